"""Pins for the oracle's FP8 form of the indexer scores (no GPU).

The DeepSeek-V3.2 page says the reference indexer runs in FP8 after a
Hadamard transform, and that the transform is orthogonal (Hq . Hk = q . k).
The oracle's reading (rotate by H / sqrt(d), one E4M3 scale amax/448 per
rotated vector) is checked here against things other than itself:

* E4M3 rounding against torch's own float8_e4m3fn conversion (a library
  routine), on every grid value, every midpoint and random values;
* the Hadamard matrix against scipy.linalg.hadamard, and its orthogonality;
* a closed case: inputs whose rotations are exactly on the scaled E4M3 grid
  must give the bf16/fp64 scores exactly (the rotation changes nothing);
* the rounding error bound: |I_fp8 - I| <= sum_j |w_j| * sum_i (dq|k| + |q|dk + dq dk)
  with dx <= max(2^-4 |x|, 2^-10 * scale) per element (half an E4M3 spacing);
* planted mistakes, each of which must fail one of the pins above.
"""
import numpy as np
import pytest
import scipy.linalg
import torch

import oracle.dsa_oracle as O

D = 128


def _grid():
    """Every finite E4M3 value, from torch's own decoding of the 256 codes."""
    codes = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    return np.unique(codes[np.isfinite(codes)])


def _torch_round(x32):
    return torch.from_numpy(x32).to(torch.float8_e4m3fn).float().numpy().astype(np.float64)


# ---------------------------------------------------------------------------
# E4M3 rounding and the Hadamard matrix against library routines
# ---------------------------------------------------------------------------
def test_e4m3_round_matches_torch_conversion():
    g = _grid()
    assert g.max() == 448.0 and g.min() == -448.0 and len(g) == 253    # +0/-0 merge; 2 NaN codes
    mids = (g[:-1] + g[1:]) / 2                                          # exact ties in fp32
    rng = np.random.default_rng(0)
    rand = np.concatenate([rng.standard_normal(20000) * s for s in (1e-4, 1e-2, 1.0, 30.0, 200.0)])
    x = np.clip(np.concatenate([g, mids, rand, [0.0, -0.0, 2.0 ** -10, 2.0 ** -9, 3 * 2.0 ** -10]]), -448, 448)
    x32 = x.astype(np.float32)
    got = O.e4m3_round(x32.astype(np.float64))
    assert np.array_equal(got, _torch_round(x32))
    assert np.array_equal(np.signbit(got[got == 0]), np.signbit(x32[got == 0]))


def test_e4m3_round_saturates():
    assert O.e4m3_round(np.array([500.0, -1e6]))[0] == 448.0
    assert O.e4m3_round(np.array([500.0, -1e6]))[1] == -448.0


@pytest.mark.parametrize("n", [1, 2, 4, 8, 16, 32, 64, 128])
def test_hadamard_is_sylvester_and_orthogonal(n):
    h = O.hadamard(n)
    assert np.array_equal(h, scipy.linalg.hadamard(n).astype(np.float64))
    assert np.array_equal(h @ h.T, n * np.eye(n))


def test_hadamard_rejects_non_powers_of_two():
    with pytest.raises(ValueError):
        O.hadamard(3)


# ---------------------------------------------------------------------------
# the FP8 scores: closed case and error bound
# ---------------------------------------------------------------------------
def _representable_inputs(rng, h, n):
    """q, k whose normalised-Hadamard rotations are (grid value) x (power-of-two scale), each row
    reaching +-448 x scale, so the FP8 form represents them exactly."""
    g = _grid()
    rot = scipy.linalg.hadamard(D) / np.sqrt(D)

    def rows(m):
        v = rng.choice(g, size=(m, D))
        v[:, 0] = np.where(rng.random(m) < 0.5, 448.0, -448.0)     # each row's amax is exactly 448
        scale = np.exp2(rng.integers(-12, -4, size=m).astype(np.float64))
        return (v * scale[:, None]) @ rot                           # rot is symmetric and orthogonal

    return rows(h), rows(n)


def _check_exact(score_fn, seed=0):
    rng = np.random.default_rng(seed)
    q, k = _representable_inputs(rng, 8, 40)
    w = rng.standard_normal(8)
    got = score_fn(q, w, k)
    ref = O.index_scores_row(q, w, k)                               # the bf16-path definition
    tol = 1e-12 * (np.abs(w) @ np.abs(q @ k.T) + 1e-30)
    return bool(np.all(np.abs(got - ref) <= tol))


def _check_bound(score_fn, seed=1):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((8, D)) / np.sqrt(D)
    k = rng.standard_normal((60, D)) / np.sqrt(D) + rng.standard_normal((60, 1)) * 0.5
    w = rng.standard_normal(8) / np.sqrt(8)
    rot = scipy.linalg.hadamard(D) / np.sqrt(D)
    qr, kr = q @ rot.T, k @ rot.T
    sq = np.abs(qr).max(axis=1) / 448.0
    sk = np.abs(kr).max(axis=1) / 448.0
    dq = np.maximum(2.0 ** -4 * np.abs(qr), 2.0 ** -10 * sq[:, None])   # half an E4M3 spacing, scaled
    dk = np.maximum(2.0 ** -4 * np.abs(kr), 2.0 ** -10 * sk[:, None])
    per_dot = dq @ np.abs(kr).T + np.abs(qr) @ dk.T + dq @ dk.T         # [H, n]
    bound = np.abs(w) @ per_dot
    err = np.abs(score_fn(q, w, k) - O.index_scores_row(q, w, k))
    return bool(np.all(err <= bound * (1 + 1e-9) + 1e-15))


def test_fp8_scores_exact_on_representable_inputs():
    for seed in range(3):
        assert _check_exact(O.index_scores_fp8_row, seed)


def test_fp8_scores_within_the_rounding_bound():
    for seed in range(1, 4):
        assert _check_bound(O.index_scores_fp8_row, seed)


def test_fp8_scores_do_differ_from_the_exact_ones():
    """On generic inputs the FP8 form is not the exact form (so the pins above are not vacuous)."""
    rng = np.random.default_rng(5)
    q = rng.standard_normal((8, D))
    k = rng.standard_normal((30, D))
    w = rng.standard_normal(8)
    assert np.abs(O.index_scores_fp8_row(q, w, k) - O.index_scores_row(q, w, k)).max() > 1e-6


# ---------------------------------------------------------------------------
# planted mistakes: each must fail the exact case or the bound
# ---------------------------------------------------------------------------
def _fp8_with(rot_q=True, rot_k=True, qmax=448.0, relu=True, rescale=True):
    def fn(q_t, w_t, k_pre):
        q, w, k = O._f64(q_t), O._f64(w_t), O._f64(k_pre)
        rot = O.hadamard(D) / np.sqrt(D)
        qr = q @ rot.T if rot_q else q
        kr = k @ rot.T if rot_k else k

        def quant(x):
            s = np.abs(x).max(axis=1) / qmax
            return O.e4m3_round(x / s[:, None]), s

        q8, sq = quant(qr)
        k8, sk = quant(kr)
        dots = q8 @ k8.T
        if rescale:
            dots = dots * sq[:, None] * sk[None, :]
        return w @ (np.maximum(dots, 0.0) if relu else dots)
    return fn


def _truncating_e4m3(x):
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    e = np.clip(np.floor(np.log2(np.where(a > 0, a, 1.0))), -6, 8)
    q = np.exp2(e - 3)
    return np.copysign(np.minimum(np.floor(a / q) * q, 448.0), x)


@pytest.mark.parametrize("name,fn", [
    ("key not rotated", _fp8_with(rot_k=False)),
    ("scale amax/127", _fp8_with(qmax=127.0)),
    ("no ReLU", _fp8_with(relu=False)),
    ("scales not applied", _fp8_with(rescale=False)),
])
def test_fp8_pins_catch_planted_mistakes(name, fn):
    assert fn is not None
    assert not (_check_exact(fn) and _check_bound(fn)), name


def test_fp8_pins_catch_truncating_rounding(monkeypatch):
    monkeypatch.setattr(O, "e4m3_round", _truncating_e4m3)
    assert not (_check_exact(O.index_scores_fp8_row) and _check_bound(O.index_scores_fp8_row))


def test_fp8_scores_from_codes_reduce_to_the_plain_definition():
    """With unit scales, scoring from given codes is the plain indexer score of those values."""
    rng = np.random.default_rng(7)
    g = _grid()
    q8 = rng.choice(g[np.abs(g) <= 8], size=(6, D))
    k8 = rng.choice(g[np.abs(g) <= 8], size=(9, D))
    w = rng.standard_normal(6)
    got = O.index_scores_fp8_codes(q8, np.ones(6), w, k8, np.ones(9))
    assert np.allclose(got, O.index_scores_row(q8, w, k8), rtol=1e-12, atol=1e-12)
    # positive scales factor out of the ReLU
    sq, sk = rng.uniform(0.5, 2.0, 6), rng.uniform(0.5, 2.0, 9)
    got2 = O.index_scores_fp8_codes(q8, sq, w, k8, sk)
    assert np.allclose(got2, sk * O.index_scores_row(q8, w * sq, k8), rtol=1e-12, atol=1e-12)
