"""Pins for the CPU oracle: checks against things other than the oracle itself.

* a pure-Python brute force written a different way (explicit loops,
  selection by repeated arg-max, softmax restricted to the selected set
  instead of an additive mask);
* closed forms: a hand-worked example, k = 1, constant value columns;
* reductions to library routines: k >= L is dense causal attention
  (torch's scaled_dot_product_attention in float64);
* invariants: orthogonal rotations of the indexer query/key (the DeepSeek-V3.2
  page's Hadamard argument, Hq.Hk = q.k), rows summing to one, the naive
  (per-head up-projected) MLA equal to the absorbed form;
* planted mistakes: each pin is re-run against a deliberately broken copy of
  the oracle and must fail there.
"""
import math

import numpy as np
import pytest
import scipy.linalg
import torch

import oracle.dsa_oracle as O

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ---------------------------------------------------------------------------
# brute force (independent restatement, pure Python)
# ---------------------------------------------------------------------------
def bf_scores(qI, w, kI, t):
    out = []
    for s in range(t + 1):
        acc = 0.0
        for j in range(len(qI)):
            d = 0.0
            for c in range(len(kI[s])):
                d += float(qI[j][c]) * float(kI[s][c])
            if d > 0.0:
                acc += float(w[j]) * d
        out.append(acc)
    return out


def bf_topk(scores, k):
    remaining = list(range(len(scores)))
    chosen = []
    while remaining and len(chosen) < k:
        best = remaining[0]
        for s in remaining[1:]:  # ascending scan: strict '>' keeps the lower position
            if scores[s] > scores[best]:
                best = s
        chosen.append(best)
        remaining.remove(best)
    chosen.sort()
    return chosen + [-1] * (k - len(chosen))


def bf_attention(q_t, kv, sel, scale, d_v):
    H = len(q_t)
    outs, lses = [], []
    for h in range(H):
        logits = []
        for s in sel:
            if s < 0:
                continue
            logits.append(scale * sum(float(a) * float(b) for a, b in zip(q_t[h], kv[s])))
        mx = max(logits)
        ex = [math.exp(z - mx) for z in logits]
        tot = sum(ex)
        valid = [s for s in sel if s >= 0]
        o = [sum(ex[i] * float(kv[s][c]) for i, s in enumerate(valid)) / tot for c in range(d_v)]
        outs.append(o)
        lses.append(mx + math.log(tot))
    return np.array(outs), np.array(lses)


def _rand_case(rng, lens, H_I=3, D_I=5, H=2, D_qk=7, d_v=4):
    T = sum(lens)
    q_idx = rng.standard_normal((T, H_I, D_I))
    w = rng.standard_normal((T, H_I))
    k_idx = rng.standard_normal((T, D_I))
    q = rng.standard_normal((T, H, D_qk))
    kv = rng.standard_normal((T, D_qk))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    return q_idx, w, k_idx, q, kv, cu


def check_bruteforce(mod, k, lens=(9, 5), seed=1, scale=0.7, d_v=4):
    rng = np.random.default_rng(seed)
    q_idx, w, k_idx, q, kv, cu = _rand_case(rng, list(lens), d_v=d_v)
    res = mod.dsa_prefill(q_idx, w, k_idx, q, kv, cu, k, scale, d_v)
    for i, r in enumerate(range(cu[-1])):
        b = int(np.searchsorted(cu, r, side="right") - 1)
        lo, hi = cu[b], cu[b + 1]
        t = r - lo
        sc = bf_scores(q_idx[r], w[r], k_idx[lo:hi], t)
        if not np.allclose(res["scores"][i], sc, rtol=1e-12, atol=1e-12):
            return False
        sel = bf_topk(sc, k)
        if list(res["idx"][i]) != sel:
            return False
        o, l = bf_attention(q[r], kv[lo:hi], sel, scale, d_v)
        if not (np.allclose(res["out"][i], o, rtol=1e-12, atol=1e-12)
                and np.allclose(res["lse"][i], l, rtol=1e-12, atol=1e-12)):
            return False
    return True


@pytest.mark.parametrize("k", [1, 3, 14])
def test_bruteforce_matches_oracle(k):
    assert check_bruteforce(O, k)


def test_bruteforce_topk_with_ties_and_signed_zero():
    rng = np.random.default_rng(3)
    for n in [1, 2, 7, 40, 200]:
        for k in [1, 5, 64]:
            s = rng.integers(-3, 4, size=n).astype(np.float64)
            s[s == 0] = np.where(rng.random((s == 0).sum()) < 0.5, 0.0, -0.0)
            assert list(O.topk_select(s, k)) == bf_topk(list(s), k)


# ---------------------------------------------------------------------------
# hand-worked example (closed form)
# ---------------------------------------------------------------------------
def test_hand_worked_example():
    # Two indexer heads of width 2; the query at position 2 has heads e0, e1
    # and weights (+1, -1), so I[2,s] = max(0, k_s[0]) - max(0, k_s[1]).
    #   k_0 = ( 1,  2) -> 1 - 2 = -1
    #   k_1 = ( 3, -1) -> 3 - 0 =  3
    #   k_2 = (-2,  1) -> 0 - 1 = -1
    # k = 2 keeps position 1 and one of the tied -1 scores: the lower
    # position, 0.  Attention (one head, scale 1): q = (ln 3, 0) against
    # keys kv_0 = (0, 5), kv_1 = (1, 7) gives logits 0 and ln 3, so
    # p = (1/4, 3/4) and O = kv[:,1] weighted = 5/4 + 21/4 = 6.5,
    # lse = log(1 + 3) = log 4.
    q_idx = np.zeros((3, 2, 2))
    q_idx[2] = [[1.0, 0.0], [0.0, 1.0]]
    w = np.zeros((3, 2))
    w[2] = [1.0, -1.0]
    k_idx = np.array([[1.0, 2.0], [3.0, -1.0], [-2.0, 1.0]])
    q = np.zeros((3, 1, 2))
    q[2, 0] = [math.log(3.0), 0.0]
    kv = np.array([[0.0, 5.0], [1.0, 7.0], [100.0, 100.0]])
    res = O.dsa_prefill(q_idx, w, k_idx, q, kv, [0, 3], 2, 1.0, 2, rows=[2])
    assert np.array_equal(res["scores"][0], [-1.0, 3.0, -1.0])
    assert list(res["idx"][0]) == [0, 1]
    assert res["out"][0, 0, 1] == pytest.approx(6.5, abs=1e-12)
    assert res["out"][0, 0, 0] == pytest.approx(0.75, abs=1e-12)
    assert res["lse"][0, 0] == pytest.approx(math.log(4.0), abs=1e-12)


# ---------------------------------------------------------------------------
# k >= L reduces to dense causal attention (library routine)
# ---------------------------------------------------------------------------
def check_dense_when_k_ge_L(mod, L=23, H=3, D=9, d_v=6, scale=0.31, seed=5):
    rng = np.random.default_rng(seed)
    q_idx, w, k_idx, q, kv, cu = _rand_case(rng, [L], H=H, D_qk=D, d_v=d_v)
    res = mod.dsa_prefill(q_idx, w, k_idx, q, kv, cu, L + 4, scale, d_v)
    qt = torch.from_numpy(q).permute(1, 0, 2)[None]                 # [1,H,L,D]
    kt = torch.from_numpy(kv)[None, None].expand(1, H, L, D)
    vt = torch.from_numpy(kv[:, :d_v])[None, None].expand(1, H, L, d_v)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True, scale=scale)
    ref = ref[0].permute(1, 0, 2).numpy()
    return np.allclose(res["out"], ref, rtol=1e-12, atol=1e-12)


def test_dense_causal_when_k_ge_L():
    assert check_dense_when_k_ge_L(O)


# ---------------------------------------------------------------------------
# invariants
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("D_I", [32, 128])
def test_index_scores_rotation_invariant(D_I):
    rng = np.random.default_rng(D_I)
    L, H_I = 17, 6
    q_idx = rng.standard_normal((L, H_I, D_I))
    w = rng.standard_normal((L, H_I))
    k_idx = rng.standard_normal((L, D_I))
    base = O.index_scores(q_idx, w, k_idx)
    R, _ = np.linalg.qr(rng.standard_normal((D_I, D_I)))
    Hd = scipy.linalg.hadamard(D_I) / math.sqrt(D_I)
    fin = np.isfinite(base)
    for M in (R, Hd):
        rot = O.index_scores(q_idx @ M.T, w, k_idx @ M.T)
        assert np.array_equal(np.isfinite(rot), fin)
        assert np.allclose(rot[fin], base[fin], rtol=1e-12, atol=1e-12)


def check_rows_sum_to_one(mod, seed=7):
    rng = np.random.default_rng(seed)
    q_idx, w, k_idx, q, kv, cu = _rand_case(rng, [30, 11], d_v=4)
    kv[:, 2] = 1.0   # a constant value column: the output there is the row sum of p
    res = mod.dsa_prefill(q_idx, w, k_idx, q, kv, cu, 5, 0.9, 4)
    return np.allclose(res["out"][:, :, 2], 1.0, rtol=0, atol=1e-12)


def test_softmax_rows_sum_to_one():
    assert check_rows_sum_to_one(O)


def test_naive_mla_equals_absorbed():
    # Naive per-head MLA (each head up-projects the shared latent into its own
    # key/value) with the additive selection mask, against the absorbed form
    # the oracle implements, followed by the per-head value up-projection.
    rng = np.random.default_rng(11)
    L, H, lat, rope, nope, vdim, k, scale = 19, 3, 16, 4, 8, 5, 6, 0.4
    c = rng.standard_normal((L, lat))            # kv latent
    k_rope = rng.standard_normal((L, rope))
    q_nope = rng.standard_normal((L, H, nope))
    q_rope = rng.standard_normal((L, H, rope))
    W_UK = rng.standard_normal((H, nope, lat))
    W_UV = rng.standard_normal((H, vdim, lat))
    q_idx = rng.standard_normal((L, 2, 3))
    w = rng.standard_normal((L, 2))
    k_idx = rng.standard_normal((L, 3))
    q_abs = np.concatenate([np.einsum("thn,hnl->thl", q_nope, W_UK), q_rope], axis=2)
    kv_abs = np.concatenate([c, k_rope], axis=1)
    res = O.dsa_prefill(q_idx, w, k_idx, q_abs, kv_abs, [0, L], k, scale, lat)
    for t in range(L):
        sel = res["idx"][t]
        mask = np.full(L, -np.inf)
        mask[sel[sel >= 0]] = 0.0
        for h in range(H):
            keys = c @ W_UK[h].T                  # [L, nope]
            vals = c @ W_UV[h].T                  # [L, vdim]
            z = scale * (keys @ q_nope[t, h] + k_rope @ q_rope[t, h]) + mask
            p = np.exp(z - z.max())
            p /= p.sum()
            naive = p @ vals
            absorbed = W_UV[h] @ res["out"][t, h]
            assert np.allclose(naive, absorbed, rtol=1e-10, atol=1e-10)


def test_k1_returns_argmax_row():
    rng = np.random.default_rng(13)
    q_idx, w, k_idx, q, kv, cu = _rand_case(rng, [25], d_v=4)
    res = O.dsa_prefill(q_idx, w, k_idx, q, kv, cu, 1, 0.5, 4)
    for t in range(25):
        s = int(np.argmax(res["scores"][t]))
        assert res["idx"][t, 0] == s
        assert np.array_equal(res["out"][t], np.broadcast_to(kv[s, :4], (2, 4)))


def test_varlen_is_per_sequence_and_decode_is_last_row():
    rng = np.random.default_rng(17)
    lens = [7, 12, 4]
    q_idx, w, k_idx, q, kv, cu = _rand_case(rng, lens, d_v=4)
    packed = O.dsa_prefill(q_idx, w, k_idx, q, kv, cu, 5, 0.8, 4)
    for b in range(3):
        lo, hi = cu[b], cu[b + 1]
        one = O.dsa_prefill(q_idx[lo:hi], w[lo:hi], k_idx[lo:hi], q[lo:hi], kv[lo:hi], [0, hi - lo], 5, 0.8, 4)
        assert np.array_equal(packed["idx"][lo:hi], one["idx"])
        assert np.array_equal(packed["out"][lo:hi], one["out"])
    # decode over caches whose valid prefix is sequence b equals its last prefill row
    max_ctx = 16
    B = 3
    idx_cache = rng.standard_normal((B, max_ctx, 5))
    kv_cache = rng.standard_normal((B, max_ctx, 7))
    last = [cu[b + 1] - 1 for b in range(B)]
    for b in range(B):
        n = lens[b]
        idx_cache[b, :n] = k_idx[cu[b]:cu[b + 1]]
        kv_cache[b, :n] = kv[cu[b]:cu[b + 1]]
    dec = O.dsa_decode(q_idx[last], w[last], q[last], idx_cache, kv_cache, lens, 5, 0.8, 4)
    assert np.array_equal(dec["idx"], packed["idx"][last])
    assert np.array_equal(dec["out"], packed["out"][last])


# ---------------------------------------------------------------------------
# planted mistakes: every pin above must catch at least one of these
# ---------------------------------------------------------------------------
class _Mutant:
    """The oracle with some of its functions replaced for the duration of a call."""

    def __init__(self, **repl):
        self._repl = repl

    def __getattr__(self, name):
        return self._repl.get(name, getattr(O, name))

    def dsa_prefill(self, *a, **kw):
        saved = {k: getattr(O, k) for k in self._repl}
        try:
            for k, v in self._repl.items():
                setattr(O, k, v)
            return O.dsa_prefill(*a, **kw)
        finally:
            for k, v in saved.items():
                setattr(O, k, v)


def _no_relu(q, w, k):
    return O._f64(w) @ (O._f64(q) @ O._f64(k).T)


def _ties_high(scores, k):
    s = O._f64(scores)
    order = np.argsort(-s[::-1], kind="stable")[: min(k, len(s))]
    out = np.full(k, -1, dtype=np.int64)
    out[: len(order)] = np.sort(len(s) - 1 - order)
    return out


def _strict_causal_mask(sel, L):
    m = np.full(L, -np.inf)
    sel = np.asarray(sel)
    m[sel[sel >= 0]] = 0.0
    m[sel[sel >= 0].max()] = -np.inf if (sel >= 0).sum() > 1 else 0.0
    return m


_ORIG_ATTN = O.masked_attention_row


def _value_from_wrong_columns(q_t, kv, mask_row, scale, d_v):
    kv = O._f64(kv)
    out, lse = _ORIG_ATTN(q_t, kv, mask_row, scale, kv.shape[1])
    return out[:, kv.shape[1] - d_v:], lse


def _unscaled(q_t, kv, mask_row, scale, d_v):
    return _ORIG_ATTN(q_t, kv, mask_row, 1.0, d_v)


@pytest.mark.parametrize("mutant", [
    {"index_scores_row": _no_relu},
    {"topk_select": _ties_high},
    {"additive_mask_row": _strict_causal_mask},
    {"masked_attention_row": _value_from_wrong_columns},
    {"masked_attention_row": _unscaled},
])
def test_pins_catch_planted_mistakes(mutant):
    m = _Mutant(**mutant)
    caught = not check_bruteforce(m, 3)
    # ties only show up with repeated scores: brute force over an integer case
    if "topk_select" in mutant:
        s = np.array([1.0, 2.0, 1.0, 2.0, 0.0])
        caught = caught or list(m.topk_select(s, 3)) != bf_topk(list(s), 3)
    assert caught
