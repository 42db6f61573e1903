"""Pins for the oracle's backward: checks against things other than the backward itself.

* central finite differences of the forward oracle (itself pinned by the
  brute force, closed forms and library reductions of the forward's pins);
* a reduction to a library routine: with every causal position selected the
  step is dense causal attention, whose gradient torch's autograd gives in
  float64;
* closed forms: one selected key (softmax of one logit has zero gradient, the
  output is that key's value row);
* invariants: the index score is positively homogeneous of degree one in each
  of w, q_I and k_I (the ReLU is), so <dw, w> = <dq, q> = <dk, k> = <g, I>;
* planted mistakes: broken copies of the backward must fail the pins.
"""
import numpy as np
import pytest
import torch

import oracle.dsa_oracle as O

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

EPS = 1e-6


def _fd(f, x, eps=EPS):
    """Central differences of the scalar f at every element of x (modified in place, restored)."""
    g = np.zeros_like(x)
    flat, gf = x.reshape(-1), g.reshape(-1)
    for i in range(flat.size):
        v = flat[i]
        flat[i] = v + eps
        hi = f()
        flat[i] = v - eps
        lo = f()
        flat[i] = v
        gf[i] = (hi - lo) / (2 * eps)
    return g


# ---------------------------------------------------------------------------
# attention (step 4 with the selection fixed)
# ---------------------------------------------------------------------------
def _attn_case(seed, H=3, L=7, dqk=10, d_v=6, n_sel=4):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((H, dqk))
    kv = rng.standard_normal((L, dqk))
    sel = np.sort(rng.choice(L, n_sel, replace=False))
    mask = O.additive_mask_row(sel, L)
    dout = rng.standard_normal((H, d_v))
    dlse = rng.standard_normal(H)
    return q, kv, mask, dout, dlse, 0.37


def check_attention_fd(bwd, seed=0, with_lse=True):
    q, kv, mask, dout, dlse, scale = _attn_case(seed)
    d_v = dout.shape[1]
    dl = dlse if with_lse else None

    def loss():
        out, lse = O.masked_attention_row(q, kv, mask, scale, d_v)
        return float(np.sum(dout * out) + (np.sum(dlse * lse) if with_lse else 0.0))

    dq, dkv = bwd(q, kv, mask, scale, d_v, dout, dl)
    ok_q = np.allclose(dq, _fd(loss, q), rtol=1e-6, atol=1e-8)
    ok_kv = np.allclose(dkv, _fd(loss, kv), rtol=1e-6, atol=1e-8)
    return ok_q and ok_kv


@pytest.mark.parametrize("with_lse", [False, True])
@pytest.mark.parametrize("seed", [0, 1])
def test_attention_backward_matches_finite_differences(seed, with_lse):
    assert check_attention_fd(O.masked_attention_row_backward, seed, with_lse)


def check_packed_attention_fd(bwd_row):
    """The packed backward against differences of the whole forward oracle (two sequences).

    Perturbing q or kv leaves the index scores (a function of q_I, w, k_I only) and so
    the selection unchanged; the forward oracle's out and lse are then smooth in q, kv.
    """
    rng = np.random.default_rng(7)
    cu = np.array([0, 5, 12])
    T, HI, DI, H, dqk, d_v, topk, scale = 12, 2, 4, 2, 6, 4, 3, 0.45
    q_idx = rng.standard_normal((T, HI, DI))
    w = rng.standard_normal((T, HI))
    k_idx = rng.standard_normal((T, DI))
    q = rng.standard_normal((T, H, dqk))
    kv = rng.standard_normal((T, dqk))
    dout = rng.standard_normal((T, H, d_v))
    dlse = rng.standard_normal((T, H))

    def loss():
        r = O.dsa_prefill(q_idx, w, k_idx, q, kv, cu, topk, scale, d_v)
        return float(np.sum(dout * r["out"]) + np.sum(dlse * r["lse"]))

    idx = O.dsa_prefill(q_idx, w, k_idx, q, kv, cu, topk, scale, d_v)["idx"]
    saved = O.masked_attention_row_backward
    O.masked_attention_row_backward = bwd_row
    try:
        res = O.sparse_attention_backward(q, kv, idx, cu, scale, d_v, dout, dlse)
    finally:
        O.masked_attention_row_backward = saved
    ok_kv = np.allclose(res["dkv"], _fd(loss, kv), rtol=1e-6, atol=1e-8)
    ok_q = np.allclose(res["dq"], _fd(loss, q), rtol=1e-6, atol=1e-8)
    return ok_kv and ok_q


def test_packed_attention_backward_matches_finite_differences():
    assert check_packed_attention_fd(O.masked_attention_row_backward)


def test_dense_causal_backward_is_autograd_of_sdpa():
    """k >= L: the packed backward equals torch autograd of dense causal attention, per sequence."""
    rng = np.random.default_rng(3)
    cu = np.array([0, 6, 15])
    T, H, dqk, d_v, scale = 15, 3, 12, 8, 0.3
    q = rng.standard_normal((T, H, dqk))
    kv = rng.standard_normal((T, dqk))
    dout = rng.standard_normal((T, H, d_v))
    dlse = rng.standard_normal((T, H))
    idx = np.full((T, 16), -1)
    for b in range(2):
        for r in range(cu[b], cu[b + 1]):
            t = r - cu[b]
            idx[r, : t + 1] = np.arange(t + 1)
    res = O.sparse_attention_backward(q, kv, idx, cu, scale, d_v, dout, dlse)
    for b in range(2):
        lo, hi = cu[b], cu[b + 1]
        L = hi - lo
        qt = torch.tensor(q[lo:hi], requires_grad=True)                 # [L,H,D]
        kt = torch.tensor(kv[lo:hi], requires_grad=True)                # [L,D]
        qh = qt.permute(1, 0, 2)[None]                                  # [1,H,L,D]
        kh = kt[None, None].expand(1, H, L, dqk)
        vh = kt[:, :d_v][None, None].expand(1, H, L, d_v)
        out = torch.nn.functional.scaled_dot_product_attention(qh, kh, vh, is_causal=True, scale=scale)
        causal = torch.full((L, L), float("-inf"), dtype=torch.float64).triu(1)
        lse = torch.logsumexp(scale * (qh @ kh.transpose(-1, -2)) + causal, dim=-1)   # [1,H,L]
        loss = (torch.tensor(dout[lo:hi]).permute(1, 0, 2)[None] * out).sum() + \
            (torch.tensor(dlse[lo:hi]).T[None] * lse).sum()
        loss.backward()
        assert np.allclose(res["dq"][lo:hi], qt.grad.numpy(), rtol=1e-10, atol=1e-12)
        assert np.allclose(res["dkv"][lo:hi], kt.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_single_selected_key_closed_form():
    """One selected key s: p = 1, O = kv[s,:d_v]; dz = dlse, so dq = scale*dlse*kv[s] and
    dkv[s] = scale*sum_h dlse_h q_h + [sum_h dO_h on the value columns]; nothing elsewhere."""
    rng = np.random.default_rng(5)
    H, L, dqk, d_v, scale = 4, 9, 10, 6, 0.8
    q = rng.standard_normal((H, dqk))
    kv = rng.standard_normal((L, dqk))
    dout = rng.standard_normal((H, d_v))
    dlse = rng.standard_normal(H)
    s = 6
    mask = O.additive_mask_row([s], L)
    dq, dkv = O.masked_attention_row_backward(q, kv, mask, scale, d_v, dout, None)
    assert np.allclose(dq, 0.0, atol=1e-14)
    want = np.zeros((L, dqk))
    want[s, :d_v] = dout.sum(axis=0)
    assert np.allclose(dkv, want, atol=1e-14)
    dq, dkv = O.masked_attention_row_backward(q, kv, mask, scale, d_v, dout, dlse)
    assert np.allclose(dq, scale * dlse[:, None] * kv[s][None, :], atol=1e-14)
    want[s] += scale * (dlse @ q)
    assert np.allclose(dkv, want, atol=1e-14)


# ---------------------------------------------------------------------------
# indexer (step 1 read at listed positions)
# ---------------------------------------------------------------------------
def _idx_case(seed, HI=3, DI=8, n=9, m=5):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((HI, DI))
    w = rng.standard_normal(HI)
    k = rng.standard_normal((n, DI))
    pos = np.sort(rng.choice(n, m, replace=False))
    g = rng.standard_normal(m)
    # the ReLU kink must stay far from every dot product for differences to apply
    assert np.min(np.abs(q @ k[pos].T)) > 1e-3
    return q, w, k, pos, g


def check_indexer_fd(bwd, seed=0):
    q, w, k, pos, g = _idx_case(seed)

    def loss():
        return float(g @ O.index_scores_row(q, w, k)[pos])

    dq, dw, dk = bwd(q, w, k, np.concatenate([pos, [-1]]), np.concatenate([g, [5.0]]))
    return (np.allclose(dq, _fd(loss, q), rtol=1e-6, atol=1e-8)
            and np.allclose(dw, _fd(loss, w), rtol=1e-6, atol=1e-8)
            and np.allclose(dk, _fd(loss, k), rtol=1e-6, atol=1e-8))


@pytest.mark.parametrize("seed", [0, 2])
def test_indexer_backward_matches_finite_differences(seed):
    assert check_indexer_fd(O.index_scores_row_backward, seed)


def test_indexer_backward_homogeneity():
    """I is positively homogeneous of degree 1 in w, in q_I and in k_I (ReLU(a x) = a ReLU(x),
    a > 0), so by Euler's theorem each gradient paired with its argument gives <g, I[pos]>."""
    rng = np.random.default_rng(11)
    HI, DI, n = 6, 16, 40
    q = rng.standard_normal((HI, DI))
    w = rng.standard_normal(HI)
    k = rng.standard_normal((n, DI))
    pos = np.arange(0, n, 3)
    g = rng.standard_normal(pos.size)
    dq, dw, dk = O.index_scores_row_backward(q, w, k, pos, g)
    gi = float(g @ O.index_scores_row(q, w, k)[pos])
    assert abs(float(np.sum(dw * w)) - gi) < 1e-12 * max(1.0, abs(gi))
    assert abs(float(np.sum(dq * q)) - gi) < 1e-12 * max(1.0, abs(gi))
    assert abs(float(np.sum(dk * k)) - gi) < 1e-12 * max(1.0, abs(gi))


def test_packed_indexer_backward_matches_finite_differences():
    """The packed form against differences of the full causal score matrices, two sequences."""
    rng = np.random.default_rng(13)
    cu = np.array([0, 4, 10])
    T, HI, DI, m = 10, 2, 6, 3
    q_idx = rng.standard_normal((T, HI, DI))
    w = rng.standard_normal((T, HI))
    k_idx = rng.standard_normal((T, DI))
    idx = np.full((T, m), -1)
    for b in range(2):
        for r in range(cu[b], cu[b + 1]):
            t = r - cu[b]
            c = min(m, t + 1)
            idx[r, :c] = np.sort(rng.choice(t + 1, c, replace=False))
    g = rng.standard_normal((T, m))

    def loss():
        tot = 0.0
        for b in range(2):
            lo, hi = cu[b], cu[b + 1]
            I = O.index_scores(q_idx[lo:hi], w[lo:hi], k_idx[lo:hi])
            for r in range(lo, hi):
                for j in range(m):
                    if idx[r, j] >= 0:
                        tot += g[r, j] * I[r - lo, idx[r, j]]
        return tot

    res = O.index_scores_backward(q_idx, w, k_idx, idx, g, cu)
    assert np.allclose(res["dk"], _fd(loss, k_idx), rtol=1e-6, atol=1e-8)
    assert np.allclose(res["dq"], _fd(loss, q_idx), rtol=1e-6, atol=1e-8)
    assert np.allclose(res["dw"], _fd(loss, w), rtol=1e-6, atol=1e-8)


# ---------------------------------------------------------------------------
# planted mistakes: the pins above must reject broken backwards
# ---------------------------------------------------------------------------
def _attn_no_value_term(q_t, kv, mask_row, scale, d_v, dout, dlse=None):
    # drops sum_h p[h,s] dO[h,:] from the value columns of dkv
    dq, dkv = O.masked_attention_row_backward(q_t, kv, mask_row, scale, d_v, dout, dlse)
    dkv = dkv.copy()
    dkv[:, :d_v] -= _value_term(q_t, kv, mask_row, scale, d_v, dout)
    return dq, dkv


def _value_term(q_t, kv, mask_row, scale, d_v, dout):
    q, k = O._f64(q_t), O._f64(kv)
    z = scale * (q @ k.T) + mask_row[None, :]
    p = np.exp(z - z.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    return p.T @ O._f64(dout)


def _attn_wrong_sign_d(q_t, kv, mask_row, scale, d_v, dout, dlse=None):
    # D added instead of subtracted: equivalent to the true backward with dlse + 2 D
    q, k, g = O._f64(q_t), O._f64(kv), O._f64(dout)
    out, _ = O.masked_attention_row(q, k, mask_row, scale, d_v)
    dd = np.sum(g * out, axis=1)
    base = np.zeros(q.shape[0]) if dlse is None else O._f64(dlse)
    return O.masked_attention_row_backward(q, k, mask_row, scale, d_v, g, base + 2 * dd)


def _attn_unscaled(q_t, kv, mask_row, scale, d_v, dout, dlse=None):
    dq, dkv = O.masked_attention_row_backward(q_t, kv, mask_row, scale, d_v, dout, dlse)
    return dq / scale, dkv


def _idx_no_w(q_idx_t, w_t, k_idx_prefix, positions, d_scores):
    return O.index_scores_row_backward(q_idx_t, np.ones_like(O._f64(w_t)), k_idx_prefix, positions, d_scores)


def _idx_transposed_dk(q_idx_t, w_t, k_idx_prefix, positions, d_scores):
    dq, dw, dk = O.index_scores_row_backward(q_idx_t, w_t, k_idx_prefix, positions, d_scores)
    return dq, dw, dk[::-1].copy()


@pytest.mark.parametrize("mutant", [_attn_no_value_term, _attn_wrong_sign_d, _attn_unscaled])
def test_attention_pins_catch_planted_mistakes(mutant):
    assert not (check_attention_fd(mutant, 0, True) and check_packed_attention_fd(mutant))


@pytest.mark.parametrize("mutant", [_idx_no_w, _idx_transposed_dk])
def test_indexer_pins_catch_planted_mistakes(mutant):
    assert not check_indexer_fd(mutant, 0)
