"""Comparison helpers shared by the GPU parity tests (no method arithmetic
beyond the tolerance denominators the acceptance criteria define)."""
from __future__ import annotations

import numpy as np
import torch

# Acceptance tolerances (bf16 inputs, fp32 accumulation on the GPU):
SCORE_REL = 2e-3        # |dI| <= 2e-3 * max(|I|, A),  A = sum_j |w_j| ReLU(q_j . k)
ATTN_MAX_ABS = 2e-2     # attention output, max abs error against the fp64 oracle
ATTN_MEAN_ABS = 2e-3    # attention output, mean abs error
LSE_ABS = 2e-3          # log-sum-exp (natural log)
# The kernels' lse = (m + log2 l) ln 2, where l sums the fp32 probabilities 2^(z - m) before
# they are rounded to bf16 for P.V.  Its error is therefore the fp32 error of the logits (bf16
# products are exact in fp32; 576-term fp32 sums are off by ~1e-7 relative to sum |q k|), the
# relative error of ex2.approx (2^-22) and of the fp32 sum of l: far below 2e-3 at every logit
# size the tests use, peaked softmax rows included.
TIE_REL = 1e-5          # near-tie band of the k-th oracle score
# fp32 inputs (general kernels, fp32 throughout): rounding ~1e-6 relative
FP32_ATTN_MAX_ABS = 1e-4
FP32_SCORE_REL = 1e-4


def f64(x):
    if isinstance(x, torch.Tensor):
        return x.detach().to("cpu", torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def score_denominator(q_idx_t, w_t, k_prefix, full=False):
    """A[s] = sum_j |w_j| * ReLU(q_j . k_s): the scale of the terms that add up to I[s].

    full=True gives sum_j |w_j| * sum_d |q_jd k_sd| instead, the scale that
    also covers cancellation inside each dot product (used for the tighter
    fp32 check, where rounding of near-zero dots is visible)."""
    if full:
        dots = np.abs(f64(q_idx_t)) @ np.abs(f64(k_prefix)).T
        return np.abs(f64(w_t)) @ dots
    dots = f64(q_idx_t) @ f64(k_prefix).T
    return np.abs(f64(w_t)) @ np.maximum(dots, 0.0)


def check_scores(gpu_row, ref_row, denom, rel):
    gpu_row = f64(gpu_row)
    bound = rel * np.maximum(np.abs(ref_row), denom) + 1e-30
    err = np.abs(gpu_row - ref_row)
    bad = np.nonzero(err > bound)[0]
    assert bad.size == 0, f"{bad.size} scores out of tolerance, e.g. s={bad[:5]} gpu={gpu_row[bad[:5]]} ref={ref_row[bad[:5]]}"


def check_selection(gpu_idx, ref_scores, ref_idx, k, score_err=None):
    """GPU selection = oracle selection, except elements tied with the k-th
    oracle score within the near-tie band.

    With score_err (the largest |GPU score - oracle score| of the row), a row
    whose only oracle score within 2*score_err of the k-th is the k-th itself
    cannot change its selection through score rounding, so it must match the
    oracle exactly.  Returns the number of differing positions."""
    g = np.asarray(gpu_idx, dtype=np.int64)
    n = len(ref_scores)
    keep = min(k, n)
    assert np.all(g[keep:] == -1), "padding must be -1"
    sel = g[:keep]
    assert np.all(np.diff(sel) > 0), "selected positions must be strictly ascending"
    assert sel.min() >= 0 and sel.max() < n
    ref = np.asarray(ref_idx[:keep], dtype=np.int64)
    if np.array_equal(sel, ref):
        return 0
    tau = np.sort(ref_scores)[::-1][keep - 1]
    if score_err is not None:
        fragile = int(np.count_nonzero(np.abs(ref_scores - tau) <= 2 * score_err))
        assert fragile >= 2, f"selection differs though no score lies within 2*err={2 * score_err:.2e} of tau"
    band = TIE_REL * abs(tau) + 1e-7 * np.max(np.abs(ref_scores))
    diff = np.setxor1d(sel, ref)
    far = diff[np.abs(ref_scores[diff] - tau) > band]
    assert far.size == 0, f"selection differs away from the k-th score: {far[:8]} (tau={tau})"
    return diff.size


def check_attention(gpu_out, ref_out, max_abs=ATTN_MAX_ABS, mean_abs=ATTN_MEAN_ABS):
    e = np.abs(f64(gpu_out) - ref_out)
    assert e.max() <= max_abs, f"max abs err {e.max():.3e} > {max_abs}"
    assert e.mean() <= mean_abs, f"mean abs err {e.mean():.3e} > {mean_abs}"
    return float(e.max()), float(e.mean())


def sample_rows(cu, k, per_seq=8, seed=0):
    """Deterministic sample of packed rows: t in {0, k-2, k-1, k, L-1} plus random rows per sequence."""
    rng = np.random.default_rng(seed)
    rows = []
    cu = [int(c) for c in cu]
    for b in range(len(cu) - 1):
        lo, hi = cu[b], cu[b + 1]
        L = hi - lo
        pos = {0, k - 2, k - 1, k, L - 1}
        pos |= set(int(x) for x in rng.integers(0, L, size=per_seq))
        rows += [lo + t for t in sorted(pos) if 0 <= t < L]
    return rows


# ---------------------------------------------------------------------------
# Backward tolerances (per-element bounds derived from the arithmetic)
# ---------------------------------------------------------------------------
# fp32 arithmetic of the backward kernels: ETA bounds the relative error of a dot
# product or a per-query sum of at most a few thousand terms (random-walk growth of
# 2^-24 per operation, with a wide margin); ETA_ACC that of the key-side sums, which
# add terms of every (query, head) that selected a key through fp32 atomics.
BWD_ETA = 1e-5
BWD_ETA_ACC = 1e-4
# Error of the forward output O the backward reads, as a multiple of sum_i p_i |v_i|:
# the tensor-core forward rounds the unnormalised probabilities to bf16 for P.V and O to
# bf16 (2^-9 each); an O rounded once to bf16 is off by 2^-9 |O|; the fp32 forward by ~1e-6.
O_REL_BF16_FORWARD = 2.0 ** -8
O_REL_BF16_ROUNDED = 2.0 ** -9
O_REL_FP32_FORWARD = 4e-6
# The tensor-core backward rounds p and scale * dz to bf16 before its dq / dkv products (2^-9
# each, round to nearest even), taken with a factor 2.
DZ_REL_BF16 = 2.0 ** -8
# A fp32 dot product of D_I bf16 products is off by at most (D_I - 1) 2^-24 sum |q k|;
# decisions [S > 0] with |S| inside 2e-5 sum |q k| may fall either way.
IDX_DECISION_REL = 2e-5


def attn_bwd_bounds(q_t, kv_sel, scale, d_v, dout_t, dlse_t, o_rel, dz_rel=0.0):
    """Error bounds of the GPU backward of one query row against the fp64 oracle.

    q_t [H, D_qk], kv_sel [m, D_qk] (the selected rows), dout_t [H, d_v], dlse_t [H].
    The gradient dz = p (dP - D + dlse) carries: the error of D = dO . O from the forward's
    O (o_rel * sum_d |dO_d| sum_i p_i |v_id|) and the fp32 errors of dP, D and p (ETA times
    the absolute sums).  dq and dkv add the fp32 error of their own sums and, with dz_rel, the
    rounding of dz and p to the MMA operand type.
    Returns (bound_dq [H, D_qk], bound_dkv [m, D_qk])."""
    q, ks, g = f64(q_t), f64(kv_sel), f64(dout_t)
    dl = np.zeros(q.shape[0]) if dlse_t is None else f64(dlse_t)
    z = scale * (q @ ks.T)
    z -= z.max(axis=1, keepdims=True)
    p = np.exp(z)
    p /= p.sum(axis=1, keepdims=True)
    v = ks[:, :d_v]
    o = p @ v
    dz = p * (g @ v.T - np.sum(g * o, axis=1)[:, None] + dl[:, None])
    e_d = o_rel * np.sum(np.abs(g) * (p @ np.abs(v)), axis=1)
    mag = np.abs(g) @ np.abs(v).T + np.sum(np.abs(g) * np.abs(o), axis=1)[:, None] + np.abs(dl)[:, None]
    a = p * (e_d[:, None] + 2 * BWD_ETA * mag)
    bq = scale * (a @ np.abs(ks)) + (BWD_ETA + dz_rel) * scale * (np.abs(dz) @ np.abs(ks))
    bkv = scale * (a.T @ np.abs(q)) + (BWD_ETA_ACC + dz_rel) * scale * (np.abs(dz).T @ np.abs(q))
    bkv[:, :d_v] += (BWD_ETA_ACC + dz_rel) * (p.T @ np.abs(g))
    return bq, bkv


def index_bwd_bounds(q_t, w_t, k_sel, g_sel, g_rel=0.0):
    """Error bounds of the GPU index-score backward of one row (listed keys k_sel [m, D_I],
    their gradients g_sel [m]).  Decisions inside the fp32 rounding of zero may differ from
    the fp64 oracle's: their whole term is allowed; the rest carries fp32 sum errors and, with
    g_rel, the rounding of G = g w to the MMA operand type.
    Returns (bound_dq [H_I, D_I], bound_dw [H_I], bound_dk [m, D_I])."""
    q, w, ks, g = f64(q_t), f64(w_t), f64(k_sel), f64(g_sel)
    s = q @ ks.T
    amb = np.abs(s) <= IDX_DECISION_REL * (np.abs(q) @ np.abs(ks).T)
    ga = np.abs(w)[:, None] * np.abs(g)[None, :]
    on = ga * (s > 0)
    bq = (BWD_ETA + g_rel) * (on @ np.abs(ks)) + (ga * amb) @ np.abs(ks)
    bw = BWD_ETA * (np.maximum(s, 0) @ np.abs(g)) + \
        (IDX_DECISION_REL * (np.abs(q) @ np.abs(ks).T)) @ np.abs(g)
    bk = (BWD_ETA_ACC + g_rel) * (on.T @ np.abs(q)) + (ga * amb).T @ np.abs(q)
    return bq, bw, bk
