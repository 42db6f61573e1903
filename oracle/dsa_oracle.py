"""CPU oracle for the DeepSeek Sparse Attention (DSA) forward step and its backward.

TEST INFRASTRUCTURE ONLY.  This module is the slow, plainly written
definition that the CUDA library is checked against.  Only the test suite,
the smoke check and the benchmark's CPU-baseline leg may import it; the
library itself never calls it and has no CPU fallback.

Everything here is numpy in float64.  Inputs arrive as whatever the caller
generated (fp32 or bf16 values); they are widened exactly to float64 before
any arithmetic.  Nothing is blocked, fused or reordered beyond what the
definitions below state.

Sources (transformers model documentation pages):

* "DeepSeek-V3.2" page, section "DeepSeek Sparse Attention (DSA)":
  - the Lightning Indexer computes an index score between each query and
    all previous keys with a light, few-head module; the port computes it
    directly in bf16/fp32 (the FP8 + Hadamard form of the original code is
    only a precision optimisation because the rotation is orthogonal);
  - fine-grained token selection keeps the ``index_topk`` most relevant
    tokens per query (2048 by default) and the main MLA attention is then
    computed only over those tokens *through an additive mask*;
  - the indexer keeps its own single-head key cache of ``index_head_dim``
    per token next to the K/V cache;
  - each layer runs its own indexer (no sharing of the selection).
* "DeepSeek-V3.2" page, ``DeepseekV32Config`` parameters: ``index_topk``
  (2048), ``index_head_dim`` (128), ``index_n_heads`` (64),
  ``kv_lora_rank`` (512), ``qk_rope_head_dim`` (64), ``qk_nope_head_dim``
  (128), ``num_attention_heads`` (128).
* "DeepSeek-V4" page, section on the attention-mask layout: an indexer slot
  with no selection is marked by a ``-1`` pointer.

The exact indexer formula is not printed on the pages.  The reading used
here is  I[t,s] = sum_j w[t,j] * ReLU(q_I[t,j,:] . k_I[s,:])  for s <= t,
with no extra scale; every other open point is listed with its reading in
the repository's design notes.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "index_scores_row",
    "index_scores",
    "e4m3_round",
    "hadamard",
    "fp8_quantize_rows",
    "index_scores_fp8_row",
    "fp8_rotate_quantize",
    "index_scores_fp8_codes",
    "topk_select",
    "additive_mask_row",
    "masked_attention_row",
    "dsa_prefill",
    "dsa_decode",
    "masked_attention_row_backward",
    "sparse_attention_backward",
    "index_scores_row_backward",
    "index_scores_backward",
]

_NEG_INF = -np.inf


def _f64(x):
    """Widen an fp32 / bf16 / fp64 array (numpy or torch) to float64 exactly."""
    try:  # torch tensors (bf16 has no numpy dtype): go through float32
        import torch  # noqa: WPS433

        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


# --------------------------------------------------------------------------
# Step 1: Lightning Indexer scores
# --------------------------------------------------------------------------
def index_scores_row(q_idx_t, w_t, k_idx_prefix):
    """Index scores of one query against every key at or before it.

    DeepSeek-V3.2 page, "DeepSeek Sparse Attention (DSA)", Lightning Indexer
    paragraph: a score between the query and all previous keys, computed by
    ``index_n_heads`` light heads of width ``index_head_dim`` against a
    single-head key cache.  Reading:  I[s] = sum_j w[j] * max(0, q[j,:].k[s,:]).

    q_idx_t:      [H_I, D_I]   indexer query heads of this token
    w_t:          [H_I]        per-head weights of this token
    k_idx_prefix: [n, D_I]     indexer keys of positions 0..n-1 (n = t+1)
    returns       [n] float64
    """
    q = _f64(q_idx_t)
    w = _f64(w_t)
    k = _f64(k_idx_prefix)
    dots = q @ k.T                      # [H_I, n]: q_I[t,j] . k_I[s]
    return w @ np.maximum(dots, 0.0)    # sum over heads of w_j * ReLU(dot)


def index_scores(q_idx, w, k_idx):
    """Full causal score matrix of one sequence.

    q_idx [L, H_I, D_I], w [L, H_I], k_idx [L, D_I]  ->  I [L, L] float64,
    with -inf where s > t (keys after the query are not "previous keys").
    """
    q = _f64(q_idx)
    L = q.shape[0]
    out = np.full((L, L), _NEG_INF)
    for t in range(L):
        out[t, : t + 1] = index_scores_row(q[t], _f64(w[t]), _f64(k_idx[: t + 1]))
    return out


# --------------------------------------------------------------------------
# Step 1, FP8 form (not yet on the GPU path)
# --------------------------------------------------------------------------
E4M3_MAX = 448.0


def e4m3_round(x):
    """Nearest FP8 E4M3 value, ties to even, saturating at +-448.

    E4M3 (the "fn" variant: 1 sign, 4 exponent bits with bias 7, 3 mantissa
    bits, no infinities): normal values m * 2^(e-3) with m in [8, 16) and
    e in [-6, 8] (largest finite value 1.75 * 2^8 = 448); subnormal values
    m * 2^-9 with m in [0, 8).  So in every binade the spacing is 2^(e-3),
    and below 2^-6 it is 2^-9.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    e = np.floor(np.log2(np.where(a > 0.0, a, 1.0)))
    e = np.clip(e, -6.0, 8.0)               # below 2^-6: the subnormal spacing 2^-9
    quantum = np.exp2(e - 3.0)
    v = np.round(a / quantum) * quantum     # numpy rounds halves to even
    return np.copysign(np.minimum(v, E4M3_MAX), x)


def hadamard(n):
    """n x n Hadamard matrix (n a power of two) by Sylvester's construction:
    H_1 = [1], H_2m = [[H_m, H_m], [H_m, -H_m]].  Entries are +-1 and
    H @ H.T = n * I, so H / sqrt(n) is orthogonal (and symmetric)."""
    if n < 1 or n & (n - 1):
        raise ValueError("n must be a power of two")
    h = np.ones((1, 1))
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h


def fp8_quantize_rows(x):
    """Each row of x quantised to E4M3 with its own scale amax / 448:
    returns (q8, scale) with x ~= q8 * scale[:, None] (q8 on the E4M3 grid).
    An all-zero row gets scale 1."""
    x = _f64(x)
    amax = np.abs(x).max(axis=1)
    scale = np.where(amax > 0.0, amax / E4M3_MAX, 1.0)
    return e4m3_round(x / scale[:, None]), scale


def index_scores_fp8_row(q_idx_t, w_t, k_idx_prefix):
    """Index scores of one query in the indexer's FP8 form.

    DeepSeek-V3.2 page, "DeepSeek Sparse Attention (DSA)", Lightning Indexer
    paragraph: the reference implementation runs the indexer in FP8 after a
    Hadamard transform (rotate_activation); the transform is orthogonal, so
    Hq . Hk = q . k, and FP8 is a precision optimisation.  The pages give no
    quantisation details; the reading here:
      1. rotate every indexer query head and every key by the normalised
         Hadamard matrix H / sqrt(index_head_dim);
      2. quantise each rotated vector (one query head, one key) to E4M3 with
         its own scale amax / 448;
      3. I[s] = sum_j w[j] * ReLU(s_q[j] * s_k[s] * (q8[j] . k8[s])).

    Shapes and result as index_scores_row.
    """
    q8, sq = fp8_rotate_quantize(q_idx_t)
    k8, sk = fp8_rotate_quantize(k_idx_prefix)
    return index_scores_fp8_codes(q8, sq, w_t, k8, sk)


def fp8_rotate_quantize(x):
    """Steps 1 and 2 of the FP8 form for a set of vectors (rows of x): the
    rotation by H / sqrt(d), then E4M3 codes with one scale amax / 448 per
    rotated row.  Returns (codes as E4M3 values, scales)."""
    x = _f64(x)
    d = x.shape[-1]
    rot = hadamard(d) / np.sqrt(d)
    return fp8_quantize_rows(x @ rot.T)


def index_scores_fp8_codes(q8, sq, w_t, k8, sk):
    """Step 3 of the FP8 form, from given codes and scales:
    I[s] = sum_j w[j] * ReLU(s_q[j] * s_k[s] * (q8[j] . k8[s]))."""
    q8, sq, w, k8, sk = (_f64(a) for a in (q8, sq, w_t, k8, sk))
    dots = (q8 @ k8.T) * sq[:, None] * sk[None, :]
    return w @ np.maximum(dots, 0.0)


# --------------------------------------------------------------------------
# Step 2: per-query top-k selection
# --------------------------------------------------------------------------
def topk_select(scores, k):
    """Indices of the ``k`` most relevant tokens of one query.

    DeepSeek-V3.2 page, "DeepSeek Sparse Attention (DSA)", fine-grained token
    selection paragraph: keep the ``index_topk`` most relevant tokens.  When
    fewer than ``k`` candidates exist every candidate is kept.  Ties are
    broken toward the lower position (order = score descending, then
    position ascending); -0.0 and +0.0 are the same score.  The kept
    positions are returned in ascending order, padded with -1 (the
    DeepSeek-V4 page's marker for an empty indexer slot) to length ``k``.

    scores: [n] scores of candidate positions 0..n-1 (n = t+1)
    returns int64 [k]
    """
    s = _f64(scores)
    n = s.shape[0]
    keep = min(k, n)
    # A stable sort on the negated score puts larger scores first and keeps
    # equal scores in ascending position order.
    order = np.argsort(-s, kind="stable")[:keep]
    out = np.full(k, -1, dtype=np.int64)
    out[:keep] = np.sort(order)
    return out


# --------------------------------------------------------------------------
# Steps 3-4: additive mask and MLA attention (absorbed latent form)
# --------------------------------------------------------------------------
def additive_mask_row(selected, L):
    """Row of the additive mask: 0 at selected positions, -inf elsewhere.

    DeepSeek-V3.2 page, "DeepSeek Sparse Attention (DSA)": the main MLA
    attention is computed only over the selected tokens via an additive
    mask.  Positions after the query are never selected, so the causal
    mask is contained in this one.
    """
    m = np.full(L, _NEG_INF)
    sel = np.asarray(selected)
    sel = sel[sel >= 0]
    m[sel] = 0.0
    return m


def masked_attention_row(q_t, kv, mask_row, scale, d_v):
    """Dense softmax attention of one query over all L keys plus the mask.

    Absorbed MLA form: each of the H heads has a query of width D_qk
    (kv_lora_rank latent + qk_rope_head_dim rope part, 512 + 64 at the
    DeepSeek-V3.2 configuration); all heads share one key row of width D_qk
    and the value is the first d_v (= kv_lora_rank) columns of that row.

    z[h,s] = scale * q[h,:].kv[s,:] + mask[s];  p = softmax_s(z);
    O[h,:] = sum_s p[h,s] kv[s,:d_v];  lse[h] = log sum_s exp(z[h,s]).

    q_t [H, D_qk], kv [L, D_qk], mask_row [L]  ->  (O [H, d_v], lse [H])
    """
    q = _f64(q_t)
    k = _f64(kv)
    z = scale * (q @ k.T) + mask_row[None, :]          # [H, L]
    zmax = np.max(z, axis=1, keepdims=True)
    e = np.exp(z - zmax)                               # exp(-inf) = 0
    denom = np.sum(e, axis=1, keepdims=True)
    p = e / denom
    out = p @ k[:, :d_v]
    lse = (zmax + np.log(denom))[:, 0]
    return out, lse


# --------------------------------------------------------------------------
# The whole forward step
# --------------------------------------------------------------------------
def _one_query(q_idx_t, w_t, k_idx_seq, q_t, kv_seq, t, topk, scale, d_v):
    """Steps 1-4 for the query at sequence position t (0-based)."""
    scores = index_scores_row(q_idx_t, w_t, k_idx_seq[: t + 1])
    sel = topk_select(scores, topk)
    L = kv_seq.shape[0]
    mask = additive_mask_row(sel, L)
    out, lse = masked_attention_row(q_t, kv_seq, mask, scale, d_v)
    return scores, sel, out, lse


def dsa_prefill(q_idx, w, k_idx, q, kv, cu_seqlens, topk, scale, d_v, rows=None):
    """DSA forward over a packed batch of causal sequences.

    Packed ("varlen") layout: sequence b owns rows cu_seqlens[b] ..
    cu_seqlens[b+1]-1 of every input; positions are sequence-local and
    every sequence is causal on its own.

    q_idx [T, H_I, D_I], w [T, H_I], k_idx [T, D_I], q [T, H, D_qk],
    kv [T, D_qk], cu_seqlens [B+1].

    rows: optional iterable of global row numbers to evaluate (the oracle
    is O(L) per row; long inputs are checked on a sample).  Default: all.

    Returns a dict with, for the evaluated rows (in the order given):
      rows   [R] int64 global rows
      pos    [R] int64 sequence-local positions
      scores list of [pos+1] float64 arrays (index scores of the row)
      idx    [R, topk] int64 selected positions (ascending, -1 padded)
      out    [R, H, d_v] float64
      lse    [R, H] float64
    """
    cu = [int(c) for c in np.asarray(cu_seqlens).reshape(-1)]
    T = cu[-1]
    if rows is None:
        rows = range(T)
    rows = [int(r) for r in rows]
    seq_of = np.searchsorted(np.asarray(cu), np.asarray(rows, dtype=np.int64), side="right") - 1
    H = q.shape[1]
    res_pos, res_scores, res_idx = [], [], []
    res_out = np.zeros((len(rows), H, d_v))
    res_lse = np.zeros((len(rows), H))
    cache = {}
    for i, (r, b) in enumerate(zip(rows, seq_of)):
        b = int(b)
        lo, hi = cu[b], cu[b + 1]
        if b not in cache:  # widen each sequence's shared tensors once
            cache = {b: (_f64(k_idx[lo:hi]), _f64(kv[lo:hi]))}
        k_seq, kv_seq = cache[b]
        t = r - lo
        sc, sel, o, l = _one_query(_f64(q_idx[r]), _f64(w[r]), k_seq, _f64(q[r]), kv_seq, t, topk, scale, d_v)
        res_pos.append(t)
        res_scores.append(sc)
        res_idx.append(sel)
        res_out[i] = o
        res_lse[i] = l
    return {
        "rows": np.asarray(rows, dtype=np.int64),
        "pos": np.asarray(res_pos, dtype=np.int64),
        "scores": res_scores,
        "idx": np.asarray(res_idx, dtype=np.int64).reshape(len(rows), topk),
        "out": res_out,
        "lse": res_lse,
    }


def dsa_decode(q_idx, w, q, idx_cache, kv_cache, cache_seqlens, topk, scale, d_v, batches=None):
    """DSA forward for one new query per sequence over its caches.

    DeepSeek-V3.2 page, "DeepSeek Sparse Attention (DSA)": the indexer keeps
    its own single-head key cache (``index_head_dim`` per token) beside the
    main K/V cache and is updated before it is read.  Reading: the caches
    already hold the new token, so ``cache_seqlens[b]`` counts it and the
    query sits at position cache_seqlens[b]-1; every cached position is a
    candidate.

    q_idx [B, H_I, D_I], w [B, H_I], q [B, H, D_qk],
    idx_cache [B, max_ctx, D_I], kv_cache [B, max_ctx, D_qk], cache_seqlens [B].
    Returns dict(batches, scores (list), idx [R, topk], out [R,H,d_v], lse [R,H]).
    """
    lens = [int(n) for n in np.asarray(cache_seqlens).reshape(-1)]
    if batches is None:
        batches = range(len(lens))
    batches = [int(b) for b in batches]
    H = q.shape[1]
    res_scores, res_idx = [], []
    res_out = np.zeros((len(batches), H, d_v))
    res_lse = np.zeros((len(batches), H))
    for i, b in enumerate(batches):
        n = lens[b]
        k_seq = _f64(idx_cache[b, :n])
        kv_seq = _f64(kv_cache[b, :n])
        sc, sel, o, l = _one_query(_f64(q_idx[b]), _f64(w[b]), k_seq, _f64(q[b]), kv_seq, n - 1, topk, scale, d_v)
        res_scores.append(sc)
        res_idx.append(sel)
        res_out[i] = o
        res_lse[i] = l
    return {
        "batches": np.asarray(batches, dtype=np.int64),
        "scores": res_scores,
        "idx": np.asarray(res_idx, dtype=np.int64).reshape(len(batches), topk),
        "out": res_out,
        "lse": res_lse,
    }


# ---------------------------------------------------------------------------
# Upstream of the path: the indexer's inputs and its key-cache update
# ---------------------------------------------------------------------------
def linear(x, weight):
    """y = x . weight^T for x [..., K] and weight [N, K] (a bias-free projection, the form of
    every projection the "DeepSeek-V3.2" page names for the indexer); float64."""
    return _f64(x) @ _f64(weight).T


def indexer_inputs(q_latent, x, wq_b, wk, w_proj, n_heads, head_dim):
    """The Lightning Indexer's inputs ("DeepSeek-V3.2" page, section "DeepSeek Sparse Attention
    (DSA)"): the indexer scores queries taken from the MLA query latent
    q_latent = q_a_layernorm(q_a_proj(x)) through its projection wq_b (sized by q_lora_rank);
    its head weights come from the weights_proj module; its single-head key of index_head_dim
    per token comes from a key projection of the hidden state x.  The page gives no further
    detail, so each is read as a plain bias-free linear map:

        q_I[t] = reshape(wq_b . q_latent[t], [n_heads, head_dim])
        k_I[t] = wk . x[t]
        w[t]   = w_proj . x[t]

    q_latent [T, q_lora_rank], x [T, hidden], wq_b [n_heads * head_dim, q_lora_rank],
    wk [head_dim, hidden], w_proj [n_heads, hidden] -> (q_I [T, n_heads, head_dim],
    k_I [T, head_dim], w [T, n_heads]), float64."""
    T = _f64(q_latent).shape[0]
    q_i = linear(q_latent, wq_b).reshape(T, n_heads, head_dim)
    return q_i, linear(x, wk), linear(x, w_proj)


def update_indexer(idx_cache, kv_cache, cache_seqlens, k_new, kv_new):
    """The decode step's cache update ("DeepSeek-V3.2" page, DSA section: the indexer keeps its
    own per-token key cache next to the K/V cache and updates it through update_indexer()).
    For every sequence b with room left, the new token's indexer key k_new[b] and latent row
    kv_new[b] are written at position cache_seqlens[b] of idx_cache[b] and kv_cache[b], and
    the length grows by one; a full cache is left as it is.  Returns new arrays
    (idx_cache, kv_cache, cache_seqlens, full) with `full` marking the sequences that had no
    room; the values are copied, not converted."""
    idx = np.array(idx_cache, copy=True)
    kv = np.array(kv_cache, copy=True)
    lens = np.array(cache_seqlens, copy=True)
    full = np.zeros(len(lens), dtype=bool)
    for b in range(len(lens)):
        p = int(lens[b])
        if p >= idx.shape[1]:
            full[b] = True
            continue
        idx[b, p] = k_new[b]
        kv[b, p] = kv_new[b]
        lens[b] = p + 1
    return idx, kv, lens, full


def paged_to_dense(pool, block_table, page_size):
    """A paged cache as the dense cache it stands for: the pool [num_pages * page_size, d] holds
    pages of page_size positions, and position s of sequence b sits in page
    block_table[b, s // page_size] at offset s % page_size ("DeepSeek-V3.2" page: the cache
    layers are dynamic or static; a block table is the plainest form of a dynamic one).
    Returns [B, max_pages * page_size, d]; positions of table entries < 0 are zero."""
    pool = np.asarray(pool)
    table = np.asarray(block_table)
    B, P = table.shape
    out = np.zeros((B, P * page_size) + pool.shape[1:], dtype=pool.dtype)
    for b in range(B):
        for j in range(P):
            pg = int(table[b, j])
            if pg >= 0:
                out[b, j * page_size:(j + 1) * page_size] = pool[pg * page_size:(pg + 1) * page_size]
    return out


# ---------------------------------------------------------------------------
# Backward of the path with the selection held fixed
# ---------------------------------------------------------------------------
# The "DeepSeek-V3.2" page calls DSA a trainable sparse attention.  The selection
# (top-k of the index scores) is piecewise constant in the scores, so no gradient
# flows through it; what is differentiable is the attention over the selected set
# (step 4, for fixed idx) and the index scores themselves (step 1), at the
# positions a loss reads them.  The pages give no training loss, so the gradients
# of the outputs arrive as inputs.
def masked_attention_row_backward(q_t, kv, mask_row, scale, d_v, dout, dlse=None):
    """Gradient of ``masked_attention_row`` with respect to q_t and kv.

    With the mask fixed the row is plain softmax attention.  For output gradients
    dO [H, d_v] and (optionally) dlse [H]:

        dP[h,s]  = dO[h,:] . kv[s,:d_v]
        D[h]     = dO[h,:] . O[h,:]            (= sum_s p[h,s] dP[h,s])
        dz[h,s]  = p[h,s] * (dP[h,s] - D[h] + dlse[h])
        dq[h,:]  = scale * sum_s dz[h,s] kv[s,:]
        dkv[s,:] = scale * sum_h dz[h,s] q[h,:],  plus sum_h p[h,s] dO[h,:] on the first d_v columns

    (softmax Jacobian dp_s/dz_u = p_s (1[s=u] - p_u); d lse / d z_s = p_s).  Masked
    positions have p = 0 and receive no gradient.

    q_t [H, D_qk], kv [L, D_qk], mask_row [L], dout [H, d_v], dlse [H] or None
    returns (dq [H, D_qk], dkv [L, D_qk]) float64
    """
    q = _f64(q_t)
    k = _f64(kv)
    g = _f64(dout)
    z = scale * (q @ k.T) + mask_row[None, :]
    zmax = np.max(z, axis=1, keepdims=True)
    e = np.exp(z - zmax)
    p = e / np.sum(e, axis=1, keepdims=True)       # [H, L]
    v = k[:, :d_v]
    out = p @ v                                    # [H, d_v]
    dp = g @ v.T                                   # [H, L]
    dd = np.sum(g * out, axis=1)                   # [H]
    dz = dp - dd[:, None]
    if dlse is not None:
        dz = dz + _f64(dlse)[:, None]
    dz = p * dz
    dq = scale * (dz @ k)
    dkv = scale * (dz.T @ q)
    dkv[:, :d_v] += p.T @ g
    return dq, dkv


def sparse_attention_backward(q, kv, idx, cu_seqlens, scale, d_v, dout, dlse=None, rows=None):
    """Backward of step 4 over a packed batch, for the selection ``idx`` held fixed.

    q [T, H, D_qk], kv [T, D_qk], idx [T, k] sequence-local positions (-1 = empty),
    cu_seqlens [B+1], dout [T, H, d_v], dlse [T, H] or None.

    rows: the rows whose output gradients are taken (default: all); the gradients
    of the other rows' outputs count as zero, so they add nothing to dkv.

    Returns a dict with
      rows [R] int64, dq [R, H, D_qk] float64 (the listed rows' query gradients),
      dkv [T, D_qk] float64 (every row of every sequence, summed over the queries
      that selected it).
    """
    cu = [int(c) for c in np.asarray(cu_seqlens).reshape(-1)]
    T = cu[-1]
    if rows is None:
        rows = range(T)
    rows = [int(r) for r in rows]
    seq_of = np.searchsorted(np.asarray(cu), np.asarray(rows, dtype=np.int64), side="right") - 1
    H, dqk = q.shape[1], q.shape[2]
    idx = np.asarray(idx)
    dq = np.zeros((len(rows), H, dqk))
    dkv = np.zeros((T, dqk))
    cache = {}
    for i, (r, b) in enumerate(zip(rows, seq_of)):
        b = int(b)
        lo, hi = cu[b], cu[b + 1]
        if b not in cache:
            cache = {b: _f64(kv[lo:hi])}
        kv_seq = cache[b]
        mask = additive_mask_row(idx[r], hi - lo)
        dl = None if dlse is None else _f64(dlse[r])
        g_q, g_kv = masked_attention_row_backward(_f64(q[r]), kv_seq, mask, scale, d_v, _f64(dout[r]), dl)
        dq[i] = g_q
        dkv[lo:hi] += g_kv
    return {"rows": np.asarray(rows, dtype=np.int64), "dq": dq, "dkv": dkv}


def index_scores_row_backward(q_idx_t, w_t, k_idx_prefix, positions, d_scores):
    """Gradient of ``index_scores_row`` read at the listed positions.

    For  I[s] = sum_j w[j] * max(0, S[j,s]),  S[j,s] = q[j,:].k[s,:],  and a loss with
    gradient g[m] on I[positions[m]]:

        dw[j]   = sum_m g[m] * max(0, S[j,s_m])
        G[j,m]  = g[m] * w[j] * [S[j,s_m] > 0]
        dq[j,:] = sum_m G[j,m] k[s_m,:]
        dk[s,:] = sum_{m: s_m = s} sum_j G[j,m] q[j,:]

    The ReLU's derivative at exactly 0 is read as 0 (max(0, x) grows only for x > 0).
    Entries with positions[m] < 0 are empty and contribute nothing.

    q_idx_t [H_I, D_I], w_t [H_I], k_idx_prefix [n, D_I], positions [m], d_scores [m]
    returns (dq [H_I, D_I], dw [H_I], dk [n, D_I]) float64
    """
    q = _f64(q_idx_t)
    w = _f64(w_t)
    k = _f64(k_idx_prefix)
    pos = np.asarray(positions, dtype=np.int64).reshape(-1)
    g = _f64(d_scores).reshape(-1)
    keep = pos >= 0
    pos, g = pos[keep], g[keep]
    ks = k[pos]                                    # [m, D_I]
    s = q @ ks.T                                   # [H_I, m]
    dw = np.maximum(s, 0.0) @ g
    G = (s > 0.0) * w[:, None] * g[None, :]
    dq = G @ ks
    dk = np.zeros_like(k)
    np.add.at(dk, pos, G.T @ q)
    return dq, dw, dk


def index_scores_backward(q_idx, w, k_idx, idx, d_scores, cu_seqlens, rows=None):
    """Backward of step 1 over a packed batch, the scores read at ``idx``.

    q_idx [T, H_I, D_I], w [T, H_I], k_idx [T, D_I], idx [T, k] sequence-local
    positions (-1 = empty), d_scores [T, k] the gradient at each listed position,
    cu_seqlens [B+1].  rows: rows whose scores carry a gradient (default: all).

    Returns a dict with rows [R], dq [R, H_I, D_I], dw [R, H_I] and dk [T, D_I]
    (summed over every query that reads the key), float64.
    """
    cu = [int(c) for c in np.asarray(cu_seqlens).reshape(-1)]
    T = cu[-1]
    if rows is None:
        rows = range(T)
    rows = [int(r) for r in rows]
    seq_of = np.searchsorted(np.asarray(cu), np.asarray(rows, dtype=np.int64), side="right") - 1
    HI, DI = q_idx.shape[1], q_idx.shape[2]
    idx = np.asarray(idx)
    dq = np.zeros((len(rows), HI, DI))
    dw = np.zeros((len(rows), HI))
    dk = np.zeros((T, DI))
    cache = {}
    for i, (r, b) in enumerate(zip(rows, seq_of)):
        b = int(b)
        lo, hi = cu[b], cu[b + 1]
        if b not in cache:
            cache = {b: _f64(k_idx[lo:hi])}
        t = r - lo
        g_q, g_w, g_k = index_scores_row_backward(_f64(q_idx[r]), _f64(w[r]), cache[b][: t + 1], idx[r],
                                                  _f64(d_scores[r]))
        dq[i] = g_q
        dw[i] = g_w
        dk[lo:lo + t + 1] += g_k
    return {"rows": np.asarray(rows, dtype=np.int64), "dq": dq, "dw": dw, "dk": dk}
