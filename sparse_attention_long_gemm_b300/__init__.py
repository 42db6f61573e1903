"""DeepSeek Sparse Attention (DSA) forward step and its backward on one B300 (sm_103a).

The compute lives in libdsa.so (CUDA kernels behind the C ABI of
include/dsa.h).  This package holds its ctypes binding (``_binding``: the C
entry points under the same names) and thin helpers that allocate outputs
and workspace with torch before calling those entry points.

The library is loaded lazily on first use; if it has not been built the
first call raises (there is no CPU fallback).
"""
from __future__ import annotations

import math

from . import _binding as C
from ._binding import (  # noqa: F401
    DSA_BF16,
    DSA_FP32,
    DSAError,
    DsaParams,
    dsa_decode_workspace_size,
    dsa_forward,
    dsa_forward_decode,
    dsa_forward_decode_paged,
    dsa_gemm_bf16,
    dsa_get_device_error,
    dsa_index_scores,
    dsa_index_scores_bwd,
    dsa_index_scores_decode,
    dsa_index_scores_fp8,
    dsa_index_scores_fp8_decode,
    dsa_indexer_inputs,
    dsa_indexer_quantize_fp8,
    dsa_path_name,
    dsa_selftest_wait_timeout,
    dsa_set_wait_timeout_ns,
    dsa_sparse_mla_attn,
    dsa_sparse_mla_attn_bwd,
    dsa_sparse_mla_attn_decode,
    dsa_topk,
    dsa_topk_decode,
    dsa_update_indexer,
    dsa_update_indexer_paged,
    dsa_workspace_size,
    make_params,
    params_from_config,
)


def indexer_inputs(p, q_latent, x, wq_b, wk, w_proj, stream=None):
    """The indexer's inputs from the query latent [T, q_lora_rank] and the hidden state
    [T, hidden] (bf16): (q_idx [T, H_I, D_I] bf16, k_idx [T, D_I] bf16, w [T, H_I] fp32)."""
    import torch

    T, R = q_latent.shape
    E = x.shape[1]
    H, D = p.n_idx_heads, p.idx_dim
    q_idx = torch.empty((T, H, D), dtype=torch.bfloat16, device=x.device)
    k_idx = torch.empty((T, D), dtype=torch.bfloat16, device=x.device)
    w = torch.empty((T, H), dtype=torch.float32, device=x.device)
    dsa_indexer_inputs(p, q_latent, x, wq_b, wk, w_proj, T, R, E, q_idx, k_idx, w, stream)
    return q_idx, k_idx, w


def _round4(x):
    return (x + 3) // 4 * 4


def index_scores(p, q_idx, w, k_idx, cu_seqlens, max_seqlen, stream=None):
    """Score rows [T, round_up(max_seqlen, 4)] (fp32; valid for s <= t only)."""
    import torch

    T = q_idx.shape[0]
    ld = _round4(max_seqlen)
    scores = torch.full((T, ld), float("nan"), dtype=torch.float32, device=q_idx.device)
    dsa_index_scores(p, q_idx, w, k_idx, cu_seqlens, cu_seqlens.numel() - 1, T, max_seqlen, scores, ld, stream)
    return scores


def topk(p, scores, cu_seqlens, max_seqlen, stream=None):
    import torch

    T, ld = scores.shape
    idx = torch.empty((T, p.topk), dtype=torch.int32, device=scores.device)
    dsa_topk(p, scores, ld, cu_seqlens, cu_seqlens.numel() - 1, T, max_seqlen, idx, stream)
    return idx


def sparse_mla_attn(p, q, kv, idx, cu_seqlens, max_seqlen, want_lse=True, stream=None):
    import torch

    T = q.shape[0]
    out = torch.empty((T, p.n_heads, p.d_v), dtype=q.dtype, device=q.device)
    lse = torch.empty((T, p.n_heads), dtype=torch.float32, device=q.device) if want_lse else None
    dsa_sparse_mla_attn(p, q, kv, idx, cu_seqlens, cu_seqlens.numel() - 1, T, max_seqlen, out, lse, stream)
    return out, lse


def sparse_mla_attn_bwd(p, q, kv, idx, cu_seqlens, max_seqlen, out, lse, dout, dlse=None, stream=None):
    """Gradients of the sparse attention for the selection idx: (dq [T, H, d_qk], dkv [T, d_qk]), fp32."""
    import torch

    T = q.shape[0]
    dq = torch.empty((T, p.n_heads, p.d_qk), dtype=torch.float32, device=q.device)
    dkv = torch.empty((T, p.d_qk), dtype=torch.float32, device=q.device)
    dsa_sparse_mla_attn_bwd(p, q, kv, idx, cu_seqlens, cu_seqlens.numel() - 1, T, max_seqlen, out, lse, dout, dlse,
                            dq, dkv, stream)
    return dq, dkv


def index_scores_bwd(p, q_idx, w, k_idx, idx, d_scores, cu_seqlens, max_seqlen, stream=None):
    """Gradients of the index scores read at idx [T, p.topk] with gradient d_scores [T, p.topk]:
    (dq_idx [T, H_I, D_I], dw [T, H_I], dk_idx [T, D_I]), fp32."""
    import torch

    T = q_idx.shape[0]
    dev = q_idx.device
    dq = torch.empty((T, p.n_idx_heads, p.idx_dim), dtype=torch.float32, device=dev)
    dw = torch.empty((T, p.n_idx_heads), dtype=torch.float32, device=dev)
    dk = torch.empty((T, p.idx_dim), dtype=torch.float32, device=dev)
    dsa_index_scores_bwd(p, q_idx, w, k_idx, idx, d_scores, cu_seqlens, cu_seqlens.numel() - 1, T, max_seqlen,
                         dq, dw, dk, stream)
    return dq, dw, dk


def prefill(p, q_idx, w, k_idx, q, kv, cu_seqlens, max_seqlen, want_lse=True, want_idx=False,
            workspace=None, stream=None):
    """Fused DSA forward over a packed batch: returns (out, lse, idx)."""
    import torch

    T = q.shape[0]
    B = cu_seqlens.numel() - 1
    dev = q.device
    out = torch.empty((T, p.n_heads, p.d_v), dtype=q.dtype, device=dev)
    lse = torch.empty((T, p.n_heads), dtype=torch.float32, device=dev) if want_lse else None
    idx = torch.empty((T, p.topk), dtype=torch.int32, device=dev) if want_idx else None
    if workspace is None:
        workspace = torch.empty(dsa_workspace_size(p, T, max_seqlen, B), dtype=torch.uint8, device=dev)
    dsa_forward(p, q_idx, w, k_idx, q, kv, cu_seqlens, B, T, max_seqlen, out, lse, idx, workspace, stream)
    return out, lse, idx


def decode(p, q_idx, w, q, idx_cache, kv_cache, cache_seqlens, want_lse=True, want_idx=False,
           workspace=None, stream=None):
    """Fused DSA forward for one new query per sequence: returns (out, lse, idx)."""
    import torch

    B, max_ctx = idx_cache.shape[0], idx_cache.shape[1]
    dev = q.device
    out = torch.empty((B, p.n_heads, p.d_v), dtype=q.dtype, device=dev)
    lse = torch.empty((B, p.n_heads), dtype=torch.float32, device=dev) if want_lse else None
    idx = torch.empty((B, p.topk), dtype=torch.int32, device=dev) if want_idx else None
    if workspace is None:
        workspace = torch.empty(dsa_decode_workspace_size(p, B, max_ctx), dtype=torch.uint8, device=dev)
    dsa_forward_decode(p, q_idx, w, q, idx_cache, kv_cache, cache_seqlens, B, max_ctx, out, lse, idx,
                       workspace, stream)
    return out, lse, idx


def index_scores_decode(p, q_idx, w, idx_cache, cache_seqlens, stream=None):
    """Decode score rows [B, round_up(max_ctx, 4)] (fp32; valid for s < cache_seqlens[b] only)."""
    import torch

    B, max_ctx = idx_cache.shape[0], idx_cache.shape[1]
    ld = _round4(max_ctx)
    scores = torch.full((B, ld), float("nan"), dtype=torch.float32, device=q_idx.device)
    dsa_index_scores_decode(p, q_idx, w, idx_cache, cache_seqlens, B, max_ctx, scores, ld, stream)
    return scores


def default_scale(qk_nope_head_dim=128, qk_rope_head_dim=64):
    return 1.0 / math.sqrt(qk_nope_head_dim + qk_rope_head_dim)
