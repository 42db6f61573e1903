"""ctypes binding of libdsa (include/dsa.h): argument marshalling only.

Every function here passes device pointers and sizes straight to the C ABI;
all arithmetic runs in the library's CUDA kernels.  torch tensors serve only
as device memory and as the source of the current CUDA stream.  If the
library is missing, loading fails loudly: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libdsa.so")

DSA_OK = 0
DSA_ERR_ARG = -1
DSA_ERR_SHAPE = -2
DSA_ERR_UNSUPPORTED = -3
DSA_ERR_CUDA = -4
DSA_ERR_TIMEOUT = -5
DSA_ERR_WORKSPACE = -6
DSA_ERR_DEVICE_DATA = -7
DSA_BF16 = 0
DSA_FP32 = 1
DSA_NOALLOC_MAX_SCORES = 4 << 20
DSA_NOALLOC_MAX_INDICES = 128 << 10

EXPORTED = [
    "dsa_status_string",
    "dsa_workspace_size",
    "dsa_decode_workspace_size",
    "dsa_index_scores",
    "dsa_topk",
    "dsa_sparse_mla_attn",
    "dsa_forward",
    "dsa_forward_decode",
    "dsa_get_device_error",
    "dsa_set_wait_timeout_ns",
    "dsa_selftest_wait_timeout",
    "dsa_path_name",
    "dsa_forward_decode_noalloc",
    "dsa_index_scores_decode",
    "dsa_topk_decode",
    "dsa_sparse_mla_attn_decode",
    "dsa_indexer_quantize_fp8",
    "dsa_index_scores_fp8",
    "dsa_index_scores_fp8_decode",
    "dsa_gemm_bf16",
    "dsa_indexer_inputs",
    "dsa_update_indexer",
    "dsa_forward_decode_paged",
    "dsa_update_indexer_paged",
    "dsa_sparse_mla_attn_bwd",
    "dsa_index_scores_bwd",
]


class DsaParams(ctypes.Structure):
    _fields_ = [
        ("n_idx_heads", ctypes.c_int),
        ("idx_dim", ctypes.c_int),
        ("n_heads", ctypes.c_int),
        ("d_qk", ctypes.c_int),
        ("d_v", ctypes.c_int),
        ("topk", ctypes.c_int),
        ("softmax_scale", ctypes.c_float),
        ("dtype", ctypes.c_int),
        ("indexer_fp8", ctypes.c_int),
    ]


class DSAError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


_lib = None


def lib():
    """The loaded libdsa.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libdsa.so not found at {LIB_PATH}; build it with "
                "`python -m sparse_attention_long_gemm_b300.build` (there is no CPU fallback)")
        L = ctypes.CDLL(LIB_PATH)
        P = ctypes.POINTER(DsaParams)
        vp, i, ll, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong, ctypes.c_size_t
        L.dsa_status_string.restype = ctypes.c_char_p
        L.dsa_status_string.argtypes = [i]
        L.dsa_path_name.restype = ctypes.c_char_p
        L.dsa_path_name.argtypes = [P]
        L.dsa_workspace_size.restype = sz
        L.dsa_workspace_size.argtypes = [P, i, i, i]
        L.dsa_decode_workspace_size.restype = sz
        L.dsa_decode_workspace_size.argtypes = [P, i, i]
        L.dsa_index_scores.restype = i
        L.dsa_index_scores.argtypes = [P, vp, vp, vp, vp, i, i, i, vp, ll, vp]
        L.dsa_topk.restype = i
        L.dsa_topk.argtypes = [P, vp, ll, vp, i, i, i, vp, vp]
        L.dsa_sparse_mla_attn.restype = i
        L.dsa_sparse_mla_attn.argtypes = [P, vp, vp, vp, vp, i, i, i, vp, vp, vp]
        L.dsa_forward.restype = i
        L.dsa_forward.argtypes = [P, vp, vp, vp, vp, vp, vp, i, i, i, vp, vp, vp, vp, sz, vp]
        L.dsa_forward_decode.restype = i
        L.dsa_forward_decode.argtypes = [P, vp, vp, vp, vp, vp, vp, i, i, vp, vp, vp, vp, sz, vp]
        L.dsa_forward_decode_noalloc.restype = i
        L.dsa_forward_decode_noalloc.argtypes = [P, vp, vp, vp, vp, vp, vp, i, i, vp, vp, vp, vp]
        L.dsa_index_scores_decode.restype = i
        L.dsa_index_scores_decode.argtypes = [P, vp, vp, vp, vp, i, i, vp, ll, vp]
        L.dsa_topk_decode.restype = i
        L.dsa_topk_decode.argtypes = [P, vp, ll, vp, i, i, vp, vp]
        L.dsa_sparse_mla_attn_decode.restype = i
        L.dsa_sparse_mla_attn_decode.argtypes = [P, vp, vp, vp, vp, i, i, vp, vp, vp]
        L.dsa_indexer_quantize_fp8.restype = i
        L.dsa_indexer_quantize_fp8.argtypes = [P, vp, ll, vp, vp, vp, vp]
        L.dsa_index_scores_fp8.restype = i
        L.dsa_index_scores_fp8.argtypes = [P, vp, vp, vp, vp, vp, i, i, i, vp, ll, vp]
        L.dsa_index_scores_fp8_decode.restype = i
        L.dsa_index_scores_fp8_decode.argtypes = [P, vp, vp, vp, vp, vp, i, i, vp, ll, vp]
        L.dsa_gemm_bf16.restype = i
        L.dsa_gemm_bf16.argtypes = [vp, ll, vp, ll, i, i, i, vp, ll, i, vp]
        L.dsa_indexer_inputs.restype = i
        L.dsa_indexer_inputs.argtypes = [P, vp, vp, vp, vp, vp, i, i, i, vp, vp, vp, vp]
        L.dsa_forward_decode_paged.restype = i
        L.dsa_forward_decode_paged.argtypes = [P, vp, vp, vp, vp, vp, i, i, vp, i, vp, i, vp, vp, vp, vp, sz, vp]
        L.dsa_update_indexer_paged.restype = i
        L.dsa_update_indexer_paged.argtypes = [P, vp, vp, i, vp, vp, vp, i, i, vp, i, vp]
        L.dsa_update_indexer.restype = i
        L.dsa_update_indexer.argtypes = [P, vp, vp, i, i, vp, vp, vp, vp]
        L.dsa_sparse_mla_attn_bwd.restype = i
        L.dsa_sparse_mla_attn_bwd.argtypes = [P, vp, vp, vp, vp, i, i, i, vp, vp, vp, vp, vp, vp, vp]
        L.dsa_index_scores_bwd.restype = i
        L.dsa_index_scores_bwd.argtypes = [P, vp, vp, vp, vp, vp, vp, i, i, i, vp, vp, vp, vp]
        L.dsa_get_device_error.restype = i
        L.dsa_get_device_error.argtypes = [vp]
        L.dsa_set_wait_timeout_ns.restype = ll
        L.dsa_set_wait_timeout_ns.argtypes = [ll]
        L.dsa_selftest_wait_timeout.restype = i
        L.dsa_selftest_wait_timeout.argtypes = [ll, vp]
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().dsa_status_string(int(status)).decode()


def make_params(n_idx_heads, idx_dim, n_heads, d_qk, d_v, topk, softmax_scale, dtype, indexer_fp8=False) -> DsaParams:
    if isinstance(dtype, str):
        dtype = DSA_BF16 if dtype == "bf16" else DSA_FP32
    return DsaParams(n_idx_heads, idx_dim, n_heads, d_qk, d_v, topk, float(softmax_scale), dtype, int(indexer_fp8))


def params_from_config(cfg, indexer_fp8=False) -> DsaParams:
    return make_params(cfg.n_idx_heads, cfg.idx_dim, cfg.n_heads, cfg.d_qk, cfg.d_v, cfg.topk,
                       cfg.softmax_scale, cfg.dtype, indexer_fp8)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is not None:
        return ctypes.c_void_p(stream)
    import torch

    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _check(rc, where):
    if rc != DSA_OK:
        raise DSAError(rc, where)


# ---------------------------------------------------------------------------
# one function per C entry point, same names
# ---------------------------------------------------------------------------
def dsa_path_name(p: DsaParams) -> str:
    return lib().dsa_path_name(ctypes.byref(p)).decode()


def dsa_workspace_size(p: DsaParams, total_q: int, max_seqlen: int, batch: int) -> int:
    return int(lib().dsa_workspace_size(ctypes.byref(p), total_q, max_seqlen, batch))


def dsa_decode_workspace_size(p: DsaParams, batch: int, max_ctx: int) -> int:
    return int(lib().dsa_decode_workspace_size(ctypes.byref(p), batch, max_ctx))


def dsa_index_scores(p, q_idx, w, k_idx, cu_seqlens, batch, total_q, max_seqlen, scores, ld, stream=None):
    rc = lib().dsa_index_scores(ctypes.byref(p), _ptr(q_idx), _ptr(w), _ptr(k_idx), _ptr(cu_seqlens), batch,
                                total_q, max_seqlen, _ptr(scores), ld, _stream(stream))
    _check(rc, "dsa_index_scores")


def dsa_topk(p, scores, ld, cu_seqlens, batch, total_q, max_seqlen, idx, stream=None):
    rc = lib().dsa_topk(ctypes.byref(p), _ptr(scores), ld, _ptr(cu_seqlens), batch, total_q, max_seqlen,
                        _ptr(idx), _stream(stream))
    _check(rc, "dsa_topk")


def dsa_sparse_mla_attn(p, q, kv, idx, cu_seqlens, batch, total_q, max_seqlen, out, lse=None, stream=None):
    rc = lib().dsa_sparse_mla_attn(ctypes.byref(p), _ptr(q), _ptr(kv), _ptr(idx), _ptr(cu_seqlens), batch,
                                   total_q, max_seqlen, _ptr(out), _ptr(lse), _stream(stream))
    _check(rc, "dsa_sparse_mla_attn")


def dsa_forward(p, q_idx, w, k_idx, q, kv, cu_seqlens, batch, total_q, max_seqlen, out, lse, idx_out,
                workspace, stream=None):
    rc = lib().dsa_forward(ctypes.byref(p), _ptr(q_idx), _ptr(w), _ptr(k_idx), _ptr(q), _ptr(kv),
                           _ptr(cu_seqlens), batch, total_q, max_seqlen, _ptr(out), _ptr(lse), _ptr(idx_out),
                           _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "dsa_forward")


def dsa_forward_decode(p, q_idx, w, q, idx_cache, kv_cache, cache_seqlens, batch, max_ctx, out, lse, idx_out,
                       workspace, stream=None):
    rc = lib().dsa_forward_decode(ctypes.byref(p), _ptr(q_idx), _ptr(w), _ptr(q), _ptr(idx_cache),
                                  _ptr(kv_cache), _ptr(cache_seqlens), batch, max_ctx, _ptr(out), _ptr(lse),
                                  _ptr(idx_out), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                  _stream(stream))
    _check(rc, "dsa_forward_decode")


def dsa_forward_decode_noalloc(p, q_idx, w, q, idx_cache, kv_cache, cache_seqlens, batch, max_ctx, out, lse,
                               idx_out, stream=None):
    """Decode forward with the library's own fixed-size scratch (no workspace argument)."""
    rc = lib().dsa_forward_decode_noalloc(ctypes.byref(p), _ptr(q_idx), _ptr(w), _ptr(q), _ptr(idx_cache),
                                          _ptr(kv_cache), _ptr(cache_seqlens), batch, max_ctx, _ptr(out),
                                          _ptr(lse), _ptr(idx_out), _stream(stream))
    _check(rc, "dsa_forward_decode_noalloc")


def dsa_index_scores_decode(p, q_idx, w, idx_cache, cache_seqlens, batch, max_ctx, scores, ld, stream=None):
    rc = lib().dsa_index_scores_decode(ctypes.byref(p), _ptr(q_idx), _ptr(w), _ptr(idx_cache), _ptr(cache_seqlens),
                                       batch, max_ctx, _ptr(scores), ld, _stream(stream))
    _check(rc, "dsa_index_scores_decode")


def dsa_topk_decode(p, scores, ld, cache_seqlens, batch, max_ctx, idx, stream=None):
    rc = lib().dsa_topk_decode(ctypes.byref(p), _ptr(scores), ld, _ptr(cache_seqlens), batch, max_ctx, _ptr(idx),
                               _stream(stream))
    _check(rc, "dsa_topk_decode")


def dsa_sparse_mla_attn_decode(p, q, kv_cache, idx, cache_seqlens, batch, max_ctx, out, lse=None, stream=None):
    rc = lib().dsa_sparse_mla_attn_decode(ctypes.byref(p), _ptr(q), _ptr(kv_cache), _ptr(idx), _ptr(cache_seqlens),
                                          batch, max_ctx, _ptr(out), _ptr(lse), _stream(stream))
    _check(rc, "dsa_sparse_mla_attn_decode")


def dsa_indexer_quantize_fp8(p, x, n_vec, w, codes, out, stream=None):
    rc = lib().dsa_indexer_quantize_fp8(ctypes.byref(p), _ptr(x), n_vec, _ptr(w), _ptr(codes), _ptr(out),
                                        _stream(stream))
    _check(rc, "dsa_indexer_quantize_fp8")


def dsa_index_scores_fp8(p, q8, wq, k8, ksc, cu_seqlens, batch, total_q, max_seqlen, scores, ld, stream=None):
    rc = lib().dsa_index_scores_fp8(ctypes.byref(p), _ptr(q8), _ptr(wq), _ptr(k8), _ptr(ksc), _ptr(cu_seqlens),
                                    batch, total_q, max_seqlen, _ptr(scores), ld, _stream(stream))
    _check(rc, "dsa_index_scores_fp8")


def dsa_index_scores_fp8_decode(p, q8, wq, k8_cache, ksc_cache, cache_seqlens, batch, max_ctx, scores, ld,
                                stream=None):
    rc = lib().dsa_index_scores_fp8_decode(ctypes.byref(p), _ptr(q8), _ptr(wq), _ptr(k8_cache), _ptr(ksc_cache),
                                           _ptr(cache_seqlens), batch, max_ctx, _ptr(scores), ld, _stream(stream))
    _check(rc, "dsa_index_scores_fp8_decode")


def dsa_gemm_bf16(a, lda, b, ldb, m, n, k, c, ldc, c_dtype, stream=None):
    rc = lib().dsa_gemm_bf16(_ptr(a), lda, _ptr(b), ldb, m, n, k, _ptr(c), ldc, c_dtype, _stream(stream))
    _check(rc, "dsa_gemm_bf16")


def dsa_indexer_inputs(p, q_latent, x, wq_b, wk, w_proj, total_q, q_lora_rank, hidden, q_idx, k_idx, w, stream=None):
    rc = lib().dsa_indexer_inputs(ctypes.byref(p), _ptr(q_latent), _ptr(x), _ptr(wq_b), _ptr(wk), _ptr(w_proj),
                                  total_q, q_lora_rank, hidden, _ptr(q_idx), _ptr(k_idx), _ptr(w), _stream(stream))
    _check(rc, "dsa_indexer_inputs")


def dsa_update_indexer(p, k_new, kv_new, batch, max_ctx, cache_seqlens, idx_cache, kv_cache, stream=None):
    rc = lib().dsa_update_indexer(ctypes.byref(p), _ptr(k_new), _ptr(kv_new), batch, max_ctx, _ptr(cache_seqlens),
                                  _ptr(idx_cache), _ptr(kv_cache), _stream(stream))
    _check(rc, "dsa_update_indexer")


def dsa_forward_decode_paged(p, q_idx, w, q, idx_pool, kv_pool, num_pages, page_size, block_table, max_pages,
                             cache_seqlens, batch, out, lse, idx_out, workspace, workspace_bytes, stream=None):
    rc = lib().dsa_forward_decode_paged(ctypes.byref(p), _ptr(q_idx), _ptr(w), _ptr(q), _ptr(idx_pool), _ptr(kv_pool),
                                        num_pages, page_size, _ptr(block_table), max_pages, _ptr(cache_seqlens), batch,
                                        _ptr(out), _ptr(lse), _ptr(idx_out), _ptr(workspace), workspace_bytes,
                                        _stream(stream))
    _check(rc, "dsa_forward_decode_paged")


def dsa_update_indexer_paged(p, k_new, kv_new, batch, cache_seqlens, idx_pool, kv_pool, num_pages, page_size,
                             block_table, max_pages, stream=None):
    rc = lib().dsa_update_indexer_paged(ctypes.byref(p), _ptr(k_new), _ptr(kv_new), batch, _ptr(cache_seqlens),
                                        _ptr(idx_pool), _ptr(kv_pool), num_pages, page_size, _ptr(block_table),
                                        max_pages, _stream(stream))
    _check(rc, "dsa_update_indexer_paged")


def dsa_sparse_mla_attn_bwd(p, q, kv, idx, cu_seqlens, batch, total_q, max_seqlen, out, lse, dout, dlse, dq, dkv,
                            stream=None):
    rc = lib().dsa_sparse_mla_attn_bwd(ctypes.byref(p), _ptr(q), _ptr(kv), _ptr(idx), _ptr(cu_seqlens), batch,
                                       total_q, max_seqlen, _ptr(out), _ptr(lse), _ptr(dout), _ptr(dlse), _ptr(dq),
                                       _ptr(dkv), _stream(stream))
    _check(rc, "dsa_sparse_mla_attn_bwd")


def dsa_index_scores_bwd(p, q_idx, w, k_idx, idx, d_scores, cu_seqlens, batch, total_q, max_seqlen, dq_idx, dw,
                         dk_idx, stream=None):
    rc = lib().dsa_index_scores_bwd(ctypes.byref(p), _ptr(q_idx), _ptr(w), _ptr(k_idx), _ptr(idx), _ptr(d_scores),
                                    _ptr(cu_seqlens), batch, total_q, max_seqlen, _ptr(dq_idx), _ptr(dw),
                                    _ptr(dk_idx), _stream(stream))
    _check(rc, "dsa_index_scores_bwd")


def dsa_get_device_error(stream=None) -> int:
    return int(lib().dsa_get_device_error(_stream(stream)))


def dsa_set_wait_timeout_ns(ns: int) -> int:
    return int(lib().dsa_set_wait_timeout_ns(int(ns)))


def dsa_selftest_wait_timeout(timeout_ns: int, stream=None):
    _check(lib().dsa_selftest_wait_timeout(int(timeout_ns), _stream(stream)), "dsa_selftest_wait_timeout")
