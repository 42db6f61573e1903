"""Host-side checks of the C ABI (no GPU needed).

The library must load, export every function that include/dsa.h declares,
and reject bad arguments on the host before anything touches a device.
"""
import ctypes
import os
import re
import subprocess

import pytest

from sparse_attention_long_gemm_b300 import _binding as B
from sparse_attention_long_gemm_b300.build import build_library

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsa.h")


@pytest.fixture(scope="module")
def L():
    build_library()
    return B.lib()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dsa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_and_library_exports_everything(L):
    names = _declared()
    assert "dsa_forward" in names and "dsa_forward_decode" in names
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB_PATH], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (dsa_[a-z0-9_]+)\b", out))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    assert set(B.EXPORTED) == set(names)
    for n in names:
        assert hasattr(L, n)


V32 = dict(n_idx_heads=64, idx_dim=128, n_heads=128, d_qk=576, d_v=512, topk=2048, softmax_scale=0.07,
           dtype="bf16")
TINY = dict(n_idx_heads=4, idx_dim=32, n_heads=8, d_qk=80, d_v=64, topk=64, softmax_scale=0.1, dtype="fp32")


def test_status_strings_and_path_names(L):
    for code in range(0, -8, -1):
        assert B.status_string(code).startswith("DSA_")
    assert B.dsa_path_name(B.make_params(**V32)) == "tcgen05"
    assert B.dsa_path_name(B.make_params(**TINY)) == "simt"
    bad = B.make_params(**{**V32, "d_v": 1000})
    assert B.dsa_path_name(bad) == "invalid"


def test_workspace_sizes(L):
    p = B.make_params(**V32)
    ws = B.dsa_workspace_size(p, 4096, 4096, 1)
    assert ws == 4096 * 4096 * 4 + 4096 * 2048 * 4
    ws = B.dsa_workspace_size(p, 10, 7, 2)          # ld rounds 7 up to 8, each part to 256 B
    assert ws == 512 + 81920
    assert B.dsa_decode_workspace_size(p, 64, 65536) == 64 * 65536 * 4 + 64 * 2048 * 4
    assert B.dsa_workspace_size(p, 10, 0, 1) == 0
    assert B.dsa_decode_workspace_size(B.make_params(**{**V32, "topk": 0}), 4, 4) == 0


def _fake(n=1 << 12):
    """A 256-byte aligned host address: never dereferenced, validation fails first."""
    return ctypes.c_void_p(0x10000)


def test_host_validation_rejects_bad_arguments(L):
    p = B.make_params(**V32)
    P = ctypes.byref(p)
    f = _fake()
    null = None
    s = None
    # null params / pointers
    assert L.dsa_index_scores(None, f, f, f, f, 1, 8, 8, f, 8, s) == B.DSA_ERR_ARG
    assert L.dsa_index_scores(P, null, f, f, f, 1, 8, 8, f, 8, s) == B.DSA_ERR_ARG
    assert L.dsa_topk(P, f, 8, null, 1, 8, 8, f, s) == B.DSA_ERR_ARG
    # ld too small / not a multiple of 4
    assert L.dsa_index_scores(P, f, f, f, f, 1, 8, 16, f, 8, s) == B.DSA_ERR_SHAPE
    assert L.dsa_topk(P, f, 10, f, 1, 8, 8, f, s) == B.DSA_ERR_SHAPE
    # misaligned pointer
    assert L.dsa_sparse_mla_attn(P, ctypes.c_void_p(0x10004), f, f, f, 1, 8, 8, f, None, s) == B.DSA_ERR_ARG
    # bad dtype / unsupported shapes
    bad = B.make_params(**{**V32, "dtype": 7})
    assert L.dsa_topk(ctypes.byref(bad), f, 8, f, 1, 8, 8, f, s) == B.DSA_ERR_ARG
    big = B.make_params(**{**V32, "topk": 20000})
    assert L.dsa_topk(ctypes.byref(big), f, 8, f, 1, 8, 8, f, s) == B.DSA_ERR_UNSUPPORTED
    wide = B.make_params(**{**V32, "n_idx_heads": 129})
    assert L.dsa_index_scores(ctypes.byref(wide), f, f, f, f, 1, 8, 8, f, 8, s) == B.DSA_ERR_UNSUPPORTED
    assert L.dsa_topk(P, f, 8, f, 0, 8, 8, f, s) == B.DSA_ERR_ARG          # batch < 1
    assert L.dsa_topk(P, f, 1 << 21, f, 1, 8, (1 << 20) + 1, f, s) == B.DSA_ERR_UNSUPPORTED
    # fused calls: missing / small / misaligned workspace
    assert L.dsa_forward(P, f, f, f, f, f, f, 1, 8, 8, f, None, None, None, 0, s) == B.DSA_ERR_WORKSPACE
    assert L.dsa_forward(P, f, f, f, f, f, f, 1, 8, 8, f, None, None, f, 100, s) == B.DSA_ERR_WORKSPACE
    need = B.dsa_workspace_size(p, 8, 8, 1)
    assert L.dsa_forward(P, f, f, f, f, f, f, 1, 8, 8, f, None, None, ctypes.c_void_p(0x10010), need,
                         s) == B.DSA_ERR_WORKSPACE
    assert L.dsa_forward_decode(P, f, f, f, f, f, f, 2, 16, f, None, None, f, 10, s) == B.DSA_ERR_WORKSPACE
    assert L.dsa_forward_decode(P, f, f, f, f, f, null, 2, 16, f, None, None, f, 1 << 20, s) == B.DSA_ERR_ARG
    # empty batch is a no-op that touches nothing
    assert L.dsa_topk(P, f, 8, f, 1, 0, 8, f, s) == B.DSA_OK


def test_wait_timeout_setting_is_clamped_and_returns_previous(L):
    old = B.dsa_set_wait_timeout_ns(5000)
    assert B.dsa_set_wait_timeout_ns(1) == 5000
    assert B.dsa_set_wait_timeout_ns(old) == 1000


def test_fp8_indexer_flag_is_checked_on_the_host(L):
    p = B.make_params(**V32, indexer_fp8=True)
    assert B.dsa_path_name(p) == "tcgen05"
    f = ctypes.c_void_p(0x10000)
    # the decode calls read a bf16 indexer key cache: the FP8 flag is refused before any launch
    rc = L.dsa_forward_decode(ctypes.byref(p), f, f, f, f, f, f, 2, 64, f, None, None, f, 1 << 30, None)
    assert rc == B.DSA_ERR_UNSUPPORTED
    rc = L.dsa_forward_decode_noalloc(ctypes.byref(p), f, f, f, f, f, f, 2, 64, f, None, None, None)
    assert rc == B.DSA_ERR_UNSUPPORTED
    # the FP8 form needs the 64 x 128 bf16 indexer
    assert B.dsa_path_name(B.make_params(**TINY, indexer_fp8=True)) == "invalid"
    bad = B.make_params(**V32)
    bad.indexer_fp8 = 2
    assert B.dsa_path_name(bad) == "invalid"
    # the fused prefill's workspace grows by the quantised operands
    q = B.make_params(**V32)
    T = 100
    extra = B.dsa_workspace_size(p, T, T, 1) - B.dsa_workspace_size(q, T, T, 1)
    assert extra == T * 64 * 128 + 25600 + 12800 + 512   # q8, w*s_q, k8, s_k, each 256-aligned
    tiny = B.make_params(**TINY)
    assert L.dsa_indexer_quantize_fp8(ctypes.byref(tiny), f, 4, None, f, f, None) == B.DSA_ERR_UNSUPPORTED


def test_indexer_inputs_and_update_are_checked_on_the_host(L):
    f = ctypes.c_void_p(0x10000)          # 16-byte aligned, never dereferenced: every case fails first
    g = ctypes.c_void_p(0x10008)          # 8-byte aligned only
    ok = (f, 64, f, 64, 128, 256, 64, f, 256, B.DSA_BF16, None)
    assert L.dsa_gemm_bf16(None, *ok[1:]) == B.DSA_ERR_ARG
    assert L.dsa_gemm_bf16(*ok[:4], 0, *ok[5:]) == B.DSA_ERR_ARG                       # m < 1
    assert L.dsa_gemm_bf16(*ok[:9], 7, None) == B.DSA_ERR_ARG                          # bad c_dtype
    assert L.dsa_gemm_bf16(f, 60, *ok[2:]) == B.DSA_ERR_SHAPE                          # lda < k
    assert L.dsa_gemm_bf16(f, 68, *ok[2:]) == B.DSA_ERR_SHAPE                          # lda not a multiple of 8
    assert L.dsa_gemm_bf16(g, *ok[1:]) == B.DSA_ERR_SHAPE                              # misaligned A
    assert L.dsa_gemm_bf16(*ok[:8], 260, B.DSA_BF16, None) == B.DSA_ERR_SHAPE          # bf16 ldc % 8
    assert L.dsa_gemm_bf16(*ok[:4], 65535 * 128 + 1, *ok[5:]) == B.DSA_ERR_UNSUPPORTED
    p = B.make_params(**V32)
    tiny = B.make_params(**TINY)
    args = (f, f, f, f, f, 100, 1536, 7168, f, f, f, None)
    assert L.dsa_indexer_inputs(ctypes.byref(tiny), *args) == B.DSA_ERR_UNSUPPORTED    # fp32 params
    assert L.dsa_indexer_inputs(ctypes.byref(p), *args[:5], 100, 1530, 7168, *args[8:]) == B.DSA_ERR_SHAPE
    assert L.dsa_indexer_inputs(ctypes.byref(p), *args[:5], -1, *args[6:]) == B.DSA_ERR_ARG
    assert L.dsa_indexer_inputs(ctypes.byref(p), *args[:5], 0, *args[6:]) == B.DSA_OK     # nothing to do
    assert L.dsa_indexer_inputs(ctypes.byref(p), None, *args[1:]) == B.DSA_ERR_ARG
    assert L.dsa_update_indexer(ctypes.byref(p), f, f, 0, 64, f, f, f, None) == B.DSA_ERR_ARG
    assert L.dsa_update_indexer(ctypes.byref(p), f, None, 2, 64, f, f, f, None) == B.DSA_ERR_ARG
    assert L.dsa_update_indexer(ctypes.byref(p), g, f, 2, 64, f, f, f, None) == B.DSA_ERR_ARG


def test_backward_calls_are_checked_on_the_host(L):
    p = B.make_params(**V32)
    P = ctypes.byref(p)
    f = _fake()
    g = ctypes.c_void_p(f.value + 4)   # not 16-byte aligned
    # q, kv, idx, cu, batch, total_q, max_seqlen, out, lse, dout, dlse, dq, dkv, stream
    ok = [f, f, f, f, 1, 8, 8, f, f, f, None, f, f, None]
    assert L.dsa_sparse_mla_attn_bwd(None, *ok) == B.DSA_ERR_ARG
    assert L.dsa_sparse_mla_attn_bwd(P, *ok[:8], None, *ok[9:]) == B.DSA_ERR_ARG      # lse is required
    assert L.dsa_sparse_mla_attn_bwd(P, *ok[:11], None, *ok[12:]) == B.DSA_ERR_ARG    # dq missing
    assert L.dsa_sparse_mla_attn_bwd(P, g, *ok[1:]) == B.DSA_ERR_ARG                  # misaligned q
    assert L.dsa_sparse_mla_attn_bwd(P, *ok[:10], g, *ok[11:]) == B.DSA_ERR_ARG       # misaligned dlse
    assert L.dsa_sparse_mla_attn_bwd(P, *ok[:4], 0, *ok[5:]) == B.DSA_ERR_ARG         # batch < 1
    assert L.dsa_sparse_mla_attn_bwd(P, *ok[:5], 0, *ok[6:]) == B.DSA_OK              # nothing to do
    wide = B.make_params(**dict(V32, d_qk=648, d_v=512))
    assert L.dsa_sparse_mla_attn_bwd(ctypes.byref(wide), *ok) == B.DSA_ERR_UNSUPPORTED
    big32 = B.make_params(**dict(TINY, n_heads=128, d_qk=576, d_v=512))   # fp32 tiles beyond 227 KB
    assert L.dsa_sparse_mla_attn_bwd(ctypes.byref(big32), *ok) == B.DSA_ERR_UNSUPPORTED
    # q_idx, w, k_idx, idx, d_scores, cu, batch, total_q, max_seqlen, dq_idx, dw, dk_idx, stream
    ik = [f, f, f, f, f, f, 1, 8, 8, f, f, f, None]
    assert L.dsa_index_scores_bwd(None, *ik) == B.DSA_ERR_ARG
    assert L.dsa_index_scores_bwd(P, *ik[:4], None, *ik[5:]) == B.DSA_ERR_ARG         # d_scores missing
    assert L.dsa_index_scores_bwd(P, *ik[:2], g, *ik[3:]) == B.DSA_ERR_ARG            # misaligned k_idx
    assert L.dsa_index_scores_bwd(P, *ik[:7], 0, *ik[8:]) == B.DSA_OK                 # nothing to do
    many = B.make_params(**dict(V32, n_idx_heads=128))
    assert L.dsa_index_scores_bwd(ctypes.byref(many), *ik) == B.DSA_ERR_UNSUPPORTED
    deep = B.make_params(**dict(V32, idx_dim=256))
    assert L.dsa_index_scores_bwd(ctypes.byref(deep), *ik) == B.DSA_ERR_UNSUPPORTED
