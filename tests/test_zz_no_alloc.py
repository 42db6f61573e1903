"""The decode entry point for callers that cannot allocate device memory.

dsa_forward_decode_noalloc serves callers that have no way to get a
workspace (plug-ins without access to their host framework's allocator,
serving loops whose memory pool they do not own).  It must give the same
result as dsa_forward_decode, which takes a caller-allocated workspace, and
keep doing so on consecutive calls that reuse the library's fixed scratch
array.  This file is collected last so that a run stopping at its first
failure has already run everything else; it also passes on its own.
"""
import ctypes

import numpy as np
import pytest
import torch

import sparse_attention_long_gemm_b300 as dsa
from sparse_attention_long_gemm_b300 import _binding as B
from sparse_attention_long_gemm_b300.build import build_library
from sparse_attention_long_gemm_b300.synth import CONFIGS, make_decode_inputs, scaled

from _helpers import ATTN_MAX_ABS, ATTN_MEAN_ABS, LSE_ABS, check_attention

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    build_library()
    B.lib()


@pytest.mark.parametrize("k, want_idx", [(2048, False), (64, True)])
def test_noalloc_decode_matches_workspace_decode_twice(k, want_idx):
    cfg = scaled(CONFIGS["decode"], batch=5, ctx_range=(1, 3000), max_ctx=3000, topk=k)
    p = B.params_from_config(cfg)
    for seed in (11, 12):      # two calls in a row, different inputs
        inp = make_decode_inputs(cfg, DEV, seed=seed)
        ref_out, ref_lse, ref_idx = dsa.decode(p, inp["q_idx"], inp["w"], inp["q"], inp["idx_cache"],
                                               inp["kv_cache"], inp["cache_seqlens"], want_idx=True)
        out = torch.empty_like(ref_out)
        lse = torch.empty_like(ref_lse)
        idx = torch.empty_like(ref_idx) if want_idx else None
        B.dsa_forward_decode_noalloc(p, inp["q_idx"], inp["w"], inp["q"], inp["idx_cache"], inp["kv_cache"],
                                     inp["cache_seqlens"], cfg.batch, cfg.max_ctx, out, lse, idx)
        torch.cuda.synchronize()
        assert B.dsa_get_device_error() == B.DSA_OK
        check_attention(out.float().cpu().numpy(), ref_out.double().cpu().numpy(), ATTN_MAX_ABS, ATTN_MEAN_ABS)
        assert np.abs(lse.cpu().numpy() - ref_lse.cpu().numpy()).max() <= LSE_ABS
        if want_idx:
            assert torch.equal(idx, ref_idx)


def test_noalloc_rejects_problems_beyond_its_scratch():
    cfg = CONFIGS["decode"]
    p = B.params_from_config(cfg)
    f = ctypes.c_void_p(0x10000)           # never dereferenced: rejected on the host
    L = B.lib()
    too_many_scores = B.DSA_NOALLOC_MAX_SCORES // 4096 + 1
    rc = L.dsa_forward_decode_noalloc(ctypes.byref(p), f, f, f, f, f, f, too_many_scores, 4096, f, None, f, None)
    assert rc == B.DSA_ERR_UNSUPPORTED
    too_many_idx = B.DSA_NOALLOC_MAX_INDICES // cfg.topk + 1   # fits the scores, not the indices
    rc = L.dsa_forward_decode_noalloc(ctypes.byref(p), f, f, f, f, f, f, too_many_idx, 8, f, None, None, None)
    assert rc == B.DSA_ERR_UNSUPPORTED
