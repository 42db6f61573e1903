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

import pytest
import torch

import sparse_attention_long_gemm_b300 as dsa
from sparse_attention_long_gemm_b300 import _binding as B
from sparse_attention_long_gemm_b300.build import build_library
from sparse_attention_long_gemm_b300.synth import CONFIGS, make_decode_inputs, scaled


pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    build_library()
    B.lib()


@pytest.mark.parametrize("k, want_idx, batch, max_ctx", [(2048, False, 5, 3000), (64, True, 5, 3000),
                                                         (2048, True, 2, 60000), (2048, False, 64, 60000)])
def test_noalloc_decode_matches_workspace_decode_twice(k, want_idx, batch, max_ctx):
    # The last two cases have caches of up to 60,000 positions (rows longer than the per-row
    # top-k kernel keeps in shared memory).  The last one fills 92% of the fixed score scratch
    # (64 x 60,000 of its 4 Mi floats) and, with no idx_out, all of its 128 Ki index entries.
    cfg = scaled(CONFIGS["decode"], batch=batch, ctx_range=(max_ctx // 2, max_ctx), max_ctx=max_ctx, topk=k)
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
        # the same kernels on the same inputs: the results must be identical, bit for bit
        assert torch.equal(out, ref_out)
        assert torch.equal(lse, ref_lse)
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
    # one sequence whose cache fits the scratch but exceeds the decode limit of 2^20 positions
    rc = L.dsa_forward_decode_noalloc(ctypes.byref(p), f, f, f, f, f, f, 1, (1 << 20) + 4, f, None, f, None)
    assert rc == B.DSA_ERR_UNSUPPORTED
