"""Parity of the CUDA library against the CPU oracle (element by element).

Every case runs through the C ABI (the ctypes binding) on cuda:0 and is
compared with oracle/ on the same seeded inputs.  Sizes span several tiles
(128-key indexer tiles, 32-key attention blocks) and ragged tails.
"""
import math

import numpy as np
import pytest
import torch

import oracle.dsa_oracle as O
import sparse_attention_long_gemm_b300 as dsa
from sparse_attention_long_gemm_b300 import _binding as B
from sparse_attention_long_gemm_b300.build import build_library
from sparse_attention_long_gemm_b300.synth import CONFIGS, make_decode_inputs, make_prefill_inputs, scaled

from _helpers import (FP32_ATTN_MAX_ABS, FP32_SCORE_REL, LSE_ABS, SCORE_REL, check_attention, check_scores,
                      check_selection, f64, score_denominator)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    build_library()
    B.lib()
    yield
    assert B.dsa_get_device_error() == B.DSA_OK


def _to(inp, dev=DEV):
    return {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


V32_SMALL = scaled(CONFIGS["v32"], seqlens=(300, 1, 129, 520), topk=128)
TINY = CONFIGS["tiny"]


# ---------------------------------------------------------------------------
# top-k: bit-exact on the same score array
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("k", [1, 7, 64, 2048])
def test_topk_bit_exact_on_same_scores(k):
    rng = np.random.default_rng(k)
    lens = [1, 5, 64, 65, 1000, 2049, 4099, 9001]
    T = sum(lens)
    ld = (max(lens) + 3) // 4 * 4
    sc = rng.standard_normal((T, ld)).astype(np.float32)
    # many exact ties, including -0.0 against +0.0
    sc[:, ::3] = np.round(sc[:, ::3] * 2) / 2
    zeros = rng.random((T, ld)) < 0.05
    sc[zeros] = np.where(rng.random(zeros.sum()) < 0.5, 0.0, -0.0).astype(np.float32)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    p = B.make_params(64, 128, 128, 576, 512, k, 0.07, "bf16")
    idx = dsa.topk(p, torch.from_numpy(sc).to(DEV), torch.from_numpy(cu).to(DEV), max(lens)).cpu().numpy()
    for b in range(len(lens)):
        for r in range(cu[b], cu[b + 1]):
            t = r - cu[b]
            ref = O.topk_select(sc[r, : t + 1], k)
            assert np.array_equal(idx[r], ref), (b, t)


def test_topk_all_equal_row_keeps_lowest_positions():
    L, k = 5000, 2048
    sc = np.full((L, L + (-L) % 4), 1.5, dtype=np.float32)
    cu = torch.tensor([0, L], dtype=torch.int32, device=DEV)
    p = B.make_params(64, 128, 128, 576, 512, k, 0.07, "bf16")
    idx = dsa.topk(p, torch.from_numpy(sc).to(DEV), cu, L).cpu().numpy()
    assert np.array_equal(idx[L - 1], np.arange(k))
    assert np.array_equal(idx[10], np.concatenate([np.arange(11), -np.ones(k - 11)]))


@pytest.mark.parametrize("n_eq", [3096, 3097])
def test_topk_candidate_list_boundary(n_eq):
    """The k-th largest key sits in a crowded top-bits bin: 1000 keys above it and n_eq equal keys
    in it give 4096 (listed, for the full row of 9000) or 4097 (refined over all keys)
    candidates; the equal keys, spread between lower scores, must be kept lowest position first
    either way."""
    k, L = 2048, 9000
    rng = np.random.default_rng(n_eq)
    row = np.full(L, 0.5, dtype=np.float32)
    pos = rng.permutation(L)
    top, eq = np.sort(pos[:1000]), np.sort(pos[1000:1000 + n_eq])
    row[top] = (100.0 + rng.random(1000)).astype(np.float32)
    row[eq] = 2.0
    sc = np.tile(row, (L, 1))
    cu = torch.tensor([0, L], dtype=torch.int32, device=DEV)
    p = B.make_params(64, 128, 128, 576, 512, k, 0.07, "bf16")
    idx = dsa.topk(p, torch.from_numpy(sc).to(DEV), cu, L).cpu().numpy()
    want = np.sort(np.concatenate([top, eq[: k - 1000]]))
    assert np.array_equal(idx[L - 1], want)
    for t in (2047, 2048, 5000, 8998):
        assert np.array_equal(idx[t], O.topk_select(sc[t, : t + 1], k)), t


def _topk_rows_decode(rows, k):
    """Top-k of each score row through the decode-form entry point (row b holds len(rows[b]) keys)."""
    n = [len(r) for r in rows]
    ld = (max(n) + 3) // 4 * 4
    sc = np.full((len(rows), ld), np.nan, dtype=np.float32)
    for b, r in enumerate(rows):
        sc[b, : len(r)] = r
    p = B.make_params(64, 128, 128, 576, 512, k, 0.07, "bf16")
    idx = torch.empty((len(rows), k), dtype=torch.int32, device=DEV)
    lens = torch.tensor(n, dtype=torch.int32, device=DEV)
    B.dsa_topk_decode(p, torch.from_numpy(sc).to(DEV), ld, lens, len(rows), max(n), idx)
    torch.cuda.synchronize()
    assert B.dsa_get_device_error() == B.DSA_OK
    return idx.cpu().numpy()


@pytest.mark.parametrize("k", [7, 2048])
def test_topk_bit_exact_rows_beyond_shared_memory(k):
    """Rows longer than the shared-memory capacity of the per-row kernel (51,200 keys), the decode
    caches' case, with exact ties, signed zeros and an all-equal row, next to short rows of the
    same call: bit-exact against the oracle on the same array."""
    rng = np.random.default_rng(100 + k)

    def noisy(n):
        r = rng.standard_normal(n).astype(np.float32)
        r[::3] = np.round(r[::3] * 2) / 2                       # exact ties
        z = rng.random(n) < 0.05
        r[z] = np.where(rng.random(z.sum()) < 0.5, 0.0, -0.0)   # -0.0 against +0.0
        return r

    crowded = np.full(65536, 0.25, dtype=np.float32)            # the k-th key in a tie of 6000
    hot = rng.choice(65536, size=k // 2, replace=False)
    crowded[hot] = 3.0
    crowded[rng.choice(65536, size=6000, replace=False)] = 1.0
    crowded[hot] = 3.0
    rows = [noisy(51201), noisy(65536), noisy(70000), np.full(65536, -1.25, dtype=np.float32), crowded,
            noisy(5), noisy(k), noisy(k + 1), noisy(3000)]
    idx = _topk_rows_decode(rows, k)
    for b, r in enumerate(rows):
        assert np.array_equal(idx[b], O.topk_select(r, k)), (b, len(r))


# ---------------------------------------------------------------------------
# indexer scores
# ---------------------------------------------------------------------------
def _check_index_scores(cfg, rel):
    inp = make_prefill_inputs(cfg, "cpu", seed=3)
    g = _to(inp)
    p = B.params_from_config(cfg)
    scores = dsa.index_scores(p, g["q_idx"], g["w"], g["k_idx"], g["cu_seqlens"], inp["max_seqlen"]).cpu().numpy()
    cu = inp["cu_seqlens"].numpy()
    for b in range(len(cu) - 1):
        lo, hi = cu[b], cu[b + 1]
        for r in range(lo, hi):
            t = r - lo
            ref = O.index_scores_row(inp["q_idx"][r], inp["w"][r], inp["k_idx"][lo: r + 1])
            den = score_denominator(inp["q_idx"][r], inp["w"][r], inp["k_idx"][lo: r + 1], full=(cfg.dtype == "fp32"))
            check_scores(scores[r, : t + 1], ref, den, rel)
            assert np.all(np.isnan(scores[r, t + 1:])), "entries s > t must stay untouched"
    return p


def test_index_scores_tensor_core_path():
    p = _check_index_scores(V32_SMALL, SCORE_REL)
    assert B.dsa_path_name(p) == "tcgen05"


def test_index_scores_decode_tensor_core_path():
    """The decode form of the tensor-core indexer (one query of 64 heads per sequence against its
    cache), element by element; entries past the cache length stay untouched."""
    cfg = scaled(CONFIGS["decode"], batch=5, ctx_range=(1, 3000), max_ctx=3000, topk=2048)
    inp = make_decode_inputs(cfg, "cpu", seed=8)
    lens = inp["lengths"]
    lens[1] = 1
    lens[2] = 128
    lens[3] = 129
    inp["cache_seqlens"] = torch.tensor(lens, dtype=torch.int32)
    g = _to(inp)
    p = B.params_from_config(cfg)
    assert B.dsa_path_name(p) == "tcgen05"
    scores = dsa.index_scores_decode(p, g["q_idx"], g["w"], g["idx_cache"], g["cache_seqlens"]).cpu().numpy()
    for b in range(cfg.batch):
        n = lens[b]
        kc = inp["idx_cache"][b, :n]
        ref = O.index_scores_row(inp["q_idx"][b], inp["w"][b], kc)
        check_scores(scores[b, :n], ref, score_denominator(inp["q_idx"][b], inp["w"][b], kc), SCORE_REL)
        assert np.all(np.isnan(scores[b, n:])), "entries past the cache length must stay untouched"


def test_tensor_core_path_beyond_256_sequences():
    """Batches longer than one indexer launch's sequence table (256) stay on the tensor cores:
    300 packed sequences (prefill) and 300 caches (decode), scores element by element."""
    rng = np.random.default_rng(9)
    lens = tuple(int(x) for x in rng.integers(1, 24, size=300))
    cfg = scaled(CONFIGS["v32"], seqlens=lens, topk=16)
    p = _check_index_scores(cfg, SCORE_REL)
    assert B.dsa_path_name(p) == "tcgen05"
    dcfg = scaled(CONFIGS["decode"], batch=300, ctx_range=(1, 300), max_ctx=300, topk=16)
    inp = make_decode_inputs(dcfg, "cpu", seed=10)
    g = _to(inp)
    scores = dsa.index_scores_decode(p, g["q_idx"], g["w"], g["idx_cache"], g["cache_seqlens"]).cpu().numpy()
    for b in range(dcfg.batch):
        n = inp["lengths"][b]
        kc = inp["idx_cache"][b, :n]
        ref = O.index_scores_row(inp["q_idx"][b], inp["w"][b], kc)
        check_scores(scores[b, :n], ref, score_denominator(inp["q_idx"][b], inp["w"][b], kc), SCORE_REL)
    # the fused forward over the same long batch, on a sample of rows
    _check_forward(cfg, 2e-2, 2e-3, rows=list(range(0, sum(lens), 53)) + [sum(lens) - 1])


def test_index_scores_general_path_fp32():
    p = _check_index_scores(TINY, FP32_SCORE_REL)
    assert B.dsa_path_name(p) == "simt"


def test_index_scores_general_path_bf16_odd_shape():
    cfg = scaled(TINY, n_idx_heads=5, idx_dim=24, dtype="bf16", seqlens=(70, 33))
    _check_index_scores(cfg, SCORE_REL)


# ---------------------------------------------------------------------------
# sparse attention over given selections
# ---------------------------------------------------------------------------
def _random_selection(rng, cu, k):
    T = cu[-1]
    idx = np.full((T, k), -1, dtype=np.int32)
    for b in range(len(cu) - 1):
        for r in range(cu[b], cu[b + 1]):
            n = r - cu[b] + 1
            m = min(k, n)
            idx[r, :m] = np.sort(rng.choice(n, size=m, replace=False))
    return idx


def _check_attention(cfg, max_abs, mean_abs, seed=5):
    inp = make_prefill_inputs(cfg, "cpu", seed=seed)
    g = _to(inp)
    p = B.params_from_config(cfg)
    cu = inp["cu_seqlens"].numpy()
    rng = np.random.default_rng(seed)
    idx = _random_selection(rng, cu, cfg.topk)
    out, lse = dsa.sparse_mla_attn(p, g["q"], g["kv"], torch.from_numpy(idx).to(DEV), g["cu_seqlens"],
                                   inp["max_seqlen"])
    out, lse = out.float().cpu().numpy(), lse.cpu().numpy()
    ref_out = np.zeros_like(out, dtype=np.float64)
    ref_lse = np.zeros_like(lse, dtype=np.float64)
    for b in range(len(cu) - 1):
        lo, hi = cu[b], cu[b + 1]
        kv_seq = f64(inp["kv"][lo:hi])
        for r in range(lo, hi):
            mask = O.additive_mask_row(idx[r], hi - lo)
            ref_out[r], ref_lse[r] = O.masked_attention_row(inp["q"][r], kv_seq, mask, cfg.softmax_scale, cfg.d_v)
    check_attention(out, ref_out, max_abs, mean_abs)
    assert np.abs(lse - ref_lse).max() <= LSE_ABS
    return p


def test_attention_tensor_core_path():
    cfg = scaled(V32_SMALL, topk=96)      # 3 blocks of 32, ragged below
    p = _check_attention(cfg, 2e-2, 2e-3)
    assert B.dsa_path_name(p) == "tcgen05"


def test_attention_tensor_core_path_k2048():
    cfg = scaled(CONFIGS["v32"], seqlens=(2100, 37), topk=2048)
    _check_attention(cfg, 2e-2, 2e-3, seed=6)


def test_attention_general_path_fp32():
    _check_attention(TINY, FP32_ATTN_MAX_ABS, FP32_ATTN_MAX_ABS)


# ---------------------------------------------------------------------------
# fused forward, end to end
# ---------------------------------------------------------------------------
def _check_forward(cfg, max_abs, mean_abs, rows=None, seed=0):
    inp = make_prefill_inputs(cfg, "cpu", seed=seed)
    g = _to(inp)
    p = B.params_from_config(cfg)
    out, lse, idx = dsa.prefill(p, g["q_idx"], g["w"], g["k_idx"], g["q"], g["kv"], g["cu_seqlens"],
                                inp["max_seqlen"], want_idx=True)
    torch.cuda.synchronize()
    out, lse, idx = out.float().cpu().numpy(), lse.cpu().numpy(), idx.cpu().numpy()
    ref = O.dsa_prefill(inp["q_idx"], inp["w"], inp["k_idx"], inp["q"], inp["kv"], inp["cu_seqlens"],
                        cfg.topk, cfg.softmax_scale, cfg.d_v, rows=rows)
    cu = inp["cu_seqlens"].numpy()
    ndiff = 0
    ref_out = ref["out"].copy()
    ref_lse = ref["lse"].copy()
    for i, r in enumerate(ref["rows"]):
        d = check_selection(idx[r], ref["scores"][i], ref["idx"][i], cfg.topk)
        if d:  # a near tie went the other way: compare attention over the GPU's own selection
            ndiff += 1
            b = int(np.searchsorted(cu, r, side="right") - 1)
            lo, hi = cu[b], cu[b + 1]
            mask = O.additive_mask_row(idx[r], hi - lo)
            ref_out[i], ref_lse[i] = O.masked_attention_row(inp["q"][r], inp["kv"][lo:hi], mask,
                                                            cfg.softmax_scale, cfg.d_v)
    check_attention(out[ref["rows"]], ref_out, max_abs, mean_abs)
    assert np.abs(lse[ref["rows"]] - ref_lse).max() <= LSE_ABS
    return ndiff


def test_forward_tiny_full():
    _check_forward(TINY, FP32_ATTN_MAX_ABS, FP32_ATTN_MAX_ABS)


def test_forward_v32_shape_small_k():
    _check_forward(V32_SMALL, 2e-2, 2e-3)


def test_forward_v32_shape_k2048_ragged():
    cfg = scaled(CONFIGS["v32"], seqlens=(2500, 300), topk=2048)
    rows = list(range(0, 2500, 97)) + [2045, 2046, 2047, 2048, 2049, 2499, 2500, 2799]
    _check_forward(cfg, 2e-2, 2e-3, rows=rows, seed=1)


def test_forward_long_offset_keys_small():
    # per-position key offsets make some keys popular: selections overlap across queries
    cfg = scaled(CONFIGS["long"], seqlens=(1500,), topk=256)
    _check_forward(cfg, 2e-2, 2e-3, rows=list(range(0, 1500, 37)) + [255, 256, 1499], seed=2)


# ---------------------------------------------------------------------------
# decode over caches
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("k", [64, 2048])
def test_decode_small(k):
    cfg = scaled(CONFIGS["decode"], batch=4, ctx_range=(1, 2600), max_ctx=2600, topk=k)
    inp = make_decode_inputs(cfg, "cpu", seed=4)
    lens = inp["lengths"]
    lens[0] = 1      # degenerate: only the new token
    inp["cache_seqlens"] = torch.tensor(lens, dtype=torch.int32)
    g = _to(inp)
    p = B.params_from_config(cfg)
    out, lse, idx = dsa.decode(p, g["q_idx"], g["w"], g["q"], g["idx_cache"], g["kv_cache"], g["cache_seqlens"],
                               want_idx=True)
    out, lse, idx = out.float().cpu().numpy(), lse.cpu().numpy(), idx.cpu().numpy()
    ref = O.dsa_decode(inp["q_idx"], inp["w"], inp["q"], inp["idx_cache"], inp["kv_cache"], lens, k,
                       cfg.softmax_scale, cfg.d_v)
    for b in range(cfg.batch):
        d = check_selection(idx[b], ref["scores"][b], ref["idx"][b], k)
        if d:
            n = lens[b]
            mask = O.additive_mask_row(idx[b], n)
            ref["out"][b], ref["lse"][b] = O.masked_attention_row(inp["q"][b], inp["kv_cache"][b, :n], mask,
                                                                  cfg.softmax_scale, cfg.d_v)
    check_attention(out, ref["out"])
    assert np.abs(lse - ref["lse"]).max() <= LSE_ABS


# ---------------------------------------------------------------------------
# device-side error reporting (no fault, no hang: bounded waits return)
# ---------------------------------------------------------------------------
def test_bounded_wait_reports_timeout():
    assert B.dsa_get_device_error() == B.DSA_OK
    B.dsa_selftest_wait_timeout(2_000_000)      # 2 ms, nothing ever arrives
    assert B.dsa_get_device_error() == B.DSA_ERR_TIMEOUT
    assert B.dsa_get_device_error() == B.DSA_OK   # the word was cleared


def test_bad_cu_seqlens_is_reported_not_faulted():
    cfg = V32_SMALL
    inp = make_prefill_inputs(cfg, "cpu", seed=1)
    g = _to(inp)
    bad = torch.tensor([0, 500, 200, 900, 950], dtype=torch.int32, device=DEV)   # decreasing, past the end
    p = B.params_from_config(cfg)
    T = g["q"].shape[0]
    dsa.prefill(p, g["q_idx"], g["w"], g["k_idx"], g["q"], g["kv"], bad, 600)
    assert B.dsa_get_device_error() == B.DSA_ERR_DEVICE_DATA
    assert T == 950
