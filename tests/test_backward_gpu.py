"""GPU parity of the backward calls against the fp64 oracle (through the C ABI).

The selection is a seeded synthetic input (random subsets of each causal prefix,
the shape the top-k step produces), fed to both sides.  The attention backward
reads the forward's out and lse: the composite tests take them from the library's
own forward, the isolated tests from the oracle (rounded to the input dtype), so
the second kind checks the backward kernel alone.  Tolerances are per-element
bounds derived from the arithmetic (tests/_helpers.py); the integer-valued
indexer case is exact.
"""
import numpy as np
import pytest
import torch

import oracle.dsa_oracle as O
from sparse_attention_long_gemm_b300 import _binding as B
from sparse_attention_long_gemm_b300.build import build_library
from sparse_attention_long_gemm_b300.synth import (CONFIGS, make_backward_inputs, make_prefill_inputs,
                                                   random_selection, scaled)

from _helpers import (DZ_REL_BF16, O_REL_BF16_FORWARD, O_REL_BF16_ROUNDED, O_REL_FP32_FORWARD, attn_bwd_bounds,
                      f64, index_bwd_bounds)

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


def _cu_list(cu):
    return [int(c) for c in cu.cpu()]


def _oracle_forward(q, kv, idx, cu, scale, d_v):
    """out, lse of the oracle for the given selection (every row)."""
    cul = _cu_list(cu)
    T, H = q.shape[0], q.shape[1]
    out = np.zeros((T, H, d_v))
    lse = np.zeros((T, H))
    qn, kvn, ix = f64(q.float().cpu()), f64(kv.float().cpu()), idx.cpu().numpy()
    for b in range(len(cul) - 1):
        lo, hi = cul[b], cul[b + 1]
        for r in range(lo, hi):
            out[r], lse[r] = O.masked_attention_row(qn[r], kvn[lo:hi], O.additive_mask_row(ix[r], hi - lo), scale,
                                                    d_v)
    return out, lse


def _attn_case(cfg, seed, qmul=1.0, rows=None, oracle_out=False, o_rel=None, dz_rel=0.0):
    inp = make_prefill_inputs(cfg, DEV, seed=seed)
    q, kv, cu = inp["q"], inp["kv"], inp["cu_seqlens"]
    if qmul != 1.0:   # larger logits: peaked softmax rows
        q = (q.float() * qmul).to(q.dtype)
    T, L = q.shape[0], inp["max_seqlen"]
    idx = random_selection(inp["lengths"], cfg.topk, seed).to(DEV)
    bw = make_backward_inputs(cfg, T, DEV, seed)
    dout, dlse = bw["dout"], bw["dlse"]
    if rows is not None:   # gradients only on the sampled rows
        keep = torch.zeros(T, dtype=torch.bool, device=DEV)
        keep[torch.tensor(rows, device=DEV)] = True
        dout = dout * keep[:, None, None].to(dout.dtype)
        dlse = dlse * keep[:, None].float()
    p = B.params_from_config(cfg)
    if oracle_out:
        o64, l64 = _oracle_forward(q, kv, idx, cu, cfg.softmax_scale, cfg.d_v)
        out = torch.tensor(o64, dtype=torch.float32).to(q.dtype).to(DEV)
        lse = torch.tensor(l64, dtype=torch.float32, device=DEV)
    else:
        out = torch.empty((T, cfg.n_heads, cfg.d_v), dtype=q.dtype, device=DEV)
        lse = torch.empty((T, cfg.n_heads), dtype=torch.float32, device=DEV)
        B.dsa_sparse_mla_attn(p, q, kv, idx, cu, len(inp["lengths"]), T, L, out, lse)
    dq = torch.full((T, cfg.n_heads, cfg.d_qk), float("nan"), dtype=torch.float32, device=DEV)
    dkv = torch.full((T, cfg.d_qk), float("nan"), dtype=torch.float32, device=DEV)
    B.dsa_sparse_mla_attn_bwd(p, q, kv, idx, cu, len(inp["lengths"]), T, L, out, lse, dout, dlse, dq, dkv)
    torch.cuda.synchronize()
    assert B.dsa_get_device_error() == B.DSA_OK

    # exact fp32 copies (bf16 widens to fp32 without change; the oracle widens them to fp64)
    qc, kvc, gc, dlc, ix = q.float().cpu(), kv.float().cpu(), dout.float().cpu(), dlse.cpu(), idx.cpu().numpy()
    ref = O.sparse_attention_backward(qc, kvc, ix, _cu_list(cu), cfg.softmax_scale, cfg.d_v, gc, dlc, rows=rows)
    # bounds, row by row (only rows with gradients add to dkv)
    cul = _cu_list(cu)
    seq_of = np.searchsorted(np.asarray(cul), np.asarray(ref["rows"]), side="right") - 1
    kvn = f64(kvc)
    bkv = np.zeros((T, cfg.d_qk))
    dq_g = dq[torch.tensor(ref["rows"], device=DEV)].cpu().double().numpy()
    for i, r in enumerate(ref["rows"]):
        lo = cul[seq_of[i]]
        sel = ix[r][ix[r] >= 0]
        bq, bk = attn_bwd_bounds(f64(qc[r]), kvn[lo + sel], cfg.softmax_scale, cfg.d_v, f64(gc[r]), f64(dlc[r]),
                                 o_rel, dz_rel)
        err = np.abs(dq_g[i] - ref["dq"][i])
        bad = np.argwhere(err > bq + 1e-30)
        assert bad.size == 0, f"row {r}: dq off at {bad[:4].tolist()}: err {err[tuple(bad[0])]:.3e} > " \
                              f"bound {bq[tuple(bad[0])]:.3e}"
        np.add.at(bkv, lo + sel, bk)
    err = np.abs(dkv.cpu().double().numpy() - ref["dkv"])
    bad = np.argwhere(err > bkv + 1e-30)
    assert bad.size == 0, f"dkv off at {bad[:4].tolist()}: err {err[tuple(bad[0])]:.3e} > bound " \
                          f"{bkv[tuple(bad[0])]:.3e}"
    return dq, dkv, ref


def test_attn_bwd_tiny_fp32():
    """fp32, 8 heads of 80/64, k = 64, two sequences: several selection blocks, a ragged tail
    (CUDA-core kernel)."""
    cfg = scaled(CONFIGS["tiny"], seqlens=(100, 157))
    _attn_case(cfg, seed=1, o_rel=O_REL_FP32_FORWARD)


def test_attn_bwd_bf16_general_shape():
    """bf16 with 48 heads (not the tensor-core shape): the CUDA-core kernel in bf16, a head group
    of 16 heads beyond the first 32, k = 64 over two sequences; out and lse from the general
    forward (fp32 arithmetic, bf16 output)."""
    cfg = scaled(CONFIGS["v32"], seqlens=(90, 131), topk=64, n_heads=48)
    _attn_case(cfg, seed=6, o_rel=O_REL_BF16_ROUNDED + O_REL_FP32_FORWARD)


@pytest.mark.parametrize("qmul", [1.0, 12.0])
def test_attn_bwd_v32_shape_after_tensor_core_forward(qmul):
    """DeepSeek-V3.2 dims (128 heads, 576/512, bf16: the tensor-core backward), k = 96 over two
    sequences; out and lse from the tensor-core forward; qmul = 12 makes the softmax rows peaked."""
    cfg = scaled(CONFIGS["v32"], seqlens=(150, 229), topk=96)
    _attn_case(cfg, seed=2, qmul=qmul, o_rel=O_REL_BF16_FORWARD, dz_rel=DZ_REL_BF16)


def test_attn_bwd_isolated_dense_causal():
    """k >= L (every causal position, long -1 tails, skipped blocks); out and lse from the
    oracle rounded to bf16, so only the backward kernel's arithmetic is measured."""
    cfg = scaled(CONFIGS["v32"], seqlens=(1, 70, 257), topk=2048)
    _attn_case(cfg, seed=3, oracle_out=True, o_rel=O_REL_BF16_ROUNDED, dz_rel=DZ_REL_BF16)


def test_attn_bwd_full_size_sampled():
    """The 4096-token DeepSeek-V3.2 workload (k = 2048), gradients on sampled rows only: the
    oracle then gives dkv exactly for the whole sequence, and every other row's dq is zero."""
    cfg = CONFIGS["v32"]
    L, k = 4096, cfg.topk
    rows = sorted({0, k - 2, k - 1, k, L - 1, 517, 3001})
    dq, dkv, ref = _attn_case(cfg, seed=4, rows=rows, o_rel=O_REL_BF16_FORWARD, dz_rel=DZ_REL_BF16)
    others = torch.ones(L, dtype=torch.bool, device=DEV)
    others[torch.tensor(rows, device=DEV)] = False
    assert torch.count_nonzero(dq[others]).item() == 0


def test_attn_bwd_bad_position_is_reported_not_faulted():
    cfg = scaled(CONFIGS["tiny"], seqlens=(40,))
    inp = make_prefill_inputs(cfg, DEV, seed=5)
    T = 40
    idx = random_selection([T], cfg.topk, 5).to(DEV)
    idx[10, 3] = 25           # position after the query (t = 10)
    idx[20, 0] = -7
    bw = make_backward_inputs(cfg, T, DEV, 5)
    p = B.params_from_config(cfg)
    out = torch.empty((T, cfg.n_heads, cfg.d_v), dtype=torch.float32, device=DEV)
    lse = torch.empty((T, cfg.n_heads), dtype=torch.float32, device=DEV)
    B.dsa_sparse_mla_attn(p, inp["q"], inp["kv"], idx, inp["cu_seqlens"], 1, T, T, out, lse)
    assert B.dsa_get_device_error() == B.DSA_ERR_DEVICE_DATA
    dq = torch.empty((T, cfg.n_heads, cfg.d_qk), dtype=torch.float32, device=DEV)
    dkv = torch.empty((T, cfg.d_qk), dtype=torch.float32, device=DEV)
    B.dsa_sparse_mla_attn_bwd(p, inp["q"], inp["kv"], idx, inp["cu_seqlens"], 1, T, T, out, lse, bw["dout"],
                              bw["dlse"], dq, dkv)
    assert B.dsa_get_device_error() == B.DSA_ERR_DEVICE_DATA
    assert torch.isfinite(dq).all() and torch.isfinite(dkv).all()


def test_bwd_empty_batch_does_nothing():
    cfg = CONFIGS["tiny"]
    p = B.params_from_config(cfg)
    cu = torch.zeros(2, dtype=torch.int32, device=DEV)
    t = torch.empty(16, dtype=torch.float32, device=DEV)
    B.dsa_sparse_mla_attn_bwd(p, t, t, t, cu, 1, 0, 1, t, t, t, None, t, t)
    B.dsa_index_scores_bwd(p, t, t, t, t, t, cu, 1, 0, 1, t, t, t)
    assert B.dsa_get_device_error() == B.DSA_OK


# ---------------------------------------------------------------------------
# index-score backward
# ---------------------------------------------------------------------------
def _index_case(cfg, q_idx, w, k_idx, idx, d_scores, cu, lengths, exact=False):
    p = B.params_from_config(cfg)
    T = q_idx.shape[0]
    dq = torch.full((T, cfg.n_idx_heads, cfg.idx_dim), float("nan"), dtype=torch.float32, device=DEV)
    dw = torch.full((T, cfg.n_idx_heads), float("nan"), dtype=torch.float32, device=DEV)
    dk = torch.full((T, cfg.idx_dim), float("nan"), dtype=torch.float32, device=DEV)
    B.dsa_index_scores_bwd(p, q_idx, w, k_idx, idx, d_scores, cu, len(lengths), T, max(lengths), dq, dw, dk)
    torch.cuda.synchronize()
    assert B.dsa_get_device_error() == B.DSA_OK
    ref = O.index_scores_backward(q_idx.cpu(), w.cpu(), k_idx.cpu(), idx.cpu().numpy(), d_scores.cpu(), _cu_list(cu))
    dq_g, dw_g, dk_g = (x.cpu().double().numpy() for x in (dq, dw, dk))
    if exact:
        assert np.array_equal(dq_g, ref["dq"]) and np.array_equal(dw_g, ref["dw"]) and np.array_equal(dk_g, ref["dk"])
        return
    cul = _cu_list(cu)
    # the V3.2 indexer shape in bf16 takes the tensor-core kernel, which rounds G = g w to bf16
    g_rel = DZ_REL_BF16 if (cfg.dtype == "bf16" and cfg.n_idx_heads == 64 and cfg.idx_dim == 128) else 0.0
    qn, wn, kn, gn, ix = f64(q_idx), f64(w), f64(k_idx), f64(d_scores), idx.cpu().numpy()
    bdk = np.zeros_like(ref["dk"])
    for b in range(len(cul) - 1):
        lo, hi = cul[b], cul[b + 1]
        for r in range(lo, hi):
            keep = ix[r] >= 0
            sel = ix[r][keep]
            bq, bw, bk = index_bwd_bounds(qn[r], wn[r], kn[lo + sel], gn[r][keep], g_rel)
            assert np.all(np.abs(dq_g[r] - ref["dq"][r]) <= bq + 1e-30), f"dq_idx row {r}"
            assert np.all(np.abs(dw_g[r] - ref["dw"][r]) <= bw + 1e-30), f"dw row {r}"
            np.add.at(bdk, lo + sel, bk)
    err = np.abs(dk_g - ref["dk"])
    bad = np.argwhere(err > bdk + 1e-30)
    assert bad.size == 0, f"dk_idx off at {bad[:4].tolist()}"


def test_index_bwd_integer_valued_inputs_are_exact():
    """Small dyadic integers: every product and sum is exact in fp32 (and G = g w exact in bf16),
    so the ReLU decisions and all gradients must equal the oracle's bit for bit (64 heads of 128,
    bf16: the tensor-core kernel; k = 96)."""
    cfg = scaled(CONFIGS["v32"], seqlens=(150, 211), topk=96)
    lengths = [150, 211]
    T = sum(lengths)
    g = torch.Generator().manual_seed(21)
    q_idx = (torch.randint(-3, 4, (T, 64, 128), generator=g).float() * 0.25).to(torch.bfloat16)
    k_idx = (torch.randint(-3, 4, (T, 128), generator=g).float() * 0.25).to(torch.bfloat16)
    w = torch.randint(-4, 5, (T, 64), generator=g).float() * 0.125
    d_scores = torch.randint(-4, 5, (T, 96), generator=g).float() * 0.0625
    idx = random_selection(lengths, 96, 21)
    cu = torch.tensor([0, 150, T], dtype=torch.int32)
    _index_case(cfg, q_idx.to(DEV), w.to(DEV), k_idx.to(DEV), idx.to(DEV), d_scores.to(DEV), cu.to(DEV), lengths,
                exact=True)


@pytest.mark.parametrize("name,lengths,topk", [("v32", (300, 77), 64), ("tiny", (256,), 64),
                                               ("v32", (190,), 2048)])
def test_index_bwd_random_inputs(name, lengths, topk):
    """Seeded workload inputs; (v32, k = 2048 > L) lists every causal position (the gradient of
    whole score rows)."""
    cfg = scaled(CONFIGS[name], seqlens=lengths, topk=topk)
    inp = make_prefill_inputs(cfg, DEV, seed=8)
    idx = random_selection(inp["lengths"], topk, 8).to(DEV)
    d_scores = make_backward_inputs(cfg, sum(lengths), DEV, 8)["d_scores"]
    _index_case(cfg, inp["q_idx"], inp["w"], inp["k_idx"], idx, d_scores, inp["cu_seqlens"], inp["lengths"])
