"""Parity of the indexer-input projections and of the key-cache append against the
CPU oracle.

The projections run on the tensor cores with fp32 accumulation and round to
bf16 (queries, keys) or keep fp32 (head weights).  Every element is checked
against the oracle's float64 product within one bf16 rounding of the exact
value plus the bound of K fp32 additions, K * 2^-23 * sum |a_k b_k| (the
products of bf16 operands are exact in fp32); the append is bit-exact.
"""
import numpy as np
import pytest
import torch

import oracle.dsa_oracle as O
import sparse_attention_long_gemm_b300 as dsa
from sparse_attention_long_gemm_b300 import _binding as B
from sparse_attention_long_gemm_b300.build import build_library
from sparse_attention_long_gemm_b300.synth import CONFIGS

from _helpers import LSE_ABS, check_attention, check_selection, f64

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


def _check_linear(got, a, w, bf16_out):
    """got [M, N] against a [M, K] . w[N, K]^T in float64."""
    a64, w64 = f64(a), f64(w)
    ref = a64 @ w64.T
    den = np.abs(a64) @ np.abs(w64).T
    g = got.float().cpu().numpy().astype(np.float64)
    rnd = (2.0 ** -8 if bf16_out else 2.0 ** -23) * np.abs(ref)
    err = np.abs(g - ref)
    acc = a64.shape[1] * 2.0 ** -23 * den   # K fp32 additions, each off by at most one ulp
    bad = err > rnd + acc + 1e-30
    assert not bad.any(), f"{bad.sum()} elements off, worst {err[bad].max()} at {np.argwhere(bad)[0]}"


@pytest.mark.parametrize("m,n,k,out", [(128, 256, 64, "bf16"), (300, 520, 200, "bf16"), (129, 64, 7168, "fp32"),
                                       (1, 1, 8, "fp32"), (257, 129, 1536, "bf16"), (64, 100, 72, "fp32")])
def test_gemm_matches_the_oracle(m, n, k, out):
    g = torch.Generator().manual_seed(m * 7 + n)
    a = (torch.randn(m, k, generator=g) / k ** 0.5).to(torch.bfloat16)
    w = torch.randn(n, k, generator=g).to(torch.bfloat16)
    dt = torch.bfloat16 if out == "bf16" else torch.float32
    ldc = (n + 7) // 8 * 8
    c = torch.full((m, ldc), float("nan"), dtype=dt, device=DEV)
    B.dsa_gemm_bf16(a.to(DEV), k, w.to(DEV), k, m, n, k, c, ldc, B.DSA_BF16 if out == "bf16" else B.DSA_FP32)
    torch.cuda.synchronize()
    _check_linear(c[:, :n], a, w, out == "bf16")
    assert torch.isnan(c[:, n:].float()).all(), "columns past n must stay untouched"


def test_gemm_with_leading_dimensions():
    m, n, k = 200, 96, 136
    g = torch.Generator().manual_seed(9)
    big_a = torch.randn(m, 160, generator=g).to(torch.bfloat16)
    big_w = torch.randn(n, 144, generator=g).to(torch.bfloat16)
    c = torch.zeros((m, 104), dtype=torch.float32, device=DEV)
    B.dsa_gemm_bf16(big_a.to(DEV), 160, big_w.to(DEV), 144, m, n, k, c, 104, B.DSA_FP32)
    torch.cuda.synchronize()
    _check_linear(c[:, :n], big_a[:, :k], big_w[:, :k], False)
    assert (c[:, n:] == 0).all()


def test_indexer_inputs_at_the_v32_sizes_match_the_oracle():
    """q_lora_rank 1536, hidden 7168, 64 x 128 indexer; T = 300 tokens (two 128-row tiles and
    a ragged tail)."""
    cfg = CONFIGS["v32"]
    p = B.params_from_config(cfg)
    T, R, E, H, D = 300, 1536, 7168, 64, 128
    g = torch.Generator().manual_seed(4)
    q_lat = torch.randn(T, R, generator=g).to(torch.bfloat16)
    x = torch.randn(T, E, generator=g).to(torch.bfloat16)
    wq_b = (torch.randn(H * D, R, generator=g) / R ** 0.5).to(torch.bfloat16)
    wk = (torch.randn(D, E, generator=g) / E ** 0.5).to(torch.bfloat16)
    wp = (torch.randn(H, E, generator=g) / E ** 0.5).to(torch.bfloat16)
    q_i, k_i, w = dsa.indexer_inputs(p, q_lat.to(DEV), x.to(DEV), wq_b.to(DEV), wk.to(DEV), wp.to(DEV))
    torch.cuda.synchronize()
    rq, rk, rw = O.indexer_inputs(q_lat, x, wq_b, wk, wp, H, D)
    assert q_i.shape == (T, H, D) and k_i.shape == (T, D) and w.shape == (T, H)
    _check_linear(q_i.reshape(T, H * D), q_lat, wq_b, True)
    _check_linear(k_i, x, wk, True)
    _check_linear(w, x, wp, False)
    assert np.allclose(f64(q_i.float().cpu()).reshape(T, H, D), rq, rtol=2 ** -7, atol=1e-3)


def test_indexer_inputs_feed_the_forward():
    """Projected inputs go straight into the indexer: its scores equal the oracle's scores of the
    same projected tensors."""
    cfg = CONFIGS["v32"]
    p = B.params_from_config(cfg)
    T, R, E, H, D = 200, 1536, 512, 64, 128
    g = torch.Generator().manual_seed(6)
    q_lat = torch.randn(T, R, generator=g).to(torch.bfloat16).to(DEV)
    x = torch.randn(T, E, generator=g).to(torch.bfloat16).to(DEV)
    wq_b = (torch.randn(H * D, R, generator=g) / R ** 0.5).to(torch.bfloat16).to(DEV)
    wk = (torch.randn(D, E, generator=g) / E ** 0.5).to(torch.bfloat16).to(DEV)
    wp = (torch.randn(H, E, generator=g) / E ** 0.5).to(torch.bfloat16).to(DEV)
    q_i, k_i, w = dsa.indexer_inputs(p, q_lat, x, wq_b, wk, wp)
    cu = torch.tensor([0, T], dtype=torch.int32, device=DEV)
    sc = dsa.index_scores(p, q_i, w, k_i, cu, T).cpu().numpy()
    qn, kn, wn = f64(q_i.float().cpu()), f64(k_i.float().cpu()), f64(w.cpu())
    for t in (0, 1, 127, 128, 199):
        ref = O.index_scores_row(qn[t], wn[t], kn[: t + 1])
        den = np.abs(wn[t]) @ np.maximum(qn[t] @ kn[: t + 1].T, 0.0)
        assert np.all(np.abs(sc[t, : t + 1] - ref) <= 2e-3 * den + 1e-6)


def test_update_indexer_is_bit_exact():
    Bn, M, D, DQK = 5, 40, 128, 576
    p = B.params_from_config(CONFIGS["v32"])
    g = torch.Generator().manual_seed(2)
    idx = torch.randn(Bn, M, D, generator=g).to(torch.bfloat16)
    kv = torch.randn(Bn, M, DQK, generator=g).to(torch.bfloat16)
    lens = torch.tensor([0, 1, 17, 39, 40], dtype=torch.int32)   # the last cache is full
    k_new = torch.randn(Bn, D, generator=g).to(torch.bfloat16)
    kv_new = torch.randn(Bn, DQK, generator=g).to(torch.bfloat16)
    ri, rkv, rl, full = O.update_indexer(idx.view(torch.int16).numpy(), kv.view(torch.int16).numpy(), lens.numpy(),
                                         k_new.view(torch.int16).numpy(), kv_new.view(torch.int16).numpy())
    di, dkv, dl = idx.to(DEV), kv.to(DEV), lens.to(DEV)
    B.dsa_update_indexer(p, k_new.to(DEV), kv_new.to(DEV), Bn, M, dl, di, dkv)
    torch.cuda.synchronize()
    assert B.dsa_get_device_error() == B.DSA_ERR_DEVICE_DATA     # the full cache is reported
    assert full.tolist() == [False, False, False, False, True]
    assert np.array_equal(dl.cpu().numpy(), rl)
    assert np.array_equal(di.cpu().view(torch.int16).numpy(), ri)
    assert np.array_equal(dkv.cpu().view(torch.int16).numpy(), rkv)


def test_update_then_decode_step():
    """Two appends, then a decode step over the grown caches equals the oracle's decode."""
    cfg = CONFIGS["v32"]
    p = B.params_from_config(cfg)
    Bn, M, H, D, DQK = 3, 300, 64, 128, 576
    g = torch.Generator().manual_seed(8)
    idx = torch.randn(Bn, M, D, generator=g).to(torch.bfloat16).to(DEV)
    kv = (torch.randn(Bn, M, DQK, generator=g) * 0.5).to(torch.bfloat16).to(DEV)
    lens = torch.tensor([5, 130, 298], dtype=torch.int32, device=DEV)
    for _ in range(2):
        B.dsa_update_indexer(p, torch.randn(Bn, D, generator=g).to(torch.bfloat16).to(DEV),
                             torch.randn(Bn, DQK, generator=g).to(torch.bfloat16).to(DEV), Bn, M, lens, idx, kv)
    torch.cuda.synchronize()
    assert lens.cpu().tolist() == [7, 132, 300]
    q_idx = torch.randn(Bn, H, D, generator=g).to(torch.bfloat16).to(DEV)
    w = torch.randn(Bn, H, generator=g).to(DEV)
    q = torch.randn(Bn, 128, DQK, generator=g).to(torch.bfloat16).to(DEV)
    out, lse, sel = dsa.decode(p, q_idx, w, q, idx, kv, lens, want_idx=True)
    torch.cuda.synchronize()
    out, lse, sel = out.float().cpu().numpy(), lse.cpu().numpy(), sel.cpu().numpy()
    qi, wn, qn = q_idx.cpu(), w.cpu(), q.cpu()
    ic, kc = idx.cpu(), kv.cpu()
    for b, n in enumerate([7, 132, 300]):
        # the appended tokens take part: the selection covers the grown cache
        ref_sc = O.index_scores_row(qi[b], wn[b], ic[b, :n])
        check_selection(sel[b], ref_sc, O.topk_select(ref_sc, cfg.topk), cfg.topk)
        ref_o, ref_l = O.masked_attention_row(qn[b], kc[b, :n], O.additive_mask_row(sel[b], n), cfg.softmax_scale,
                                              cfg.d_v)
        check_attention(out[b], ref_o)
        assert np.abs(lse[b] - ref_l).max() <= LSE_ABS


def test_update_indexer_fp32_caches_are_bit_exact():
    """The fp32 shape (4 x 32 indexer, 80-wide latent rows): the append copies bytes for either
    dtype."""
    cfg = CONFIGS["tiny"]
    p = B.params_from_config(cfg)
    Bn, M = 3, 17
    g = torch.Generator().manual_seed(5)
    idx = torch.randn(Bn, M, cfg.idx_dim, generator=g)
    kv = torch.randn(Bn, M, cfg.d_qk, generator=g)
    lens = torch.tensor([0, 9, 16], dtype=torch.int32)
    k_new = torch.randn(Bn, cfg.idx_dim, generator=g)
    kv_new = torch.randn(Bn, cfg.d_qk, generator=g)
    ri, rkv, rl, full = O.update_indexer(idx.view(torch.int32).numpy(), kv.view(torch.int32).numpy(), lens.numpy(),
                                         k_new.view(torch.int32).numpy(), kv_new.view(torch.int32).numpy())
    di, dkv, dl = idx.to(DEV), kv.to(DEV), lens.to(DEV)
    B.dsa_update_indexer(p, k_new.to(DEV), kv_new.to(DEV), Bn, M, dl, di, dkv)
    torch.cuda.synchronize()
    assert B.dsa_get_device_error() == B.DSA_OK and not full.any()
    assert np.array_equal(dl.cpu().numpy(), rl)
    assert np.array_equal(di.cpu().view(torch.int32).numpy(), ri)
    assert np.array_equal(dkv.cpu().view(torch.int32).numpy(), rkv)
