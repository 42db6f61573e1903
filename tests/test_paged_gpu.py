"""Decode over paged caches (page pools plus a block table) against the dense decode and the
CPU oracle.

The paged calls read the same values as the dense ones, only from other rows, and do the same
arithmetic, so their outputs must equal the dense decode over the caches the pages stand for
bit for bit; the oracle checks the selection and attention as for the dense decode.
"""
import numpy as np
import pytest
import torch

import oracle.dsa_oracle as O
import sparse_attention_long_gemm_b300 as dsa
from sparse_attention_long_gemm_b300 import _binding as B
from sparse_attention_long_gemm_b300.build import build_library
from sparse_attention_long_gemm_b300.synth import CONFIGS, scaled

from _helpers import LSE_ABS, check_attention, check_selection

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


def _paged_problem(cfg_name, lens, page_size, max_pages, seed):
    cfg = CONFIGS[cfg_name]
    p = B.params_from_config(cfg)
    Bn = len(lens)
    need = [(n + page_size - 1) // page_size for n in lens]
    num_pages = sum(need) + 3                      # spare pages that no sequence owns
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(num_pages, generator=g).tolist()
    table = torch.full((Bn, max_pages), -1, dtype=torch.int32)
    it = iter(perm)
    for b in range(Bn):
        for j in range(need[b]):
            table[b, j] = next(it)
    table_dev = table.clone()
    table_dev[table_dev < 0] = 0                   # entries past a sequence's pages are never read
    dt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    idx_pool = torch.randn(num_pages * page_size, cfg.idx_dim, generator=g).to(dt)
    kv_pool = (torch.randn(num_pages * page_size, cfg.d_qk, generator=g) * 0.5).to(dt)
    q_idx = torch.randn(Bn, cfg.n_idx_heads, cfg.idx_dim, generator=g).to(dt)
    w = torch.randn(Bn, cfg.n_idx_heads, generator=g)
    q = torch.randn(Bn, cfg.n_heads, cfg.d_qk, generator=g).to(dt)
    return cfg, p, num_pages, table, table_dev, idx_pool, kv_pool, q_idx, w, q


@pytest.mark.parametrize("cfg_name,lens,page_size,max_pages", [
    ("v32", [1, 127, 128, 129, 3000, 5000], 128, 40),
    ("v32", [300, 2048, 2049, 7000], 256, 28),
    ("tiny", [1, 200, 333], 128, 3),
])
def test_paged_decode_equals_dense_decode(cfg_name, lens, page_size, max_pages):
    cfg, p, num_pages, table, table_dev, idx_pool, kv_pool, q_idx, w, q = _paged_problem(
        cfg_name, lens, page_size, max_pages, seed=len(lens) * page_size)
    Bn, M = len(lens), max_pages * page_size
    lens_t = torch.tensor(lens, dtype=torch.int32)
    dense_idx = torch.from_numpy(O.paged_to_dense(idx_pool.view(torch.int16 if idx_pool.dtype == torch.bfloat16
                                                                 else torch.int32).numpy(), table.numpy(), page_size))
    dense_kv = torch.from_numpy(O.paged_to_dense(kv_pool.view(torch.int16 if kv_pool.dtype == torch.bfloat16
                                                               else torch.int32).numpy(), table.numpy(), page_size))
    dense_idx = dense_idx.view(idx_pool.dtype)
    dense_kv = dense_kv.view(kv_pool.dtype)
    g = {k: v.to(DEV) for k, v in dict(q_idx=q_idx, w=w, q=q, lens=lens_t).items()}
    ref_out, ref_lse, ref_sel = dsa.decode(p, g["q_idx"], g["w"], g["q"], dense_idx.to(DEV), dense_kv.to(DEV),
                                           g["lens"], want_idx=True)
    out = torch.empty_like(ref_out)
    lse = torch.empty_like(ref_lse)
    sel = torch.empty_like(ref_sel)
    ws = torch.empty(B.dsa_decode_workspace_size(p, Bn, M), dtype=torch.uint8, device=DEV)
    B.dsa_forward_decode_paged(p, g["q_idx"], g["w"], g["q"], idx_pool.to(DEV), kv_pool.to(DEV), num_pages,
                               page_size, table_dev.to(DEV), max_pages, g["lens"], Bn, out, lse, sel, ws, ws.numel())
    torch.cuda.synchronize()
    assert B.dsa_get_device_error() == B.DSA_OK
    assert torch.equal(sel, ref_sel) and torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
    # and against the oracle, on the dense view
    outn, lsen, seln = out.float().cpu().numpy(), lse.cpu().numpy(), sel.cpu().numpy()
    for b, n in enumerate(lens):
        if b % 2 and n > 1:
            continue
        ref_sc = O.index_scores_row(q_idx[b], w[b], dense_idx[b, :n])
        check_selection(seln[b], ref_sc, O.topk_select(ref_sc, cfg.topk), cfg.topk)
        ro, rl = O.masked_attention_row(q[b], dense_kv[b, :n], O.additive_mask_row(seln[b], n), cfg.softmax_scale,
                                        cfg.d_v)
        check_attention(outn[b], ro)
        assert np.abs(lsen[b] - rl).max() <= LSE_ABS


def test_paged_update_indexer_is_bit_exact():
    cfg, p, num_pages, table, table_dev, idx_pool, kv_pool, *_ = _paged_problem("v32", [5, 128, 255, 256], 128, 3, 7)
    Bn, M = 4, 3 * 128
    lens = torch.tensor([5, 128, 255, 256], dtype=torch.int32)
    g = torch.Generator().manual_seed(1)
    k_new = torch.randn(Bn, cfg.idx_dim, generator=g).to(torch.bfloat16)
    kv_new = torch.randn(Bn, cfg.d_qk, generator=g).to(torch.bfloat16)
    # the dense view before the append, with a fresh page for the sequence whose pages are full
    # every sequence whose next position starts a page gets one that no sequence owns
    tab = table.clone()
    spare = sorted(set(range(num_pages)) - set(table[table >= 0].tolist()))
    for b, n in enumerate(lens.tolist()):
        if n % 128 == 0:
            tab[b, n // 128] = spare.pop()
    dense_idx = O.paged_to_dense(idx_pool.view(torch.int16).numpy(), tab.numpy(), 128)
    dense_kv = O.paged_to_dense(kv_pool.view(torch.int16).numpy(), tab.numpy(), 128)
    ri, rkv, rl, full = O.update_indexer(dense_idx, dense_kv, lens.numpy(), k_new.view(torch.int16).numpy(),
                                         kv_new.view(torch.int16).numpy())
    di, dkv, dl = idx_pool.to(DEV), kv_pool.to(DEV), lens.to(DEV)
    tab_dev = tab.clone()
    tab_dev[tab_dev < 0] = 0
    B.dsa_update_indexer_paged(p, k_new.to(DEV), kv_new.to(DEV), Bn, dl, di, dkv, num_pages, 128, tab_dev.to(DEV), 3)
    torch.cuda.synchronize()
    assert B.dsa_get_device_error() == B.DSA_OK and not full.any()
    assert np.array_equal(dl.cpu().numpy(), rl)
    assert np.array_equal(O.paged_to_dense(di.cpu().view(torch.int16).numpy(), tab.numpy(), 128), ri)
    assert np.array_equal(O.paged_to_dense(dkv.cpu().view(torch.int16).numpy(), tab.numpy(), 128), rkv)


def test_bad_page_index_is_reported_not_faulted():
    cfg, p, num_pages, table, table_dev, idx_pool, kv_pool, q_idx, w, q = _paged_problem("v32", [300, 200], 128, 3, 3)
    bad = table_dev.clone()
    bad[0, 1] = num_pages + 5                      # outside the pool
    out = torch.empty((2, cfg.n_heads, cfg.d_v), dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(B.dsa_decode_workspace_size(p, 2, 384), dtype=torch.uint8, device=DEV)
    B.dsa_forward_decode_paged(p, q_idx.to(DEV), w.to(DEV), q.to(DEV), idx_pool.to(DEV), kv_pool.to(DEV), num_pages,
                               128, bad.to(DEV), 3, torch.tensor([300, 200], dtype=torch.int32, device=DEV), 2, out,
                               None, None, ws, ws.numel())
    assert B.dsa_get_device_error() == B.DSA_ERR_DEVICE_DATA


def test_paged_update_with_a_bad_page_writes_nothing():
    cfg, p, num_pages, table, table_dev, idx_pool, kv_pool, *_ = _paged_problem("v32", [128, 5], 128, 2, 11)
    bad = table_dev.clone()
    bad[0, 1] = -3                                 # sequence 0's next position has no valid page
    di, dkv = idx_pool.to(DEV), kv_pool.to(DEV)
    lens = torch.tensor([128, 5], dtype=torch.int32, device=DEV)
    g = torch.Generator().manual_seed(2)
    k_new = torch.randn(2, cfg.idx_dim, generator=g).to(torch.bfloat16).to(DEV)
    kv_new = torch.randn(2, cfg.d_qk, generator=g).to(torch.bfloat16).to(DEV)
    B.dsa_update_indexer_paged(p, k_new, kv_new, 2, lens, di, dkv, num_pages, 128, bad.to(DEV), 2)
    torch.cuda.synchronize()
    assert B.dsa_get_device_error() == B.DSA_ERR_DEVICE_DATA
    assert lens.cpu().tolist() == [128, 6]         # sequence 1 appended, sequence 0 not
    pg1 = int(table[1, 0])
    changed = (di != idx_pool.to(DEV)).any(dim=1).nonzero().flatten().tolist()
    assert changed == [pg1 * 128 + 5]              # the one row of sequence 1, nothing else
    assert torch.equal(di[pg1 * 128 + 5], k_new[1]) and torch.equal(dkv[pg1 * 128 + 5], kv_new[1])
