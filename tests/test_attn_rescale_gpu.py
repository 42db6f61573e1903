"""Attention parity on inputs that drive the online-softmax rescaling.

With the standard Gaussian inputs every logit is tiny, so the running row
maximum is set by the first 64-key block and never grows enough to make the
kernel rescale O (it rescales lazily, when the maximum grows by more than 8
in log2 units).  Here the logits of half the heads rise steadily along the
selected positions (ascending, as the top-k emits them), so those heads
rescale every few blocks, while the other heads' logits fall and never
rescale.  The heads are shuffled, so one warp holds heads of both kinds.
Each rescale decision is taken by the CTA of the pair that owns the head's
softmax and sent, with P, to the other CTA; both halves of O must agree
with the fp64 additive-mask oracle.

A negative softmax scale takes the kernel's other softmax branch (the row
maximum on the scaled scores instead of on the raw ones).
"""
import numpy as np
import pytest
import torch

import oracle.dsa_oracle as O
import sparse_attention_long_gemm_b300 as dsa
from sparse_attention_long_gemm_b300 import _binding as B
from sparse_attention_long_gemm_b300.build import build_library

from _helpers import ATTN_MAX_ABS, ATTN_MEAN_ABS, LSE_ABS, check_attention, f64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
H, DQK, DV, K = 128, 576, 512, 2048


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    build_library()
    B.lib()
    yield
    assert B.dsa_get_device_error() == B.DSA_OK


def _rising_inputs(L, seed):
    """q, kv (bf16, on the device) whose logits along key position s grow like g_h * s for head h."""
    gen = torch.Generator(device=DEV).manual_seed(seed)
    e = torch.randn(DQK, generator=gen, device=DEV)
    e /= e.norm()
    scale = 1.0 / np.sqrt(192.0)
    # the growth sits in q (large, exact in bf16), so the values kv[s, :512] and hence the
    # outputs stay below ~0.2, where bf16 output rounding is far inside the tolerance
    c = torch.linspace(0.0, 1.0, L, device=DEV)
    g = torch.linspace(-1.0, 1.0, H, device=DEV)[torch.randperm(H, generator=gen, device=DEV)]
    kv = 0.05 * torch.randn(L, DQK, generator=gen, device=DEV) + c[:, None] * e[None, :]
    q = 0.05 * torch.randn(L, H, DQK, generator=gen, device=DEV) + (60.0 / scale) * g[None, :, None] * e[None, None, :]
    return q.to(torch.bfloat16), kv.to(torch.bfloat16), scale


def _selection(L, seed):
    rng = np.random.default_rng(seed)
    idx = np.full((L, K), -1, dtype=np.int32)
    for t in range(L):
        n = t + 1
        m = min(K, n)
        idx[t, :m] = np.sort(rng.choice(n, size=m, replace=False))
    return idx


def _run_and_check(q, kv, idx, scale, rows):
    L = q.shape[0]
    p = B.make_params(64, 128, H, DQK, DV, K, scale, "bf16")
    assert B.dsa_path_name(p) == "tcgen05"
    cu = torch.tensor([0, L], dtype=torch.int32, device=DEV)
    out, lse = dsa.sparse_mla_attn(p, q, kv, torch.from_numpy(idx).to(DEV), cu, L)
    torch.cuda.synchronize()
    assert B.dsa_get_device_error() == B.DSA_OK
    out = out.float().cpu().numpy()[rows]
    lse = lse.cpu().numpy()[rows]
    kv64 = f64(kv)
    q_rows = q[rows].cpu()
    ref_out = np.zeros((len(rows), H, DV))
    ref_lse = np.zeros((len(rows), H))
    for i, r in enumerate(rows):
        mask = O.additive_mask_row(idx[r], L)
        ref_out[i], ref_lse[i] = O.masked_attention_row(q_rows[i], kv64, mask, scale, DV)
    check_attention(out, ref_out, ATTN_MAX_ABS, ATTN_MEAN_ABS)
    assert np.abs(lse - ref_lse).max() <= LSE_ABS


def test_attention_rescaling_rising_logits():
    L = 2100
    q, kv, scale = _rising_inputs(L, seed=11)
    idx = _selection(L, seed=12)
    # rows with 2048 selected keys (32 blocks) and a few shorter ones
    rows = [100, 700, 2047, 2048, 2050, 2099]
    _run_and_check(q, kv, idx, scale, rows)


def test_attention_negative_scale():
    L = 700
    gen = torch.Generator(device=DEV).manual_seed(21)
    q = (torch.randn(L, H, DQK, generator=gen, device=DEV) / np.sqrt(DQK)).to(torch.bfloat16)
    kv = (torch.randn(L, DQK, generator=gen, device=DEV) / np.sqrt(DQK)).to(torch.bfloat16)
    idx = _selection(L, seed=22)
    _run_and_check(q, kv, idx, -3.0, [0, 63, 64, 500, 699])
