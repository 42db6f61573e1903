"""Parity of the Lightning Indexer's FP8 form (Hadamard rotation, E4M3 codes,
one scale per vector) against the CPU oracle.

The GPU rotates in fp32 and the oracle in fp64, so an E4M3 code may round the
other way when the exact value sits within rounding distance of a midpoint
between two codes; such codes are allowed to differ by one step and nothing
else.  Scores are checked element by element against the oracle's FP8 form
evaluated on the GPU's own codes and scales (the acceptance tolerance of the
indexer, 2e-3 with the cancellation-aware denominator), and against the
oracle's FP8 form of the raw inputs.
"""
import numpy as np
import pytest
import torch

import oracle.dsa_oracle as O
import sparse_attention_long_gemm_b300 as dsa
from sparse_attention_long_gemm_b300 import _binding as B
from sparse_attention_long_gemm_b300.build import build_library
from sparse_attention_long_gemm_b300.synth import CONFIGS, make_decode_inputs, make_prefill_inputs, scaled

from _helpers import LSE_ABS, SCORE_REL, check_attention, check_scores, check_selection, f64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
D = 128


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    build_library()
    B.lib()
    yield
    assert B.dsa_get_device_error() == B.DSA_OK


def _decode_codes(c_u8):
    return c_u8.view(torch.float8_e4m3fn).float().cpu().numpy().astype(np.float64)


def _quantize(p, x, w=None):
    """GPU rotation + E4M3 codes of the rows of x [n, 128] (bf16): (codes as values, out)."""
    n = x.shape[0]
    codes = torch.empty((n, D), dtype=torch.uint8, device=DEV)
    out = torch.empty(n, dtype=torch.float32, device=DEV)
    B.dsa_indexer_quantize_fp8(p, x, n, w, codes, out)
    torch.cuda.synchronize()
    return codes, out


def _check_codes(x_bf16, codes_u8, scales):
    """Codes equal the oracle's, except single steps at rounding midpoints; scales within 1e-6."""
    ref8, ref_s = O.fp8_rotate_quantize(x_bf16)
    got8 = _decode_codes(codes_u8)
    got_s = scales.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got_s - ref_s) <= 1e-6 * ref_s), "scales differ"
    diff = np.nonzero(got8 != ref8)
    if diff[0].size:
        # the oracle's value before rounding, and the midpoint between the two codes
        x = f64(x_bf16)
        v = (x @ (O.hadamard(D) / np.sqrt(D)).T) / ref_s[:, None]
        vv, a, b = v[diff], ref8[diff], got8[diff]
        mid = (a + b) / 2
        assert np.all(np.abs(vv - mid) <= 4e-6 * np.maximum(np.abs(vv), 2.0 ** -9)), "a code is off away from a tie"
        steps = np.abs(a - b) / np.exp2(np.clip(np.floor(np.log2(np.maximum(np.abs(mid), 2.0 ** -9))), -6, 8) - 3)
        assert np.all(steps <= 1.0 + 1e-9), "a code is off by more than one step"
    return got8, diff[0].size


def test_fp8_rotate_quantize_matches_oracle():
    p = B.params_from_config(CONFIGS["v32"])
    g = torch.Generator().manual_seed(5)
    x = torch.randn(3000, D, generator=g) / np.sqrt(D)
    x[7] = 0.0                                  # all-zero vector: scale 1, codes 0
    x[8] = 0.0
    x[8, 3] = 1e-3                              # one-hot: the rotation spreads it over every element
    x[9] *= 1e4                                 # large values
    x[10, :64] = 2.0 ** -20                     # tiny values (E4M3 subnormals after scaling)
    xb = x.to(torch.bfloat16)
    codes, s = _quantize(p, xb.to(DEV))
    got8, nflip = _check_codes(xb, codes, s)
    assert np.all(got8[7] == 0) and s[7].item() == 1.0
    assert nflip <= 5
    # query heads: w * s_q in place of s_q
    w = torch.randn(3000, generator=g)
    codes2, ws = _quantize(p, xb.to(DEV), w.to(DEV))
    assert torch.equal(codes2, codes)
    assert torch.allclose(ws.cpu(), w * s.cpu(), rtol=1e-6, atol=0)


def _fp8_inputs(p, inp):
    """Rotated and quantised q_I (with w * s_q) and k_I of a prefill input."""
    T = inp["q_idx"].shape[0]
    q8, wq = _quantize(p, inp["q_idx"].reshape(T * 64, D).to(DEV), inp["w"].reshape(-1).to(DEV))
    k8, ks = _quantize(p, inp["k_idx"].to(DEV))
    return q8.reshape(T, 64, D), wq.reshape(T, 64), k8, ks


def test_fp8_index_scores_prefill_from_codes():
    cfg = scaled(CONFIGS["v32"], seqlens=(300, 1, 129, 520), topk=128)
    inp = make_prefill_inputs(cfg, "cpu", seed=3)
    p = B.params_from_config(cfg)
    q8, wq, k8, ks = _fp8_inputs(p, inp)
    T, maxL = q8.shape[0], inp["max_seqlen"]
    ld = (maxL + 3) // 4 * 4
    scores = torch.full((T, ld), float("nan"), dtype=torch.float32, device=DEV)
    cu = inp["cu_seqlens"].to(DEV)
    B.dsa_index_scores_fp8(p, q8, wq, k8, ks, cu, len(inp["lengths"]), T, maxL, scores, ld)
    torch.cuda.synchronize()
    sc = scores.cpu().numpy()
    q8v, k8v = _decode_codes(q8), _decode_codes(k8)
    wqv, ksv = f64(wq), f64(ks)
    cun = inp["cu_seqlens"].numpy()
    for b in range(len(cun) - 1):
        lo, hi = cun[b], cun[b + 1]
        for r in range(lo, hi):
            t = r - lo
            ref = O.index_scores_fp8_codes(q8v[r], np.ones(64), wqv[r], k8v[lo:r + 1], ksv[lo:r + 1])
            den = np.abs(wqv[r]) @ np.maximum(q8v[r] @ k8v[lo:r + 1].T, 0.0) * ksv[lo:r + 1]
            check_scores(sc[r, : t + 1], ref, den, SCORE_REL)
            assert np.all(np.isnan(sc[r, t + 1:])), "entries s > t must stay untouched"
            if r % 37 == 0:   # and the oracle's FP8 form of the raw inputs
                raw = O.index_scores_fp8_row(inp["q_idx"][r], inp["w"][r], inp["k_idx"][lo:r + 1])
                check_scores(sc[r, : t + 1], raw, den, SCORE_REL)


def test_fp8_index_scores_decode_over_an_fp8_cache():
    cfg = scaled(CONFIGS["decode"], batch=5, ctx_range=(1, 3000), max_ctx=3000, topk=2048)
    inp = make_decode_inputs(cfg, "cpu", seed=8)
    lens = inp["lengths"]
    lens[1] = 1
    lens[2] = 129
    p = B.params_from_config(cfg)
    Bn, M = cfg.batch, cfg.max_ctx
    q8, wq = _quantize(p, inp["q_idx"].reshape(Bn * 64, D).to(DEV), inp["w"].reshape(-1).to(DEV))
    k8, ks = _quantize(p, inp["idx_cache"].reshape(Bn * M, D).to(DEV))
    ld = M
    scores = torch.full((Bn, ld), float("nan"), dtype=torch.float32, device=DEV)
    cs = torch.tensor(lens, dtype=torch.int32, device=DEV)
    B.dsa_index_scores_fp8_decode(p, q8, wq, k8, ks, cs, Bn, M, scores, ld)
    torch.cuda.synchronize()
    sc = scores.cpu().numpy()
    q8v, k8v, wqv, ksv = _decode_codes(q8).reshape(Bn, 64, D), _decode_codes(k8).reshape(Bn, M, D), f64(wq).reshape(
        Bn, 64), f64(ks).reshape(Bn, M)
    for b in range(Bn):
        n = lens[b]
        ref = O.index_scores_fp8_codes(q8v[b], np.ones(64), wqv[b], k8v[b, :n], ksv[b, :n])
        den = np.abs(wqv[b]) @ np.maximum(q8v[b] @ k8v[b, :n].T, 0.0) * ksv[b, :n]
        check_scores(sc[b, :n], ref, den, SCORE_REL)
        assert np.all(np.isnan(sc[b, n:]))


def test_forward_with_fp8_indexer():
    """dsa_forward with the FP8 indexer: selections against the oracle's FP8 scores (near ties
    exempt), attention against the oracle on the GPU's own selection."""
    cfg = scaled(CONFIGS["v32"], seqlens=(2500, 300), topk=2048)
    inp = make_prefill_inputs(cfg, "cpu", seed=1)
    g = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    p = B.params_from_config(cfg, indexer_fp8=True)
    assert B.dsa_workspace_size(p, 2800, 2500, 2) > B.dsa_workspace_size(B.params_from_config(cfg), 2800, 2500, 2)
    out, lse, idx = dsa.prefill(p, g["q_idx"], g["w"], g["k_idx"], g["q"], g["kv"], g["cu_seqlens"],
                                inp["max_seqlen"], want_idx=True)
    torch.cuda.synchronize()
    out, lse, idx = out.float().cpu().numpy(), lse.cpu().numpy(), idx.cpu().numpy()
    rows = list(range(0, 2500, 131)) + [2047, 2048, 2049, 2499, 2500, 2799]
    cun = inp["cu_seqlens"].numpy()
    for r in rows:
        b = int(np.searchsorted(cun, r, side="right") - 1)
        lo, hi = cun[b], cun[b + 1]
        ref_sc = O.index_scores_fp8_row(inp["q_idx"][r], inp["w"][r], inp["k_idx"][lo:r + 1])
        check_selection(idx[r], ref_sc, O.topk_select(ref_sc, cfg.topk), cfg.topk)
        mask = O.additive_mask_row(idx[r], hi - lo)
        ref_o, ref_l = O.masked_attention_row(inp["q"][r], inp["kv"][lo:hi], mask, cfg.softmax_scale, cfg.d_v)
        check_attention(out[r], ref_o)
        assert np.abs(lse[r] - ref_l).max() <= LSE_ABS

