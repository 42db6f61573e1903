"""Seeded synthetic inputs for the DSA forward step.

This module only draws input tensors; it holds none of the method's
arithmetic, so both the CUDA library's tests/benchmark and the CPU oracle
can take their inputs from it.

Recipe (all workloads): a ``torch.Generator`` seeded with ``seed`` on the
target device draws (``Tensor.normal_``), in this order, q_I, k_I, w, q, kv
as float32 standard normals; q_I, k_I, q and kv are divided by sqrt(last dim) and w by
sqrt(H_I); bf16 workloads then round to bfloat16.  The long-prefill
workload adds one scalar per key position, drawn from N(0, std 0.5), to
every element of that position's indexer key (so that some keys score high
for most queries and the top-k sets are not trivial).  Sequence lengths
(varlen) and cache lengths (decode) come from a second generator seeded
with ``seed + 1`` on the CPU, so the lengths do not depend on the device.

Large workloads are drawn on the GPU (the CPU generator is far too slow for
billions of values); the oracle then receives host copies of exactly those
tensors.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch

__all__ = ["DSAConfig", "CONFIGS", "make_prefill_inputs", "make_decode_inputs", "scaled"]


@dataclass(frozen=True)
class DSAConfig:
    name: str
    n_idx_heads: int          # H_I  (index_n_heads)
    idx_dim: int              # D_I  (index_head_dim)
    topk: int                 # k    (index_topk)
    n_heads: int              # H    (num_attention_heads)
    d_qk: int                 # latent + rope width of query / key
    d_v: int                  # latent width (value)
    dtype: str                # "bf16" | "fp32"
    softmax_scale: float
    seqlens: tuple = ()       # prefill: lengths of the packed sequences
    decode: bool = False
    batch: int = 0            # decode: number of sequences
    ctx_range: tuple = (0, 0) # decode: cache lengths uniform in [lo, hi]
    max_ctx: int = 0          # decode: cache capacity per sequence
    varlen_range: tuple = ()  # varlen: lengths uniform in [lo, hi] (count = len(seqlens))
    key_offset_std: float = 0.0

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    @property
    def total_q(self):
        return self.batch if self.decode else int(sum(self.seqlens))


_S192 = 1.0 / math.sqrt(192.0)   # qk_nope_head_dim 128 + qk_rope_head_dim 64

CONFIGS = {
    # B=1, L=256, indexer 4 x 32, k=64, MLA 8 heads, kv latent 64 + rope 16, fp32
    "tiny": DSAConfig("tiny", 4, 32, 64, 8, 80, 64, "fp32", 1.0 / math.sqrt(80.0), seqlens=(256,)),
    # B=1, L=4096, DeepSeek-V3.2 dimensions, bf16
    "v32": DSAConfig("v32", 64, 128, 2048, 128, 576, 512, "bf16", _S192, seqlens=(4096,)),
    # B=1, L=32768, same dimensions, per-position indexer-key offset
    "long": DSAConfig("long", 64, 128, 2048, 128, 576, 512, "bf16", _S192, seqlens=(32768,),
                      key_offset_std=0.5),
    # 64 sequences, one new query each, cache lengths uniform in [8192, 65536]
    "decode": DSAConfig("decode", 64, 128, 2048, 128, 576, 512, "bf16", _S192, decode=True,
                        batch=64, ctx_range=(8192, 65536), max_ctx=65536),
    # 8 packed sequences with lengths uniform in [1024, 16384]
    "varlen": DSAConfig("varlen", 64, 128, 2048, 128, 576, 512, "bf16", _S192,
                        seqlens=(0,) * 8, varlen_range=(1024, 16384)),
}


def scaled(cfg: DSAConfig, **kw) -> DSAConfig:
    """A copy of ``cfg`` with some fields replaced (small parity cases)."""
    return replace(cfg, **kw)


def _lengths(cfg: DSAConfig, seed: int):
    g = torch.Generator().manual_seed(seed + 1)
    if cfg.decode:
        lo, hi = cfg.ctx_range
        return [int(x) for x in torch.randint(lo, hi + 1, (cfg.batch,), generator=g)]
    if cfg.varlen_range:
        lo, hi = cfg.varlen_range
        return [int(x) for x in torch.randint(lo, hi + 1, (len(cfg.seqlens),), generator=g)]
    return [int(x) for x in cfg.seqlens]


def _draw(g, shape, denom, device):
    x = torch.empty(*shape, device=device, dtype=torch.float32).normal_(generator=g)
    x.div_(denom)
    return x


def make_prefill_inputs(cfg: DSAConfig, device="cpu", seed: int = 0):
    """Packed prefill inputs: dict of q_idx, w, k_idx, q, kv, cu_seqlens (+ lengths)."""
    assert not cfg.decode
    lens = _lengths(cfg, seed)
    T = sum(lens)
    g = torch.Generator(device=device).manual_seed(seed)
    dt = cfg.torch_dtype
    q_idx = _draw(g, (T, cfg.n_idx_heads, cfg.idx_dim), math.sqrt(cfg.idx_dim), device)
    k_idx = _draw(g, (T, cfg.idx_dim), math.sqrt(cfg.idx_dim), device)
    w = _draw(g, (T, cfg.n_idx_heads), math.sqrt(cfg.n_idx_heads), device)
    q = _draw(g, (T, cfg.n_heads, cfg.d_qk), math.sqrt(cfg.d_qk), device).to(dt)
    kv = _draw(g, (T, cfg.d_qk), math.sqrt(cfg.d_qk), device).to(dt)
    if cfg.key_offset_std > 0:
        off = torch.empty(T, 1, device=device, dtype=torch.float32).normal_(generator=g) * cfg.key_offset_std
        k_idx.add_(off)
    cu = torch.zeros(len(lens) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0).to(torch.int32)
    return {
        "q_idx": q_idx.to(dt),
        "w": w,
        "k_idx": k_idx.to(dt),
        "q": q,
        "kv": kv,
        "cu_seqlens": cu.to(device),
        "lengths": lens,
        "max_seqlen": max(lens),
    }


def make_decode_inputs(cfg: DSAConfig, device="cpu", seed: int = 0):
    """Decode inputs: one query per sequence over indexer-key and latent-KV caches."""
    assert cfg.decode
    lens = _lengths(cfg, seed)
    B = cfg.batch
    g = torch.Generator(device=device).manual_seed(seed)
    dt = cfg.torch_dtype
    q_idx = _draw(g, (B, cfg.n_idx_heads, cfg.idx_dim), math.sqrt(cfg.idx_dim), device).to(dt)
    idx_cache = _draw(g, (B, cfg.max_ctx, cfg.idx_dim), math.sqrt(cfg.idx_dim), device).to(dt)
    w = _draw(g, (B, cfg.n_idx_heads), math.sqrt(cfg.n_idx_heads), device)
    q = _draw(g, (B, cfg.n_heads, cfg.d_qk), math.sqrt(cfg.d_qk), device).to(dt)
    kv_cache = _draw(g, (B, cfg.max_ctx, cfg.d_qk), math.sqrt(cfg.d_qk), device).to(dt)
    return {
        "q_idx": q_idx,
        "w": w,
        "idx_cache": idx_cache,
        "q": q,
        "kv_cache": kv_cache,
        "cache_seqlens": torch.tensor(lens, dtype=torch.int32, device=device),
        "lengths": lens,
        "max_ctx": cfg.max_ctx,
    }


def random_selection(lengths, topk, seed: int = 0):
    """A seeded selection of the shape the top-k step produces: for the query at position t
    of each packed sequence, min(topk, t + 1) distinct positions of 0..t in ascending order,
    padded with -1 to topk (every position when t + 1 <= topk, a uniform random subset
    otherwise).  int32 [sum(lengths), topk] on the CPU."""
    g = torch.Generator().manual_seed(seed + 7)
    rows = []
    for L in lengths:
        for t in range(L):
            n = t + 1
            if n <= topk:
                sel = torch.arange(n, dtype=torch.int32)
            else:
                sel = torch.randperm(n, generator=g)[:topk].sort().values.to(torch.int32)
            row = torch.full((topk,), -1, dtype=torch.int32)
            row[: sel.numel()] = sel
            rows.append(row)
    if not rows:
        return torch.empty((0, topk), dtype=torch.int32)
    return torch.stack(rows)


def make_backward_inputs(cfg: DSAConfig, T: int, device="cpu", seed: int = 0):
    """Gradients arriving at the forward's outputs (the pages give no loss): dout
    [T, H, d_v] in the config's dtype, dlse [T, H] fp32, and a gradient on the index scores
    d_scores [T, topk] fp32, all N(0, 1)."""
    g = torch.Generator(device=device).manual_seed(seed + 11)
    dout = _draw(g, (T, cfg.n_heads, cfg.d_v), 1.0, device).to(cfg.torch_dtype)
    dlse = _draw(g, (T, cfg.n_heads), 1.0, device)
    d_scores = _draw(g, (T, cfg.topk), 1.0, device)
    return {"dout": dout, "dlse": dlse, "d_scores": d_scores}
