"""Benchmark of the DSA forward step on B300.

Workload (default): long prefill, B=1, L=32768, indexer 64 heads x 128,
index_topk 2048, MLA 128 heads, 576/512, bf16, seeded synthetic inputs.
One step = one pass of the whole path: Lightning Indexer -> top-k ->
sparse MLA attention (the kernels dsa_forward launches, called stage by
stage so that each kernel is timed with CUDA events on its stream).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 (under torchrun): every rank runs its own independent problem of the
same size (weak scaling, no collective on the data path); the time is the
max over ranks.  --impl reference times the CPU oracle (numpy fp64) on a
bounded sample of query rows of the same workload.

Prints ONE JSON line (rank 0).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "DSA fwd queries/s and TFLOP/s per stage at L=32K, as % of B300 roofline"


def flop_per_pair_idx(cfg):
    """Indexer flop per causal (t, s) pair: H_I dot products of width D_I (16,384 at 64 x 128)."""
    return 2 * cfg.n_idx_heads * cfg.idx_dim


def flop_per_pair_attn(cfg):
    """Attention flop per selected (t, s) pair: q.k over d_qk and p.v over d_v for each head
    (278,528 at 128 heads, 576 / 512)."""
    return 2 * cfg.n_heads * (cfg.d_qk + cfg.d_v)


def _peaks():
    """Roofline denominators: the measured HBM copy bandwidth and bf16 GEMM throughput of this
    pool's B300s (burst for kernels timed alone, sustained for seconds-long loops), else the
    fallback figures.  The record's values and date travel in the bench line."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured", "when": d.get("when"), "gpu": d.get("gpu_name"), "how": d.get("how")}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback",
                "when": None, "gpu": None, "how": "fallback figures of the profiling recipe"}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(ms, ws, device):
    """The slowest rank's time (every rank gets it): the job is as fast as its slowest rank."""
    import torch
    import torch.distributed as dist

    t = torch.tensor([ms], dtype=torch.float64, device=device)
    if ws > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(units_per_rank, ws, ms_max):
    """Whole-job throughput: every rank processed units_per_rank in at most ms_max."""
    return units_per_rank * ws / (ms_max / 1e3)


def _workload_desc(cfg, lens):
    return (f"{cfg.name} prefill: B={len(lens)}, L={max(lens)} causal, indexer {cfg.n_idx_heads}x{cfg.idx_dim}, "
            f"index_topk={cfg.topk}, MLA {cfg.n_heads} heads {cfg.d_qk}/{cfg.d_v}, {cfg.dtype}")


def _work_counts(lens, k):
    causal = sum(L * (L + 1) // 2 for L in lens)
    selected = sum(sum(min(k, t + 1) for t in range(L)) for L in lens)
    return causal, selected


def clock_tail(step, flush, dev, timed_ms, min_ms=500.0, max_steps=20000):
    """nvidia-smi samples every 50 ms, so a timed region shorter than that holds no sample: keep
    the same untimed steps running after it until about min_ms of GPU work has passed, so the
    sampler (still running) sees the clocks of this work.  Returns the number of extra steps."""
    import torch

    total = sum(timed_ms)
    if total >= min_ms:
        return 0
    per = max(total / max(1, len(timed_ms)), 1e-3)
    extra = min(max_steps, int((min_ms - total) / per) + 1)
    for _ in range(extra):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    return extra


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    def __init__(self, index, path):
        self.path = path
        self.proc = None
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.f = open(path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(index), f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def _attn_traffic(cfg):
    """DRAM bytes per attention launch from the committed ncu summary, or None when the
    kernel source has changed since the counters were taken (or for other workloads)."""
    import hashlib

    if cfg.name != "long" or tuple(cfg.seqlens) != (32768,):
        return None
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)["attn_tc_kernel_long"]
        with open(os.path.join(ROOT, "sparse_attention_long_gemm_b300", "csrc", "attn_tc.cuh"), "rb") as f:
            sha = hashlib.sha1(f.read()).hexdigest()
    except (OSError, ValueError, KeyError):
        return None
    return rec["bytes_per_launch"] if rec.get("source_sha1") == sha else None


def _cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_sample(cfg, inp_cpu, rows):
    """Time the CPU oracle on the given rows; returns (seconds, rows)."""
    import oracle.dsa_oracle as O

    t0 = time.perf_counter()
    O.dsa_prefill(inp_cpu["q_idx"], inp_cpu["w"], inp_cpu["k_idx"], inp_cpu["q"], inp_cpu["kv"],
                  inp_cpu["cu_seqlens"], cfg.topk, cfg.softmax_scale, cfg.d_v, rows=rows)
    return time.perf_counter() - t0


def _sample_rows(L, k, n_extra, seed):
    import numpy as np

    rng = np.random.default_rng(seed)
    base = [0, k - 2, k - 1, k, L - 1]
    extra = [int(x) for x in rng.integers(0, L, size=n_extra)]
    return sorted(set(t for t in base + extra if 0 <= t < L))


def _host_copy_for_oracle(inp, rows):
    """Host copies the oracle needs: whole k_I / kv, and only the sampled rows of the per-query tensors."""
    out = {"k_idx": inp["k_idx"].cpu(), "kv": inp["kv"].cpu(), "cu_seqlens": inp["cu_seqlens"].cpu()}
    for name in ("q_idx", "w", "q"):
        out[name] = _RowView(inp[name][rows].cpu(), rows)
    return out


class _RowView:
    """Row-indexable view of a few host rows of a large device tensor (oracle input)."""

    def __init__(self, sub, rows):
        self.sub = sub
        self.pos = {r: i for i, r in enumerate(rows)}
        self.shape = (None,) + tuple(sub.shape[1:])

    def __getitem__(self, r):
        return self.sub[self.pos[int(r)]]


def run_reference(args, cfg):
    """--impl reference: the CPU oracle, as it stands, on a bounded sample of rows per step."""
    import torch

    ws, rank, _ = _dist()
    if rank != 0:
        return
    if cfg.decode:
        return run_reference_decode(args, cfg)
    from sparse_attention_long_gemm_b300.synth import make_prefill_inputs

    dev = "cuda:0" if torch.cuda.is_available() else "cpu"
    inp = make_prefill_inputs(cfg, dev, seed=0)
    L = inp["max_seqlen"]
    lens = inp["lengths"]
    rows_per_step = args.ref_rows
    rows = _sample_rows(L, cfg.topk, 4 * rows_per_step, seed=1)
    host = _host_copy_for_oracle(inp, rows)
    del inp
    import numpy as np

    rng = np.random.default_rng(2)
    times, done = [], 0
    for i in range(args.warmup + args.steps):
        step_rows = sorted(rng.choice(rows, size=min(rows_per_step, len(rows)), replace=False).tolist())
        dt = oracle_sample(cfg, host, step_rows)
        if i >= args.warmup:
            times.append(dt)
            done += len(step_rows)
    total = sum(times)
    v = done / total
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "queries/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": _workload_desc(cfg, lens), "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": v, "unit": "queries/s", "cores": _cpu_cores(), "kind": "oracle",
                         "sample": f"{rows_per_step} query rows per step drawn from positions {rows[:8]}..."
                                   f" (t in {{0,k-2,k-1,k,L-1}} + uniform), dense additive-mask oracle"},
        "e2e": {"value": v, "unit": "queries/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_reference_decode(args, cfg):
    """--impl reference, decode workload: the oracle's decode form on a sample of sequences per step."""
    import numpy as np
    import torch

    import oracle.dsa_oracle as O
    from sparse_attention_long_gemm_b300.synth import make_decode_inputs

    ws, _, _ = _dist()
    dev = "cuda:0" if torch.cuda.is_available() else "cpu"
    inp = make_decode_inputs(cfg, dev, seed=0)
    rng = np.random.default_rng(2)
    per_step = max(1, args.ref_seqs)
    times, done = [], 0
    for i in range(args.warmup + args.steps):
        bs = sorted(rng.choice(cfg.batch, size=per_step, replace=False).tolist())
        host = {n: inp[n][bs].cpu() for n in ("q_idx", "w", "q", "idx_cache", "kv_cache")}
        lens = [inp["lengths"][b] for b in bs]
        t0 = time.perf_counter()
        O.dsa_decode(host["q_idx"], host["w"], host["q"], host["idx_cache"], host["kv_cache"], lens, cfg.topk,
                     cfg.softmax_scale, cfg.d_v)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
            done += per_step
    total = sum(times)
    v = done / total
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "queries/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": _decode_desc(cfg), "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": v, "unit": "queries/s", "cores": _cpu_cores(), "kind": "oracle",
                         "sample": f"{per_step} of the {cfg.batch} decode sequences per step, dense additive-mask "
                                   f"oracle over the whole cache"},
        "e2e": {"value": v, "unit": "queries/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _decode_desc(cfg):
    return (f"decode: batch {cfg.batch} sequences, 1 query each, cache lengths U[{cfg.ctx_range[0]}, "
            f"{cfg.ctx_range[1]}] (max_ctx {cfg.max_ctx}), indexer {cfg.n_idx_heads}x{cfg.idx_dim} bf16 key cache, "
            f"latent KV cache {cfg.d_qk} bf16, MLA {cfg.n_heads} heads, index_topk={cfg.topk}")


def decode_bytes(cfg, lens):
    """Algorithmic HBM bytes of the decode stages (every stage streams or gathers from HBM)."""
    B, k = len(lens), cfg.topk
    ctx = sum(lens)
    sel = sum(min(k, n) for n in lens)
    idx_b = ctx * (cfg.idx_dim * 2 + 4) + B * cfg.n_idx_heads * (cfg.idx_dim * 2 + 4)   # keys, scores, q_I, w
    topk_b = ctx * 4 + B * k * 4                                                         # scores, indices
    attn_b = (sel * cfg.d_qk * 2 + B * k * 4                                             # gathered rows, indices
              + B * cfg.n_heads * (cfg.d_qk * 2 + cfg.d_v * 2 + 4))                      # q, out, lse
    return idx_b, topk_b, attn_b


def run_ours_decode(args, cfg):
    """Decode workload: the three decode-form stage calls timed with CUDA events, every stage
    against HBM bandwidth (they all stream or gather from HBM)."""
    import torch
    import torch.distributed as dist

    import sparse_attention_long_gemm_b300 as dsa
    from sparse_attention_long_gemm_b300.build import build_library
    from sparse_attention_long_gemm_b300.synth import make_decode_inputs

    ws, rank, local = _dist()
    if ws > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        build_library()
    if ws > 1:
        dist.barrier()
    p = dsa.params_from_config(cfg)
    inp = make_decode_inputs(cfg, dev, seed=rank)
    lens = inp["lengths"]
    Bn, max_ctx = cfg.batch, cfg.max_ctx
    ld = (max_ctx + 3) // 4 * 4
    scores = torch.empty((Bn, ld), dtype=torch.float32, device=dev)
    idx = torch.empty((Bn, cfg.topk), dtype=torch.int32, device=dev)
    out = torch.empty((Bn, cfg.n_heads, cfg.d_v), dtype=inp["q"].dtype, device=dev)
    lse = torch.empty((Bn, cfg.n_heads), dtype=torch.float32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)   # > L2 (126 MB)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream

    def step(evs=None):
        if evs:
            evs[0].record(stream)
        dsa.dsa_index_scores_decode(p, inp["q_idx"], inp["w"], inp["idx_cache"], inp["cache_seqlens"], Bn, max_ctx,
                                    scores, ld, sp)
        if evs:
            evs[1].record(stream)
        dsa.dsa_topk_decode(p, scores, ld, inp["cache_seqlens"], Bn, max_ctx, idx, sp)
        if evs:
            evs[2].record(stream)
        dsa.dsa_sparse_mla_attn_decode(p, inp["q"], inp["kv_cache"], idx, inp["cache_seqlens"], Bn, max_ctx, out,
                                       lse, sp)
        if evs:
            evs[3].record(stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    if dsa.dsa_get_device_error(sp) != 0:
        raise RuntimeError("device error during warm-up")
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    clocks_dir = os.environ.get("DSA_CLOCKS_DIR") or tempfile.gettempdir()
    sampler = ClockSampler(local, os.path.join(clocks_dir, f"dsa_clocks_rank{rank}.csv"))
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    for s_ in range(args.steps):
        flush.zero_()
        step(evs[s_])
    torch.cuda.synchronize(dev)
    if ws > 1:
        dist.barrier()
    st = [[e[i].elapsed_time(e[i + 1]) for i in range(3)] for e in evs]
    extra = clock_tail(step, flush, dev, [sum(x) for x in st])
    clocks = sampler.stop()
    if clocks is not None:
        clocks["untimed_steps_after"] = extra
    if dsa.dsa_get_device_error(sp) != 0:
        raise RuntimeError("device error during timing")
    step_ms = statistics.median(sum(x) for x in st)
    stage_ms = [statistics.median(x[i] for x in st) for i in range(3)]
    step_ms_max = max_over_ranks(step_ms, ws, dev)

    # ---- end to end: the step's per-query inputs from pinned host memory, the output back ----
    e2e = None
    if not args.no_e2e:
        names = ["q_idx", "w", "q", "cache_seqlens"]
        host = {n: inp[n].cpu().pin_memory() for n in names}
        dev_in = {n: torch.empty_like(inp[n]) for n in names}
        h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        wsb = torch.empty(dsa.dsa_decode_workspace_size(p, Bn, max_ctx), dtype=torch.uint8, device=dev)
        h2d = sum(v.numel() * v.element_size() for v in host.values())
        d2h = h_out.numel() * h_out.element_size()

        def e2e_step():
            for n in names:
                dev_in[n].copy_(host[n], non_blocking=True)
            dsa.dsa_forward_decode(p, dev_in["q_idx"], dev_in["w"], dev_in["q"], inp["idx_cache"], inp["kv_cache"],
                                   dev_in["cache_seqlens"], Bn, max_ctx, out, None, None, wsb, sp)
            h_out.copy_(out, non_blocking=True)

        for _ in range(max(1, min(args.warmup, 3))):
            e2e_step()
        torch.cuda.synchronize(dev)
        ne = max(3, args.steps)
        times = []
        for _ in range(ne):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            e2e_step()
            e1.record(stream)
            times.append((e0, e1))
        torch.cuda.synchronize(dev)
        e_ms = max_over_ranks(statistics.median(a.elapsed_time(b) for a, b in times), ws, dev)
        e2e = {"value": weak_scaling_value(Bn, ws, e_ms), "unit": "queries/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": ne,
               "note": "per-step inputs are the new queries (q_I, w, q) and cache lengths; the caches are "
                       "resident device state"}
        if dsa.dsa_get_device_error(sp) != 0:
            raise RuntimeError("device error during the end-to-end loop")

    if rank != 0:
        if ws > 1:
            dist.barrier()
            dist.destroy_process_group()
        return
    peaks = _peaks()
    hbm = peaks["hbm_gbs"]
    nbytes = decode_bytes(cfg, lens)
    gbs = [b / (ms * 1e-3) / 1e9 for b, ms in zip(nbytes, stage_ms)]
    names = ["index_scores", "topk", "sparse_mla_attn"]
    kernels = ["indexer_tc_kernel<1,5,2>", "topk", "attn_tc_kernel"]
    dom = max(range(3), key=lambda i: stage_ms[i])
    cpu = None
    if not args.no_cpu_baseline:
        cpu = cpu_baseline_decode(cfg, inp, args)
    line = {
        "metric": METRIC,
        "value": weak_scaling_value(Bn, ws, step_ms_max),
        "unit": "queries/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": step_ms_max,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": _decode_desc(cfg), "l2": "flushed (256 MB write) between timed steps",
                   "per_rank": "independent problem per rank (seed = rank)",
                   "timing": f"median of {args.steps} steps, CUDA events per stage"},
        "stages": {n: {"ms": ms, "gbs": g, "bytes": b, "frac_of_peak": g / hbm}
                   for n, ms, g, b in zip(names, stage_ms, gbs, nbytes)},
        "roofline": {"bound": "hbm", "kernel": kernels[dom], "achieved": gbs[dom], "peak": hbm, "unit": "GB/s",
                     "frac": gbs[dom] / hbm, "traffic": None, "peak_kind": f"HBM copy, {peaks['source']}",
                     "step_floor_us": sum(nbytes) / (hbm * 1e9) * 1e6, "peak_record": peaks},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "clocks": clocks,
        "gpu_launches": 3 * args.steps,
        "path": dsa.dsa_path_name(p),
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()


def cpu_baseline_decode(cfg, inp, args):
    """The oracle's decode form as it stands, on a bounded sample of the sequences."""
    import numpy as np

    import oracle.dsa_oracle as O

    rng = np.random.default_rng(1)
    batches = sorted(rng.choice(cfg.batch, size=min(cfg.batch, args.cpu_seqs), replace=False).tolist())
    host = {n: inp[n][batches].cpu() for n in ("q_idx", "w", "q", "idx_cache", "kv_cache")}
    lens = [inp["lengths"][b] for b in batches]
    t0 = time.perf_counter()
    O.dsa_decode(host["q_idx"], host["w"], host["q"], host["idx_cache"], host["kv_cache"], lens, cfg.topk,
                 cfg.softmax_scale, cfg.d_v)
    dt = time.perf_counter() - t0
    return {"value": len(batches) / dt, "unit": "queries/s", "cores": _cpu_cores(), "kind": "oracle",
            "sample": f"{len(batches)} of the {cfg.batch} decode sequences (cache lengths {lens}), "
                      f"{dt:.1f} s of CPU work"}


def run_ours(args, cfg):
    import torch
    import torch.distributed as dist

    import sparse_attention_long_gemm_b300 as dsa
    from sparse_attention_long_gemm_b300.build import build_library
    from sparse_attention_long_gemm_b300.synth import make_prefill_inputs

    if cfg.decode:
        return run_ours_decode(args, cfg)
    ws, rank, local = _dist()
    if ws > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        build_library()
    if ws > 1:
        dist.barrier()
    p = dsa.params_from_config(cfg, indexer_fp8=(args.indexer == "fp8"))
    inp = make_prefill_inputs(cfg, dev, seed=rank)   # weak scaling: one independent problem per rank
    lens = inp["lengths"]
    T = sum(lens)
    B = len(lens)
    maxL = inp["max_seqlen"]
    ld = (maxL + 3) // 4 * 4
    causal, selected = _work_counts(lens, cfg.topk)
    scores = torch.empty((T, ld), dtype=torch.float32, device=dev)
    idx = torch.empty((T, cfg.topk), dtype=torch.int32, device=dev)
    out = torch.empty((T, cfg.n_heads, cfg.d_v), dtype=inp["q"].dtype, device=dev)
    lse = torch.empty((T, cfg.n_heads), dtype=torch.float32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)   # > L2 (126 MB)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    fp8 = args.indexer == "fp8"
    if fp8:   # the indexer's FP8 operands: rotated E4M3 codes, w * s_q, s_k
        q8 = torch.empty((T, cfg.n_idx_heads, cfg.idx_dim), dtype=torch.uint8, device=dev)
        wq = torch.empty((T, cfg.n_idx_heads), dtype=torch.float32, device=dev)
        k8 = torch.empty((T, cfg.idx_dim), dtype=torch.uint8, device=dev)
        ks = torch.empty(T, dtype=torch.float32, device=dev)
        qev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]

    def step(evs=None, si=None):
        if evs:
            evs[0].record(stream)
        if fp8:
            dsa.dsa_indexer_quantize_fp8(p, inp["q_idx"], T * cfg.n_idx_heads, inp["w"], q8, wq, sp)
            dsa.dsa_indexer_quantize_fp8(p, inp["k_idx"], T, None, k8, ks, sp)
            if evs:
                qev[si].record(stream)
            dsa.dsa_index_scores_fp8(p, q8, wq, k8, ks, inp["cu_seqlens"], B, T, maxL, scores, ld, sp)
        else:
            dsa.dsa_index_scores(p, inp["q_idx"], inp["w"], inp["k_idx"], inp["cu_seqlens"], B, T, maxL, scores, ld,
                                 sp)
        if evs:
            evs[1].record(stream)
        dsa.dsa_topk(p, scores, ld, inp["cu_seqlens"], B, T, maxL, idx, sp)
        if evs:
            evs[2].record(stream)
        dsa.dsa_sparse_mla_attn(p, inp["q"], inp["kv"], idx, inp["cu_seqlens"], B, T, maxL, out, lse, sp)
        if evs:
            evs[3].record(stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    err = dsa.dsa_get_device_error(sp)
    if err != 0:
        raise RuntimeError(f"device error during warm-up: {err}")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    # raw samples go to DSA_CLOCKS_DIR when set (to keep them), else to the temp directory
    clocks_dir = os.environ.get("DSA_CLOCKS_DIR") or tempfile.gettempdir()
    sampler = ClockSampler(local, os.path.join(clocks_dir, f"dsa_clocks_rank{rank}.csv"))
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    for s in range(args.steps):
        flush.zero_()          # L2 flushed between steps (not inside the timed events)
        step(evs[s], s)
    torch.cuda.synchronize(dev)
    if ws > 1:
        dist.barrier()
    st = [[e[i].elapsed_time(e[i + 1]) for i in range(3)] for e in evs]
    quant_ms = statistics.median(evs[i][0].elapsed_time(qev[i]) for i in range(args.steps)) if fp8 else 0.0
    extra = clock_tail(step, flush, dev, [sum(x) for x in st])
    clocks = sampler.stop()
    if clocks is not None:
        clocks["untimed_steps_after"] = extra
    err = dsa.dsa_get_device_error(sp)
    if err != 0:
        raise RuntimeError(f"device error during timing: {err}")
    step_ms = statistics.median(sum(x) for x in st)
    stage_ms = [statistics.median(x[i] for x in st) for i in range(3)]
    step_ms_max = max_over_ranks(step_ms, ws, dev)

    # ---- end to end: host buffers, H2D + fused dsa_forward + D2H inside the timed region ----
    e2e = None
    if not args.no_e2e:
        names = ["q_idx", "w", "k_idx", "q", "kv", "cu_seqlens"]
        host = {n: inp[n].cpu().pin_memory() for n in names}
        h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        dev_in = {n: torch.empty_like(inp[n]) for n in names}
        del inp
        wsb = torch.empty(dsa.dsa_workspace_size(p, T, maxL, B), dtype=torch.uint8, device=dev)
        h2d = sum(v.numel() * v.element_size() for v in host.values())
        d2h = h_out.numel() * h_out.element_size()

        def e2e_step():
            for n in names:
                dev_in[n].copy_(host[n], non_blocking=True)
            dsa.dsa_forward(p, dev_in["q_idx"], dev_in["w"], dev_in["k_idx"], dev_in["q"], dev_in["kv"],
                            dev_in["cu_seqlens"], B, T, maxL, out, None, None, wsb, sp)
            h_out.copy_(out, non_blocking=True)

        for _ in range(max(1, min(args.warmup, 2))):
            e2e_step()
        torch.cuda.synchronize(dev)
        ne = max(2, min(args.steps, 5))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if ws > 1:
            dist.barrier()
        e0.record(stream)
        for _ in range(ne):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e_ms = max_over_ranks(e0.elapsed_time(e1) / ne, ws, dev)
        e2e = {"value": weak_scaling_value(T, ws, e_ms), "unit": "queries/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": ne}
        if dsa.dsa_get_device_error(sp) != 0:
            raise RuntimeError("device error during the end-to-end loop")

    if rank != 0:
        if ws > 1:
            dist.barrier()
            dist.destroy_process_group()
        return

    peaks = _peaks()
    idx_tf = causal * flop_per_pair_idx(cfg) / (stage_ms[0] * 1e-3) / 1e12
    topk_bytes = causal * 4 + T * cfg.topk * 4
    topk_gbs = topk_bytes / (stage_ms[1] * 1e-3) / 1e9
    attn_tf = selected * flop_per_pair_attn(cfg) / (stage_ms[2] * 1e-3) / 1e12
    peak_t = peaks["bf16_tflops"]
    peak_s = peaks["bf16_tflops_sustained"]
    traffic = _attn_traffic(cfg)
    if fp8:
        # the FP8 scores contraction alone, against the FP8 peak (the measured bf16 peak times the
        # nominal fp8 / bf16 ratio of 2)
        idx_tf = causal * flop_per_pair_idx(cfg) / ((stage_ms[0] - quant_ms) * 1e-3) / 1e12
        qbytes = T * (cfg.n_idx_heads + 1) * cfg.idx_dim * 3 + T * (cfg.n_idx_heads * 8 + 4)
    cpu = None
    if not args.no_cpu_baseline:
        cpu = cpu_baseline(cfg, args)
    line = {
        "metric": METRIC,
        "value": weak_scaling_value(T, ws, step_ms_max),
        "unit": "queries/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": step_ms_max,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": _workload_desc(cfg, lens), "l2": "flushed (256 MB write) between timed steps",
                   "per_rank": "independent problem per rank (seed = rank)",
                   "timing": f"median of {args.steps} steps, CUDA events per stage",
                   "indexer": "FP8 (Hadamard rotation, E4M3)" if fp8 else cfg.dtype},
        "stages": {
            "index_scores": ({"ms": stage_ms[0], "quantize_ms": quant_ms,
                              "quantize_gbs": qbytes / (quant_ms * 1e-3) / 1e9 if fp8 else None,
                              "scores_ms": stage_ms[0] - quant_ms, "tflops": idx_tf,
                              "frac_of_peak": idx_tf / (2 * peak_t), "peak": "fp8 = 2 x measured bf16"}
                             if fp8 else
                             {"ms": stage_ms[0], "tflops": idx_tf, "frac_of_peak": idx_tf / peak_t,
                              "frac_of_sustained": idx_tf / peak_s}),
            "topk": {"ms": stage_ms[1], "gbs": topk_gbs, "frac_of_peak": topk_gbs / peaks["hbm_gbs"]},
            "sparse_mla_attn": {"ms": stage_ms[2], "tflops": attn_tf, "frac_of_peak": attn_tf / peak_t,
                                "frac_of_sustained": attn_tf / peak_s,
                                # the gather inside the kernel: every selected row's d_qk elements (split
                                # between the two CTAs of a cluster, none fetched twice), from L2 or HBM
                                "gather_gbs": selected * cfg.d_qk * (2 if cfg.dtype == "bf16" else 4)
                                / (stage_ms[2] * 1e-3) / 1e9},
        },
        "roofline": {"bound": "tensor", "kernel": "attn_tc_kernel", "achieved": attn_tf, "peak": peak_t,
                     "unit": "TFLOP/s", "frac": attn_tf / peak_t, "traffic": traffic,
                     "peak_kind": f"bf16 dense, burst, {peaks['source']}",
                     "frac_of_sustained": attn_tf / peak_s, "peak_record": peaks},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "clocks": clocks,
        "gpu_launches": (5 if fp8 else 3) * args.steps,
        "path": dsa.dsa_path_name(p),
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()


def cpu_baseline(cfg, args):
    """The oracle as it stands on the host cores, on a bounded sample of the same workload."""
    import torch

    from sparse_attention_long_gemm_b300.synth import make_prefill_inputs

    inp = make_prefill_inputs(cfg, "cuda:0", seed=0)
    L = inp["max_seqlen"]
    rows = _sample_rows(L, cfg.topk, args.cpu_rows, seed=1)
    host = _host_copy_for_oracle(inp, rows)
    del inp
    torch.cuda.empty_cache()
    dt = oracle_sample(cfg, host, rows)
    return {"value": len(rows) / dt, "unit": "queries/s", "cores": _cpu_cores(), "kind": "oracle",
            "sample": f"{len(rows)} query rows of the same workload (t in {{0,k-2,k-1,k,L-1}} + uniform), "
                      f"{dt:.1f} s of CPU work"}


Q_LORA_RANK = 1536    # DeepseekV3Config defaults (q_lora_rank, hidden_size), shared by V3.2
HIDDEN = 7168


def run_inputs(args, cfg):
    """Upstream of the path: the indexer's input projections for every token of the prefill
    workload (q_idx = q_latent . wq_b^T, k_idx = x . wk^T, w = x . w_proj^T) on the tensor cores,
    and one update_indexer append per sequence of the decode workload.  One JSON line, its own
    metric (the projections' TFLOP/s against the bf16 peak); not the step of the headline."""
    import torch

    import sparse_attention_long_gemm_b300 as dsa
    from sparse_attention_long_gemm_b300.synth import CONFIGS

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    p = dsa.params_from_config(cfg)
    T, H, D = sum(cfg.seqlens), cfg.n_idx_heads, cfg.idx_dim
    g = torch.Generator(device=dev).manual_seed(0)
    q_lat = torch.randn(T, Q_LORA_RANK, device=dev, generator=g).to(torch.bfloat16)
    x = torch.randn(T, HIDDEN, device=dev, generator=g).to(torch.bfloat16)
    wq_b = (torch.randn(H * D, Q_LORA_RANK, device=dev, generator=g) / Q_LORA_RANK ** 0.5).to(torch.bfloat16)
    wk = (torch.randn(D, HIDDEN, device=dev, generator=g) / HIDDEN ** 0.5).to(torch.bfloat16)
    wp = (torch.randn(H, HIDDEN, device=dev, generator=g) / HIDDEN ** 0.5).to(torch.bfloat16)
    q_idx = torch.empty((T, H, D), dtype=torch.bfloat16, device=dev)
    k_idx = torch.empty((T, D), dtype=torch.bfloat16, device=dev)
    w = torch.empty((T, H), dtype=torch.float32, device=dev)
    # decode caches of the decode workload, one append per sequence
    dc = CONFIGS["decode"]
    Bn, M = dc.batch, dc.max_ctx
    idx_cache = torch.zeros((Bn, M, D), dtype=torch.bfloat16, device=dev)
    kv_cache = torch.zeros((Bn, M, dc.d_qk), dtype=torch.bfloat16, device=dev)
    k_new = torch.randn(Bn, D, device=dev, generator=g).to(torch.bfloat16)
    kv_new = torch.randn(Bn, dc.d_qk, device=dev, generator=g).to(torch.bfloat16)
    lens = torch.zeros(Bn, dtype=torch.int32, device=dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    shapes = [(q_lat, Q_LORA_RANK, wq_b, H * D, q_idx, dsa.DSA_BF16), (x, HIDDEN, wk, D, k_idx, dsa.DSA_BF16),
              (x, HIDDEN, wp, H, w, dsa.DSA_FP32)]

    def step(evs=None):
        for i, (a, kk, b, n, c, dt) in enumerate(shapes):
            if evs is not None:
                evs[i].record()
            dsa.dsa_gemm_bf16(a, kk, b, kk, T, n, kk, c, n, dt)
        if evs is not None:
            evs[3].record()
        lens.zero_()
        dsa.dsa_update_indexer(p, k_new, kv_new, Bn, M, lens, idx_cache, kv_cache)
        if evs is not None:
            evs[4].record()

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    clocks_dir = os.environ.get("DSA_CLOCKS_DIR") or tempfile.gettempdir()
    sampler = ClockSampler(0, os.path.join(clocks_dir, "dsa_clocks_inputs.csv"))
    torch.cuda.synchronize(dev)
    for s_ in range(args.steps):
        flush.zero_()
        step(evs[s_])
    torch.cuda.synchronize(dev)
    st = [[e[i].elapsed_time(e[i + 1]) for i in range(4)] for e in evs]
    extra = clock_tail(step, flush, dev, [sum(x) for x in st])
    clocks = sampler.stop()
    if clocks is not None:
        clocks["untimed_steps_after"] = extra
    if dsa.dsa_get_device_error() != 0:
        raise RuntimeError("device error during timing")
    ms = [statistics.median(x[i] for x in st) for i in range(4)]
    peaks = _peaks()
    flops = [2.0 * T * kk * n for (_, kk, _, n, _, _) in shapes]
    tf = [f / (m * 1e9) for f, m in zip(flops, ms[:3])]
    tot_tf = sum(flops) / (sum(ms[:3]) * 1e9)
    upd_bytes = 2 * Bn * (D + dc.d_qk) * 2 + 2 * Bn * 4   # rows read and written, lengths read and written
    upd_gbs = upd_bytes / (ms[3] * 1e6)
    names = ["q_idx = q_latent.wq_b^T", "k_idx = x.wk^T", "w = x.w_proj^T"]
    line = {
        "metric": "indexer input projections TFLOP/s (q_lora_rank 1536, hidden 7168)",
        "value": tot_tf, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": sum(ms[:3]), "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{cfg.name}: {T} tokens; update_indexer: {Bn} sequences of the decode caches",
                   "l2": "flushed (256 MB write) between timed steps", "timing": f"median of {args.steps} steps"},
        "stages": {nm: {"m": T, "n": n, "k": kk, "ms": m, "tflops": t, "frac_of_peak": t / peaks["bf16_tflops"]}
                   for nm, (_, kk, _, n, _, _), m, t in zip(names, shapes, ms[:3], tf)},
        "update_indexer": {"us": ms[3] * 1e3, "bytes": upd_bytes, "gbs": upd_gbs},
        "roofline": {"bound": "tensor", "kernel": "gemm_tc_kernel<256,true>", "achieved": tf[0],
                     "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": tf[0] / peaks["bf16_tflops"],
                     "peak_kind": f"bf16 dense, burst, {peaks['source']}"},
        "clocks": clocks, "gpu_launches": 4 * args.steps,
    }
    print(json.dumps(line), flush=True)


def flop_per_pair_attn_bwd(cfg):
    """Attention-backward flop per selected (t, s) pair: the logits q.k (d_qk) and dP = dO.v (d_v)
    recomputed, dq += dz.kv (d_qk), dkv += dz.q (d_qk) + p.dO (d_v), for each head (704,512 at
    128 heads, 576 / 512)."""
    return 2 * cfg.n_heads * (3 * cfg.d_qk + 2 * cfg.d_v)


def flop_per_pair_idx_bwd(cfg):
    """Index-score-backward flop per listed (t, s) pair: S = q_I.k_I, dq_I += G.k_I and
    dk_I += G.q_I for each indexer head (49,152 at 64 x 128)."""
    return 3 * 2 * cfg.n_idx_heads * cfg.idx_dim


def run_backward(args, cfg):
    """Backward of the path with the selection fixed (training): the attention's dq and dkv and
    the index scores' dq_I, dw, dk_I at the selected positions, for the output gradients of a
    loss the pages do not give (seeded N(0, 1) inputs).  The selection, out and lse come from the
    library's forward over the same inputs (untimed).  One JSON line with its own metric: the
    two kernels' TFLOP/s against the CUDA cores' fp32 FMA peak (they run in fp32 on the CUDA
    cores) and, for reference, the bf16 tensor peak."""
    import torch

    import sparse_attention_long_gemm_b300 as dsa
    from sparse_attention_long_gemm_b300.build import build_library
    from sparse_attention_long_gemm_b300.synth import make_backward_inputs, make_prefill_inputs

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    build_library()
    p = dsa.params_from_config(cfg)
    inp = make_prefill_inputs(cfg, dev, seed=0)
    lens = inp["lengths"]
    T, B, maxL = sum(lens), len(lens), inp["max_seqlen"]
    ld = (maxL + 3) // 4 * 4
    _, selected = _work_counts(lens, cfg.topk)
    scores = torch.empty((T, ld), dtype=torch.float32, device=dev)
    idx = torch.empty((T, cfg.topk), dtype=torch.int32, device=dev)
    out = torch.empty((T, cfg.n_heads, cfg.d_v), dtype=inp["q"].dtype, device=dev)
    lse = torch.empty((T, cfg.n_heads), dtype=torch.float32, device=dev)
    cu = inp["cu_seqlens"]
    dsa.dsa_index_scores(p, inp["q_idx"], inp["w"], inp["k_idx"], cu, B, T, maxL, scores, ld)
    dsa.dsa_topk(p, scores, ld, cu, B, T, maxL, idx)
    dsa.dsa_sparse_mla_attn(p, inp["q"], inp["kv"], idx, cu, B, T, maxL, out, lse)
    del scores
    bw = make_backward_inputs(cfg, T, dev, seed=0)
    dq = torch.empty((T, cfg.n_heads, cfg.d_qk), dtype=torch.float32, device=dev)
    dkv = torch.empty((T, cfg.d_qk), dtype=torch.float32, device=dev)
    dqi = torch.empty((T, cfg.n_idx_heads, cfg.idx_dim), dtype=torch.float32, device=dev)
    dwi = torch.empty((T, cfg.n_idx_heads), dtype=torch.float32, device=dev)
    dki = torch.empty((T, cfg.idx_dim), dtype=torch.float32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)   # > L2 (126 MB)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream

    def step(evs=None):
        if evs:
            evs[0].record(stream)
        dsa.dsa_sparse_mla_attn_bwd(p, inp["q"], inp["kv"], idx, cu, B, T, maxL, out, lse, bw["dout"], bw["dlse"],
                                    dq, dkv, sp)
        if evs:
            evs[1].record(stream)
        dsa.dsa_index_scores_bwd(p, inp["q_idx"], inp["w"], inp["k_idx"], idx, bw["d_scores"], cu, B, T, maxL, dqi,
                                 dwi, dki, sp)
        if evs:
            evs[2].record(stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    if dsa.dsa_get_device_error() != 0:
        raise RuntimeError("device error during warm-up")
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    clocks_dir = os.environ.get("DSA_CLOCKS_DIR") or tempfile.gettempdir()
    sampler = ClockSampler(0, os.path.join(clocks_dir, "dsa_clocks_backward.csv"))
    torch.cuda.synchronize(dev)
    for s_ in range(args.steps):
        flush.zero_()
        step(evs[s_])
    torch.cuda.synchronize(dev)
    st = [[e[i].elapsed_time(e[i + 1]) for i in range(2)] for e in evs]
    extra = clock_tail(step, flush, dev, [sum(x) for x in st])
    clocks = sampler.stop()
    if clocks is not None:
        clocks["untimed_steps_after"] = extra
    if dsa.dsa_get_device_error() != 0:
        raise RuntimeError("device error during timing")
    ms = [statistics.median(x[i] for x in st) for i in range(2)]
    peaks = _peaks()
    props = torch.cuda.get_device_properties(dev)
    mhz = (clocks or {}).get("sm_max_mhz") or 2032.0
    # fp32 FMA peak of the CUDA cores: 128 lanes per SM, 2 flop per FMA, at the maximum SM clock
    alu_peak = props.multi_processor_count * 128 * 2 * mhz * 1e6 / 1e12
    fl = [selected * flop_per_pair_attn_bwd(cfg), selected * flop_per_pair_idx_bwd(cfg)]
    # the DeepSeek-V3.2 shape in bf16 takes the tensor-core backward (warp-level MMAs)
    idx_tc = cfg.dtype == "bf16" and cfg.n_idx_heads == 64 and cfg.idx_dim == 128
    tc_shape = idx_tc and cfg.n_heads == 128 and cfg.d_qk == 576 and cfg.d_v == 512
    tf = [f / (m * 1e9) for f, m in zip(fl, ms)]
    line = {
        "metric": "DSA backward (selection fixed) TFLOP/s: sparse attention + index scores",
        "value": sum(fl) / (sum(ms) * 1e9), "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": sum(ms), "higher_is_better": True, "dtype": "f32 (bf16 inputs)",
        "data": "synthetic",
        "config": {"workload": _workload_desc(cfg, lens) + f"; {selected} selected pairs",
                   "l2": "flushed (256 MB write) between timed steps", "timing": f"median of {args.steps} steps"},
        "stages": {
            "sparse_mla_attn_bwd": {"ms": ms[0], "tflops": tf[0], "flop_per_pair": flop_per_pair_attn_bwd(cfg),
                                    "kernel": "attn_bwd_mma_kernel (bf16 mma.sync)" if tc_shape
                                    else "attn_bwd_kernel (fp32 CUDA cores)",
                                    "frac_of_bf16_peak": tf[0] / peaks["bf16_tflops"],
                                    "frac_of_alu_peak": None if tc_shape else tf[0] / alu_peak},
            "index_scores_bwd": {"ms": ms[1], "tflops": tf[1], "flop_per_pair": flop_per_pair_idx_bwd(cfg),
                                 "kernel": "index_scores_bwd_mma_kernel (bf16 mma.sync)" if idx_tc
                                 else "index_scores_bwd_kernel (fp32 CUDA cores)",
                                 "frac_of_bf16_peak": tf[1] / peaks["bf16_tflops"],
                                 "frac_of_alu_peak": None if idx_tc else tf[1] / alu_peak},
        },
        "roofline": ({"bound": "tensor", "kernel": "attn_bwd_mma_kernel", "achieved": tf[0],
                      "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": tf[0] / peaks["bf16_tflops"],
                      "peak_kind": f"bf16 dense, burst, {peaks['source']} (warp-level MMA, not tcgen05)"}
                     if tc_shape else
                     {"bound": "alu", "kernel": "attn_bwd_kernel", "achieved": tf[0], "peak": alu_peak,
                      "unit": "TFLOP/s", "frac": tf[0] / alu_peak,
                      "peak_kind": f"fp32 FMA on the CUDA cores: {props.multi_processor_count} SMs x 128 lanes x "
                                   f"2 flop x {mhz:.0f} MHz"}),
        "clocks": clocks, "gpu_launches": 4 * args.steps,   # two zero fills and the two backward kernels
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="long")
    ap.add_argument("--seqlen", type=int, default=0, help="override: one prefill sequence of this length")
    ap.add_argument("--indexer", default="native", choices=["native", "fp8"],
                    help="fp8: the indexer's FP8 form (rotation + E4M3 codes) in place of bf16")
    ap.add_argument("--stage", default="forward", choices=["forward", "inputs", "backward"],
                    help="inputs: time the indexer's input projections and the cache append instead; "
                         "backward: time the backward calls (selection fixed)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-rows", type=int, default=24)
    ap.add_argument("--ref-rows", type=int, default=6)
    ap.add_argument("--cpu-seqs", type=int, default=4)
    ap.add_argument("--ref-seqs", type=int, default=1)
    args = ap.parse_args()
    from sparse_attention_long_gemm_b300.synth import CONFIGS

    cfg = CONFIGS[args.config]
    if args.seqlen:   # a smaller single-sequence prefill of the same shape (profiling captures)
        from sparse_attention_long_gemm_b300.synth import scaled

        cfg = scaled(cfg, seqlens=(args.seqlen,), varlen_range=())
    if args.stage == "inputs":
        run_inputs(args, cfg)
    elif args.stage == "backward":
        run_backward(args, cfg)
    elif args.impl == "reference":
        run_reference(args, cfg)
    else:
        run_ours(args, cfg)


if __name__ == "__main__":
    main()
