#!/usr/bin/env python3
"""Benchmark of one MLA decode step (absorb_q → decode_fwd → combine_up_v) on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload all|NAME] [--no-cpu-baseline]

Prints ONE JSON line on rank 0. A "step" is one pass of the whole hot path over one
batch of synthetic inputs; the latent cache and the weights are resident in HBM
(they are the layer's state) and L2 is flushed (256 MiB write) before every timed
step (the write is followed by a 256 MiB read so that no dirty lines of the flush
are written back inside the timed kernels). `value` = latent-cache bytes per step ÷
step time (GB/s), summed over ranks; each rank decodes its own batch (weak scaling,
no data-path collective).

The headline is the DeepSeek-V2 shape (B = 32 × 4096 tokens); with `--workload all`
(the default) the other four workloads are measured in the same run and reported
under "workloads", each with its own roofline, per-call times, e2e and CPU baseline.
`--impl reference` times the fp64 CPU oracle on a fixed bounded sample instead.
"""
from __future__ import annotations

import argparse
import gc
import json
import math
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "MLA decode latent-cache GB/s, tokens/s, % HBM roofline on 1 B300"
HEADLINE = "v2_b32_l4096"
L2_FLUSH_BYTES = 256 << 20
N_CALLS = 3                                  # absorb_q, decode_fwd, combine_up_v
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}

# The oracle's bounded sample of each workload: (sequence, heads or None = all). The
# same sample serves the CPU baseline of our arm and every step of the reference arm,
# sized to a few seconds of fp64 work on a many-core host.
ORACLE_SAMPLE = {
    "tiny_h16_b1_l256": [(0, None)],
    "v2_b32_l4096": [(b, None) for b in range(4)],
    "paged_b64_l1k_32k": [(b, list(range(32))) for b in range(4)],
    "long_b4_l128k": [(0, list(range(16)))],
    "fp8_b128_l8192": [(b, list(range(64))) for b in range(8)],
}


# ------------------------------- distributed --------------------------------------
class Dist:
    """Rank bookkeeping; a world of 1 needs no process group."""

    def __init__(self, backend: str | None = None):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist

            dist.init_process_group(backend=backend or "nccl")
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, x: float, device=None) -> float:
        if self.pg is None:
            return float(x)
        import torch

        t = torch.tensor([float(x)], dtype=torch.float64, device=device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def sum(self, x: float, device=None) -> float:
        if self.pg is None:
            return float(x)
        import torch

        t = torch.tensor([float(x)], dtype=torch.float64, device=device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


def rank_workload(w: W.Workload, rank: int) -> W.Workload:
    """Each rank decodes its own batch: same shape, its own seed."""
    return w if rank == 0 else w.with_(seed=w.seed + 1000 * rank)


# ------------------------------- helpers -------------------------------------------
def load_peaks() -> tuple[dict, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi sampling (200 ms) during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info

        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return host_cores()


def num_splits_for(w: W.Workload, lens) -> int:
    """The split count the library resolves num_splits = 0 to (a host-only query)."""
    import mla_latent_kv_69_b300 as mla

    return mla.num_splits(w.batch, int(np.max(lens)) if len(lens) else 0, w.n_h)


def workload_config(w: W.Workload, lens, n_splits: int) -> dict:
    """`config` of a JSON line; both arms print the same dict for the same workload."""
    return {"workload": w.name, "n_h": w.n_h, "batch_per_gpu": w.batch, "ctx": int(np.max(lens)),
            "tokens_per_gpu": int(np.sum(lens, dtype=np.int64)), "kv": w.kv,
            "layout": "paged-64" if w.paged else "contiguous", "n_splits": int(n_splits),
            "schedule": "library default (num_splits = 0): slots per sequence = n_splits",
            "l2": "flushed before every timed step (256 MiB write, then a 256 MiB read; both outside the timed "
                  "intervals); the cache of every workload but the tiny one is also larger than L2"}


def oracle_sample_desc(w: W.Workload) -> str:
    parts = [f"seq {b} ({'all' if h is None else len(h)} heads)" for b, h in ORACLE_SAMPLE[w.name]]
    return f"{w.name}: " + ", ".join(parts) + "; fp64 explicit (non-absorbed) form"


class OracleSample:
    """The workload's fixed oracle sample, generated once; run() times one pass."""

    def __init__(self, w: W.Workload):
        from oracle import fp8_e4m3

        self.w = w
        lens = W.seq_lens(w)
        qb = W.gen_q(w)
        self.wk, self.wv = W.bf16_bits_to_f32(W.gen_w_uk(w)), W.bf16_bits_to_f32(W.gen_w_uv(w))
        per_tok = W.D_ROW * 2 if w.kv == "bf16" else W.D_ROW + 4
        self.items, self.bytes = [], 0.0
        for b, heads in ORACLE_SAMPLE[w.name]:
            L = int(lens[b])
            rows = W.bf16_bits_to_f32(W.gen_rows(w, b, L))
            if w.kv == "fp8":
                codes, scales = fp8_e4m3.quantize_rows(rows)
                rows = fp8_e4m3.dequantize_rows(codes, scales)
            self.items.append((W.bf16_bits_to_f32(qb[b]), rows, heads, max(L - 1, 0)))
            self.bytes += L * per_tok * (w.n_h if heads is None else len(heads)) / w.n_h

    def run(self) -> float:
        from oracle import mla_oracle

        t0 = time.perf_counter()
        for q, rows, heads, pos in self.items:
            mla_oracle.attend_explicit(q, rows[:, :512], rows[:, 512:], self.wk, self.wv, pos_q=pos, heads=heads)
        return time.perf_counter() - t0


def cpu_baseline(w: W.Workload, budget_s: float) -> dict:
    """The oracle as it stands, on the host cores, repeating the fixed sample for about
    `budget_s` seconds: cache GB/s equivalent (bytes scaled by the heads evaluated)."""
    smp = OracleSample(w)
    spent, reps = 0.0, 0
    while reps == 0 or spent < budget_s:
        spent += smp.run()
        reps += 1
    return {"value": round(smp.bytes * reps / spent / 1e9, 5), "unit": "GB/s", "cores": _blas_threads(),
            "kind": "oracle", "sample": oracle_sample_desc(w) + f"; {reps} pass(es)", "seconds": round(spent, 2)}


# ------------------------------- our arm -------------------------------------------
def measure_ours(name: str, args, dist: Dist, headline: bool) -> dict:
    """One workload on this rank's GPU: device-timed step (CUDA graph), per-call
    intervals, end-to-end through the public call with host buffers, roofline."""
    import torch

    import mla_latent_kv_69_b300 as mla

    dev = torch.device("cuda", dist.local_rank)
    w = rank_workload(W.WORKLOADS[name], dist.rank)
    case = W.DeviceInputs(w, dev)
    if w.kv == "fp8":                     # the library's own cache writer makes the e4m3 cache
        codes, scales = mla.quantize_fp8(case.source)
        cache = mla.Cache(codes, scales, case.block_table)
        del case.source
    else:
        cache = mla.Cache(case.source, None, case.block_table)
    B, n_h = case.B, case.n_h
    S = mla.num_splits(B, case.max_len, n_h)   # slots of the library's own schedule (n_splits = 0)
    bufs = dict(
        q_lat=torch.empty(B, n_h, 576, dtype=torch.bfloat16, device=dev),
        o_part=torch.empty(B, S, n_h, 512, dtype=torch.float32, device=dev),
        lse_part=torch.empty(B, S, n_h, dtype=torch.float32, device=dev),
        o=torch.empty(B, n_h, 128, dtype=torch.float32, device=dev),
    )
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    drain = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    drain_out = torch.empty(1, dtype=torch.float32, device=dev)

    def flush_l2():
        # Write a buffer larger than L2, then read another one: the read evicts the
        # written lines (their write-back happens here), so the timed kernels start
        # with a cold L2 that holds no dirty lines of the flush.
        flush.zero_()
        torch.sum(drain, dim=0, keepdim=True, out=drain_out)

    cache_bytes = W.cache_bytes(w, case.lens)
    weight_bytes = 2 * n_h * 128 * 512 * 2
    io_bytes = B * n_h * (192 * 2 + 576 * 2 * 2 + 128 * 4)     # q read, q_lat write+read, o write
    stream = torch.cuda.current_stream()

    def call(i):
        if i == 0:
            mla.absorb_q(case.q, case.w_uk, case.pos, q_lat=bufs["q_lat"])
        elif i == 1:
            mla.decode_fwd(bufs["q_lat"], cache, case.seq_lens, case.max_len, n_splits=0,
                           o_part=bufs["o_part"], lse_part=bufs["lse_part"])
        else:   # the merge of the split partials and W_UV, one launch; o only
            mla.combine_up_v(bufs["o_part"], bufs["lse_part"], case.w_uv, o=bufs["o"])

    def step():
        for i in range(N_CALLS):
            call(i)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # The timed step is one CUDA-graph replay: an L2 flush (outside the timed interval),
    # then the three library calls between two device-side events. Consecutive kernels of
    # the step overlap their launch and prologue with the previous kernel's tail
    # (programmatic dependent launch), so no event may sit between them in this graph;
    # a second graph with events between the calls gives the per-call breakdown.
    ev_step = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(2)]
    ev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(N_CALLS + 1)]
    graph, graph_parts = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        step()                              # the first call on a stream sets up kernel attributes
        torch.cuda.synchronize()
        with torch.cuda.graph(graph, stream=cap):
            flush_l2()
            ev_step[0].record()
            step()
            ev_step[1].record()
        with torch.cuda.graph(graph_parts, stream=cap):
            flush_l2()
            ev[0].record()
            for i in range(N_CALLS):
                call(i)
                ev[i + 1].record()
    torch.cuda.current_stream().wait_stream(cap)
    for _ in range(max(args.warmup, 3)):
        graph.replay()
        graph_parts.replay()
    torch.cuda.synchronize()

    # The e2e and cache-write timings come before the clock-sampling window: host API
    # calls of this process ran several times slower for a few hundred ms after the
    # nvidia-smi sampler stopped, which would charge the sampler to the library.
    # e2e through the public API with host buffers: per step, H2D of the new queries
    # (+ positions, lengths) from pinned memory, the three calls, and D2H of o. The
    # eager form makes the three Python calls every step (mla.decode_step); beside it,
    # the step captured once as a CUDA graph (mla.DecodeStepGraph).
    h_q = case.q.cpu().pin_memory()
    h_pos = case.pos.cpu().pin_memory()
    h_len = case.seq_lens.cpu().pin_memory()
    h_o = torch.empty(B, n_h, 128, dtype=torch.float32).pin_memory()
    d_q, d_pos, d_len = torch.empty_like(case.q), torch.empty_like(case.pos), torch.empty_like(case.seq_lens)
    e2e_bufs = dict(bufs)

    def eager_step():
        d_q.copy_(h_q, non_blocking=True)
        d_pos.copy_(h_pos, non_blocking=True)
        d_len.copy_(h_len, non_blocking=True)
        mla.decode_step(d_q, case.w_uk, case.w_uv, cache, d_len, d_pos, case.max_len, n_splits=0, bufs=e2e_bufs,
                        latent=False)
        h_o.copy_(e2e_bufs["o"], non_blocking=True)

    g = mla.DecodeStepGraph(case.w_uk, case.w_uv, cache, B, case.max_len)
    g.h_q.copy_(h_q)
    g.h_pos.copy_(h_pos)
    g.h_seq_lens.copy_(h_len)

    def time_e2e(run, st):
        for _ in range(max(args.warmup, 10)):   # first calls pay one-time host setup
            run()
        torch.cuda.synchronize()
        e2e_ms, host_ms = [], []
        for _ in range(max(args.steps, 30)):
            flush_l2()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(st)
            t0 = time.perf_counter()
            run()
            host_ms.append(1e3 * (time.perf_counter() - t0))
            b.record(st)
            b.synchronize()
            e2e_ms.append(a.elapsed_time(b))
        return e2e_ms, host_ms

    e2e_ms, host_ms = time_e2e(g.replay, g.stream)
    eager_ms, eager_host_ms = time_e2e(eager_step, stream)
    torch.cuda.synchronize()
    same_o = bool(torch.equal(g.h_o, h_o))   # both forms computed the same step
    e2e_mean = dist.max(float(np.mean(e2e_ms)), dev)
    eager_mean = dist.max(float(np.mean(eager_ms)), dev)
    del g

    # The cache write of the step's new tokens (mla_cache_append): one token per
    # sequence, hidden size 5120, written over each sequence's newest row.
    d_model = W.D_MODEL
    h_new = W.bits_to_torch_bf16(W.gen_hidden(w.seed, B, d_model), dev)
    w_dkv = W.bits_to_torch_bf16(W.gen_w_dkv(w.seed, d_model), dev)
    w_kr = W.bits_to_torch_bf16(W.gen_w_kr(w.seed, d_model), dev)
    a_seq = torch.arange(B, dtype=torch.int32, device=dev)
    a_pos = torch.clamp(case.seq_lens - 1, min=0)
    a_stage = torch.empty(B, 576, dtype=torch.bfloat16, device=dev) if w.kv == "fp8" else None
    for _ in range(3):
        mla.cache_append(h_new, w_dkv, w_kr, a_seq, a_pos, cache, staging=a_stage)
    torch.cuda.synchronize()
    app_ms = []
    for _ in range(args.steps):
        flush_l2()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        mla.cache_append(h_new, w_dkv, w_kr, a_seq, a_pos, cache, staging=a_stage)
        b.record(stream)
        b.synchronize()
        app_ms.append(a.elapsed_time(b))
    app_mean = float(np.mean(app_ms))
    row_bytes = 576 * 2 if w.kv == "bf16" else 576 + 4 + 2 * 576 * 2   # e4m3: codes + scale, staging out and in
    app_bytes = 576 * d_model * 2 + B * d_model * 2 + B * row_bytes
    del h_new, w_dkv, w_kr, a_seq, a_pos, a_stage

    K = args.steps
    sampler = ClockSampler(dist.local_rank if "CUDA_VISIBLE_DEVICES" not in os.environ else 0)
    sampler.start()
    # Keep the GPU under this load for a while so nvidia-smi's 200 ms samples cover it;
    # the timed steps follow immediately inside the same sampling window.
    t_soak = time.perf_counter()
    while time.perf_counter() - t_soak < args.soak:
        for _ in range(20):
            graph.replay()
        torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    steps = []
    for _ in range(K):
        graph.replay()
        torch.cuda.synchronize()
        steps.append(ev_step[0].elapsed_time(ev_step[1]))   # ms
    torch.cuda.synchronize()
    dist.barrier()
    clocks = sampler.stop()
    per = []
    for _ in range(K):
        graph_parts.replay()
        torch.cuda.synchronize()
        per.append([ev[i].elapsed_time(ev[i + 1]) for i in range(N_CALLS)])   # ms
    per = np.array(per)
    step_ms = float(np.mean(steps))
    kern_ms = per.mean(axis=0)
    step_ms_max = dist.max(step_ms, dev)


    peaks, peaks_src = load_peaks()
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    total_cache = dist.sum(cache_bytes, dev)
    value = total_cache / (step_ms_max / 1e3) / 1e9
    decode_ms = float(kern_ms[1])
    achieved = cache_bytes / (decode_ms / 1e3) / 1e9
    # Which pipe bounds the decode kernel: QK^T over 576 and PV over 512 columns per
    # (token, head) against the cache bytes; a bf16 cache sits just under the measured
    # ridge (HBM-bound), an e4m3 cache, whose f16 MMAs run on converted codes, above it.
    flops = 2.0 * (576 + 512) * n_h * float(np.sum(case.lens))
    tensor_peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))   # f16 dense = bf16 dense
    tensor_bound = flops / cache_bytes > tensor_peak * 1e12 / (hbm_peak * 1e9)
    achieved_tflops = flops / (decode_ms / 1e3) / 1e12
    traffic = None
    prof = os.path.join(ROOT, "profiles", "decode_traffic.json")
    if os.path.exists(prof):
        with open(prof) as f:
            pj = json.load(f)
        rec = pj.get(w.name) if isinstance(pj, dict) else None
        if rec and rec.get("kernel_source_hash") == _kernel_hash():
            traffic = rec.get("dram_bytes_per_launch")
    roof_common = {"kernel": "mla_decode_fwd", "traffic": traffic, "algorithmic_bytes_per_launch": cache_bytes,
                   "algorithmic_flops_per_launch": flops}
    if tensor_bound:
        roofline = {"bound": "tensor", "achieved": round(achieved_tflops, 1), "peak": tensor_peak,
                    "unit": "TFLOP/s", "frac": round(achieved_tflops / tensor_peak, 4),
                    "peak_source": f"{peaks_src} bf16_tflops (the f16 dense rate is the same)",
                    "hbm_achieved_gbs": round(achieved, 1), "hbm_frac": round(achieved / hbm_peak, 4),
                    **roof_common}
    else:
        roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                    "frac": round(achieved / hbm_peak, 4), "peak_source": f"{peaks_src} hbm_gbs",
                    "tensor_achieved_tflops": round(achieved_tflops, 1),
                    "tensor_frac": round(achieved_tflops / tensor_peak, 4), **roof_common}
    res = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "ms_per_step": round(step_ms_max, 5),
        "dtype": mla.compute_dtype(n_h, w.kv),
        "config": workload_config(w, case.lens, S),
        "decode_tokens_per_s": round(B * dist.world / (step_ms_max / 1e3), 1),
        "decode_tokens_per_s_note": "sequences decoded per second, one MLA layer",
        "hbm_roofline_frac_step": round((cache_bytes + weight_bytes + io_bytes) / (step_ms / 1e3) / 1e9 / hbm_peak,
                                        4),
        "kernel_ms": {"absorb_q": round(float(kern_ms[0]), 5), "decode_fwd": round(decode_ms, 5),
                      "combine_up_v": round(float(kern_ms[2]), 5)},
        "decode_kernel": mla.decode_kernel(w.kv, n_h),
        "roofline": roofline,
        "e2e": {"value": round(total_cache / (eager_mean / 1e3) / 1e9, 2), "unit": "GB/s",
                "ms_per_step": round(eager_mean, 5), "host_ms_per_step": round(float(np.mean(eager_host_ms)), 4),
                "steps": len(eager_ms), "ms_median": round(float(np.median(eager_ms)), 5),
                "ms_max": round(float(np.max(eager_ms)), 5),
                "device_step_ratio": round(eager_mean / step_ms, 2),
                "h2d_bytes_per_step": int(h_q.numel() * 2 + h_pos.numel() * 4 + h_len.numel() * 4),
                "d2h_bytes_per_step": int(h_o.numel() * 4),
                "path": "mla.decode_step (three Python calls over the C ABI) with H2D of q, pos and seq_lens from "
                        "pinned host buffers and D2H of o into a pinned buffer, every step",
                "same_o_as_graph": same_o,
                "graph": {"value": round(total_cache / (e2e_mean / 1e3) / 1e9, 2), "unit": "GB/s",
                          "ms_per_step": round(e2e_mean, 5),
                          "host_ms_per_step": round(float(np.mean(host_ms)), 4),
                          "ms_median": round(float(np.median(e2e_ms)), 5),
                          "path": "mla.DecodeStepGraph.replay: the same copies around the three calls captured "
                                  "once as a CUDA graph"}},
        "cache_append": {"ms": round(app_mean, 5), "tokens": B, "d_model": d_model,
                         "algorithmic_bytes": int(app_bytes),
                         "achieved_gbs": round(app_bytes / (app_mean / 1e3) / 1e9, 1),
                         "frac": round(app_bytes / (app_mean / 1e3) / 1e9 / hbm_peak, 4),
                         "bound": "hbm", "peak_gbs": hbm_peak,
                         "note": "W_DKV and W_KR read once, the new tokens' hidden states and rows; "
                                 "CUDA events around one call, L2 flushed before each"},
        "clocks": {**clocks, "window": f"{args.soak:.1f} s soak + the timed steps"},
    }
    del case, cache, bufs, e2e_bufs, flush, drain, graph, graph_parts
    gc.collect()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    if not args.no_cpu_baseline and dist.world == 1 and dist.rank == 0:
        res["cpu_baseline"] = cpu_baseline(W.WORKLOADS[name], args.cpu_budget if headline else args.cpu_budget / 2)
    return res


def run_ours(args, dist: Dist) -> dict | None:
    import torch

    torch.cuda.set_device(dist.local_rank)
    names = [HEADLINE] + [n for n in W.WORKLOAD_ORDER if n != HEADLINE] if args.workload == "all" else [args.workload]
    recs = {n: measure_ours(n, args, dist, headline=(i == 0)) for i, n in enumerate(names)}
    if dist.rank != 0:
        return None
    head = recs[names[0]]
    res = {
        "metric": METRIC, "value": head["value"], "unit": "GB/s", "n_gpus": dist.world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": head["dtype"],
        "data": "synthetic (seeded N(0,1) bf16 cache and queries, N(0,1/512) weights; no checkpoint)",
        **{k: v for k, v in head.items() if k not in ("metric", "value", "unit", "ms_per_step", "dtype")},
        "gpu_launches": N_CALLS * args.steps,
        "timing": "CUDA-graph replay of the step between two device-side events; kernel_ms from a second graph "
                  "with events between the three calls (no launch overlap there, so they sum to more than the step)",
        "step": "absorb_q + decode_fwd + combine_up_v (log-sum-exp merge of the splits and W_UV in one kernel), "
                "one MLA layer",
    }
    if len(names) > 1:
        res["workloads"] = {n: recs[n] for n in names[1:]}
        res["gpu_launches_all_workloads"] = N_CALLS * args.steps * len(names)
    return res


def _kernel_hash() -> str:
    import hashlib

    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mla_latent_kv_69_b300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.startswith("decode") or f.endswith((".cuh", ".h")):
            h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


# ------------------------------- reference arm -------------------------------------
def run_reference(args, dist: Dist) -> dict | None:
    """The oracle as it stands, on the host cores, rank 0 only: each step is one pass of
    the headline workload's fixed oracle sample."""
    if dist.rank != 0:
        return None
    name = HEADLINE if args.workload == "all" else args.workload
    w = W.WORKLOADS[name]
    lens = W.seq_lens(w)
    smp = OracleSample(w)
    for _ in range(args.warmup):
        smp.run()
    secs = [smp.run() for _ in range(args.steps)]
    mean_s = float(np.mean(secs))
    value = smp.bytes / mean_s / 1e9
    return {
        "metric": METRIC, "impl": "reference", "value": round(value, 5), "unit": "GB/s", "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * mean_s, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) bf16 cache and queries, N(0,1/512) weights; no checkpoint)",
        "config": workload_config(w, lens, num_splits_for(w, lens)),
        "cpu_baseline": {"value": round(value, 5), "unit": "GB/s", "cores": _blas_threads(), "kind": "oracle",
                         "sample": oracle_sample_desc(w), "seconds": round(float(np.sum(secs)), 2)},
        "e2e": {"value": round(value, 5), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "step": "one pass of the fp64 oracle (explicit form) over the fixed sample; GB/s counts the sample's "
                "cache bytes scaled by the heads evaluated",
    }


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="all", choices=["all"] + list(W.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--soak", type=float, default=1.5, help="seconds of untimed load before the timed steps "
                    "(nvidia-smi clock samples span soak + timed region)")
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="oracle seconds for the headline cpu_baseline "
                    "(half of it for each other workload)")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        print("note: fewer than 3 warm-up steps", file=sys.stderr)
    dist = Dist(backend="gloo" if args.impl == "reference" else None)
    try:
        res = run_reference(args, dist) if args.impl == "reference" else run_ours(args, dist)
    finally:
        dist.close()
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
