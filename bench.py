#!/usr/bin/env python3
"""Benchmark of one MLA decode step (absorb_q → decode_fwd → combine → up_v) on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-cpu-baseline]

Prints ONE JSON line on rank 0. A "step" is one pass of the whole hot path over one
batch of synthetic inputs; the latent cache and the weights are resident in HBM
(they are the layer's state) and L2 is flushed (256 MiB write) before every timed
step (the write is followed by a 256 MiB read so that no dirty lines of the flush
are written back inside the timed kernels). `value` = latent-cache bytes per step ÷ step time (GB/s), summed over
ranks; each rank decodes its own batch (weak scaling, no data-path collective).
`--impl reference` times the fp64 CPU oracle on a bounded sample instead.
"""
from __future__ import annotations

import argparse
import json
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
DEFAULT_WORKLOAD = "v2_b32_l4096"
L2_FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


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


def cpu_oracle_sample(w: W.Workload, budget_s: float = 12.0, min_seqs: int = 1):
    """Time the fp64 oracle (as it stands) on whole sequences of the workload until
    the time budget is spent. Returns (GB/s of cache processed, seconds, sample text)."""
    from oracle import fp8_e4m3, mla_oracle

    lens = W.seq_lens(w)
    qb, wk, wv = W.gen_q(w), W.bf16_bits_to_f32(W.gen_w_uk(w)), W.bf16_bits_to_f32(W.gen_w_uv(w))
    order = list(np.argsort(lens, kind="stable"))          # cheapest sequences first keeps the bound
    spent, done_bytes, seqs = 0.0, 0, []
    per_tok = W.D_ROW * 2 if w.kv == "bf16" else W.D_ROW + 4
    for b in order:
        if spent >= budget_s and len(seqs) >= min_seqs:
            break
        L = int(lens[b])
        rows = W.bf16_bits_to_f32(W.gen_rows(w, int(b), L))
        if w.kv == "fp8":
            codes, scales = fp8_e4m3.quantize_rows(rows)
            rows = fp8_e4m3.dequantize_rows(codes, scales)
        q = W.bf16_bits_to_f32(qb[b])
        t0 = time.perf_counter()
        mla_oracle.attend_explicit(q, rows[:, :512], rows[:, 512:], wk, wv, pos_q=max(L - 1, 0))
        spent += time.perf_counter() - t0
        done_bytes += L * per_tok
        seqs.append(int(b))
    gbs = done_bytes / spent / 1e9 if spent > 0 else 0.0
    return gbs, spent, f"{len(seqs)} whole sequence(s) {seqs[:4]}{'...' if len(seqs) > 4 else ''} of {w.name}, all {w.n_h} heads, fp64 explicit form"


# ------------------------------- our arm -------------------------------------------
def run_ours(args, dist: Dist) -> dict | None:
    import torch

    import mla_latent_kv_69_b300 as mla

    torch.cuda.set_device(dist.local_rank)
    dev = torch.device("cuda", dist.local_rank)
    w = rank_workload(W.WORKLOADS[args.workload], dist.rank)
    case = W.DeviceInputs(w, dev)
    if w.kv == "fp8":                     # the library's own cache writer makes the e4m3 cache
        codes, scales = mla.quantize_fp8(case.source)
        case.cache = mla.Cache(codes, scales, case.block_table)
        del case.source
    else:
        case.cache = mla.Cache(case.source, None, case.block_table)
    B, n_h = case.B, case.n_h
    S = mla.num_splits(B, case.max_len, n_h)
    bufs = dict(
        q_lat=torch.empty(B, n_h, 576, dtype=torch.bfloat16, device=dev),
        o_part=torch.empty(B, S, n_h, 512, dtype=torch.float32, device=dev),
        lse_part=torch.empty(B, S, n_h, dtype=torch.float32, device=dev),
        o_lat=torch.empty(B, n_h, 512, dtype=torch.float32, device=dev),
        lse=torch.empty(B, n_h, dtype=torch.float32, device=dev),
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

    def step():
        mla.absorb_q(case.q, case.w_uk, case.pos, q_lat=bufs["q_lat"])
        mla.decode_fwd(bufs["q_lat"], case.cache, case.seq_lens, case.max_len, n_splits=S,
                       o_part=bufs["o_part"], lse_part=bufs["lse_part"])
        mla.combine(bufs["o_part"], bufs["lse_part"], o_lat=bufs["o_lat"], lse=bufs["lse"])
        mla.up_v(bufs["o_lat"], case.w_uv, o=bufs["o"])

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # The timed step is one CUDA-graph replay: an L2 flush (outside the timed interval),
    # then the four library calls between two device-side events. Consecutive kernels of
    # the step overlap their launch and prologue with the previous kernel's tail
    # (programmatic dependent launch), so no event may sit between them in this graph;
    # a second graph with events between the calls gives the per-kernel breakdown.
    ev_step = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(2)]
    ev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(5)]
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
            mla.absorb_q(case.q, case.w_uk, case.pos, q_lat=bufs["q_lat"])
            ev[1].record()
            mla.decode_fwd(bufs["q_lat"], case.cache, case.seq_lens, case.max_len, n_splits=S,
                           o_part=bufs["o_part"], lse_part=bufs["lse_part"])
            ev[2].record()
            mla.combine(bufs["o_part"], bufs["lse_part"], o_lat=bufs["o_lat"], lse=bufs["lse"])
            ev[3].record()
            mla.up_v(bufs["o_lat"], case.w_uv, o=bufs["o"])
            ev[4].record()
    torch.cuda.current_stream().wait_stream(cap)
    for _ in range(max(args.warmup, 3)):
        graph.replay()
        graph_parts.replay()
    torch.cuda.synchronize()

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
    for k in range(K):
        graph.replay()
        torch.cuda.synchronize()
        steps.append(ev_step[0].elapsed_time(ev_step[1]))   # ms
    torch.cuda.synchronize()
    dist.barrier()
    clocks = sampler.stop()
    per = []
    for k in range(K):
        graph_parts.replay()
        torch.cuda.synchronize()
        per.append([ev[i].elapsed_time(ev[i + 1]) for i in range(4)])   # ms
    per = np.array(per)
    step_ms = float(np.mean(steps))
    kern_ms = per.mean(axis=0)
    step_ms_max = dist.max(step_ms, dev)

    # e2e through the public API with host buffers: per step, H2D of the new queries
    # (+ positions, lengths) from pinned memory and D2H of the outputs o.
    h_q = case.q.cpu().pin_memory()
    h_pos = case.pos.cpu().pin_memory()
    h_len = case.seq_lens.cpu().pin_memory()
    h_o = torch.empty(B, n_h, 128, dtype=torch.float32).pin_memory()
    d_q, d_pos, d_len = torch.empty_like(case.q), torch.empty_like(case.pos), torch.empty_like(case.seq_lens)

    def e2e_step():
        d_q.copy_(h_q, non_blocking=True)
        d_pos.copy_(h_pos, non_blocking=True)
        d_len.copy_(h_len, non_blocking=True)
        mla.absorb_q(d_q, case.w_uk, d_pos, q_lat=bufs["q_lat"])
        mla.decode_fwd(bufs["q_lat"], case.cache, d_len, case.max_len, n_splits=S,
                       o_part=bufs["o_part"], lse_part=bufs["lse_part"])
        mla.combine(bufs["o_part"], bufs["lse_part"], o_lat=bufs["o_lat"], lse=bufs["lse"])
        mla.up_v(bufs["o_lat"], case.w_uv, o=bufs["o"])
        h_o.copy_(bufs["o"], non_blocking=True)

    for _ in range(max(args.warmup, 1)):
        e2e_step()
    torch.cuda.synchronize()
    e2e_ms = []
    for _ in range(K):
        flush_l2()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        e2e_step()
        b.record(stream)
        b.synchronize()
        e2e_ms.append(a.elapsed_time(b))
    e2e_mean = dist.max(float(np.mean(e2e_ms)), dev)

    peaks, peaks_src = load_peaks()
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    total_cache = dist.sum(cache_bytes, dev)
    value = total_cache / (step_ms_max / 1e3) / 1e9
    decode_ms = float(kern_ms[1])
    achieved = cache_bytes / (decode_ms / 1e3) / 1e9
    # Which pipe bounds the decode kernel: QK^T over 576 and PV over 512 columns per
    # (token, head) against the cache bytes; a bf16 cache sits just under the measured
    # ridge (HBM-bound), an e4m3 cache, whose f16 MMAs run on dequantised codes, above it.
    flops = 2.0 * (576 + 512) * n_h * float(np.sum(case.lens))
    tensor_peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))   # f16 dense = bf16 dense
    tensor_bound = flops / cache_bytes > tensor_peak * 1e12 / (hbm_peak * 1e9)
    achieved_tflops = flops / (decode_ms / 1e3) / 1e12
    traffic = None
    prof = os.path.join(ROOT, "profiles", "decode_traffic.json")
    if os.path.exists(prof):
        with open(prof) as f:
            pj = json.load(f)
        if pj.get("workload") == w.name and pj.get("kernel_source_hash") == _kernel_hash():
            traffic = pj.get("dram_bytes_per_launch")
    if dist.rank != 0:
        return None
    res = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": dist.world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms_max, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": _compute_dtype(w, n_h),
        "data": "synthetic (seeded N(0,1) bf16 cache and queries, N(0,1/512) weights; no checkpoint)",
        "config": {
            "workload": w.name, "n_h": n_h, "batch_per_gpu": B, "ctx": int(case.max_len), "kv": w.kv,
            "layout": "paged-64" if w.paged else "contiguous", "n_splits": S,
            "l2": "flushed before every timed step (256 MiB write, then a 256 MiB read that drains the written lines; both outside the timed intervals)",
            "timing": "CUDA-graph replay of the step between two device-side events; kernel_ms from a second graph with events between the four calls",
            "decode_kernel": mla.decode_kernel(w.kv, n_h),
            "step": "absorb_q + decode_fwd + combine + up_v, one MLA layer",
        },
        "decode_tokens_per_s": round(B * dist.world / (step_ms_max / 1e3), 1),
        "hbm_roofline_frac_step": round((cache_bytes + weight_bytes + io_bytes) / (step_ms / 1e3) / 1e9 / hbm_peak, 4),
        "kernel_ms": {"absorb_q": round(float(kern_ms[0]), 5), "decode_fwd": round(decode_ms, 5),
                      "combine": round(float(kern_ms[2]), 5), "up_v": round(float(kern_ms[3]), 5)},
        "roofline": ({"kernel": "mla_decode_fwd", "bound": "tensor", "achieved": round(achieved_tflops, 1),
                      "peak": tensor_peak, "unit": "TFLOP/s", "frac": round(achieved_tflops / tensor_peak, 4),
                      "traffic": traffic, "peak_source": f"{peaks_src} bf16_tflops (the f16 dense rate is the same)",
                      "algorithmic_flops_per_launch": flops, "algorithmic_bytes_per_launch": cache_bytes,
                      "hbm_achieved_gbs": round(achieved, 1), "hbm_frac": round(achieved / hbm_peak, 4)}
                     if tensor_bound else
                     {"kernel": "mla_decode_fwd", "bound": "hbm", "achieved": round(achieved, 1),
                      "peak": hbm_peak, "unit": "GB/s", "frac": round(achieved / hbm_peak, 4),
                      "traffic": traffic, "peak_source": f"{peaks_src} hbm_gbs",
                      "algorithmic_bytes_per_launch": cache_bytes, "algorithmic_flops_per_launch": flops,
                      "tensor_achieved_tflops": round(achieved_tflops, 1),
                      "tensor_frac": round(achieved_tflops / tensor_peak, 4)}),
        "cache_gbs_decode_combine": round(cache_bytes / ((decode_ms + float(kern_ms[2])) / 1e3) / 1e9, 1),
        "e2e": {"value": round(total_cache / (e2e_mean / 1e3) / 1e9, 2), "unit": "GB/s",
                "ms_per_step": round(e2e_mean, 5),
                "h2d_bytes_per_step": int(h_q.numel() * 2 + h_pos.numel() * 4 + h_len.numel() * 4),
                "d2h_bytes_per_step": int(h_o.numel() * 4)},
        "gpu_launches": 4 * K,
        "kernel_ms_note": "per-call intervals from a graph with events between the calls (no launch overlap there); their sum exceeds ms_per_step",
        "clocks": {**clocks, "window": f"{args.soak:.1f} s soak + the timed steps"},
    }
    if not args.no_cpu_baseline and dist.world == 1:
        gbs, spent, sample = cpu_oracle_sample(w, budget_s=args.cpu_budget)
        res["cpu_baseline"] = {"value": round(gbs, 4), "unit": "GB/s", "cores": _blas_threads(),
                               "kind": "oracle", "sample": sample, "seconds": round(spent, 2)}
    return res


def _compute_dtype(w, n_h) -> str:
    try:
        import mla_latent_kv_69_b300 as mla

        return mla.compute_dtype(n_h, w.kv)
    except AttributeError:
        return "f32"


def _kernel_hash() -> str:
    import hashlib

    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mla_latent_kv_69_b300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.startswith("decode") or f.endswith((".cuh", ".h")):
            h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def _blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info

        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return host_cores()


# ------------------------------- reference arm -------------------------------------
def run_reference(args, dist: Dist) -> dict | None:
    """The oracle as it stands, on the host cores, rank 0 only."""
    if dist.rank != 0:
        return None
    w = W.WORKLOADS[args.workload]
    per_step_budget = max(1.0, args.ref_budget / max(args.steps + args.warmup, 1))
    for _ in range(args.warmup):
        cpu_oracle_sample(w, budget_s=per_step_budget)
    vals, secs, sample = [], [], ""
    for _ in range(args.steps):
        gbs, spent, sample = cpu_oracle_sample(w, budget_s=per_step_budget)
        vals.append(gbs)
        secs.append(spent)
    value = float(np.mean(vals))
    return {
        "metric": METRIC, "impl": "reference", "value": round(value, 4), "unit": "GB/s", "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * float(np.mean(secs)), 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) bf16 cache and queries, N(0,1/512) weights; no checkpoint)",
        "config": {"workload": w.name, "n_h": w.n_h, "batch_per_gpu": w.batch, "kv": w.kv,
                   "layout": "paged-64" if w.paged else "contiguous",
                   "step": "fp64 oracle, explicit form, on a bounded sample of whole sequences"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": _blas_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=list(W.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--soak", type=float, default=1.5, help="seconds of untimed load before the timed steps "
                    "(nvidia-smi clock samples span soak + timed region)")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--ref-budget", type=float, default=60.0, help="total oracle seconds for --impl reference")
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
