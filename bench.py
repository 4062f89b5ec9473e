#!/usr/bin/env python
"""Throughput of libq4mm on GB300: decode weight-GB/s and prefill TFLOP/s, as fractions of
the measured HBM and dense-bf16 rooflines.

Headline workload (one "step"): the INT4 group-32 affine decode GEMV at every shape of the
decode configuration -- M in {1, 4, 16} x (K, N) in {(4096, 14336), (14336, 4096),
(4096, 4096)} -- one q4_gemv call per shape, each on a weight replica that is not in L2.
value = algorithmic bytes of a step / device time of a step (GB/s).  The prefill GEMM,
LUT4 and Q4_0 MoE paths are timed in the same run and reported beside it.

Timing: inputs resident in HBM; steps are CUDA-graph replays timed with CUDA events on the
launching stream; weights rotate through a ring of replicas whose total is >= 4x L2, so
every call reads its weights from HBM.  nvidia-smi clocks are sampled during the timed
region.  `--impl reference` times the CPU oracle on the host cores instead (a deliberately
slow baseline on a bounded sample of the same workload).

Multi-GPU: the path does not shard (replicas only); under torchrun every rank runs the same
workload on its own GPU, and value = units of all ranks / max time over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "int4 qmm decode weight-GB/s & prefill TFLOP/s, % of GB300 roofline"
DECODE_KN = [(4096, 14336), (14336, 4096), (4096, 4096)]
DECODE_M = [1, 4, 16]
PREFILL_KN = [(4096, 14336), (14336, 4096), (4096, 6144)]
PREFILL_M = [512, 2048, 8192]
HEADLINE = (1, 4096, 14336)   # (M, K, N) of the kernel whose roofline is reported


def profiled_traffic(summary: str):
    """DRAM bytes per launch from a committed ncu summary, or None once the kernel source
    has changed since the capture (the summary records the source file's SHA-256)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", summary)
    try:
        fields = dict(line.split(": ", 1) for line in open(path).read().splitlines() if ": " in line
                      and line.split(": ", 1)[0] in ("traffic_bytes_per_launch", "source", "source_sha256"))
        src = os.path.join(ROOT, fields["source"])
        if hashlib.sha256(open(src, "rb").read()).hexdigest() != fields["source_sha256"]:
            return None
        return int(fields["traffic_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


def max_over_ranks(seconds: float, device) -> float:
    """The slowest rank's time: every rank's timed region ends when the last one's does."""
    import torch
    t = torch.tensor([seconds], device=device, dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_step: int, steps: int, world: int, seconds: float) -> float:
    """Whole-job GB/s: every rank (an independent replica) processes bytes_per_step each
    step, and the job takes the slowest rank's time."""
    return bytes_per_step * steps * world / seconds / 1e9


def decode_shapes():
    return [(M, K, N) for (K, N) in DECODE_KN for M in DECODE_M]


def int4_bytes(M, K, N):
    """Algorithmic bytes of one INT4 matmul call: codes + scales/biases + x + y."""
    return N * K // 2 + N * (K // 32) * 4 + 2 * M * K + 2 * M * N


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# ------------------------------------------------------------------------------------------
# clocks
# ------------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[str] = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, flag in zip(names, parts[5:9]):
                if flag.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": float(max(mx)) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------------------
# our arm
# ------------------------------------------------------------------------------------------
def under_profiler() -> bool:
    """Nsight Compute injects itself into the target (it sets the NV_NSIGHT_INJECTION_*
    variables); kernel nodes of CUDA graphs do not replay under it, so the same command
    then issues every launch eagerly (timings taken that way are never bench values)."""
    return any(k.startswith("NV_NSIGHT_INJECTION") for k in os.environ) or \
        bool(os.environ.get("CUDA_INJECTION64_PATH"))


class EagerGraph:
    """Stand-in for torch.cuda.CUDAGraph that re-issues the captured calls on replay()."""

    def __init__(self, fn):
        self.fn = fn

    def replay(self):
        self.fn()


def run_ours(args, rank, world, local_rank):
    import torch

    import weight_only_bit_int4_gb300 as q
    from weight_only_bit_int4_gb300 import synth

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2 ** 20))
    pk = peaks()

    def to_dev(a):
        a = np.ascontiguousarray(a)
        view = {np.dtype(np.uint16): np.int16, np.dtype(np.uint32): np.int32}.get(a.dtype, a.dtype)
        return torch.from_numpy(a.view(view)).to(dev)

    def ring_of(tensors, nbytes):
        """Replicas of `tensors` so that the ring holds >= 4x L2."""
        R = max(2, math.ceil(4 * l2 / nbytes))
        return [tensors] + [tuple(t.clone() for t in tensors) for _ in range(R - 1)]

    eager = under_profiler()

    def time_graph(build_calls, launches_per_replay, replays, warmup=3):
        """Capture build_calls() into a graph; return (seconds per replay)."""
        if eager:
            replays, warmup = 1, 1
            for _ in range(warmup):
                build_calls(0)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            build_calls(0)
            torch.cuda.synchronize()
            return (time.perf_counter() - t0) / replays
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            build_calls(0)       # eager warm-up outside capture (first-call set-up)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            build_calls(1)
        for _ in range(warmup):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(replays):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / 1e3 / replays

    # ---------------- decode workload ----------------
    rings = {}
    for i, (K, N) in enumerate(DECODE_KN):
        w, s, b = synth.int4_weights(1000 + i, N, K)
        rings[(K, N)] = ring_of((to_dev(w), to_dev(s), to_dev(b)), N * K * 9 // 16)
    xs, ys = {}, {}
    for j, (M, K, N) in enumerate(decode_shapes()):
        xs[(M, K, N)] = to_dev(synth.activations_bf16(1100 + j, M, K))
        ys[(M, K, N)] = torch.empty((M, N), dtype=torch.int16, device=dev)
    P = max(len(r) for r in rings.values())
    step_bytes = sum(int4_bytes(*shp) for shp in decode_shapes())

    # eager warm-up of every shape (first-call attribute set-up happens outside capture)
    for shp in decode_shapes():
        M, K, N = shp
        q.q4_gemv(xs[shp], *rings[(K, N)][0], ys[shp])
    torch.cuda.synchronize()

    # Decode weights are static, so each call is launched to overlap the previous one's tail
    # (Q4MM_GEMV_STATIC_WEIGHTS); the per-shape table also times plain launches.
    def step_calls(p):
        for shp in decode_shapes():
            M, K, N = shp
            r = rings[(K, N)]
            q.q4_gemv(xs[shp], *r[p % len(r)], ys[shp], static_weights=True)

    graphs = []
    if eager:
        graphs = [EagerGraph(lambda p=p: step_calls(p)) for p in range(P)]
    else:
        cap = torch.cuda.Stream()
        cap.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(cap):
            for p in range(P):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=cap):
                    step_calls(p)
                graphs.append(g)
    torch.cuda.synchronize()
    launches_per_step = len(decode_shapes())

    for i in range(max(3, args.warmup)):
        graphs[i % P].replay()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(args.steps):
        graphs[i % P].replay()
    e1.record()
    torch.cuda.synchronize()
    elapsed = e0.elapsed_time(e1) / 1e3
    if world > 1:
        torch.distributed.barrier()
        elapsed = max_over_ranks(elapsed, dev)
    # per-shape and headline-kernel timings (same run, same clock sampling)
    shape_rows = []
    headline = None
    for shp in decode_shapes():
        M, K, N = shp
        r = rings[(K, N)]
        L = 2 * len(r)
        def calls(_, shp=shp, r=r, L=L, sw=True):
            for l in range(L):
                q.q4_gemv(xs[shp], *r[l % len(r)], ys[shp], static_weights=sw)
        t = time_graph(calls, L, replays=max(5, args.steps // 10)) / L
        t_plain = time_graph(lambda p_: calls(p_, sw=False), L, replays=max(5, args.steps // 10)) / L
        by = int4_bytes(M, K, N)
        row = {"M": M, "K": K, "N": N, "us": round(t * 1e6, 3), "GB_s": round(by / t / 1e9, 1),
               "frac_hbm": round(by / t / 1e9 / pk["hbm_gbs"], 3),
               "us_plain_launch": round(t_plain * 1e6, 3)}
        shape_rows.append(row)
        if shp == HEADLINE:
            headline = (t, by)
    clocks = sampler.stop()

    value = job_throughput(step_bytes, args.steps, world, elapsed)
    out = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(elapsed / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "INT4 g32 affine decode GEMV, M in {1,4,16} x (K,N) in "
                               "{(4096,14336),(14336,4096),(4096,4096)}, one call per shape per step",
                   "l2": f"weights rotate through replicas totalling >= 4x L2 ({l2 >> 20} MiB)",
                   "timing": "CUDA-graph replays, CUDA events on the launching stream",
                   "launch": "q4_gemv_ex with Q4MM_GEMV_STATIC_WEIGHTS: each call streams its weights "
                             "while the previous call finishes; x and y wait for it",
                   "parallelism": f"replicas x{world}"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "decode_shapes": shape_rows,
    }
    t_h, by_h = headline
    # The decode kernel of each shape: the K-split group-column kernel at M <= 2, the TMA-fed
    # warp-specialised kernel at 3 <= M <= 16 (every bench shape has K % 256 == 0).
    def kernel_of(M):
        return "gemv_ks_kernel" if M <= 2 else "gemv_tma_kernel"
    by_kernel = {}
    for r in shape_rows:
        k = kernel_of(r["M"])
        r["kernel"] = k
        tb = by_kernel.setdefault(k, [0.0, 0, 0])
        tb[0] += r["us"] * 1e-6
        tb[1] += int4_bytes(r["M"], r["K"], r["N"])
        tb[2] += 1
    dom = max(by_kernel, key=lambda k: by_kernel[k][0])
    t_d, by_d, n_d = by_kernel[dom]
    share = t_d / sum(v[0] for v in by_kernel.values())
    out["roofline"] = {
        "bound": "hbm", "kernel": f"{dom} (q4_gemv_ex, static weights): the step's dominant kernel, "
                                  f"{n_d} of 9 launches, {share:.0%} of the summed per-shape time",
        "achieved": round(by_d / t_d / 1e9, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
        "frac": round(by_d / t_d / 1e9 / pk["hbm_gbs"], 3),
        "frac_vs_8TBs": round(by_d / t_d / 8e12, 3),
        "peak_source": pk["source"] + " (hbm_gbs, burst copy)",
        "traffic": profiled_traffic(f"{dom}_q4_gemv_M16_K14336_N4096.md"),
        "traffic_note": "ncu DRAM bytes (read + write) of one launch of the M=16, K=14336, N=4096 shape, "
                        "whose algorithmic bytes are 37224448",
        "algorithmic_bytes_per_launch": round(by_d / n_d),
        "step_frac": round(value / pk["hbm_gbs"], 3),
        "headline_shape": {"M": HEADLINE[0], "K": HEADLINE[1], "N": HEADLINE[2], "kernel": kernel_of(HEADLINE[0]),
                           "achieved": round(by_h / t_h / 1e9, 1), "frac": round(by_h / t_h / 1e9 / pk["hbm_gbs"], 3),
                           "traffic": profiled_traffic("gemv_ks_kernel_q4_gemv_M1_K4096_N14336.md"),
                           "algorithmic_bytes_per_launch": by_h},
        # per decode shape: [M, K, N, us, GB/s, fraction of the measured HBM peak]
        "shapes": [[r["M"], r["K"], r["N"], r["us"], r["GB_s"], r["frac_hbm"]] for r in shape_rows]}

    # ---------------- e2e through the public API with host buffers ----------------
    out["e2e"] = e2e_decode(args, q, synth, rings, dev)

    if not args.quick:
        out["prefill"] = bench_prefill(args, q, synth, to_dev, time_graph, dev, pk)
        out["lut4"] = bench_lut4(args, q, synth, to_dev, ring_of, time_graph, dev, pk)
        out["moe"] = bench_moe(args, q, synth, to_dev, ring_of, time_graph, dev, pk)
        out["dispatch"] = bench_dispatch(q, synth, to_dev, dev, calls=10 if eager else 3000)
        try:
            out["dequant"] = bench_dequant(q, synth, to_dev, ring_of, rings, time_graph, dev, pk)
        except Exception as e:   # an auxiliary section never costs the headline line
            out["dequant"] = {"error": f"{type(e).__name__}: {e}"[:300]}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        gpu_ms = {"0": small_case_ms(q, synth, to_dev, time_graph, dev), "1": elapsed / args.steps * 1e3}
        if not args.quick:
            gpu_ms["2"] = sum(r["us"] for r in out["prefill"]["shapes"]) / 1e3
            gpu_ms["3"] = sum(r["us"] for r in out["lut4"]["shapes"]) / 1e3
            gpu_ms["4"] = sum(r["us"] for r in out["moe"]["shapes"]) / 1e3
        out["cpu_baseline"] = cpu_baseline(gpu_ms, with_configs=not args.quick)
    # last, so that a tail of the printed line keeps it: per decode shape [M, K, N, us, frac]
    out["decode_summary"] = [[r["M"], r["K"], r["N"], r["us"], r["frac_hbm"]] for r in shape_rows]
    return out


def small_case_ms(q, synth, to_dev, time_graph, dev):
    """GPU ms per call of the small INT4 case (M=16, K=512, N=256) through q4_gemv."""
    import torch
    M, K, N = 16, 512, 256
    w, s, b = synth.int4_weights(1000, N, K)
    W = (to_dev(w), to_dev(s), to_dev(b))
    x = to_dev(synth.activations_bf16(1001, M, K))
    y = torch.empty((M, N), dtype=torch.int16, device=dev)
    L = 50
    return time_graph(lambda _: [q.q4_gemv(x, *W, y) for _ in range(L)], L, replays=5) / L * 1e3


def e2e_decode(args, q, synth, rings, dev):
    """The decode step end to end through the public API: every step copies all nine x
    from pinned host memory in one transfer, replays the nine dispatch records (q4_gemv_record,
    static weights, planned once before timing) in one q4_gemv_record_launch_n call, copies
    all nine y back in one transfer and waits for it."""
    import torch
    shapes = decode_shapes()
    xsz = [s[0] * s[1] for s in shapes]
    ysz = [s[0] * s[2] for s in shapes]
    xh = torch.empty(sum(xsz), dtype=torch.int16).pin_memory()
    yh = torch.empty(sum(ysz), dtype=torch.int16).pin_memory()
    off = 0
    for j, (s, n) in enumerate(zip(shapes, xsz)):
        xh[off:off + n].copy_(torch.from_numpy(synth.activations_bf16(1100 + j, s[0], s[1]).view(np.int16).reshape(-1)))
        off += n
    xd = torch.empty(sum(xsz), dtype=torch.int16, device=dev)
    yd = torch.empty(sum(ysz), dtype=torch.int16, device=dev)
    xv, yv, ox, oy = [], [], 0, 0
    for s, nx, ny in zip(shapes, xsz, ysz):
        xv.append(xd[ox:ox + nx].view(s[0], s[1]))
        yv.append(yd[oy:oy + ny].view(s[0], s[2]))
        ox += nx
        oy += ny
    recs = [q.q4_gemv_record(M, N, K, static_weights=True) for (M, K, N) in shapes]
    steps = max(3, min(args.steps, 50))
    # One prepared batch per phase of the weight-replica rotation (a server's buffers would
    # be fixed, so its batch would be prepared once).
    period = 1
    for (M, K, N) in shapes:
        period = math.lcm(period, len(rings[(K, N)]))
    batches = []
    for i in range(period):
        wsb = [rings[(K, N)][i % len(rings[(K, N)])] for (M, K, N) in shapes]
        batches.append(q.RecordBatch(recs, xv, [t[0] for t in wsb], [t[1] for t in wsb], [t[2] for t in wsb], yv))

    def one(i):
        xd.copy_(xh, non_blocking=True)
        batches[i % period].launch()
        yh.copy_(yd, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    for i in range(3):
        one(i)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(steps):
        one(i)
    t = (time.perf_counter() - t0) / steps
    by = sum(int4_bytes(*s) for s in shapes)
    for r in recs:
        r.close()
    return {"value": round(by / t / 1e9, 1), "unit": "GB/s",
            "h2d_bytes_per_step": 2 * sum(xsz),
            "d2h_bytes_per_step": 2 * sum(ysz),
            "ms_per_step": round(t * 1e3, 3),
            "note": "per step: one pinned H2D copy of the nine x, the nine dispatch records replayed "
                    "in one q4_gemv_record_launch_n call (a prepared RecordBatch, static weights), one "
                    "D2H copy of the nine y, host wait; weights resident"}


def bench_prefill(args, q, synth, to_dev, time_graph, dev, pk):
    import torch
    rows = []
    gen = torch.Generator(device=dev)
    for i, (K, N) in enumerate(PREFILL_KN):
        w, s, b = synth.int4_weights(2000 + i, N, K)
        W = (to_dev(w), to_dev(s), to_dev(b))
        gen.manual_seed(2100 + i)
        xmax = torch.randn((max(PREFILL_M), K), generator=gen, device=dev, dtype=torch.float32)
        out_cols = torch.randperm(K, generator=gen, device=dev)[: max(1, round(0.01 * K))]
        xmax[:, out_cols] *= 20.0
        xmax = xmax.to(torch.bfloat16).view(torch.int16)
        for M in PREFILL_M:
            x = xmax[:M]
            y = torch.empty((M, N), dtype=torch.int16, device=dev)
            flops = 2.0 * M * N * K
            L = 2 if M == 8192 else 4
            t = time_graph(lambda _: [q.q4_gemm(x, *W, y) for _ in range(L)], L,
                           replays=3 if M == 8192 else 5) / L
            tf = flops / t / 1e12
            rows.append({"M": M, "K": K, "N": N, "us": round(t * 1e6, 2), "TFLOP_s": round(tf, 1),
                         "frac_bf16_burst": round(tf / pk["bf16_tflops"], 3),
                         "tokens_s": round(M / t, 0)})
        del xmax
        torch.cuda.empty_cache()
    tot_f = sum(2.0 * r["M"] * r["K"] * r["N"] for r in rows)
    tot_t = sum(r["us"] for r in rows) / 1e6
    return {"kernel": "qgemm_tma_kernel (q4_gemm: tcgen05, TMA-fed; every bench shape has K % 256 == 0)", "shapes": rows,
            "aggregate_TFLOP_s": round(tot_f / tot_t / 1e12, 1),
            "aggregate_frac_bf16_burst": round(tot_f / tot_t / 1e12 / pk["bf16_tflops"], 3),
            "x": "bf16 N(0,1), 1% columns x20, seeded torch generator on device"}


def bench_dispatch(q, synth, to_dev, dev, calls: int = 3000):
    """Host time per call on the smallest decode shape (M=16, K=512, N=256, whose kernel is
    shorter than its launch): the direct entry point, which plans every call, against a
    dispatch record planned once.  Python -> ctypes -> C ABI both ways; the calls are
    enqueued without synchronising, and the device is drained before and after."""
    import torch
    M, K, N = 16, 512, 256
    w, s, b = synth.int4_weights(1000, N, K)
    W = (to_dev(w), to_dev(s), to_dev(b))
    x = to_dev(synth.activations_bf16(1001, M, K))
    y = torch.empty((M, N), dtype=torch.int16, device=dev)
    rec = q.q4_gemv_record(M, N, K)
    res = {"shape": {"M": M, "K": K, "N": N}, "calls": calls}
    for name, fn in (("direct_us", lambda: q.q4_gemv(x, *W, y)), ("record_us", lambda: rec.gemv(x, *W, y))):
        for _ in range(min(50, calls)):
            fn()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(calls):
            fn()
        res[name] = round((time.perf_counter() - t0) / calls * 1e6, 2)
        torch.cuda.synchronize()
    rec.close()
    return res


def bench_lut4(args, q, synth, to_dev, ring_of, time_graph, dev, pk):
    import torch
    N = K = 4096
    packed, scales, book = synth.lut4_weights(3000, N, K, 64)
    ring = ring_of((to_dev(packed), to_dev(scales)), packed.nbytes + scales.nbytes)
    rows = []
    for M in (1, 512):
        x = to_dev(synth.activations_bf16(3100 + M, M, K))
        y = torch.empty((M, N), dtype=torch.int16, device=dev)
        L = 2 * len(ring)
        # Static weights (lut4_matmul_ex, Q4MM_GEMV_STATIC_WEIGHTS) as in the decode step; the
        # flag only changes the decode-kernel (M <= 16) launches.
        t = time_graph(lambda _: [q.lut4_matmul(x, *ring[l % len(ring)], book, y, N, K, 64, 1, static_weights=True)
                                  for l in range(L)], L, replays=10) / L
        by = packed.nbytes + scales.nbytes + 64 + 2 * M * K + 2 * M * N
        fl = 2.0 * M * N * K
        row = {"M": M, "K": K, "N": N, "us": round(t * 1e6, 3), "GB_s": round(by / t / 1e9, 1),
               "frac_hbm": round(by / t / 1e9 / pk["hbm_gbs"], 3),
               "TFLOP_s": round(fl / t / 1e12, 2),
               "frac_bf16_burst": round(fl / t / 1e12 / pk["bf16_tflops"], 3)}
        if M <= 16:
            tp = time_graph(lambda _: [q.lut4_matmul(x, *ring[l % len(ring)], book, y, N, K, 64, 1)
                                       for l in range(L)], L, replays=10) / L
            row["us_plain_launch"] = round(tp * 1e6, 3)
            # the rounded-weight variants (Q4MM_LUT4_ROUND_F16 / _BF16), same launches; at
            # M = 512 bf16 is the same GEMM and f16 the CUDA-core row kernel (about 2 ms a call)
            for r in ("f16", "bf16"):
                tr = time_graph(lambda _: [q.lut4_matmul(x, *ring[l % len(ring)], book, y, N, K, 64, 1,
                                                         static_weights=True, rounding=r)
                                           for l in range(L)], L, replays=10) / L
                row[f"us_round_{r}"] = round(tr * 1e6, 3)
        rows.append(row)
    return {"shapes": rows}


def bench_dequant(q, synth, to_dev, ring_of, rings, time_graph, dev, pk):
    """Standalone dequants to a dense bf16 matrix: INT4 (N = 14336, K = 4096) and LUT4
    (K = N = 4096, block 64).  HBM-bound: codes and scales (and biases) are read once and the
    dense matrix is written.  16 calls per graph walk the weight replicas; the outputs rotate
    through buffers whose total exceeds L2, so the writes reach DRAM."""
    import torch
    rows = []
    K, N = 4096, 14336
    r = rings[(K, N)]
    outs = [torch.empty((N, K), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    L = 16
    t = time_graph(lambda _: [q.q4_dequant(*r[l % len(r)], outs[l % 2]) for l in range(L)], L, replays=5) / L
    by = N * K // 2 + N * (K // 32) * 4 + N * K * 2   # codes, bf16 scales + biases, bf16 out
    rows.append({"op": "q4_dequant", "N": N, "K": K, "out": "bf16", "us": round(t * 1e6, 3),
                 "GB_s": round(by / t / 1e9, 1), "frac_hbm": round(by / t / 1e9 / pk["hbm_gbs"], 3)})
    Kl = Nl = 4096
    packed, scales, book = synth.lut4_weights(3000, Nl, Kl, 64)
    lr = ring_of((to_dev(packed), to_dev(scales)), packed.nbytes + scales.nbytes)
    louts = [torch.empty((Nl, Kl), dtype=torch.bfloat16, device=dev) for _ in range(6)]
    t = time_graph(lambda _: [q.lut4_dequant(*lr[l % len(lr)], book, Nl, Kl, 64, louts[l % 6]) for l in range(L)],
                   L, replays=5) / L
    by = packed.nbytes + scales.nbytes + 64 + Nl * Kl * 2
    rows.append({"op": "lut4_dequant", "N": Nl, "K": Kl, "block": 64, "out": "bf16", "us": round(t * 1e6, 3),
                 "GB_s": round(by / t / 1e9, 1), "frac_hbm": round(by / t / 1e9 / pk["hbm_gbs"], 3)})
    return {"shapes": rows}


def bench_moe(args, q, synth, to_dev, ring_of, time_graph, dev, pk):
    import torch
    E, top_k, N, K = 64, 8, 1408, 2048
    w, stride = synth.q4_0_experts(4000, E, N, K)
    ring = ring_of((to_dev(w),), w.nbytes)
    rows = []
    for n_tokens in (1, 512):
        ids = synth.routing_ids(4100 + n_tokens, n_tokens, top_k, E)
        x = to_dev(synth.activations_f32(4200 + n_tokens, n_tokens, K))
        idd = to_dev(ids.view(np.int32))
        out = torch.empty((n_tokens * top_k, N), dtype=torch.float32, device=dev)
        ws = torch.empty(q.q4_0_matmul_id_workspace_size(n_tokens, top_k, N, K, E), dtype=torch.uint8,
                         device=dev)
        touched = len(np.unique(ids))
        by = touched * N * (K // 32) * 18 + x.numel() * 4 + out.numel() * 4 + ids.nbytes
        fl = 2.0 * n_tokens * top_k * N * K
        for mode in ((1,) if n_tokens == 1 else (2,)):
            L = 2 * len(ring)
            t = time_graph(lambda _: [q.q4_0_matmul_id(x, ring[l % len(ring)][0], idd, out, top_k, N, K, E,
                                                       stride, mode=mode, workspace=ws)
                                      for l in range(L)], L, replays=5) / L
            rows.append({"n_tokens": n_tokens, "mode": {1: "mv", 2: "mm"}[mode], "us": round(t * 1e6, 2),
                         "GB_s": round(by / t / 1e9, 1), "frac_hbm": round(by / t / 1e9 / pk["hbm_gbs"], 3),
                         "TFLOP_s": round(fl / t / 1e12, 2)})
    # Fused SwiGLU routed mat-vec: the down projection of the same MoE (K = 1408 -> N = 2048),
    # one decode token; gate/up rows per routed row.
    Nd, Kd, n_tokens = K, N, 1
    wd, stride_d = synth.q4_0_experts(4300, E, Nd, Kd)
    ring_d = ring_of((to_dev(wd),), wd.nbytes)
    ids = synth.routing_ids(4400, n_tokens, top_k, E)
    idd = to_dev(ids.view(np.int32))
    gate = to_dev(synth.activations_f32(4500, n_tokens * top_k, Kd))
    up = to_dev(synth.activations_f32(4501, n_tokens * top_k, Kd))
    out = torch.empty((n_tokens * top_k, Nd), dtype=torch.float32, device=dev)
    by = len(np.unique(ids)) * Nd * (Kd // 32) * 18 + 2 * gate.numel() * 4 + out.numel() * 4 + ids.nbytes
    L = 2 * len(ring_d)
    t = time_graph(lambda _: [q.q4_0_matmul_id_swiglu(gate, up, ring_d[l % len(ring_d)][0], idd, out, top_k,
                                                      Nd, Kd, E, stride_d) for l in range(L)], L, replays=5) / L
    swiglu = {"n_tokens": n_tokens, "N": Nd, "K": Kd, "us": round(t * 1e6, 2), "GB_s": round(by / t / 1e9, 1),
              "frac_hbm": round(by / t / 1e9 / pk["hbm_gbs"], 3)}
    # GGML Q8_0 routed matmul on the same MoE shape (34-byte blocks): mat-vec at one token
    # (tensor cores, two nibble planes), mat-mat (route, scale, gather, tcgen05) at 512 tokens.
    w8, stride8 = synth.q8_0_experts(4700, E, N, K)
    ring8 = ring_of((to_dev(w8),), w8.nbytes)
    q8 = []
    for n_tokens, mode in ((1, 1), (512, 2)):
        ids = synth.routing_ids(4100 + n_tokens, n_tokens, top_k, E)
        x = to_dev(synth.activations_f32(4200 + n_tokens, n_tokens, K))
        idd = to_dev(ids.view(np.int32))
        out = torch.empty((n_tokens * top_k, N), dtype=torch.float32, device=dev)
        ws = torch.empty(max(1, q.q8_0_matmul_id_workspace_size(n_tokens, top_k, N, K, E)), dtype=torch.uint8,
                         device=dev)
        by = len(np.unique(ids)) * N * (K // 32) * 34 + x.numel() * 4 + out.numel() * 4 + ids.nbytes
        L = 2 * len(ring8) if n_tokens == 1 else 2
        t = time_graph(lambda _: [q.q8_0_matmul_id(x, ring8[l % len(ring8)][0], idd, out, top_k, N, K, E,
                                                   stride8, mode=mode, workspace=ws)
                                  for l in range(L)], L, replays=5 if n_tokens == 1 else 2) / L
        q8.append({"n_tokens": n_tokens, "mode": {1: "mv", 2: "mm"}[mode], "us": round(t * 1e6, 2),
                   "GB_s": round(by / t / 1e9, 1), "frac_hbm": round(by / t / 1e9 / pk["hbm_gbs"], 3)})
    return {"experts": E, "top_k": top_k, "N": N, "K": K, "shapes": rows, "swiglu_down_mv": swiglu,
            "q8_0": q8}


# ------------------------------------------------------------------------------------------
# CPU oracle timing (the cpu_baseline leg and the reference arm)
# ------------------------------------------------------------------------------------------
def _host_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def _split_run(fn, n: int, threads: int) -> float:
    """fn(i0, i1) over [0, n) in `threads` contiguous slices on a thread pool (the oracle's C
    calls release the GIL, so the slices run in parallel).  Returns wall seconds."""
    from concurrent.futures import ThreadPoolExecutor
    threads = max(1, min(threads, n))
    step = -(-n // threads)
    t0 = time.perf_counter()
    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(lambda i: fn(i * step, min(n, (i + 1) * step)), range(threads)))
    return time.perf_counter() - t0


def decode_oracle_pass(n_rows: int, cache: dict, threads: int):
    """The decode workload (all 9 shapes, all M tokens, full K) on the oracle, restricted to
    the first n_rows weight rows of every shape (n_rows >= N: the full shapes), split over
    weight rows on `threads` threads.  Returns (seconds, algorithmic bytes of that work)."""
    import oracle
    from weight_only_bit_int4_gb300 import synth
    t = 0.0
    by = 0
    for j, (M, K, N) in enumerate(decode_shapes()):
        key = (M, K, N)
        if key not in cache:
            i = DECODE_KN.index((K, N))
            w, s, b = synth.int4_weights(1000 + i, N, K)
            cache[key] = (synth.activations_bf16(1100 + j, M, K), w, s, b)
        x, w, s, b = cache[key]
        rows = min(n_rows, N)
        t += _split_run(lambda r0, r1: oracle.q4_matmul(x, w[r0:r1], s[r0:r1], b[r0:r1], M, r1 - r0, K),
                        rows, threads)
        by += int4_bytes(M, K, rows)
    return t, by


def oracle_configs(threads: int, gpu_ms: dict):
    """The oracle on every configuration of the workload list, on `threads` host threads:
    0, 1, 3 and 4 in full, 2 (prefill, up to 1.5 T multiply-adds) on 8 sampled token rows
    per weight shape, scaled to the full token count.  Each is also timed on one thread over a
    1/threads share of its work and scaled up (the one-core figure).  Returns per config the
    oracle time per call (all threads and one core), the GPU time per call of the same work
    (from this bench run) and their ratio."""
    import oracle
    from weight_only_bit_int4_gb300 import synth
    out = {}

    def entry(cfg, what, t_all, t_one, scale=1.0):
        e = {"what": what, "oracle_ms": round(t_all * scale * 1e3, 2),
             "oracle_ms_1core": round(t_one * scale * 1e3, 2)}
        g = gpu_ms.get(cfg)
        if g:
            e["gpu_ms"] = round(g, 5)
            e["gpu_speedup_vs_oracle"] = round(t_all * scale * 1e3 / g, 1)
        out[cfg] = e

    # 0: INT4 M=16 K=512 N=256
    M, K, N = 16, 512, 256
    w, s, b = synth.int4_weights(1000, N, K)
    x = synth.activations_bf16(1001, M, K)
    f = lambda r0, r1: oracle.q4_matmul(x, w[r0:r1], s[r0:r1], b[r0:r1], M, r1 - r0, K)
    entry("0", "INT4 M=16 K=512 N=256", _split_run(f, N, threads), _split_run(f, -(-N // threads), 1) * threads)
    # 1: decode, nine shapes
    cache = {}
    t_all, _ = decode_oracle_pass(1 << 30, cache, threads)
    t_one = 0.0
    for (M, K, N) in decode_shapes():
        x, w, s, b = cache[(M, K, N)]
        share = -(-N // threads)
        t_one += _split_run(lambda r0, r1: oracle.q4_matmul(x, w[r0:r1], s[r0:r1], b[r0:r1], M, r1 - r0, K),
                            share, 1) * (N / share)
    entry("1", "INT4 decode, 9 shapes (one step)", t_all, t_one)
    # 2: prefill, 9 shapes, 8 token rows sampled per weight shape, scaled to the full M
    t_all = t_one = 0.0
    for i, (K, N) in enumerate(PREFILL_KN):
        w, s, b = synth.int4_weights(2000 + i, N, K)
        x = synth.activations_bf16(2100 + i, 8, K, outlier_frac=0.01)
        f = lambda r0, r1: oracle.q4_matmul(x, w[r0:r1], s[r0:r1], b[r0:r1], 8, r1 - r0, K)
        share = -(-N // threads)
        ta, to = _split_run(f, N, threads), _split_run(f, share, 1) * (N / share)
        tot_m = sum(PREFILL_M)
        t_all += ta * tot_m / 8
        t_one += to * tot_m / 8
    entry("2", "INT4 prefill, 9 shapes (sampled: 8 token rows per weight shape)", t_all, t_one)
    # 3: LUT4 M in {1, 512}, K = N = 4096, block 64
    Kl = Nl = 4096
    packed, sc, book = synth.lut4_weights(3000, Nl, Kl, 64)
    t_all = t_one = 0.0
    for Ml in (1, 512):
        xl = synth.activations_bf16(3100 + Ml, Ml, Kl)
        if Ml == 1:   # split over weight rows (the packed rows of [N, K/2] are contiguous)
            f = lambda r0, r1: oracle.lut4_matmul(xl, packed[r0 * Kl // 2:r1 * Kl // 2],
                                                  sc[r0 * Kl // 64:r1 * Kl // 64], book, 1, r1 - r0, Kl, 64, 1)
            n = Nl
        else:         # split over tokens
            f = lambda r0, r1: oracle.lut4_matmul(xl[r0:r1], packed, sc, book, r1 - r0, Nl, Kl, 64, 1)
            n = Ml
        share = -(-n // threads)
        t_all += _split_run(f, n, threads)
        t_one += _split_run(f, share, 1) * (n / share)
    entry("3", "LUT4 M in {1, 512}, K = N = 4096", t_all, t_one)
    # 4: Q4_0 MoE, 64 experts, top 8, K = 2048, N = 1408, n_tokens in {1, 512}
    E, top_k, Nm, Km = 64, 8, 1408, 2048
    wq, stride = synth.q4_0_experts(4000, E, Nm, Km)
    t_all = t_one = 0.0
    for nt in (1, 512):
        ids = synth.routing_ids(4100 + nt, nt, top_k, E)
        xm = synth.activations_f32(4200 + nt, nt, Km)
        if nt == 1:   # split over routed rows
            f = lambda r0, r1: oracle.q4_0_matmul_id_rows(xm, wq, ids, top_k, Nm, Km, E, stride,
                                                          np.arange(r0, r1))
            n = top_k
        else:         # split over tokens
            f = lambda r0, r1: oracle.q4_0_matmul_id(xm[r0:r1], wq, ids[r0 * top_k:r1 * top_k], r1 - r0, top_k,
                                                     Nm, Km, E, stride)
            n = nt
        share = -(-n // threads)
        t_all += _split_run(f, n, threads)
        t_one += _split_run(f, share, 1) * (n / share)
    entry("4", "Q4_0 MoE, 64 experts top 8, n_tokens in {1, 512}", t_all, t_one)
    return out


def cpu_baseline(gpu_ms: dict, with_configs: bool = True):
    """The oracle on the GPU machine's host cores: `value` is the full decode workload (one step
    of the nine shapes) in the metric's unit on every host thread; `configs` gives every
    configuration's oracle time per call and the GPU's speed-up over it."""
    threads = _host_threads()
    t, by = decode_oracle_pass(1 << 30, {}, threads)
    res = {"value": round(by / t / 1e9, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
           "sample": f"decode workload, all 9 shapes in full (one step), split over weight rows on "
                     f"{threads} threads, {t:.1f} s"}
    if with_configs:
        res["configs"] = oracle_configs(threads, gpu_ms)
    return res


def run_reference(args, rank, world):
    if rank != 0:
        return None
    threads = _host_threads()
    # rows per shape so that the whole run spends about --reference-seconds
    cache = {}
    t1, by1 = decode_oracle_pass(64, cache, threads)
    per_row = t1 / 64
    n_rows = max(16, int(args.reference_seconds / max(1, args.steps + args.warmup) / per_row))
    for _ in range(args.warmup):
        decode_oracle_pass(n_rows, cache, threads)
    t_tot, by_tot = 0.0, 0
    for _ in range(args.steps):
        t, by = decode_oracle_pass(n_rows, cache, threads)
        t_tot += t
        by_tot += by
    value = by_tot / t_tot / 1e9
    sample = (f"decode workload, first {min(n_rows, 14336)} weight rows of each of the 9 shapes per step "
              f"(all M tokens, full K), {threads} threads")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(t_tot / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "INT4 g32 affine decode GEMV, M in {1,4,16} x (K,N) in "
                                   "{(4096,14336),(14336,4096),(4096,4096)} (bounded row sample)",
                       "parallelism": f"cpu oracle, {threads} threads"},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


CASES = {
    "gemv_m1": "q4_gemv M=1 K=4096 N=14336",
    "gemv_m16": "q4_gemv M=16 K=14336 N=4096",
    "gemm_m2048": "q4_gemm M=2048 K=4096 N=14336",
    "gemm_m8192": "q4_gemm M=8192 K=14336 N=4096 (384-token tiles)",
    "lut4_m1": "lut4_matmul M=1 K=N=4096",
    "lut4_m512": "lut4_matmul M=512 K=N=4096",
    "lut4_f16_m1": "lut4_matmul M=1 K=N=4096, weights rounded to f16 (CUDA-core row kernel)",
    "moe_n1": "q4_0_matmul_id n_tokens=1 (mat-vec)",
    "moe_n512": "q4_0_matmul_id n_tokens=512 (mat-mat)",
    "moe_q8_n1": "q8_0_matmul_id n_tokens=1 (mat-vec)",
    "moe_q8_n512": "q8_0_matmul_id n_tokens=512 (mat-mat)",
    "swiglu_n1": "q4_0_matmul_id_swiglu n_tokens=1, K=1408 -> N=2048 (fused SwiGLU mat-vec)",
}


def run_case(name: str, launches: int = 3):
    """One named small workload, `launches` eager calls: the unit that profiler captures use.
    Prints a wall-clock figure for orientation only (never a bench value)."""
    import torch

    import weight_only_bit_int4_gb300 as q
    from weight_only_bit_int4_gb300 import synth
    dev = torch.device("cuda", 0)

    def to_dev(a):
        a = np.ascontiguousarray(a)
        view = {np.dtype(np.uint16): np.int16, np.dtype(np.uint32): np.int32}.get(a.dtype, a.dtype)
        return torch.from_numpy(a.view(view)).to(dev)

    if name.startswith("gemv") or name.startswith("gemm"):
        M, K, N = {"gemv_m1": (1, 4096, 14336), "gemv_m16": (16, 14336, 4096),
                   "gemm_m2048": (2048, 4096, 14336), "gemm_m8192": (8192, 14336, 4096)}[name]
        w, s, b = synth.int4_weights(1000, N, K)
        x = to_dev(synth.activations_bf16(1100, M, K, outlier_frac=0.01 if M > 16 else 0.0))
        W = (to_dev(w), to_dev(s), to_dev(b))
        y = torch.empty((M, N), dtype=torch.int16, device=dev)
        fn = (lambda: q.q4_gemv(x, *W, y)) if name.startswith("gemv") else (lambda: q.q4_gemm(x, *W, y))
    elif name.startswith("lut4"):
        M = 512 if name == "lut4_m512" else 1
        N = K = 4096
        packed, scales, book = synth.lut4_weights(3000, N, K, 64)
        x = to_dev(synth.activations_bf16(3100 + M, M, K))
        P, S = to_dev(packed), to_dev(scales)
        y = torch.empty((M, N), dtype=torch.int16, device=dev)
        rounding = "f16" if name == "lut4_f16_m1" else None
        fn = lambda: q.lut4_matmul(x, P, S, book, y, N, K, 64, 1, rounding=rounding)
    elif name == "swiglu_n1":
        E, top_k, N, K = 64, 8, 2048, 1408
        w, stride = synth.q4_0_experts(4300, E, N, K)
        ids = synth.routing_ids(4400, 1, top_k, E)
        gate = to_dev(synth.activations_f32(4500, top_k, K))
        up = to_dev(synth.activations_f32(4501, top_k, K))
        Wd, idd = to_dev(w), to_dev(ids.view(np.int32))
        out = torch.empty((top_k, N), dtype=torch.float32, device=dev)
        fn = lambda: q.q4_0_matmul_id_swiglu(gate, up, Wd, idd, out, top_k, N, K, E, stride)
    elif name in ("moe_q8_n1", "moe_q8_n512"):
        n_tokens = 1 if name == "moe_q8_n1" else 512
        E, top_k, N, K = 64, 8, 1408, 2048
        w, stride = synth.q8_0_experts(4000, E, N, K)
        ids = synth.routing_ids(4100 + n_tokens, n_tokens, top_k, E)
        x = to_dev(synth.activations_f32(4200 + n_tokens, n_tokens, K))
        Wd, idd = to_dev(w), to_dev(ids.view(np.int32))
        out = torch.empty((n_tokens * top_k, N), dtype=torch.float32, device=dev)
        ws = torch.empty(q.q8_0_matmul_id_workspace_size(n_tokens, top_k, N, K, E), dtype=torch.uint8,
                         device=dev)
        mode = 1 if n_tokens == 1 else 2
        fn = lambda: q.q8_0_matmul_id(x, Wd, idd, out, top_k, N, K, E, stride, mode=mode, workspace=ws)
    else:
        n_tokens = 1 if name == "moe_n1" else 512
        E, top_k, N, K = 64, 8, 1408, 2048
        w, stride = synth.q4_0_experts(4000, E, N, K)
        ids = synth.routing_ids(4100 + n_tokens, n_tokens, top_k, E)
        x = to_dev(synth.activations_f32(4200 + n_tokens, n_tokens, K))
        Wd, idd = to_dev(w), to_dev(ids.view(np.int32))
        out = torch.empty((n_tokens * top_k, N), dtype=torch.float32, device=dev)
        ws = torch.empty(q.q4_0_matmul_id_workspace_size(n_tokens, top_k, N, K, E), dtype=torch.uint8,
                         device=dev)
        mode = 1 if n_tokens == 1 else 2
        fn = lambda: q.q4_0_matmul_id(x, Wd, idd, out, top_k, N, K, E, stride, mode=mode, workspace=ws)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(launches):
        fn()
    torch.cuda.synchronize()
    print(json.dumps({"case": name, "what": CASES[name], "launches": launches,
                      "wall_ms_per_call_orientation_only": round((time.perf_counter() - t0) / launches * 1e3, 3)}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--quick", action="store_true", help="headline workload only")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--reference-seconds", type=float, default=120.0,
                    help="--impl reference: oracle seconds for the whole warmup + steps run")
    ap.add_argument("--case", choices=sorted(CASES), help="run one small named workload (profiling)")
    args = ap.parse_args()
    if args.case:
        run_case(args.case)
        return
    args.warmup = max(3, args.warmup)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        out = run_reference(args, rank, world)
        if out is not None:
            print(json.dumps(out), flush=True)
        return

    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    out = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
