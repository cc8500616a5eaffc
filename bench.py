#!/usr/bin/env python
"""Throughput of the block-scaled FP8 GEMM on the dense workload, printed as one JSON line.

Workload (one "step"): the dense normal FP8 GEMM NT, D[M,N] = A[M,K] . B[N,K]^T with 1x128 / 128x128
FP32 block scales and BF16 output, for every M in {64, 128, 4096} and (N, K) in {(2112, 7168),
(24576, 1536), (32768, 512), (7168, 16384), (4096, 7168), (7168, 2048)}: 18 GEMMs, each on its own
device buffers (about 1.5 GB in all, far above the 129 MB L2, so no GEMM finds its inputs cached from
its previous run). Inputs are seeded synthetic N(0,1) values block-quantised to e4m3.

value: FP8 TFLOP/s over the whole step (sum of 2MNK / device time of the step), summed over ranks.
e2e:   the same through the public API with host buffers: pinned host -> device copies of every GEMM's
       inputs, the call, and the device -> host copy of every output inside the timed region.
roofline: the kernel with the largest share of the step, against the measured tensor (FP8 = 2 x the
       measured BF16 rate) or HBM peak, whichever bounds that shape.
cpu_baseline / --impl reference: the CPU oracle on a bounded row sample of the same 18 GEMMs.

Launch: python bench.py [--gpus N --steps K --warmup W] [--impl reference]; for N > 1 under
torch.distributed.run, one replica per rank (the GEMMs are independent; there is no exchange).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "FP8 GEMM TFLOP/s per shape on 1 GB300; fraction of min(FP8 peak, HBM roofline)"
MS = (64, 128, 4096)
NKS = ((2112, 7168), (24576, 1536), (32768, 512), (7168, 16384), (4096, 7168), (7168, 2048))
SHAPES = [(M, N, K) for (N, K) in NKS for M in MS]
WORKLOAD = ("dense normal FP8 GEMM NT (e4m3, 1x128 / 128x128 FP32 scales, BF16 out), "
            "M in {64,128,4096} x (N,K) in {(2112,7168),(24576,1536),(32768,512),(7168,16384),(4096,7168),(7168,2048)}")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
CPU_SAMPLE_ROWS = 64      # cpu_baseline: rows per GEMM
REF_SAMPLE_ROWS = 16      # --impl reference: rows per GEMM per step


def flops(M, N, K):
    return 2.0 * M * N * K


def algo_bytes(M, N, K):
    kb, nb = K // 128, (N + 127) // 128
    return M * K + N * K + 4 * M * kb + 4 * nb * kb + 2 * M * N


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def roofline_time(M, N, K, peaks):
    fp8 = 2.0 * peaks["bf16_tflops_sustained"] * 1e12
    bw = peaks["hbm_gbs"] * 1e9
    tf, tb = flops(M, N, K) / fp8, algo_bytes(M, N, K) / bw
    return max(tf, tb), ("tensor" if tf >= tb else "hbm")


def kernel_source_digest():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "moe_grouped_gemm_tma_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(shape):
    """DRAM bytes per launch from the committed ncu record, if it was taken on the current kernels."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    if rec.get("kernel_source_digest") != kernel_source_digest():
        return None
    return rec.get("per_launch_bytes", {}).get("x".join(map(str, shape)))


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while the timed region runs."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            sel = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
            self.proc = subprocess.Popen(["nvidia-smi", "-i", sel, f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(name)
        busy = sorted(sm)[len(sm) // 2:] if sm else []
        return {"sm_mhz": float(np.median(busy)) if busy else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def make_inputs():
    """Host inputs per (N, K): A for the largest M (smaller M take its first rows) and B, with scales."""
    from moe_grouped_gemm_tma_gb300 import inputs as I
    need = {}
    for (M, N, K) in SHAPES:
        need[(N, K)] = max(need.get((N, K), 0), M)
    return {(N, K): I.make_normal(I.seed_for(1, 0), M, N, K) for (N, K), M in need.items()}


def cpu_oracle_rate(host, rows_per_gemm):
    """Oracle TFLOP/s on the first `rows_per_gemm` rows of each of the 18 GEMMs, all host threads."""
    from oracle import oracle as O
    total_flops, t0 = 0.0, time.perf_counter()
    for (M, N, K) in SHAPES:
        c = host[(N, K)]
        r = min(rows_per_gemm, M)
        O.gemm_fp8_nt(c.A[:r], c.sfa[:r], c.B, c.sfb)
        total_flops += flops(r, N, K)
    dt = time.perf_counter() - t0
    return total_flops / dt / 1e12, dt, total_flops, O.hardware_threads()


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    from oracle import oracle as O
    O.build()
    host = make_inputs()
    for _ in range(args.warmup):
        cpu_oracle_rate(host, REF_SAMPLE_ROWS)
    times, fl = [], 0.0
    for _ in range(args.steps):
        _, dt, fl, threads = cpu_oracle_rate(host, REF_SAMPLE_ROWS)
        times.append(dt)
    total = sum(times)
    value = fl * args.steps / total / 1e12
    sample = f"first {REF_SAMPLE_ROWS} rows of each of the 18 GEMMs per step ({fl / 1e9:.1f} GFLOP)"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample": sample},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import moe_grouped_gemm_tma_gb300 as dg

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    dg.load()
    peaks, peak_kind = load_peaks()

    host = make_inputs()
    # device buffers: every GEMM gets its own copies (distinct addresses keep each run L2-cold)
    bufs = []
    for (M, N, K) in SHAPES:
        c = host[(N, K)]
        bufs.append(dict(
            shape=(M, N, K),
            A=c.A[:M].to(dev), sfa=c.sfa[:M].to(dev), B=c.B.to(dev), sfb=c.sfb.to(dev),
            D=torch.empty(M, N, dtype=torch.bfloat16, device=dev)))
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()

    def step():
        for b in bufs:
            dg.dg_gemm_fp8_nt(b["A"], b["sfa"], b["B"], b["sfb"], b["D"], stream=stream)

    host_s = []
    for _ in range(max(args.warmup, 0)):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        step()
        host_s.append(time.perf_counter() - t0)
    if dg.dg_device_status(stream) != 0:
        raise RuntimeError("device-side timeout during warm-up")
    # Small GEMMs run for a few microseconds, less than the host needs to enqueue one call, so the GPU
    # is first kept busy by a spin kernel for longer than the host takes to enqueue every timed launch;
    # the events then measure device time only (the e2e figure below keeps the host in the loop).
    enqueue_s = (min(host_s) if host_s else 0.01) * (args.steps + 1)
    spin_cycles = int(min(2.0, 1.5 * enqueue_s + 0.005) * 2.1e9)

    n = len(bufs)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(dev.index)
    time.sleep(0.3)
    # timed region: K steps back to back, only a start and a stop event (events between launches would
    # serialise them and hide the overlap of one GEMM's set-up with the previous one's tail)
    torch.cuda._sleep(spin_cycles)
    start.record(stream)
    for _ in range(args.steps):
        step()
    stop.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    if dg.dg_device_status(stream) != 0:
        raise RuntimeError("device-side timeout in the timed region")
    total_ms = start.elapsed_time(stop)
    if world > 1:
        t = torch.tensor([total_ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        total_ms = float(t.item())

    # per-launch breakdown (roofline of the dominant kernel): a second pass with an event after every
    # launch, also behind a spin kernel
    prof_steps = max(1, min(args.steps, 20))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(n + 1)] for _ in range(prof_steps)]
    torch.cuda.synchronize()
    torch.cuda._sleep(int(min(2.0, 1.5 * (min(host_s) if host_s else 0.01) * (prof_steps + 1) + 0.005) * 2.1e9))
    for s_ in range(prof_steps):
        ev[s_][0].record(stream)
        for i, b in enumerate(bufs):
            dg.dg_gemm_fp8_nt(b["A"], b["sfa"], b["B"], b["sfb"], b["D"], stream=stream)
            ev[s_][i + 1].record(stream)
    torch.cuda.synchronize()
    per_launch = np.array([[ev[s_][i].elapsed_time(ev[s_][i + 1]) for i in range(n)] for s_ in range(prof_steps)])
    avg_ms = per_launch.mean(axis=0)
    step_flops = sum(flops(*b["shape"]) for b in bufs)
    value = step_flops * args.steps * world / (total_ms * 1e-3) / 1e12

    per_shape = []
    for i, b in enumerate(bufs):
        M, N, K = b["shape"]
        t_roof, bound = roofline_time(M, N, K, peaks)
        per_shape.append({"M": M, "N": N, "K": K, "ms": round(float(avg_ms[i]), 5),
                          "tflops": round(flops(M, N, K) / (avg_ms[i] * 1e-3) / 1e12, 1),
                          "gbs": round(algo_bytes(M, N, K) / (avg_ms[i] * 1e-3) / 1e9, 1),
                          "bound": bound, "roofline_frac": round(t_roof / (avg_ms[i] * 1e-3), 3)})
    dom = int(np.argmax(avg_ms))
    M, N, K = bufs[dom]["shape"]
    _, bound = roofline_time(M, N, K, peaks)
    if bound == "tensor":
        achieved = flops(M, N, K) / (avg_ms[dom] * 1e-3) / 1e12
        peak = 2.0 * peaks["bf16_tflops_sustained"]
        unit = "TFLOP/s"
    else:
        achieved = algo_bytes(M, N, K) / (avg_ms[dom] * 1e-3) / 1e9
        peak = peaks["hbm_gbs"]
        unit = "GB/s"
    roofline = {"bound": bound, "achieved": round(achieved, 1), "peak": peak, "unit": unit,
                "frac": round(achieved / peak, 4), "traffic": ncu_traffic((M, N, K)),
                "kernel": f"dg_gemm_kernel normal M={M} N={N} K={K}",
                "peak_source": f"{peak_kind} ({'2 x bf16_tflops_sustained' if bound == 'tensor' else 'hbm_gbs'})",
                "share": round(float(avg_ms[dom] / avg_ms.sum()), 3)}

    # end to end through the public API with host buffers: pinned H2D of every input, the call, D2H
    pinned = []
    h2d = d2h = 0
    for (M, N, K) in SHAPES:
        c = host[(N, K)]
        hb = dict(A=c.A[:M].contiguous().pin_memory(), sfa=c.sfa[:M].contiguous().pin_memory(),
                  B=c.B.pin_memory(), sfb=c.sfb.pin_memory(),
                  D=torch.empty(M, N, dtype=torch.bfloat16).pin_memory())
        h2d += sum(hb[k].numel() * hb[k].element_size() for k in ("A", "sfa", "B", "sfb"))
        d2h += hb["D"].numel() * hb["D"].element_size()
        pinned.append(hb)

    def e2e_step():
        for b, hb in zip(bufs, pinned):
            for k in ("A", "sfa", "B", "sfb"):
                b[k].copy_(hb[k], non_blocking=True)
            dg.dg_gemm_fp8_nt(b["A"], b["sfa"], b["B"], b["sfb"], b["D"], stream=stream)
            hb["D"].copy_(b["D"], non_blocking=True)

    for _ in range(max(1, min(args.warmup, 3))):
        e2e_step()
    e2e_steps = max(1, min(args.steps, 10))
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    if world > 1:
        t = torch.tensor([e2e_ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        e2e_ms = float(t.item())
    e2e_value = step_flops * e2e_steps * world / (e2e_ms * 1e-3) / 1e12

    if rank == 0:
        cpu_tf, cpu_s, cpu_fl, threads = cpu_oracle_rate(host, CPU_SAMPLE_ROWS)
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "fp8_e4m3", "data": "synthetic",
            "config": {"workload": WORKLOAD if len(SHAPES) > 1 else f"single GEMM M,N,K = {SHAPES[0]}",
                       "gemms_per_step": n,
                       "l2": "inputs larger than L2: each GEMM has its own buffers, ~1.5 GB per step in all",
                       "parallelism": "replicas" if world > 1 else "single GPU",
                       "timing": "device time: CUDA events around the K steps, enqueued behind a GPU spin "
                                 "kernel so host launch cost is excluded (e2e includes it); per_shape and "
                                 "roofline from a second pass with an event after every launch"},
            "roofline": roofline,
            "cpu_baseline": {"value": cpu_tf, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                             "sample": f"first {CPU_SAMPLE_ROWS} rows of each of the 18 GEMMs "
                                       f"({cpu_fl / 1e9:.1f} GFLOP in {cpu_s:.1f} s)"},
            "e2e": {"value": round(e2e_value, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps},
            "clocks": clk,
            "gpu_launches": n * args.steps,
            "per_shape": per_shape,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--shape", default=None,
                    help="M,N,K: time only this GEMM of the workload (for profiler captures)")
    args = ap.parse_args()
    if args.shape:
        global SHAPES
        SHAPES = [tuple(int(x) for x in args.shape.split(","))]
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
