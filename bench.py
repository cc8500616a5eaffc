#!/usr/bin/env python
"""Throughput of the block-scaled FP8 GEMM and its MoE variants, printed as one JSON line.

With no --workload, every workload below runs in turn; the line's top-level numbers are the dense
workload's (the headline configuration) and `per_workload` holds each workload's own value, roofline,
e2e, clocks, CPU baseline and per-case figures. One "step" = every case of a workload once, each on its
own device buffers.

* dense (headline): the normal FP8 GEMM NT, D[M,N] = A[M,K] . B[N,K]^T, 1x128 / 128x128 FP32 block
  scales, BF16 out, for M in {64, 128, 4096} x (N, K) in {(2112, 7168), (24576, 1536), (32768, 512),
  (7168, 16384), (4096, 7168), (7168, 2048)}: 18 GEMMs, about 1.5 GB of buffers in all.
* tiny: the parity-sized normal GEMM, M=128, N=256, K=512 (launch-bound; reported for completeness).
* contiguous: m-grouped contiguous layout, G in {4, 8} experts, rows per expert U[0.7, 1.3] x {8192,
  4096} padded to 128, (N, K) in {(4096, 7168), (7168, 2048)}.
* masked: m-grouped masked layout (decode), G in {1, 2, 4, 16}, (max_m, expected_m) in {(256, 64),
  (512, 128), (1024, 256)}, masked_m U[0.7, 1.0] x expected_m, (N, K) as above.
* kgrouped: k-grouped FP32 weight gradient, G in {4, 8}, tokens per expert U[0.5, 1.5] x 4096 padded
  to 128, (M, N) in {(7168, 4096), (2048, 7168)}.
* layouts: the M=4096 dense GEMMs with A and/or B stored transposed (TN, NN, TT).
* ue8m0: the dense workload with power-of-two block scales on the block-scaled (UE8M0) path.

Inputs are seeded synthetic N(0,1) values block-quantised to e4m3 (drawn on the GPU with the same
counter-based generator the tests use on the CPU). Every case has its own buffers, so the working set of
a step is far above the 129 MB L2 and no case finds its inputs cached from its previous run.

value: TFLOP/s over the whole step (2MNK per case, real rows only), summed over ranks; device time of K
       steps between a start and a stop event, enqueued behind a GPU spin kernel so host launch cost
       is excluded.
e2e:   the same through the public API with host buffers: pinned host -> device copies of every case's
       inputs, the call, and the device -> host copy of every output inside the timed region.
roofline: the case with the largest share of the step, against the measured peak that bounds it: the
       FP8 tensor peak = 2 x the measured burst BF16 rate (the kernels are timed launch by launch, well
       under a second), or the measured HBM copy rate. `frac_of_sustained` restates it against 2 x the
       sustained BF16 rate. per_case lists every case against the same peaks.
cpu_baseline / --impl reference: the CPU oracle on a bounded row sample of the same cases.

Launch: python bench.py [--gpus N --steps K --warmup W] [--workload W] [--impl reference]; for N > 1
under torch.distributed.run, one replica per rank (the GEMMs are independent; there is no exchange).
--timed-only runs the warm-up and timed steps alone (for profiler captures).
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
HEADLINE = "dense"
WORKLOAD_ORDER = ("dense", "tiny", "contiguous", "masked", "kgrouped", "layouts", "ue8m0")
WORKLOADS = {
    "tiny": "parity-sized normal FP8 GEMM NT, M=128, N=256, K=512, BF16 out",
    "dense": ("dense normal FP8 GEMM NT (e4m3, 1x128 / 128x128 FP32 scales, BF16 out), M in {64,128,4096} x "
              "(N,K) in {(2112,7168),(24576,1536),(32768,512),(7168,16384),(4096,7168),(7168,2048)}"),
    "contiguous": ("m-grouped contiguous FP8 GEMM (MoE prefill / training forward), G in {4,8}, rows per expert "
                   "U[0.7,1.3] x {8192,4096} padded to 128, (N,K) in {(4096,7168),(7168,2048)}, BF16 out"),
    "masked": ("m-grouped masked FP8 GEMM (MoE decode), G in {1,2,4,16}, (max_m, expected_m) in {(256,64),"
               "(512,128),(1024,256)}, masked_m U[0.7,1.0] x expected_m, (N,K) in {(4096,7168),(7168,2048)}"),
    "ue8m0": ("dense normal FP8 GEMM NT as the dense workload, with power-of-two block scales (amax/448 rounded up), "
              "on the block-scaled UE8M0 tensor-core path, BF16 out"),
    "layouts": ("dense normal FP8 GEMM, M=4096, (N,K) as the dense workload, with transposed operand storage: "
                "TN (A stored [K,M]), NN (B stored [K,N]), TT (both); BF16 out"),
    "kgrouped": ("k-grouped FP8 weight-gradient GEMM, FP32 accumulated, G in {4,8}, tokens per expert "
                 "U[0.5,1.5] x 4096 padded to 128, (M,N) in {(7168,4096),(2048,7168)}"),
}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
CPU_SAMPLE_ROWS = 1024    # cpu_baseline of the headline: rows per case (all rows of a smaller case); ~10 s on 16 cores
CPU_SAMPLE_ROWS_OTHER = 128   # ... of every other workload (a few seconds each)
STREAM_COPY_BYTES = 256 << 20   # per-case in-stream timing: input copies cycled per case (2 x L2)
REF_SAMPLE_ROWS = 16      # --impl reference: rows per case per step


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_digest():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "moe_grouped_gemm_tma_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload, name):
    """DRAM bytes per launch (keyed "workload:case") from the committed ncu record, if it was taken on the
    current kernels."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    if rec.get("kernel_source_digest") != kernel_source_digest():
        return None
    return rec.get("per_launch_bytes", {}).get(f"{workload}:{name}")


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
                                          "--format=csv,noheader,nounits", "-lms", "100"],
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
        return parse_clock_samples(out)


def parse_clock_samples(text):
    """Clock record of a timed region from nvidia-smi CSV lines (ClockSampler.FIELDS, no header, no
    units): the median SM clock over the busier half of the samples (the sampler starts and stops a
    little outside the region), the maximum SM clock, and every throttle reason seen active. Lines that
    do not parse (fewer fields, "[N/A]") are skipped."""
    sm, smax, reasons = [], [], set()
    names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
    for line in text.strip().splitlines():
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


def max_over_ranks(ms, world, device):
    """The slowest rank's time, on every rank (the job ends when its last replica does)."""
    if world <= 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tflops(step_flops, steps, world, ms):
    """Whole-job throughput: every replica ran `steps` steps of `step_flops` within `ms`."""
    return step_flops * steps * world / (ms * 1e-3) / 1e12


# ------------------------------------------------------------------------------------------------ cases
class Case:
    """One GEMM of a workload: its inputs (on the generation device), work counts and calls."""

    def __init__(self, name, flops, nbytes, inputs, out_shape, out_dtype, call, oracle, init_out=None):
        self.name, self.flops, self.bytes = name, float(flops), float(nbytes)
        self.inputs = inputs              # ordered dict name -> tensor (copied H2D in e2e)
        self.out_shape, self.out_dtype = out_shape, out_dtype
        self.call = call                  # call(dev_inputs, dev_out, stream)
        self.oracle = oracle              # oracle(cpu_inputs, rows) -> sampled flops
        self.init_out = init_out          # output buffer contents that the call accumulates into


def ue8m0_cases():
    """The dense workload's 18 GEMMs with power-of-two block scales, on the block-scaled (UE8M0) path."""
    import moe_grouped_gemm_tma_gb300 as dg
    cases = dense_cases(pow2=True)
    for c in cases:
        c.call = lambda d, o, s: dg.dg_gemm_fp8_nt_ue8m0(d["A"], d["sfa"], d["B"], d["sfb"], o, stream=s)
    return cases


def dense_cases(only=None, pow2=False, seed_config=1):
    import moe_grouped_gemm_tma_gb300 as dg
    from moe_grouped_gemm_tma_gb300 import inputs as I
    from oracle import oracle as O
    shapes = [(M, N, K) for (N, K) in NKS for M in MS] if only is None else [only]
    need = {}
    for (M, N, K) in shapes:
        need[(N, K)] = max(need.get((N, K), 0), M)
    big = {(N, K): I.make_normal(I.seed_for(seed_config, 0), M, N, K, pow2=pow2) for (N, K), M in need.items()}
    cases = []
    for (M, N, K) in shapes:
        c = big[(N, K)]
        kb, nb = K // 128, (N + 127) // 128
        inp = {"A": c.A[:M].contiguous(), "sfa": c.sfa[:M].contiguous(), "B": c.B, "sfb": c.sfb}
        cases.append(Case(
            f"{M}x{N}x{K}", 2.0 * M * N * K, M * K + N * K + 4 * M * kb + 4 * nb * kb + 2 * M * N, inp, (M, N),
            torch.bfloat16,
            lambda d, o, s: dg.dg_gemm_fp8_nt(d["A"], d["sfa"], d["B"], d["sfb"], o, stream=s),
            lambda h, r: (O.gemm_fp8_nt(h["A"][:r], h["sfa"][:r], h["B"], h["sfb"]),
                          2.0 * min(r, h["A"].shape[0]) * h["B"].shape[0] * h["B"].shape[1])[1]))
    return cases


def layouts_cases():
    """The M=4096 dense GEMMs with transposed operand storage: TN (A stored [K, M]), NN (B stored
    [K, N]) and TT (both)."""
    import moe_grouped_gemm_tma_gb300 as dg
    from moe_grouped_gemm_tma_gb300 import inputs as I
    from oracle import oracle as O
    M = 4096
    cases = []
    for (N, K) in NKS:
        c = I.make_normal(I.seed_for(1, 0), M, N, K)
        kb, nb = K // 128, (N + 127) // 128
        for name, a_mn, b_mn in (("TN", True, False), ("NN", False, True), ("TT", True, True)):
            inp = {"A": c.A.t().contiguous() if a_mn else c.A, "sfa": c.sfa,
                   "B": c.B.t().contiguous() if b_mn else c.B, "sfb": c.sfb}
            cases.append(Case(
                f"{name} {M}x{N}x{K}", 2.0 * M * N * K, M * K + N * K + 4 * M * kb + 4 * nb * kb + 2 * M * N, inp,
                (M, N), torch.bfloat16,
                (lambda a, b: lambda d, o, s: dg.dg_gemm_fp8(d["A"], d["sfa"], d["B"], d["sfb"], o, a_mn_major=a,
                                                              b_mn_major=b, stream=s))(a_mn, b_mn),
                (lambda a, b, n_, k_: lambda h, r: (O.gemm_fp8_nt((h["A"].t() if a else h["A"])[:r].contiguous(), h["sfa"][:r],
                                                                  (h["B"].t() if b else h["B"]).contiguous(), h["sfb"]),
                                                    2.0 * min(r, M) * n_ * k_)[1])(a_mn, b_mn, N, K)))
    return cases


CONTIGUOUS_SHAPES = tuple((G, base, N, K) for (N, K) in ((4096, 7168), (7168, 2048)) for G, base in ((4, 8192), (8, 4096)))


def contiguous_cases(shapes=CONTIGUOUS_SHAPES):
    import moe_grouped_gemm_tma_gb300 as dg
    from moe_grouped_gemm_tma_gb300 import inputs as I
    from oracle import oracle as O
    cases = []
    for (G, base, N, K) in shapes:
        seed = I.seed_for(2, G * 10 + base // 4096 + N)
        sizes = I.contiguous_group_sizes(seed, G, base)
        c = I.make_contiguous(seed, G, N, K, sizes)
        rows = sum(sizes)
        kb, nb = K // 128, (N + 127) // 128
        inp = {"A": c.A, "sfa": c.sfa, "B": c.B, "sfb": c.sfb, "m_indices": c.m_indices}
        cases.append(Case(
            f"G{G}x{rows}rows N{N} K{K}", 2.0 * rows * N * K,
            rows * K + G * N * K + 4 * rows * kb + 4 * G * nb * kb + 2 * rows * N + 4 * c.Mt, inp, (c.Mt, N),
            torch.bfloat16,
            lambda d, o, s: dg.dg_m_grouped_contiguous(d["A"], d["sfa"], d["B"], d["sfb"], d["m_indices"], o, stream=s),
            lambda h, r: (O.m_grouped_contiguous(h["A"][:r], h["sfa"][:r], h["B"], h["sfb"], h["m_indices"][:r]),
                          2.0 * int((h["m_indices"][:r] >= 0).sum()) * h["B"].shape[1] * h["B"].shape[2])[1]))
    return cases


MASKED_SHAPES = tuple((G, max_m, em, N, K) for (N, K) in ((4096, 7168), (7168, 2048)) for G in (1, 2, 4, 16)
                      for max_m, em in ((256, 64), (512, 128), (1024, 256)))


def masked_sample_rows(masked_m, max_m, r):
    """Flattened rows (g * max_m + i) of a bounded oracle sample spread over every expert: the first
    rows of each group, up to ceil(r / G) of them, r in all at most."""
    G = len(masked_m)
    per = max(1, -(-r // G))
    rows = [g * max_m + i for g in range(G) for i in range(min(per, max(0, min(int(masked_m[g]), max_m))))]
    return rows[:r]


def masked_cases(shapes=MASKED_SHAPES):
    import moe_grouped_gemm_tma_gb300 as dg
    from moe_grouped_gemm_tma_gb300 import inputs as I
    from oracle import oracle as O
    cases = []
    for (G, max_m, em, N, K) in shapes:
        seed = I.seed_for(3, G * 1000 + max_m + em + N)
        sizes = I.masked_sizes(seed, G, em, max_m)
        c = I.make_masked(seed, G, max_m, N, K, sizes, em)
        rows = sum(sizes)
        kb, nb = K // 128, (N + 127) // 128
        inp = {"A": c.A, "sfa": c.sfa, "B": c.B, "sfb": c.sfb, "masked_m": c.masked_m}

        def oracle_leg(h, r, max_m=max_m):
            sample = masked_sample_rows(h["masked_m"].tolist(), max_m, r)
            if sample:
                O.m_grouped_masked(h["A"], h["sfa"], h["B"], h["sfb"], h["masked_m"], rows=sample)
            return 2.0 * len(sample) * h["B"].shape[1] * h["B"].shape[2]

        cases.append(Case(
            f"G{G} max_m{max_m} E[m]{em} rows{rows} N{N} K{K}", 2.0 * rows * N * K,
            rows * K + G * N * K + 4 * rows * kb + 4 * G * nb * kb + 2 * rows * N, inp, (G, max_m, N),
            torch.bfloat16,
            (lambda em_: lambda d, o, s: dg.dg_m_grouped_masked(d["A"], d["sfa"], d["B"], d["sfb"], d["masked_m"], o,
                                                                 expected_m=em_, stream=s))(em),
            oracle_leg))
    return cases


KGROUPED_SHAPES = tuple((G, M, N, 4096) for (M, N) in ((7168, 4096), (2048, 7168)) for G in (4, 8))


def kgrouped_cases(shapes=KGROUPED_SHAPES):
    import moe_grouped_gemm_tma_gb300 as dg
    from moe_grouped_gemm_tma_gb300 import inputs as I
    from oracle import oracle as O
    cases = []
    for (G, M, N, base_k) in shapes:
        seed = I.seed_for(4, G * 10 + M)
        ks = I.kgrouped_sizes(seed, G, base_k)
        c = I.make_kgrouped(seed, G, M, N, ks)
        sumK = sum(ks)
        inp = {"A": c.A, "sfa": c.sfa, "B": c.B, "sfb": c.sfb}
        cases.append(Case(
            f"G{G} M{M} N{N} sumK{sumK}", 2.0 * M * N * sumK,
            (M + N) * sumK + 4 * (M + N) * sumK // 128 + 8 * G * M * N, inp, (G, M, N), torch.float32,
            (lambda ks_: lambda d, o, s: dg.dg_k_grouped_wgrad(d["A"], d["sfa"], d["B"], d["sfb"], ks_, o, stream=s))(ks),
            (lambda ks_: lambda h, r: (O.k_grouped_wgrad(h["A"][:r], h["sfa"][:r], h["B"], h["sfb"], ks_,
                                                        np.zeros((len(ks_), min(r, h["A"].shape[0]), h["B"].shape[0]), np.float32)),
                                       2.0 * min(r, h["A"].shape[0]) * h["B"].shape[0] * sum(ks_))[1])(ks),
            init_out=c.D_in))
    return cases


def tiny_cases():
    """The parity-sized normal GEMM, 128 x 256 x 512."""
    return dense_cases(only=(128, 256, 512), seed_config=0)


def build_cases(workload, shape=None, only=None):
    if workload == "dense":
        cases = dense_cases(shape)
    elif workload == "tiny":
        cases = tiny_cases()
    else:
        cases = {"contiguous": contiguous_cases, "masked": masked_cases, "kgrouped": kgrouped_cases,
                 "layouts": layouts_cases, "ue8m0": ue8m0_cases}[workload]()
    if only:
        cases = [c for c in cases if only in c.name]
        if not cases:
            raise SystemExit(f"no case of the {workload} workload matches {only!r}")
    return cases


def cpu_oracle_rate(cases, rows_per_case):
    """Oracle TFLOP/s on the first `rows_per_case` rows of every case, all host threads."""
    from oracle import oracle as O
    host = [{k: v.cpu() for k, v in c.inputs.items()} for c in cases]
    total_flops, t0 = 0.0, time.perf_counter()
    for c, h in zip(cases, host):
        total_flops += c.oracle(h, rows_per_case)
    dt = time.perf_counter() - t0
    return total_flops / dt / 1e12, dt, total_flops, O.hardware_threads()


# ------------------------------------------------------------------------------------------------ arms
def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    from oracle import oracle as O
    from moe_grouped_gemm_tma_gb300 import inputs as I
    O.build()
    cases = build_cases(args.workload, args.shape, args.case)
    for _ in range(args.warmup):
        cpu_oracle_rate(cases, REF_SAMPLE_ROWS)
    times, fl, threads = [], 0.0, 0
    for _ in range(args.steps):
        _, dt, fl, threads = cpu_oracle_rate(cases, REF_SAMPLE_ROWS)
        times.append(dt)
    total = sum(times)
    value = fl * args.steps / total / 1e12
    sample = f"first {REF_SAMPLE_ROWS} rows of each of the {len(cases)} cases per step ({fl / 1e9:.1f} GFLOP)"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOADS[args.workload], "sample": sample},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def spin_cycles_for(host_step_s, steps):
    # keep the GPU busy for longer than the host needs to enqueue every timed launch (capped at 2 s)
    return int(min(2.0, 1.5 * host_step_s * (steps + 1) + 0.005) * 2.1e9)


def _peaks_line(peaks):
    """(FP8 tensor peak from the burst BF16 rate, the same from the sustained rate, HBM rate)."""
    return 2.0 * peaks["bf16_tflops"], 2.0 * peaks["bf16_tflops_sustained"], peaks["hbm_gbs"]


def roofline_of(workload, cases, avg_ms, peaks, peak_kind):
    """The dominant case's roofline record and every case's fraction, against the burst FP8 peak (2 x the
    measured burst BF16 rate) or the measured HBM rate, whichever bounds the case."""
    fp8_peak, fp8_sustained, bw = _peaks_line(peaks)
    per = []
    for i, c in enumerate(cases):
        t_tc, t_bw = c.flops / (fp8_peak * 1e12), c.bytes / (bw * 1e9)
        per.append({"case": c.name, "ms": round(float(avg_ms[i]), 5),
                    "tflops": round(c.flops / (avg_ms[i] * 1e-3) / 1e12, 1),
                    "gbs": round(c.bytes / (avg_ms[i] * 1e-3) / 1e9, 1),
                    "bound": "tensor" if t_tc >= t_bw else "hbm",
                    "roofline_frac": round(max(t_tc, t_bw) / (avg_ms[i] * 1e-3), 3)})
    dom = int(np.argmax(avg_ms))
    c = cases[dom]
    if per[dom]["bound"] == "tensor":
        achieved, peak, unit, src = c.flops / (avg_ms[dom] * 1e-3) / 1e12, fp8_peak, "TFLOP/s", "2 x bf16_tflops (burst)"
        sustained = round(achieved / fp8_sustained, 4)
    else:
        achieved, peak, unit, src = c.bytes / (avg_ms[dom] * 1e-3) / 1e9, bw, "GB/s", "hbm_gbs"
        sustained = None
    kernel = "dg_gemm_bs_kernel" if workload == "ue8m0" else "dg_gemm_kernel"
    roof = {"bound": per[dom]["bound"], "achieved": round(achieved, 1), "peak": round(peak, 1), "unit": unit,
            "frac": round(achieved / peak, 4), "traffic": ncu_traffic(workload, c.name),
            "kernel": f"{kernel}, {workload} case {c.name}", "peak_source": f"{peak_kind} ({src})",
            "frac_of_sustained": sustained, "share": round(float(avg_ms[dom] / avg_ms.sum()), 3)}
    return roof, per


def run_workload(workload, args, dev, world, rank, peaks, peak_kind, headline):
    """Time one workload: the K-step timed region, the per-case and in-stream passes, e2e through host
    buffers and the CPU oracle leg. Returns the workload's record (every rank) or None."""
    import moe_grouped_gemm_tma_gb300 as dg
    from moe_grouped_gemm_tma_gb300 import inputs as I

    I.set_generation_device(dev)
    cases = build_cases(workload, args.shape, args.case)
    I.set_generation_device("cpu")
    # device buffers: every case its own copies (distinct addresses keep each run L2-cold)
    bufs = []
    for c in cases:
        d = {k: v.to(dev).clone() for k, v in c.inputs.items()}
        out = (c.init_out.to(dev).clone() if c.init_out is not None
               else torch.empty(c.out_shape, dtype=c.out_dtype, device=dev))
        bufs.append((d, out))
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()

    def step():
        for c, (d, out) in zip(cases, bufs):
            c.call(d, out, stream)

    host_s = []
    for _ in range(max(args.warmup, 0)):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        step()
        host_s.append(time.perf_counter() - t0)
    if dg.dg_device_status(stream) != 0:
        raise RuntimeError(f"{workload}: device-side error during warm-up")
    host_step = min(host_s) if host_s else 0.01

    n = len(cases)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(dev.index)
    time.sleep(0.3)
    # timed region: K steps back to back between one start and one stop event (events between launches
    # would serialise them and hide the overlap of one GEMM's set-up with the previous one's tail)
    torch.cuda._sleep(spin_cycles_for(host_step, args.steps))
    start.record(stream)
    for _ in range(args.steps):
        step()
    stop.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    if dg.dg_device_status(stream) != 0:
        raise RuntimeError(f"{workload}: device-side error in the timed region")
    total_ms = max_over_ranks(start.elapsed_time(stop), world, dev)
    step_flops = sum(c.flops for c in cases)
    value = job_tflops(step_flops, args.steps, world, total_ms)
    rec = {"value": round(value, 2), "unit": "TFLOP/s", "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(total_ms / args.steps, 4), "cases_per_step": n,
           "gpu_launches": n * args.steps, "clocks": clk, "config": WORKLOADS[workload]
           if args.shape is None else f"single dense GEMM M,N,K = {args.shape}"}
    if args.timed_only:
        return rec

    # per-case breakdown: a second pass with an event after every launch, also behind a spin kernel
    prof_steps = max(1, min(args.steps, 20))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(n + 1)] for _ in range(prof_steps)]
    torch.cuda.synchronize()
    torch.cuda._sleep(spin_cycles_for(host_step, prof_steps))
    for s_ in range(prof_steps):
        ev[s_][0].record(stream)
        for i, (c, (d, out)) in enumerate(zip(cases, bufs)):
            c.call(d, out, stream)
            ev[s_][i + 1].record(stream)
    torch.cuda.synchronize()
    avg_ms = np.array([[ev[s_][i].elapsed_time(ev[s_][i + 1]) for i in range(n)] for s_ in range(prof_steps)]).mean(axis=0)

    # In-stream time per launch: each case launched back to back (programmatic dependent launch lets a
    # launch's set-up overlap the previous one's tail, as in a stream of expert GEMMs) on enough distinct
    # buffer copies that none is L2-resident when it runs; one event pair around the run.
    stream_ms = []
    for c, (d, out) in zip(cases, bufs):
        in_bytes = sum(v.numel() * v.element_size() for v in d.values())
        reps = int(min(16, max(2, -(-STREAM_COPY_BYTES // max(in_bytes, 1)))))
        copies = [(d, out)] + [({k: v.clone() for k, v in d.items()}, out.clone()) for _ in range(reps - 1)]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for dd, oo in copies:                       # warm every copy's launch path once
            c.call(dd, oo, stream)
        torch.cuda.synchronize()
        rounds = max(1, min(args.steps, 10))
        torch.cuda._sleep(spin_cycles_for(host_step / max(n, 1) * reps, rounds))
        e0.record(stream)
        for _ in range(rounds):
            for dd, oo in copies:
                c.call(dd, oo, stream)
        e1.record(stream)
        torch.cuda.synchronize()
        stream_ms.append(e0.elapsed_time(e1) / (rounds * reps))
        del copies
    torch.cuda.empty_cache()

    roof, per_case = roofline_of(workload if args.shape is None else "dense", cases, avg_ms, peaks, peak_kind)
    fp8_peak, _, bw = _peaks_line(peaks)
    for pc, c, ms in zip(per_case, cases, stream_ms):
        t_bound = max(c.flops / (fp8_peak * 1e12), c.bytes / (bw * 1e9))
        pc["ms_stream"] = round(float(ms), 5)
        pc["roofline_frac_stream"] = round(t_bound / (ms * 1e-3), 3)
    rec["roofline"] = roof
    rec["per_case"] = per_case

    # end to end through the public API with host buffers: pinned H2D of every input, the call, D2H
    pinned, h2d, d2h = [], 0, 0
    for c in cases:
        hb = {k: v.cpu().contiguous().pin_memory() for k, v in c.inputs.items()}
        if c.init_out is not None:
            hb["__out_in"] = c.init_out.cpu().contiguous().pin_memory()
        hb["__out"] = torch.empty(c.out_shape, dtype=c.out_dtype).pin_memory()
        h2d += sum(v.numel() * v.element_size() for k, v in hb.items() if k != "__out")
        d2h += hb["__out"].numel() * hb["__out"].element_size()
        pinned.append(hb)

    # Three streams, as a serving loop would run them: host-to-device copies of case i+1 and the
    # device-to-host read of case i-1 overlap the GEMM of case i. Per-case events keep every buffer
    # safe across steps: a case's inputs are rewritten only after its previous GEMM has read them, and
    # its output only after the previous result has been copied out.
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in cases]      # inputs of case i are on the device
    ev_done = [torch.cuda.Event() for _ in cases]    # GEMM of case i has run (its inputs may be reused)
    ev_out = [torch.cuda.Event() for _ in cases]     # result of case i is on the host (output reusable)
    for i in range(n):
        ev_done[i].record(stream)
        ev_out[i].record(stream)

    def e2e_step():
        for i, (c, (d, out), hb) in enumerate(zip(cases, bufs, pinned)):
            s_in.wait_event(ev_done[i])
            with torch.cuda.stream(s_in):
                for k in c.inputs:
                    d[k].copy_(hb[k], non_blocking=True)
                if "__out_in" in hb:
                    s_in.wait_event(ev_out[i])
                    out.copy_(hb["__out_in"], non_blocking=True)
            ev_in[i].record(s_in)
            stream.wait_event(ev_in[i])
            stream.wait_event(ev_out[i])
            c.call(d, out, stream)
            ev_done[i].record(stream)
            s_out.wait_event(ev_done[i])
            with torch.cuda.stream(s_out):
                hb["__out"].copy_(out, non_blocking=True)
            ev_out[i].record(s_out)

    for _ in range(max(1, min(args.warmup, 3))):
        e2e_step()
    e2e_steps = max(1, min(args.steps, 10))
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    for _ in range(e2e_steps):
        e2e_step()
    for i in range(n):
        stream.wait_event(ev_out[i])
    stream.wait_event(ev_in[n - 1])
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    rec["e2e"] = {"value": round(job_tflops(step_flops, e2e_steps, world, e2e_ms), 2), "unit": "TFLOP/s",
                  "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                  "pipeline": "pinned H2D, GEMM and D2H on three streams with per-case events"}
    if dg.dg_device_status(stream) != 0:
        raise RuntimeError(f"{workload}: device-side error in the e2e pass")
    del pinned, bufs
    torch.cuda.synchronize()
    torch.cuda.empty_cache()

    if rank == 0:
        rows = CPU_SAMPLE_ROWS if headline else CPU_SAMPLE_ROWS_OTHER
        cpu_tf, cpu_s, cpu_fl, threads = cpu_oracle_rate(cases, rows)
        rec["cpu_baseline"] = {"value": cpu_tf, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                               "sample": f"up to {rows} rows of each of the {n} cases (all rows of a smaller "
                                         f"case; for the masked layout spread over the experts), "
                                         f"{cpu_fl / 1e9:.1f} GFLOP in {cpu_s:.1f} s"}
    return rec


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

    names = list(WORKLOAD_ORDER) if args.workload == "all" else [args.workload]
    results = {}
    for name in names:
        results[name] = run_workload(name, args, dev, world, rank, peaks, peak_kind, headline=(name == names[0]))
    head = results[names[0]]

    if rank == 0:
        line = {
            "metric": METRIC, "value": head["value"], "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "fp8_e4m3", "data": "synthetic",
            "config": {"workload": head["config"], "headline": names[0], "cases_per_step": head["cases_per_step"],
                       "workloads_run": names,
                       "l2": "inputs larger than L2: every case has its own buffers, far above L2 per step",
                       "parallelism": "replicas" if world > 1 else "single GPU",
                       "timing": "device time: CUDA events around the K steps, enqueued behind a GPU spin "
                                 "kernel so host launch cost is excluded (e2e includes it); per_case ms and "
                                 "roofline from a second pass with an event after every launch; per_case "
                                 "ms_stream from back-to-back launches of one case on distinct buffer copies"},
            "roofline": head.get("roofline"),
            "cpu_baseline": head.get("cpu_baseline"),
            "e2e": head.get("e2e"),
            "clocks": head["clocks"],
            "gpu_launches": head["gpu_launches"],
            "per_case": head.get("per_case"),
            "per_workload": {k: v for k, v in results.items() if k != names[0]},
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=["all"] + sorted(WORKLOADS), default="all",
                    help="one workload, or all of them (the default; the dense workload is the headline)")
    ap.add_argument("--timed-only", action="store_true",
                    help="run the warm-up and timed steps alone (no per-case, e2e or CPU passes): for profiler captures")
    ap.add_argument("--shape", default=None,
                    help="M,N,K: time only this GEMM of the dense workload (for profiler captures)")
    ap.add_argument("--case", default=None,
                    help="time only the cases of the workload whose name contains this text (for profiler captures)")
    args = ap.parse_args()
    if args.shape:
        args.shape = tuple(int(x) for x in args.shape.split(","))
        args.workload = "dense"
    if args.impl == "reference":
        if args.workload == "all":
            args.workload = HEADLINE
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
