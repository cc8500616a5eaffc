"""Host logic of bench.py's multi-rank launch, on CPU with two gloo ranks: the timed region's
max-over-ranks reduction, the whole-job throughput, and the reference arm's rank-0-only rule."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # each replica timed its own K steps; the job's time is the slowest one
        slowest = bench.max_over_ranks(10.0 + 5.0 * rank, world, torch.device("cpu"))
        # the reference arm runs on rank 0 only; every other rank exits 0 at once without work
        class Args:
            workload, shape, case, warmup, steps, gpus = "dense", None, None, 0, 1, world
        ref_rc = bench.run_reference(Args) if rank != 0 else 0
        results[rank] = (slowest, ref_rc, bench.dist_env())
    finally:
        dist.destroy_process_group()


def test_two_rank_reduction_and_rank0_rule():
    world = 2
    results = mp.get_context("spawn").Manager().dict()   # no fork of this multi-threaded process
    mp.spawn(_worker, args=(world, _free_port(), results), nprocs=world, join=True)
    for rank in range(world):
        slowest, ref_rc, env = results[rank]
        assert slowest == pytest.approx(15.0)
        assert ref_rc == 0
        assert env == (world, rank, rank)


def test_single_rank_passthrough_and_job_throughput():
    assert bench.max_over_ranks(3.25, 1, torch.device("cpu")) == 3.25
    # 2 replicas x 10 steps x 1 TFLOP in 2 s (2000 ms) = 10 TFLOP/s for the whole job
    assert bench.job_tflops(1e12, 10, 2, 2000.0) == pytest.approx(10.0)


def test_traffic_record_matches_current_kernels_only(monkeypatch):
    # roofline.traffic comes from the committed ncu record only while it was taken on the current
    # kernel source, and is keyed by workload and case (the dense and UE8M0 workloads share case names)
    import json
    rec = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    current = rec["kernel_source_digest"] == bench.kernel_source_digest()
    for key in rec["per_launch_bytes"]:
        workload, case = key.split(":", 1)
        assert workload in bench.WORKLOADS, key
        assert bench.ncu_traffic(workload, case) == (rec["per_launch_bytes"][key] if current else None)
    if current:
        assert bench.ncu_traffic("dense", "4096x7168x16384") != bench.ncu_traffic("ue8m0", "4096x7168x16384")
    assert bench.ncu_traffic("dense", "no such case") is None
    # after any change to the kernel sources the record no longer applies
    monkeypatch.setattr(bench, "kernel_source_digest", lambda: "0" * 16)
    assert bench.ncu_traffic("dense", "4096x7168x16384") is None


# nvidia-smi lines as the sampler asks for them: sm, max sm, power, active mask, hw_slowdown,
# hw_thermal_slowdown, sw_thermal_slowdown, sw_power_cap
_IDLE = "1980, 2070, 300.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active"
_BUSY = "2070, 2070, 1100.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active"
_CAPPED = "1995, 2070, 1398.7, 0x0000000000000004, Not Active, Not Active, Not Active, Active"
_HOT = "1500, 2070, 1200.0, 0x0000000000000040, Not Active, Active, Not Active, Not Active"


def test_clock_record_median_of_the_busy_half_and_reasons():
    rec = bench.parse_clock_samples("\n".join([_IDLE, _BUSY, _BUSY, _CAPPED, _BUSY, _IDLE]) + "\n")
    # sorted 1980 1980 1995 2070 2070 2070: the busier half is 2070 x 3
    assert rec == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 6}
    rec = bench.parse_clock_samples("\n".join([_HOT, _BUSY, _CAPPED, _BUSY]))
    assert rec["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    assert rec["sm_mhz"] == pytest.approx(2070.0)


def test_clock_record_skips_unparsable_lines_and_reports_no_samples():
    rec = bench.parse_clock_samples("[N/A], [N/A], [N/A], [N/A], [N/A], [N/A], [N/A], [N/A]\nshort, line\n" + _BUSY)
    assert rec["samples"] == 1 and rec["sm_mhz"] == 2070.0 and rec["reasons"] == []
    assert bench.parse_clock_samples("") == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}


def test_clock_sampler_stop_reads_its_process_output():
    class FakeProc:
        def __init__(self, text):
            self.text, self.terminated = text, False

        def terminate(self):
            self.terminated = True

        def communicate(self, timeout=None):
            return self.text, None

    sampler = bench.ClockSampler.__new__(bench.ClockSampler)
    sampler.proc = FakeProc("\n".join([_CAPPED, _BUSY, _BUSY]))
    rec = sampler.stop()
    assert sampler.proc.terminated
    assert rec["samples"] == 3 and rec["sm_mhz"] == 2070.0 and rec["reasons"] == ["sw_power_cap"]
    sampler.proc = None
    assert sampler.stop()["reasons"] == ["nvidia-smi unavailable"]


@pytest.mark.parametrize("workload", ["dense", "layouts"])
def test_cpu_baseline_counts_each_cases_own_flops(workload, monkeypatch):
    # the oracle legs report 2 * rows * N * K for the rows they computed, each case with its own N and K
    # (the oracle call itself is stubbed out: only the count is checked here)
    from oracle import oracle as O
    monkeypatch.setattr(O, "gemm_fp8_nt", lambda *a, **k: None)
    cases = bench.build_cases(workload)
    assert len(cases) == 18
    for c in cases:
        M, N, K = (int(x) for x in c.name.split()[-1].split("x"))
        host = {k: v for k, v in c.inputs.items()}
        for r in (16, 100, 5000):
            assert c.oracle(host, r) == 2.0 * min(r, M) * N * K, (c.name, r)
        assert c.flops == 2.0 * M * N * K


def test_cpu_baseline_counts_grouped_layouts_flops():
    # the grouped workloads' oracle legs, on small shapes built by the same case builders: each reports
    # 2 * (rows it computed) * N * K, and the masked leg samples every expert, not only the first
    import numpy as np
    for c in bench.contiguous_cases(shapes=((2, 256, 256, 256),)):
        host = dict(c.inputs)
        N, K = c.inputs["B"].shape[1], c.inputs["B"].shape[2]
        for r in (16, 300, 10 ** 6):
            valid = int((c.inputs["m_indices"][:r] >= 0).sum())
            assert c.oracle(host, r) == 2.0 * valid * N * K
    for c in bench.masked_cases(shapes=((3, 64, 32, 256, 256),)):
        mm = c.inputs["masked_m"].tolist()
        assert len(mm) == 3 and all(m > 0 for m in mm)
        rows = bench.masked_sample_rows(mm, 64, 6)
        assert sorted({r // 64 for r in rows}) == [0, 1, 2]          # every expert is sampled
        assert all(r % 64 < mm[r // 64] for r in rows)               # only valid rows
        host = dict(c.inputs)
        assert c.oracle(host, 6) == 2.0 * len(rows) * 256 * 256
        assert c.oracle(host, 10 ** 6) == 2.0 * sum(mm) * 256 * 256
        assert c.flops == 2.0 * sum(mm) * 256 * 256
    for c in bench.kgrouped_cases(shapes=((2, 128, 128, 256),)):
        sumK = c.inputs["A"].shape[1]
        host = dict(c.inputs)
        for r in (16, 1000):
            assert c.oracle(host, r) == 2.0 * min(r, 128) * 128 * sumK
    assert bench.masked_sample_rows([0, 5, 0], 8, 4) == [8, 9]                  # ceil(4 / 3) rows a group
    assert bench.masked_sample_rows([100, 100], 64, 3) == [0, 1, 64]


def test_default_run_covers_every_workload():
    assert set(bench.WORKLOAD_ORDER) == set(bench.WORKLOADS)
    assert bench.WORKLOAD_ORDER[0] == bench.HEADLINE == "dense"
    for w in ("contiguous", "masked", "kgrouped", "tiny"):
        assert w in bench.WORKLOAD_ORDER
