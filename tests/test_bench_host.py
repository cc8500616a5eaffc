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
    results = mp.Manager().dict()
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
