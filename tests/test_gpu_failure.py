"""The failure path of the bounded device waits, exercised without a GPU fault.

Every wait in the kernels is bounded; when one runs out the kernel records DG_DEVICE_TIMEOUT, drains
the copies and MMAs it has in flight, frees its tensor memory and returns. The test hook
dg_testing_arm_wait_timeout makes exactly that happen on one launch: the launch's waits are bounded by
a few milliseconds and its TMA producer leaves its first stage unfilled, so the MMA issuer's wait on
that stage runs out (nothing ever arrives; nothing faults). The test then checks that the status is
reported once and cleared, and that the next ordinary call in the same process is correct, which it
could not be if the aborted launch had left tensor memory allocated or copies in flight.
"""
import time

import numpy as np
import pytest
import torch

import moe_grouped_gemm_tma_gb300 as dg
from moe_grouped_gemm_tma_gb300 import inputs as I
from oracle import oracle as O
from tests.gpu_util import bf16_bits, check_bf16, dev, sentinel_bf16

pytestmark = pytest.mark.gpu

DG_DEVICE_TIMEOUT = 6


def _normal(c, D):
    dg.dg_gemm_fp8_nt(dev(c.A), dev(c.sfa), dev(c.B), dev(c.sfb), D)


@pytest.mark.parametrize("M,N,K", [(256, 512, 1024), (512, 2112, 2048)])
def test_expired_wait_is_reported_and_the_next_call_is_correct(M, N, K):
    c = I.make_normal(I.seed_for(9, M + N), M, N, K)
    assert dg.dg_device_status() == 0
    dg.dg_testing_arm_wait_timeout(5_000_000)        # 5 ms bound on this launch's waits
    D = sentinel_bf16(M, N)
    t0 = time.perf_counter()
    _normal(c, D)
    assert dg.dg_device_status() == DG_DEVICE_TIMEOUT
    elapsed = time.perf_counter() - t0
    assert elapsed < 5.0, f"the aborted launch took {elapsed:.2f} s"
    assert dg.dg_device_status() == 0                # reported once, then cleared
    # the hook is one-shot: this call runs normally, on the same context
    D2 = sentinel_bf16(M, N)
    _normal(c, D2)
    assert dg.dg_device_status() == 0
    check_bf16(bf16_bits(D2), O.gemm_fp8_nt(c.A, c.sfa, c.B, c.sfb), f"after timeout {M}x{N}x{K}")


def test_grouped_layouts_run_after_an_expired_wait():
    # an aborted launch of one specialisation leaves the others usable too
    c = I.make_normal(I.seed_for(9, 7), 384, 1024, 512)
    dg.dg_testing_arm_wait_timeout(2_000_000)
    _normal(c, sentinel_bf16(384, 1024))
    assert dg.dg_device_status() == DG_DEVICE_TIMEOUT
    G, max_m, N, K = 3, 256, 512, 768
    sizes = [200, 0, 256]
    m = I.make_masked(I.seed_for(9, 8), G, max_m, N, K, sizes, 128)
    D = sentinel_bf16(G, max_m, N)
    dg.dg_m_grouped_masked(dev(m.A), dev(m.sfa), dev(m.B), dev(m.sfb), dev(m.masked_m), D, expected_m=128)
    assert dg.dg_device_status() == 0
    want = O.m_grouped_masked(m.A, m.sfa, m.B, m.sfb, m.masked_m,
                              rows=[g * max_m + r for g in range(G) for r in range(sizes[g])])
    got = bf16_bits(D).reshape(G * max_m, N)
    check_bf16(got[[g * max_m + r for g in range(G) for r in range(sizes[g])]], want, "masked after timeout")


def test_arming_needs_a_positive_limit():
    with pytest.raises(dg.DGError):
        dg.dg_testing_arm_wait_timeout(0)
