"""Seeded random shapes through every entry point, with the library's own choice of tile width, CTA
split, swapped-operand kernel and staging path (no overrides), compared element by element with the
CPU oracle. The shapes are drawn so that most are ragged in M and N (N a multiple of 8, K of 128) and
small enough for the oracle to take every row."""
import numpy as np
import pytest
import torch

import moe_grouped_gemm_tma_gb300 as dg
from moe_grouped_gemm_tma_gb300 import inputs as I
from oracle import oracle as O
from tests.gpu_util import SENTINEL, bf16_bits, check_bf16, check_f32, dev, sentinel_bf16

pytestmark = pytest.mark.gpu

RNG_SEED = 0x5EED


def _shapes(count, seed):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(count):
        m = int(rng.choice([1, 7, 64, 100, 128, 129, 200, 257, 384, 520, 700]))
        n = int(8 * rng.integers(1, 400))            # 8 .. 3192
        k = int(128 * rng.integers(1, 24))           # 128 .. 2944
        out.append((m, n, k))
    return out


@pytest.mark.parametrize("idx,shape", list(enumerate(_shapes(16, RNG_SEED))))
def test_random_normal(idx, shape):
    M, N, K = shape
    c = I.make_normal(I.seed_for(20, idx), M, N, K)
    D = sentinel_bf16(M, N)
    dg.dg_gemm_fp8_nt(dev(c.A), dev(c.sfa), dev(c.B), dev(c.sfb), D)
    assert dg.dg_device_status() == 0
    check_bf16(bf16_bits(D), O.gemm_fp8_nt(c.A, c.sfa, c.B, c.sfb), f"normal {M}x{N}x{K}")


@pytest.mark.parametrize("idx,shape", list(enumerate(_shapes(12, RNG_SEED + 1))))
def test_random_ue8m0(idx, shape):
    M, N, K = shape
    c = I.make_normal(I.seed_for(21, idx), M, N, K, pow2=True)
    D = sentinel_bf16(M, N)
    dg.dg_gemm_fp8_nt_ue8m0(dev(c.A), dev(c.sfa), dev(c.B), dev(c.sfb), D)
    assert dg.dg_device_status() == 0
    check_bf16(bf16_bits(D), O.gemm_fp8_nt(c.A, c.sfa, c.B, c.sfb), f"ue8m0 {M}x{N}x{K}")


@pytest.mark.parametrize("idx", range(8))
def test_random_contiguous(idx):
    rng = np.random.default_rng(RNG_SEED + 100 + idx)
    G = int(rng.integers(1, 6))
    sizes = [int(x) for x in rng.choice([0, 1, 60, 128, 129, 300, 511], size=G)]
    if sum(sizes) == 0:
        sizes[0] = 77
    N = int(8 * rng.integers(1, 300))
    K = int(128 * rng.integers(1, 16))
    c = I.make_contiguous(I.seed_for(22, idx), G, N, K, sizes)
    D = sentinel_bf16(c.Mt, N)
    dg.dg_m_grouped_contiguous(dev(c.A), dev(c.sfa), dev(c.B), dev(c.sfb), dev(c.m_indices), D)
    assert dg.dg_device_status() == 0
    got = bf16_bits(D)
    valid = c.m_indices.numpy() >= 0
    want = O.m_grouped_contiguous(c.A, c.sfa, c.B, c.sfb, c.m_indices)
    check_bf16(got[valid], want[valid], f"contiguous G={G} sizes={sizes} N={N} K={K}")


@pytest.mark.parametrize("idx", range(8))
def test_random_masked(idx):
    rng = np.random.default_rng(RNG_SEED + 200 + idx)
    G = int(rng.integers(1, 9))
    max_m = int(rng.choice([128, 192, 256, 384, 512]))
    masked = [int(x) for x in rng.integers(0, max_m + 1, size=G)]
    expected = int(rng.choice([0, 32, 64, 128]))
    N = int(8 * rng.integers(1, 300))
    K = int(128 * rng.integers(1, 16))
    c = I.make_masked(I.seed_for(23, idx), G, max_m, N, K, masked, expected)
    D = sentinel_bf16(G, max_m, N)
    dg.dg_m_grouped_masked(dev(c.A), dev(c.sfa), dev(c.B), dev(c.sfb), dev(c.masked_m), D, expected)
    assert dg.dg_device_status() == 0
    got = bf16_bits(D).reshape(G * max_m, N)
    valid = np.zeros(G * max_m, dtype=bool)
    for g, m in enumerate(masked):
        valid[g * max_m: g * max_m + m] = True
    assert (got[~valid] == SENTINEL).all(), "rows past masked_m were written"
    rows = np.nonzero(valid)[0]
    if rows.size:
        want = O.m_grouped_masked(c.A, c.sfa, c.B, c.sfb, c.masked_m, rows=rows)
        check_bf16(got[rows], want, f"masked G={G} max_m={max_m} masked={masked} N={N} K={K}")


@pytest.mark.parametrize("idx", range(6))
def test_random_kgrouped(idx):
    rng = np.random.default_rng(RNG_SEED + 300 + idx)
    G = int(rng.integers(1, 5))
    ks = [int(128 * x) for x in rng.integers(0, 8, size=G)]
    M = int(rng.choice([64, 128, 200, 300]))
    N = int(8 * rng.integers(1, 60))
    c = I.make_kgrouped(I.seed_for(24, idx), G, M, N, ks)
    D = dev(c.D_in)
    dg.dg_k_grouped_wgrad(dev(c.A), dev(c.sfa), dev(c.B), dev(c.sfb), c.ks, D)
    assert dg.dg_device_status() == 0
    got = D.cpu().numpy()
    want = O.k_grouped_wgrad(c.A, c.sfa, c.B, c.sfb, c.ks, c.D_in)
    for g in range(G):
        check_f32(got[g], want[g], f"k-grouped G={G} ks={ks} M={M} N={N} g={g}")
