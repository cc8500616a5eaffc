"""The block-scaled (UE8M0) normal GEMM for power-of-two scales, through the C ABI: compared with the
oracle of the same product, bitwise on integer-exact inputs, and the report of a scale that is not a
power of two."""
import numpy as np
import pytest
import torch

import moe_grouped_gemm_tma_gb300 as dg
from moe_grouped_gemm_tma_gb300 import inputs as I
from oracle import oracle as O
from tests.gpu_util import bf16_bits, check_bf16, dev, pack_ue8m0, sentinel_bf16

pytestmark = pytest.mark.gpu


def run_ue8m0(A, sfa, B, sfb, M, N):
    D = sentinel_bf16(M, N)
    dg.dg_gemm_fp8_nt_ue8m0(dev(A), dev(sfa), dev(B), dev(sfb), D)
    return D


@pytest.mark.parametrize("bn", [0, 128, 192, 224, 256])
@pytest.mark.parametrize("M,N,K", [(128, 256, 512), (200, 1000, 768), (1, 2112, 1024), (520, 4096, 2048)])
def test_ue8m0_parity(M, N, K, bn, tune):
    # power-of-two block scales (amax/448 rounded up to a power of two); ragged M and N; every tile width
    if bn:
        tune(bn=bn)
    c = I.make_normal(I.seed_for(7, M + N + K), M, N, K, pow2=True)
    assert bool((torch.frexp(c.sfa)[0] == 0.5).all()) and bool((torch.frexp(c.sfb)[0] == 0.5).all())
    D = run_ue8m0(c.A, c.sfa, c.B, c.sfb, M, N)
    assert dg.dg_device_status() == 0
    check_bf16(bf16_bits(D), O.gemm_fp8_nt(c.A, c.sfa, c.B, c.sfb), f"ue8m0 BN={bn} {M}x{N}x{K}")


@pytest.mark.parametrize("bn", [0, 256])
def test_ue8m0_rows_short_of_one_tile(bn, tune):
    # 40 rows and 4 K blocks (no split-K): the output boxes of rows 40..127 are not issued
    if bn:
        tune(bn=bn)
    c = I.make_normal(I.seed_for(7, 4040 + bn), 40, 1000, 512, pow2=True)
    D = run_ue8m0(c.A, c.sfa, c.B, c.sfb, 40, 1000)
    assert dg.dg_device_status() == 0
    check_bf16(bf16_bits(D), O.gemm_fp8_nt(c.A, c.sfa, c.B, c.sfb), f"ue8m0 BN={bn} 40x1000x512")


def test_ue8m0_integer_exact_bitwise():
    # values in {-1, 0, 1} and power-of-two scales 2^-2 .. 2^2 per block: every 32-element slice sums
    # exactly, every output is a multiple of 2^-4 below 2^13, so the FP32 accumulation is exact and the
    # only rounding is the final one to BF16, which the oracle takes from the exact value too
    rng = np.random.default_rng(13)
    M, N, K = 256, 384, 512
    codes = np.array([0xB8, 0x00, 0x38], dtype=np.uint8)
    A = torch.from_numpy(rng.choice(codes, size=(M, K)))
    B = torch.from_numpy(rng.choice(codes, size=(N, K)))
    sfa = torch.from_numpy(np.ldexp(1.0, rng.integers(-2, 3, size=(M, K // 128))).astype(np.float32))
    sfb = torch.from_numpy(np.ldexp(1.0, rng.integers(-2, 3, size=(N // 128, K // 128))).astype(np.float32))
    D = run_ue8m0(A, sfa, B, sfb, M, N)
    assert dg.dg_device_status() == 0
    np.testing.assert_array_equal(bf16_bits(D), O.gemm_fp8_nt(A, sfa, B, sfb))


def test_ue8m0_reports_non_power_of_two_scales():
    c = I.make_normal(I.seed_for(7, 1), 128, 256, 256)      # FP32 scales amax/448: not powers of two
    run_ue8m0(c.A, c.sfa, c.B, c.sfb, 128, 256)
    assert dg.dg_device_status() == 7                       # DG_SCALE_NOT_UE8M0
    assert dg.dg_device_status() == 0                       # reported once, then cleared


@pytest.mark.parametrize("bad", [float("inf"), float("nan")])
def test_ue8m0_reports_infinite_or_nan_scale(bad):
    # an exponent byte of all ones is not a power of two that UE8M0 can hold (it stands for NaN there)
    c = I.make_normal(I.seed_for(7, 3), 128, 256, 256, pow2=True)
    sfa = c.sfa.clone()
    sfa[5, 1] = bad
    run_ue8m0(c.A, sfa, c.B, c.sfb, 128, 256)
    assert dg.dg_device_status() == 7
    assert dg.dg_device_status() == 0


@pytest.mark.parametrize("split", [2, 4, 8])
@pytest.mark.parametrize("M,N,K", [(64, 1000, 3200), (100, 2112, 1024)])
def test_ue8m0_split_k(split, M, N, K, tune):
    # a cluster of `split` CTAs shares each tile's K blocks (unevenly when they do not divide); each
    # accumulates its range in TMEM and the FP32 partials are reduced through distributed shared memory
    tune(split=split)
    c = I.make_normal(I.seed_for(7, 50 + split + M), M, N, K, pow2=True)
    D = run_ue8m0(c.A, c.sfa, c.B, c.sfb, M, N)
    assert dg.dg_device_status() == 0
    check_bf16(bf16_bits(D), O.gemm_fp8_nt(c.A, c.sfa, c.B, c.sfb), f"ue8m0 split={split} {M}x{N}x{K}")


def test_ue8m0_split_k_reports_non_power_of_two_scales(tune):
    tune(split=4)
    c = I.make_normal(I.seed_for(7, 2), 64, 512, 2048)
    run_ue8m0(c.A, c.sfa, c.B, c.sfb, 64, 512)
    assert dg.dg_device_status() == 7


@pytest.mark.parametrize("bn", [128, 256])
@pytest.mark.parametrize("M,N,K", [(200, 1000, 768), (520, 4096, 2048), (256, 264, 384)])
def test_ue8m0_cta_pairs(M, N, K, bn, tune):
    # 256-row tiles over a CTA pair (cta_group::2): each CTA writes the exponents of its own rows and all
    # of B's; ragged M leaves the second CTA of the last pair partly or wholly past M
    tune(pair=2)
    tune(bn=bn)
    c = I.make_normal(I.seed_for(7, 70 + bn + M), M, N, K, pow2=True)
    D = run_ue8m0(c.A, c.sfa, c.B, c.sfb, M, N)
    assert dg.dg_device_status() == 0
    check_bf16(bf16_bits(D), O.gemm_fp8_nt(c.A, c.sfa, c.B, c.sfb), f"ue8m0 pair BN={bn} {M}x{N}x{K}")


def test_ue8m0_cta_pairs_integer_exact_bitwise(tune):
    tune(pair=2)
    rng = np.random.default_rng(17)
    M, N, K = 512, 384, 512
    codes = np.array([0xB8, 0x00, 0x38], dtype=np.uint8)
    A = torch.from_numpy(rng.choice(codes, size=(M, K)))
    B = torch.from_numpy(rng.choice(codes, size=(N, K)))
    sfa = torch.from_numpy(np.ldexp(1.0, rng.integers(-2, 3, size=(M, K // 128))).astype(np.float32))
    sfb = torch.from_numpy(np.ldexp(1.0, rng.integers(-2, 3, size=(N // 128, K // 128))).astype(np.float32))
    D = run_ue8m0(A, sfa, B, sfb, M, N)
    assert dg.dg_device_status() == 0
    np.testing.assert_array_equal(bf16_bits(D), O.gemm_fp8_nt(A, sfa, B, sfb))


@pytest.mark.parametrize("N,K", [(2112, 7168), (24576, 1536), (32768, 512), (7168, 16384), (4096, 7168), (7168, 2048)])
def test_ue8m0_workload_sampled_rows(N, K):
    # the block-scaled workload at full size (M in {64, 128, 4096}: split-K clusters for few rows, CTA
    # pairs for M = 4096), as the bench runs it; the oracle recomputes a sample of rows
    from tests.gpu_util import sample_rows
    big = I.make_normal(I.seed_for(1, 0), 4096, N, K, pow2=True)
    for M in (64, 128, 4096):
        A, sfa = big.A[:M], big.sfa[:M]
        D = run_ue8m0(A, sfa, big.B, big.sfb, M, N)
        assert dg.dg_device_status() == 0
        rows = sample_rows(M, 24, seed=M + N + K)
        want = O.gemm_fp8_nt(A, sfa, big.B, big.sfb, rows=rows)
        check_bf16(bf16_bits(D)[rows], want, f"ue8m0 {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(1, 256, 128), (200, 1000, 640), (129, 2112, 1408), (64, 4096, 7168),
                                   (520, 264, 896), (4096, 2112, 1536)])
def test_ue8m0_packed_matches_fp32_scales_bitwise(M, N, K):
    # the packed format carries the same exponents, so the two entry points run the same tensor-core
    # arithmetic: bit-identical outputs, and the oracle agrees within the tolerance
    c = I.make_normal(I.seed_for(7, 500 + M + N + K), M, N, K, pow2=True)
    D_f32 = run_ue8m0(c.A, c.sfa, c.B, c.sfb, M, N)
    assert dg.dg_device_status() == 0
    D_pk = sentinel_bf16(M, N)
    dg.dg_gemm_fp8_nt_ue8m0_packed(dev(c.A), dev(pack_ue8m0(c.sfa)), dev(c.B), dev(pack_ue8m0(c.sfb)), D_pk)
    assert dg.dg_device_status() == 0
    np.testing.assert_array_equal(bf16_bits(D_pk), bf16_bits(D_f32))
    rows = np.unique(np.linspace(0, M - 1, min(M, 48)).astype(int))
    want = O.gemm_fp8_nt(c.A, c.sfa, c.B, c.sfb, rows=rows)
    check_bf16(bf16_bits(D_pk)[rows], want, f"ue8m0 packed {M}x{N}x{K}")


def test_ue8m0_packed_rejects_wrong_shapes():
    c = I.make_normal(I.seed_for(7, 3), 128, 256, 640, pow2=True)
    D = sentinel_bf16(128, 256)
    with pytest.raises(ValueError):
        dg.dg_gemm_fp8_nt_ue8m0_packed(dev(c.A), dev(pack_ue8m0(c.sfa))[:, :1].contiguous(), dev(c.B),
                                       dev(pack_ue8m0(c.sfb)), D)
    with pytest.raises(TypeError):
        dg.dg_gemm_fp8_nt_ue8m0_packed(dev(c.A), dev(c.sfa), dev(c.B), dev(c.sfb), D)
