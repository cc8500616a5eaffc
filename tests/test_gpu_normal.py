"""GPU parity of the normal GEMM (dg_gemm_fp8_nt) against the CPU oracle on identical seeded inputs."""
import os

import numpy as np
import pytest
import torch

import moe_grouped_gemm_tma_gb300 as dg
from moe_grouped_gemm_tma_gb300 import inputs as I
from oracle import oracle as O
from tests.gpu_util import bf16_bits, bits_to_f64, check_bf16, dev, sample_rows, sentinel_bf16

pytestmark = pytest.mark.gpu


def run_normal(c, D=None):
    if D is None:
        D = sentinel_bf16(c.M, c.N)
    dg.dg_gemm_fp8_nt(dev(c.A), dev(c.sfa), dev(c.B), dev(c.sfb), D)
    assert dg.dg_device_status() == 0
    return D


def test_tiny_config_full_parity():
    # the small workload: M=128, N=256, K=512
    c = I.make_normal(I.seed_for(0), 128, 256, 512)
    D = run_normal(c)
    check_bf16(bf16_bits(D), O.gemm_fp8_nt(c.A, c.sfa, c.B, c.sfb), "tiny")


@pytest.mark.parametrize("M,N,K", [
    (1, 256, 128), (64, 2112, 1024), (200, 2112, 768), (300, 1000, 384), (129, 4096, 256), (512, 7168, 2048),
])
def test_normal_shapes_full_parity(M, N, K):
    c = I.make_normal(I.seed_for(1, M + N + K), M, N, K)
    D = run_normal(c)
    check_bf16(bf16_bits(D), O.gemm_fp8_nt(c.A, c.sfa, c.B, c.sfb), f"{M}x{N}x{K}")


SPECS = [(bn, 1) for bn in (64, 96, 128, 160, 192, 224, 256)] + [(bn, 2) for bn in (128, 160, 192, 224, 256)]


@pytest.mark.parametrize("bn,pair", SPECS)
@pytest.mark.parametrize("M", [200, 520])
def test_every_tile_shape(bn, pair, M, tune):
    # ragged in M (the last row block partial; for CTA pairs also a pair whose second CTA has no rows)
    # and in N, for every tile width, single-CTA and CTA-pair tiles
    tune(bn=bn)
    tune(pair=pair)
    c = I.make_normal(I.seed_for(1, 900 + bn + M), M, 1000, 512)
    D = run_normal(c)
    check_bf16(bf16_bits(D), O.gemm_fp8_nt(c.A, c.sfa, c.B, c.sfb), f"BN={bn} pair={pair}")


@pytest.mark.parametrize("bn,pair", [(64, 1), (128, 1), (192, 1), (256, 2)])
@pytest.mark.parametrize("M", [40, 100])
def test_output_boxes_past_the_last_row(bn, pair, M, tune):
    # fewer rows than one tile, without split-K: the whole-tile staging issues only the TMA store boxes
    # that start inside D (the others lie wholly past its last row)
    tune(bn=bn)
    tune(pair=pair)
    tune(split=1)
    c = I.make_normal(I.seed_for(1, 950 + bn + M), M, 1000, 512)
    D = run_normal(c)
    check_bf16(bf16_bits(D), O.gemm_fp8_nt(c.A, c.sfa, c.B, c.sfb), f"BN={bn} pair={pair} M={M}")


@pytest.mark.parametrize("split", [2, 4, 8])
@pytest.mark.parametrize("M,N,K", [(64, 1000, 4096), (128, 2112, 1024), (100, 512, 3200)])
def test_split_k(split, M, N, K, tune):
    # the standard kernel's split-K: a cluster of `split` CTAs shares each tile's K blocks (unevenly when
    # they do not divide) and reduces the partial sums through distributed shared memory
    tune(split=split, swap=0)
    c = I.make_normal(I.seed_for(1, 700 + split + M + N), M, N, K)
    D = run_normal(c)
    check_bf16(bf16_bits(D), O.gemm_fp8_nt(c.A, c.sfa, c.B, c.sfb), f"split={split}")


def test_integer_exact_bitwise():
    # unit scales and values in {-1, 0, 1}: every output is an integer <= 256, exact in BF16
    rng = np.random.default_rng(5)
    M, N, K = 256, 512, 256
    codes = np.array([0xB8, 0x00, 0x38], dtype=np.uint8)
    A = torch.from_numpy(rng.choice(codes, size=(M, K)))
    B = torch.from_numpy(rng.choice(codes, size=(N, K)))
    sfa, sfb = torch.ones(M, K // 128), torch.ones(N // 128, K // 128)
    D = sentinel_bf16(M, N)
    dg.dg_gemm_fp8_nt(dev(A), dev(sfa), dev(B), dev(sfb), D)
    assert dg.dg_device_status() == 0
    np.testing.assert_array_equal(bf16_bits(D), O.gemm_fp8_nt(A, sfa, B, sfb))


def test_pow2_scale_rules_bitwise():
    c = I.make_normal(I.seed_for(1, 77), 256, 512, 512)
    base = bits_to_f64(bf16_bits(run_normal(c)))
    sfa = c.sfa.clone()
    sfa[5] *= 8.0
    sfb = c.sfb.clone()
    sfb[2] *= 0.25
    c2 = I.NormalCase(c.M, c.N, c.K, c.A, sfa, c.B, sfb)
    got = bits_to_f64(bf16_bits(run_normal(c2)))
    want = base.copy()
    want[5] *= 8.0
    want[:, 256:384] *= 0.25
    np.testing.assert_array_equal(got, want)


def test_k_zero_writes_zeros():
    D = sentinel_bf16(4, 16)
    e = torch.empty(0, dtype=torch.uint8, device="cuda")
    s = torch.empty(0, dtype=torch.float32, device="cuda")
    st = dg.load().dg_gemm_fp8_nt(e.data_ptr(), s.data_ptr(), e.data_ptr(), s.data_ptr(), D.data_ptr(), 4, 16, 0,
                                  torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    assert (D.float() == 0).all()


@pytest.mark.parametrize("N,K", [(2112, 7168), (24576, 1536), (32768, 512), (7168, 16384), (4096, 7168), (7168, 2048)])
def test_dense_workload_sampled_rows(N, K):
    # the dense workload at full size (M in {64, 128, 4096}), in the launch configuration the bench
    # times; the oracle recomputes a sample of rows, including tile-boundary rows
    big = I.make_normal(I.seed_for(1, 0), 4096, N, K)
    for M in (64, 128, 4096):
        c = I.NormalCase(M, N, K, big.A[:M], big.sfa[:M], big.B, big.sfb)
        D = run_normal(c)
        rows = sample_rows(M, 24, seed=M + N + K)
        want = O.gemm_fp8_nt(c.A, c.sfa, c.B, c.sfb, rows=rows)
        check_bf16(bf16_bits(D)[rows], want, f"{M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [
    (1, 256, 128), (17, 1000, 512), (33, 200, 384), (50, 4096, 2048), (64, 7168, 2048), (100, 2112, 1024),
    (128, 4096, 7168), (64, 2112, 7168), (32, 24576, 1536), (128, 32768, 512),
])
def test_decode_small_m(M, N, K, tune):
    # the few-row (decode) kernel (D^T = B . A^T on the tensor cores), with the tile height and split-K
    # clusters it picks itself, on ragged M and N
    tune(swap=1)
    c = I.make_normal(I.seed_for(1, 500 + M + N + K), M, N, K)
    D = run_normal(c)
    check_bf16(bf16_bits(D), O.gemm_fp8_nt(c.A, c.sfa, c.B, c.sfb), f"decode {M}x{N}x{K}")


@pytest.mark.parametrize("split", [1, 2, 4, 8])
@pytest.mark.parametrize("M", [20, 64, 120])
def test_decode_every_split(M, split, tune):
    # each tile height (32, 64, 128 rows) with each split-K cluster size, K blocks shared unevenly
    tune(split=split, swap=1)
    c = I.make_normal(I.seed_for(1, 600 + M + split), M, 1000, 1408)
    D = run_normal(c)
    check_bf16(bf16_bits(D), O.gemm_fp8_nt(c.A, c.sfa, c.B, c.sfb), f"decode M={M} split={split}")


def test_decode_integer_exact_bitwise(tune):
    tune(swap=1)
    rng = np.random.default_rng(21)
    M, N, K = 96, 512, 512
    codes = np.array([0xB8, 0x00, 0x38], dtype=np.uint8)
    A = torch.from_numpy(rng.choice(codes, size=(M, K)))
    B = torch.from_numpy(rng.choice(codes, size=(N, K)))
    sfa, sfb = torch.ones(M, K // 128), torch.ones(N // 128, K // 128)
    D = sentinel_bf16(M, N)
    dg.dg_gemm_fp8_nt(dev(A), dev(sfa), dev(B), dev(sfb), D)
    assert dg.dg_device_status() == 0
    np.testing.assert_array_equal(bf16_bits(D), O.gemm_fp8_nt(A, sfa, B, sfb))
