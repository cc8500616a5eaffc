"""The normal GEMM with transposed operand storage (TN, NN, TT as well as NT), through the C ABI:
A stored [K, M] and/or B stored [K, N], compared with the oracle of the same logical product."""
import numpy as np
import pytest
import torch

import moe_grouped_gemm_tma_gb300 as dg
from moe_grouped_gemm_tma_gb300 import inputs as I
from oracle import oracle as O
from tests.gpu_util import bf16_bits, check_bf16, dev, sentinel_bf16

pytestmark = pytest.mark.gpu

LAYOUTS = [(False, False), (True, False), (False, True), (True, True)]


def run_layout(A, sfa, B, sfb, M, N, a_mn, b_mn):
    A_st = A.t().contiguous() if a_mn else A
    B_st = B.t().contiguous() if b_mn else B
    D = sentinel_bf16(M, N)
    dg.dg_gemm_fp8(dev(A_st), dev(sfa), dev(B_st), dev(sfb), D, a_mn_major=a_mn, b_mn_major=b_mn)
    assert dg.dg_device_status() == 0
    return D


@pytest.mark.parametrize("a_mn,b_mn", LAYOUTS)
@pytest.mark.parametrize("M,N,K", [(128, 256, 512), (208, 272, 384), (512, 1024, 2048), (16, 4096, 1024)])
def test_layout_parity(M, N, K, a_mn, b_mn):
    # ragged M and N (whole 16s, as MN-major storage needs), several tiles and a split-K small-M case
    c = I.make_normal(I.seed_for(6, M + N + K), M, N, K)
    D = run_layout(c.A, c.sfa, c.B, c.sfb, M, N, a_mn, b_mn)
    check_bf16(bf16_bits(D), O.gemm_fp8_nt(c.A, c.sfa, c.B, c.sfb), f"a_mn={a_mn} b_mn={b_mn} {M}x{N}x{K}")


@pytest.mark.parametrize("a_mn,b_mn,bn", [(a, b, bn) for (a, b) in LAYOUTS for bn in (128, 256)] +
                         [(True, False, bn) for bn in (64, 192, 224)])
def test_layout_every_tile_width(a_mn, b_mn, bn, tune):
    # every layout at the tile widths it takes (MN-major B: whole 128-column boxes, so 128 and 256; an
    # MN-major A alone takes every width); ragged M and N
    tune(bn=bn)
    M, N, K = 208, 272, 384
    c = I.make_normal(I.seed_for(6, 5000 + bn), M, N, K)
    D = run_layout(c.A, c.sfa, c.B, c.sfb, M, N, a_mn, b_mn)
    check_bf16(bf16_bits(D), O.gemm_fp8_nt(c.A, c.sfa, c.B, c.sfb), f"a_mn={a_mn} b_mn={b_mn} bn={bn}")


@pytest.mark.parametrize("a_mn,b_mn", LAYOUTS)
def test_layout_integer_exact_bitwise(a_mn, b_mn):
    # unit scales and values in {-1, 0, 1}: every output is an integer <= 256, exact in BF16
    rng = np.random.default_rng(11)
    M, N, K = 256, 512, 256
    codes = np.array([0xB8, 0x00, 0x38], dtype=np.uint8)
    A = torch.from_numpy(rng.choice(codes, size=(M, K)))
    B = torch.from_numpy(rng.choice(codes, size=(N, K)))
    sfa, sfb = torch.ones(M, K // 128), torch.ones(N // 128, K // 128)
    D = run_layout(A, sfa, B, sfb, M, N, a_mn, b_mn)
    np.testing.assert_array_equal(bf16_bits(D), O.gemm_fp8_nt(A, sfa, B, sfb))


def test_mn_major_needs_whole_16s():
    # B stored [K, N] with N = 216: its rows are not a whole number of 16 bytes
    with pytest.raises(dg.DGError):
        dg.dg_gemm_fp8(torch.zeros(64, 128, dtype=torch.uint8, device="cuda"), torch.ones(64, 1, device="cuda"),
                       torch.zeros(128, 216, dtype=torch.uint8, device="cuda"), torch.ones(2, 1, device="cuda"),
                       torch.empty(64, 216, dtype=torch.bfloat16, device="cuda"), b_mn_major=True)
