"""GPU parity of the MoE layouts against the CPU oracle on identical seeded inputs: m-grouped
contiguous (dg_m_grouped_contiguous), m-grouped masked (dg_m_grouped_masked, with sentinel checks of
every row past masked_m) and the k-grouped FP32 weight gradient (dg_k_grouped_wgrad)."""
import numpy as np
import pytest
import torch

import moe_grouped_gemm_tma_gb300 as dg
from moe_grouped_gemm_tma_gb300 import inputs as I
from oracle import oracle as O
from tests.gpu_util import SENTINEL, bf16_bits, check_bf16, check_f32, dev, sample_rows, sentinel_bf16

pytestmark = pytest.mark.gpu


# ------------------------------------------------------------------------------------------ contiguous
def run_contiguous(c, m_indices=None):
    mi = c.m_indices if m_indices is None else m_indices
    D = sentinel_bf16(c.Mt, c.N)
    dg.dg_m_grouped_contiguous(dev(c.A), dev(c.sfa), dev(c.B), dev(c.sfb), dev(mi), D)
    assert dg.dg_device_status() == 0
    return bf16_bits(D)


@pytest.mark.parametrize("G,group_m,N,K", [
    (3, [130, 0, 77], 256, 256),
    (4, [128, 1, 255, 300], 2112, 512),
    (2, [600, 50], 1000, 384),
])
def test_contiguous_small_full_parity(G, group_m, N, K):
    c = I.make_contiguous(I.seed_for(2, sum(group_m)), G, N, K, group_m)
    got = run_contiguous(c)
    valid = c.m_indices.numpy() >= 0
    want = O.m_grouped_contiguous(c.A, c.sfa, c.B, c.sfb, c.m_indices)
    check_bf16(got[valid], want[valid], f"contiguous G={G}")


@pytest.mark.parametrize("bn", [128, 160, 192, 224, 256])
def test_contiguous_every_tile_width(bn, tune):
    # every tile width the contiguous layout takes, against a ragged N (264: a partial last column block
    # at every width) and experts whose last row block is partly padding
    tune(bn=bn)
    G, group_m, N, K = 3, [130, 0, 77], 264, 384
    c = I.make_contiguous(I.seed_for(2, 600 + bn), G, N, K, group_m)
    got = run_contiguous(c)
    valid = c.m_indices.numpy() >= 0
    want = O.m_grouped_contiguous(c.A, c.sfa, c.B, c.sfb, c.m_indices)
    check_bf16(got[valid], want[valid], f"contiguous bn={bn}")


def test_contiguous_skips_blocks_that_start_with_padding():
    c = I.make_contiguous(I.seed_for(2, 5), 2, 256, 256, [128, 128])
    mi = c.m_indices.clone()
    mi[128:256] = -1   # the second expert's whole block marked as padding
    got = run_contiguous(c, mi)
    assert (got[128:256] == SENTINEL).all()
    want = O.gemm_fp8_nt(c.A[:128], c.sfa[:128], c.B[0], c.sfb[0])
    check_bf16(got[:128], want, "first block")


@pytest.mark.parametrize("G,base,N,K", [(4, 4096, 7168, 2048), (8, 8192, 4096, 7168)])
def test_contiguous_workload_sampled_rows(G, base, N, K):
    # the MoE prefill / training-forward workload at full size; rows sampled around every expert boundary
    sizes = I.contiguous_group_sizes(I.seed_for(2, G), G, base)
    c = I.make_contiguous(I.seed_for(2, G), G, N, K, sizes)
    got = run_contiguous(c)
    mi = c.m_indices.numpy()
    starts = np.concatenate([[0], np.cumsum([(m + 127) // 128 * 128 for m in sizes])[:-1]])
    must = [int(s + d) for s, m in zip(starts, sizes) for d in (0, 1, 127, 128, m - 1)]
    rows = sample_rows(c.Mt, 64, seed=G + base, must=must)
    rows = rows[mi[rows] >= 0]
    want = O.m_grouped_contiguous(c.A, c.sfa, c.B, c.sfb, c.m_indices, rows=rows)
    check_bf16(got[rows], want, f"contiguous G={G} base={base}")


# ------------------------------------------------------------------------------------------ masked
def run_masked(c, masked_m=None, expected_m=0):
    mm = c.masked_m if masked_m is None else masked_m
    D = sentinel_bf16(c.G, c.max_m, c.N)
    dg.dg_m_grouped_masked(dev(c.A), dev(c.sfa), dev(c.B), dev(c.sfb), dev(mm), D, expected_m=expected_m)
    assert dg.dg_device_status() == 0
    return bf16_bits(D).reshape(c.G * c.max_m, c.N)


def _check_masked(c, got, mm_list, rows=None):
    valid = np.zeros(c.G * c.max_m, dtype=bool)
    for g, m in enumerate(mm_list):
        valid[g * c.max_m: g * c.max_m + min(max(m, 0), c.max_m)] = True
    assert (got[~valid] == SENTINEL).all(), f"{(got[~valid] != SENTINEL).any(axis=1).sum()} masked rows written"
    if rows is None:
        rows = np.nonzero(valid)[0]
    else:
        rows = rows[valid[rows]]
    want = O.m_grouped_masked(c.A, c.sfa, c.B, c.sfb, c.masked_m, rows=rows)
    check_bf16(got[rows], want, "masked")


@pytest.mark.parametrize("G,max_m,masked,N,K", [
    (3, 256, [10, 0, 256], 256, 256),
    (4, 192, [129, 128, 127, 1], 2112, 512),
    (2, 64, [64, 33], 4096, 384),
])
def test_masked_small_full_parity_and_untouched_rows(G, max_m, masked, N, K):
    c = I.make_masked(I.seed_for(3, G * max_m), G, max_m, N, K, masked)
    got = run_masked(c)
    _check_masked(c, got, masked)


@pytest.mark.parametrize("kernel", ["standard", "decode"])
def test_masked_largest_expert_count(kernel, tune):
    # the largest expert count the call takes (1024): the device-side tile count and its prefix scan over
    # every expert, with empty experts and experts at max_m among them
    tune(swap=1 if kernel == "decode" else 0)
    G, max_m, N, K = 1024, 32, 128, 256
    rng = np.random.default_rng(11)
    masked = [int(x) for x in rng.integers(0, max_m + 1, size=G)]
    c = I.make_masked(I.seed_for(3, 7000), G, max_m, N, K, masked)
    got = run_masked(c, expected_m=16)
    _check_masked(c, got, masked)


def test_masked_all_empty_and_over_max():
    c = I.make_masked(I.seed_for(3, 1), 2, 128, 256, 256, [0, 0])
    got = run_masked(c)
    assert (got == SENTINEL).all()
    over = torch.tensor([1000, 3], dtype=torch.int32)
    c2 = I.MaskedCase(c.G, c.max_m, c.N, c.K, 0, c.A, c.sfa, c.B, c.sfb, over)
    got = run_masked(c2)
    _check_masked(c2, got, [128, 3])


@pytest.mark.parametrize("bn,pair", [(64, 1), (128, 1), (192, 1), (224, 1), (256, 1), (128, 2), (256, 2)])
def test_masked_every_tile_shape(bn, pair, tune):
    tune(bn=bn)
    tune(pair=pair)
    c = I.make_masked(I.seed_for(3, bn), 3, 384, 1000, 384, [300, 5, 129])
    _check_masked(c, run_masked(c), [300, 5, 129])


@pytest.mark.parametrize("bn", [64, 128])
@pytest.mark.parametrize("split", [2, 4, 8])
def test_masked_split_k(bn, split, tune):
    # clusters of `split` CTAs share a tile's K blocks; one cluster per possible tile, the ones past the
    # device-side tile count have no work; an empty expert and rows past masked_m stay untouched
    tune(bn=bn)
    tune(split=split)
    sizes = [300, 0, 129]
    c = I.make_masked(I.seed_for(3, 100 + bn + split), 3, 384, 256, 1024, sizes)
    _check_masked(c, run_masked(c), sizes)


@pytest.mark.parametrize("expected_m", [24, 64, 128])
@pytest.mark.parametrize("split", [None, 1, 2, 4, 8])
def test_masked_decode_kernel(expected_m, split, tune):
    # the few-row (decode) kernel: tiles of 32 / 64 / 128 rows per expert from expected_m, split-K
    # clusters of each size, an expert with more rows than a tile (several row blocks, counted on the
    # device), an empty expert, max_m not a multiple of the tile height and N not a multiple of 128
    tune(swap=1)
    if split is not None:
        tune(split=split)
    G, max_m, N, K = 4, 300, 1000, 1024
    sizes = [expected_m, 0, max_m, 3]
    c = I.make_masked(I.seed_for(3, 300 + expected_m + (split or 0)), G, max_m, N, K, sizes, expected_m)
    _check_masked(c, run_masked(c, expected_m=expected_m), sizes)


@pytest.mark.parametrize("kernel", ["decode", "standard"])
def test_masked_few_rows_both_kernels_agree_with_the_oracle(kernel, tune):
    # the same decode-shaped problem through the decode kernel and through the standard masked kernel
    tune(swap=0 if kernel == "standard" else 1)
    sizes = [45, 64, 0, 17, 63, 1]
    c = I.make_masked(I.seed_for(3, 77), 6, 128, 2112, 2048, sizes, 64)
    _check_masked(c, run_masked(c, expected_m=64), sizes)


@pytest.mark.parametrize("G,max_m,expected_m,N,K", [
    (16, 256, 64, 4096, 7168), (4, 512, 128, 7168, 2048), (1, 1024, 256, 4096, 7168), (2, 256, 256, 7168, 2048),
    (1, 256, 64, 4096, 7168), (2, 512, 128, 7168, 2048), (4, 256, 64, 4096, 7168),
])
def test_masked_workload_sampled_rows(G, max_m, expected_m, N, K):
    # the MoE decode workload at full size; every row past masked_m is sentinel-checked
    sizes = I.masked_sizes(I.seed_for(3, G), G, expected_m, max_m)
    c = I.make_masked(I.seed_for(3, G), G, max_m, N, K, sizes, expected_m)
    got = run_masked(c, expected_m=expected_m)
    must = [g * max_m + d for g, m in enumerate(sizes) for d in (0, m - 1) if m > 0]
    rows = sample_rows(G * max_m, 48, seed=G * max_m, must=must)
    _check_masked(c, got, sizes, rows=rows)


# ------------------------------------------------------------------------------------------ k-grouped
def run_kgrouped(c):
    D = dev(c.D_in)
    dg.dg_k_grouped_wgrad(dev(c.A), dev(c.sfa), dev(c.B), dev(c.sfb), c.ks, D)
    assert dg.dg_device_status() == 0
    return D.cpu().numpy()


@pytest.mark.parametrize("bn,pair", [(0, 1), (128, 1), (192, 1), (224, 1), (256, 1), (0, 2)])
@pytest.mark.parametrize("ks,M,N", [([256, 0, 384], 200, 264), ([128], 128, 128), ([512, 128, 1024, 256], 300, 1000)])
def test_kgrouped_small_full_parity(ks, M, N, bn, pair, tune):
    tune(pair=pair)
    if bn:
        tune(bn=bn)
    c = I.make_kgrouped(I.seed_for(4, sum(ks) + M), len(ks), M, N, ks)
    got = run_kgrouped(c)
    want = O.k_grouped_wgrad(c.A, c.sfa, c.B, c.sfb, c.ks, c.D_in)
    for g in range(len(ks)):
        check_f32(got[g], want[g], f"k-grouped g={g}")
        if ks[g] == 0:   # an expert with no tokens leaves its gradient buffer bit-for-bit unchanged
            np.testing.assert_array_equal(got[g], c.D_in[g].numpy())


@pytest.mark.parametrize("bn", [0, 224])
@pytest.mark.parametrize("G,M,N,seed", [(32, 136, 200, 1), (128, 128, 64, 2)])
def test_kgrouped_many_short_experts(G, M, N, seed, bn, tune):
    # many experts with K windows of 0-3 blocks: scale patches shorter than four K blocks, windows that
    # start at any K block, empty experts, up to the largest expert count the call takes
    if bn:
        tune(bn=bn)
    rng = np.random.default_rng(seed)
    ks = [int(k) for k in rng.integers(0, 4, size=G) * 128]
    ks[0] = max(ks[0], 128)
    c = I.make_kgrouped(I.seed_for(4, 1000 + seed), G, M, N, ks)
    got = run_kgrouped(c)
    want = O.k_grouped_wgrad(c.A, c.sfa, c.B, c.sfb, c.ks, c.D_in)
    for g in range(G):
        check_f32(got[g], want[g], f"k-grouped G={G} g={g}")
        if ks[g] == 0:
            np.testing.assert_array_equal(got[g], c.D_in[g].numpy())


def test_kgrouped_integer_exact_bitwise():
    rng = np.random.default_rng(9)
    M, N, ks = 256, 256, [256, 128]
    vals = np.array([0x00, 0x38, 0x40, 0x44, 0x48, 0xB8, 0xC0, 0xC4, 0xC8], dtype=np.uint8)
    A = torch.from_numpy(rng.choice(vals, size=(M, sum(ks))))
    B = torch.from_numpy(rng.choice(vals, size=(N, sum(ks))))
    sfa, sfb = torch.ones(M, 3), torch.ones(N, 3)
    D_in = torch.from_numpy(rng.integers(-100, 100, size=(2, M, N)).astype(np.float32))
    c = I.KGroupedCase(2, M, N, ks, A, sfa, B, sfb, D_in)
    np.testing.assert_array_equal(run_kgrouped(c), O.k_grouped_wgrad(A, sfa, B, sfb, ks, D_in))


@pytest.mark.parametrize("G,M,N", [(4, 7168, 4096), (8, 2048, 7168)])
def test_kgrouped_workload_sampled_rows(G, M, N):
    # the MoE weight-gradient workload at full size (token counts per expert around 4096)
    ks = I.kgrouped_sizes(I.seed_for(4, G), G, 4096)
    c = I.make_kgrouped(I.seed_for(4, G), G, M, N, ks)
    got = run_kgrouped(c)
    rows = sample_rows(M, 16, seed=G + M)
    want = O.k_grouped_wgrad(c.A, c.sfa, c.B, c.sfb, c.ks, c.D_in, rows=rows)
    for g in range(G):
        check_f32(got[g][rows], want[g], f"k-grouped g={g}")


# --------------------------------------------------------------------------- dense weight gradient
@pytest.mark.parametrize("accumulate", [True, False])
@pytest.mark.parametrize("M,N,K", [(200, 264, 384), (128, 128, 128), (300, 1000, 1024), (1024, 2048, 4096)])
def test_dense_wgrad_parity(M, N, K, accumulate):
    # the single-expert weight gradient, accumulating (D += X^T dY) or overwriting (D = X^T dY)
    c = I.make_kgrouped(I.seed_for(5, M + N + K), 1, M, N, [K])
    D = dev(c.D_in[0]) if accumulate else torch.full((M, N), float("nan"), device="cuda")
    dg.dg_wgrad_fp8_nt(dev(c.A), dev(c.sfa), dev(c.B), dev(c.sfb), D, accumulate=accumulate)
    assert dg.dg_device_status() == 0
    D_in = c.D_in if accumulate else torch.zeros(1, M, N)
    want = O.k_grouped_wgrad(c.A, c.sfa, c.B, c.sfb, [K], D_in)[0]
    check_f32(D.cpu().numpy(), want, f"dense wgrad accumulate={accumulate}")


@pytest.mark.parametrize("bn", [128, 192, 224, 256])
def test_dense_wgrad_overwrite_every_tile_width(bn, tune):
    # the overwriting form at every tile width: 32-column TMEM load batches where the warpgroup's columns
    # start on a 32-column boundary, 16-column ones at BN = 224; ragged M and N (N % 16 == 8)
    tune(bn=bn)
    M, N, K = 200, 264, 512
    c = I.make_kgrouped(I.seed_for(5, bn), 1, M, N, [K])
    D = torch.full((M, N), float("nan"), device="cuda")
    dg.dg_wgrad_fp8_nt(dev(c.A), dev(c.sfa), dev(c.B), dev(c.sfb), D, accumulate=False)
    assert dg.dg_device_status() == 0
    want = O.k_grouped_wgrad(c.A, c.sfa, c.B, c.sfb, [K], torch.zeros(1, M, N))[0]
    check_f32(D.cpu().numpy(), want, f"dense wgrad overwrite bn={bn}")


def test_dense_wgrad_k_zero():
    M, N = 130, 64
    D = torch.full((M, N), 3.0, device="cuda")
    dg.dg_wgrad_fp8_nt(torch.empty(M, 0, dtype=torch.uint8, device="cuda"), torch.empty(M, 0, device="cuda"),
                       torch.empty(N, 0, dtype=torch.uint8, device="cuda"), torch.empty(N, 0, device="cuda"), D,
                       accumulate=True)
    assert dg.dg_device_status() == 0
    assert bool((D == 3.0).all())          # nothing to add: unchanged
    dg.dg_wgrad_fp8_nt(torch.empty(M, 0, dtype=torch.uint8, device="cuda"), torch.empty(M, 0, device="cuda"),
                       torch.empty(N, 0, dtype=torch.uint8, device="cuda"), torch.empty(N, 0, device="cuda"), D,
                       accumulate=False)
    assert dg.dg_device_status() == 0
    assert bool((D == 0.0).all())          # the empty product, stored


@pytest.mark.parametrize("kernel", ["standard", "decode"])
def test_masked_replayed_from_a_cuda_graph(kernel, tune):
    # decode runs the masked layout under CUDA graphs: one capture, replayed with new per-expert counts
    # written into the same device buffer; every argument the host sees stays fixed
    tune(swap=1 if kernel == "decode" else 0)
    G, max_m, N, K = 4, 256, 1024, 512
    first = [100, 0, 256, 37]
    c = I.make_masked(I.seed_for(3, 900), G, max_m, N, K, first, 128)
    dA, dsfa, dB, dsfb = dev(c.A), dev(c.sfa), dev(c.B), dev(c.sfb)
    mm = dev(c.masked_m)
    D = sentinel_bf16(G, max_m, N)
    dg.dg_m_grouped_masked(dA, dsfa, dB, dsfb, mm, D, expected_m=128)   # one-time set-up outside capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        dg.dg_m_grouped_masked(dA, dsfa, dB, dsfb, mm, D, expected_m=128)
    for sizes in (first, [1, 255, 0, 129], [256, 256, 256, 256]):
        mm.copy_(torch.tensor(sizes, dtype=torch.int32))
        D.view(torch.int16).fill_(SENTINEL - 65536)
        graph.replay()
        torch.cuda.synchronize()
        assert dg.dg_device_status() == 0
        c2 = I.MaskedCase(c.G, c.max_m, c.N, c.K, 128, c.A, c.sfa, c.B, c.sfb, torch.tensor(sizes, dtype=torch.int32))
        _check_masked(c2, bf16_bits(D).reshape(G * max_m, N), sizes)
