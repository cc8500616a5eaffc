"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test fixes one part of what the block-scaled FP8 GEMM computes (DeepGEMM pages: "fine-grained
scaling", two-level accumulation, NT layout, grouped contiguous / masked layouts, FP32 weight
gradients) with an independent route: torch's e4m3 / bf16 casts, exact rational arithmetic,
integer matrix products, power-of-two scaling identities and per-group decompositions.
"""
import bisect
from fractions import Fraction

import numpy as np
import pytest
import torch

from moe_grouped_gemm_tma_gb300 import inputs as I
from oracle import oracle as O

E4M3_CODES = torch.arange(256, dtype=torch.int32).to(torch.uint8)
E4M3_F32 = E4M3_CODES.view(torch.float8_e4m3fn).to(torch.float32).numpy()


# ----------------------------------------------------------------------------------------- e4m3 decode
def test_e4m3_decode_all_codes_match_torch():
    for c in range(256):
        v = O.e4m3_value(c)
        t = float(E4M3_F32[c])
        if np.isnan(t):
            assert np.isnan(v), c
        else:
            assert v == t and np.signbit(v) == np.signbit(t), (c, v, t)


@pytest.mark.parametrize("code,value", [
    (0x00, 0.0), (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9), (0x08, 2.0 ** -6), (0x38, 1.0),
    (0x3F, 1.875), (0x40, 2.0), (0x7E, 448.0), (0xFE, -448.0), (0xB8, -1.0), (0x81, -(2.0 ** -9)),
])
def test_e4m3_decode_closed_forms(code, value):
    # OCP E4M3: bias 7, subnormals f*2^-9, largest finite (1+6/8)*2^8 = 448
    assert O.e4m3_value(code) == value


def test_e4m3_nan_codes_and_no_infinity():
    assert np.isnan(O.e4m3_value(0x7F)) and np.isnan(O.e4m3_value(0xFF))
    finite = [abs(O.e4m3_value(c)) for c in range(256) if c not in (0x7F, 0xFF)]
    assert max(finite) == 448.0 and all(np.isfinite(finite))


# ----------------------------------------------------------------------------------------- BF16 rounding
def _bf16_table():
    """All finite non-negative BF16 values (decoded by torch), sorted, with their bit patterns."""
    bits = torch.arange(0, 0x7F80, dtype=torch.int32).to(torch.int16)
    vals = bits.view(torch.bfloat16).to(torch.float32).numpy().astype(np.float64)
    return [Fraction(float(v)) for v in vals], list(range(0, 0x7F80))


_BF16_VALS, _BF16_BITS = _bf16_table()


def bf16_nearest_even(q: Fraction) -> int:
    """BF16 bits nearest to the rational q, ties to the even pattern, by exact search over the table."""
    sign = 0x8000 if q < 0 else 0
    a = -q if q < 0 else q
    top = _BF16_VALS[-1]
    if a > top:  # beyond the largest finite: rounds to infinity when at least half an ulp past it
        ulp = top - _BF16_VALS[-2]
        return sign | (0x7F80 if a >= top + ulp / 2 else _BF16_BITS[-1])
    i = bisect.bisect_left(_BF16_VALS, a)
    if i < len(_BF16_VALS) and _BF16_VALS[i] == a:
        return sign | _BF16_BITS[i]
    lo, hi = i - 1, i
    dlo, dhi = a - _BF16_VALS[lo], _BF16_VALS[hi] - a
    if dlo < dhi:
        pick = lo
    elif dhi < dlo:
        pick = hi
    else:
        pick = lo if _BF16_BITS[lo] % 2 == 0 else hi
    return sign | _BF16_BITS[pick]


def test_bf16_rounding_matches_torch_on_float32():
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.standard_normal(3000).astype(np.float32),
        (rng.standard_normal(1000) * 1e30).astype(np.float32),
        (rng.standard_normal(1000) * 1e-39).astype(np.float32),  # float32 subnormals
        # exact BF16 ties: a BF16 value plus half its ulp (low 16 bits 0x8000)
        (rng.integers(0x0080, 0x7F00, 1000).astype(np.uint32) << 16 | 0x8000).view(np.float32),
        np.array([0.0, -0.0, 1.0, -1.0, 3.0e38, -3.0e38], dtype=np.float32),
    ])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    got = np.array([O.bf16_bits(float(v)) for v in x], dtype=np.uint16)
    np.testing.assert_array_equal(got, ref)


def test_bf16_rounding_from_double_is_single_rounding():
    # doubles just above / below BF16 ties, by 2^-30 relative: visible in FP64 but lost when rounding
    # through FP32 first, which would turn them into exact ties
    rng = np.random.default_rng(11)
    vals = []
    for b in rng.integers(0x0100, 0x7E00, 300):
        lo = Fraction(float(torch.tensor([int(b)], dtype=torch.int32).to(torch.int16)
                            .view(torch.bfloat16).float()))
        hi = Fraction(float(torch.tensor([int(b) + 1], dtype=torch.int32).to(torch.int16)
                            .view(torch.bfloat16).float()))
        mid = (lo + hi) / 2
        for eps in (Fraction(1, 2 ** 30), -Fraction(1, 2 ** 30), 0):
            v = mid * (1 + eps)
            vals.append(float(v))
    vals += list(rng.standard_normal(500) * 10.0 ** rng.integers(-40, 38, 500))
    vals += [2.0 ** -133, 2.0 ** -134, 3 * 2.0 ** -135, 1e-50, 3.4e38, 3.3961e38]
    for v in vals:
        assert O.bf16_bits(v) == bf16_nearest_even(Fraction(v)), v


# ----------------------------------------------------------------------------------------- helpers
def _frac_codes(codes: np.ndarray):
    return [[Fraction(float(E4M3_F32[c])) for c in row] for row in codes]


def exact_gemm(A, sfa, B, sfb, sfb_per_row=False, kb_range=None):
    """Exact rational D[m,n] = sum_kb sfa[m,kb] sfb[.,kb] sum_k a b (no rounding anywhere)."""
    A = np.asarray(A); B = np.asarray(B)
    sfa = np.asarray(sfa, dtype=np.float32); sfb = np.asarray(sfb, dtype=np.float32)
    M, K = A.shape
    N = B.shape[0]
    fa, fb = _frac_codes(A), _frac_codes(B)
    kbs = K // 128
    kbr = range(kbs) if kb_range is None else range(*kb_range)
    out = [[Fraction(0)] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            tot = Fraction(0)
            for kb in kbr:
                p = sum(fa[m][k] * fb[n][k] for k in range(kb * 128, kb * 128 + 128))
                sb = sfb[n, kb] if sfb_per_row else sfb[n // 128, kb]
                tot += Fraction(float(sfa[m, kb])) * Fraction(float(sb)) * p
            out[m][n] = tot
    return out


def _with_edge_codes(A: torch.Tensor) -> torch.Tensor:
    A = A.clone()
    flat = A.view(-1)
    edge = torch.tensor([0x01, 0x81, 0x07, 0x7E, 0xFE, 0x00, 0x80, 0x08], dtype=torch.uint8)
    flat[: len(edge)] = edge
    return A


# ----------------------------------------------------------------------------------------- contraction
@pytest.mark.parametrize("M,N,K", [(3, 5, 128), (2, 136, 256), (4, 7, 384)])
def test_normal_gemm_matches_exact_rational_bruteforce(M, N, K):
    c = I.make_normal(1234 + M * N + K, M, N, K)
    A = _with_edge_codes(c.A)
    got = O.gemm_fp8_nt(A, c.sfa, c.B, c.sfb)
    ex = exact_gemm(A.numpy(), c.sfa.numpy(), c.B.numpy(), c.sfb.numpy())
    want = np.array([[bf16_nearest_even(v) for v in row] for row in ex], dtype=np.uint16)
    np.testing.assert_array_equal(got, want)


def _ternary_codes(rng, shape):
    # e4m3 codes of -1, 0, +1
    return torch.from_numpy(rng.choice(np.array([0xB8, 0x00, 0x38], dtype=np.uint8), size=shape))


@pytest.mark.parametrize("K", [128, 256])
def test_normal_gemm_integer_exact(K):
    # all scales 1, values in {-1,0,1}: |D| <= K <= 256, so BF16 holds every result exactly
    rng = np.random.default_rng(K)
    M, N = 5, 260
    A, B = _ternary_codes(rng, (M, K)), _ternary_codes(rng, (N, K))
    sfa = torch.ones(M, K // 128)
    sfb = torch.ones((N + 127) // 128, K // 128)
    got = O.gemm_fp8_nt(A, sfa, B, sfb)
    ai = np.rint(E4M3_F32[A.numpy()]).astype(np.int64)
    bi = np.rint(E4M3_F32[B.numpy()]).astype(np.int64)
    d = ai @ bi.T
    want = torch.from_numpy(d.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    np.testing.assert_array_equal(got, want)


def test_worked_example_closed_form():
    # A codes all 1.0 with sfa 0.5, B codes all 2.0 with sfb 0.25, K = 384:
    # D = 3 blocks * 128 * (1*0.5) * (2*0.25) = 96
    M, N, K = 2, 3, 384
    A = torch.full((M, K), 0x38, dtype=torch.uint8)
    B = torch.full((N, K), 0x40, dtype=torch.uint8)
    got = O.gemm_fp8_nt(A, torch.full((M, 3), 0.5), B, torch.full((1, 3), 0.25))
    assert (O.bf16_bits_to_float(got) == 96.0).all()


def test_pow2_scaling_of_sfa_row_scales_output_row_exactly():
    c = I.make_normal(99, 6, 260, 384)
    base = O.bf16_bits_to_float(O.gemm_fp8_nt(c.A, c.sfa, c.B, c.sfb)).astype(np.float64)
    for row, k in ((2, 3), (5, -4)):
        sfa = c.sfa.clone()
        sfa[row] *= 2.0 ** k
        got = O.bf16_bits_to_float(O.gemm_fp8_nt(c.A, sfa, c.B, c.sfb)).astype(np.float64)
        want = base.copy()
        want[row] *= 2.0 ** k
        np.testing.assert_array_equal(got, want)


def test_pow2_scaling_of_sfb_block_row_scales_its_128_columns_exactly():
    c = I.make_normal(98, 4, 300, 256)   # nb = 3, the last block has 44 rows
    base = O.bf16_bits_to_float(O.gemm_fp8_nt(c.A, c.sfa, c.B, c.sfb)).astype(np.float64)
    for j, k in ((0, 2), (1, -3), (2, 5)):
        sfb = c.sfb.clone()
        sfb[j] *= 2.0 ** k
        got = O.bf16_bits_to_float(O.gemm_fp8_nt(c.A, c.sfa, c.B, sfb)).astype(np.float64)
        want = base.copy()
        want[:, 128 * j:128 * (j + 1)] *= 2.0 ** k
        np.testing.assert_array_equal(got, want)


def test_row_subset_equals_full_rows():
    c = I.make_normal(5, 40, 136, 256)
    full = O.gemm_fp8_nt(c.A, c.sfa, c.B, c.sfb)
    rows = [0, 39, 17, 3]
    np.testing.assert_array_equal(O.gemm_fp8_nt(c.A, c.sfa, c.B, c.sfb, rows=rows), full[rows])


def test_zero_block_scale_floor():
    # an all-zero 1x128 block gets the floor scale; its codes are all zero and contribute nothing
    x = torch.zeros(2, 256)
    x[:, 128:] = 1.0
    q, s = I.quantize_1x128(x)
    assert (q[:, :128] == 0).all() and torch.allclose(s[:, 0], torch.tensor(1e-4 / 448))
    B = torch.full((3, 256), 0x38, dtype=torch.uint8)
    got = O.bf16_bits_to_float(O.gemm_fp8_nt(q, s, B, torch.ones(1, 2)))
    assert np.allclose(got, 128.0, rtol=1e-2)


# ----------------------------------------------------------------------------------------- grouped
def test_contiguous_equals_per_group_normal_and_skips_padding():
    G, N, K = 3, 136, 256
    c = I.make_contiguous(17, G, N, K, [130, 0, 77])
    sentinel = np.full((c.Mt, N), I.BF16_SENTINEL, dtype=np.uint16)
    got = O.m_grouped_contiguous(c.A, c.sfa, c.B, c.sfb, c.m_indices, D_init=sentinel)
    mi = c.m_indices.numpy()
    for g in range(G):
        r = np.nonzero(mi == g)[0]
        if len(r) == 0:
            continue
        want = O.gemm_fp8_nt(c.A[r], c.sfa[r], c.B[g], c.sfb[g])
        np.testing.assert_array_equal(got[r], want)
    assert (got[mi < 0] == I.BF16_SENTINEL).all()
    assert (mi < 0).sum() == c.Mt - 207


def test_contiguous_bruteforce_small():
    c = I.make_contiguous(23, 2, 8, 128, [3, 2])
    got = O.m_grouped_contiguous(c.A, c.sfa, c.B, c.sfb, c.m_indices)
    mi = c.m_indices.numpy()
    for r in np.nonzero(mi >= 0)[0]:
        g = mi[r]
        ex = exact_gemm(c.A[r:r + 1].numpy(), c.sfa[r:r + 1].numpy(), c.B[g].numpy(), c.sfb[g].numpy())
        assert [bf16_nearest_even(v) for v in ex[0]] == list(got[r])


def test_masked_equals_per_group_normal_and_leaves_rows_untouched():
    G, max_m, N, K = 3, 64, 136, 256
    c = I.make_masked(31, G, max_m, N, K, [10, 0, 64])
    sentinel = np.full((G * max_m, N), I.BF16_SENTINEL, dtype=np.uint16)
    got = O.m_grouped_masked(c.A, c.sfa, c.B, c.sfb, c.masked_m, D_init=sentinel).reshape(G, max_m, N)
    for g, mm in enumerate([10, 0, 64]):
        if mm:
            want = O.gemm_fp8_nt(c.A[g, :mm], c.sfa[g, :mm], c.B[g], c.sfb[g])
            np.testing.assert_array_equal(got[g, :mm], want)
        assert (got[g, mm:] == I.BF16_SENTINEL).all()


def test_masked_m_above_max_m_is_clamped():
    G, max_m, N, K = 2, 32, 16, 128
    c = I.make_masked(32, G, max_m, N, K, [32, 5])
    over = torch.tensor([1000, 5], dtype=torch.int32)
    np.testing.assert_array_equal(O.m_grouped_masked(c.A, c.sfa, c.B, c.sfb, over),
                                  O.m_grouped_masked(c.A, c.sfa, c.B, c.sfb, c.masked_m))


# ----------------------------------------------------------------------------------------- k-grouped
def test_kgrouped_bruteforce_with_accumulation():
    c = I.make_kgrouped(41, 2, 3, 5, [128, 256])
    got = O.k_grouped_wgrad(c.A, c.sfa, c.B, c.sfb, c.ks, c.D_in)
    koff = 0
    for g, kg in enumerate(c.ks):
        ex = exact_gemm(c.A.numpy(), c.sfa.numpy(), c.B.numpy(), c.sfb.numpy(), sfb_per_row=True,
                        kb_range=(koff // 128, (koff + kg) // 128))
        for m in range(c.M):
            for n in range(c.N):
                want = float(Fraction(float(c.D_in[g, m, n])) + ex[m][n])  # Fraction -> nearest double
                want32 = np.float32(want)   # double -> float32, nearest even
                assert got[g, m, n] == want32, (g, m, n)
        koff += kg


def test_kgrouped_empty_group_leaves_buffer_unchanged():
    c = I.make_kgrouped(42, 3, 4, 8, [128, 0, 128])
    got = O.k_grouped_wgrad(c.A, c.sfa, c.B, c.sfb, c.ks, c.D_in)
    np.testing.assert_array_equal(got[1], c.D_in[1].numpy())


def test_kgrouped_integer_exact_and_split_additivity():
    # values in {-4..4} with unit scales: every partial sum is an integer below 2^24, exact in FP32
    rng = np.random.default_rng(3)
    M, N, sumK = 6, 9, 384
    vals = np.array([0x00, 0x38, 0x40, 0x44, 0x48, 0xB8, 0xC0, 0xC4, 0xC8], dtype=np.uint8)  # 0,1,2,3,4,-1..-4
    A = torch.from_numpy(rng.choice(vals, size=(M, sumK)))
    B = torch.from_numpy(rng.choice(vals, size=(N, sumK)))
    ones_a, ones_b = torch.ones(M, sumK // 128), torch.ones(N, sumK // 128)
    ai = np.rint(E4M3_F32[A.numpy()]).astype(np.int64)
    bi = np.rint(E4M3_F32[B.numpy()]).astype(np.int64)
    d0 = np.zeros((1, M, N), dtype=np.float32)
    one = O.k_grouped_wgrad(A, ones_a, B, ones_b, [384], d0)
    np.testing.assert_array_equal(one[0], (ai @ bi.T).astype(np.float32))
    two = O.k_grouped_wgrad(A, ones_a, B, ones_b, [256, 128], np.zeros((2, M, N), dtype=np.float32))
    np.testing.assert_array_equal(two[0], (ai[:, :256] @ bi[:, :256].T).astype(np.float32))
    np.testing.assert_array_equal(two[0] + two[1], one[0])


def test_kgrouped_g1_equals_dense_definition():
    c = I.make_kgrouped(43, 1, 4, 7, [256])
    got = O.k_grouped_wgrad(c.A, c.sfa, c.B, c.sfb, c.ks, np.zeros((1, 4, 7), dtype=np.float32))
    ex = exact_gemm(c.A.numpy(), c.sfa.numpy(), c.B.numpy(), c.sfb.numpy(), sfb_per_row=True)
    want = np.array([[np.float32(float(v)) for v in row] for row in ex], dtype=np.float32)
    np.testing.assert_array_equal(got[0], want)


# ----------------------------------------------------------------------------------------- generator
def test_torch_generator_matches_numpy_definition():
    # the bench may draw inputs with torch ops on the GPU; they must be the same numbers
    for seed, n in ((I._stream_seed(5, 1), 1001), (I._stream_seed(0xD6E0, 2), 4097)):
        a = I.normals(seed, n)
        b = I.normals_torch(seed, n, "cpu").numpy()
        np.testing.assert_array_equal(a, b)
