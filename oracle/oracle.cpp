// CPU oracle for the block-scaled FP8 GEMM and its MoE grouped variants.
//
// TEST INFRASTRUCTURE ONLY. Nothing in the product path (the CUDA library and its Python binding)
// may link, load or call this file; only the tests, the package's smoke check and the bench's CPU
// baseline use it. It shares no code, header, table or constant with the CUDA path.
//
// What it computes (restated from the DeepGEMM pages, "DeepSeek DeepGEMM" usage example and feature
// list; "DeepSeek Open Source Week - Dia 3", technical features):
//   * operands are float8 e4m3 codes, K-contiguous ("NT": A is [M,K], B is [N,K]);
//   * fine-grained scaling: one FP32 scale per 1x128 row block of A (sfa [M, K/128]) and per 128x128
//     block of B (sfb [ceil(N/128), K/128]), real value = code value * scale;
//   * two-level accumulation: each 128-wide K block is contracted, then multiplied by its two scales
//     and added to a higher-precision running sum;
//   * BF16 output for the normal and m-grouped GEMMs, FP32 output for the weight-gradient GEMM.
// The oracle writes out the plain definition D[m,n] = sum_kb sfa[m,kb]*sfb[n/128,kb]*sum_{k in kb}
// a[m,k]*b[n,k] in FP64 and rounds once. Per 128-K block the FP64 partial is exact (each e4m3 product
// has at most 8 significant bits within 2^-18..2^17; 128 of them need < 53 bits); the scale product
// sfa*sfb of two FP32 values is exact in FP64; the scaled terms are summed in FP64; the total is
// rounded once to BF16 (round to nearest even, directly from FP64) or FP32.
//
// Parity pins live in the CPU tests: e4m3 decode of all 256 codes, BF16 rounding, exact rational
// brute force, integer-exact products, power-of-two scaling rules and grouped = per-group identities.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <algorithm>
#include <thread>
#include <vector>

namespace {

// OCP 8-bit floating point, E4M3 ("fn" variant, as torch.float8_e4m3fn): sign bit 7, exponent bits
// 6..3 with bias 7, mantissa bits 2..0; exponent 0 is subnormal (f * 2^-9); S.1111.111 is NaN; there
// are no infinities, so the largest finite magnitude is 1.75 * 2^8 = 448.
double e4m3_value(uint8_t code) {
    const int s = code >> 7;
    const int e = (code >> 3) & 0xF;
    const int f = code & 0x7;
    if (e == 15 && f == 7) return std::nan("");
    const double mag = (e == 0) ? std::ldexp(static_cast<double>(f), -9)
                                : std::ldexp(static_cast<double>(8 + f), e - 10);  // (1 + f/8) 2^(e-7)
    return s ? -mag : mag;
}

struct Table {
    double v[256];
    Table() { for (int i = 0; i < 256; ++i) v[i] = e4m3_value(static_cast<uint8_t>(i)); }
};
const Table& table() { static Table t; return t; }

// IEEE bfloat16 (1 sign, 8 exponent bits with bias 127, 7 stored mantissa bits) from FP64 with one
// round-to-nearest-even step. Magnitudes are written r * 2^q with r an integer of at most 8 bits:
// q = max(floor(log2|x|), -126) - 7 (the subnormal quantum is 2^-133).
uint16_t bf16_bits(double x) {
    if (std::isnan(x)) return 0x7FC0;
    const uint16_t sign = std::signbit(x) ? 0x8000 : 0;
    const double a = std::fabs(x);
    if (a == 0.0) return sign;
    if (std::isinf(a)) return sign | 0x7F80;
    int e2;
    std::frexp(a, &e2);                     // a in [2^(e2-1), 2^e2)
    int q = std::max(e2 - 1, -126) - 7;
    double r = std::nearbyint(std::ldexp(a, -q));   // default rounding mode: to nearest, ties even
    if (r >= 256.0) { r = 128.0; q += 1; }
    if (q + 7 > 127) return sign | 0x7F80;  // overflow to infinity
    const uint32_t ri = static_cast<uint32_t>(r);
    if (ri < 128) return sign | static_cast<uint16_t>(ri);           // subnormal (or zero)
    const uint32_t bexp = static_cast<uint32_t>(q + 7 + 127);
    return sign | static_cast<uint16_t>((bexp << 7) | (ri - 128));
}

// One output row of the block-scaled contraction, written to out[0..N).
// sfa_row: the row's K/128 scales; sfb: [ceil(N/128), kbs] (per_col_sfb = 0) or [N, kbs] (= 1).
// kb0/kb1: the K blocks [kb0, kb1) that take part; kbs: the row stride of both scale tensors.
void row_sums(const uint8_t* a_row, const float* sfa_row, const uint8_t* B, const float* sfb,
              int64_t N, int64_t K, int64_t kbs, int64_t kb0, int64_t kb1, bool per_col_sfb,
              std::vector<double>& a_dec, double* out) {
    const double* tab = table().v;
    for (int64_t k = kb0 * 128; k < kb1 * 128; ++k) a_dec[k] = tab[a_row[k]];
    for (int64_t n = 0; n < N; ++n) {
        const uint8_t* b_row = B + n * K;
        const float* sfb_row = sfb + (per_col_sfb ? n : n / 128) * kbs;
        double acc = 0.0;
        for (int64_t kb = kb0; kb < kb1; ++kb) {
            double p = 0.0;   // exact: see the header
            for (int64_t k = kb * 128; k < kb * 128 + 128; ++k) p += a_dec[k] * tab[b_row[k]];
            const double s = static_cast<double>(sfa_row[kb]) * static_cast<double>(sfb_row[kb]);
            acc += s * p;
        }
        out[n] = acc;
    }
}

template <class F>
void parallel_rows(int64_t n_rows, int n_threads, F&& f) {
    if (n_threads <= 0) n_threads = static_cast<int>(std::max(1u, std::thread::hardware_concurrency()));
    n_threads = static_cast<int>(std::min<int64_t>(n_threads, std::max<int64_t>(n_rows, 1)));
    std::vector<std::thread> th;
    for (int t = 0; t < n_threads; ++t)
        th.emplace_back([&, t] { for (int64_t i = t; i < n_rows; i += n_threads) f(i); });
    for (auto& x : th) x.join();
}

}  // namespace

extern "C" {

double oracle_e4m3_value(uint8_t code) { return e4m3_value(code); }

uint16_t oracle_bf16_bits(double x) {
    return bf16_bits(x);
}

int oracle_hardware_threads(void) { return static_cast<int>(std::thread::hardware_concurrency()); }

// D = A . B^T for the rows listed in `rows` (all M rows when rows == NULL); D is [n_rows, N] BF16 bits.
int oracle_gemm_fp8_nt(const uint8_t* A, const float* sfa, const uint8_t* B, const float* sfb,
                       uint16_t* D, int64_t M, int64_t N, int64_t K,
                       const int64_t* rows, int64_t n_rows, int n_threads) {
    if (K % 128 != 0 || M < 0 || N < 0) return 1;
    const int64_t kbs = K / 128;
    if (!rows) n_rows = M;
    parallel_rows(n_rows, n_threads, [&](int64_t i) {
        const int64_t m = rows ? rows[i] : i;
        std::vector<double> a_dec(K), acc(N);
        row_sums(A + m * K, sfa + m * kbs, B, sfb, N, K, kbs, 0, kbs, false, a_dec, acc.data());
        for (int64_t n = 0; n < N; ++n) D[i * N + n] = oracle_bf16_bits(acc[n]);
    });
    return 0;
}

// m-grouped contiguous layout: row r of A belongs to group m_indices[r]; B is [G, N, K], sfb is
// [G, ceil(N/128), K/128]. Rows whose group is outside [0, G) are left as they are in D.
int oracle_m_grouped_contiguous(const uint8_t* A, const float* sfa, const uint8_t* B, const float* sfb,
                                const int32_t* m_indices, uint16_t* D, int64_t Mt, int64_t N, int64_t K,
                                int64_t G, const int64_t* rows, int64_t n_rows, int n_threads) {
    if (K % 128 != 0) return 1;
    const int64_t kbs = K / 128, nb = (N + 127) / 128;
    if (!rows) n_rows = Mt;
    parallel_rows(n_rows, n_threads, [&](int64_t i) {
        const int64_t r = rows ? rows[i] : i;
        const int64_t g = m_indices[r];
        if (g < 0 || g >= G) return;
        std::vector<double> a_dec(K), acc(N);
        row_sums(A + r * K, sfa + r * kbs, B + g * N * K, sfb + g * nb * kbs, N, K, kbs, 0, kbs, false,
                 a_dec, acc.data());
        for (int64_t n = 0; n < N; ++n) D[i * N + n] = bf16_bits(acc[n]);
    });
    return 0;
}

// m-grouped masked layout: A [G, max_m, K], D [G, max_m, N]; row r of group g is computed when
// r < min(masked_m[g], max_m) and left as it is otherwise. `rows` index the flattened G*max_m rows.
int oracle_m_grouped_masked(const uint8_t* A, const float* sfa, const uint8_t* B, const float* sfb,
                            const int32_t* masked_m, uint16_t* D, int64_t G, int64_t max_m, int64_t N,
                            int64_t K, const int64_t* rows, int64_t n_rows, int n_threads) {
    if (K % 128 != 0) return 1;
    const int64_t kbs = K / 128, nb = (N + 127) / 128;
    if (!rows) n_rows = G * max_m;
    parallel_rows(n_rows, n_threads, [&](int64_t i) {
        const int64_t gr = rows ? rows[i] : i;
        const int64_t g = gr / max_m, r = gr % max_m;
        const int64_t lim = std::min<int64_t>(std::max<int32_t>(masked_m[g], 0), max_m);
        if (r >= lim) return;
        std::vector<double> a_dec(K), acc(N);
        row_sums(A + gr * K, sfa + gr * kbs, B + g * N * K, sfb + g * nb * kbs, N, K, kbs, 0, kbs, false,
                 a_dec, acc.data());
        for (int64_t n = 0; n < N; ++n) D[i * N + n] = bf16_bits(acc[n]);
    });
    return 0;
}

// k-grouped weight gradient: A = X^T [M, sumK], B = dY^T [N, sumK], 1x128 scales along K for both
// (sfa [M, sumK/128], sfb [N, sumK/128]); group g owns K columns [koff_g, koff_g + ks[g]).
// D is [G, n_rows, N] FP32 holding the values to accumulate into; on return
// D[g, i, n] = fp32(D_in[g, i, n] + sum over group g's K blocks), the add done in FP64.
int oracle_k_grouped_wgrad(const uint8_t* A, const float* sfa, const uint8_t* B, const float* sfb,
                           const int64_t* ks, float* D, int64_t G, int64_t M, int64_t N,
                           const int64_t* rows, int64_t n_rows, int n_threads) {
    int64_t sumK = 0;
    for (int64_t g = 0; g < G; ++g) { if (ks[g] % 128 != 0 || ks[g] < 0) return 1; sumK += ks[g]; }
    const int64_t kbs = sumK / 128;
    if (!rows) n_rows = M;
    parallel_rows(n_rows, n_threads, [&](int64_t i) {
        const int64_t m = rows ? rows[i] : i;
        std::vector<double> a_dec(std::max<int64_t>(sumK, 1)), acc(N);
        int64_t koff = 0;
        for (int64_t g = 0; g < G; ++g) {
            const int64_t kb0 = koff / 128, kb1 = (koff + ks[g]) / 128;
            row_sums(A + m * sumK, sfa + m * kbs, B, sfb, N, sumK, kbs, kb0, kb1, true, a_dec, acc.data());
            float* drow = D + (g * n_rows + i) * N;
            for (int64_t n = 0; n < N; ++n)
                drow[n] = static_cast<float>(static_cast<double>(drow[n]) + acc[n]);
            koff += ks[g];
        }
    });
    return 0;
}

}  // extern "C"
