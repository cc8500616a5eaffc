// Persistent, warp-specialised block-scaled FP8 GEMM for sm_103a.
//
// What it computes is the DeepGEMM method as its pages describe it ("DeepSeek DeepGEMM": fine-grained
// scaling with BLOCK_K = 128, two-level accumulation, TMA loads/stores, persistent warp
// specialisation, unaligned block sizes; "DeepSeek Open Source Week - Dia 3": promotion of tensor-core
// partial sums into a higher-precision accumulator):
//
//   D[m,n] = sum_kb sfa[m,kb] * sfb(n,kb) * P_kb[m,n],   P_kb[m,n] = sum_{k in block kb} A[m,k] B[n,k]
//
// One CTA per SM runs a static round-robin over output tiles of 128 x BN. Its warps have fixed roles:
//   warp 0      TMA producer: one lane streams the A [128 x 128] and B [BN x 128] e4m3 tiles of every
//               K block into a STAGES-deep shared-memory ring (128-byte swizzle), signalling `full`.
//   warp 1      TMEM owner and MMA issuer: one lane issues four tcgen05.mma (M=128, N=BN, K=32) per
//               K block into one of NACC TMEM accumulators, then commits to the stage's `empty`
//               barrier (smem reusable) and the accumulator's `tmem_full` barrier.
//   warps 2..9  promotion / epilogue: two warpgroups split the BN columns; each thread owns one tile
//               row (its TMEM lane) and BN/2 FP32 running sums in registers. Per K block they read the
//               block partial out of TMEM, multiply by sfa[m,kb] * sfb and add (packed f32x2 FMA), and
//               release the accumulator (`tmem_empty`). At the end of a tile they round to BF16 (or
//               add into FP32 for the weight gradient) and store.
// The MMA of K block kb+1.. overlaps the promotion of block kb (NACC accumulators in flight), and the
// store of one tile overlaps the first MMAs of the next.
//
// Every wait is bounded: after WAIT_LIMIT_NS a waiter records DG_DEVICE_TIMEOUT in the status word,
// raises a CTA-wide abort flag, and the CTA drains its own in-flight copies and MMAs (bounded too),
// frees TMEM and exits.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "dg_ptx.cuh"

namespace dg {

constexpr int BM = 128;                 // tile rows = UMMA M (one TMEM lane per row)
constexpr int BK = 128;                 // K block = scaling block
constexpr int UMMA_K = 32;              // K of one kind::f8f6f4 MMA
constexpr int EPI_WARPS = 8;
constexpr int THREADS = 64 + 32 * EPI_WARPS;
constexpr int TMEM_COLS = 512;
constexpr int MAX_MASKED_G = 1024;
constexpr int MAX_KGROUPS = 128;
constexpr int SMEM_LIMIT = 232448;      // 227 KB per CTA on sm_100-family parts
constexpr uint64_t WAIT_LIMIT_NS = 1000000000ull;
constexpr uint64_t DRAIN_LIMIT_NS = 50000000ull;
constexpr int STATUS_TIMEOUT = 6;       // DG_DEVICE_TIMEOUT

enum Mode : int { kNormal = 0, kContiguous = 1, kMasked = 2, kKGrouped = 3 };

struct Params {
    const float* sfa;          // scales of A rows, row stride kbs
    const float* sfb;          // scales of B: [G][sfb_rows][kbs]
    void* d;                   // output (bf16, or fp32 for k-grouped)
    const int32_t* m_indices;  // contiguous: expert per row
    const int32_t* masked_m;   // masked: valid rows per expert
    int* status;               // device status word
    int rows;                  // A rows per group: M (normal, k-grouped), Mt (contiguous), max_m (masked)
    int n;
    int kbs;                   // K blocks per scale row (K/128, or sumK/128)
    int groups;
    int sfb_rows;              // ceil(N/128), or N for the per-row k-grouped scales
    int m_blocks;              // ceil(rows / BM)
    int n_blocks;              // ceil(n / BN)
    int tiles;                 // tile count when known on the host (not masked)
    int kb_off[MAX_KGROUPS + 1];  // k-grouped: first K block of each expert, kb_off[G] = sumK/128
};

template <int MODE, int BN>
struct Cfg {
    static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "BN must be a multiple of 32 in [32, 256]");
    static constexpr int A_BYTES = BM * BK;
    static constexpr int B_BYTES = BN * BK;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int SFB_BYTES = (MODE == kKGrouped) ? 2 * BN * 4 : 0;
    static constexpr int STATIC_RESERVE = 512 + (MODE == kMasked ? 4 * (MAX_MASKED_G + 1) : 0);
    static constexpr int STAGES_FIT = (SMEM_LIMIT - 1024 - SFB_BYTES - STATIC_RESERVE) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
    static constexpr int NACC_FIT = TMEM_COLS / BN;
    static constexpr int NACC = NACC_FIT > 4 ? 4 : NACC_FIT;
    static constexpr int DYN_SMEM = 1024 + STAGES * STAGE_BYTES + SFB_BYTES;
    static constexpr int COLS = BN / 2;        // columns per epilogue warpgroup
    static constexpr int CHUNKS = COLS / 16;   // 16-column TMEM loads per K block
    static_assert(STAGES >= 2, "not enough shared memory for two stages");
};

struct TileInfo {
    int g, m0, n0;
    int kb0, nkb;        // K blocks [kb0, kb0 + nkb)
    int a_row, b_row;    // TMA row coordinates of the first A / B row
    int d_row;           // output row of the tile's first row
    int rows_valid;      // rows of the tile that are stored
    bool valid;
};

template <int MODE, int BN>
__device__ __forceinline__ TileInfo decode_tile(const Params& p, int t, const int* s_prefix) {
    TileInfo ti;
    ti.valid = true;
    ti.g = 0;
    ti.kb0 = 0;
    ti.nkb = p.kbs;
    if (MODE == kNormal || MODE == kContiguous) {
        const int mb = t % p.m_blocks, nb = t / p.m_blocks;
        ti.m0 = mb * BM;
        ti.n0 = nb * BN;
        ti.a_row = ti.m0;
        ti.d_row = ti.m0;
        ti.rows_valid = min(BM, p.rows - ti.m0);
        ti.b_row = ti.n0;
        if (MODE == kContiguous) {
            const int g = __ldg(p.m_indices + ti.m0);
            ti.valid = (g >= 0 && g < p.groups);
            ti.g = ti.valid ? g : 0;
            ti.b_row = ti.g * p.n + ti.n0;
        }
    } else if (MODE == kMasked) {
        // s_prefix[g] = tiles of experts < g; find the expert whose tile range holds t
        int lo = 0, hi = p.groups;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (s_prefix[mid] <= t) lo = mid; else hi = mid;
        }
        const int g = lo;
        const int local = t - s_prefix[g];
        const int mblk = (s_prefix[g + 1] - s_prefix[g]) / p.n_blocks;
        const int mb = local % mblk, nb = local / mblk;
        const int mm = min(max(__ldg(p.masked_m + g), 0), p.rows);
        ti.g = g;
        ti.m0 = mb * BM;
        ti.n0 = nb * BN;
        ti.a_row = g * p.rows + ti.m0;
        ti.d_row = ti.a_row;
        ti.b_row = g * p.n + ti.n0;
        ti.rows_valid = min(BM, mm - ti.m0);
    } else {  // kKGrouped
        const int per_g = p.m_blocks * p.n_blocks;
        const int g = t / per_g, local = t - g * per_g;
        const int mb = local % p.m_blocks, nb = local / p.m_blocks;
        ti.g = g;
        ti.m0 = mb * BM;
        ti.n0 = nb * BN;
        ti.kb0 = p.kb_off[g];
        ti.nkb = p.kb_off[g + 1] - p.kb_off[g];
        ti.valid = ti.nkb > 0;
        ti.a_row = ti.m0;
        ti.b_row = ti.n0;
        ti.d_row = g * p.rows + ti.m0;
        ti.rows_valid = min(BM, p.rows - ti.m0);
    }
    return ti;
}

// Bounded mbarrier wait. Returns false when this CTA is aborting (this waiter timed out, or another
// role did); the first waiter to time out records the status and raises the abort flag.
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                             int* status) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > WAIT_LIMIT_NS) {
            *abort_flag = 1;
            atomicExch(status, STATUS_TIMEOUT);
            return false;
        }
    }
}

// Short bounded wait used only while draining after an abort.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_timer_ns() - t0 > DRAIN_LIMIT_NS) return;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

template <int MODE, int BN>
__global__ void __launch_bounds__(THREADS, 1)
dg_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
               const __grid_constant__ Params p) {
    using C = Cfg<MODE, BN>;
    constexpr int STAGES = C::STAGES;
    constexpr int NACC = C::NACC;
    constexpr int COLS = C::COLS;
    constexpr int CHUNKS = C::CHUNKS;
    constexpr uint32_t IDESC = idesc_e4m3_f32(BM, BN);

    extern __shared__ uint8_t dyn_smem[];
    __shared__ uint64_t full_bar[STAGES], empty_bar[STAGES];
    __shared__ uint64_t tmem_full_bar[NACC], tmem_empty_bar[NACC];
    __shared__ uint32_t s_tmem_base;
    __shared__ int s_abort;
    __shared__ int s_prefix[MODE == kMasked ? MAX_MASKED_G + 1 : 1];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // 1024-byte aligned operand ring (128-byte swizzle atoms are 1024 bytes)
    const uint32_t raw = smem_u32(dyn_smem);
    uint8_t* smem = dyn_smem + (((raw + 1023u) & ~1023u) - raw);
    uint8_t* smem_a = smem;
    uint8_t* smem_b = smem + STAGES * C::A_BYTES;
    float* s_sfb = reinterpret_cast<float*>(smem + STAGES * C::STAGE_BYTES);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        for (int a = 0; a < NACC; ++a) {
            mbar_init(&tmem_full_bar[a], 1);
            mbar_init(&tmem_empty_bar[a], EPI_WARPS);
        }
        s_abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&s_tmem_base, TMEM_COLS);
        tmem_relinquish();
    }
    if (MODE == kMasked) {
        // per-expert tile counts, then an exclusive prefix sum (one warp)
        for (int g = threadIdx.x; g < p.groups; g += THREADS) {
            const int mm = min(max(__ldg(p.masked_m + g), 0), p.rows);
            s_prefix[g + 1] = ((mm + BM - 1) / BM) * p.n_blocks;
        }
        __syncthreads();
        if (warp == 0) {
            int carry = 0;
            for (int base = 0; base < p.groups; base += 32) {
                const int i = base + lane;
                int v = (i < p.groups) ? s_prefix[i + 1] : 0;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int u = __shfl_up_sync(0xffffffffu, v, o);
                    if (lane >= o) v += u;
                }
                if (i < p.groups) s_prefix[i + 1] = carry + v;
                carry += __shfl_sync(0xffffffffu, v, 31);
            }
            if (lane == 0) s_prefix[0] = 0;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const uint32_t tmem_base = s_tmem_base;
    volatile int* abort_flag = &s_abort;
    const int num_tiles = (MODE == kMasked) ? s_prefix[p.groups] : p.tiles;

    if (warp == 0) {
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tmap(&tmap_a);
            prefetch_tmap(&tmap_b);
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued = 0, issued_parity = 0;   // per-stage bits, for the abort drain
            bool ok = true;
            for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                const TileInfo ti = decode_tile<MODE, BN>(p, t, s_prefix);
                if (!ti.valid) continue;
                for (int kb = 0; kb < ti.nkb; ++kb) {
                    if (!wait_bounded(&empty_bar[stage], phase ^ 1u, abort_flag, p.status)) { ok = false; break; }
                    mbar_arrive_expect_tx(&full_bar[stage], C::STAGE_BYTES);
                    const int x = (ti.kb0 + kb) * BK;
                    tma_load_2d(&tmap_a, &full_bar[stage], smem_a + stage * C::A_BYTES, x, ti.a_row);
                    tma_load_2d(&tmap_b, &full_bar[stage], smem_b + stage * C::B_BYTES, x, ti.b_row);
                    issued |= 1u << stage;
                    issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) {
                for (int s = 0; s < STAGES; ++s)
                    if (issued & (1u << s)) drain_wait(&full_bar[s], (issued_parity >> s) & 1u);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true, any = false;
            int last_acc = 0;
            uint32_t last_parity = 0;
            const uint32_t a_base = smem_u32(smem_a), b_base = smem_u32(smem_b);
            for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                const TileInfo ti = decode_tile<MODE, BN>(p, t, s_prefix);
                if (!ti.valid) continue;
                for (int kb = 0; kb < ti.nkb; ++kb) {
                    if (!wait_bounded(&tmem_empty_bar[acc], acc_phase ^ 1u, abort_flag, p.status)) { ok = false; break; }
                    if (!wait_bounded(&full_bar[stage], phase, abort_flag, p.status)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                    const uint32_t a_addr = a_base + stage * C::A_BYTES;
                    const uint32_t b_addr = b_base + stage * C::B_BYTES;
#pragma unroll
                    for (int k = 0; k < BK / UMMA_K; ++k)
                        mma_f8f6f4(d_tmem, sw128_kmajor_desc(a_addr + k * UMMA_K),
                                   sw128_kmajor_desc(b_addr + k * UMMA_K), IDESC, k > 0 ? 1u : 0u);
                    mma_commit(&empty_bar[stage]);
                    mma_commit(&tmem_full_bar[acc]);
                    any = true;
                    last_acc = acc;
                    last_parity = acc_phase;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                    if (++acc == NACC) { acc = 0; acc_phase ^= 1u; }
                }
            }
            if (!ok && any) drain_wait(&tmem_full_bar[last_acc], last_parity);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------------ promotion + epilogue
        const int ew = warp - 2;               // 0..7
        const int q = warp & 3;                // TMEM lane quarter this warp may access
        const int h = ew >> 2;                 // column half of the tile
        const int row_in_tile = q * 32 + lane;
        const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + h * COLS;
        int acc = 0;
        uint32_t acc_phase = 0;
        uint32_t it = 0;                       // K blocks processed so far (scale-slot parity)
        bool ok = true;

        for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
            const TileInfo ti = decode_tile<MODE, BN>(p, t, s_prefix);
            if (!ti.valid) continue;
            const int cstart = ti.n0 + h * COLS;   // first output column of this thread
            const int arow = min(ti.a_row + row_in_tile, (MODE == kMasked ? p.groups * p.rows : p.rows) - 1);
            const float* sfa_row = p.sfa + static_cast<size_t>(arow) * p.kbs + ti.kb0;

            float accum[COLS];
            if (MODE == kKGrouped) {
                const float* drow = reinterpret_cast<const float*>(p.d) +
                                    static_cast<size_t>(ti.d_row + row_in_tile) * p.n + cstart;
                const bool row_ok = row_in_tile < ti.rows_valid;
#pragma unroll
                for (int j = 0; j < COLS; j += 4) {
                    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (row_ok && cstart + j < p.n) v = *reinterpret_cast<const float4*>(drow + j);
                    accum[j] = v.x; accum[j + 1] = v.y; accum[j + 2] = v.z; accum[j + 3] = v.w;
                }
            } else {
#pragma unroll
                for (int j = 0; j < COLS; ++j) accum[j] = 0.f;
            }

            // sfb rows that this thread's columns fall into
            const float* sfb_g = p.sfb + static_cast<size_t>(ti.g) * p.sfb_rows * p.kbs + ti.kb0;
            const int bblk = cstart / 128;
            const int split = (128 * (bblk + 1) - cstart) / 16;     // chunks before the next 128-block
            const float* sfb0 = sfb_g + static_cast<size_t>(min(bblk, p.sfb_rows - 1)) * p.kbs;
            const float* sfb1 = sfb_g + static_cast<size_t>(min(bblk + 1, p.sfb_rows - 1)) * p.kbs;
            // k-grouped: this thread stages one per-column scale per K block
            const int my_col = cstart + (threadIdx.x & 127);
            const bool stage_col = (MODE == kKGrouped) && ((threadIdx.x & 127) < COLS) && my_col < p.n;
            const float* sfb_col = p.sfb + static_cast<size_t>(stage_col ? my_col : 0) * p.kbs + ti.kb0;

            float sa_next = __ldg(sfa_row);
            float sb0_next = (MODE == kKGrouped) ? 0.f : __ldg(sfb0);
            float sb1_next = (MODE == kKGrouped) ? 0.f : __ldg(sfb1);
            float sc_next = stage_col ? __ldg(sfb_col) : 0.f;

            for (int kb = 0; kb < ti.nkb; ++kb) {
                const float sa = sa_next, sb0 = sb0_next, sb1 = sb1_next, sc = sc_next;
                if (kb + 1 < ti.nkb) {           // prefetch the next K block's scales
                    sa_next = __ldg(sfa_row + kb + 1);
                    if (MODE != kKGrouped) {
                        sb0_next = __ldg(sfb0 + kb + 1);
                        sb1_next = __ldg(sfb1 + kb + 1);
                    } else if (stage_col) {
                        sc_next = __ldg(sfb_col + kb + 1);
                    }
                }
                // k-grouped: publish this K block's per-column scales to the warpgroup; the slot
                // alternates on a running counter, so a slot is rewritten only after every thread
                // of the warpgroup has passed the barrier of the block that last used it
                float* slot = s_sfb + (it & 1) * BN + h * COLS;
                ++it;
                if (MODE == kKGrouped && (threadIdx.x & 127) < COLS) slot[threadIdx.x & 127] = sc;

                const bool got = wait_bounded(&tmem_full_bar[acc], acc_phase, abort_flag, p.status);
                // abort decisions are uniform per warp (and per warpgroup when it shares a barrier)
                const bool all_ok = (MODE == kKGrouped) ? named_bar_and(1 + h, 128, got)
                                                        : __all_sync(0xffffffffu, got);
                if (!all_ok) { ok = false; break; }
                tc_fence_after();
                const uint32_t taddr = lane_addr + static_cast<uint32_t>(acc * BN);

#pragma unroll
                for (int c0 = 0; c0 < CHUNKS; c0 += 2) {
                    uint32_t r0[16], r1[16];
                    tmem_ld_x16(taddr + c0 * 16, r0);
                    if (c0 + 1 < CHUNKS) tmem_ld_x16(taddr + (c0 + 1) * 16, r1);
                    tmem_ld_wait();
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {
                        const int c = c0 + cc;
                        if (c >= CHUNKS) break;
                        const uint32_t* r = cc ? r1 : r0;
                        if (MODE == kKGrouped) {
                            const float2 sa2 = make_float2(sa, sa);
#pragma unroll
                            for (int j = 0; j < 16; j += 4) {
                                const float4 sv = *reinterpret_cast<const float4*>(slot + c * 16 + j);
                                float2 a0 = make_float2(accum[c * 16 + j], accum[c * 16 + j + 1]);
                                float2 a1 = make_float2(accum[c * 16 + j + 2], accum[c * 16 + j + 3]);
                                const float2 p0 = __fmul2_rn(make_float2(__uint_as_float(r[j]), __uint_as_float(r[j + 1])),
                                                             make_float2(sv.x, sv.y));
                                const float2 p1 = __fmul2_rn(make_float2(__uint_as_float(r[j + 2]), __uint_as_float(r[j + 3])),
                                                             make_float2(sv.z, sv.w));
                                a0 = __ffma2_rn(p0, sa2, a0);
                                a1 = __ffma2_rn(p1, sa2, a1);
                                accum[c * 16 + j] = a0.x; accum[c * 16 + j + 1] = a0.y;
                                accum[c * 16 + j + 2] = a1.x; accum[c * 16 + j + 3] = a1.y;
                            }
                        } else {
                            const float s = sa * ((c < split) ? sb0 : sb1);
                            const float2 s2 = make_float2(s, s);
#pragma unroll
                            for (int j = 0; j < 16; j += 2) {
                                float2 a = make_float2(accum[c * 16 + j], accum[c * 16 + j + 1]);
                                a = __ffma2_rn(make_float2(__uint_as_float(r[j]), __uint_as_float(r[j + 1])), s2, a);
                                accum[c * 16 + j] = a.x;
                                accum[c * 16 + j + 1] = a.y;
                            }
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tmem_empty_bar[acc]);
                if (++acc == NACC) { acc = 0; acc_phase ^= 1u; }
            }
            if (!ok) break;

            // ---- store the tile
            if (row_in_tile < ti.rows_valid) {
                if (MODE == kKGrouped) {
                    float* drow = reinterpret_cast<float*>(p.d) + static_cast<size_t>(ti.d_row + row_in_tile) * p.n + cstart;
#pragma unroll
                    for (int j = 0; j < COLS; j += 4)
                        if (cstart + j < p.n)
                            st_global_v4(drow + j, __float_as_uint(accum[j]), __float_as_uint(accum[j + 1]),
                                         __float_as_uint(accum[j + 2]), __float_as_uint(accum[j + 3]));
                } else {
                    __nv_bfloat16* drow = reinterpret_cast<__nv_bfloat16*>(p.d) +
                                          static_cast<size_t>(ti.d_row + row_in_tile) * p.n + cstart;
#pragma unroll
                    for (int j = 0; j < COLS; j += 8)
                        if (cstart + j < p.n)
                            st_global_v4(drow + j, pack_bf16x2(accum[j], accum[j + 1]), pack_bf16x2(accum[j + 2], accum[j + 3]),
                                         pack_bf16x2(accum[j + 4], accum[j + 5]), pack_bf16x2(accum[j + 6], accum[j + 7]));
                }
            }
        }
    }

    // ---------------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

}  // namespace dg
