// Block-scaled variant of the normal GEMM for power-of-two scales, for sm_103a.
//
// Same product as dg_gemm_kernel in the normal layout,
//   D[m,n] = sum_kb sfa[m,kb] * sfb[n/128,kb] * sum_{k in block kb} A[m,k] B[n,k],
// but when every scale is a power of two the scaling can be done by the tensor core itself:
// tcgen05.mma.kind::mxf8f6f4.block_scale multiplies each 32-element slice of A's row m and B's row n by
// an 8-bit exponent (UE8M0) read from TMEM while it accumulates, so the whole K of a tile accumulates in
// one TMEM accumulator and nothing is promoted per K block (the pages' "UE8M0 block-scaled path" for
// SM100; the 1x128 and 128x128 FP32 scales become the same exponent for all four 32-element slices of a
// 128-K block).
//
// Warp roles (384 threads; no register re-split, no role holds large state):
//   warp 0      TMA producer: A and B tiles of every K block into a STAGES-deep ring.
//   warp 1      TMEM owner and MMA issuer: per K block four block-scaled MMAs (K = 32, scale bytes 0..3)
//               into the tile's accumulator, then commits the stage and the scale slot; at the end of a
//               tile commits the accumulator.
//   warp 2      scale stager: per K block, cp.async copies of the block's 128 sfa values and 4 sfb
//               block rows into a shared-memory ring (as in dg_gemm_kernel), ahead of the writers.
//   warps 4..11 two sets of four (one warp per TMEM lane quarter in each). Set 0 writes the scales of the
//               even K blocks (counted across tiles), set 1 those of the odd ones: each turns the staged
//               FP32 scales into exponents and stores them with tcgen05.st into a TMEM scale slot: A's row
//               m (lane m) in four columns (the MMA reads row m's from column m / 32), B's row n
//               (replicated in every lane quarter, lane n % 32) in column n / 32 after them. A scale
//               that is not a power of two is reported (DG_SCALE_NOT_UE8M0); packed UE8M0 input (four
//               exponent bytes per 32-bit word) is used as it is. Once a tile's scales are
//               written, each set reads its half of the tile's columns out of the accumulator,
//               releases it, rounds to BF16 and TMA-stores 32 x 16 boxes. (One set of writers was the
//               pacing loop: about 930 cycles per K block against about 640 for the MMAs.)
// CTA pairs (PAIR = 2): a cluster of two CTAs computes a 256-row tile with cta_group::2 MMAs issued by
// the leader. Each CTA stages its 128 A rows and half of B's rows (the peer's loads complete on the
// leader's barrier), writes the exponents of its own A rows and of all of B's rows into its own TMEM
// slot (the MMA reads both CTAs' slots at the same address), and reads out and stores its own rows;
// the peer's slot and accumulator releases arrive on the leader's barriers.
// Every wait is bounded as in dg_gemm_kernel.
#pragma once

#include "dg_kernel.cuh"

namespace dg {

constexpr int STATUS_SCALE_NOT_UE8M0 = 7;   // DG_SCALE_NOT_UE8M0

template <int BN, int PAIR>
struct CfgBS {
    static_assert(BN % 32 == 0 && BN >= 64 && BN <= 256, "BN must be a multiple of 32 in [64, 256]");
    static_assert(PAIR == 1 || PAIR == 2, "PAIR is 1 or 2");
    static constexpr int A_BYTES = BM * BK;
    static constexpr int B_ROWS = BN / PAIR;                      // B rows staged by each CTA
    static constexpr int B_BYTES = B_ROWS * BK;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int OUT_WARPS = 8;                          // both writer/output sets
    static constexpr int STORE_BYTES = OUT_WARPS * 2048;
    static constexpr int STATIC_RESERVE = 640;
    static constexpr int SCALE_SLOTS = 16;                       // shared-memory ring of staged FP32 scales
    static constexpr int SLOT_FLOATS = BM + 4;
    static constexpr int SCALE_BYTES = SCALE_SLOTS * SLOT_FLOATS * 4;
    static constexpr int STAGES = ring_stages(STAGE_BYTES, SCALE_BYTES, STORE_BYTES, STATIC_RESERVE);
    // TMEM: NACC accumulators of BN columns, then scale slots of 16 columns (A: 4, B: from +8, one per
    // 32 rows of B, at most 8)
    static constexpr int SLOT_COLS = 16;
    static constexpr int SFB_OFF = 8;
    static constexpr int NACC = (2 * BN + 2 * SLOT_COLS <= TMEM_COLS) ? 2 : 1;
    static constexpr int SF_COL0 = NACC * BN;
    static constexpr int SLOTS_FIT = (TMEM_COLS - SF_COL0) / SLOT_COLS;
    static constexpr int SLOTS = SLOTS_FIT > 8 ? 8 : SLOTS_FIT;
    static constexpr int STORE_OFF = ((STAGES * STAGE_BYTES + SCALE_BYTES + 1023) / 1024) * 1024;
    static constexpr int DYN_SMEM = 1024 + STORE_OFF + STORE_BYTES;
    // split-K partial sums: [128 rows][BN + 4] FP32 in the operand ring, idle once the tile's MMAs are done
    static constexpr int PSTRIDE = BN + 4;
    static_assert(BM * PSTRIDE * 4 <= STAGES * STAGE_BYTES, "split-K partials must fit in the operand ring");
    static_assert(SLOTS >= 2, "at least two scale slots");
    static_assert(STAGES >= 2, "not enough shared memory for two stages");
    static_assert(B_BYTES % 1024 == 0, "B stage must keep 1024-byte swizzle-atom alignment");
};

// Exponent byte of a power-of-two FP32 scale, replicated into the four bytes of a TMEM cell (one per
// 32-element slice of the 128-K block). Anything else (sign, mantissa bits, zero, infinity, NaN) is flagged in `bad`,
// which the caller reports once; its exponent is used. (A per-value branch with an atomic here made
// the scale writers the pacing loop: 476 against 358 us on 4096 x 7168 x 16384.)
__device__ __forceinline__ uint32_t ue8m0x4(float s, uint32_t& bad) {
    const uint32_t bits = __float_as_uint(s);
    // sign or mantissa bits; a zero exponent (bits - 2^23 borrows into the sign bit); the all-ones
    // exponent of infinity and NaN, which UE8M0 cannot hold (bits + 2^23 carries into the sign bit)
    bad |= (bits & 0x807FFFFFu) | ((bits - 0x00800000u) & 0x80000000u) | ((bits + 0x00800000u) & 0x80000000u);
    return ((bits >> 23) & 0xFFu) * 0x01010101u;
}

__device__ __forceinline__ uint32_t pick4u(uint32_t e0, uint32_t e1, uint32_t e2, uint32_t e3, int i) {
    return i == 0 ? e0 : (i == 1 ? e1 : (i == 2 ? e2 : e3));
}

template <int BN, int PAIR>
__global__ void __launch_bounds__(THREADS, 1)
dg_gemm_bs_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                  const __grid_constant__ CUtensorMap tmap_d, const __grid_constant__ Params p) {
    using C = CfgBS<BN, PAIR>;
    constexpr int STAGES = C::STAGES;
    constexpr int NACC = C::NACC;
    constexpr int SLOTS = C::SLOTS;
    constexpr uint32_t IDESC = idesc_bs_e4m3(BM * PAIR, BN);

    extern __shared__ uint8_t dyn_smem[];
    __shared__ uint64_t full_bar[STAGES], empty_bar[STAGES];
    __shared__ uint64_t tmem_full_bar[NACC], tmem_empty_bar[NACC];
    __shared__ uint64_t sf_full_bar[SLOTS], sf_empty_bar[SLOTS];
    __shared__ uint64_t scale_full_bar[C::SCALE_SLOTS], scale_empty_bar[C::SCALE_SLOTS];
    __shared__ uint32_t s_tmem_base;
    __shared__ int s_abort;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // split-K (few tiles): a cluster of p.split CTAs shares one tile, each CTA a K range, and the FP32
    // partial sums are reduced through distributed shared memory (not persistent: one tile per cluster)
    // CTA pairs (cta_group::2, 256-row tiles): each CTA stages its 128 A rows and half of B's rows;
    // the leader issues the MMAs; both CTAs write their own scale slots and store their own rows
    const bool split_k = PAIR == 1 && p.split > 1;
    const int crank = (PAIR == 2 || split_k) ? static_cast<int>(cluster_ctarank()) : 0;
    const int rank = (PAIR == 2) ? crank : 0;
    const bool leader = (rank == 0);
    const int srank = split_k ? crank : 0;
    const int csize = (PAIR == 2) ? 2 : (split_k ? p.split : 1);
    const int unit = static_cast<int>(blockIdx.x) / csize;
    const int num_units = static_cast<int>(gridDim.x) / csize;
    const uint32_t raw = smem_u32(dyn_smem);
    uint8_t* smem = dyn_smem + (((raw + 1023u) & ~1023u) - raw);
    uint8_t* smem_a = smem;
    uint8_t* smem_b = smem + STAGES * C::A_BYTES;
    float* s_scales = reinterpret_cast<float*>(smem + STAGES * C::STAGE_BYTES);
    uint8_t* s_store = smem + C::STORE_OFF;

    if (threadIdx.x == 0) {
        // the tensor maps are fetched while the barriers and TMEM are set up (they are kernel
        // parameters, not data of the previous grid, so this may precede the dependency wait)
        prefetch_tmap(&tmap_a);
        prefetch_tmap(&tmap_b);
        prefetch_tmap(&tmap_d);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        for (int a = 0; a < NACC; ++a) {
            mbar_init(&tmem_full_bar[a], 1);
            mbar_init(&tmem_empty_bar[a], C::OUT_WARPS * PAIR);
        }
        for (int s = 0; s < SLOTS; ++s) {
            mbar_init(&sf_full_bar[s], 4 * PAIR);
            mbar_init(&sf_empty_bar[s], 1);
        }
        for (int s = 0; s < C::SCALE_SLOTS; ++s) {
            mbar_init(&scale_full_bar[s], 32);
            mbar_init(&scale_empty_bar[s], 4);
        }
        s_abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        if (PAIR == 2) {
            tmem_alloc_pair(&s_tmem_base, TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(&s_tmem_base, TMEM_COLS);
            tmem_relinquish();
        }
    }
    grid_dependency_wait();
    grid_launch_dependents();
    tc_fence_before();
    if (PAIR == 2) cluster_sync(); else __syncthreads();
    tc_fence_after();

    const uint32_t tmem_base = s_tmem_base;
    volatile int* abort_flag = &s_abort;
    const int num_tiles = p.tiles;

    if (warp == 0) {
        // ---------------------------------------------------------------------- TMA producer
        const bool issuer = elect_one();
        int stage = 0;
        uint32_t phase = 0;
        uint32_t issued = 0, issued_parity = 0;
        bool ok = true;
        for (int t = unit; t < num_tiles && ok; t += num_units) {
            const TileInfo ti = decode_tile<kNormal, BN, PAIR>(p, t, nullptr, rank, srank);
            for (int kb = 0; kb < ti.nkb; ++kb) {
                const bool got = wait_bounded(&empty_bar[stage], phase ^ 1u, abort_flag, p.status, p.wait_limit_ns);
                if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
                if (issuer) {
                    const int x = (ti.kb0 + kb) * BK;
                    if (PAIR == 1 || leader) {
                        mbar_arrive_expect_tx(&full_bar[stage], PAIR * C::STAGE_BYTES);
                        tma_load_2d(&tmap_a, &full_bar[stage], smem_a + stage * C::A_BYTES, x, ti.a_row);
                        tma_load_2d(&tmap_b, &full_bar[stage], smem_b + stage * C::B_BYTES, x, ti.b_row);
                    } else {
                        // the peer's halves complete on the leader's barrier
                        const uint32_t bar = mapa_shared(smem_u32(&full_bar[stage]), 0);
                        tma_load_2d_pair(&tmap_a, bar, smem_a + stage * C::A_BYTES, x, ti.a_row);
                        tma_load_2d_pair(&tmap_b, bar, smem_b + stage * C::B_BYTES, x, ti.b_row);
                    }
                }
                __syncwarp();
                issued |= 1u << stage;
                issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
        }
        if (ok) {
            // every stage this CTA filled has been consumed before the CTA may exit
            for (int i = 0; i < STAGES && ok; ++i) {
                const bool got = wait_bounded(&empty_bar[stage], phase ^ 1u, abort_flag, p.status, p.wait_limit_ns);
                if (!__all_sync(0xffffffffu, got)) ok = false;
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
        }
        if (!ok && (PAIR == 1 || leader) && issuer) {
            for (int s = 0; s < STAGES; ++s)
                if (issued & (1u << s)) drain_wait(&full_bar[s], (issued_parity >> s) & 1u);
        }
    } else if (warp == 1 && leader) {
        // ---------------------------------------------------------------------- MMA issuer
        const bool issuer = elect_one();
        int stage = 0, slot = 0, acc = 0;
        uint32_t phase = 0, sphase = 0, aphase = 0;
        bool ok = true, any = false;
        int last_acc = 0;
        uint32_t last_parity = 0;
        const uint32_t a_base = smem_u32(smem_a), b_base = smem_u32(smem_b);
        for (int t = unit; t < num_tiles && ok; t += num_units) {
            const TileInfo ti = decode_tile<kNormal, BN, PAIR>(p, t, nullptr, rank, srank);
            // the tile's accumulator must have been read out by the output warps
            const bool free_acc = wait_bounded(&tmem_empty_bar[acc], aphase ^ 1u, abort_flag, p.status, p.wait_limit_ns);
            if (!__all_sync(0xffffffffu, free_acc)) { ok = false; break; }
            const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
            for (int kb = 0; kb < ti.nkb; ++kb) {
                bool got = (static_cast<unsigned>(mbar_try_wait(&full_bar[stage], phase)) &
                            static_cast<unsigned>(mbar_try_wait(&sf_full_bar[slot], sphase))) != 0u;
                if (!got)
                    got = wait_bounded(&full_bar[stage], phase, abort_flag, p.status, p.wait_limit_ns) &&
                          wait_bounded(&sf_full_bar[slot], sphase, abort_flag, p.status, p.wait_limit_ns);
                if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
                tc_fence_after();
                const uint64_t a_desc = sw128_kmajor_desc(a_base + stage * C::A_BYTES);
                const uint64_t b_desc = sw128_kmajor_desc(b_base + stage * C::B_BYTES);
                const uint32_t sfa_t = tmem_base + static_cast<uint32_t>(C::SF_COL0 + slot * C::SLOT_COLS);
                const uint32_t sfb_t = sfa_t + C::SFB_OFF;
                if (issuer) {
#pragma unroll
                    for (int k = 0; k < BK / UMMA_K; ++k) {
                        // 32-element slice k of the block: scale byte k of every cell
                        const uint64_t ad = a_desc + static_cast<uint64_t>(k * (UMMA_K >> 4));
                        const uint64_t bd = b_desc + static_cast<uint64_t>(k * (UMMA_K >> 4));
                        const uint32_t id = IDESC | IDESC_BS_SFA(k) | IDESC_BS_SFB(k);
                        if (PAIR == 2) mma_f8f6f4_bs_pair(d_tmem, ad, bd, id, sfa_t, sfb_t, (kb > 0 || k > 0) ? 1u : 0u);
                        else mma_f8f6f4_bs(d_tmem, ad, bd, id, sfa_t, sfb_t, (kb > 0 || k > 0) ? 1u : 0u);
                    }
                    if (PAIR == 2) {
                        mma_commit_pair(&empty_bar[stage], 0x3);
                        mma_commit_pair(&sf_empty_bar[slot], 0x3);
                    } else {
                        mma_commit(&empty_bar[stage]);
                        mma_commit(&sf_empty_bar[slot]);
                    }
                }
                __syncwarp();
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                if (++slot == SLOTS) { slot = 0; sphase ^= 1u; }
            }
            if (!ok) break;
            if (issuer) {
                if (PAIR == 2) mma_commit_pair(&tmem_full_bar[acc], 0x3);
                else mma_commit(&tmem_full_bar[acc]);
            }
            __syncwarp();
            any = true;
            last_acc = acc;
            last_parity = aphase;
            if (++acc == NACC) { acc = 0; aphase ^= 1u; }
        }
        if (!ok && any && issuer) drain_wait(&tmem_full_bar[last_acc], last_parity);
    } else if (warp == 2) {
        // ---------------------------------------------------------------------- scale stager
        int slot = 0;
        uint32_t sphase = 0;
        for (int t = unit; t < num_tiles; t += num_units) {
            const TileInfo ti = decode_tile<kNormal, BN, PAIR>(p, t, nullptr, rank, srank);
            // FP32 scales: one value per K block; packed UE8M0: the 32-bit word holding the block's
            // exponent (the writers pick its byte)
            const int row_stride = p.sf_packed ? p.sf_words : p.kbs;
            const float* sfa_rows[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                sfa_rows[i] = p.sfa + static_cast<size_t>(min(ti.a_row + lane + 32 * i, p.rows - 1)) * row_stride;
            const float* sfb_src = p.sfb + static_cast<size_t>(min(ti.n0 / 128 + (lane & 3), p.sfb_rows - 1)) * row_stride;
            bool ok = true;
            for (int kb = 0; kb < ti.nkb; ++kb) {
                const bool got = wait_bounded(&scale_empty_bar[slot], sphase ^ 1u, abort_flag, p.status, p.wait_limit_ns);
                if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
                float* dst = s_scales + slot * C::SLOT_FLOATS;
                const int kidx = p.sf_packed ? ((ti.kb0 + kb) >> 2) : (ti.kb0 + kb);
#pragma unroll
                for (int i = 0; i < 4; ++i) cp_async_4(dst + lane + 32 * i, sfa_rows[i] + kidx);
                if (lane < 4) cp_async_4(dst + BM + lane, sfb_src + kidx);
                cp_async_arrive_noinc(&scale_full_bar[slot]);
                if (++slot == C::SCALE_SLOTS) { slot = 0; sphase ^= 1u; }
            }
            if (!ok) break;
        }
        cp_async_wait_all();
    } else if (warp >= 4) {
        // ---------------------------------------------------------------------- scale writers + output
        const int set = (warp >= 8) ? 1 : 0;
        const int q = warp & 3;
        const int ow = warp - 4;
        const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
        uint32_t bad = 0;   // a scale that is not a power of two was seen (reported once, below)
        int gbase = 0;      // K blocks of this CTA's earlier tiles: the global K-block count picks slots
        int acc = 0;
        uint32_t aphase = 0, store_round = 0;
        uint8_t* wbuf = s_store + ow * 2048;
        const int sw = (lane >> 2) & 1;
        bool ok = true;
        for (int t = unit; t < num_tiles && ok; t += num_units) {
            const TileInfo ti = decode_tile<kNormal, BN, PAIR>(p, t, nullptr, rank, srank);
            // staged sfb block row of this lane's columns n0 + 32 j + lane (columns past N reuse the last)
            int bidx[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) bidx[j] = min(min(ti.n0 + 32 * j + lane, p.n - 1) / 128 - ti.n0 / 128, 3);
            for (int kb = ((gbase & 1) == set) ? 0 : 1; kb < ti.nkb; kb += 2) {
                const int gk = gbase + kb;
                const int slot = gk % SLOTS, sslot = gk % C::SCALE_SLOTS;
                const uint32_t tphase = static_cast<uint32_t>(gk / SLOTS) & 1u;
                const uint32_t sphase = static_cast<uint32_t>(gk / C::SCALE_SLOTS) & 1u;
                bool got = (static_cast<unsigned>(mbar_try_wait(&sf_empty_bar[slot], tphase ^ 1u)) &
                            static_cast<unsigned>(mbar_try_wait(&scale_full_bar[sslot], sphase))) != 0u;
                if (!got)
                    got = wait_bounded(&sf_empty_bar[slot], tphase ^ 1u, abort_flag, p.status, p.wait_limit_ns) &&
                          wait_bounded(&scale_full_bar[sslot], sphase, abort_flag, p.status, p.wait_limit_ns);
                if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
                const float* sl = s_scales + sslot * C::SLOT_FLOATS;
                const float4 b4 = *reinterpret_cast<const float4*>(sl + BM);
                uint32_t va, vb[8];
                if (p.sf_packed) {
                    // byte (K block mod 4) of the staged words, replicated into the cell's four bytes
                    const uint32_t sh = 8u * static_cast<uint32_t>((ti.kb0 + kb) & 3);
                    va = ((__float_as_uint(sl[q * 32 + lane]) >> sh) & 0xFFu) * 0x01010101u;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        vb[j] = (j < BN / 32) ? ((__float_as_uint(pick4(b4, bidx[j])) >> sh) & 0xFFu) * 0x01010101u : 0u;
                } else {
                    va = ue8m0x4(sl[q * 32 + lane], bad);
                    // the (at most four) 128-column blocks' exponents, converted once and picked per column
                    const uint32_t e0 = ue8m0x4(b4.x, bad), e1 = ue8m0x4(b4.y, bad);
                    const uint32_t e2 = ue8m0x4(b4.z, bad), e3 = ue8m0x4(b4.w, bad);
#pragma unroll
                    for (int j = 0; j < 8; ++j) vb[j] = (j < BN / 32) ? pick4u(e0, e1, e2, e3, bidx[j]) : 0u;
                }
                const uint32_t col = static_cast<uint32_t>(C::SF_COL0 + slot * C::SLOT_COLS);
                // A's exponent in the slot's first eight columns: the MMA reads row m's from column m / 32
                // (of the CTA's own rows, or of the pair's 256)
                const uint32_t va8[8] = {va, va, va, va, va, va, va, va};
                tmem_st_x8(lane_base + col, va8);
                tmem_st_x8(lane_base + col + C::SFB_OFF, vb);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (PAIR == 2 && !leader) mbar_arrive_cluster(mapa_shared(smem_u32(&sf_full_bar[slot]), 0));
                    else mbar_arrive(&sf_full_bar[slot]);
                    mbar_arrive(&scale_empty_bar[sslot]);
                }
            }
            gbase += ti.nkb;
            if (!ok) break;

            // this set's half of the tile: columns [set * BN/2, (set + 1) * BN/2)
            const bool full = wait_bounded(&tmem_full_bar[acc], aphase, abort_flag, p.status, p.wait_limit_ns);
            if (!__all_sync(0xffffffffu, full)) break;
            tc_fence_after();
            const uint32_t taddr = lane_base + static_cast<uint32_t>(acc * BN);
            const int y = ti.m0 + q * 32;
            constexpr int CH = BN / 32;            // 16-column chunks per set
            const int c0 = set * CH;
            if (split_k) {
                // park this CTA's FP32 partial sums (its half of the columns) in the idle operand ring;
                // rows padded to BN + 4 floats, so the 16-byte stores of a warp hit every bank
                float* prow = reinterpret_cast<float*>(smem) + (q * 32 + lane) * C::PSTRIDE + c0 * 16;
#pragma unroll 1
                for (int i = 0; i < CH; ++i) {
                    uint32_t r[16];
                    tmem_ld_x16(taddr + (c0 + i) * 16, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; j += 4)
                        *reinterpret_cast<float4*>(prow + i * 16 + j) =
                            make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]), __uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tmem_empty_bar[acc]);
                if (++acc == NACC) { acc = 0; aphase ^= 1u; }
                continue;
            }
            // loads of chunk c + 1 are in flight while chunk c is rounded and staged
            uint32_t rb[2][16];
            tmem_ld_x16(taddr + c0 * 16, rb[0]);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < CH; ++i) {
                const int b = i & 1;
                const int c = c0 + i;
                if (i + 1 < CH) {
                    tmem_ld_x16(taddr + (c + 1) * 16, rb[b ^ 1]);
                } else {
                    // every load of this half has completed: release it to the next tile's MMAs (on the
                    // leader's barrier for a pair)
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        if (PAIR == 2 && !leader) mbar_arrive_cluster(mapa_shared(smem_u32(&tmem_empty_bar[acc]), 0));
                        else mbar_arrive(&tmem_empty_bar[acc]);
                    }
                }
                uint8_t* half = wbuf + (store_round & 1u) * 1024;
                ++store_round;
                if (lane == 0) bulk_wait_read_1();
                __syncwarp();
                const uint32_t* r = rb[b];
                uint4* rowp = reinterpret_cast<uint4*>(half + lane * 32);
                rowp[sw] = make_uint4(pack_bf16x2(__uint_as_float(r[0]), __uint_as_float(r[1])),
                                      pack_bf16x2(__uint_as_float(r[2]), __uint_as_float(r[3])),
                                      pack_bf16x2(__uint_as_float(r[4]), __uint_as_float(r[5])),
                                      pack_bf16x2(__uint_as_float(r[6]), __uint_as_float(r[7])));
                rowp[sw ^ 1] = make_uint4(pack_bf16x2(__uint_as_float(r[8]), __uint_as_float(r[9])),
                                          pack_bf16x2(__uint_as_float(r[10]), __uint_as_float(r[11])),
                                          pack_bf16x2(__uint_as_float(r[12]), __uint_as_float(r[13])),
                                          pack_bf16x2(__uint_as_float(r[14]), __uint_as_float(r[15])));
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    // only boxes that start inside the output are issued (rows past M, columns past N)
                    if (y < p.rows && ti.n0 + c * 16 < p.n) tma_store_2d(&tmap_d, half, ti.n0 + c * 16, y);
                    bulk_commit();
                }
                if (i + 1 < CH) tmem_ld_wait();
            }
            if (++acc == NACC) { acc = 0; aphase ^= 1u; }
        }
        if (bad != 0u) record_status(p.status, STATUS_SCALE_NOT_UE8M0);
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }

    // ------------------------------------------------------------------------ split-K reduction
    if (split_k) {
        // every CTA's partials are visible cluster-wide after this barrier; CTA s of the cluster then
        // reduces rows [s*128/S, (s+1)*128/S) of the tile over all S partials (fixed order s = 0..S-1),
        // rounds to BF16 and stores; the second barrier keeps every CTA's shared memory alive until all
        // remote reads are done
        cluster_sync();
        if (warp >= 4 && !*abort_flag && unit < num_tiles) {
            const TileInfo ti = decode_tile<kNormal, BN, PAIR>(p, unit, nullptr, rank, srank);
            const int rows_per = BM / p.split;
            const int groups = rows_per * (BN / 4);
            const uint32_t part_local = smem_u32(smem);
            for (int gi = static_cast<int>(threadIdx.x) - 128; gi < groups; gi += 256) {
                const int row = srank * rows_per + gi / (BN / 4);
                const int c4 = (gi % (BN / 4)) * 4;
                const float4 sum = cluster_sum_v4(part_local + static_cast<uint32_t>((row * C::PSTRIDE + c4) * 4), p.split);
                if (row < ti.rows_valid && ti.n0 + c4 < p.n) {
                    __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(p.d) + static_cast<size_t>(ti.m0 + row) * p.n + ti.n0 + c4;
                    st_global_v2(dst, pack_bf16x2(sum.x, sum.y), pack_bf16x2(sum.z, sum.w));
                }
            }
        }
        cluster_sync();
    }

    // ------------------------------------------------------------------------ teardown
    tc_fence_before();
    if (PAIR == 2) cluster_sync(); else __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        if (PAIR == 2) tmem_dealloc_pair(tmem_base, TMEM_COLS);
        else tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

}  // namespace dg
