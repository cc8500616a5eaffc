// Few-row ("decode") variant of the block-scaled FP8 GEMM for sm_103a: the normal layout with M <= 128
// and the masked m-grouped layout with few rows per expert (MoE decode: "DeepSeek DeepGEMM", the
// grouped-GEMM section: the masked layout serves inference decoding, under CUDA graphs).
//
// Same product and scales as dg_gemm_kernel, computed transposed: a tile is 128 columns of D (n) x BMT
// rows of D (m), and the MMA runs with B's 128 rows as its M operand and A's BMT rows as its N operand,
// so TMEM lane n holds column n of the tile and TMEM column m holds row m. With few rows this stages 128
// B rows -- the bytes that come from HBM -- plus BMT A rows per K block, instead of 128 A rows (mostly
// past M) plus a few B rows. Scales: sfb[n0/128, kb] is one value per tile and K block (the tile's 128
// columns are one sfb block) and sfa[m, kb] varies along the MMA's N, so the promotion is
// acc[m] += P[m] * (sfa[m] * sfb).
//
// These shapes are bound by streaming B from HBM, and a tile has little arithmetic, so the kernel is
// built to keep every SM's loads in flight and to pay few round trips per K block:
//   * split-K over a cluster of S CTAs sized so that the tiles times S fill the SMs; each CTA streams
//     K/S of the tile and the FP32 partials are reduced through distributed shared memory;
//   * the MMA issuer commits a group of KG consecutive K blocks (KG TMEM accumulators of BMT columns)
//     at once, and the epilogue takes a whole group per wait: one wait, one batch of TMEM loads, one
//     release per KG blocks;
//   * the two epilogue warpgroups split the tile's BMT rows (each its own TMEM columns), so both work
//     on every group and no exchange is needed at the end of a tile;
//   * persistent: a CTA (or cluster) loops over tiles; the masked layout counts its tiles on the device
//     from masked_m, so the launch needs no host synchronisation (graph-capturable).
//
// Warp roles: warp 0 TMA producer, warp 1 TMEM owner and MMA issuer, warp 2 scale stager (sfa and sfb of
// each group into a shared-memory slot with cp.async), warp 3 idle, warps 4..11 promotion and store
// (setmaxnreg 56 / 224). Every wait is bounded as in dg_gemm_kernel.
#pragma once

#include "dg_kernel.cuh"

namespace dg {

template <int BMT>
struct CfgDec {
    static_assert(BMT == 32 || BMT == 64 || BMT == 128, "BMT is 32, 64 or 128");
    static constexpr int BNT = 128;                      // D columns per tile = MMA M = TMEM lanes
    static constexpr int A_BYTES = BMT * BK;             // A rows of the tile (the MMA's N operand)
    static constexpr int B_BYTES = BNT * BK;             // B rows of the tile (the MMA's M operand)
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int HALF = BMT / 2;                 // rows of D promoted by each epilogue warpgroup
    static constexpr int NSLOT = TMEM_COLS / BMT;        // TMEM accumulators (one K block each)
    static constexpr int KG = (NSLOT / 2) > 8 ? 8 : NSLOT / 2;   // K blocks per group: 8, 4, 2
    static constexpr int NGRP = NSLOT / KG;              // groups in TMEM at once
    static constexpr int SGROUPS = 4;                    // scale slots (one group each)
    static constexpr int SROW = BMT + 4;                 // per K block: BMT sfa values, sfb, padding
    static constexpr int SLOT_FLOATS = KG * SROW;
    static constexpr int SCALE_BYTES = SGROUPS * SLOT_FLOATS * 4;
    static constexpr int STATIC_RESERVE = 640 + 4 * (MAX_MASKED_G + 1);
    static constexpr int STAGES = ring_stages(STAGE_BYTES, SCALE_BYTES, 0, STATIC_RESERVE);
    static constexpr int DYN_SMEM = 1024 + STAGES * STAGE_BYTES + SCALE_BYTES;
    static constexpr int PARTIAL_BYTES = BMT * BNT * 4;  // split-K partials [BMT rows][128 columns] in the ring
    static_assert(PARTIAL_BYTES <= STAGES * STAGE_BYTES, "split-K partials must fit in the operand ring");
    static_assert(STAGES >= 2, "not enough shared memory for two stages");
    static_assert(HALF % 16 == 0, "each warpgroup loads whole 16-column chunks");
};

struct DecTile {
    int g, m0, n0;       // expert, first row within the expert, first column
    int kb0, nkb;        // K blocks [kb0, kb0 + nkb) of this CTA
    int a_row, b_row;    // TMA row coordinates of the tile's first A / B row
    int rows_valid;      // rows of the tile that are stored
};

// Tiles: row block fastest (the row blocks of one expert and column block share B, read back to back),
// then column block, then expert; the K blocks are shared by the CTAs of a split-K cluster.
template <int MODE, int BMT>
__device__ __forceinline__ DecTile decode_dec(const Params& p, int t, const int* s_prefix, int srank) {
    DecTile ti;
    if (MODE == kMasked) {
        int lo = 0, hi = p.groups;   // s_prefix[g] = tiles of experts < g
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
        ti.m0 = mb * BMT;
        ti.n0 = nb * 128;
        ti.a_row = g * p.rows + ti.m0;
        ti.b_row = g * p.n + ti.n0;
        ti.rows_valid = min(BMT, mm - ti.m0);
    } else {
        const int mb = t % p.m_blocks, nb = t / p.m_blocks;
        ti.g = 0;
        ti.m0 = mb * BMT;
        ti.n0 = nb * 128;
        ti.a_row = ti.m0;
        ti.b_row = ti.n0;
        ti.rows_valid = min(BMT, p.rows - ti.m0);
    }
    ti.kb0 = 0;
    ti.nkb = p.kbs;
    if (p.split > 1) {
        ti.kb0 = (srank * p.kbs) / p.split;
        ti.nkb = ((srank + 1) * p.kbs) / p.split - ti.kb0;
    }
    return ti;
}

template <int MODE, int BMT>
__global__ void __launch_bounds__(THREADS, 1)
dg_decode_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                 const __grid_constant__ Params p) {
    using C = CfgDec<BMT>;
    constexpr int STAGES = C::STAGES;
    constexpr int KG = C::KG;
    constexpr int NGRP = C::NGRP;
    constexpr int SG = C::SGROUPS;
    constexpr int HALF = C::HALF;
    constexpr int HCH = HALF / 16;                        // 16-column TMEM loads per K block and thread
    constexpr int LB = (HALF + KG * HALF > 160) ? 1 : KG; // K blocks per batch of TMEM loads
    constexpr uint32_t IDESC = idesc_e4m3_f32(128, BMT);

    extern __shared__ uint8_t dyn_smem[];
    __shared__ uint64_t full_bar[STAGES], empty_bar[STAGES];
    __shared__ uint64_t tmem_full_bar[NGRP], tmem_empty_bar[NGRP];
    __shared__ uint64_t scale_full_bar[SG], scale_empty_bar[SG];
    __shared__ uint32_t s_tmem_base;
    __shared__ int s_abort;
    __shared__ int s_prefix[MODE == kMasked ? MAX_MASKED_G + 1 : 1];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const bool split_k = p.split > 1;
    const int srank = split_k ? static_cast<int>(cluster_ctarank()) : 0;
    const int csize = split_k ? p.split : 1;
    const int unit = static_cast<int>(blockIdx.x) / csize;
    const int num_units = static_cast<int>(gridDim.x) / csize;

    const uint32_t raw = smem_u32(dyn_smem);
    uint8_t* smem = dyn_smem + (((raw + 1023u) & ~1023u) - raw);
    uint8_t* smem_a = smem;
    uint8_t* smem_b = smem + STAGES * C::A_BYTES;
    float* s_scales = reinterpret_cast<float*>(smem + STAGES * C::STAGE_BYTES);

    if (threadIdx.x == 0) {
        // the tensor maps are kernel parameters, not data of the previous grid: fetched before the wait
        prefetch_tmap(&tmap_a);
        prefetch_tmap(&tmap_b);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        for (int a = 0; a < NGRP; ++a) {
            mbar_init(&tmem_full_bar[a], 1);
            mbar_init(&tmem_empty_bar[a], EPI_WARPS);
        }
        for (int s = 0; s < SG; ++s) {
            mbar_init(&scale_full_bar[s], 32);
            mbar_init(&scale_empty_bar[s], EPI_WARPS);
        }
        s_abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&s_tmem_base, TMEM_COLS);
        tmem_relinquish();
    }
    // global memory is read from here on: wait for the previous grid in the stream (programmatic
    // dependent launch), and let the next one start its own set-up
    grid_dependency_wait();
    grid_launch_dependents();
    if (MODE == kMasked) {
        // per-expert tile counts from the device-resident masked_m, then an exclusive prefix sum
        for (int g = threadIdx.x; g < p.groups; g += THREADS) {
            const int mm = min(max(__ldg(p.masked_m + g), 0), p.rows);
            s_prefix[g + 1] = ((mm + BMT - 1) / BMT) * p.n_blocks;
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
    const int a_rows_total = (MODE == kMasked) ? p.groups * p.rows : p.rows;


    // Every CTA of a split-K cluster sees the same tile sequence (the cluster's unit), and every warp of
    // the CTA passes the two cluster barriers of every tile: the control warps right after issuing the
    // tile's work, the epilogue warps around the reduction. A role that is aborting keeps iterating
    // without work so that it still does.
    if (warp < EPI_WARP0) {
        regs_dec<CTRL_REGS>();
        const bool issuer = elect_one();
        int stage = 0, grp = 0, sslot = 0;
        uint32_t phase = 0, gphase = 0, sphase = 0;
        uint32_t issued = 0, issued_parity = 0;      // producer: per-stage bits, for the abort drain
        int last_grp = -1;                            // MMA issuer: last committed group, for the abort drain
        uint32_t last_gparity = 0;
        bool ok = true;
        const uint32_t a_base = smem_u32(smem_a), b_base = smem_u32(smem_b);
        for (int t = unit; t < num_tiles; t += num_units) {
            const DecTile ti = decode_dec<MODE, BMT>(p, t, s_prefix, srank);
            if (warp == 0) {
                // ------------------------------------------------------------ TMA producer
                for (int kb = 0; kb < ti.nkb && ok; ++kb) {
                    // a stage never filled before is free: the first pass over the ring issues its loads
                    // without a barrier round trip
                    if (issued & (1u << stage)) {
                        const bool got = wait_bounded(&empty_bar[stage], phase ^ 1u, abort_flag, p.status, p.wait_limit_ns);
                        if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
                    }
                    if (issuer) {
                        const int x = (ti.kb0 + kb) * BK;
                        mbar_arrive_expect_tx(&full_bar[stage], C::STAGE_BYTES);
                        tma_load_2d(&tmap_a, &full_bar[stage], smem_a + stage * C::A_BYTES, x, ti.a_row);
                        tma_load_2d(&tmap_b, &full_bar[stage], smem_b + stage * C::B_BYTES, x, ti.b_row);
                    }
                    issued |= 1u << stage;
                    issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                    __syncwarp();
                }
            } else if (warp == 1) {
                // ------------------------------------------------------------ MMA issuer
                for (int kb = 0; kb < ti.nkb && ok; ++kb) {
                    const int j = kb % KG;
                    bool got = true;
                    if (j == 0) got = wait_bounded(&tmem_empty_bar[grp], gphase ^ 1u, abort_flag, p.status, p.wait_limit_ns);
                    got = got && wait_bounded(&full_bar[stage], phase, abort_flag, p.status, p.wait_limit_ns);
                    if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>((grp * KG + j) * BMT);
                    // the MMA's M operand is the B tile (128 columns of D), its N operand the A tile
                    const uint64_t m_desc = sw128_kmajor_desc(b_base + stage * C::B_BYTES);
                    const uint64_t n_desc = sw128_kmajor_desc(a_base + stage * C::A_BYTES);
                    const bool group_end = (j == KG - 1) || (kb + 1 == ti.nkb);
                    if (issuer) {
#pragma unroll
                        for (int k = 0; k < BK / UMMA_K; ++k)
                            mma_f8f6f4(d_tmem, m_desc + static_cast<uint64_t>(k * (UMMA_K >> 4)),
                                       n_desc + static_cast<uint64_t>(k * (UMMA_K >> 4)), IDESC, k > 0 ? 1u : 0u);
                        mma_commit(&empty_bar[stage]);
                        if (group_end) mma_commit(&tmem_full_bar[grp]);
                    }
                    __syncwarp();
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                    if (group_end) {
                        last_grp = grp;
                        last_gparity = gphase;
                        if (++grp == NGRP) { grp = 0; gphase ^= 1u; }
                    }
                }
            } else if (warp == 2) {
                // ------------------------------------------------------------ scale stager
                const float* sfa_rows[BMT / 32];
#pragma unroll
                for (int i = 0; i < BMT / 32; ++i)
                    sfa_rows[i] = p.sfa + static_cast<size_t>(min(ti.a_row + lane + 32 * i, a_rows_total - 1)) * p.kbs + ti.kb0;
                const float* sfb_src = p.sfb + (static_cast<size_t>(ti.g) * p.sfb_rows + ti.n0 / 128) * p.kbs + ti.kb0;
                for (int kb = 0; kb < ti.nkb && ok; kb += KG) {
                    const bool got = wait_bounded(&scale_empty_bar[sslot], sphase ^ 1u, abort_flag, p.status, p.wait_limit_ns);
                    if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
                    float* dst = s_scales + sslot * C::SLOT_FLOATS;
                    const int ng = min(KG, ti.nkb - kb);
                    for (int j = 0; j < ng; ++j) {
#pragma unroll
                        for (int i = 0; i < BMT / 32; ++i) cp_async_4(dst + j * C::SROW + lane + 32 * i, sfa_rows[i] + kb + j);
                        if (lane == 0) cp_async_4(dst + j * C::SROW + BMT, sfb_src + kb + j);
                    }
                    cp_async_arrive_noinc(&scale_full_bar[sslot]);
                    if (++sslot == SG) { sslot = 0; sphase ^= 1u; }
                }
            }
            if (split_k) {
                if (warp == 0 && ok) {
                    // every stage of this tile has been consumed (its MMAs have completed) before the
                    // ring holds partial sums; this also leaves no MMA-completion arrival in flight
                    // when the CTA exits after its last tile. The ring position is not advanced: the
                    // wait is the one the next refill of each stage would make.
                    int s = stage;
                    uint32_t ph = phase;
                    for (int i = 0; i < STAGES && ok; ++i) {
                        const bool got = wait_bounded(&empty_bar[s], ph ^ 1u, abort_flag, p.status, p.wait_limit_ns);
                        if (!__all_sync(0xffffffffu, got)) ok = false;
                        if (++s == STAGES) { s = 0; ph ^= 1u; }
                    }
                }
                // the epilogue warps park, reduce and store between these two barriers
                cluster_sync();
                cluster_sync();
            }
        }
        // ------------------------------------------------------------------ drain
        if (warp == 0 && ok && !split_k) {
            // every stage this CTA filled has been consumed, so no MMA-completion arrival is still in
            // flight towards this CTA when it exits (split-K tiles drained the ring before their
            // reduction already)
            int s = stage;
            uint32_t ph = phase;
            for (int i = 0; i < STAGES && ok; ++i) {
                const bool got = wait_bounded(&empty_bar[s], ph ^ 1u, abort_flag, p.status, p.wait_limit_ns);
                if (!__all_sync(0xffffffffu, got)) ok = false;
                if (++s == STAGES) { s = 0; ph ^= 1u; }
            }
        }
        if (warp == 0 && !ok && issuer) {
            for (int s = 0; s < STAGES; ++s)
                if (issued & (1u << s)) drain_wait(&full_bar[s], (issued_parity >> s) & 1u);
        }
        if (warp == 1 && !ok && issuer && last_grp >= 0) drain_wait(&tmem_full_bar[last_grp], last_gparity);
        if (warp == 2) cp_async_wait_all();
        __syncwarp();
    } else {
        // -------------------------------------------------------------------- promotion + store
        regs_inc<EPI_REGS>();
        const int ew = warp - EPI_WARP0;          // 0..7
        const int q = warp & 3;                   // TMEM lane quarter: columns q*32 .. q*32+31 of the tile
        const int h = ew >> 2;                    // warpgroup: rows [h*HALF, (h+1)*HALF) of the tile
        const int n_in_tile = q * 32 + lane;
        const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(h * HALF);
        int grp = 0, sslot = 0;
        uint32_t gphase = 0, sphase = 0;
        bool ok = true;
        for (int t = unit; t < num_tiles; t += num_units) {
            const DecTile ti = decode_dec<MODE, BMT>(p, t, s_prefix, srank);
            float acc[HALF];
#pragma unroll
            for (int m = 0; m < HALF; ++m) acc[m] = 0.f;
            for (int kb = 0; kb < ti.nkb && ok; kb += KG) {
                const int ng = min(KG, ti.nkb - kb);
                bool got = (static_cast<unsigned>(mbar_try_wait(&tmem_full_bar[grp], gphase)) &
                            static_cast<unsigned>(mbar_try_wait(&scale_full_bar[sslot], sphase))) != 0u;
                if (!got)
                    got = wait_bounded(&tmem_full_bar[grp], gphase, abort_flag, p.status, p.wait_limit_ns) &&
                          wait_bounded(&scale_full_bar[sslot], sphase, abort_flag, p.status, p.wait_limit_ns);
                if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
                tc_fence_after();
                // the group's partials of this thread's rows in batches of LB K blocks (the whole group
                // at once unless the registers do not hold it), one wait per batch; the accumulators are
                // released once the last batch is in registers, before its FMAs
                const float* sl = s_scales + sslot * C::SLOT_FLOATS;
#pragma unroll
                for (int jb = 0; jb < KG; jb += LB) {
                    if (jb >= ng) break;
                    uint32_t r[LB][HCH][16];
#pragma unroll
                    for (int j = 0; j < LB; ++j)
#pragma unroll
                        for (int c = 0; c < HCH; ++c)
                            if (jb + j < ng) tmem_ld_x16(lane_addr + static_cast<uint32_t>((grp * KG + jb + j) * BMT + c * 16), r[j][c]);
                    tmem_ld_wait();
                    if (jb + LB >= ng) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&tmem_empty_bar[grp]);
                    }
#pragma unroll
                    for (int j = 0; j < LB; ++j) {
                        if (jb + j < ng) {
                            const float sb = sl[(jb + j) * C::SROW + BMT];
                            const float* sa = sl + (jb + j) * C::SROW + h * HALF;
#pragma unroll
                            for (int c = 0; c < HCH; ++c) {
#pragma unroll
                                for (int e = 0; e < 16; e += 4) {
                                    const float4 s4 = *reinterpret_cast<const float4*>(sa + c * 16 + e);
                                    const int m = c * 16 + e;
                                    acc[m + 0] = fmaf(__uint_as_float(r[j][c][e + 0]), s4.x * sb, acc[m + 0]);
                                    acc[m + 1] = fmaf(__uint_as_float(r[j][c][e + 1]), s4.y * sb, acc[m + 1]);
                                    acc[m + 2] = fmaf(__uint_as_float(r[j][c][e + 2]), s4.z * sb, acc[m + 2]);
                                    acc[m + 3] = fmaf(__uint_as_float(r[j][c][e + 3]), s4.w * sb, acc[m + 3]);
                                }
                            }
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&scale_empty_bar[sslot]);
                if (++grp == NGRP) { grp = 0; gphase ^= 1u; }
                if (++sslot == SG) { sslot = 0; sphase ^= 1u; }
            }
            if (ok) {
                if (split_k) {
                    // park this CTA's partial sums [row m][column n] in the operand ring (every stage of
                    // the tile has been consumed by an MMA that has completed, and the producer issues
                    // nothing more before the second cluster barrier below): a warp writes 128
                    // contiguous bytes per row, and each CTA's share of rows is one contiguous block
                    float* pcol = reinterpret_cast<float*>(smem) + (h * HALF) * C::BNT + n_in_tile;
#pragma unroll
                    for (int m = 0; m < HALF; ++m) pcol[m * C::BNT] = acc[m];
                } else {
                    // column n of D for this warpgroup's rows: a warp writes 64 contiguous bytes per row
                    const int n = ti.n0 + n_in_tile;
                    if (n < p.n) {
                        __nv_bfloat16* dcol = reinterpret_cast<__nv_bfloat16*>(p.d) + n;
                        const size_t d_row = static_cast<size_t>(ti.a_row);
#pragma unroll
                        for (int m = 0; m < HALF; ++m) {
                            const int rr = h * HALF + m;
                            if (rr < ti.rows_valid) dcol[(d_row + rr) * p.n] = __float2bfloat16_rn(acc[m]);
                        }
                    }
                }
            }
            if (split_k) {
                // ------------------------------------------------------------ split-K reduction
                // every CTA's partials are visible cluster-wide after this barrier; CTA s reduces rows
                // [s*BMT/S, (s+1)*BMT/S) of the tile, a contiguous block of every CTA's partials read
                // with consecutive threads on consecutive 16-byte chunks, over all S partials in fixed
                // order (s = 0..S-1), and stores BF16 rows (8 bytes a thread, a warp 256 contiguous
                // bytes); the second barrier keeps every CTA's ring untouched until all remote reads are
                // done (only then does the producer refill it with the next tile)
                cluster_sync();
                if (!*abort_flag) {
                    const int rows_per = BMT / p.split;
                    const int chunks = rows_per * (C::BNT / 4);
                    const uint32_t part_local = smem_u32(smem);
                    for (int f = static_cast<int>(threadIdx.x) - EPI_WARP0 * 32; f < chunks; f += EPI_WARPS * 32) {
                        const int m = srank * rows_per + f / (C::BNT / 4);
                        const int n4 = (f % (C::BNT / 4)) * 4;
                        const float4 sum = cluster_sum_v4(part_local + static_cast<uint32_t>((m * C::BNT + n4) * 4), p.split);
                        if (m < ti.rows_valid && ti.n0 + n4 < p.n) {
                            __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(p.d) +
                                                 static_cast<size_t>(ti.a_row + m) * p.n + ti.n0 + n4;
                            st_global_v2(dst, pack_bf16x2(sum.x, sum.y), pack_bf16x2(sum.z, sum.w));
                        }
                    }
                }
                cluster_sync();
            }
        }
        __syncwarp();
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
