// Swapped-operand variant of the normal GEMM for few rows (small M), for sm_103a.
//
// Same product and scales as dg_gemm_kernel in the normal layout, computed transposed: the tile is
// 128 columns of D (n) x BMT rows of D (m), and the MMA runs with B's 128 rows as its M operand and A's
// BMT rows as its N operand, so TMEM lane n holds column n of the tile and TMEM column m holds row m.
// With few rows this stages 128 B rows (the bytes that come from HBM) plus BMT A rows per K block,
// instead of 128 A rows (mostly past M) plus BN B rows: per K block an SM moves about twice the useful
// bytes. Scales: sfb[n0/128, kb] is one value per tile and K block (the tile's 128 columns are one sfb
// block), sfa[m, kb] varies along the MMA's N, so the promotion is acc[m] += (P[m] * sfa[m]) * sfb.
//
// Warp roles as in dg_gemm_kernel (warp 0 TMA producer, warp 1 TMEM owner and MMA issuer, warp 2 scale
// stager, warps 4..11 promotion and store, setmaxnreg 56 / 224); the two epilogue warpgroups take
// alternate K blocks over all BMT rows and exchange the halves they store once per tile. Each thread
// stores its column n of D for its half of the rows (2-byte stores; a warp writes 64 contiguous bytes
// per row). Split-K over a cluster reduces the FP32 partials through distributed shared memory.
// Every wait is bounded as in dg_gemm_kernel.
#pragma once

#include "dg_kernel.cuh"

namespace dg {

template <int BMT>
struct CfgSW {
    static_assert(BMT == 32 || BMT == 64 || BMT == 128, "BMT is 32, 64 or 128");
    static constexpr int BNT = 128;                      // D columns per tile = MMA M = TMEM lanes
    static constexpr int A_BYTES = BMT * BK;             // A rows of the tile (the MMA's N operand)
    static constexpr int B_BYTES = BNT * BK;             // B rows of the tile (the MMA's M operand)
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int SLOT_FLOATS = BMT + 4;          // sfa of the tile's rows, then sfb
    static constexpr int SCALE_BYTES = SCALE_SLOTS_MAX * SLOT_FLOATS * 4;
    static constexpr int HALF = BMT / 2;                 // rows of D each epilogue warpgroup stores
    static constexpr int XCHG_PASS = HALF < 32 ? HALF : 32;
    static constexpr int XCHG_BYTES = 2 * BNT * XCHG_PASS * 4;
    static constexpr int STATIC_RESERVE = 640;
    static constexpr int STAGES = ring_stages(STAGE_BYTES, SCALE_BYTES + XCHG_BYTES, 0, STATIC_RESERVE);
    static constexpr int NACC_FIT = TMEM_COLS / BMT;
    static constexpr int NACC = NACC_FIT > 8 ? 8 : NACC_FIT;
    static constexpr int XCHG_OFF = STAGES * STAGE_BYTES + SCALE_BYTES;
    static constexpr int DYN_SMEM = 1024 + XCHG_OFF + XCHG_BYTES;
    static constexpr int PSTRIDE = BMT + 4;              // split-K partials [128][BMT + 4] in the ring
    static constexpr int PARTIAL_BYTES = BNT * PSTRIDE * 4;
    static_assert(PARTIAL_BYTES <= STAGES * STAGE_BYTES, "split-K partials must fit in the operand ring");
    static_assert(STAGES >= 2, "not enough shared memory for two stages");
};

struct SwTile {
    int m0, n0, kb0, nkb, rows_valid;
};

// Tiles: column block fastest (few row blocks), K shared by the CTAs of a split-K cluster.
template <int BMT>
__device__ __forceinline__ SwTile decode_sw(const Params& p, int t, int srank) {
    SwTile ti;
    const int nb = t % p.n_blocks, mb = t / p.n_blocks;
    ti.m0 = mb * BMT;
    ti.n0 = nb * 128;
    ti.rows_valid = min(BMT, p.rows - ti.m0);
    ti.kb0 = 0;
    ti.nkb = p.kbs;
    if (p.split > 1) {
        ti.kb0 = (srank * p.kbs) / p.split;
        ti.nkb = ((srank + 1) * p.kbs) / p.split - ti.kb0;
    }
    return ti;
}

template <int BMT>
__global__ void __launch_bounds__(THREADS, 1)
dg_gemm_swap_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                    const __grid_constant__ CUtensorMap tmap_d, const __grid_constant__ Params p) {
    using C = CfgSW<BMT>;
    constexpr int STAGES = C::STAGES;
    constexpr int NACC = C::NACC;
    constexpr int SLOTS = SCALE_SLOTS_MAX;
    constexpr int HALF = C::HALF;
    constexpr uint32_t IDESC = idesc_e4m3_f32(128, BMT);

    extern __shared__ uint8_t dyn_smem[];
    __shared__ uint64_t full_bar[STAGES], empty_bar[STAGES];
    __shared__ uint64_t tmem_full_bar[NACC], tmem_empty_bar[NACC];
    __shared__ uint64_t scale_full_bar[SLOTS], scale_empty_bar[SLOTS];
    __shared__ uint64_t xchg_full_bar, xchg_free_bar;
    __shared__ uint32_t s_tmem_base;
    __shared__ int s_abort;

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
    float* s_xchg = reinterpret_cast<float*>(smem + C::XCHG_OFF);

    if (threadIdx.x == 0) {
        // the tensor maps are fetched while the barriers and TMEM are set up (they are kernel
        // parameters, not data of the previous grid, so this may precede the dependency wait)
        prefetch_tmap(&tmap_a);
        prefetch_tmap(&tmap_b);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        for (int a = 0; a < NACC; ++a) {
            mbar_init(&tmem_full_bar[a], 1);
            mbar_init(&tmem_empty_bar[a], EPI_WARPS / 2);   // one warpgroup promotes each K block
        }
        for (int s = 0; s < SLOTS; ++s) {
            mbar_init(&scale_full_bar[s], 32);
            mbar_init(&scale_empty_bar[s], EPI_WARPS / 2);
        }
        mbar_init(&xchg_full_bar, EPI_WARPS);
        mbar_init(&xchg_free_bar, EPI_WARPS);
        s_abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&s_tmem_base, TMEM_COLS);
        tmem_relinquish();
    }
    grid_dependency_wait();
    grid_launch_dependents();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const uint32_t tmem_base = s_tmem_base;
    volatile int* abort_flag = &s_abort;
    const int num_tiles = p.tiles;

    if (warp < EPI_WARP0) {
        regs_dec<CTRL_REGS>();
        if (warp == 0) {
            // ------------------------------------------------------------------ TMA producer
            const bool issuer = elect_one();
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued = 0, issued_parity = 0;
            bool ok = true;
            for (int t = unit; t < num_tiles && ok; t += num_units) {
                const SwTile ti = decode_sw<BMT>(p, t, srank);
                for (int kb = 0; kb < ti.nkb;) {
                    // a second stage in the same pass when it is free already (narrow-tile pass cost)
                    int s1 = stage + 1;
                    uint32_t ph1 = phase;
                    if (s1 == STAGES) { s1 = 0; ph1 ^= 1u; }
                    const bool more = kb + 1 < ti.nkb;
                    const bool f0 = mbar_try_wait(&empty_bar[stage], phase ^ 1u);
                    const bool f1 = more && mbar_test_wait(&empty_bar[s1], ph1 ^ 1u);
                    const bool got = f0 || wait_bounded(&empty_bar[stage], phase ^ 1u, abort_flag, p.status);
                    if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
                    const int take = __all_sync(0xffffffffu, f1) ? 2 : 1;
                    for (int j = 0; j < take; ++j) {
                        if (issuer) {
                            const int x = (ti.kb0 + kb + j) * BK;
                            mbar_arrive_expect_tx(&full_bar[stage], C::STAGE_BYTES);
                            tma_load_2d(&tmap_a, &full_bar[stage], smem_a + stage * C::A_BYTES, x, ti.m0);
                            tma_load_2d(&tmap_b, &full_bar[stage], smem_b + stage * C::B_BYTES, x, ti.n0);
                        }
                        issued |= 1u << stage;
                        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                    }
                    __syncwarp();
                    kb += take;
                }
            }
            if (ok) {
                for (int i = 0; i < STAGES && ok; ++i) {
                    const bool got = wait_bounded(&empty_bar[stage], phase ^ 1u, abort_flag, p.status);
                    if (!__all_sync(0xffffffffu, got)) ok = false;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok && issuer) {
                for (int s = 0; s < STAGES; ++s)
                    if (issued & (1u << s)) drain_wait(&full_bar[s], (issued_parity >> s) & 1u);
            }
        } else if (warp == 1) {
            // ------------------------------------------------------------------ MMA issuer
            const bool issuer = elect_one();
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true, any = false;
            int last_acc = 0;
            uint32_t last_parity = 0;
            const uint32_t a_base = smem_u32(smem_a), b_base = smem_u32(smem_b);
            for (int t = unit; t < num_tiles && ok; t += num_units) {
                const SwTile ti = decode_sw<BMT>(p, t, srank);
                for (int kb = 0; kb < ti.nkb;) {
                    int s1 = stage + 1, a1 = acc + 1;
                    uint32_t ph1 = phase, ap1 = acc_phase;
                    if (s1 == STAGES) { s1 = 0; ph1 ^= 1u; }
                    if (a1 == NACC) { a1 = 0; ap1 ^= 1u; }
                    const bool more = kb + 1 < ti.nkb;
                    const bool r0 = (static_cast<unsigned>(mbar_try_wait(&tmem_empty_bar[acc], acc_phase ^ 1u)) &
                                     static_cast<unsigned>(mbar_try_wait(&full_bar[stage], phase))) != 0u;
                    const bool r1 = more && (static_cast<unsigned>(mbar_test_wait(&tmem_empty_bar[a1], ap1 ^ 1u)) &
                                             static_cast<unsigned>(mbar_test_wait(&full_bar[s1], ph1))) != 0u;
                    bool got = r0;
                    if (!got)
                        got = wait_bounded(&tmem_empty_bar[acc], acc_phase ^ 1u, abort_flag, p.status) &&
                              wait_bounded(&full_bar[stage], phase, abort_flag, p.status);
                    if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
                    const int take = __all_sync(0xffffffffu, r1) ? 2 : 1;
                    tc_fence_after();
                    for (int j = 0; j < take; ++j) {
                        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BMT);
                        // the MMA's M operand is the B tile (128 columns of D), its N operand the A tile
                        const uint64_t m_desc = sw128_kmajor_desc(b_base + stage * C::B_BYTES);
                        const uint64_t n_desc = sw128_kmajor_desc(a_base + stage * C::A_BYTES);
                        if (issuer) {
#pragma unroll
                            for (int k = 0; k < BK / UMMA_K; ++k)
                                mma_f8f6f4(d_tmem, m_desc + static_cast<uint64_t>(k * (UMMA_K >> 4)),
                                           n_desc + static_cast<uint64_t>(k * (UMMA_K >> 4)), IDESC, k > 0 ? 1u : 0u);
                            mma_commit(&empty_bar[stage]);
                            mma_commit(&tmem_full_bar[acc]);
                        }
                        last_acc = acc;
                        last_parity = acc_phase;
                        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                        if (++acc == NACC) { acc = 0; acc_phase ^= 1u; }
                    }
                    __syncwarp();
                    any = true;
                    kb += take;
                }
            }
            if (!ok && any && issuer) drain_wait(&tmem_full_bar[last_acc], last_parity);
        } else if (warp == 2) {
            // ------------------------------------------------------------------ scale stager
            int slot = 0;
            uint32_t sphase = 0;
            for (int t = unit; t < num_tiles; t += num_units) {
                const SwTile ti = decode_sw<BMT>(p, t, srank);
                const float* sfa_rows[BMT / 32];
#pragma unroll
                for (int i = 0; i < BMT / 32; ++i)
                    sfa_rows[i] = p.sfa + static_cast<size_t>(min(ti.m0 + lane + 32 * i, p.rows - 1)) * p.kbs + ti.kb0;
                const float* sfb_src = p.sfb + static_cast<size_t>(ti.n0 / 128) * p.kbs + ti.kb0;
                bool ok = true;
                for (int kb = 0; kb < ti.nkb; ++kb) {
                    const bool got = wait_bounded(&scale_empty_bar[slot], sphase ^ 1u, abort_flag, p.status);
                    if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
                    float* dst = s_scales + slot * C::SLOT_FLOATS;
#pragma unroll
                    for (int i = 0; i < BMT / 32; ++i) cp_async_4(dst + lane + 32 * i, sfa_rows[i] + kb);
                    if (lane == 0) cp_async_4(dst + BMT, sfb_src + kb);
                    cp_async_arrive_noinc(&scale_full_bar[slot]);
                    if (++slot == SLOTS) { slot = 0; sphase ^= 1u; }
                }
                if (!ok) break;
            }
            cp_async_wait_all();
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------------ promotion + store
        regs_inc<EPI_REGS>();
        const int ew = warp - EPI_WARP0;        // 0..7
        const int q = warp & 3;                 // TMEM lane quarter: columns q*32 .. q*32+31 of the tile
        const int h = ew >> 2;                  // K-block parity promoted, and half of the rows stored
        const int lane_row = q * 32 + lane;     // this thread's column of the tile
        const uint32_t row_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
        int acc = 0, slot = 0;
        uint32_t acc_phase = 0, sphase = 0, xphase = 0;
        bool ok = true;
        for (int t = unit; t < num_tiles && ok; t += num_units) {
            const SwTile ti = decode_sw<BMT>(p, t, srank);
            float accf[BMT];
#pragma unroll
            for (int j = 0; j < BMT; ++j) accf[j] = 0.f;
            for (int kb = 0; kb < ti.nkb; ++kb) {
                if ((kb & 1) == h) {
                    bool got = (static_cast<unsigned>(mbar_try_wait(&tmem_full_bar[acc], acc_phase)) &
                                static_cast<unsigned>(mbar_try_wait(&scale_full_bar[slot], sphase))) != 0u;
                    if (!got)
                        got = wait_bounded(&tmem_full_bar[acc], acc_phase, abort_flag, p.status) &&
                              wait_bounded(&scale_full_bar[slot], sphase, abort_flag, p.status);
                    if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
                    tc_fence_after();
                    constexpr int NCH = BMT / 16;
                    constexpr int LB = NCH < 4 ? NCH : 4;
                    const float* sl = s_scales + slot * C::SLOT_FLOATS;
                    const float sb = sl[BMT];
#pragma unroll
                    for (int b = 0; b < NCH / LB; ++b) {
                        uint32_t rb[LB][16];
#pragma unroll
                        for (int c = 0; c < LB; ++c)
                            tmem_ld_x16(row_addr + static_cast<uint32_t>(acc * BMT + (b * LB + c) * 16), rb[c]);
                        tmem_ld_wait();
                        if (b + 1 == NCH / LB) {
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&tmem_empty_bar[acc]);
                        }
                        // per-column scale sfa[m] (staged), row scale sfb
#pragma unroll
                        for (int c = 0; c < LB; ++c) promote_chunk<kKGrouped, BMT>(accf, rb[c], b * LB + c, 0.f, sb, sl);
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&scale_empty_bar[slot]);
                }
                if (++acc == NACC) { acc = 0; acc_phase ^= 1u; }
                if (++slot == SLOTS) { slot = 0; sphase ^= 1u; }
            }
            if (!ok) break;
            // Exchange: warpgroup h keeps rows [h*HALF, (h+1)*HALF) and hands the other half to the
            // other warpgroup, XCHG_PASS rows per pass, 16-byte chunks swizzled by lane (chunk ^ (lane
            // & (HC - 1))).
            constexpr int PASS = C::XCHG_PASS;
            constexpr int HC = PASS / 4;
            float send[HALF], keep[HALF], accum[HALF];
            if (h == 0) {
#pragma unroll
                for (int j = 0; j < HALF; ++j) { send[j] = accf[HALF + j]; keep[j] = accf[j]; }
            } else {
#pragma unroll
                for (int j = 0; j < HALF; ++j) { send[j] = accf[j]; keep[j] = accf[HALF + j]; }
            }
            float4* mine = reinterpret_cast<float4*>(s_xchg) + (h * 128 + lane_row) * HC;
            const float4* theirs = reinterpret_cast<const float4*>(s_xchg) + ((1 - h) * 128 + lane_row) * HC;
#pragma unroll
            for (int ps = 0; ps < HALF / PASS; ++ps) {
                const bool freed = wait_bounded(&xchg_free_bar, xphase ^ 1u, abort_flag, p.status);
                if (!__all_sync(0xffffffffu, freed)) { ok = false; break; }
#pragma unroll
                for (int c = 0; c < HC; ++c) {
                    const int j = ps * PASS + c * 4;
                    mine[c ^ (lane_row & (HC - 1))] = make_float4(send[j], send[j + 1], send[j + 2], send[j + 3]);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&xchg_full_bar);
                const bool full = wait_bounded(&xchg_full_bar, xphase, abort_flag, p.status);
                if (!__all_sync(0xffffffffu, full)) { ok = false; break; }
#pragma unroll
                for (int c = 0; c < HC; ++c) {
                    const float4 v = theirs[c ^ (lane_row & (HC - 1))];
                    const int j = ps * PASS + c * 4;
                    accum[j + 0] = keep[j + 0] + v.x;
                    accum[j + 1] = keep[j + 1] + v.y;
                    accum[j + 2] = keep[j + 2] + v.z;
                    accum[j + 3] = keep[j + 3] + v.w;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&xchg_free_bar);
                xphase ^= 1u;
            }
            if (!ok) break;
            if (split_k) {
                // park this CTA's partial sums [column][row] in the (idle) operand ring
                float* prow = reinterpret_cast<float*>(smem) + lane_row * C::PSTRIDE + h * HALF;
#pragma unroll
                for (int j = 0; j < HALF; j += 4)
                    *reinterpret_cast<float4*>(prow + j) = make_float4(accum[j], accum[j + 1], accum[j + 2], accum[j + 3]);
                continue;
            }
            // column n of D for this warpgroup's rows; a warp writes 64 contiguous bytes per row
            const int n = ti.n0 + lane_row;
            if (n < p.n) {
                __nv_bfloat16* dcol = reinterpret_cast<__nv_bfloat16*>(p.d) + n;
#pragma unroll
                for (int j = 0; j < HALF; ++j) {
                    const int r = h * HALF + j;
                    if (r < ti.rows_valid) dcol[static_cast<size_t>(ti.m0 + r) * p.n] = __float2bfloat16_rn(accum[j]);
                }
            }
        }
        __syncwarp();
    }

    // ---------------------------------------------------------------------- split-K reduction
    if (split_k) {
        // CTA s reduces columns [s*128/S, (s+1)*128/S) of the tile over all S partials (fixed order),
        // consecutive threads taking consecutive columns so each row of D is written contiguously
        cluster_sync();
        if (warp >= EPI_WARP0 && !*abort_flag) {
            const SwTile ti = decode_sw<BMT>(p, unit, srank);
            const int cols_per = 128 / p.split;
            const int groups = cols_per * (BMT / 4);
            const uint32_t part_local = smem_u32(smem);
            for (int gi = static_cast<int>(threadIdx.x) - EPI_WARP0 * 32; gi < groups; gi += EPI_WARPS * 32) {
                const int col = srank * cols_per + gi % cols_per;
                const int r4 = (gi / cols_per) * 4;
                const uint32_t off = static_cast<uint32_t>((col * C::PSTRIDE + r4) * 4);
                const float4 sum = cluster_sum_v4(part_local + off, p.split);
                const int n = ti.n0 + col;
                if (n < p.n) {
                    __nv_bfloat16* dcol = reinterpret_cast<__nv_bfloat16*>(p.d) + n;
                    const float vals[4] = {sum.x, sum.y, sum.z, sum.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if (r4 + i < ti.rows_valid) dcol[static_cast<size_t>(ti.m0 + r4 + i) * p.n] = __float2bfloat16_rn(vals[i]);
                }
            }
        }
        cluster_sync();
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
