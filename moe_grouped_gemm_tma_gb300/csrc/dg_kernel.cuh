// Persistent, warp-specialised block-scaled FP8 GEMM for sm_103a.
//
// What it computes is the DeepGEMM method as its pages describe it ("DeepSeek DeepGEMM": fine-grained
// scaling with BLOCK_K = 128, two-level accumulation, TMA loads/stores, persistent warp
// specialisation, unaligned block sizes; "DeepSeek Open Source Week - Dia 3": promotion of tensor-core
// partial sums into a higher-precision accumulator):
//
//   D[m,n] = sum_kb sfa[m,kb] * sfb(n,kb) * P_kb[m,n],   P_kb[m,n] = sum_{k in block kb} A[m,k] B[n,k]
//
// Output tiles are (128 * PAIR) x BN. With PAIR = 1 one CTA owns a 128-row tile; with PAIR = 2 a
// cluster of two CTAs on two SMs owns a 256-row tile: each CTA loads its own 128 rows of A and half
// (BN/2 rows) of B, the leader CTA issues tcgen05.mma.cta_group::2 (M = 256) which reads both CTAs'
// shared memory and writes each CTA's 128 accumulator rows into that CTA's TMEM. Per SM this halves
// the B bytes staged per K block.
//
// Warp roles (every CTA; 3 warpgroups):
//   warp 0      TMA producer: one lane streams the A and B tiles of every K block into a STAGES-deep
//               shared-memory ring (128-byte swizzle). The leader's `full` barrier expects the bytes
//               of both CTAs; the peer's loads signal it across the pair.
//   warp 1      TMEM owner (512 columns) and, in the leader, the MMA issuer: one lane issues four
//               MMAs (K = 32) per K block into one of NACC TMEM accumulators, then commits (to both
//               CTAs of a pair) the stage's `empty` barrier and the accumulator's `tmem_full` barrier.
//               Where the accumulators pair up (two of them, one K block per pass) warp 3 issues the
//               odd accumulators' blocks and warp 1 the even ones.
//   warp 2      scale stager (k-grouped layout and narrow tiles): cp.async copies of each K block's sfa
//               column (this CTA's 128 rows) and of the sfb values the tile needs into a
//               SCALE_SLOTS-deep shared ring, ahead of the epilogue; k-grouped tiles load patches of
//               KG_PATCH K blocks per pass. Wide tiles of the other layouts read their scales directly.
//   warps 4..11 promotion / epilogue (two warpgroups, registers raised with setmaxnreg): each thread
//               owns one tile row (its TMEM lane) -- in the k-grouped layout, 4 rows x 2 columns of every
//               8-column group (the 16x256b TMEM load shape), so that it reads a quarter of the
//               per-column scales. Per K block a thread reads the block partial out of TMEM, releases
//               the accumulator (`tmem_empty` in the leader) once its loads have completed, and adds
//               partial * sfa[m,kb] * sfb into FP32 running sums (packed f32x2 FMAs). Wide tiles: the
//               warpgroups split the BN columns. Narrow tiles (BN <= 64): each
//               warpgroup takes every other K block over all columns, and the two partial sums are
//               exchanged once per tile through shared memory. At the end of a tile they round to BF16
//               and either stage the whole tile in shared memory for TMA stores that complete in the
//               background (where that fits beside a four-stage ring) or write it with coalesced plain
//               stores; the weight gradient is added into D with coalesced FP32 vector reductions.
// The MMA of K block kb+1.. overlaps the promotion of block kb (NACC accumulators in flight), and the
// store of one tile overlaps the first MMAs of the next. Small-M GEMMs split K over a cluster of CTAs
// and reduce the FP32 partials through distributed shared memory.
//
// Barrier round trips cost about a hundred cycles each, so the loops probe all barriers of a pass at
// once, and on narrow tiles the producer, MMA issuer and stager take a second ready K block per pass.
//
// Every wait is bounded: after the launch's wait limit (WAIT_LIMIT_NS unless a test shortens it) a
// waiter records DG_DEVICE_TIMEOUT in the status word (the first error recorded wins), raises a
// CTA-wide abort flag, and the CTA drains its own in-flight copies and MMAs (bounded too), frees TMEM
// and exits.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "dg_ptx.cuh"

namespace dg {

constexpr int BM = 128;                 // rows per CTA = UMMA M per CTA (one TMEM lane per row)
constexpr int BK = 128;                 // K block = scaling block
constexpr int UMMA_K = 32;              // K of one kind::f8f6f4 MMA
constexpr int EPI_WARP0 = 4;            // first epilogue warp
constexpr int EPI_WARPS = 8;
constexpr int THREADS = 128 + 32 * EPI_WARPS;
constexpr int CTRL_REGS = 56;           // registers per thread of warpgroup 0 after setmaxnreg
constexpr int EPI_REGS = 224;           // ... of the epilogue warpgroups (128*56 + 256*224 = 384*168)
constexpr int TMEM_COLS = 512;
constexpr int SCALE_SLOTS_MAX = 16;
constexpr int MAX_MASKED_G = 1024;
constexpr int MAX_KGROUPS = 128;
// k-grouped: K blocks per scale patch the stager loads in one pass (a power of two dividing 32 and the
// scale ring's slot count)
constexpr int KG_PATCH = 4;
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
    int m_blocks;              // row blocks of (BM * PAIR) rows: ceil(rows / (BM * PAIR))
    int n_blocks;              // ceil(n / BN)
    int tiles;                 // tile count when known on the host (not masked)
    int split;                 // normal layout, single-CTA tiles: CTAs (a cluster) sharing one tile's K
    int group_m;               // normal / contiguous: row blocks per raster band (row block fastest)
    int overwrite;             // k-grouped: store the tile (D = ...) instead of adding it (D += ...)
    int a_mn, b_mn;            // normal layout: A stored [K, M] / B stored [K, N] (MN-major operands)
    int sf_packed;             // block-scaled: sfa / sfb hold UE8M0 exponents, four K blocks per int32
    int sf_words;              // block-scaled, packed: int32 words per scale row, ceil(kbs / 4)
    int l2_hint;               // normal layout, long K: A loads evict-last, B loads evict-first in L2
    unsigned long long wait_limit_ns;  // bound of every wait (0 = WAIT_LIMIT_NS); tests shorten it
    int fault_skip_first_fill;  // test only (0 in every product call): the producer leaves its first
                                // stage unfilled, so the MMA issuer's wait on it runs out
    int kb_off[MAX_KGROUPS + 1];  // k-grouped: first K block of each expert, kb_off[G] = sumK/128
};

// Deepest operand ring (at most 8 stages) whose dynamic layout -- alignment slack, ring and scale slots
// rounded up to 1 KB, output staging -- fits next to the static shared memory.
constexpr int ring_stages(int stage_bytes, int scale_bytes, int store_bytes, int static_bytes) {
    int s = 8;
    while (s > 1 && 1024 + ((s * stage_bytes + scale_bytes + 1023) / 1024) * 1024 + store_bytes + static_bytes > SMEM_LIMIT)
        --s;
    return s;
}

template <int MODE, int BN, int PAIR>
struct Cfg {
    static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "BN must be a multiple of 32 in [32, 256]");
    static_assert(PAIR == 1 || PAIR == 2, "PAIR is 1 or 2");
    static constexpr int TILE_M = BM * PAIR;
    static constexpr int A_BYTES = BM * BK;
    static constexpr int B_ROWS = BN / PAIR;            // B rows staged by each CTA
    static constexpr int B_BYTES = B_ROWS * BK;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    // scale slot: sfa of the CTA's 128 rows, then sfb: 4 block rows (from n0/128), or, k-grouped, BN
    // per-column values in the epilogue's lane order: per warpgroup column block, four runs of KG_CS
    // floats (lane class t%4: the two columns 2(t%4), 2(t%4)+1 of every 8-column group), each run padded
    // so that the four classes' 16-byte reads fall in distinct banks (KG_CS / 4 odd); the slot is padded
    // by 8 more floats, so that the stager's patch writes -- 8 consecutive positions x 4 consecutive slots
    // per instruction -- fall in distinct banks
    static constexpr int KG_CS = (BN / 8) + (((BN / 32) % 2 == 0) ? 4 : 0);
    static constexpr int SB = (MODE == kKGrouped) ? 2 * 4 * KG_CS + 8 : 4;
    static constexpr int SLOT_FLOATS = BM + SB;
    // the k-grouped slots hold BN per-column values, so they get a shallower ring (eight: six would
    // leave room for a fifth operand stage at BN = 192, but the stager's scattered per-column loads
    // then fall behind, measured 15% slower)
    static constexpr int SCALE_SLOTS = (MODE == kKGrouped) ? 8 : SCALE_SLOTS_MAX;
    static constexpr int SCALE_BYTES = SCALE_SLOTS * SLOT_FLOATS * 4;
    // Epilogue warpgroups (each a column block of the tile); the launch's registers are re-split so
    // that the control warpgroup keeps CTRL_REGS. Three (512 threads, 152 registers each, 64 columns
    // per thread) measured slower than two for the k-grouped layout at BN = 192 (1353 against 1570
    // TFLOP/s), so every specialisation uses two.
    static constexpr int NWG = 2;
    static constexpr int EPI_WARPS_C = 4 * NWG;
    static constexpr int THREADS_C = 128 + 32 * EPI_WARPS_C;
    static constexpr int LAUNCH_REGS = ((65536 / THREADS_C) / 8) * 8;
    static constexpr int EPI_REGS_C = ((THREADS_C * LAUNCH_REGS - 128 * CTRL_REGS) / (THREADS_C - 128) / 8) * 8;
    static constexpr int COLS = BN / NWG;      // columns per epilogue warpgroup
    // static shared memory: barriers and flags (under 640 bytes), plus the masked prefix table
    static constexpr int STATIC_RESERVE = 640 + (MODE == kMasked ? 4 * (MAX_MASKED_G + 1) : 0);
    // Narrow tiles: the two epilogue warpgroups take alternate K blocks over all BN columns (two
    // independent per-block chains in flight) instead of one column half each; once per tile each hands
    // the other the half it does not store, XCHG_PASS columns at a time through shared memory.
    static constexpr bool KPAR = (BN <= 64 && MODE != kKGrouped && NWG == 2);
    static constexpr int XCHG_PASS = (BN / 2) < 32 ? (BN / 2) : 32;
    static constexpr int XCHG_BYTES = KPAR ? 2 * BM * XCHG_PASS * 4 : 0;
    static constexpr int EPI_ARRIVALS = KPAR ? EPI_WARPS_C / 2 : EPI_WARPS_C;   // warps releasing one block
    // Output staging. BF16 out, where it fits next to a ring of at least four stages: the whole CTA tile
    // (each epilogue warp its 32 rows x COLS columns as boxes of 32 x 32 with the 64-byte swizzle),
    // written by TMA stores that the warp does not wait for until it stages its next tile (a tile's
    // 64 KB take the SM's store path several thousand cycles, which would otherwise stall promotion).
    // Otherwise, for BF16 out, 2 KB per epilogue warp: one buffer of 32 rows x 32 columns, written with
    // plain stores. The k-grouped FP32 output needs none: lanes pair up their registers by shuffles into
    // coalesced vector reductions. (Shared memory is kept small for the k-grouped layout: its scale
    // stager relies on what L1 keeps beside it.)
    static constexpr bool FULL_STAGE = MODE != kKGrouped && COLS % 32 == 0 &&
        ring_stages(STAGE_BYTES, SCALE_BYTES + XCHG_BYTES, BM * BN * 2, STATIC_RESERVE) >= 4;
    static constexpr int STORE_WARP_BYTES = FULL_STAGE ? 32 * COLS * 2 : (MODE == kKGrouped ? 0 : 2048);
    static constexpr int STORE_BYTES = EPI_WARPS_C * STORE_WARP_BYTES;
    static constexpr int STAGES = ring_stages(STAGE_BYTES, SCALE_BYTES + XCHG_BYTES, STORE_BYTES, STATIC_RESERVE);
    static constexpr int NACC_FIT = TMEM_COLS / BN;
    static constexpr int NACC = NACC_FIT > 8 ? 8 : NACC_FIT;
    static constexpr int XCHG_OFF = STAGES * STAGE_BYTES + SCALE_BYTES;
    static constexpr int STORE_OFF = ((XCHG_OFF + XCHG_BYTES + 1023) / 1024) * 1024;
    static constexpr int DYN_SMEM = 1024 + STORE_OFF + STORE_BYTES;
    static_assert(COLS % 16 == 0, "each epilogue warpgroup takes whole 16-column chunks");
    static_assert(MODE != kKGrouped || (NWG == 2 && KG_CS >= COLS / 4 && (KG_CS / 4) % 2 == 1),
                  "k-grouped scale runs: one per lane class, a quarter of a warpgroup's columns, odd in 16 bytes");
    static constexpr int CHUNKS = COLS / 16;   // 16-column TMEM loads per K block
    // Narrow tiles (four or more accumulators) and the k-grouped layout let the producer, the MMA issuer
    // and the scale stager take a second K block in the same pass of their loops when it is ready
    // already: a pass costs several hundred cycles of barrier round trips, more than the MMA of a narrow
    // block. (Measured: it slows the wide two-accumulator tiles of the other layouts.)
    static constexpr bool KB_PAIRING = (NACC >= 4) || MODE == kKGrouped;
    // MMA issue takes issue slots from the epilogue warps on the issuing warp's sub-partition (per-block
    // clock stamps: those two warps released each accumulator ~350 cycles after the other six, and
    // moving the issuer to another warp moved the lag with it). Where the accumulators pair up (an even
    // count, one K block per pass), two warps on different sub-partitions share the issue: warp 1 the
    // even accumulators, warp 3 the odd ones.
    static constexpr int MMA_WARPS = (!KB_PAIRING && NACC % 2 == 0) ? 2 : 1;
    // Up to 96 columns a thread, a whole K block fits in registers beside the running sums: all its loads
    // are issued and waited on once, and the accumulator is released before any FMA, which keeps the
    // promotion arithmetic off the two-accumulator MMA -> release -> MMA loop.
    static constexpr bool EPI_ONE = MODE != kKGrouped && COLS <= 96;
    // Wide tiles outside the k-grouped layout read their two scales per K block straight from global
    // memory (L1-resident after a tile's first block), one block ahead, instead of from the scale
    // stager's slots: that takes a barrier round trip per block off the epilogue and leaves the stager
    // warp idle, whose issue slots the epilogue warps of its sub-partition then get (per-block clock
    // stamps showed those warps releasing the accumulator last).
    static constexpr bool DIRECT_SCALES = !KPAR && MODE != kKGrouped;
    // split-K partial sums: [128 rows][BN + 4] FP32 (padded rows: conflict-free 16-byte stores), in the
    // operand ring, which is idle once the tile's last MMA has completed
    static constexpr int PSTRIDE = BN + 4;
    static constexpr int PARTIAL_BYTES = BM * PSTRIDE * 4;
    static_assert(!((MODE == kNormal || MODE == kMasked) && PAIR == 1) || PARTIAL_BYTES <= STAGES * STAGE_BYTES,
                  "split-K partials must fit in the operand ring");
    static_assert(STAGES >= 2, "not enough shared memory for two stages");
    static_assert(B_BYTES % 1024 == 0, "B stage must keep 1024-byte swizzle-atom alignment");
};

struct TileInfo {
    int g, m0, n0;       // m0: first row of this CTA's 128-row part (within the expert for masked)
    int kb0, nkb;        // K blocks [kb0, kb0 + nkb)
    int a_row, b_row;    // TMA row coordinates of this CTA's first A / B row
    int d_row;           // output row of this CTA's first row
    int rows_valid;      // rows of this CTA's part that are stored (may be <= 0)
    bool valid;
};

template <int MODE, int BN, int PAIR>
__device__ __forceinline__ TileInfo decode_tile(const Params& p, int t, const int* s_prefix, int rank, int srank) {
    constexpr int TILE_M = BM * PAIR;
    constexpr int B_ROWS = BN / PAIR;
    TileInfo ti;
    ti.valid = true;
    ti.g = 0;
    ti.kb0 = 0;
    ti.nkb = p.kbs;
    if (MODE == kNormal || MODE == kContiguous) {
        // bands of group_m row blocks; within a band the row block varies fastest. Odd bands take the
        // column blocks in reverse (serpentine), so a band starts on the B column blocks the previous
        // band read last, which may still be in L2 (DRAM reads of 4096 x 7168 x 16384: 324.8 -> 318.2
        // MB; 4096 x 24576 x 1536: 81.7 -> 69.3 MB).
        const int band_tiles = p.group_m * p.n_blocks;
        const int band = t / band_tiles, r = t - band * band_tiles;
        const int m_first = band * p.group_m;
        const int gm = min(p.group_m, p.m_blocks - m_first);
        const int mb = m_first + r % gm;
        const int nb = (band & 1) ? (p.n_blocks - 1 - r / gm) : (r / gm);
        ti.m0 = mb * TILE_M + rank * BM;
        ti.n0 = nb * BN;
        ti.a_row = ti.m0;
        ti.d_row = ti.m0;
        ti.rows_valid = min(BM, p.rows - ti.m0);
        ti.b_row = ti.n0 + rank * B_ROWS;
        if (MODE == kNormal && p.split > 1) {   // this CTA's share of the tile's K blocks
            ti.kb0 = (srank * p.kbs) / p.split;
            ti.nkb = ((srank + 1) * p.kbs) / p.split - ti.kb0;
        }
        if (MODE == kContiguous) {
            const int g = __ldg(p.m_indices + mb * TILE_M);
            ti.valid = (g >= 0 && g < p.groups);
            ti.g = ti.valid ? g : 0;
            ti.b_row += ti.g * p.n;
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
        ti.m0 = mb * TILE_M + rank * BM;
        ti.n0 = nb * BN;
        ti.a_row = g * p.rows + ti.m0;
        ti.d_row = ti.a_row;
        ti.b_row = g * p.n + ti.n0 + rank * B_ROWS;
        ti.rows_valid = min(BM, mm - ti.m0);
        if (p.split > 1) {   // this CTA's share of the tile's K blocks
            ti.kb0 = (srank * p.kbs) / p.split;
            ti.nkb = ((srank + 1) * p.kbs) / p.split - ti.kb0;
        }
    } else {  // kKGrouped
        const int per_g = p.m_blocks * p.n_blocks;
        const int g = t / per_g, local = t - g * per_g;
        const int mb = local % p.m_blocks, nb = local / p.m_blocks;
        ti.g = g;
        ti.m0 = mb * TILE_M + rank * BM;
        ti.n0 = nb * BN;
        ti.kb0 = p.kb_off[g];
        ti.nkb = p.kb_off[g + 1] - p.kb_off[g];
        ti.valid = ti.nkb > 0;
        ti.a_row = ti.m0;
        ti.b_row = ti.n0 + rank * B_ROWS;
        ti.d_row = g * p.rows + ti.m0;
        ti.rows_valid = min(BM, p.rows - ti.m0);
    }
    return ti;
}

// Record a device-side error in the status word unless one is recorded already (the first error since
// the host last read and cleared the word wins; a later one does not overwrite it).
__device__ __forceinline__ void record_status(int* status, int code) { atomicCAS(status, 0, code); }

// Bounded mbarrier wait. Returns false when this CTA is aborting (this waiter timed out, or another
// role did); the first waiter to time out records the status and raises the abort flag. `limit_ns` is
// the launch's wait limit (0 = WAIT_LIMIT_NS). Between checks of the flag and the clock the thread
// waits in try_wait with a 1 us suspend hint, so that a waiting warp is suspended instead of polling:
// a polling warp takes issue slots from the epilogue warps of its sub-partition (per-block clock stamps:
// a control warp polling with plain try_wait delayed those warps' accumulator release by ~350 cycles
// per K block; test_wait with a 32 ns sleep between polls, 0.5-1% slower than the suspend hint).
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                             int* status, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t limit = limit_ns ? limit_ns : WAIT_LIMIT_NS;
    const uint64_t t0 = global_timer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 8; ++i)
            if (mbar_try_wait_hint(bar, parity, 1000)) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > limit) {
            *abort_flag = 1;
            record_status(status, STATUS_TIMEOUT);
            return false;
        }
    }
}

// Short bounded wait used only while draining.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_timer_ns() - t0 > DRAIN_LIMIT_NS) return;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ float pick4(const float4& v, int i) {
    return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// Promotion of one 16-column chunk c of a K block's partial sums r into the running sums:
// acc += r * s (s = sfa * sfb of the chunk's 128-column block).
template <int COLS>
__device__ __forceinline__ void promote_chunk(float (&accum)[COLS], const uint32_t* r, int c, float s) {
    const float2 s2 = make_float2(s, s);
#pragma unroll
    for (int j = 0; j < 16; j += 2) {
        float2 a = make_float2(accum[c * 16 + j], accum[c * 16 + j + 1]);
        a = __ffma2_rn(make_float2(__uint_as_float(r[j]), __uint_as_float(r[j + 1])), s2, a);
        accum[c * 16 + j] = a.x;
        accum[c * 16 + j + 1] = a.y;
    }
}

// k-grouped promotion of one 16-column chunk c (8-column groups 2c and 2c + 1) in the 16x256b register
// layout: lo holds the lanes base .. base + 15 (the lane's rows 0 and 1), hi base + 16 .. base + 31
// (rows 2 and 3); sv the lane's column scales (group 2c: x, y; group 2c + 1: z, w), sa its four row
// scales. accum[(j * 4 + i) * 2 + e] += (P * sfb) * sfa for group j, row i, column e of the lane's pair.
template <int COLS>
__device__ __forceinline__ void promote_kg_chunk(float (&accum)[COLS], const uint32_t* lo, const uint32_t* hi, int c,
                                                 const float4& sv, const float4& sa) {
#pragma unroll
    for (int m = 0; m < 2; ++m) {
        const float2 sb = m ? make_float2(sv.z, sv.w) : make_float2(sv.x, sv.y);
        const int j = 2 * c + m;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t* w = (i < 2 ? lo : hi) + 4 * m + 2 * (i & 1);
            const float s = i == 0 ? sa.x : (i == 1 ? sa.y : (i == 2 ? sa.z : sa.w));
            float2 a = make_float2(accum[(j * 4 + i) * 2], accum[(j * 4 + i) * 2 + 1]);
            const float2 pr = __fmul2_rn(make_float2(__uint_as_float(w[0]), __uint_as_float(w[1])), sb);
            a = __ffma2_rn(pr, make_float2(s, s), a);
            accum[(j * 4 + i) * 2] = a.x;
            accum[(j * 4 + i) * 2 + 1] = a.y;
        }
    }
}

template <int MODE, int BN, int PAIR>
__global__ void __launch_bounds__(Cfg<MODE, BN, PAIR>::THREADS_C, 1)
dg_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
               const __grid_constant__ CUtensorMap tmap_d, const __grid_constant__ Params p) {
    using C = Cfg<MODE, BN, PAIR>;
    constexpr int STAGES = C::STAGES;
    constexpr int NACC = C::NACC;
    constexpr int COLS = C::COLS;
    constexpr int CHUNKS = C::CHUNKS;
    constexpr uint32_t IDESC = idesc_e4m3_f32(C::TILE_M, BN);

    extern __shared__ uint8_t dyn_smem[];
    __shared__ uint64_t full_bar[STAGES], empty_bar[STAGES];
    __shared__ uint64_t tmem_full_bar[NACC], tmem_empty_bar[NACC];
    __shared__ uint64_t scale_full_bar[C::SCALE_SLOTS], scale_empty_bar[C::SCALE_SLOTS];
    __shared__ uint64_t xchg_full_bar, xchg_free_bar;   // narrow-tile partial-sum exchange
    __shared__ uint32_t s_tmem_base;
    __shared__ int s_abort;
    __shared__ int s_prefix[MODE == kMasked ? MAX_MASKED_G + 1 : 1];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // split-K: a cluster of p.split CTAs shares one tile (one tile per cluster), each CTA a K range
    const bool split_k = ((MODE == kNormal || MODE == kMasked) && PAIR == 1 && p.split > 1);
    const int crank = (PAIR == 2 || split_k) ? static_cast<int>(cluster_ctarank()) : 0;
    const int rank = (PAIR == 2) ? crank : 0;      // row half of a CTA-pair tile
    const int srank = split_k ? crank : 0;         // K share of a split-K tile
    const bool leader = (rank == 0);
    const int csize = (PAIR == 2) ? 2 : (split_k ? p.split : 1);
    const int unit = static_cast<int>(blockIdx.x) / csize;
    const int num_units = static_cast<int>(gridDim.x) / csize;

    // 1024-byte aligned operand ring (128-byte swizzle atoms are 1024 bytes); identical offsets in
    // both CTAs of a pair, which the pair MMA relies on
    const uint32_t raw = smem_u32(dyn_smem);
    uint8_t* smem = dyn_smem + (((raw + 1023u) & ~1023u) - raw);
    uint8_t* smem_a = smem;
    uint8_t* smem_b = smem + STAGES * C::A_BYTES;
    float* s_scales = reinterpret_cast<float*>(smem + STAGES * C::STAGE_BYTES);
    uint8_t* s_store = smem + C::STORE_OFF;
    float* s_xchg = reinterpret_cast<float*>(smem + C::XCHG_OFF);

    if (threadIdx.x == 0) {
        // the tensor maps are fetched while the barriers and TMEM are set up (they are kernel
        // parameters, not data of the previous grid, so this may precede the dependency wait)
        prefetch_tmap(&tmap_a);
        prefetch_tmap(&tmap_b);
        if (MODE != kKGrouped) prefetch_tmap(&tmap_d);   // the gradient is added without a tensor map
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        for (int a = 0; a < NACC; ++a) {
            mbar_init(&tmem_full_bar[a], 1);
            mbar_init(&tmem_empty_bar[a], C::EPI_ARRIVALS * PAIR);
        }
        for (int s = 0; s < C::SCALE_SLOTS; ++s) {
            mbar_init(&scale_full_bar[s], 32);
            mbar_init(&scale_empty_bar[s], C::EPI_ARRIVALS);
        }
        {
            mbar_init(&xchg_full_bar, C::EPI_WARPS_C);
            mbar_init(&xchg_free_bar, C::EPI_WARPS_C);
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
    // Everything above touches only shared memory, TMEM and kernel parameters; from here on global
    // memory is read or written, so wait for the previous grid in the stream (programmatic dependent
    // launch), and let the next one start its own set-up.
    grid_dependency_wait();
    grid_launch_dependents();
    if (MODE == kMasked) {
        // per-expert tile counts, then an exclusive prefix sum (one warp)
        for (int g = threadIdx.x; g < p.groups; g += C::THREADS_C) {
            const int mm = min(max(__ldg(p.masked_m + g), 0), p.rows);
            s_prefix[g + 1] = ((mm + C::TILE_M - 1) / C::TILE_M) * p.n_blocks;
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
    if (PAIR == 2) cluster_sync(); else __syncthreads();
    tc_fence_after();

    const uint32_t tmem_base = s_tmem_base;
    volatile int* abort_flag = &s_abort;
    const int num_tiles = (MODE == kMasked) ? s_prefix[p.groups] : p.tiles;

    if (warp < EPI_WARP0) {
        regs_dec<CTRL_REGS>();
        if (warp == 0) {
            // ------------------------------------------------------------------ TMA producer
            // The whole warp runs the loop (warp-uniform operands); one elected lane issues.
            const bool issuer = elect_one();
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued = 0, issued_parity = 0;   // per-stage bits, for the abort drain
            bool ok = true;
            bool skip_fill = p.fault_skip_first_fill != 0;   // test only: leave the first stage empty
            // L2 policies for the long-K normal layout: a band's A row blocks are read again by the next
            // round of tiles, B's column blocks only by tiles in flight at the same time
            const uint64_t pol_a = policy_evict_last(), pol_b = policy_evict_first();
            const bool hint = (MODE == kNormal && PAIR == 1 && p.l2_hint != 0);
            for (int t = unit; t < num_tiles && ok; t += num_units) {
                const TileInfo ti = decode_tile<MODE, BN, PAIR>(p, t, s_prefix, rank, srank);
                if (!ti.valid) continue;
                for (int kb = 0; kb < ti.nkb;) {
                    // The next stage and, when the tile has another K block, the one after it are probed
                    // at once; the second is filled in the same pass only if it is free already. (Each
                    // pass of this loop costs several hundred cycles of barrier round trips, which
                    // narrow tiles would otherwise pay per K block.)
                    int s1 = stage + 1;
                    uint32_t ph1 = phase;
                    if (s1 == STAGES) { s1 = 0; ph1 ^= 1u; }
                    const bool more = C::KB_PAIRING && kb + 1 < ti.nkb;
                    const bool f0 = mbar_try_wait(&empty_bar[stage], phase ^ 1u);
                    const bool f1 = more && mbar_test_wait(&empty_bar[s1], ph1 ^ 1u);
                    const bool got = f0 || wait_bounded(&empty_bar[stage], phase ^ 1u, abort_flag, p.status, p.wait_limit_ns);
                    if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
                    const int take = __all_sync(0xffffffffu, f1) ? 2 : 1;
                    for (int j = 0; j < take; ++j) {
                        const int x = (ti.kb0 + kb + j) * BK;
                        uint8_t* a_dst = smem_a + stage * C::A_BYTES;
                        uint8_t* b_dst = smem_b + stage * C::B_BYTES;
                        if (skip_fill) {
                            // test only: no expect_tx, no copy, so this stage's `full` phase never
                            // completes and the MMA issuer's bounded wait on it expires
                            skip_fill = false;
                            if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                            continue;
                        }
                        if (PAIR == 1 || leader) {
                            if (issuer) {
                                mbar_arrive_expect_tx(&full_bar[stage], PAIR * C::STAGE_BYTES);
                                // MN-major operands: boxes of 128 M (N) bytes x 128 k rows; B takes one
                                // box per 128 columns of the tile (the host allows it for BN % 128 == 0)
                                if ((MODE == kNormal && p.a_mn)) tma_load_2d(&tmap_a, &full_bar[stage], a_dst, ti.a_row, x);
                                else if (hint) tma_load_2d_hint(&tmap_a, &full_bar[stage], a_dst, x, ti.a_row, pol_a);
                                else tma_load_2d(&tmap_a, &full_bar[stage], a_dst, x, ti.a_row);
                                if ((MODE == kNormal && p.b_mn)) {
                                    for (int j = 0; j < C::B_ROWS / 128; ++j)
                                        tma_load_2d(&tmap_b, &full_bar[stage], b_dst + j * (128 * BK), ti.b_row + 128 * j, x);
                                } else if (hint) {
                                    tma_load_2d_hint(&tmap_b, &full_bar[stage], b_dst, x, ti.b_row, pol_b);
                                } else {
                                    tma_load_2d(&tmap_b, &full_bar[stage], b_dst, x, ti.b_row);
                                }
                            }
                        } else {
                            const uint32_t bar = mapa_shared(smem_u32(&full_bar[stage]), 0);
                            if (issuer) {
                                tma_load_2d_pair(&tmap_a, bar, a_dst, x, ti.a_row);
                                tma_load_2d_pair(&tmap_b, bar, b_dst, x, ti.b_row);
                            }
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
                // wait until every stage this CTA filled has been consumed, so no MMA-completion
                // arrival can still be in flight towards this CTA when it exits
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
        } else if ((warp == 1 || (C::MMA_WARPS == 2 && warp == 3)) && leader) {
            // ------------------------------------------------------------------ MMA issuer
            // The whole warp runs the loop so descriptors and TMEM addresses are warp-uniform (kept in
            // uniform registers); one elected lane issues the MMAs and commits. With two issuing warps
            // (see Cfg::MMA_WARPS) warp 1 takes the K blocks of the even accumulators and warp 3 those of
            // the odd ones; each walks every block to keep the ring positions.
            const bool issuer = elect_one();
            const int mine = (warp == 3) ? 1 : 0;
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true, any = false;
            int last_acc = 0;
            uint32_t last_parity = 0;
            const uint32_t a_base = smem_u32(smem_a), b_base = smem_u32(smem_b);
            for (int t = unit; t < num_tiles && ok; t += num_units) {
                const TileInfo ti = decode_tile<MODE, BN, PAIR>(p, t, s_prefix, rank, srank);
                if (!ti.valid) continue;
                for (int kb = 0; kb < ti.nkb;) {
                    if (C::MMA_WARPS == 2 && (acc & 1) != mine) {
                        // the other issuing warp's block: only the ring positions move
                        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                        if (++acc == NACC) { acc = 0; acc_phase ^= 1u; }
                        ++kb;
                        continue;
                    }
                    // This K block's accumulator and stage and, when the tile has another K block, the
                    // next ones are probed at once; the second block is issued in the same pass only if it
                    // is ready already (never waited for, so a two-accumulator tile keeps its overlap).
                    int s1 = stage + 1, a1 = acc + 1;
                    uint32_t ph1 = phase, ap1 = acc_phase;
                    if (s1 == STAGES) { s1 = 0; ph1 ^= 1u; }
                    if (a1 == NACC) { a1 = 0; ap1 ^= 1u; }
                    const bool more = C::KB_PAIRING && kb + 1 < ti.nkb;
                    const bool r0 = (static_cast<unsigned>(mbar_try_wait(&tmem_empty_bar[acc], acc_phase ^ 1u)) &
                                     static_cast<unsigned>(mbar_try_wait(&full_bar[stage], phase))) != 0u;
                    const bool r1 = more && (static_cast<unsigned>(mbar_test_wait(&tmem_empty_bar[a1], ap1 ^ 1u)) &
                                             static_cast<unsigned>(mbar_test_wait(&full_bar[s1], ph1))) != 0u;
                    bool got = r0;
                    if (!got)
                        got = wait_bounded(&tmem_empty_bar[acc], acc_phase ^ 1u, abort_flag, p.status, p.wait_limit_ns) &&
                              wait_bounded(&full_bar[stage], phase, abort_flag, p.status, p.wait_limit_ns);
                    if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
                    const int take = __all_sync(0xffffffffu, r1) ? 2 : 1;
                    tc_fence_after();
                    for (int j = 0; j < take; ++j) {
                        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                        const uint32_t a_addr = a_base + stage * C::A_BYTES, b_addr = b_base + stage * C::B_BYTES;
                        const uint64_t a_desc = (MODE == kNormal && p.a_mn) ? sw128_mnmajor_desc(a_addr, 128 * BK) : sw128_kmajor_desc(a_addr);
                        const uint64_t b_desc = (MODE == kNormal && p.b_mn) ? sw128_mnmajor_desc(b_addr, 128 * BK) : sw128_kmajor_desc(b_addr);
                        // K-major: K = 32 is 32 bytes along the swizzled row (>> 4 = 2); MN-major: 32 rows
                        // of k, four whole 1024-byte atoms (>> 4 = 256)
                        const uint32_t a_kstep = (MODE == kNormal && p.a_mn) ? (32 * 128) >> 4 : UMMA_K >> 4;
                        const uint32_t b_kstep = (MODE == kNormal && p.b_mn) ? (32 * 128) >> 4 : UMMA_K >> 4;
                        const uint32_t idesc = IDESC | ((MODE == kNormal && p.a_mn) ? IDESC_A_MN : 0u) | ((MODE == kNormal && p.b_mn) ? IDESC_B_MN : 0u);
                        if (issuer) {
#pragma unroll
                            for (int k = 0; k < BK / UMMA_K; ++k) {
                                const uint64_t ad = a_desc + static_cast<uint64_t>(k * a_kstep);
                                const uint64_t bd = b_desc + static_cast<uint64_t>(k * b_kstep);
                                if (PAIR == 2) mma_f8f6f4_pair(d_tmem, ad, bd, idesc, k > 0 ? 1u : 0u);
                                else mma_f8f6f4(d_tmem, ad, bd, idesc, k > 0 ? 1u : 0u);
                            }
                            if (PAIR == 2) {
                                mma_commit_pair(&empty_bar[stage], 0x3);
                                mma_commit_pair(&tmem_full_bar[acc], 0x3);
                            } else {
                                mma_commit(&empty_bar[stage]);
                                mma_commit(&tmem_full_bar[acc]);
                            }
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
        } else if (warp == 2 && !C::DIRECT_SCALES) {
            // ------------------------------------------------------------------ scale stager
            int slot = 0;
            uint32_t sphase = 0;
            const int a_rows_total = (MODE == kMasked) ? p.groups * p.rows : p.rows;
            for (int t = unit; t < num_tiles; t += num_units) {
                const TileInfo ti = decode_tile<MODE, BN, PAIR>(p, t, s_prefix, rank, srank);
                if (!ti.valid) continue;
                const float* sfa_rows[4];
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    sfa_rows[i] = p.sfa + static_cast<size_t>(min(ti.a_row + lane + 32 * i, a_rows_total - 1)) * p.kbs + ti.kb0;
                const int blk = min(ti.n0 / 128 + (lane & 3), p.sfb_rows - 1);
                const float* sfb_src = p.sfb + (static_cast<size_t>(ti.g) * p.sfb_rows + blk) * p.kbs + ti.kb0;
                bool ok = true;
                if constexpr (MODE == kKGrouped) {
                    // Patches of KG_PATCH consecutive K blocks: lane (r, kk) fills slot positions r, r + 8,
                    // ... for the patch's K block kk, so that each load instruction reads 8 rows x 16
                    // contiguous bytes instead of 32 scattered words; each lane then arrives on every slot
                    // of the patch, which completes when all of the patch has landed. Positions are in the
                    // epilogue's lane order: sfa position 32w + 4a + i holds row 32w + 8i + a, and the
                    // sfb run of lane class cls in column block hh holds, at 2j + e, column
                    // hh * COLS + 8j + 2cls + e.
                    const int kk = lane & (KG_PATCH - 1), rc = lane / KG_PATCH;
                    for (int kb = 0; kb < ti.nkb;) {
                        const int np = min(KG_PATCH, ti.nkb - kb);
                        bool got = true;
                        int s = slot;
                        uint32_t ph = sphase;
                        for (int j = 0; j < np; ++j) {
                            got = got && (mbar_try_wait(&scale_empty_bar[s], ph ^ 1u) ||
                                          wait_bounded(&scale_empty_bar[s], ph ^ 1u, abort_flag, p.status, p.wait_limit_ns));
                            if (++s == C::SCALE_SLOTS) { s = 0; ph ^= 1u; }
                        }
                        if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
                        if (kk < np) {
                            const int my = (slot + kk) % C::SCALE_SLOTS;
                            float* dst = s_scales + my * C::SLOT_FLOATS;
                            const int k = ti.kb0 + kb + kk;
                            // sfa: lane rc fills positions rc + 8 it, i.e. rows ra + 32 (it / 4) + 2 (it % 4)
                            const int ra = 8 * (rc & 3) + (rc >> 2);
                            const int rmax = a_rows_total - 1 - ti.a_row;
                            const float* sa_k = p.sfa + static_cast<size_t>(ti.a_row) * p.kbs + k;
#pragma unroll 4
                            for (int it = 0; it < BM / 8; ++it) {
                                const int r = min(ra + 32 * (it >> 2) + 2 * (it & 3), rmax);
                                cp_async_4(dst + rc + 8 * it, sa_k + static_cast<size_t>(r) * p.kbs);
                            }
                            // sfb: lane rc fills positions rc + 8 j of every run (hh, cls), i.e. columns
                            // cb + hh * COLS + 2 cls + 32 j
                            constexpr int RUN = COLS / 4;
                            const int cb = 8 * (rc >> 1) + (rc & 1);
                            const int cmax = p.n - 1 - ti.n0;
                            const float* sb_k = p.sfb + static_cast<size_t>(ti.n0) * p.kbs + k;
#pragma unroll 1
                            for (int run = 0; run < 8; ++run) {
                                const int hh = run >> 2, cls = run & 3;
#pragma unroll
                                for (int j = 0; j < (RUN + 7) / 8; ++j) {
                                    if (8 * j + 8 <= RUN || rc + 8 * j < RUN) {
                                        const int c = min(cb + hh * COLS + 2 * cls + 32 * j, cmax);
                                        cp_async_4(dst + BM + hh * 4 * C::KG_CS + cls * C::KG_CS + rc + 8 * j,
                                                   sb_k + static_cast<size_t>(c) * p.kbs);
                                    }
                                }
                            }
                        }
                        for (int j = 0; j < np; ++j) {
                            cp_async_arrive_noinc(&scale_full_bar[slot]);
                            if (++slot == C::SCALE_SLOTS) { slot = 0; sphase ^= 1u; }
                        }
                        kb += np;
                    }
                } else {
                    for (int kb = 0; kb < ti.nkb;) {
                        // as in the producer: a second slot is filled in the same pass if it is free already
                        int s1 = slot + 1;
                        uint32_t sp1 = sphase;
                        if (s1 == C::SCALE_SLOTS) { s1 = 0; sp1 ^= 1u; }
                        const bool more = C::KB_PAIRING && kb + 1 < ti.nkb;
                        const bool f0 = mbar_try_wait(&scale_empty_bar[slot], sphase ^ 1u);
                        const bool f1 = more && mbar_test_wait(&scale_empty_bar[s1], sp1 ^ 1u);
                        // the stager runs several slots ahead, so the wake-up latency of its suspended wait
                        // is hidden
                        const bool got = f0 || wait_bounded(&scale_empty_bar[slot], sphase ^ 1u, abort_flag, p.status, p.wait_limit_ns);
                        if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
                        const int take = __all_sync(0xffffffffu, f1) ? 2 : 1;
                        for (int j = 0; j < take; ++j) {
                            const int k = kb + j;
                            float* dst = s_scales + slot * C::SLOT_FLOATS;
#pragma unroll
                            for (int i = 0; i < 4; ++i) cp_async_4(dst + lane + 32 * i, sfa_rows[i] + k);
                            if (lane < 4) {
                                cp_async_4(dst + BM + lane, sfb_src + k);
                            }
                            cp_async_arrive_noinc(&scale_full_bar[slot]);
                            if (++slot == C::SCALE_SLOTS) { slot = 0; sphase ^= 1u; }
                        }
                        kb += take;
                    }
                }
                if (!ok) break;
            }
            cp_async_wait_all();
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------------ promotion + epilogue
        regs_inc<C::EPI_REGS_C>();
        const int ew = warp - EPI_WARP0;       // 0..7
        const int q = warp & 3;                // TMEM lane quarter this warp may access
        const int h = ew >> 2;                 // epilogue warpgroup: its column block of the tile
        const int row_in_tile = q * 32 + lane;
        const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + h * COLS;
        uint32_t xphase = 0;                   // narrow-tile exchange rounds so far (parity)
        int acc = 0, slot = 0;
        uint32_t acc_phase = 0, sphase = 0;
        bool ok = true;

        for (int t = unit; t < num_tiles && ok; t += num_units) {
            const TileInfo ti = decode_tile<MODE, BN, PAIR>(p, t, s_prefix, rank, srank);
            if (!ti.valid) continue;
            const int cstart = ti.n0 + h * COLS;   // first output column of this thread
            const int split = (128 * (cstart / 128 + 1) - cstart) / 16;   // chunks before the next block

            // the k-grouped output is added into D at the tile's end, so every layout starts the tile's
            // sum at zero
            float accum[COLS];
#pragma unroll
            for (int j = 0; j < COLS; ++j) accum[j] = 0.f;

            if constexpr (C::DIRECT_SCALES) {
                // sfa of this thread's row and the sfb of its (at most two) 128-column blocks, read one K
                // block ahead
                const int a_rows_total = (MODE == kMasked) ? p.groups * p.rows : p.rows;
                const float* sfa_row = p.sfa + static_cast<size_t>(min(ti.a_row + row_in_tile, a_rows_total - 1)) * p.kbs + ti.kb0;
                const float* sfb_0 = p.sfb + (static_cast<size_t>(ti.g) * p.sfb_rows + min(cstart / 128, p.sfb_rows - 1)) * p.kbs + ti.kb0;
                const float* sfb_1 = p.sfb + (static_cast<size_t>(ti.g) * p.sfb_rows + min(cstart / 128 + 1, p.sfb_rows - 1)) * p.kbs + ti.kb0;
                float sa_n = __ldg(sfa_row), b0_n = __ldg(sfb_0), b1_n = __ldg(sfb_1);
                // Each K block's TMEM loads in two halves: the first half is loaded and promoted, then the
                // second half is loaded and the accumulator released before its FMAs, so the MMA of block
                // kb + NACC waits for half a block's FMAs instead of three quarters (EPI_ONE tiles load the
                // whole block before any FMA).
                constexpr int H1 = C::EPI_ONE ? CHUNKS : (CHUNKS + 1) / 2;
                constexpr int H2 = CHUNKS - H1;
                for (int kb = 0; kb < ti.nkb; ++kb) {
                    const float sa = sa_n, b0 = b0_n, b1 = b1_n;
                    if (kb + 1 < ti.nkb) {
                        sa_n = __ldg(sfa_row + kb + 1);
                        b0_n = __ldg(sfb_0 + kb + 1);
                        b1_n = __ldg(sfb_1 + kb + 1);
                    }
                    bool got = mbar_try_wait(&tmem_full_bar[acc], acc_phase);
                    if (!got) got = wait_bounded(&tmem_full_bar[acc], acc_phase, abort_flag, p.status, p.wait_limit_ns);
                    if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t taddr = lane_addr + static_cast<uint32_t>(acc * BN);
                    const float s0 = sa * b0, s1 = sa * b1;
                    uint32_t rb[H1][16];
#pragma unroll
                    for (int c = 0; c < H1; ++c) tmem_ld_x16(taddr + c * 16, rb[c]);
                    tmem_ld_wait();
                    if constexpr (H2 > 0) {
#pragma unroll
                        for (int c = 0; c < H1; ++c) promote_chunk<COLS>(accum, rb[c], c, (c < split) ? s0 : s1);
#pragma unroll
                        for (int c = 0; c < H2; ++c) tmem_ld_x16(taddr + (H1 + c) * 16, rb[c]);
                        tmem_ld_wait();
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        // the accumulator is released on the leader's barrier (the peer's is unused)
                        if (PAIR == 2 && !leader) mbar_arrive_cluster(mapa_shared(smem_u32(&tmem_empty_bar[acc]), 0));
                        else mbar_arrive(&tmem_empty_bar[acc]);
                    }
                    if constexpr (H2 > 0) {
#pragma unroll
                        for (int c = 0; c < H2; ++c)
                            promote_chunk<COLS>(accum, rb[c], H1 + c, (H1 + c < split) ? s0 : s1);
                    } else {
#pragma unroll
                        for (int c = 0; c < H1; ++c) promote_chunk<COLS>(accum, rb[c], c, (c < split) ? s0 : s1);
                    }
                    if (++acc == NACC) { acc = 0; acc_phase ^= 1u; }
                }
            } else if constexpr (MODE == kKGrouped) {
                // Per-column scales (weight gradient). The TMEM loads take the 16x256b shape: a lane holds
                // rows t/4 + 8i (i = 0..3) of the warp's 32 and, of every 8-column group, columns 2(t%4)
                // and 2(t%4) + 1, so it needs the column scales of only a quarter of its column block.
                // The stager stores them in that order: one 16-byte read gives the lane's four row
                // scales, one more its column scales of two groups. Loads in batches of two 16-column
                // chunks, double-buffered; the accumulator is released once the last batch has landed,
                // before its FMAs; the scale slot after the FMAs that read it.
                constexpr int GC = 2;
                constexpr int NG = (CHUNKS + GC - 1) / GC;
                const float* sa_src = s_scales + q * 32 + (lane >> 2) * 4;
                const float* sb_src = s_scales + BM + h * 4 * C::KG_CS + (lane & 3) * C::KG_CS;
                bool pre = false;   // this block's barriers were found complete by the probe below
                for (int kb = 0; kb < ti.nkb; ++kb) {
                    bool got = pre;
                    if (!got)
                        got = (static_cast<unsigned>(mbar_try_wait(&tmem_full_bar[acc], acc_phase)) &
                               static_cast<unsigned>(mbar_try_wait(&scale_full_bar[slot], sphase))) != 0u;
                    if (!got)
                        got = wait_bounded(&tmem_full_bar[acc], acc_phase, abort_flag, p.status, p.wait_limit_ns) &&
                              wait_bounded(&scale_full_bar[slot], sphase, abort_flag, p.status, p.wait_limit_ns);
                    if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t taddr = lane_addr + static_cast<uint32_t>(acc * BN);
                    const float4 sa4 = *reinterpret_cast<const float4*>(sa_src + slot * C::SLOT_FLOATS);
                    const float4* sb4 = reinterpret_cast<const float4*>(sb_src + slot * C::SLOT_FLOATS);
                    uint32_t rb[2][2][GC * 8];   // [buffer][lane half][chunk * 8 + word]
                    // a whole batch of 32 columns per load where every batch starts on a 32-column boundary
                    // (column blocks of 64, 96 and 128), two 16-column loads otherwise
                    constexpr bool X4 = (GC == 2) && (COLS % 32 == 0);
                    auto load_batch = [&](int g, uint32_t (&dst)[2][GC * 8]) {
                        if constexpr (X4) {
                            const uint32_t col = static_cast<uint32_t>(g * 32);
                            tmem_ld_16x256b_x4(taddr + col, &dst[0][0]);
                            tmem_ld_16x256b_x4(taddr + (16u << 16) + col, &dst[1][0]);
                        } else {
#pragma unroll
                            for (int cc = 0; cc < GC; ++cc)
                                if (g * GC + cc < CHUNKS) {
                                    const uint32_t col = static_cast<uint32_t>((g * GC + cc) * 16);
                                    tmem_ld_16x256b_x2(taddr + col, &dst[0][cc * 8]);
                                    tmem_ld_16x256b_x2(taddr + (16u << 16) + col, &dst[1][cc * 8]);
                                }
                        }
                    };
                    load_batch(0, rb[0]);
                    tmem_ld_wait();
#pragma unroll
                    for (int g = 0; g < NG; ++g) {
                        const int b = g & 1;
                        if (g + 1 < NG) {
                            load_batch(g + 1, rb[b ^ 1]);
                        } else {
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) {
                                // the accumulator is released on the leader's barrier (the peer's is unused)
                                if (PAIR == 2 && !leader) mbar_arrive_cluster(mapa_shared(smem_u32(&tmem_empty_bar[acc]), 0));
                                else mbar_arrive(&tmem_empty_bar[acc]);
                            }
                            // probe the next block's two barriers here, before the last batch's FMAs, so
                            // that their round trips overlap them (1-1.5% on the weight-gradient workload;
                            // the same probe slowed the other layouts' epilogue by 1.5-4%)
                            int an = acc + 1, sn = slot + 1;
                            uint32_t apn = acc_phase, spn = sphase;
                            if (an == NACC) { an = 0; apn ^= 1u; }
                            if (sn == C::SCALE_SLOTS) { sn = 0; spn ^= 1u; }
                            pre = (kb + 1 < ti.nkb) &&
                                  ((static_cast<unsigned>(mbar_test_wait(&tmem_full_bar[an], apn)) &
                                    static_cast<unsigned>(mbar_test_wait(&scale_full_bar[sn], spn))) != 0u);
                        }
#pragma unroll
                        for (int cc = 0; cc < GC; ++cc) {
                            const int c = GC * g + cc;
                            if (c >= CHUNKS) break;
                            promote_kg_chunk<COLS>(accum, &rb[b][0][cc * 8], &rb[b][1][cc * 8], c, sb4[c], sa4);
                        }
                        if (g + 1 < NG) tmem_ld_wait();
                    }
                    // every lane has read its scales (the FMAs above used them)
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&scale_empty_bar[slot]);
                    if (++acc == NACC) { acc = 0; acc_phase ^= 1u; }
                    if (++slot == C::SCALE_SLOTS) { slot = 0; sphase ^= 1u; }
                }
            } else {
                // all BN columns of every other K block (this warpgroup's parity); the columns lie in one
                // 128-column sfb block (BN divides 128, n0 is a multiple of BN), so one scale sfa * sfb
                // serves the row
                float accf[BN];
#pragma unroll
                for (int j = 0; j < BN; ++j) accf[j] = 0.f;
                const uint32_t row_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
                for (int kb = 0; kb < ti.nkb; ++kb) {
                    if ((kb & 1) == h) {
                        bool got = (static_cast<unsigned>(mbar_try_wait(&tmem_full_bar[acc], acc_phase)) &
                                    static_cast<unsigned>(mbar_try_wait(&scale_full_bar[slot], sphase))) != 0u;
                        if (!got)
                            got = wait_bounded(&tmem_full_bar[acc], acc_phase, abort_flag, p.status, p.wait_limit_ns) &&
                                  wait_bounded(&scale_full_bar[slot], sphase, abort_flag, p.status, p.wait_limit_ns);
                        if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
                        tc_fence_after();
                        // TMEM loads in batches of up to 64 columns (the registers next to BN running
                        // sums), each waited on once; the accumulator is released after the last batch
                        constexpr int NCH = BN / 16;
                        constexpr int LB = NCH < 4 ? NCH : 4;
                        const float* sl = s_scales + slot * C::SLOT_FLOATS;
                        const float sab = sl[row_in_tile] * sl[BM];
#pragma unroll
                        for (int b = 0; b < NCH / LB; ++b) {
                            uint32_t rb[LB][16];
#pragma unroll
                            for (int c = 0; c < LB; ++c)
                                tmem_ld_x16(row_addr + static_cast<uint32_t>(acc * BN + (b * LB + c) * 16), rb[c]);
                            tmem_ld_wait();
                            if (b + 1 == NCH / LB) {
                                tc_fence_before();
                                __syncwarp();
                                if (lane == 0) {
                                    if (PAIR == 2 && !leader) mbar_arrive_cluster(mapa_shared(smem_u32(&tmem_empty_bar[acc]), 0));
                                    else mbar_arrive(&tmem_empty_bar[acc]);
                                }
                            }
#pragma unroll
                            for (int c = 0; c < LB; ++c) promote_chunk<BN>(accf, rb[c], b * LB + c, sab);
                        }
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&scale_empty_bar[slot]);
                    }
                    if (++acc == NACC) { acc = 0; acc_phase ^= 1u; }
                    if (++slot == C::SCALE_SLOTS) { slot = 0; sphase ^= 1u; }
                }
                if (!ok) break;
                // Exchange: warpgroup h stores columns [h*BN/2, (h+1)*BN/2) and hands the other half to
                // the other warpgroup, XCHG_PASS columns per pass. Region h holds what warpgroup h wrote:
                // rows of XCHG_PASS floats in 16-byte chunks swizzled by row (chunk ^ (row & 7)), so
                // neither side bank-conflicts.
                constexpr int PASS = C::XCHG_PASS;
                constexpr int HC = PASS / 4;   // 16-byte chunks per row and pass
                // split by h with compile-time indices only (so accf stays in registers)
                float send[COLS], keep[COLS];
                if (h == 0) {
#pragma unroll
                    for (int j = 0; j < COLS; ++j) { send[j] = accf[COLS + j]; keep[j] = accf[j]; }
                } else {
#pragma unroll
                    for (int j = 0; j < COLS; ++j) { send[j] = accf[j]; keep[j] = accf[COLS + j]; }
                }
                float4* mine = reinterpret_cast<float4*>(s_xchg) + (h * BM + row_in_tile) * HC;
                const float4* theirs = reinterpret_cast<const float4*>(s_xchg) + ((1 - h) * BM + row_in_tile) * HC;
#pragma unroll
                for (int ps = 0; ps < COLS / PASS; ++ps) {
                    const bool freed = wait_bounded(&xchg_free_bar, xphase ^ 1u, abort_flag, p.status, p.wait_limit_ns);
                    if (!__all_sync(0xffffffffu, freed)) { ok = false; break; }
#pragma unroll
                    for (int c = 0; c < HC; ++c) {
                        const int j = ps * PASS + c * 4;
                        mine[c ^ (row_in_tile & (HC - 1))] = make_float4(send[j], send[j + 1], send[j + 2], send[j + 3]);
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&xchg_full_bar);
                    const bool full = wait_bounded(&xchg_full_bar, xphase, abort_flag, p.status, p.wait_limit_ns);
                    if (!__all_sync(0xffffffffu, full)) { ok = false; break; }
#pragma unroll
                    for (int c = 0; c < HC; ++c) {
                        const float4 v = theirs[c ^ (row_in_tile & (HC - 1))];
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
            }
            if (!ok) break;

            if (split_k) {
                // ---- split-K: park this CTA's FP32 partial sums in shared memory for the reduction
                float* prow = reinterpret_cast<float*>(smem) + row_in_tile * C::PSTRIDE + h * COLS;
#pragma unroll
                for (int j = 0; j < COLS; j += 4)
                    *reinterpret_cast<float4*>(prow + j) = make_float4(accum[j], accum[j + 1], accum[j + 2], accum[j + 3]);
                continue;
            }
            // ---- store this CTA's rows of the tile
            if constexpr (MODE == kKGrouped) {
                // D[g] += tile (or D[g] = tile in the overwriting form). Per 16-column chunk and row i, the
                // lanes of a class pair (t, t ^ 1) swap one column pair, so that each lane holds 4
                // contiguous columns: the even lane of its group 2c, the odd lane of group 2c + 1. One
                // instruction then covers 8 rows x 64 contiguous bytes. The adds are vector reductions
                // at L2: one add per element, so the result does not depend on timing.
                float* d_g = static_cast<float*>(p.d) + static_cast<size_t>(ti.g) * p.rows * p.n;
                const int y0 = ti.m0 + q * 32 + (lane >> 2);
                const bool odd = (lane & 1) != 0;
                const int coff = odd ? 8 + 2 * ((lane & 3) - 1) : 2 * (lane & 3);
#pragma unroll
                for (int c = 0; c < CHUNKS; ++c) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int e0 = ((2 * c) * 4 + i) * 2, e1 = ((2 * c + 1) * 4 + i) * 2;
                        const float s0 = odd ? accum[e0] : accum[e1];
                        const float s1 = odd ? accum[e0 + 1] : accum[e1 + 1];
                        const float r0 = __shfl_xor_sync(0xffffffffu, s0, 1);
                        const float r1 = __shfl_xor_sync(0xffffffffu, s1, 1);
                        const float4 v = odd ? make_float4(r0, r1, accum[e1], accum[e1 + 1])
                                             : make_float4(accum[e0], accum[e0 + 1], r0, r1);
                        const int row = y0 + 8 * i;
                        const int col = cstart + c * 16 + coff;
                        if (row < p.rows && col < p.n) {
                            float* dst = d_g + static_cast<size_t>(row) * p.n + col;
                            if (p.overwrite) st_global_v4(dst, __float_as_uint(v.x), __float_as_uint(v.y), __float_as_uint(v.z), __float_as_uint(v.w));
                            else red_add_v4_f32(dst, v.x, v.y, v.z, v.w);
                        }
                    }
                }
            } else if constexpr (C::FULL_STAGE) {
                // BF16 out: the warp's 32 rows x COLS columns go to its staging boxes (32 x 32, 64 bytes a
                // row, 16-byte chunks swizzled by row pair as the 64-byte TMA swizzle expects: chunk ^
                // ((row >> 1) & 3); eight consecutive lanes touch every bank once), then one lane issues
                // the TMA stores and the warp moves on. The boxes are rewritten one tile later, after
                // their previous stores have read them. A masked tile with rows past masked_m is written
                // with plain stores of its valid rows instead (four lanes a row, 16 bytes each).
                uint8_t* wbuf = s_store + ew * C::STORE_WARP_BYTES;
                if (lane == 0) bulk_wait_read_n<0>();
                __syncwarp();
#pragma unroll
                for (int r = 0; r < COLS / 32; ++r) {
                    uint4* mine = reinterpret_cast<uint4*>(wbuf + r * 2048 + lane * 64);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int j = r * 32 + c * 8;
                        mine[c ^ ((lane >> 1) & 3)] = make_uint4(pack_bf16x2(accum[j], accum[j + 1]), pack_bf16x2(accum[j + 2], accum[j + 3]),
                                                                 pack_bf16x2(accum[j + 4], accum[j + 5]), pack_bf16x2(accum[j + 6], accum[j + 7]));
                    }
                }
                if (MODE != kMasked || ti.rows_valid >= BM) {
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        // boxes that lie wholly past the output's last row or column are not issued: a TMA
                        // store is given only boxes that start inside the tensor
                        const int y = ti.d_row + q * 32;
                        const int out_rows = (MODE == kMasked) ? p.groups * p.rows : p.rows;
                        if (y < out_rows) {
#pragma unroll
                            for (int r = 0; r < COLS / 32; ++r)
                                if (cstart + r * 32 < p.n) tma_store_2d(&tmap_d, wbuf + r * 2048, cstart + r * 32, y);
                        }
                        bulk_commit();
                    }
                } else {
                    __syncwarp();
                    __nv_bfloat16* dtile = reinterpret_cast<__nv_bfloat16*>(p.d) + static_cast<size_t>(ti.d_row + q * 32) * p.n;
                    const int rows_here = ti.rows_valid - q * 32;
                    const int cc = lane & 3;
#pragma unroll
                    for (int r = 0; r < COLS / 32; ++r) {
                        const int col = cstart + r * 32 + cc * 8;
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int row = i * 8 + (lane >> 2);
                            const uint4 v = *reinterpret_cast<const uint4*>(wbuf + r * 2048 + row * 64 + ((cc ^ ((row >> 1) & 3)) << 4));
                            if (row < rows_here && col < p.n)
                                st_global_v4(dtile + static_cast<size_t>(row) * p.n + col, v.x, v.y, v.z, v.w);
                        }
                    }
                }
            } else {
                // BF16 out through the warp's 2 KB staging buffer, 32 columns a round: each lane writes
                // its row's 64 bytes, then four lanes a row read them back and store 16 bytes each, so
                // one store instruction covers eight rows of 64 contiguous bytes (whole sectors). The
                // 16-byte chunks of a row are swizzled by row pair (chunk ^ ((row >> 1) & 3)): eight
                // consecutive lanes touch every bank once, writing and reading. A 16-column tail round
                // uses two lanes a row (chunk ^ ((row >> 2) & 1)). Rows past rows_valid (the matrix
                // edge, or masked_m) and columns past N are not written. Plain stores need no proxy
                // fence or bulk-store wait, and are not waited on: the warp moves on to its next tile.
                uint8_t* wbuf = s_store + ew * C::STORE_WARP_BYTES;
                __nv_bfloat16* dtile = reinterpret_cast<__nv_bfloat16*>(p.d) + static_cast<size_t>(ti.d_row + q * 32) * p.n;
                const int rows_here = ti.rows_valid - q * 32;   // valid rows of this warp's 32
#pragma unroll
                for (int r = 0; r < COLS / 32; ++r) {
                    __syncwarp();   // the previous round's reads are done
                    uint4* mine = reinterpret_cast<uint4*>(wbuf + lane * 64);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int j = r * 32 + c * 8;
                        mine[c ^ ((lane >> 1) & 3)] = make_uint4(pack_bf16x2(accum[j], accum[j + 1]), pack_bf16x2(accum[j + 2], accum[j + 3]),
                                                                 pack_bf16x2(accum[j + 4], accum[j + 5]), pack_bf16x2(accum[j + 6], accum[j + 7]));
                    }
                    __syncwarp();
                    const int cc = lane & 3;
                    const int col = cstart + r * 32 + cc * 8;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int row = i * 8 + (lane >> 2);
                        const uint4 v = *reinterpret_cast<const uint4*>(wbuf + row * 64 + ((cc ^ ((row >> 1) & 3)) << 4));
                        if (row < rows_here && col < p.n)
                            st_global_v4(dtile + static_cast<size_t>(row) * p.n + col, v.x, v.y, v.z, v.w);
                    }
                }
                if constexpr (COLS % 32 != 0) {
                    constexpr int j0 = (COLS / 32) * 32;
                    __syncwarp();
                    uint4* mine = reinterpret_cast<uint4*>(wbuf + lane * 32);
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const int j = j0 + c * 8;
                        mine[c ^ ((lane >> 2) & 1)] = make_uint4(pack_bf16x2(accum[j], accum[j + 1]), pack_bf16x2(accum[j + 2], accum[j + 3]),
                                                                 pack_bf16x2(accum[j + 4], accum[j + 5]), pack_bf16x2(accum[j + 6], accum[j + 7]));
                    }
                    __syncwarp();
                    const int cc = lane & 1;
                    const int col = cstart + j0 + cc * 8;
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const int row = i * 16 + (lane >> 1);
                        const uint4 v = *reinterpret_cast<const uint4*>(wbuf + row * 32 + ((cc ^ ((row >> 2) & 1)) << 4));
                        if (row < rows_here && col < p.n)
                            st_global_v4(dtile + static_cast<size_t>(row) * p.n + col, v.x, v.y, v.z, v.w);
                    }
                }
            }
        }
        // every TMA store of this warp has completed (and released its staging buffer) before exit
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }

    // ---------------------------------------------------------------------- split-K reduction
    if (split_k) {
        // every CTA's partials are visible cluster-wide after this barrier; CTA s of the cluster then
        // reduces rows [s*128/S, (s+1)*128/S) of the tile over all S partials (fixed order s = 0..S-1),
        // rounds to BF16 and stores; the second barrier keeps every CTA's shared memory alive until
        // all remote reads are done
        cluster_sync();
        // (a masked launch covers every possible tile; clusters past the device-side count have none)
        if (warp >= EPI_WARP0 && !*abort_flag && unit < num_tiles) {
            const TileInfo ti = decode_tile<MODE, BN, PAIR>(p, unit, s_prefix, rank, srank);
            const int rows_per = BM / p.split;
            const int groups = rows_per * (BN / 4);
            const uint32_t part_local = smem_u32(smem);
            for (int gi = static_cast<int>(threadIdx.x) - EPI_WARP0 * 32; gi < groups; gi += C::EPI_WARPS_C * 32) {
                const int row = srank * rows_per + gi / (BN / 4);
                const int c4 = (gi % (BN / 4)) * 4;
                const uint32_t off = static_cast<uint32_t>((row * C::PSTRIDE + c4) * 4);
                const float4 sum = cluster_sum_v4(part_local + off, p.split);
                if (row < ti.rows_valid && ti.n0 + c4 < p.n) {
                    __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(p.d) +
                                         static_cast<size_t>(ti.d_row + row) * p.n + ti.n0 + c4;
                    st_global_v2(dst, pack_bf16x2(sum.x, sum.y), pack_bf16x2(sum.z, sum.w));
                }
            }
        }
        cluster_sync();
    }

    // ---------------------------------------------------------------------- teardown
    tc_fence_before();
    if (PAIR == 2) cluster_sync(); else __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        if (PAIR == 2) tmem_dealloc_pair(tmem_base, TMEM_COLS);
        else tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

}  // namespace dg
