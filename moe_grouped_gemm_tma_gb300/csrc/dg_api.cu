// The C ABI declared in include/dg.h: argument checks, tile-shape choice, TMA descriptors, launch.
//
// Tile-shape choice follows the pages' "unaligned block sizes" and automatic block-size selection:
// BN (the tile's N extent) is picked per problem from multiples of 32 up to 256 so that the number
// of output tiles fills the SMs in as few, as full waves as possible.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "dg.h"
#include "dg_launch.cuh"
#include "dg_tuning.h"

namespace dg {

__device__ int g_status_word;

namespace {

// Tuning knobs (dg_tuning.h) and the armed test fault. The environment is read once, at load, and only
// when DG_TUNING=1.
std::atomic<int> g_tune[DG_TUNE_COUNT];
std::atomic<unsigned long long> g_armed_wait_fault{0};

struct TuneInit {
    TuneInit() {
        for (auto& k : g_tune) k.store(DG_TUNE_AUTO);
        const char* on = getenv("DG_TUNING");
        if (!on || strcmp(on, "1") != 0) return;
        const char* names[DG_TUNE_COUNT] = {"DG_BN", "DG_PAIR", "DG_SPLIT", "DG_SWAP", "DG_GROUP_M", "DG_PDL"};
        for (int i = 0; i < DG_TUNE_COUNT; ++i)
            if (const char* v = getenv(names[i])) g_tune[i].store(atoi(v));
    }
} g_tune_init;

}  // namespace

int tune(int knob) {
    return (knob >= 0 && knob < DG_TUNE_COUNT) ? g_tune[knob].load(std::memory_order_relaxed) : DG_TUNE_AUTO;
}

unsigned long long take_armed_wait_fault() {
    if (g_armed_wait_fault.load(std::memory_order_relaxed) == 0) return 0;
    return g_armed_wait_fault.exchange(0);
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

constexpr int kMaxDevices = 64;
struct DeviceInfo {
    bool ready = false;
    bool supported = false;
    int sms = 0;
    int l2_bytes = 0;
    int* status = nullptr;
};
DeviceInfo g_devices[kMaxDevices];
std::mutex g_devices_mutex;

dg_status device_info(DeviceInfo* out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DG_CUDA_ERROR;
    std::lock_guard<std::mutex> lock(g_devices_mutex);
    DeviceInfo& d = g_devices[dev];
    if (!d.ready) {
        int major = 0, minor = 0, sms = 0, l2 = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess)
            return DG_CUDA_ERROR;
        d.supported = (major == 10 && minor == 3);
        d.sms = sms;
        d.l2_bytes = l2;
        if (d.supported) {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return DG_CUDA_ERROR;
            d.status = static_cast<int*>(p);
        }
        d.ready = true;
    }
    *out = d;
    return d.supported ? DG_OK : DG_NO_DEVICE_SUPPORT;
}

dg_status encoder() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode ? DG_OK : DG_CUDA_ERROR;
}

// Row-major e4m3 matrix [rows, k] (k contiguous) read in boxes of box_rows x 128 with the 128-byte
// swizzle the MMA descriptors expect.
dg_status make_operand_map(CUtensorMap* m, const void* base, int64_t rows, int64_t k, int box_rows) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(k), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(k)};
    cuuint32_t box[2] = {128u, static_cast<cuuint32_t>(box_rows)};
    cuuint32_t es[2] = {1u, 1u};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? DG_OK : DG_CUDA_ERROR;
}

// MN-major e4m3 operand stored [k, cols] (cols contiguous: A as [K, M] or B as [K, N]) read in boxes of
// 128 columns x 128 k rows with the 128-byte swizzle, the layout of the MN-major MMA descriptors.
dg_status make_mn_operand_map(CUtensorMap* m, const void* base, int64_t k, int64_t cols) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(k)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols)};
    cuuint32_t box[2] = {128u, 128u};
    cuuint32_t es[2] = {1u, 1u};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? DG_OK : DG_CUDA_ERROR;
}

// Row-major BF16 output [rows, n] written in boxes of 32 rows x 16 columns (32 bytes) with the
// 32-byte swizzle the epilogue's staging buffers use.
dg_status make_output_map(CUtensorMap* m, void* base, int64_t rows, int64_t n) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(n), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(n) * 2};
    cuuint32_t box[2] = {16u, 32u};
    cuuint32_t es[2] = {1u, 1u};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
                          CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? DG_OK : DG_CUDA_ERROR;
}

// Row-major BF16 output [rows, n] written in boxes of 32 rows x 32 columns (64 bytes) with the
// 64-byte swizzle of the main kernel's whole-tile staging.
dg_status make_tile_output_map(CUtensorMap* m, void* base, int64_t rows, int64_t n) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(n), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(n) * 2};
    cuuint32_t box[2] = {32u, 32u};
    cuuint32_t es[2] = {1u, 1u};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                          CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? DG_OK : DG_CUDA_ERROR;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int cdiv(int64_t a, int64_t b) { return static_cast<int>((a + b - 1) / b); }

// Specialisations per layout: (BN, PAIR); each must be instantiated in the matching dg_inst_*.cu.
struct Spec {
    int bn, pair;
};
constexpr Spec kNormalSpecs1[] = {{64, 1}, {96, 1}, {128, 1}, {160, 1}, {192, 1}, {224, 1}, {256, 1}};
constexpr Spec kNormalSpecs2[] = {{128, 2}, {160, 2}, {192, 2}, {224, 2}, {256, 2}};
// block-scaled (UE8M0) normal GEMM
constexpr Spec kBlockScaledSpecs[] = {{128, 1}, {192, 1}, {224, 1}, {256, 1}};
constexpr Spec kBlockScaledSpecs2[] = {{128, 2}, {256, 2}};
// B stored MN-major is staged in whole 128-column boxes
constexpr Spec kNormalSpecsBMN[] = {{128, 1}, {256, 1}};
constexpr Spec kContiguousSpecs[] = {{128, 1}, {160, 1}, {192, 1}, {224, 1}, {256, 1}};
constexpr Spec kMaskedSpecs1[] = {{64, 1}, {128, 1}, {192, 1}, {224, 1}, {256, 1}};
constexpr Spec kMaskedSpecs2[] = {{128, 2}, {256, 2}};
constexpr Spec kKGroupedSpecs1[] = {{128, 1}, {192, 1}, {224, 1}, {256, 1}};
// automatic k-grouped choice: its per-column promotion makes tiles wider than 192 slower
constexpr Spec kKGroupedAuto1[] = {{128, 1}, {192, 1}, {256, 1}};
constexpr Spec kKGroupedSpecs2[] = {{128, 2}};

// Pick BN minimising waves * (BN + per-tile overhead), ties to the larger BN: the time of one wave of
// (128 * PAIR) x BN tiles grows with BN, and the number of waves is the tile count over the number of
// tiles that run at once (SMs / PAIR). The overhead term (96 columns' worth) is the measured cost of a
// narrower tile: each 128-K block still stages and feeds the whole 128-row A tile and pays the same
// epilogue round trip, so a BN=160 tile takes well over 160/256 of a BN=256 tile's time.
template <size_t NC>
Spec choose_spec(const Spec (&cands)[NC], int64_t row_units, int n, int sms) {
    Spec best = cands[NC - 1];
    int64_t best_cost = INT64_MAX;
    for (size_t i = 0; i < NC; ++i) {
        const int bn = cands[i].bn;
        const int64_t slots = sms / cands[i].pair;
        const int64_t tiles = row_units * cdiv(n, bn);
        const int64_t waves = (tiles + slots - 1) / slots;
        const int64_t cost = waves * (bn + 96);
        if (cost <= best_cost) { best_cost = cost; best = cands[i]; }
    }
    return best;
}

// Optional override of the tile width (the DG_TUNE_BN knob); ignored unless the layout has that width.
template <size_t NC>
Spec spec_override(const Spec (&cands)[NC], Spec chosen) {
    const int v = tune(DG_TUNE_BN);
    if (v < 0) return chosen;
    for (size_t i = 0; i < NC; ++i)
        if (cands[i].bn == v) return cands[i];
    return chosen;
}

// Tile raster for the normal and contiguous layouts: bands of group_m row blocks, row block fastest
// within a band. A band's A rows (group_m * 128 * PAIR * K bytes, at most a third of L2) stay resident
// while the band sweeps every column block; with the plain row-fastest order a wave spans up to 152 row
// blocks of one column block, and once A outgrows L2 every column block re-reads A from DRAM (measured
// on the contiguous layout with 31k rows, K = 7168: 803 us row-fastest, 691 us in bands of 16).
// The DG_TUNE_GROUP_M knob forces the band height.
int choose_group_m(int m_blocks, int tile_m, int64_t k, const DeviceInfo& dev) {
    int gm = std::min(m_blocks, 16);
    const int64_t band_bytes = static_cast<int64_t>(tile_m) * k;
    if (band_bytes > 0 && dev.l2_bytes > 0) {
        const int64_t fit = (static_cast<int64_t>(dev.l2_bytes) / 3) / band_bytes;
        gm = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(fit, gm)));
    }
    if (const int v = tune(DG_TUNE_GROUP_M); v > 0) gm = std::min(v, m_blocks);
    return std::max(gm, 1);
}

// Split-K for problems whose tiles cannot fill half the SMs (small M): a cluster of S CTAs shares a
// tile, each CTA streaming K/S of it, so more SMs pull operands at once. Picks (BN, S in {2, 4}) with
// the most CTAs that still fit in one wave, at least `min_kb` K blocks per CTA (4; the block-scaled
// kernel, whose per-CTA set-up is longer, asks for 8: 64 x 7168 x 2048 took 22.7 us as 4 CTAs of 4
// blocks per tile, against 14.4 us unsplit); ties go to the smaller S.
// The DG_TUNE_SPLIT knob forces S (2, 4 or 8; 1 disables); a forced tile width disables the split.
template <size_t NC>
int choose_split(const Spec (&cands)[NC], Spec* sp, int64_t row_blocks, int n, int kbs, int sms, int min_kb = 4) {
    if (const int s = tune(DG_TUNE_SPLIT); s >= 0) return (s == 2 || s == 4 || s == 8) && kbs >= s ? s : 1;
    if (tune(DG_TUNE_BN) >= 0) return 1;
    if (row_blocks * cdiv(n, sp->bn) * 2 > sms) return 1;
    int best_split = 1;
    int64_t best_ctas = row_blocks * cdiv(n, sp->bn);
    for (int s = 2; s <= 4; s *= 2) {   // clusters of 8 do not all fit at once with one CTA per SM
        if (kbs < min_kb * s) break;
        for (size_t i = 0; i < NC; ++i) {
            const int64_t ctas = row_blocks * cdiv(n, cands[i].bn) * s;
            if (ctas <= sms && ctas > best_ctas) {
                best_ctas = ctas;
                best_split = s;
                *sp = cands[i];
            }
        }
    }
    return best_split;
}

// CTA-pair (256-row) tiles halve the per-SM B traffic, but with the promotion epilogue as the limit
// they currently lose to single-CTA tiles on every measured shape (the cross-SM accumulator handoff
// lengthens the MMA/promotion loop), so they are opt-in: the DG_TUNE_PAIR knob at 2 (only for more
// than 128 rows).
bool use_pair(int64_t rows_per_group) { return tune(DG_TUNE_PAIR) == 2 && rows_per_group > 128; }

template <int MODE>
cudaError_t launch_spec(Spec sp, const Launch& L);

#define DG_CASE(M, B, P) \
    if (sp.bn == B && sp.pair == P) return launch<M, B, P>(L);

template <>
cudaError_t launch_spec<kNormal>(Spec sp, const Launch& L) {
    DG_CASE(kNormal, 64, 1) DG_CASE(kNormal, 96, 1) DG_CASE(kNormal, 128, 1) DG_CASE(kNormal, 160, 1)
    DG_CASE(kNormal, 192, 1) DG_CASE(kNormal, 224, 1) DG_CASE(kNormal, 256, 1)
    DG_CASE(kNormal, 128, 2) DG_CASE(kNormal, 160, 2) DG_CASE(kNormal, 192, 2) DG_CASE(kNormal, 224, 2)
    DG_CASE(kNormal, 256, 2)
    return cudaErrorInvalidValue;
}

template <>
cudaError_t launch_spec<kContiguous>(Spec sp, const Launch& L) {
    DG_CASE(kContiguous, 128, 1) DG_CASE(kContiguous, 160, 1) DG_CASE(kContiguous, 192, 1)
    DG_CASE(kContiguous, 224, 1) DG_CASE(kContiguous, 256, 1)
    return cudaErrorInvalidValue;
}

template <>
cudaError_t launch_spec<kMasked>(Spec sp, const Launch& L) {
    DG_CASE(kMasked, 64, 1) DG_CASE(kMasked, 128, 1) DG_CASE(kMasked, 192, 1) DG_CASE(kMasked, 224, 1) DG_CASE(kMasked, 256, 1)
    DG_CASE(kMasked, 128, 2) DG_CASE(kMasked, 256, 2)
    return cudaErrorInvalidValue;
}

template <>
cudaError_t launch_spec<kKGrouped>(Spec sp, const Launch& L) {
    DG_CASE(kKGrouped, 128, 1) DG_CASE(kKGrouped, 192, 1) DG_CASE(kKGrouped, 224, 1) DG_CASE(kKGrouped, 256, 1)
    DG_CASE(kKGrouped, 128, 2)
    return cudaErrorInvalidValue;
}
#undef DG_CASE

// The few-row (decode) kernel's plan: tile height BMT (tokens per tile, the MMA's N) from the expected
// rows per expert, and the split-K cluster size S. Time per wave of clusters ~ K blocks per CTA plus a
// fixed per-tile cost (the reduction through distributed shared memory for S > 1), so S is the one that
// minimises waves x (K/S + overhead) over the clusters that can be resident at once; ties go to the
// smaller S. The DG_TUNE_SPLIT knob forces S (1, 2, 4 or 8, at most the K blocks).
struct DecodePlan {
    int bmt = 64;
    int split = 1;
    int units = 0;   // clusters (or CTAs) launched: persistent, at most one wave
};

template <int MODE>
int decode_capacity(int bmt, int split, int sms) {
    switch (bmt) {
        case 32: return decode_cluster_capacity<MODE, 32>(split, sms);
        case 64: return decode_cluster_capacity<MODE, 64>(split, sms);
        default: return decode_cluster_capacity<MODE, 128>(split, sms);
    }
}

template <int MODE>
DecodePlan plan_decode(int64_t groups, int rows_hint, int rows_max, int n, int kbs, int sms) {
    DecodePlan pl;
    pl.bmt = rows_hint <= 32 ? 32 : (rows_hint <= 64 ? 64 : 128);
    const int64_t nt = cdiv(n, 128);
    const int64_t tiles_exp = std::max<int64_t>(1, groups * cdiv(std::max(rows_hint, 1), pl.bmt) * nt);
    const int64_t tiles_max = groups * cdiv(std::max(rows_max, 1), pl.bmt) * nt;
    const int forced = tune(DG_TUNE_SPLIT);
    const bool force = (forced == 1 || forced == 2 || forced == 4 || forced == 8) && kbs >= forced;
    int64_t best = INT64_MAX;
    for (int s = 1; s <= 8; s *= 2) {
        if (force ? s != forced : (s > 1 && kbs < 2 * s)) continue;
        const int cap = std::max(1, decode_capacity<MODE>(pl.bmt, s, sms));
        const int64_t waves = (tiles_exp + cap - 1) / cap;
        const int64_t cost = waves * (cdiv(kbs, s) + (s > 1 ? 3 : 1));
        if (cost < best) {
            best = cost;
            pl.split = s;
            pl.units = static_cast<int>(std::min<int64_t>(tiles_max, cap));
        }
    }
    return pl;
}

template <int MODE>
cudaError_t launch_decode_bmt(int bmt, const Launch& L) {
    switch (bmt) {
        case 32: return launch_decode<MODE, 32>(L);
        case 64: return launch_decode<MODE, 64>(L);
        case 128: return launch_decode<MODE, 128>(L);
    }
    return cudaErrorInvalidValue;
}

dg_status common_prologue(DeviceInfo* dev) {
    dg_status st = device_info(dev);
    if (st != DG_OK) return st;
    return encoder();
}

}  // namespace
}  // namespace dg

using namespace dg;

// Both weight-gradient entry points: experts g own consecutive K windows of widths ks_host[g]; the tile
// is added into D (D += ...) or, with overwrite, stored (D = ...).
static dg_status wgrad_impl(const uint8_t* A, const float* sfa, const uint8_t* B, const float* sfb,
                            const int32_t* ks_host, float* D, int G, int M, int N, bool overwrite,
                            cudaStream_t stream) {
    if (G < 0 || M < 0 || N < 0) return DG_INVALID_ARG;
    if (G == 0 || M == 0 || N == 0) return DG_OK;
    if (G > MAX_KGROUPS || !ks_host) return DG_INVALID_ARG;
    int64_t sumK = 0;
    for (int g = 0; g < G; ++g) {
        if (ks_host[g] < 0) return DG_INVALID_ARG;
        if (ks_host[g] % 128 != 0) return DG_UNSUPPORTED_SHAPE;
        sumK += ks_host[g];
    }
    if (N % 8 != 0) return DG_UNSUPPORTED_SHAPE;
    if (sumK == 0) return DG_OK;
    if (sumK > INT32_MAX || static_cast<int64_t>(G) * M > INT32_MAX) return DG_UNSUPPORTED_SHAPE;
    if (!A || !B || !sfa || !sfb || !D) return DG_INVALID_ARG;
    if (!aligned(A, 16) || !aligned(B, 16) || !aligned(D, 16) || !aligned(sfa, 4) || !aligned(sfb, 4))
        return DG_MISALIGNED;
    DeviceInfo dev;
    dg_status st = common_prologue(&dev);
    if (st != DG_OK) return st;

    const bool pair = use_pair(M);
    const Spec sp = pair ? spec_override(kKGroupedSpecs2, choose_spec(kKGroupedSpecs2, static_cast<int64_t>(G) * cdiv(M, 2 * BM), N, dev.sms))
                         : spec_override(kKGroupedSpecs1, choose_spec(kKGroupedAuto1, static_cast<int64_t>(G) * cdiv(M, BM), N, dev.sms));
    const int bn = sp.bn;
    Launch L;
    std::memset(&L, 0, sizeof(L));
    if (make_operand_map(&L.tmap_a, A, M, sumK, BM) != DG_OK) return DG_CUDA_ERROR;
    if (make_operand_map(&L.tmap_b, B, N, sumK, bn / sp.pair) != DG_OK) return DG_CUDA_ERROR;
    Params& p = L.params;
    p.sfa = sfa;
    p.sfb = sfb;
    p.d = D;
    p.status = dev.status;
    p.overwrite = overwrite ? 1 : 0;
    p.rows = M;
    p.n = N;
    p.kbs = static_cast<int>(sumK / 128);
    p.groups = G;
    p.sfb_rows = N;
    p.m_blocks = cdiv(M, BM * sp.pair);
    p.n_blocks = cdiv(N, bn);
    int off = 0;
    for (int g = 0; g < G; ++g) {
        p.kb_off[g] = off;
        off += ks_host[g] / 128;
    }
    p.kb_off[G] = off;
    const int64_t tiles = static_cast<int64_t>(G) * p.m_blocks * p.n_blocks;
    if (tiles > INT32_MAX) return DG_UNSUPPORTED_SHAPE;
    p.tiles = static_cast<int>(tiles);
    L.units = p.tiles;
    L.sms = dev.sms;
    L.stream = stream;
    return launch_spec<kKGrouped>(sp, L) == cudaSuccess ? DG_OK : DG_CUDA_ERROR;
}


// The normal GEMM for every operand layout: A stored [M, K] or (a_mn) [K, M], B stored [N, K] or
// (b_mn) [K, N]. MN-major operands need their contiguous extent to be a multiple of 16 (TMA row
// strides); MN-major B is tiled in whole 128-column boxes; CTA pairs serve the K-major layout only.
static dg_status gemm_impl(const uint8_t* A, const float* sfa, const uint8_t* B, const float* sfb, void* D,
                           int M, int N, int K, bool a_mn, bool b_mn, cudaStream_t stream) {
    if (M < 0 || N < 0 || K < 0) return DG_INVALID_ARG;
    if (M == 0 || N == 0) return DG_OK;
    if (!D) return DG_INVALID_ARG;
    if (K % 128 != 0 || N % 8 != 0) return DG_UNSUPPORTED_SHAPE;
    if ((a_mn && M % 16 != 0) || (b_mn && N % 16 != 0)) return DG_UNSUPPORTED_SHAPE;
    if (!aligned(D, 16)) return DG_MISALIGNED;
    DeviceInfo dev;
    dg_status st = common_prologue(&dev);
    if (st != DG_OK) return st;
    if (K == 0)
        return cudaMemsetAsync(D, 0, static_cast<size_t>(M) * N * 2, stream) == cudaSuccess ? DG_OK : DG_CUDA_ERROR;
    if (!A || !B || !sfa || !sfb) return DG_INVALID_ARG;
    if (!aligned(A, 16) || !aligned(B, 16) || !aligned(sfa, 4) || !aligned(sfb, 4)) return DG_MISALIGNED;

    // Short K (at most four K blocks) on pair tiles that fill every SM: 256-column CTA pairs, in which
    // each SM stages half of B, so less traffic shares an SM's TMA path with the tile's output stores
    // (in-stream, 4096 x 32768 x 512: 102.3 -> 98.2 us; from K = 1536 on, and for narrower pair tiles,
    // the single-CTA tiles measured as fast or faster).
    const bool short_k_pair = !a_mn && !b_mn && tune(DG_TUNE_PAIR) < 0 && tune(DG_TUNE_BN) < 0 && K <= 512 && M > 256 &&
                              static_cast<int64_t>(cdiv(M, 2 * BM)) * cdiv(N, 256) >= dev.sms;
    const bool pair = !a_mn && !b_mn && (use_pair(M) || short_k_pair);
    Spec sp;
    int split = 1;
    if (b_mn) {
        sp = spec_override(kNormalSpecsBMN, choose_spec(kNormalSpecsBMN, cdiv(M, BM), N, dev.sms));
        split = choose_split(kNormalSpecsBMN, &sp, cdiv(M, BM), N, K / 128, dev.sms);
    } else if (short_k_pair) {
        sp = Spec{256, 2};
    } else if (pair) {
        sp = spec_override(kNormalSpecs2, choose_spec(kNormalSpecs2, cdiv(M, 2 * BM), N, dev.sms));
    } else {
        sp = spec_override(kNormalSpecs1, choose_spec(kNormalSpecs1, cdiv(M, BM), N, dev.sms));
        split = choose_split(kNormalSpecs1, &sp, cdiv(M, BM), N, K / 128, dev.sms);
    }
    const int bn = sp.bn;
    Launch L;
    std::memset(&L, 0, sizeof(L));
    const int kbs = K / 128;
    // Few rows, long K, 32..64 column tiles of 128: the decode kernel (swapped operands, K-block groups,
    // split-K clusters sized to fill the SMs). Measured in-stream against the standard kernel with
    // split-K, fraction of the HBM roofline: 64 x 7168 x 16384 0.55 against 0.45, 64 x 4096 x 7168 0.35
    // against 0.31. Outside that range the standard kernel was as fast or faster (64 x 2112 x 7168,
    // 17 column tiles: 0.20 against 0.22; 128-row tiles: 128 x 7168 x 16384 0.44 against 0.46; short K
    // or 192..256 column tiles: 0.22-0.37 against 0.26-0.52). The DG_TUNE_SWAP knob forces the choice
    // (1 = decode kernel, 0 = standard kernel).
    DecodePlan pl;
    bool decode = false;
    if (!a_mn && !b_mn && !pair && M <= 128 && tune(DG_TUNE_BN) < 0) {
        const int col_tiles = cdiv(N, 128);
        decode = M <= 64 && K >= 7168 && col_tiles >= 32 && col_tiles <= 64;
        if (const int v = tune(DG_TUNE_SWAP); v >= 0) decode = (v == 1);
        if (decode) pl = plan_decode<kNormal>(1, M, M, N, kbs, dev.sms);
    }
    if (decode) {
        if (make_operand_map(&L.tmap_a, A, M, K, pl.bmt) != DG_OK) return DG_CUDA_ERROR;
        if (make_operand_map(&L.tmap_b, B, N, K, 128) != DG_OK) return DG_CUDA_ERROR;
        Params& p = L.params;
        p.sfa = sfa;
        p.sfb = sfb;
        p.d = D;
        p.status = dev.status;
        p.rows = M;
        p.n = N;
        p.kbs = kbs;
        p.groups = 1;
        p.sfb_rows = cdiv(N, 128);
        p.m_blocks = cdiv(M, pl.bmt);
        p.n_blocks = cdiv(N, 128);
        p.split = pl.split;
        p.tiles = p.m_blocks * p.n_blocks;
        L.units = pl.units;
        L.sms = dev.sms;
        L.stream = stream;
        return launch_decode_bmt<kNormal>(pl.bmt, L) == cudaSuccess ? DG_OK : DG_CUDA_ERROR;
    }
    if ((a_mn ? make_mn_operand_map(&L.tmap_a, A, K, M) : make_operand_map(&L.tmap_a, A, M, K, BM)) != DG_OK)
        return DG_CUDA_ERROR;
    if ((b_mn ? make_mn_operand_map(&L.tmap_b, B, K, N) : make_operand_map(&L.tmap_b, B, N, K, bn / sp.pair)) != DG_OK)
        return DG_CUDA_ERROR;
    if (make_tile_output_map(&L.tmap_d, D, M, N) != DG_OK) return DG_CUDA_ERROR;
    Params& p = L.params;
    p.sfa = sfa;
    p.sfb = sfb;
    p.d = D;
    p.status = dev.status;
    p.rows = M;
    p.n = N;
    p.kbs = K / 128;
    p.groups = 1;
    p.sfb_rows = cdiv(N, 128);
    p.m_blocks = cdiv(M, BM * sp.pair);
    p.n_blocks = cdiv(N, bn);
    p.group_m = choose_group_m(p.m_blocks, BM * sp.pair, K, dev);
    p.split = split;
    p.a_mn = a_mn ? 1 : 0;
    p.b_mn = b_mn ? 1 : 0;
    // Long K: a band's A row blocks (2 MB each at K = 16384) are evicted before the band's next round of
    // tiles reads them again, unless A is marked evict-last and B (read only by tiles in flight
    // together) evict-first. Measured on 4096 x 7168 x 16384: DRAM traffic per launch 483 -> 355 MB
    // (algorithmic 243 MB), 330.6 -> 325.7 us; on K <= 7168 shapes it measured 0.5-1.5% slower.
    p.l2_hint = (!a_mn && !b_mn && K >= 8192) ? 1 : 0;
    const int64_t tiles = static_cast<int64_t>(p.m_blocks) * p.n_blocks;
    if (tiles > INT32_MAX) return DG_UNSUPPORTED_SHAPE;
    p.tiles = static_cast<int>(tiles);
    L.units = p.tiles;
    L.sms = dev.sms;
    L.stream = stream;
    return launch_spec<kNormal>(sp, L) == cudaSuccess ? DG_OK : DG_CUDA_ERROR;
}

extern "C" {

const char* dg_status_string(dg_status s) {
    switch (s) {
        case DG_OK: return "DG_OK";
        case DG_INVALID_ARG: return "DG_INVALID_ARG";
        case DG_UNSUPPORTED_SHAPE: return "DG_UNSUPPORTED_SHAPE";
        case DG_MISALIGNED: return "DG_MISALIGNED";
        case DG_CUDA_ERROR: return "DG_CUDA_ERROR";
        case DG_NO_DEVICE_SUPPORT: return "DG_NO_DEVICE_SUPPORT";
        case DG_DEVICE_TIMEOUT: return "DG_DEVICE_TIMEOUT";
        case DG_SCALE_NOT_UE8M0: return "DG_SCALE_NOT_UE8M0";
    }
    return "DG_UNKNOWN_STATUS";
}

dg_status dg_tuning_set(int knob, int value) {
    if (knob < 0 || knob >= DG_TUNE_COUNT) return DG_INVALID_ARG;
    g_tune[knob].store(value < 0 ? DG_TUNE_AUTO : value);
    return DG_OK;
}

int dg_tuning_get(int knob) { return tune(knob); }

void dg_tuning_reset(void) {
    for (auto& k : g_tune) k.store(DG_TUNE_AUTO);
}

dg_status dg_testing_arm_wait_timeout(uint64_t wait_limit_ns) {
    if (wait_limit_ns == 0) return DG_INVALID_ARG;
    g_armed_wait_fault.store(static_cast<unsigned long long>(wait_limit_ns));
    return DG_OK;
}

dg_status dg_device_status(cudaStream_t stream) {
    DeviceInfo dev;
    dg_status st = device_info(&dev);
    if (st != DG_OK) return st;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return DG_CUDA_ERROR;
    int v = 0;
    if (cudaMemcpy(&v, dev.status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return DG_CUDA_ERROR;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpy(dev.status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return DG_CUDA_ERROR;
        return v == DG_SCALE_NOT_UE8M0 ? DG_SCALE_NOT_UE8M0 : DG_DEVICE_TIMEOUT;
    }
    return DG_OK;
}

dg_status dg_gemm_fp8_nt(const uint8_t* A, const float* sfa, const uint8_t* B, const float* sfb, void* D,
                         int M, int N, int K, cudaStream_t stream) {
    return gemm_impl(A, sfa, B, sfb, D, M, N, K, false, false, stream);
}

dg_status dg_gemm_fp8(const uint8_t* A, const float* sfa, const uint8_t* B, const float* sfb, void* D, int M,
                      int N, int K, int a_mn_major, int b_mn_major, cudaStream_t stream) {
    return gemm_impl(A, sfa, B, sfb, D, M, N, K, a_mn_major != 0, b_mn_major != 0, stream);
}

// The block-scaled GEMM behind both UE8M0 entry points: FP32 power-of-two scales (converted and checked
// on the device) or packed UE8M0 exponents (four K blocks per int32, used as they are).
static dg_status ue8m0_impl(const uint8_t* A, const void* sfa, const uint8_t* B, const void* sfb, void* D,
                            int M, int N, int K, bool packed, cudaStream_t stream) {
    if (M < 0 || N < 0 || K < 0) return DG_INVALID_ARG;
    if (M == 0 || N == 0) return DG_OK;
    if (!D) return DG_INVALID_ARG;
    if (K % 128 != 0 || N % 8 != 0) return DG_UNSUPPORTED_SHAPE;
    if (!aligned(D, 16)) return DG_MISALIGNED;
    DeviceInfo dev;
    dg_status st = common_prologue(&dev);
    if (st != DG_OK) return st;
    if (K == 0)
        return cudaMemsetAsync(D, 0, static_cast<size_t>(M) * N * 2, stream) == cudaSuccess ? DG_OK : DG_CUDA_ERROR;
    if (!A || !B || !sfa || !sfb) return DG_INVALID_ARG;
    if (!aligned(A, 16) || !aligned(B, 16) || !aligned(sfa, 4) || !aligned(sfb, 4)) return DG_MISALIGNED;

    // CTA pairs halve each SM's B bytes per K block, which the block-scaled kernel (no per-block
    // promotion loop) turns into speed: 4096 x 7168 x 16384 in 279 us against 308 us single-CTA, and
    // faster on every M = 4096 dense shape. They are taken when the pair tiles fill at least one wave
    // of CTAs; fewer tiles go to single-CTA tiles with split-K. The DG_TUNE_PAIR knob forces the choice.
    bool pair = M > BM && static_cast<int64_t>(cdiv(M, 2 * BM)) * cdiv(N, 256) * 2 >= dev.sms;
    if (const int v = tune(DG_TUNE_PAIR); v >= 0) pair = (v == 2) && M > BM;
    Spec sp = pair ? spec_override(kBlockScaledSpecs2, choose_spec(kBlockScaledSpecs2, cdiv(M, 2 * BM), N, dev.sms))
                   : spec_override(kBlockScaledSpecs, choose_spec(kBlockScaledSpecs, cdiv(M, BM), N, dev.sms));
    const int split = pair ? 1 : choose_split(kBlockScaledSpecs, &sp, cdiv(M, BM), N, K / 128, dev.sms, 8);
    const int bn = sp.bn;
    Launch L;
    std::memset(&L, 0, sizeof(L));
    if (make_operand_map(&L.tmap_a, A, M, K, BM) != DG_OK) return DG_CUDA_ERROR;
    if (make_operand_map(&L.tmap_b, B, N, K, bn / sp.pair) != DG_OK) return DG_CUDA_ERROR;
    if (make_output_map(&L.tmap_d, D, M, N) != DG_OK) return DG_CUDA_ERROR;
    Params& p = L.params;
    p.sfa = static_cast<const float*>(sfa);
    p.sfb = static_cast<const float*>(sfb);
    p.sf_packed = packed ? 1 : 0;
    p.sf_words = cdiv(K / 128, 4);
    p.d = D;
    p.status = dev.status;
    p.rows = M;
    p.n = N;
    p.kbs = K / 128;
    p.groups = 1;
    p.sfb_rows = cdiv(N, 128);
    p.m_blocks = cdiv(M, BM * sp.pair);
    p.n_blocks = cdiv(N, bn);
    p.group_m = choose_group_m(p.m_blocks, BM * sp.pair, K, dev);
    p.split = split;
    const int64_t tiles = static_cast<int64_t>(p.m_blocks) * p.n_blocks;
    if (tiles > INT32_MAX) return DG_UNSUPPORTED_SHAPE;
    p.tiles = static_cast<int>(tiles);
    L.units = p.tiles;
    L.sms = dev.sms;
    L.stream = stream;
    cudaError_t e = cudaErrorInvalidValue;
    if (pair) {
        switch (bn) {
            case 128: e = launch_bs<128, 2>(L); break;
            case 256: e = launch_bs<256, 2>(L); break;
        }
    } else {
        switch (bn) {
            case 128: e = launch_bs<128, 1>(L); break;
            case 192: e = launch_bs<192, 1>(L); break;
            case 224: e = launch_bs<224, 1>(L); break;
            case 256: e = launch_bs<256, 1>(L); break;
        }
    }
    return e == cudaSuccess ? DG_OK : DG_CUDA_ERROR;
}

dg_status dg_gemm_fp8_nt_ue8m0(const uint8_t* A, const float* sfa, const uint8_t* B, const float* sfb, void* D,
                               int M, int N, int K, cudaStream_t stream) {
    return ue8m0_impl(A, sfa, B, sfb, D, M, N, K, false, stream);
}

dg_status dg_gemm_fp8_nt_ue8m0_packed(const uint8_t* A, const int32_t* sfa, const uint8_t* B, const int32_t* sfb,
                                      void* D, int M, int N, int K, cudaStream_t stream) {
    return ue8m0_impl(A, sfa, B, sfb, D, M, N, K, true, stream);
}

dg_status dg_m_grouped_contiguous(const uint8_t* A, const float* sfa, const uint8_t* B, const float* sfb,
                                  const int32_t* m_indices, void* D, int Mt, int N, int K, int G,
                                  cudaStream_t stream) {
    if (Mt < 0 || N < 0 || K < 0 || G < 0) return DG_INVALID_ARG;
    if (Mt == 0 || N == 0) return DG_OK;
    if (G == 0) return DG_INVALID_ARG;
    if (K % 128 != 0 || K == 0 || N % 8 != 0 || Mt % 128 != 0) return DG_UNSUPPORTED_SHAPE;
    if (!A || !B || !sfa || !sfb || !m_indices || !D) return DG_INVALID_ARG;
    if (!aligned(A, 16) || !aligned(B, 16) || !aligned(D, 16) || !aligned(sfa, 4) || !aligned(sfb, 4) ||
        !aligned(m_indices, 4))
        return DG_MISALIGNED;
    if (static_cast<int64_t>(G) * N > INT32_MAX) return DG_UNSUPPORTED_SHAPE;
    DeviceInfo dev;
    dg_status st = common_prologue(&dev);
    if (st != DG_OK) return st;

    const Spec sp = spec_override(kContiguousSpecs, choose_spec(kContiguousSpecs, cdiv(Mt, BM), N, dev.sms));
    const int bn = sp.bn;
    Launch L;
    std::memset(&L, 0, sizeof(L));
    if (make_operand_map(&L.tmap_a, A, Mt, K, BM) != DG_OK) return DG_CUDA_ERROR;
    if (make_tile_output_map(&L.tmap_d, D, Mt, N) != DG_OK) return DG_CUDA_ERROR;
    if (make_operand_map(&L.tmap_b, B, static_cast<int64_t>(G) * N, K, bn) != DG_OK) return DG_CUDA_ERROR;
    Params& p = L.params;
    p.sfa = sfa;
    p.sfb = sfb;
    p.d = D;
    p.m_indices = m_indices;
    p.status = dev.status;
    p.rows = Mt;
    p.n = N;
    p.kbs = K / 128;
    p.groups = G;
    p.sfb_rows = cdiv(N, 128);
    p.m_blocks = Mt / BM;
    p.group_m = choose_group_m(p.m_blocks, BM, K, dev);
    p.n_blocks = cdiv(N, bn);
    const int64_t tiles = static_cast<int64_t>(p.m_blocks) * p.n_blocks;
    if (tiles > INT32_MAX) return DG_UNSUPPORTED_SHAPE;
    p.tiles = static_cast<int>(tiles);
    L.units = p.tiles;
    L.sms = dev.sms;
    L.stream = stream;
    return launch_spec<kContiguous>(sp, L) == cudaSuccess ? DG_OK : DG_CUDA_ERROR;
}

dg_status dg_m_grouped_masked(const uint8_t* A, const float* sfa, const uint8_t* B, const float* sfb,
                              const int32_t* masked_m, void* D, int G, int max_m, int N, int K, int expected_m,
                              cudaStream_t stream) {
    if (G < 0 || max_m < 0 || N < 0 || K < 0) return DG_INVALID_ARG;
    if (G == 0 || max_m == 0 || N == 0) return DG_OK;
    if (G > MAX_MASKED_G) return DG_INVALID_ARG;
    if (K % 128 != 0 || K == 0 || N % 8 != 0) return DG_UNSUPPORTED_SHAPE;
    if (!A || !B || !sfa || !sfb || !masked_m || !D) return DG_INVALID_ARG;
    if (!aligned(A, 16) || !aligned(B, 16) || !aligned(D, 16) || !aligned(sfa, 4) || !aligned(sfb, 4) ||
        !aligned(masked_m, 4))
        return DG_MISALIGNED;
    if (static_cast<int64_t>(G) * max_m > INT32_MAX || static_cast<int64_t>(G) * N > INT32_MAX)
        return DG_UNSUPPORTED_SHAPE;
    DeviceInfo dev;
    dg_status st = common_prologue(&dev);
    if (st != DG_OK) return st;

    const int hint = (expected_m > 0 && expected_m < max_m) ? expected_m : max_m;
    // Decode with few tiles (a single expert of up to 128 expected rows, long K): the decode kernel.
    // Measured in-stream, fraction of the HBM roofline, one expert, N = 4096, K = 7168: 0.32 against 0.26
    // (expected_m = 64) and 0.28 against 0.23 (128). With more experts, or short K, the standard kernel
    // was as fast or faster (G = 2..16: 0.39-0.73 against 0.44-0.85). DG_TUNE_SWAP forces the choice.
    bool decode = hint <= 128 && K >= 7168 &&
                  static_cast<int64_t>(G) * cdiv(hint, hint <= 32 ? 32 : (hint <= 64 ? 64 : 128)) * cdiv(N, 128) <= 32;
    if (const int v = tune(DG_TUNE_SWAP); v >= 0) decode = (v == 1) && hint <= 128;
    if (decode && tune(DG_TUNE_PAIR) != 2 && tune(DG_TUNE_BN) < 0) {
        // The decode kernel (swapped operands: B's rows fill the MMA's 128 lanes, the tokens are its N)
        // counts each expert's row blocks on the device from masked_m; the plan (tile height, split-K)
        // follows expected_m, and any masked_m up to max_m stays correct.
        const DecodePlan pl = plan_decode<kMasked>(G, hint, max_m, N, K / 128, dev.sms);
        Launch L;
        std::memset(&L, 0, sizeof(L));
        if (make_operand_map(&L.tmap_a, A, static_cast<int64_t>(G) * max_m, K, pl.bmt) != DG_OK) return DG_CUDA_ERROR;
        if (make_operand_map(&L.tmap_b, B, static_cast<int64_t>(G) * N, K, 128) != DG_OK) return DG_CUDA_ERROR;
        Params& p = L.params;
        p.sfa = sfa;
        p.sfb = sfb;
        p.d = D;
        p.masked_m = masked_m;
        p.status = dev.status;
        p.rows = max_m;
        p.n = N;
        p.kbs = K / 128;
        p.groups = G;
        p.sfb_rows = cdiv(N, 128);
        p.m_blocks = cdiv(max_m, pl.bmt);
        p.n_blocks = cdiv(N, 128);
        if (static_cast<int64_t>(G) * p.m_blocks * p.n_blocks > INT32_MAX) return DG_UNSUPPORTED_SHAPE;
        p.tiles = 0;  // counted on the device from masked_m
        p.split = pl.split;
        L.units = pl.units;
        L.sms = dev.sms;
        L.stream = stream;
        return launch_decode_bmt<kMasked>(pl.bmt, L) == cudaSuccess ? DG_OK : DG_CUDA_ERROR;
    }
    const bool pair = use_pair(hint);
    Spec sp = pair ? spec_override(kMaskedSpecs2, choose_spec(kMaskedSpecs2, static_cast<int64_t>(G) * cdiv(hint, 2 * BM), N, dev.sms))
                   : spec_override(kMaskedSpecs1, choose_spec(kMaskedSpecs1, static_cast<int64_t>(G) * cdiv(hint, BM), N, dev.sms));
    int split = 1;
    if (!pair) {
        // Split-K when the expected tiles (from expected_m) fill under half the SMs. The launch holds a
        // cluster for every possible tile (the count is known only on the device), and clusters past the
        // count still pay their set-up, so the split is dropped when that grid exceeds two waves
        // (measured with one expert of 59 rows, N = 4096, K = 7168: 25.2 -> 23.2 us at max_m = 256; at
        // max_m = 512, four waves of mostly empty clusters, 24.6 -> 26.9 us).
        Spec s2 = sp;
        split = choose_split(kMaskedSpecs1, &s2, static_cast<int64_t>(G) * cdiv(hint, BM), N, K / 128, dev.sms);
        if (split > 1 && static_cast<int64_t>(G) * cdiv(max_m, BM) * cdiv(N, s2.bn) * split > 2 * static_cast<int64_t>(dev.sms))
            split = 1;
        if (split > 1) sp = s2;
    }
    const int bn = sp.bn;
    Launch L;
    std::memset(&L, 0, sizeof(L));
    if (make_operand_map(&L.tmap_a, A, static_cast<int64_t>(G) * max_m, K, BM) != DG_OK) return DG_CUDA_ERROR;
    if (make_tile_output_map(&L.tmap_d, D, static_cast<int64_t>(G) * max_m, N) != DG_OK) return DG_CUDA_ERROR;
    if (make_operand_map(&L.tmap_b, B, static_cast<int64_t>(G) * N, K, bn / sp.pair) != DG_OK) return DG_CUDA_ERROR;
    Params& p = L.params;
    p.sfa = sfa;
    p.sfb = sfb;
    p.d = D;
    p.masked_m = masked_m;
    p.status = dev.status;
    p.rows = max_m;
    p.n = N;
    p.kbs = K / 128;
    p.groups = G;
    p.sfb_rows = cdiv(N, 128);
    p.m_blocks = cdiv(max_m, BM * sp.pair);
    p.n_blocks = cdiv(N, bn);
    const int64_t max_tiles = static_cast<int64_t>(G) * p.m_blocks * p.n_blocks;
    if (max_tiles > INT32_MAX) return DG_UNSUPPORTED_SHAPE;
    p.tiles = 0;  // counted on the device from masked_m
    p.split = split;
    L.units = static_cast<int>(max_tiles);
    L.sms = dev.sms;
    L.stream = stream;
    return launch_spec<kMasked>(sp, L) == cudaSuccess ? DG_OK : DG_CUDA_ERROR;
}

dg_status dg_k_grouped_wgrad(const uint8_t* A, const float* sfa, const uint8_t* B, const float* sfb,
                             const int32_t* ks_host, float* D, int G, int M, int N, cudaStream_t stream) {
    return wgrad_impl(A, sfa, B, sfb, ks_host, D, G, M, N, false, stream);
}

dg_status dg_wgrad_fp8_nt(const uint8_t* A, const float* sfa, const uint8_t* B, const float* sfb, float* D,
                          int M, int N, int K, int accumulate, cudaStream_t stream) {
    if (M < 0 || N < 0 || K < 0) return DG_INVALID_ARG;
    if (M == 0 || N == 0) return DG_OK;
    if (K % 128 != 0 || N % 8 != 0) return DG_UNSUPPORTED_SHAPE;
    if (K == 0) {
        if (accumulate) return DG_OK;
        if (!D) return DG_INVALID_ARG;
        if (!aligned(D, 16)) return DG_MISALIGNED;
        DeviceInfo dev;
        dg_status st = common_prologue(&dev);
        if (st != DG_OK) return st;
        return cudaMemsetAsync(D, 0, static_cast<size_t>(M) * N * sizeof(float), stream) == cudaSuccess
                   ? DG_OK : DG_CUDA_ERROR;
    }
    const int32_t ks[1] = {K};
    return wgrad_impl(A, sfa, B, sfb, ks, D, 1, M, N, accumulate == 0, stream);
}

}  // extern "C"
