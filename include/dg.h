/*
 * dg — block-scaled FP8 GEMM and MoE grouped GEMM for GB300 (sm_103a): the C ABI.
 *
 * The operation (DeepGEMM pages: "DeepSeek DeepGEMM" feature list and usage example;
 * "DeepSeek Open Source Week - Dia 3", technical features):
 *
 *   D[m,n] = sum_kb  sfa[m,kb] * sfb[n/128,kb] * sum_{k in block kb} A[m,k] * B[n,k]
 *
 * A and B hold float8 e4m3 codes ("fn" variant), K-contiguous ("NT": A is [M,K], B is [N,K]).
 * Fine-grained scaling gives one FP32 scale per 1x128 row block of A and per 128x128 block of B;
 * every 128-wide K block is contracted on the tensor cores and then promoted, scaled by its two
 * scales, into an FP32 running sum ("two-level accumulation"). Results are rounded to BF16
 * (round to nearest even) for the normal and m-grouped GEMMs; the k-grouped weight gradient
 * accumulates into FP32.
 *
 * Conventions shared by every entry point:
 *   - All tensors are caller-owned DEVICE memory, row-major and densely packed, unless stated
 *     otherwise. The library keeps no pointer after a call returns and allocates no memory.
 *   - Calls are asynchronous on `stream` (0 = the legacy default stream). Argument errors are
 *     returned synchronously before anything is launched; launch errors return DG_CUDA_ERROR.
 *   - K (and every k-grouped ks[g]) must be a multiple of 128, the scaling block ("K dimension
 *     aligned to 128" in the pages' requirements). N must be a multiple of 8 (16-byte output rows).
 *   - A and B must be 16-byte aligned (TMA), D 16-byte aligned, scales 4-byte aligned.
 *   - Zero-sized problems (M = 0, Mt = 0, G = 0) are valid and launch nothing.
 *   - The library runs on compute capability 10.3 only (sm_103a code); other devices get
 *     DG_NO_DEVICE_SUPPORT.
 *   - Device-side waits are bounded; a kernel that gives up records DG_DEVICE_TIMEOUT, which
 *     dg_device_status() reports. Tuning overrides and a test hook for this path: dg_tuning.h.
 *   - Distinct streams may call concurrently (no mutable host state after first use per device).
 */
#ifndef DG_H
#define DG_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int dg_status;
enum {
    DG_OK = 0,
    DG_INVALID_ARG = 1,        /* null pointer with a non-empty shape, negative size, G out of range */
    DG_UNSUPPORTED_SHAPE = 2,  /* K % 128, N % 8, ks[g] % 128, or a size beyond the supported range */
    DG_MISALIGNED = 3,         /* a pointer not aligned as stated above */
    DG_CUDA_ERROR = 4,         /* a CUDA runtime/driver call or launch failed */
    DG_NO_DEVICE_SUPPORT = 5,  /* current device is not compute capability 10.3 */
    DG_DEVICE_TIMEOUT = 6,     /* a kernel's bounded wait expired (reported by dg_device_status) */
    DG_SCALE_NOT_UE8M0 = 7     /* a UE8M0-path scale was not a power of two (reported by dg_device_status) */
};

/*
 * Normal GEMM (pages: gemm_fp8_fp8_bf16_nt).
 *   A   [M, K]            e4m3 codes          sfa [M, K/128]            fp32
 *   B   [N, K]            e4m3 codes          sfb [ceil(N/128), K/128]  fp32
 *   D   [M, N]            bf16, overwritten
 * The usage example on the pages (M=4096, K=7168, N=2112) has sfa [4096, 56] and sfb [17, 56]:
 * sfb has ceil(N/128) rows, row j scaling B rows [128j, 128j+128).
 */
dg_status dg_gemm_fp8_nt(const uint8_t* A, const float* sfa, const uint8_t* B, const float* sfb,
                         void* D, int M, int N, int K, cudaStream_t stream);

/*
 * The normal GEMM for the other operand layouts (the pages list NT, TN, NN and TT for SM100): the same
 * product D = A . B^T with the same scales, but A may be stored transposed, [K, M] with M contiguous
 * (a_mn_major != 0), and B transposed, [K, N] with N contiguous (b_mn_major != 0). sfa stays
 * [M, K/128] and sfb [ceil(N/128), K/128]. An MN-major operand needs its contiguous extent (M or N)
 * to be a multiple of 16 (DG_UNSUPPORTED_SHAPE otherwise). dg_gemm_fp8(..., 0, 0, ...) is
 * dg_gemm_fp8_nt.
 */
dg_status dg_gemm_fp8(const uint8_t* A, const float* sfa, const uint8_t* B, const float* sfb, void* D,
                      int M, int N, int K, int a_mn_major, int b_mn_major, cudaStream_t stream);

/*
 * The normal GEMM for power-of-two scales, on the block-scaled tensor-core path (pages: the SM100
 * UE8M0 scale format): same arguments and result as dg_gemm_fp8_nt, but every sfa and sfb entry must
 * be a positive power of two in [2^-126, 2^127]. The tensor core applies the scales as 8-bit exponents
 * while it accumulates, so no per-128-K promotion runs. A scale that is not a power of two is
 * reported by dg_device_status as DG_SCALE_NOT_UE8M0 (its result is then unspecified).
 */
dg_status dg_gemm_fp8_nt_ue8m0(const uint8_t* A, const float* sfa, const uint8_t* B, const float* sfb, void* D,
                               int M, int N, int K, cudaStream_t stream);

/*
 * The same block-scaled GEMM with the scales already in the packed UE8M0 format (pages: the SM100
 * scale layout, four UE8M0 values in one int32):
 *   sfa  [M, ceil(K/512)] int32          sfb  [ceil(N/128), ceil(K/512)] int32
 * Byte j (least significant first) of word w of a row is the biased exponent e of K block 4w + j; the
 * scale it stands for is 2^(e - 127). Bytes past the last K block are ignored. The exponents are used
 * as they are (no check; e = 255 is not a number). Result as dg_gemm_fp8_nt with those scales.
 * Device pointers, 4-byte aligned; errors as dg_gemm_fp8_nt.
 */
dg_status dg_gemm_fp8_nt_ue8m0_packed(const uint8_t* A, const int32_t* sfa, const uint8_t* B, const int32_t* sfb,
                                      void* D, int M, int N, int K, cudaStream_t stream);

/*
 * m-grouped GEMM, contiguous layout (pages: m_grouped_gemm_fp8_fp8_bf16_nt_contiguous; for training
 * forward and inference prefill). The experts' token rows are stacked along M; each expert's segment
 * starts on a multiple of 128 rows (segments padded to 128).
 *   A         [Mt, K]                 sfa [Mt, K/128]
 *   B         [G, N, K]               sfb [G, ceil(N/128), K/128]
 *   m_indices [Mt] int32 (device)     expert of each row, -1 on padding rows
 *   D         [Mt, N] bf16
 * Row r gets D[r] = A[r] . B[m_indices[r]]^T. The expert of a 128-row block is read from its first
 * row; a block whose first row is -1 (or >= G) is skipped and its D rows are left untouched. Rows
 * tagged -1 inside a computed block receive that block's expert's product (their content is
 * unspecified). Mt must be a multiple of 128.
 */
dg_status dg_m_grouped_contiguous(const uint8_t* A, const float* sfa, const uint8_t* B, const float* sfb,
                                  const int32_t* m_indices, void* D, int Mt, int N, int K, int G,
                                  cudaStream_t stream);

/*
 * m-grouped GEMM, masked layout (pages: m_grouped_gemm_fp8_fp8_bf16_nt_masked; for decode, including
 * under CUDA graphs, since every shape argument is static and the per-expert counts stay on device).
 *   A        [G, max_m, K]            sfa [G, max_m, K/128]
 *   B        [G, N, K]                sfb [G, ceil(N/128), K/128]
 *   masked_m [G] int32 (device)       valid rows per expert, clamped to [0, max_m] on device
 *   D        [G, max_m, N] bf16
 * For r < masked_m[g]: D[g,r] = A[g,r] . B[g]^T. Rows r >= masked_m[g] are never written.
 * expected_m is a performance hint (typical masked_m); <= 0 means unknown. 1 <= G <= 1024.
 */
dg_status dg_m_grouped_masked(const uint8_t* A, const float* sfa, const uint8_t* B, const float* sfb,
                              const int32_t* masked_m, void* D, int G, int max_m, int N, int K,
                              int expected_m, cudaStream_t stream);

/*
 * k-grouped weight-gradient GEMM with FP32 output (pages: k_grouped_wgrad_gemm_fp8_fp8_fp32_nt; the
 * MoE backward dW = X^T . dY per expert). Each expert g owns a window of ks[g] columns of the
 * token dimension, windows laid out in order:
 *   A  = X^T  [M, sumK]   e4m3        sfa [M, sumK/128]   (1x128 scales along K)
 *   B  = dY^T [N, sumK]   e4m3        sfb [N, sumK/128]   (1x128 scales along K, per row)
 *   ks_host [G] int32, HOST memory, each a multiple of 128 (0 allowed), sumK = sum(ks)
 *   D  [G, M, N] fp32, accumulated: D[g] += A[:, win_g] . B[:, win_g]^T
 * 1 <= G <= 128.
 */
dg_status dg_k_grouped_wgrad(const uint8_t* A, const float* sfa, const uint8_t* B, const float* sfb,
                             const int32_t* ks_host, float* D, int G, int M, int N,
                             cudaStream_t stream);

/*
 * Dense weight-gradient GEMM with FP32 output (pages: wgrad_gemm_fp8_fp8_fp32_nt; dW = X^T . dY of a
 * dense layer in the backward pass). The single-expert case of dg_k_grouped_wgrad, plus an
 * overwriting form:
 *   A = X^T  [M, K]   e4m3        sfa [M, K/128]   (1x128 scales along K)
 *   B = dY^T [N, K]   e4m3        sfb [N, K/128]   (1x128 scales along K, per row)
 *   D        [M, N]   fp32: D += A . B^T if accumulate != 0, else D = A . B^T (old contents ignored)
 * K must be a multiple of 128. K == 0 leaves D unchanged when accumulating and zeroes it otherwise.
 */
dg_status dg_wgrad_fp8_nt(const uint8_t* A, const float* sfa, const uint8_t* B, const float* sfb,
                          float* D, int M, int N, int K, int accumulate, cudaStream_t stream);

/* Human-readable name of a status code (static storage). */
const char* dg_status_string(dg_status status);

/*
 * Synchronises `stream`, then reports (and clears) the device-side error recorded by any dg kernel on
 * the current device since the last call: DG_DEVICE_TIMEOUT, or DG_SCALE_NOT_UE8M0 from the UE8M0
 * path, else DG_CUDA_ERROR if the synchronisation failed, else DG_OK. Kernels record only the first
 * error (a later one does not overwrite it). Reading and clearing are two steps: an error that a dg
 * kernel on another stream records between them is lost, so call this while no other dg work runs on
 * the device when every error must be seen.
 */
dg_status dg_device_status(cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DG_H */
