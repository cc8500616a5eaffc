// Host-side launch of one kernel specialisation (mode, BN). Each dg_inst_*.cu file instantiates the
// specialisations of one mode, so the kernels compile in parallel translation units.
#pragma once

#include <cuda_runtime.h>

#include "dg_kernel.cuh"

namespace dg {

struct Launch {
    CUtensorMap tmap_a;
    CUtensorMap tmap_b;
    Params params;
    int grid;
    cudaStream_t stream;
};

template <int MODE, int BN>
cudaError_t launch(const Launch& L);

template <int MODE, int BN>
int dyn_smem_bytes() { return Cfg<MODE, BN>::DYN_SMEM; }

#ifdef DG_DEFINE_LAUNCH
template <int MODE, int BN>
cudaError_t launch(const Launch& L) {
    using C = Cfg<MODE, BN>;
    auto kern = dg_gemm_kernel<MODE, BN>;
    // the attribute is per function and cheap to set; setting it every call keeps this free of
    // per-device caches
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::DYN_SMEM);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(L.grid), 1, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = C::DYN_SMEM;
    cfg.stream = L.stream;
    cfg.attrs = nullptr;
    cfg.numAttrs = 0;
    return cudaLaunchKernelEx(&cfg, kern, L.tmap_a, L.tmap_b, L.params);
}
#endif

}  // namespace dg
