// Specialisations of the block-scaled (UE8M0) normal GEMM, and their launch.
#include <cuda_runtime.h>

#include <mutex>

#include "dg_kernel_bs.cuh"
#include "dg_launch.cuh"

namespace dg {

template <int BN>
cudaError_t launch_bs(const Launch& L) {
    using C = CfgBS<BN>;
    auto kern = dg_gemm_bs_kernel<BN>;
    static std::mutex mu;
    static int ready[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!ready[dev]) {
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::DYN_SMEM);
            if (e != cudaSuccess) return e;
            ready[dev] = 1;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = C::DYN_SMEM;
    cfg.stream = L.stream;
    cfg.attrs = attr;
    cfg.numAttrs = 0;
    if (L.params.split > 1) {
        // split-K: one cluster of `split` CTAs per tile, not persistent
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(L.params.split);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.numAttrs = 1;
        cfg.gridDim = dim3(static_cast<unsigned>(L.units * L.params.split), 1, 1);
    } else {
        const int units = L.units < L.sms ? L.units : L.sms;
        cfg.gridDim = dim3(static_cast<unsigned>(units), 1, 1);
    }
    if (cfg.gridDim.x == 0) return cudaSuccess;
    if (pdl_enabled()) {
        attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
        cfg.numAttrs += 1;
    }
    return cudaLaunchKernelEx(&cfg, kern, L.tmap_a, L.tmap_b, L.tmap_d, L.params);
}

template cudaError_t launch_bs<128>(const Launch&);
template cudaError_t launch_bs<192>(const Launch&);
template cudaError_t launch_bs<224>(const Launch&);
template cudaError_t launch_bs<256>(const Launch&);

}  // namespace dg
