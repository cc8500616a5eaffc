// Specialisations of the swapped-operand (small-M) normal GEMM, and their launch.
#include <cuda_runtime.h>

#include <mutex>

#include "dg_kernel_swap.cuh"
#include "dg_launch.cuh"

namespace dg {

template <int BMT>
cudaError_t launch_swap(const Launch& L) {
    using C = CfgSW<BMT>;
    auto kern = dg_gemm_swap_kernel<BMT>;
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
            // the warpgroups re-split the launch's registers with setmaxnreg (see launch<>)
            cudaFuncAttributes fa;
            e = cudaFuncGetAttributes(&fa, kern);
            if (e != cudaSuccess) return e;
            if (fa.numRegs * THREADS != CTRL_REGS * 128 + EPI_REGS * (THREADS - 128)) return cudaErrorInvalidConfiguration;
            ready[dev] = 1;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = C::DYN_SMEM;
    cfg.stream = L.stream;
    cfg.numAttrs = 0;
    if (L.params.split > 1) {
        // one cluster of `split` CTAs per tile, not persistent
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
    cfg.attrs = cfg.numAttrs ? attr : nullptr;
    return cudaLaunchKernelEx(&cfg, kern, L.tmap_a, L.tmap_b, L.tmap_d, L.params);
}

template cudaError_t launch_swap<32>(const Launch&);
template cudaError_t launch_swap<64>(const Launch&);
template cudaError_t launch_swap<128>(const Launch&);

}  // namespace dg
