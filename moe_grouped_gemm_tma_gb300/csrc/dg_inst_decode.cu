// Specialisations of the few-row ("decode") kernel, their launch, and the cluster capacity the host
// plans split-K with.
#include <cuda_runtime.h>

#include <mutex>

#include "dg_kernel_decode.cuh"
#include "dg_launch.cuh"

namespace dg {

namespace {

template <int MODE, int BMT>
cudaError_t setup_decode(int dev) {
    using C = CfgDec<BMT>;
    auto kern = dg_decode_kernel<MODE, BMT>;
    static std::mutex mu;
    static int ready[64] = {0};
    std::lock_guard<std::mutex> lock(mu);
    if (ready[dev]) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::DYN_SMEM);
    if (e != cudaSuccess) return e;
    // the warpgroups re-split the launch's registers with setmaxnreg; the split must equal what the kernel
    // was compiled to launch with, or a raising warpgroup would wait forever
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    if (fa.numRegs * THREADS != CTRL_REGS * 128 + EPI_REGS * (THREADS - 128)) return cudaErrorInvalidConfiguration;
    ready[dev] = 1;
    return cudaSuccess;
}

}  // namespace

template <int MODE, int BMT>
int decode_cluster_capacity(int split, int sms) {
    using C = CfgDec<BMT>;
    if (split <= 1) return sms;
    static std::mutex mu;
    static int cache[64][9] = {{0}};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || split > 8) return sms / split;
    if (setup_decode<MODE, BMT>(dev) != cudaSuccess) return sms / split;
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev][split]) {
        cudaLaunchConfig_t q = {};
        cudaLaunchAttribute qa[1];
        qa[0].id = cudaLaunchAttributeClusterDimension;
        qa[0].val.clusterDim.x = static_cast<unsigned>(split);
        qa[0].val.clusterDim.y = 1;
        qa[0].val.clusterDim.z = 1;
        q.attrs = qa;
        q.numAttrs = 1;
        q.blockDim = dim3(THREADS, 1, 1);
        q.dynamicSmemBytes = C::DYN_SMEM;
        q.gridDim = dim3(static_cast<unsigned>(split * (sms / split)), 1, 1);
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, dg_decode_kernel<MODE, BMT>, &q) != cudaSuccess || clusters <= 0)
            clusters = sms / split;
        cache[dev][split] = clusters;
    }
    return cache[dev][split];
}

template <int MODE, int BMT>
cudaError_t launch_decode(const Launch& L) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    e = setup_decode<MODE, BMT>(dev);
    if (e != cudaSuccess) return e;
    using C = CfgDec<BMT>;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = C::DYN_SMEM;
    cfg.stream = L.stream;
    cfg.numAttrs = 0;
    const int split = L.params.split > 1 ? L.params.split : 1;
    if (split > 1) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(split);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.numAttrs = 1;
    }
    // persistent: L.units clusters (or CTAs), each looping over tiles
    cfg.gridDim = dim3(static_cast<unsigned>(L.units * split), 1, 1);
    if (cfg.gridDim.x == 0) return cudaSuccess;
    if (pdl_enabled()) {
        attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
        cfg.numAttrs += 1;
    }
    cfg.attrs = cfg.numAttrs ? attr : nullptr;
    return cudaLaunchKernelEx(&cfg, dg_decode_kernel<MODE, BMT>, L.tmap_a, L.tmap_b, L.params);
}

template int decode_cluster_capacity<kNormal, 32>(int, int);
template int decode_cluster_capacity<kNormal, 64>(int, int);
template int decode_cluster_capacity<kNormal, 128>(int, int);
template int decode_cluster_capacity<kMasked, 32>(int, int);
template int decode_cluster_capacity<kMasked, 64>(int, int);
template int decode_cluster_capacity<kMasked, 128>(int, int);
template cudaError_t launch_decode<kNormal, 32>(const Launch&);
template cudaError_t launch_decode<kNormal, 64>(const Launch&);
template cudaError_t launch_decode<kNormal, 128>(const Launch&);
template cudaError_t launch_decode<kMasked, 32>(const Launch&);
template cudaError_t launch_decode<kMasked, 64>(const Launch&);
template cudaError_t launch_decode<kMasked, 128>(const Launch&);

}  // namespace dg
