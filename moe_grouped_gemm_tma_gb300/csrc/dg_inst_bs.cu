// Specialisations of the block-scaled (UE8M0) normal GEMM, and their launch.
#include <cuda_runtime.h>

#include <mutex>

#include "dg_kernel_bs.cuh"
#include "dg_launch.cuh"

namespace dg {

template <int BN, int PAIR>
cudaError_t launch_bs(const Launch& L) {
    using C = CfgBS<BN, PAIR>;
    auto kern = dg_gemm_bs_kernel<BN, PAIR>;
    static std::mutex mu;
    static int ready[64] = {0};
    static int pair_clusters[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!ready[dev]) {
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::DYN_SMEM);
            if (e != cudaSuccess) return e;
            if (PAIR == 2) {
                // persistent pairs: as many as can be resident at once (one CTA per SM)
                cudaLaunchConfig_t q = {};
                cudaLaunchAttribute qa[1];
                qa[0].id = cudaLaunchAttributeClusterDimension;
                qa[0].val.clusterDim.x = 2;
                qa[0].val.clusterDim.y = 1;
                qa[0].val.clusterDim.z = 1;
                q.attrs = qa;
                q.numAttrs = 1;
                q.blockDim = dim3(THREADS, 1, 1);
                q.dynamicSmemBytes = C::DYN_SMEM;
                q.gridDim = dim3(2u * static_cast<unsigned>(L.sms / 2), 1, 1);
                int clusters = 0;
                if (cudaOccupancyMaxActiveClusters(&clusters, kern, &q) != cudaSuccess || clusters <= 0)
                    clusters = L.sms / 2;
                pair_clusters[dev] = clusters;
            }
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
    if (PAIR == 2) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.numAttrs = 1;
        const int units = L.units < pair_clusters[dev] ? L.units : pair_clusters[dev];
        cfg.gridDim = dim3(static_cast<unsigned>(2 * units), 1, 1);
    } else if (L.params.split > 1) {
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

template cudaError_t launch_bs<128, 1>(const Launch&);
template cudaError_t launch_bs<192, 1>(const Launch&);
template cudaError_t launch_bs<224, 1>(const Launch&);
template cudaError_t launch_bs<256, 1>(const Launch&);
template cudaError_t launch_bs<128, 2>(const Launch&);
template cudaError_t launch_bs<256, 2>(const Launch&);

}  // namespace dg
