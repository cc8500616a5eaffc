// Host-side launch of one kernel specialisation (mode, BN, CTA pair). Each dg_inst_*.cu file
// instantiates the specialisations of one mode, so the kernels compile in parallel translation units.
#pragma once

#include <cuda_runtime.h>

#include <mutex>

#include "dg_kernel.cuh"
#include "dg_tuning.h"

namespace dg {

struct Launch {
    CUtensorMap tmap_a;
    CUtensorMap tmap_b;
    CUtensorMap tmap_d;     // the BF16 output for TMA stores (unused by the k-grouped gradient)
    Params params;
    int units;          // work units wanted: tiles (single CTA) or tile pairs (CTA pairs)
    int sms;
    cudaStream_t stream;
};

template <int MODE, int BN, int PAIR>
cudaError_t launch(const Launch& L);

// The block-scaled (UE8M0) normal GEMM (dg_inst_bs.cu).
template <int BN, int PAIR>
cudaError_t launch_bs(const Launch& L);

// The few-row ("decode") kernel, normal or masked layout (dg_inst_decode.cu): L.units clusters of
// L.params.split CTAs (or CTAs, unsplit), persistent over the tiles.
template <int MODE, int BMT>
cudaError_t launch_decode(const Launch& L);

// Clusters of `split` decode CTAs that can be resident at once (SMs for split 1).
template <int MODE, int BMT>
int decode_cluster_capacity(int split, int sms);

// Tuning knobs (dg_tuning.h): the knob's value, or DG_TUNE_AUTO (-1) for the automatic choice.
int tune(int knob);

// The one-shot wait-limit fault armed by dg_testing_arm_wait_timeout (0 when none is armed); taking it
// disarms it, so exactly one launch carries it.
unsigned long long take_armed_wait_fault();

// Programmatic dependent launch is on unless the DG_TUNE_PDL knob is 0.
inline bool pdl_enabled() { return tune(DG_TUNE_PDL) != 0; }

#ifdef DG_DEFINE_LAUNCH
template <int MODE, int BN, int PAIR>
cudaError_t launch(const Launch& L) {
    using C = Cfg<MODE, BN, PAIR>;
    auto kern = dg_gemm_kernel<MODE, BN, PAIR>;
    // One-time set-up per device for this specialisation (the shared-memory attribute and the checks
    // below are per function and device; caching them keeps the per-call host cost low).
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
            // the warpgroups re-split the launch's registers with setmaxnreg; that split must equal what
            // the kernel was compiled to launch with, or a raising warpgroup would wait forever
            cudaFuncAttributes fa;
            e = cudaFuncGetAttributes(&fa, kern);
            if (e != cudaSuccess) return e;
            if (fa.numRegs * C::THREADS_C != CTRL_REGS * 128 + C::EPI_REGS_C * (C::THREADS_C - 128))
                return cudaErrorInvalidConfiguration;
            if (PAIR == 2) {
                cudaLaunchConfig_t q = {};
                cudaLaunchAttribute qa[1];
                qa[0].id = cudaLaunchAttributeClusterDimension;
                qa[0].val.clusterDim.x = 2;
                qa[0].val.clusterDim.y = 1;
                qa[0].val.clusterDim.z = 1;
                q.attrs = qa;
                q.numAttrs = 1;
                q.blockDim = dim3(C::THREADS_C, 1, 1);
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
    cfg.blockDim = dim3(C::THREADS_C, 1, 1);
    cfg.dynamicSmemBytes = C::DYN_SMEM;
    cfg.stream = L.stream;
    if ((MODE == kNormal || MODE == kMasked) && PAIR == 1 && L.params.split > 1) {
        // split-K: one cluster of `split` CTAs per tile (masked: per possible tile), not persistent
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(L.params.split);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cfg.gridDim = dim3(static_cast<unsigned>(L.units * L.params.split), 1, 1);
    } else if (PAIR == 2) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        // persistent: as many pairs as can be resident at once (one CTA per SM)
        const int clusters = pair_clusters[dev];
        const int units = L.units < clusters ? L.units : clusters;
        cfg.gridDim = dim3(static_cast<unsigned>(2 * units), 1, 1);
    } else {
        cfg.attrs = nullptr;
        cfg.numAttrs = 0;
        const int units = L.units < L.sms ? L.units : L.sms;
        cfg.gridDim = dim3(static_cast<unsigned>(units), 1, 1);
    }
    if (cfg.gridDim.x == 0) return cudaSuccess;
    // programmatic dependent launch: the kernel waits (griddepcontrol.wait) before its first global
    // memory access, so its set-up may overlap the tail of the previous grid in the stream
    if (pdl_enabled()) {
        attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs += 1;
    }
    Params prm = L.params;
    if (const unsigned long long ns = take_armed_wait_fault()) {
        prm.wait_limit_ns = ns;
        prm.fault_skip_first_fill = 1;
    }
    return cudaLaunchKernelEx(&cfg, kern, L.tmap_a, L.tmap_b, L.tmap_d, prm);
}
#endif

}  // namespace dg
