// Kernel specialisations of the contiguous layout (one translation unit per layout).
#define DG_DEFINE_LAUNCH
#include "dg_launch.cuh"

namespace dg {
template cudaError_t launch<kContiguous, 128, 1>(const Launch&);
template cudaError_t launch<kContiguous, 160, 1>(const Launch&);
template cudaError_t launch<kContiguous, 192, 1>(const Launch&);
template cudaError_t launch<kContiguous, 224, 1>(const Launch&);
template cudaError_t launch<kContiguous, 256, 1>(const Launch&);
}  // namespace dg
