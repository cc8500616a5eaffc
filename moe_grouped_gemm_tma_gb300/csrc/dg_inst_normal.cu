// Kernel specialisations of the normal layout (one translation unit per layout).
#define DG_DEFINE_LAUNCH
#include "dg_launch.cuh"

namespace dg {
template cudaError_t launch<kNormal, 64, 1>(const Launch&);
template cudaError_t launch<kNormal, 96, 1>(const Launch&);
template cudaError_t launch<kNormal, 128, 1>(const Launch&);
template cudaError_t launch<kNormal, 160, 1>(const Launch&);
template cudaError_t launch<kNormal, 192, 1>(const Launch&);
template cudaError_t launch<kNormal, 224, 1>(const Launch&);
template cudaError_t launch<kNormal, 256, 1>(const Launch&);
template cudaError_t launch<kNormal, 128, 2>(const Launch&);
template cudaError_t launch<kNormal, 160, 2>(const Launch&);
template cudaError_t launch<kNormal, 192, 2>(const Launch&);
template cudaError_t launch<kNormal, 224, 2>(const Launch&);
template cudaError_t launch<kNormal, 256, 2>(const Launch&);
}  // namespace dg
