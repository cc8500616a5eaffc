// Kernel specialisations of the masked layout (one translation unit per layout).
#define DG_DEFINE_LAUNCH
#include "dg_launch.cuh"

namespace dg {
template cudaError_t launch<kMasked, 64, 1>(const Launch&);
template cudaError_t launch<kMasked, 128, 1>(const Launch&);
template cudaError_t launch<kMasked, 192, 1>(const Launch&);
template cudaError_t launch<kMasked, 224, 1>(const Launch&);
template cudaError_t launch<kMasked, 256, 1>(const Launch&);
template cudaError_t launch<kMasked, 128, 2>(const Launch&);
template cudaError_t launch<kMasked, 256, 2>(const Launch&);
}  // namespace dg
