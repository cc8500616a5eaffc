// Kernel specialisations of the kgrouped layout (one translation unit per layout).
#define DG_DEFINE_LAUNCH
#include "dg_launch.cuh"

namespace dg {
template cudaError_t launch<kKGrouped, 128, 1>(const Launch&);
template cudaError_t launch<kKGrouped, 192, 1>(const Launch&);
template cudaError_t launch<kKGrouped, 224, 1>(const Launch&);
template cudaError_t launch<kKGrouped, 256, 1>(const Launch&);
template cudaError_t launch<kKGrouped, 128, 2>(const Launch&);
}  // namespace dg
