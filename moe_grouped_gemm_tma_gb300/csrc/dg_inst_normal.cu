// Kernel specialisations of the normal layout (one translation unit per layout).
#define DG_DEFINE_LAUNCH
#include "dg_launch.cuh"

namespace dg {
template cudaError_t launch<kNormal, 64>(const Launch&);
template cudaError_t launch<kNormal, 96>(const Launch&);
template cudaError_t launch<kNormal, 128>(const Launch&);
template cudaError_t launch<kNormal, 160>(const Launch&);
template cudaError_t launch<kNormal, 192>(const Launch&);
template cudaError_t launch<kNormal, 224>(const Launch&);
template cudaError_t launch<kNormal, 256>(const Launch&);
}  // namespace dg
