// Kb: tcgen05 / TMEM grouped implicit GEMM (placeholder until implemented).
#include "kernels.h"

namespace gconv {

bool tc_supported(const Geometry&, DType, const LaunchArgs*) { return false; }

cudaError_t tc_launch(const Geometry&, const LaunchArgs&, const DeviceInfo&) { return cudaErrorNotSupported; }

}  // namespace gconv
