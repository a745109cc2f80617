// Depthwise direct kernel (Ka) instantiations for __nv_bfloat16 storage.
#include "dw_launch.cuh"

namespace gconv {
cudaError_t dw_launch_bf16(const Geometry& g, const LaunchArgs& a, const DeviceInfo& dev) {
  return dw::dw_launch_typed<__nv_bfloat16>(g, a, dev);
}
}  // namespace gconv
