// Depthwise direct kernel (Ka) instantiations for float storage.
#include "dw_launch.cuh"

namespace gconv {
cudaError_t dw_launch_f32(const Geometry& g, const LaunchArgs& a, const DeviceInfo& dev) {
  return dw::dw_launch_typed<float>(g, a, dev);
}
int dw_col_regs_f32(int S, int DL, int form) { return dw::col_kernel_regs<float>(S, DL, form); }
}  // namespace gconv
