// Depthwise direct kernel (Ka) instantiations for __half storage.
#include "dw_launch.cuh"

namespace gconv {
cudaError_t dw_launch_f16(const Geometry& g, const LaunchArgs& a, const DeviceInfo& dev) {
  return dw::dw_launch_typed<__half>(g, a, dev);
}
int dw_col_regs_f16(int S, int DL, int form) { return dw::col_kernel_regs<__half>(S, DL, form); }
}  // namespace gconv
