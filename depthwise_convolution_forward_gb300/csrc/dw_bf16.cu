// Depthwise direct kernel (Ka) instantiations for __nv_bfloat16 storage.
#include "dw_launch.cuh"

namespace gconv {
cudaError_t dw_launch_bf16(const Geometry& g, const LaunchArgs& a, const DeviceInfo& dev) {
  return dw::dw_launch_typed<__nv_bfloat16>(g, a, dev);
}
int dw_col_regs_bf16(int S, int DL, int form) { return dw::col_kernel_regs<__nv_bfloat16>(S, DL, form); }
}  // namespace gconv
