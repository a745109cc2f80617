// Test harness (host only): the selector's support checks against the
// launchers' own planners, for a given SM count and shared-memory limit, on
// problems read from stdin; one JSON line per problem on stdout.  Built and
// run by tests/test_plans.py; nothing here launches a kernel.
#include "../../depthwise_convolution_forward_gb300/csrc/dw.cu"
#include "../../depthwise_convolution_forward_gb300/csrc/tc.cu"

#include <cstdio>

namespace gconv {
CUresult encode_tiled(CUtensorMap*, CUtensorMapDataType, uint32_t, const void*, const uint64_t*, const uint64_t*,
                      const uint32_t*, const uint32_t*, CUtensorMapSwizzle) {
  return CUDA_ERROR_NOT_SUPPORTED;
}
// The per-dtype depthwise launchers are never called here.
cudaError_t dw_launch_f32(const Geometry&, const LaunchArgs&, const DeviceInfo&) { return cudaErrorNotSupported; }
cudaError_t dw_launch_f16(const Geometry&, const LaunchArgs&, const DeviceInfo&) { return cudaErrorNotSupported; }
cudaError_t dw_launch_bf16(const Geometry&, const LaunchArgs&, const DeviceInfo&) { return cudaErrorNotSupported; }
int dw_col_regs_f32(int, int, int) { return -1; }
int dw_col_regs_f16(int, int, int) { return -1; }
int dw_col_regs_bf16(int, int, int) { return -1; }
}  // namespace gconv

using namespace gconv;

int main() {
  Geometry g{};
  int dt, sms, smem, regs;
  long long N;
  // per problem: geometry, dtype (0 f32, 1 f16, 2 bf16), SM count, opt-in
  // shared memory per block, registers per thread of the column kernel
  while (scanf("%lld %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d", &N, &g.G,
               &g.Cg, &g.Kg, &g.D, &g.H, &g.W, &g.Do, &g.Ho, &g.Wo, &g.Z, &g.Y, &g.X, &g.sD, &g.sH, &g.sW, &g.pD,
               &g.pH, &g.pW, &g.dD, &g.dH, &g.dW, &g.ndim, &dt, &sms, &smem, &regs) == 27) {
    g.N = N;
    const DType t = (DType)dt;
    const int es = dtype_bytes(t);
    const bool dw_sel = dw_supported(g, t, nullptr, sms);
    const bool tc_sel = tc_supported(g, t, nullptr, sms, smem);
    // what the launchers plan: the column form with the kernel's registers
    // when the depth filter is 1 (else the row-blocked form); the tensor-core
    // planner with the device's SM count and shared memory
    dw::Plan dp{};
    bool dw_plan = false;
    if (g.Z == 1) dw_plan = dw::make_col_plan(g, es, nullptr, sms, dw::col_form(es, nullptr, g.Cg), regs, &dp);
    if (!dw_plan && g.Cg == 1) dw_plan = dw::make_plan(g, es, nullptr, sms, &dp);
    dw_plan = dw_plan && dp.smem_bytes <= (uint32_t)smem;
    TcPlan tp;
    std::memset(&tp, 0, sizeof(tp));
    const bool tc_plan = t != kF32 && make_tc_plan(g, t == kBF16, sms, smem, nullptr, &tp);
    printf("{\"dw_sel\": %d, \"dw_plan\": %d, \"tc_sel\": %d, \"tc_plan\": %d, \"dw_smem\": %u, \"dw_TC\": %d, "
           "\"tc_grid\": %d}\n",
           (int)dw_sel, (int)dw_plan, (int)tc_sel, (int)tc_plan, dp.smem_bytes, dp.TC, tp.grid);
  }
  return 0;
}
