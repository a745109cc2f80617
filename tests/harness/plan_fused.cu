// Test harness (host only): the fused depthwise + projection planner on
// problems read from stdin (the geometry, then bf16, K, act), one JSON line
// per problem on stdout.  Built and run by tests/test_plans.py; nothing here
// launches a kernel.
#include "../../depthwise_convolution_forward_gb300/csrc/fused.cu"

#include <cstdio>

namespace gconv {
// The planner never encodes a tensor map; the launch path that would is not run.
CUresult encode_tiled(CUtensorMap*, CUtensorMapDataType, uint32_t, const void*, const uint64_t*, const uint64_t*,
                      const uint32_t*, const uint32_t*, CUtensorMapSwizzle) {
  return CUDA_ERROR_NOT_SUPPORTED;
}
}  // namespace gconv

using namespace gconv;

int main() {
  Geometry g{};
  int bf16, K, act;
  long long N;
  while (scanf("%lld %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d", &N, &g.G, &g.Cg,
               &g.Kg, &g.D, &g.H, &g.W, &g.Do, &g.Ho, &g.Wo, &g.Z, &g.Y, &g.X, &g.sD, &g.sH, &g.sW, &g.pD, &g.pH,
               &g.pW, &g.dD, &g.dH, &g.dW, &g.ndim, &bf16, &K, &act) == 26) {
    g.N = N;
    DwPwPlan p;
    if (!make_dw_pw_plan(g, bf16 != 0, K, act, kDefaultSmemOptin, nullptr, &p)) {
      printf("{\"ok\": false}\n");
      continue;
    }
    const fz::DwPwArgs& a = p.a;
    printf("{\"ok\": true, \"smem\": %u, \"threads\": %d, \"C\": %d, \"K\": %d, \"Np\": %d, \"G\": %d, "
           "\"TH\": %d, \"TW\": %d, \"tiles_h\": %d, \"tiles_w\": %d, \"tiles\": %d, \"Win\": %d, \"Hin\": %d, "
           "\"CH\": %d, \"GC\": %d, \"GT\": %d, \"cpt\": %d, \"chunks\": %d, \"stages\": %d, \"nA\": %d, \"NS\": %d, \"rps\": %d, "
           "\"x_stage_bytes\": %u, \"x_stage_stride\": %u, \"a_bytes\": %u, \"wdw_off\": %u, \"bdw_off\": %u, "
           "\"bpw_off\": %u, \"b_off\": %u, \"a_off\": %u, \"x_off\": %u, \"tmem_cols\": %u, \"idesc\": %u, "
           "\"compute_threads\": %d, \"atom\": %u, \"max_stages\": %d, \"inline_mma\": %d}\n",
           p.smem_bytes, a.cpt == 8 ? fz::Cfg<8>::kThreads : fz::Cfg<4>::kThreads, a.C, a.K, a.Np, a.G, a.TH, a.TW, a.tiles_h, a.tiles_w, a.tiles, a.Win, a.Hin,
           a.CH, a.GC, a.GT, a.cpt, a.chunks, a.stages, a.nA, a.NS, a.rps, a.x_stage_bytes, a.x_stage_stride, a.a_bytes,
           a.wdw_off, a.bdw_off, a.bpw_off, a.b_off, a.a_off, a.x_off, a.tmem_cols, a.idesc, compute_threads(a.cpt),
           fz::kAtomBytes, fz::kMaxStages, a.inline_mma);
  }
  return 0;
}
