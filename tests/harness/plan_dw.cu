// Test harness (host only): the depthwise kernel's tile planners (column and
// row-blocked forms) on problems (with optional tile overrides) read from
// stdin, one JSON line per problem
// on stdout.  Built and run by tests/test_plans.py; nothing here launches a
// kernel.  The register count the column planner needs is an input.
#include "../../depthwise_convolution_forward_gb300/csrc/dw_launch.cuh"

#include <cstdio>

namespace gconv {
CUresult encode_tiled(CUtensorMap*, CUtensorMapDataType, uint32_t, const void*, const uint64_t*, const uint64_t*,
                      const uint32_t*, const uint32_t*, CUtensorMapSwizzle) {
  return CUDA_ERROR_NOT_SUPPORTED;
}
}  // namespace gconv

using namespace gconv;

int main() {
  Geometry g{};
  int es, regs, ov[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  long long N;
  // per problem: geometry, element size, registers, then overrides TH TW stages ctas (0 = automatic)
  while (scanf("%lld %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d", &N, &g.G,
               &g.Cg, &g.Kg, &g.D, &g.H, &g.W, &g.Do, &g.Ho, &g.Wo, &g.Z, &g.Y, &g.X, &g.sD, &g.sH, &g.sW, &g.pD,
               &g.pH, &g.pW, &g.dD, &g.dH, &g.dW, &g.ndim, &es, &regs, &ov[0], &ov[1], &ov[3], &ov[4]) == 29) {
    g.N = N;
    const bool any_ov = ov[0] || ov[1] || ov[3] || ov[4];
    dw::Plan p{};
    bool ok;
    int form = 0;
    if (g.Z == 1) {
      form = dw::col_form(es, nullptr, g.Cg);
      ok = dw::make_col_plan(g, es, any_ov ? ov : nullptr, 152, form, regs, &p);
    } else {
      ok = dw::make_plan(g, es, any_ov ? ov : nullptr, 152, &p);
    }
    if (!ok) {
      printf("{\"ok\": false}\n");
      continue;
    }
    printf("{\"ok\": true, \"col\": %d, \"form\": %d, \"max_threads\": %d, \"TH\": %d, \"TW\": %d, \"TC\": %d, "
           "\"Dh\": %d, \"Hh\": %d, \"Wh\": %d, \"tiles_c\": %d, \"tiles_w\": %d, \"tiles_h\": %d, "
           "\"num_tiles\": %lld, \"stage_bytes\": %u, \"stage_stride\": %u, \"stage_off\": %u, \"smem\": %u, "
           "\"stages\": %d, \"ctas\": %d, \"threads\": %d, \"direct\": %d, \"h0\": %d}\n",
           p.col, form, dw::col_max_threads(form), p.TH, p.TW, p.TC, p.Dh, p.Hh, p.Wh, p.tiles_c, p.tiles_w,
           p.tiles_h, (long long)p.num_tiles, p.stage_bytes, p.stage_stride, p.stage_off, p.smem_bytes, p.stages,
           p.ctas_per_sm, p.threads, p.direct, p.h0);
  }
  return 0;
}
