// Test harness (host only): the tensor-core kernel's tile planner on problems
// read from stdin, one JSON line per problem on stdout.  Built and run by
// tests/test_plans.py; nothing here launches a kernel.
#include "../../depthwise_convolution_forward_gb300/csrc/tc.cu"

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
  int bf16, ov[8];
  long long N;
  while (scanf("%lld %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d", &N, &g.G,
               &g.Cg, &g.Kg, &g.D, &g.H, &g.W, &g.Do, &g.Ho, &g.Wo, &g.Z, &g.Y, &g.X, &g.sD, &g.sH, &g.sW, &g.pD,
               &g.pH, &g.pW, &g.dD, &g.dH, &g.dW, &g.ndim, &bf16, &ov[0], &ov[2], &ov[3], &ov[4], &ov[5]) == 29) {
    g.N = N;
    ov[1] = ov[6] = ov[7] = 0;
    const bool any_ov = ov[0] || ov[2] || ov[3] || ov[4] || ov[5];
    TcPlan p;
    std::memset(&p, 0, sizeof(p));
    const int m = merge_factor(g);
    const bool ok = m > 0 && make_tc_plan(g, bf16 != 0, 152, 232448, any_ov ? ov : nullptr, &p);
    if (!ok) {
      printf("{\"ok\": false, \"m\": %d}\n", m);
      continue;
    }
    const tc::TcArgs& a = p.a;
    uint32_t max_a = 0, max_b = 0, min_a = 0xffffffffu;
    for (int i = 0; i < a.ntab; ++i) {
      const uint2 e = a.tab[i];
      if ((e.y >> 16) & 2u) continue;  // skipped slot
      max_a = std::max(max_a, (e.x & 0xffffu) << 4);
      min_a = std::min(min_a, (e.x & 0xffffu) << 4);
      max_b = std::max(max_b, (e.x >> 16) << 4);
    }
    printf("{\"ok\": true, \"m\": %d, \"sw\": %d, \"smem\": %u, \"grid\": %d, \"tmem_cols\": %u, \"np\": %d, "
           "\"nmt\": %d, \"sc\": %d, \"Nn\": %d, \"KS\": %d, \"TH\": %d, \"TWo\": %d, \"P\": %d, \"Hh\": %d, "
           "\"Dh\": %d, \"stages\": %d, \"a_off\": %u, \"b_off\": %u, \"a_stage_bytes\": %u, \"plane_stride\": %u, "
           "\"nphase\": %d, \"nchunks\": %d, \"tx_bytes\": %u, \"tiles_h\": %d, \"tiles_w\": %d, \"spatial\": %d, "
           "\"cpg\": %d, \"n_gc\": %d, \"ntab\": %d, \"max_a\": %u, \"min_a\": %u, \"shift\": %d, \"max_b\": %u, \"tab_off\": %u, "
           "\"bias_off\": %u, \"epi_off\": %u, \"epi_w\": %d, \"epi_slices\": %d, \"epi_slice_bytes\": %u, "
           "\"nbuf\": %d, \"plane_cx\": [%d, %d, %d, %d, %d, %d, %d, %d], \"tap_phase\": [%d, %d, %d, %d, %d, %d, %d, %d, %d], "
           "\"tap_off\": [%d, %d, %d, %d, %d, %d, %d, %d, %d]}\n",
           m, (int)p.sw, p.smem_bytes, p.grid, a.tmem_cols, a.np, a.nmt, a.sc, a.Nn, a.KS, a.TH, a.TWo, a.P, a.Hh,
           a.Dh, a.stages, a.a_off, a.b_off, a.a_stage_bytes, a.plane_stride, a.nphase, a.nchunks, a.tx_bytes,
           a.tiles_h, a.tiles_w, a.spatial_tiles, a.cpg, a.n_gc, a.ntab, max_a, min_a, a.shift, max_b, a.tab_off, a.bias_off,
           a.epi_off, a.epi_w, a.epi_slices, a.epi_slice_bytes, a.nbuf, a.plane_cx[0], a.plane_cx[1], a.plane_cx[2],
           a.plane_cx[3], a.plane_cx[4], a.plane_cx[5], a.plane_cx[6], a.plane_cx[7], a.tap_phase[0], a.tap_phase[1],
           a.tap_phase[2], a.tap_phase[3], a.tap_phase[4], a.tap_phase[5], a.tap_phase[6], a.tap_phase[7],
           a.tap_phase[8], a.tap_off[0], a.tap_off[1], a.tap_off[2], a.tap_off[3], a.tap_off[4], a.tap_off[5],
           a.tap_off[6], a.tap_off[7], a.tap_off[8]);
  }
  return 0;
}
