// Test harness (host only): the tensor-core backward-weight planner on
// problems read from stdin, one JSON line per problem on stdout.  Built and
// run by tests/test_plans.py; nothing here launches a kernel.
#include "../../depthwise_convolution_forward_gb300/csrc/bwdw_tc.cu"

#include <cstdio>

namespace gconv {
CUresult encode_tiled(CUtensorMap*, CUtensorMapDataType, uint32_t, const void*, const uint64_t*, const uint64_t*,
                      const uint32_t*, const uint32_t*, CUtensorMapSwizzle) {
  return CUDA_ERROR_NOT_SUPPORTED;
}
cudaError_t bwd_weight_reduce_launch(const Geometry&, const LaunchArgs&, float*, int, const DeviceInfo&) {
  return cudaErrorNotSupported;
}
}  // namespace gconv

using namespace gconv;

int main() {
  Geometry g{};
  int half;
  long long N;
  while (scanf("%lld %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d", &N, &g.G, &g.Cg, &g.Kg,
               &g.D, &g.H, &g.W, &g.Do, &g.Ho, &g.Wo, &g.Z, &g.Y, &g.X, &g.sD, &g.sH, &g.sW, &g.pD, &g.pH, &g.pW,
               &g.dD, &g.dH, &g.dW, &g.ndim, &half) == 24) {
    g.N = N;
    BwtPlan p;
    if (!make_bwt_plan(g, half != 0, &p)) {
      printf("{\"ok\": false}\n");
      continue;
    }
    const bwt::BwtArgs& a = p.a;
    printf("{\"ok\": true, \"smem\": %u, \"grid\": %d, \"S\": %d, \"E\": %lld, \"tiles\": %lld, \"tiles_h\": %d, "
           "\"TH\": %d, \"P\": %d, \"Kp\": %d, \"stages\": %d, \"nplane\": %d, \"dy_bytes\": %u, "
           "\"plane_bytes\": %u, \"stage_bytes\": %u, \"tx_bytes\": %u, \"ncols\": %u, \"tmem_cols\": %u, "
           "\"rows\": %d, \"chunks\": %d, \"qx_min\": %d, \"plane_px\": [%d, %d], \"runs\": [",
           p.smem_bytes, p.grid, a.S, (long long)a.E, (long long)a.tiles, a.tiles_h, a.TH, a.P, a.Kp, a.stages,
           a.nplane, a.dy_bytes, a.plane_bytes, a.stage_bytes, a.tx_bytes, a.ncols, a.tmem_cols, a.rows, a.chunks,
           a.qx_min, a.plane_px[0], a.plane_px[1]);
    for (int q = 0; q < a.nruns; ++q) {
      printf("%s{\"len\": %d, \"u0\": %d, \"du\": %d, \"plane\": %d, \"idesc\": %u, \"kx\": [", q ? ", " : "",
             a.run_len[q], a.run_u0[q], a.run_du[q], a.run_plane[q], a.run_idesc[q]);
      for (int b = 0; b < a.run_len[q]; ++b) printf("%s%d", b ? ", " : "", a.run_kx[q][b]);
      printf("]}");
    }
    printf("], \"row_qy\": [");
    for (int r = 0; r < a.rows; ++r) printf("%s%d", r ? ", " : "", a.row_qy[r]);
    printf("], \"row_py\": [");
    for (int r = 0; r < a.rows; ++r) printf("%s%d", r ? ", " : "", a.row_py[r]);
    printf("]}\n");
  }
  return 0;
}
