// Ka dispatch: support check and per-dtype launch.
#include <cstring>

#include "dw_launch.cuh"
#include "kernels.h"
#include "plan_cache.h"

namespace gconv {

cudaError_t dw_launch_f32(const Geometry& g, const LaunchArgs& a, const DeviceInfo& dev);
cudaError_t dw_launch_f16(const Geometry& g, const LaunchArgs& a, const DeviceInfo& dev);
cudaError_t dw_launch_bf16(const Geometry& g, const LaunchArgs& a, const DeviceInfo& dev);
int dw_col_regs_f32(int S, int DL, int form);
int dw_col_regs_f16(int S, int DL, int form);
int dw_col_regs_bf16(int S, int DL, int form);

// Depthwise (Cg == Kg == 1), or groups of two channels (Cg == Kg == 2,
// 16-bit data, depth filter 1: the column form's two-channel dot products),
// 3x3 spatial filter, equal H/W stride and dilation in {1, 2}; channels a
// multiple of one 16-byte vector; x and y 16-byte aligned (TMA and
// vector-store requirements).  Any depth filter for depthwise, as long as
// the planner finds a tile that fits shared memory for this device's SM
// count (num_sms).
bool dw_supported(const Geometry& g, DType dt, const LaunchArgs* a, int num_sms) {
  const int es = dtype_bytes(dt);
  const int vec = 16 / es;
  const bool group2 = g.Cg == 2 && g.Kg == 2 && es == 2 && g.Z == 1;
  if (!((g.Cg == 1 && g.Kg == 1) || group2)) return false;
  if (g.Y != 3 || g.X != 3) return false;
  if (g.sH != g.sW || g.dH != g.dW) return false;
  if (g.sH < 1 || g.sH > 2 || g.dH < 1 || g.dH > 2) return false;
  if (g.C() % vec != 0) return false;
  if (g.Z > 7 || (g.Z - 1) * g.dD + 1 > 16) return false;
  if (g.W > (1 << 30) || g.H > (1 << 30)) return false;
  // the image index is a 32-bit tensor-map coordinate (element offsets are 64-bit)
  if (g.N >= (int64_t)1 << 31) return false;
  // all weights stay resident in shared memory (fp32 copy, at most 64 KB)
  if ((int64_t)g.taps() * g.C() * g.Cg * 4 > 64 * 1024) return false;
  if (a) {
    if ((reinterpret_cast<uintptr_t>(a->x) & 15) || (reinterpret_cast<uintptr_t>(a->y) & 15)) return false;
  }
  struct Key {
    Geometry g;
    int tile[8];
    int es, num_sms, with_device;
  } key;
  std::memset(&key, 0, sizeof(key));
  key.g = g;
  if (a) std::memcpy(key.tile, a->tile, sizeof(key.tile));
  key.es = es;
  key.with_device = a != nullptr;
  key.num_sms = num_sms;
  static PlanCache<int> cache;
  int ok = 0;
  if (cache.get(key, &ok)) return ok != 0;
  // With launch arguments a device is at hand: plan with the column kernel's
  // real register count, as the launch does (tile overrides may need it);
  // the host-only query plans with the most it can have.
  // The TMA forms run a layer whose taps read one stride phase as the
  // stride-1 layer over the subsampled input (dw::phase_subsample), and fall
  // back to the layer as it is; the launch plans in the same order.
  const int form = dw::col_form(es, a ? a->tile : nullptr, g.Cg);
  Geometry gs;
  const bool sub = !(a && a->tile[6] == 2) && dw::phase_subsample(g, &gs);
  for (int attempt = sub ? 0 : 1; attempt < 2 && !ok; ++attempt) {
    const Geometry& gq = attempt == 0 ? gs : g;
    int regs = dw::col_max_regs(form);
    if (a && gq.Z == 1) {
      const int r = dt == kF32 ? dw_col_regs_f32(gq.sH, gq.dH, form)
                               : (dt == kF16 ? dw_col_regs_f16(gq.sH, gq.dH, form)
                                             : dw_col_regs_bf16(gq.sH, gq.dH, form));
      if (r > 0) regs = r;
    }
    ok = dw::plannable(gq, es, a ? a->tile : nullptr, num_sms, regs) ? 1 : 0;
  }
  cache.put(key, ok);
  return ok != 0;
}

cudaError_t dw_launch(const Geometry& g, const LaunchArgs& a, const DeviceInfo& dev) {
  switch (a.dt) {
    case kF32: return dw_launch_f32(g, a, dev);
    case kF16: return dw_launch_f16(g, a, dev);
    case kBF16: return dw_launch_bf16(g, a, dev);
  }
  return cudaErrorNotSupported;
}

}  // namespace gconv
