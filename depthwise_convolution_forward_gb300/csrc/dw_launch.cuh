// Host-side planning and launch of the depthwise direct kernel (Ka) for one
// element type.  Included once per dtype translation unit so the template
// instantiations compile in parallel.
#pragma once

#include <algorithm>

#include "dw_impl.cuh"
#include "dwc_impl.cuh"
#include "plan_cache.h"

namespace gconv {
namespace dw {

struct Plan {
  int TH, TW, TC, WB, stages, ctas_per_sm, mode;
  int direct;  // 1: direct-load variant (dw_ldg_kernel), 0: TMA-staged pipeline
  int col;     // 1: column form (dw_col_kernel)
  int h0;      // column form: halo rows of a tile's first copy (Hh: one copy)
  int Dh, Hh, Wh;
  int tiles_c, tiles_w, tiles_h;
  int64_t num_tiles;
  uint32_t stage_bytes, stage_stride, stage_off, smem_bytes;
  int threads;
  int sub;  // > 1: planned for the input subsampled by this stride (phase_subsample)
};

constexpr int kDwK = 3;  // compiled filter extent (Y == X == 3)
constexpr uint32_t kStageBudget = 48 * 1024;
constexpr int kDwModeDefault16 = kMixedFma;    // 16-bit storage
constexpr int kDwModeDefault32 = kWidenFfma2;  // fp32 storage

inline int ceil_div(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }
inline uint32_t align_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

// Choose TC (channels per tile): the whole pixel when it fits a TMA box,
// otherwise the largest divisor of C that is a multiple of VEC and <= 256.
inline int pick_tc(int C, int vec) {
  if (C <= 256) return C;
  for (int tc = 256 / vec * vec; tc >= vec; tc -= vec)
    if (C % tc == 0) return tc;
  return 256 / vec * vec;
}

// Row-blocked form for channel tile TC (see make_plan).
inline bool make_plan_tc(const Geometry& g, int es, const int* tile_override, int num_sms, int TC, Plan* out) {
  const int vec = 16 / es;
  const int direct = (tile_override && tile_override[6] == 2) ? 1 : 0;
  const int S = g.sH, DL = g.dH;
  Plan best{};
  double best_cost = 1e30;
  const int NV = TC / vec;
  const int Dh = (g.Z - 1) * g.dD + 1;
  for (int WB : {4, 8}) {
    if (tile_override && tile_override[2] && tile_override[2] != WB) continue;
    const int tw_max = std::min(ceil_div(g.Wo, WB) * WB, 64);
    for (int TW = WB; TW <= tw_max; TW += WB) {
      if (tile_override && tile_override[1] && tile_override[1] != TW) continue;
      const int Wh = (TW - 1) * S + (kDwK - 1) * DL + 1;
      if (Wh > 256) break;
      for (int TH = 1; TH <= std::min(g.Ho, 64); ++TH) {
        if (tile_override && tile_override[0] && tile_override[0] != TH) continue;
        const int Hh = (TH - 1) * S + (kDwK - 1) * DL + 1;
        if (Hh > 256) break;
        const uint32_t bytes = (uint32_t)Dh * Hh * Wh * TC * es;
        const int items = NV * (TW / WB) * TH;
        if (items > (direct ? 256 : (WB >= 8 ? 256 : 480))) break;
        if (!direct && bytes > kStageBudget && !(tile_override && tile_override[0])) break;
        const int tiles_w = ceil_div(g.Wo, TW), tiles_h = ceil_div(g.Ho, TH);
        const int tiles_c = ceil_div(g.C(), TC);
        const int64_t tiles = (int64_t)tiles_c * tiles_w * tiles_h * g.Do * g.N;
        // cost: shared-memory fill bytes per useful output byte, plus idle
        // compute slots, plus a penalty for too few threads per CTA and for
        // grids that leave SMs without work.
        const double fill = (double)tiles * bytes;
        const double useful = (double)g.N * g.Do * g.Ho * g.Wo * g.C() * es;
        const double slots = (double)tiles * TH * TW * TC;
        const double outs = (double)g.N * g.Do * g.Ho * g.Wo * g.C();
        double cost = fill / useful + 0.5 * (slots / outs);
        if (items < 128) cost += 0.5;
        if (tiles < num_sms) cost += 1.0;
        if (cost < best_cost) {
          best_cost = cost;
          best.TH = TH, best.TW = TW, best.TC = TC, best.WB = WB;
          best.Dh = Dh, best.Hh = Hh, best.Wh = Wh;
          best.tiles_c = tiles_c, best.tiles_w = tiles_w, best.tiles_h = tiles_h;
          best.num_tiles = tiles;
          best.stage_bytes = bytes;
          best.threads = (direct ? 0 : 32) + (items + 31) / 32 * 32;  // (producer warp) + consumers
        }
      }
    }
  }
  if (best_cost >= 1e30) return false;
  best.direct = direct;
  best.stage_stride = align_up(best.stage_bytes, 1024);
  // FMA form: override 1 = widen + fp32 FMA, 2 = mixed f16/bf16, 3 = widen + fp32x2
  const int ov_mode = tile_override ? tile_override[5] : 0;
  int mode = es == 2 ? kDwModeDefault16 : kDwModeDefault32;
  if (ov_mode >= 1 && ov_mode <= 3) mode = ov_mode - 1;
  if (mode == kMixedFma && es != 2) mode = kWidenFfma;
  best.mode = mode;
  best.stage_off = align_up(fixed_smem_bytes<kDwK>(g.Z, g.C(), es, mode), 1024);
  // Prefer two CTAs per SM (two independent copy/compute streams) with two
  // stages each; fall back to one CTA with up to four stages.
  const int ov_stages = tile_override ? tile_override[3] : 0;
  const int ov_ctas = tile_override ? tile_override[4] : 0;
  const uint32_t half_sm = 113 * 1024, full_sm = 220 * 1024;
  int ctas = ov_ctas ? ov_ctas : (best.stage_off + 2 * best.stage_stride <= half_sm ? 2 : 1);
  int stages = ov_stages ? std::min(ov_stages, kDwMaxStages) : (ctas == 2 ? 2 : kDwMaxStages);
  const uint32_t cap = ctas == 2 ? half_sm : full_sm;
  while (!ov_stages && stages > 2 && best.stage_off + stages * best.stage_stride > cap) --stages;
  best.stages = stages;
  best.ctas_per_sm = ctas;
  best.smem_bytes = best.stage_off + stages * best.stage_stride;
  if (direct) {
    best.stages = 0;
    best.smem_bytes = weight_smem_bytes(g.Z * kDwK * kDwK, best.TC, es, mode) + 4u * (uint32_t)best.TC;
  }
  *out = best;
  return true;
}

// Row-blocked (and direct-load) form: the channel tile is the whole pixel or
// the largest divisor of C up to 256 channels; when even the smallest spatial
// tile of that channel tile overflows the stage budget (deep filters, wide
// fp32 channels), narrower channel tiles (divisors of C, multiples of one
// 16-byte vector) are tried in turn.
inline bool make_plan(const Geometry& g, int es, const int* tile_override, int num_sms, Plan* out) {
  const int vec = 16 / es;
  const int tc0 = pick_tc(g.C(), vec);
  if (make_plan_tc(g, es, tile_override, num_sms, tc0, out)) return true;
  for (int tc = tc0 - vec; tc >= vec; tc -= vec)
    if (g.C() % tc == 0 && make_plan_tc(g, es, tile_override, num_sms, tc, out)) return true;
  return false;
}

// Operand form of the column kernel (override slot 5): 1 split 16-bit /
// scalar fp32, 2 packed 16-bit x4, 3 widened fp32x2, 4 packed 16-bit x8;
// automatic: packed x4 for 16-bit storage (as fast as the others and the
// fewest registers), scalar for fp32.
inline int col_form(int es, const int* ov, int cg = 1) {
  if (cg == 2) return kColGroup2;  // groups of two channels have one form
  const int ov_form = ov ? ov[5] : 0;
  int form = es == 2 ? kColPacked : kColSplit;
  if (ov_form == 1) form = kColSplit;
  if (ov_form == 2 && es == 2) form = kColPacked;
  if (ov_form == 3) form = kColWide;
  if (ov_form == 4 && es == 2) form = kColPacked8;
  return form;
}

// Column form (dw_col_kernel): depth filter 1 only.  Each consumer thread
// owns one output column of the tile and CPT channels, so a tile is TW
// columns x TC channels of threads and TH rows deep.  The plan minimises
//   (tiles / SMs) x (Hh + 3.7) x max(1, busiest scheduler's warps / 4) x k(CTAs per SM)
// A thread walks the Hh input rows of its column in sequence (each costs
// three loads and the taps it feeds), so a tile takes about as long as Hh
// rows plus a fixed start-up.  Resident CTAs overlap each other's copies and
// start-up but share the SM's issue slots: k = 1, 0.79, 0.72 for 1, 2, 3
// CTAs per SM.  The constants are fitted to measured times (C = 512, 28x28,
// tiles of 10 / 14 / 28 rows with one or two CTAs, and the MobileNetV2
// layers): a second CTA is worth 1.27x, not 2x, so tall tiles with less halo
// per output row can win.  Warps of a CTA are dealt to the SM's 4
// schedulers in turn, so the busiest one holds ceil(consumer warps / 4) per
// CTA; beyond about 4 warps a scheduler is issue-bound and its tiles slow
// down in proportion (9 consumer warps per CTA measured slower than 8).
// Resident CTAs per SM are bounded by shared memory, threads and the
// kernel's registers per thread (`regs`).
inline bool make_col_plan(const Geometry& g, int es, const int* ov, int num_sms, int form, int regs, Plan* out) {
  if (g.Z != 1) return false;
  const int S = g.sH, DL = g.dH;
  const int vec = 16 / es;
  const int cpt = col_cpt(es, form);
  const int TC = pick_tc(g.C(), vec);
  const int NQ = TC / cpt;
  const uint32_t fixed = align_up(col_fixed_smem_bytes(g.C()), 1024);
  const uint32_t half_sm = 113 * 1024, third_sm = 75 * 1024, full_sm = 220 * 1024;
  const int ov_th = ov ? ov[0] : 0, ov_tw = ov ? ov[1] : 0, ov_stages = ov ? ov[3] : 0, ov_ctas = ov ? ov[4] : 0;
  const int tiles_c = ceil_div(g.C(), TC);
  const int regs_warp = (regs + 7) / 8 * 8 * 32;
  Plan best{};
  double best_cost = 1e30;
  const int tw_max = std::min(g.Wo, (col_max_threads(form) - 32) / NQ);
  for (int TW = 1; TW <= tw_max; ++TW) {
    if (ov_tw && ov_tw != TW) continue;
    const int Wh = (TW - 1) * S + 2 * DL + 1;
    if (Wh > 256) break;
    const int ncons = (TW * NQ + 31) / 32 * 32;
    const int warps = ncons / 32;
    const int tiles_w = ceil_div(g.Wo, TW);
    for (int TH = 1; TH <= std::min(g.Ho, 64); ++TH) {
      if (ov_th && ov_th != TH) continue;
      const int Hh = (TH - 1) * S + 2 * DL + 1;
      if (Hh > 256) break;
      const uint32_t bytes = (uint32_t)Hh * Wh * TC * es;
      const uint32_t stride = align_up(bytes, 1024);
      for (int ctas = 1; ctas <= 3; ++ctas) {
        if (ov_ctas && ov_ctas != ctas) continue;
        const uint32_t cap = ctas == 1 ? full_sm : (ctas == 2 ? half_sm : third_sm);
        const int stages = ov_stages ? std::min(ov_stages, kDwMaxStages) : 2;
        if (fixed + (uint32_t)stages * stride > cap) continue;
        if (ctas * (ncons + 32) > 2048) continue;
        if (ctas * (warps + 1) * regs_warp > 65536) continue;
        const int tiles_h = ceil_div(g.Ho, TH);
        const int64_t tiles = (int64_t)tiles_c * tiles_w * tiles_h * g.Do * g.N;
        const double per_sm = (double)tiles / (double)num_sms;
        const int busiest = ctas * ((warps + 3) / 4);
        const double k = ctas == 1 ? 1.0 : (ctas == 2 ? 0.71 : 0.65);
        const double wide = warps > 8 ? 1.6 : 1.0;
        const double cost = per_sm * (Hh + 8.0) * std::max(1.0, busiest / 4.0) * k * wide;
        if (cost < best_cost) {
          best_cost = cost;
          best = Plan{};
          best.TH = TH, best.TW = TW, best.TC = TC;
          best.Dh = 1, best.Hh = Hh, best.Wh = Wh;
          best.tiles_c = tiles_c, best.tiles_w = tiles_w, best.tiles_h = tiles_h;
          best.num_tiles = tiles;
          best.stage_bytes = bytes;
          best.stage_stride = stride;
          best.stage_off = fixed;
          best.stages = stages;
          best.ctas_per_sm = ctas;
          best.threads = 32 + ncons;
        }
      }
    }
  }
  if (best_cost >= 1e30) return false;
  best.col = 1;
  best.mode = form;
  // Two copies per tile: the first ends at a multiple of the row block
  // (U = NA*S rows) near the middle, with the second copy's shared-memory
  // destination on a 128-byte boundary; otherwise one copy.
  {
    const int U = ((2 * DL) / S + 1) * S;
    const uint32_t row_bytes = (uint32_t)best.Wh * best.TC * es;
    best.h0 = best.Hh;
    for (int h0 = best.Hh / 2 / U * U; h0 >= U; h0 -= U)
      if (((uint32_t)h0 * row_bytes) % 128u == 0) {
        best.h0 = h0;
        break;
      }
    // The split measured slower than one copy (all CTAs' first copies compete
    // for DRAM either way), so it is used only on request: override slot 2 = 2.
    if (!(ov && ov[2] == 2)) best.h0 = best.Hh;
  }
  best.smem_bytes = best.stage_off + best.stages * best.stage_stride;
  *out = best;
  return true;
}

// Most registers a thread of the column kernel can have: its launch bound
// leaves at most 65536 / max threads, in steps of 8.
inline int col_max_regs(int form) { return 65536 / col_max_threads(form) / 8 * 8; }

// Whether some launch plan exists for the depthwise kernel (host only): the
// column form when the depth filter is 1, else the row-blocked form.  The
// column form is planned with `regs` registers per thread: the kernel's own
// count when the caller knows it, else col_max_regs (a plan found with that
// many is found with fewer too).  tile[6] picks the form as in
// dw_launch_typed.
inline bool plannable(const Geometry& g, int es, const int* ov, int num_sms, int regs) {
  Plan p;
  const int kind = ov ? ov[6] : 0;
  const int form = col_form(es, ov, g.Cg);
  if ((kind == 0 || kind == 3) && g.Z == 1 && make_col_plan(g, es, ov, num_sms, form, regs, &p)) return true;
  if (kind == 3 || g.Cg != 1) return false;  // groups of two channels: column form only
  return make_plan(g, es, ov, num_sms, &p);
}

// Every tap of a layer with stride s = dilation s >= 2 and padding a
// multiple of s reads only input rows and columns that are multiples of s
// (input row s*oh + s*ky - p = s*(oh + ky - p/s)).  Such a layer is the
// stride-1, dilation-1 layer with padding p/s over the input subsampled by s
// (extents ceil(H/s), ceil(W/s)), and the tensor map of that subsampled
// input is the dense one with its W and H strides multiplied by s: the
// copies then read only the positions the taps use (a quarter of x at
// s = 2) instead of whole haloed boxes.
inline bool phase_subsample(const Geometry& g, Geometry* gs) {
  const int s = g.sH;
  if (s < 2 || g.sW != s || g.dH != s || g.dW != s || g.pH % s != 0 || g.pW % s != 0) return false;
  Geometry t = g;
  t.H = (g.H + s - 1) / s, t.W = (g.W + s - 1) / s;
  t.sH = t.sW = t.dH = t.dW = 1;
  t.pH = g.pH / s, t.pW = g.pW / s;
  if (t.H + 2 * t.pH - (t.Y - 1) != g.Ho || t.W + 2 * t.pW - (t.X - 1) != g.Wo) return false;
  *gs = t;
  return true;
}

template <typename T>
inline CUtensorMapDataType tma_type() {
  if (std::is_same<T, float>::value) return CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  if (std::is_same<T, __half>::value) return CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  return CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
}

template <typename T>
using DwKernel = void (*)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const DwArgs);

// The compiled variant for (stride, dilation, register block, FMA form).
template <typename T>
DwKernel<T> pick_kernel(int S, int DL, int WB, int mode) {
#define GCONV_DW_CASE(s_, d_, wb_)                                               \
  if (S == s_ && DL == d_ && WB == wb_) {                                        \
    if constexpr (sizeof(T) == 2) {                                              \
      if (mode == kMixedFma) return dw_kernel<T, kDwK, s_, d_, wb_, kMixedFma>;  \
    }                                                                            \
    if (mode == kWidenFfma2) return dw_kernel<T, kDwK, s_, d_, wb_, kWidenFfma2>; \
    return dw_kernel<T, kDwK, s_, d_, wb_, kWidenFfma>;                          \
  }
  GCONV_DW_CASE(1, 1, 4)
  GCONV_DW_CASE(1, 1, 8)
  GCONV_DW_CASE(2, 1, 4)
  GCONV_DW_CASE(2, 1, 8)
  GCONV_DW_CASE(1, 2, 4)
  GCONV_DW_CASE(1, 2, 8)
  GCONV_DW_CASE(2, 2, 4)
  GCONV_DW_CASE(2, 2, 8)
#undef GCONV_DW_CASE
  return nullptr;
}

template <typename T>
DwKernel<T> pick_col_kernel(int S, int DL, int form) {
#define GCONV_COL_CASE(s_, d_)                                                      \
  if (S == s_ && DL == d_) {                                                        \
    if constexpr (sizeof(T) == 2) {                                                 \
      if (form == kColPacked) return dw_col_kernel<T, s_, d_, kColPacked>;          \
      if (form == kColPacked8) return dw_col_kernel<T, s_, d_, kColPacked8>;        \
      if (form == kColGroup2) return dw_col_kernel<T, s_, d_, kColGroup2>;          \
    } else {                                                                        \
      if (form == kColGroup2) return nullptr;                                       \
    }                                                                               \
    if (form == kColWide) return dw_col_kernel<T, s_, d_, kColWide>;                \
    return dw_col_kernel<T, s_, d_, kColSplit>;                                     \
  }
  GCONV_COL_CASE(1, 1)
  GCONV_COL_CASE(2, 1)
  GCONV_COL_CASE(1, 2)
  GCONV_COL_CASE(2, 2)
#undef GCONV_COL_CASE
  return nullptr;
}

template <typename T>
using DwLdgKernel = void (*)(const DwArgs);

template <typename T>
DwLdgKernel<T> pick_ldg_kernel(int S, int DL, int WB, int mode) {
#define GCONV_DW_CASE(s_, d_, wb_)                                                   \
  if (S == s_ && DL == d_ && WB == wb_) {                                            \
    if constexpr (sizeof(T) == 2) {                                                  \
      if (mode == kMixedFma) return dw_ldg_kernel<T, kDwK, s_, d_, wb_, kMixedFma>;  \
    }                                                                                \
    if (mode == kWidenFfma2) return dw_ldg_kernel<T, kDwK, s_, d_, wb_, kWidenFfma2>; \
    return dw_ldg_kernel<T, kDwK, s_, d_, wb_, kWidenFfma>;                          \
  }
  GCONV_DW_CASE(1, 1, 4)
  GCONV_DW_CASE(1, 1, 8)
  GCONV_DW_CASE(2, 1, 4)
  GCONV_DW_CASE(2, 1, 8)
  GCONV_DW_CASE(1, 2, 4)
  GCONV_DW_CASE(1, 2, 8)
  GCONV_DW_CASE(2, 2, 4)
  GCONV_DW_CASE(2, 2, 8)
#undef GCONV_DW_CASE
  return nullptr;
}

// Registers per thread of the column kernel for (stride, dilation, operand
// form), or -1 when there is no such kernel or the query fails.
template <typename T>
int col_kernel_regs(int S, int DL, int form) {
  DwKernel<T> k = pick_col_kernel<T>(S, DL, form);
  cudaFuncAttributes fa{};
  if (k == nullptr || cudaFuncGetAttributes(&fa, k) != cudaSuccess) return -1;
  return fa.numRegs;
}

template <typename T>
cudaError_t dw_launch_typed(const Geometry& g, const LaunchArgs& la, const DeviceInfo& dev) {
  const int es = sizeof(T);
  struct Key {
    Geometry g;
    int tile[8];
    int num_sms;
    int device;
  } key;
  std::memset(&key, 0, sizeof(key));
  key.g = g;
  std::memcpy(key.tile, la.tile, sizeof(key.tile));
  key.num_sms = dev.num_sms;
  key.device = dev.device;
  static PlanCache<Plan> cache;
  Plan p;
  static SmemAttr attr[2][2][2][3];  // [S-1][DL-1][WB==8][mode]
  static SmemAttr attr_col[2][2][4];  // [S-1][DL-1][form]
  // The TMA forms run a layer whose taps read one stride phase on the
  // subsampled input (phase_subsample); the direct-load variant reads x
  // itself and keeps the layer as it is.
  Geometry gs;
  const bool can_sub = la.tile[6] != 2 && phase_subsample(g, &gs);
  if (!cache.get(key, &p)) {
    // tile[6]: 0 automatic (column form when the depth filter is 1),
    // 1 row-blocked form, 2 direct-load variant, 3 column form only.
    const int kind = la.tile[6];
    bool planned = false;
    for (int attempt = can_sub ? 0 : 1; attempt < 2 && !planned; ++attempt) {
      const Geometry& gq = attempt == 0 ? gs : g;
      if ((kind == 0 || kind == 3) && gq.Z == 1) {
        const int form = col_form(es, la.tile, gq.Cg);
        DwKernel<T> k = pick_col_kernel<T>(gq.sH, gq.dH, form);
        cudaFuncAttributes fa{};
        if (k == nullptr) return cudaErrorNotSupported;
        cudaError_t e = cudaFuncGetAttributes(&fa, k);
        if (e != cudaSuccess) return e;
        planned = make_col_plan(gq, es, la.tile, dev.num_sms, form, fa.numRegs, &p);
      }
      if (!planned && kind != 3 && gq.Cg == 1) planned = make_plan(gq, es, la.tile, dev.num_sms, &p);
      p.sub = attempt == 0 ? g.sH : 1;
    }
    if (!planned) return cudaErrorNotSupported;
    const Geometry& gq = p.sub > 1 ? gs : g;
    if (p.direct) {
      // one CTA per tile: the grid's x extent bounds the tile count
      if (p.sub > 1 || p.num_tiles >= ((int64_t)1 << 31) ||
          pick_ldg_kernel<T>(gq.sH, gq.dH, p.WB, p.mode) == nullptr)
        return cudaErrorNotSupported;
    } else {
      DwKernel<T> k = p.col ? pick_col_kernel<T>(gq.sH, gq.dH, p.mode) : pick_kernel<T>(gq.sH, gq.dH, p.WB, p.mode);
      if (k == nullptr || p.smem_bytes > (uint32_t)dev.max_smem_optin) return cudaErrorNotSupported;
      SmemAttr& at =
          p.col ? attr_col[gq.sH - 1][gq.dH - 1][p.mode] : attr[gq.sH - 1][gq.dH - 1][p.WB == 8][p.mode];
      cudaError_t e = at.ensure(k, dev.device, (int)p.smem_bytes);
      if (e != cudaSuccess) return e;
      int occ = 0;
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, p.threads, p.smem_bytes);
      if (e != cudaSuccess) return e;
      if (occ < 1) return cudaErrorNotSupported;
      p.ctas_per_sm = std::min(occ, p.ctas_per_sm);
    }
    cache.put(key, p);
  }
  const Geometry& gq = p.sub > 1 ? gs : g;
  if (p.direct) {
    DwArgs a{};
    a.x = la.x;
    a.D = gq.D, a.H = gq.H, a.W = gq.W;
    a.w = la.w;
    a.bias = la.bias;
    a.y = la.y;
    a.C = gq.C();
    a.Do = gq.Do, a.Ho = gq.Ho, a.Wo = gq.Wo;
    a.Z = gq.Z, a.dD = gq.dD, a.sD = gq.sD, a.pD = gq.pD, a.pH = gq.pH, a.pW = gq.pW;
    a.TH = p.TH, a.TW = p.TW, a.TC = p.TC;
    a.tiles_c = p.tiles_c, a.tiles_w = p.tiles_w, a.tiles_h = p.tiles_h;
    a.num_tiles = p.num_tiles;
    a.status = la.status;
    a.wait_limit_ns = la.wait_limit_ns;
    DwLdgKernel<T> k = pick_ldg_kernel<T>(gq.sH, gq.dH, p.WB, p.mode);
    return launch_kernel(k, dim3((unsigned)p.num_tiles), dim3(p.threads), p.smem_bytes, la, a);
  }

  // x viewed as a 5-D tensor (C, W, H, D, N), innermost first.
  CUtensorMap map;
  const uint64_t C = gq.C();
  uint64_t dims[5] = {C, (uint64_t)gq.W, (uint64_t)gq.H, (uint64_t)gq.D, (uint64_t)gq.N};
  // (subsampled input: rows and columns s apart in the dense tensor g)
  const uint64_t sub = (uint64_t)p.sub;
  uint64_t strides[4] = {C * es * sub, C * es * g.W * sub, C * es * g.W * g.H, C * es * g.W * g.H * g.D};
  const int h0 = p.col ? p.h0 : p.Hh;
  uint32_t box[5] = {(uint32_t)p.TC, (uint32_t)p.Wh, (uint32_t)p.Hh, (uint32_t)p.Dh, 1u};
  uint32_t estr[5] = {1, 1, 1, 1, 1};
  if (encode_tiled(&map, tma_type<T>(), 5, la.x, dims, strides, box, estr) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  // column form, a CTA's first tile in two copies: rows 0 .. h0-1, h0 .. Hh-1
  CUtensorMap map0 = map, map1 = map;
  if (h0 < p.Hh) {
    box[2] = (uint32_t)h0;
    if (encode_tiled(&map0, tma_type<T>(), 5, la.x, dims, strides, box, estr) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    box[2] = (uint32_t)(p.Hh - h0);
    if (encode_tiled(&map1, tma_type<T>(), 5, la.x, dims, strides, box, estr) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }

  DwArgs a{};
  a.x = la.x;
  a.D = gq.D, a.H = gq.H, a.W = gq.W;
  a.w = la.w;
  a.bias = la.bias;
  a.y = la.y;
  a.C = gq.C();
  a.Do = gq.Do, a.Ho = gq.Ho, a.Wo = gq.Wo;
  a.Z = gq.Z, a.dD = gq.dD, a.sD = gq.sD, a.pD = gq.pD, a.pH = gq.pH, a.pW = gq.pW;
  a.TH = p.TH, a.TW = p.TW, a.TC = p.TC;
  a.Dh = p.Dh, a.Hh = p.Hh, a.Wh = p.Wh;
  a.tiles_c = p.tiles_c, a.tiles_w = p.tiles_w, a.tiles_h = p.tiles_h;
  a.num_tiles = p.num_tiles;
  a.stages = p.stages;
  a.stage_bytes = p.stage_bytes;
  a.stage_stride = p.stage_stride;
  a.stage_off = p.stage_off;
  a.status = la.status;
  a.wait_limit_ns = la.wait_limit_ns;
  a.test_flags = la.test_flags;

  const int64_t grid64 = std::min<int64_t>(p.num_tiles, (int64_t)dev.num_sms * p.ctas_per_sm);
  const int grid = (int)std::max<int64_t>(1, grid64);
  DwKernel<T> kern = p.col ? pick_col_kernel<T>(gq.sH, gq.dH, p.mode) : pick_kernel<T>(gq.sH, gq.dH, p.WB, p.mode);
  a.h0 = h0;
  a.bytes0 = (uint32_t)h0 * p.Wh * p.TC * p.Dh * es;
  return launch_kernel(kern, dim3(grid), dim3(p.threads), p.smem_bytes, la, map, map0, map1, a);
}

}  // namespace dw
}  // namespace gconv
