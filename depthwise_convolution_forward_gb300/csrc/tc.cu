// Kb host side: support check, tile planning, tensor-map encoding, launch.
#include <algorithm>
#include <cmath>
#include <cstring>

#include "kernels.h"
#include "plan_cache.h"
#include "tc_impl.cuh"

namespace gconv {
namespace {

using tc::TcArgs;

inline int mod_pos(int v, int m) { return ((v % m) + m) % m; }
inline uint32_t round_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

// Smallest merge factor m (groups per MMA) with K = m*Cg and N = m*Kg both
// multiples of 16 (tcgen05 kind::f16 with M = 128 wants N % 16 == 0 and each
// MMA consumes K = 16), or 0 if none within 16 groups.
int merge_factor(const Geometry& g) {
  for (int m = 1; m <= 16; ++m) {
    if (g.G % m) continue;
    if ((m * g.Cg) % 16 == 0 && (m * g.Kg) % 16 == 0 && m * g.Kg <= 256 && m * g.Cg <= 256) return m;
  }
  return 0;
}

struct TcPlan {
  TcArgs a;  // everything except pointers / status
  bool sw;   // 128-byte swizzled rows of 64 channels (else 16-byte chunk planes)
  uint32_t smem_bytes;
  int grid;
  bool ok;
};

// aligned: (128-byte rows only) one copy of the tile per stride phase and
// column shift cx of the taps, each copy shifted left by cx and laid out
// with a pitch rounded up to 8 pixels, so every tap's A operand starts on
// an 8-row boundary.  MMAs whose A start is not a multiple of 8 rows
// measured about 57 cycles against 39-48 aligned (M = 128, N <= 64) on
// GB300; the copies cost shared memory (up to 3x the input tile).
bool make_tc_plan_mode(const Geometry& g, bool bf16, int num_sms, int max_smem, const int* ov, bool allow_sw,
                       bool aligned, TcPlan* out, double* cost_out) {
  TcArgs a;
  std::memset(&a, 0, sizeof(a));
  const int m = merge_factor(g);
  if (m == 0) return false;
  if (g.sH != g.sW || g.sH < 1 || g.sH > 2) return false;
  const int taps = g.taps();
  if (taps > tc::kMaxTaps) return false;
  a.G = g.G, a.Cg = g.Cg, a.Kg = g.Kg, a.m = m;
  a.Do = g.Do, a.Ho = g.Ho, a.Wo = g.Wo, a.Ktot = g.K();
  a.sD = g.sD, a.pD = g.pD, a.taps_total = taps;
  a.s = g.sH;
  a.Kt = m * g.Cg, a.Nn = m * g.Kg, a.KS = a.Kt / 16, a.nchunks = a.Kt / 8;
  a.n_gc = g.G / m;
  // 128-byte rows: 64 input channels per pixel cover sc = 64 / Kt group
  // chunks, read by one TMA box per phase (override 6: 1 = chunk planes).
  const bool sw = allow_sw && g.C() % 64 == 0 && 64 % a.Kt == 0 && a.n_gc % (64 / a.Kt) == 0 && !(ov && ov[6] == 1);
  a.sc = sw ? 64 / a.Kt : 1;
  if (sw) a.nchunks = 1;
  if (aligned && !sw) return false;
  a.ntaps = taps;
  a.Dh = (g.Z - 1) * g.dD + 1;
  // Phase decomposition: input row of tap ky for output row oh is
  // s*(oh + qy) + py with py in [0, s).
  int qy[16], py[16], qx[16], px[16];
  if (g.Y > 16 || g.X > 16) return false;
  int qy_min = 1 << 30, qy_max = -(1 << 30), qx_min = 1 << 30, qx_max = -(1 << 30);
  for (int ky = 0; ky < g.Y; ++ky) {
    const int v = ky * g.dH - g.pH;
    py[ky] = mod_pos(v, a.s);
    qy[ky] = (v - py[ky]) / a.s;
    qy_min = std::min(qy_min, qy[ky]);
    qy_max = std::max(qy_max, qy[ky]);
  }
  for (int kx = 0; kx < g.X; ++kx) {
    const int v = kx * g.dW - g.pW;
    px[kx] = mod_pos(v, a.s);
    qx[kx] = (v - px[kx]) / a.s;
    qx_min = std::min(qx_min, qx[kx]);
    qx_max = std::max(qx_max, qx[kx]);
  }
  a.qy_min = qy_min, a.qx_min = qx_min;
  // used planes: one per stride phase (py, px), and in aligned mode one per
  // (phase, column shift cx = qx - qx_min); plane_of[ky][kx]
  int plane_of[16][16];
  a.nphase = 0;
  for (int ky = 0; ky < g.Y; ++ky)
    for (int kx = 0; kx < g.X; ++kx) {
      const int cx = aligned ? qx[kx] - qx_min : 0;
      int pl = -1;
      for (int q = 0; q < a.nphase; ++q)
        if (a.phase_py[q] == py[ky] && a.phase_px[q] == px[kx] && a.plane_cx[q] == cx) pl = q;
      if (pl < 0) {
        if (a.nphase == tc::kMaxPhases) return false;
        pl = a.nphase++;
        a.phase_py[pl] = py[ky], a.phase_px[pl] = px[kx], a.plane_cx[pl] = cx;
      }
      plane_of[ky][kx] = pl;
    }
  const int range_x = aligned ? 0 : qx_max - qx_min, range_y = qy_max - qy_min;
  const uint32_t budget = (uint32_t)std::min(max_smem, 227 * 1024);
  // Tile shape: full output rows when they fit, TH rows so the flattened
  // M = TH * pitch fills nmt MMAs of 128 rows.  Every candidate nmt is
  // planned completely; the cheapest one that fits shared and tensor memory
  // wins (cost = MMA rows issued + a per-tile overhead).
  const int tw_cap = std::min(256 / a.s, 128 * 4) - range_x;
  if (tw_cap < 1) return false;
  double best = 1e30;
  TcPlan bestp;
  std::memset(&bestp, 0, sizeof(bestp));
  // Candidates: nmt M tiles per CTA tile x np partial accumulators.
  for (int combo = 0; combo < 12; ++combo) {
    const int nmt = combo / 3 + 1, np_cand = 1 << (combo % 3);
    if (ov && ov[2] && ov[2] != nmt) continue;
    TcArgs c = a;
    int TWo = std::min(g.Wo, std::min(tw_cap, 128 * nmt - range_x));
    if (aligned) TWo = std::min(TWo, (std::min(256 / a.s, 128 * nmt) / 8) * 8);  // pitch round_up(TWo, 8) fits
    if (TWo < 1) continue;
    const int P = aligned ? (int)round_up((uint32_t)TWo, 8) : TWo + range_x;
    int TH = std::min(g.Ho, (128 * nmt) / P);
    if (ov && ov[0]) TH = std::min(ov[0], (128 * nmt) / P);
    if (TH < 1) continue;
    if (a.s * (TH + range_y) > 256) continue;
    c.TH = TH, c.TWo = TWo, c.nmt = nmt, c.P = P, c.Hh = TH + range_y;
    c.tiles_w = (g.Wo + TWo - 1) / TWo;
    c.tiles_h = (g.Ho + TH - 1) / TH;
    const double sp = (double)g.N * g.Do * c.tiles_h * c.tiles_w;
    if (sp >= 2e9) continue;
    c.spatial_tiles = (int)sp;
    int max_off = 0;
    for (int z = 0; z < g.Z; ++z)
      for (int ky = 0; ky < g.Y; ++ky)
        for (int kx = 0; kx < g.X; ++kx) {
          const int t = (z * g.Y + ky) * g.X + kx;
          c.tap_phase[t] = plane_of[ky][kx];
          c.tap_off[t] = z * g.dD * c.Hh * c.P + (qy[ky] - qy_min) * c.P + (aligned ? 0 : qx[kx] - qx_min);
          max_off = std::max(max_off, c.tap_off[t]);
        }
    // Row shift (shift <= 0): accumulator row f of a tile holds flattened
    // output f + shift, so tap t's A operand starts at plane row mt * 128 +
    // shift + tap_off[t].  An MMA whose A starts on an 8-row boundary costs
    // about 39 cycles on GB300 against 57 off it (M = 128, N <= 64), so the
    // shift that puts the most taps on that boundary is taken, while the
    // tile's TH * P outputs still fit its nmt * 128 rows.  The rows before
    // the first output read whatever precedes the plane in shared memory and
    // are never stored.
    {
      int best = -1;
      c.shift = 0;
      for (int sh = 0; sh > -8; --sh) {
        if (c.TH * c.P - sh > nmt * 128) break;
        int cnt = 0;
        for (int t = 0; t < taps; ++t) cnt += ((c.tap_off[t] + sh) & 7) == 0;
        if (cnt > best) best = cnt, c.shift = sh;
      }
    }
    const uint32_t plane_px = round_up((uint32_t)std::max(c.Dh * c.Hh * c.P, c.nmt * 128 + max_off), 8);
    const uint32_t row_bytes = sw ? 128u : 16u;
    c.plane_stride = plane_px * row_bytes;
    c.a_stage_bytes = round_up((uint32_t)(c.nphase * c.nchunks) * c.plane_stride, 1024);
    c.tx_bytes = (uint32_t)(c.nphase * c.nchunks) * (uint32_t)(c.Dh * c.Hh * c.P) * row_bytes;
    const uint32_t b_bytes = round_up((uint32_t)(c.sc * taps * c.Kt * c.Nn * 2), 1024);
    // Partial accumulators (taps split np ways, summed by the epilogue): the
    // smallest count that gives the tile kIssuers independent units of MMA
    // work, within 512 TMEM columns.  More partials only add tensor-memory
    // reads to the epilogue: on GB300 they measured 2-5% slower on the
    // stride-1 sweeps and ResNeXt (a).  An explicit count (override slot 4)
    // replaces it (issuers without a unit then only commit).
    const int G2 = c.sc * c.nmt;
    int np = 1;
    while (np * 2 <= tc::kIssuers && G2 * np < tc::kIssuers && np * 2 <= taps &&
           2 * (np * 2) * G2 * c.Nn <= 512)
      np *= 2;
    if (ov && ov[4]) {
      if (np_cand != 1 || ov[4] < 1 || ov[4] > taps) continue;
      np = ov[4];
    } else {
      if (np_cand != np) continue;
    }
    c.np = np;
    // per-issuer MMA lists: 32 bytes per entry
    uint32_t entries = 0;
    {
      const int units = G2 * np, steps = ((taps + np - 1) / np) * c.KS;
      for (int w = 0; w < tc::kIssuers; ++w)
        entries += (uint32_t)(steps * (units > w ? (units - w + tc::kIssuers - 1) / tc::kIssuers : 0));
    }
    c.bias_off = 1024;
    c.tab_off = round_up(c.bias_off + (uint32_t)(c.sc * c.Nn) * 4u, 16);
    const uint32_t tab_bytes = entries * 32u;
    c.b_off = round_up(c.tab_off + tab_bytes, 1024);
    c.a_off = c.b_off + b_bytes;
    c.ntab = 0;
    if (entries <= (uint32_t)tc::kMaxTab) {
      // The same lists the kernel would build, with shared-memory offsets
      // instead of descriptors (the kernel adds its shared-memory base).
      const int units = G2 * np, steps = ((taps + np - 1) / np) * c.KS;
      const uint32_t slab = (uint32_t)c.Nn * 16u;  // one (chunk, K step, K half, tap) slab of B
      int base = 0;
      for (int w = 0; w < tc::kIssuers; ++w) {
        const int nu = units > w ? (units - w + tc::kIssuers - 1) / tc::kIssuers : 0;
        for (int i = 0; i < steps * nu; ++i) {
          const int st = i / nu, ui = i - st * nu;
          const int u = w + tc::kIssuers * ui;
          const int grp = u / np, pp = u - grp * np;
          const int t = pp + np * (st / c.KS), ks = st % c.KS;
          const int mt = grp / c.sc, j = grp - mt * c.sc;
          uint2 e = make_uint2(0u, 2u << 16);  // skip
          if (t < taps) {
            uint32_t aoff;
            if (sw)
              aoff = c.a_off + (uint32_t)c.tap_phase[t] * c.plane_stride + (uint32_t)(mt * 128 + c.shift + c.tap_off[t]) * 128u +
                     (uint32_t)(j * c.Kt * 2 + ks * 32);
            else
              aoff = c.a_off + (uint32_t)(c.tap_phase[t] * c.nchunks + 2 * ks) * c.plane_stride +
                     (uint32_t)(mt * 128 + c.shift + c.tap_off[t]) * 16u;
            const uint32_t boff = c.b_off + (uint32_t)((j * c.KS + ks) * 2 * taps + t) * slab;
            e = make_uint2((aoff >> 4) | ((boff >> 4) << 16),
                           (uint32_t)((pp * G2 + grp) * c.Nn) | ((st == 0 ? 0u : 1u) << 16));
          }
          c.tab[base + i] = e;
        }
        base += steps * nu;
      }
      c.ntab = (int)entries;
    }
    // Epilogue: stores straight from registers by default.  On request
    // (override 7 < 0) the tile's output box is staged in shared memory and
    // written with TMA tensor stores, one per channel slice of W bytes per
    // pixel (the CTA's sc * Nn channels, at most 128 bytes per slice), when
    // the staging fits beside two input stages.  The TMA-store epilogue
    // measured no faster on GB300 (within -5..+2% on the tensor-core
    // workloads): the scattered 32-byte stores are not what bounds a tile.
    const uint32_t chan_bytes = (uint32_t)(c.sc * c.Nn) * 2u;
    c.epi_w = (int)std::min<uint32_t>(128u, chan_bytes);
    c.epi_slices = (int)(chan_bytes / (uint32_t)c.epi_w);
    c.epi_slice_bytes = round_up((uint32_t)(c.TH * c.TWo) * (uint32_t)c.epi_w, 1024);
    const uint32_t epi_bytes = (uint32_t)c.epi_slices * c.epi_slice_bytes;
    const bool want_epi = ov && ov[7] < 0;
    // At stride 1, three stages of 128-byte-row planes by default: a fourth,
    // requested at launch with every CTA's first copies, measured 1.5% slower
    // on ResNeXt (a).  At stride 2 the fourth measured 2-5% faster.
    int stages = (ov && ov[3]) ? ov[3] : ((sw && a.s == 1) ? 3 : tc::kMaxStages);
    stages = std::min(stages, tc::kMaxStages);
    auto a_end_of = [&](int st) { return c.a_off + (uint32_t)st * c.a_stage_bytes; };
    bool epi = want_epi && a_end_of(2) + epi_bytes <= budget;
    while (stages > 2 && a_end_of(stages) + (epi ? epi_bytes : 0u) > budget) --stages;
    if (a_end_of(stages) > budget) continue;
    c.stages = stages;
    c.epi_off = epi ? a_end_of(stages) : 0u;
    // Accumulator buffers: as many as 512 tensor-memory columns hold (at
    // most kMaxAccBufs, at least 2), or at most override slot 1.  With two
    // buffers the MMAs of tile k wait for the epilogue of tile k - 2, which
    // itself waited for the MMAs of tile k - 2 to complete.
    const uint32_t per_buf = (uint32_t)(np * G2 * c.Nn);
    int nbuf = (int)std::min<uint32_t>((uint32_t)tc::kMaxAccBufs, 512u / per_buf);
    if (ov && ov[1]) nbuf = std::min(nbuf, ov[1]);
    if (nbuf < 2) continue;
    c.nbuf = nbuf;
    uint32_t cols = 32;
    while (cols < (uint32_t)nbuf * per_buf) cols <<= 1;
    if (cols > 512) continue;
    c.tmem_cols = cols;
    c.idesc = tc::idesc_f16(bf16, 128, c.Nn);
    // A CTA keeps one group chunk (its weights stay resident); the chunk's
    // spatial tiles are dealt round-robin to cpg CTAs.
    const int n_sc = c.n_gc / c.sc;
    c.cpg = std::max(1, num_sms / n_sc);
    TcPlan p;
    p.a = c;
    p.sw = sw;
    p.smem_bytes = c.a_off + stages * c.a_stage_bytes + (c.epi_off ? epi_bytes : 0u);
    // Keep a second CTA off the SM when both could not hold their tensor
    // memory at once (its allocation would wait for the first CTA to exit).
    if (cols > 256) p.smem_bytes = std::max<uint32_t>(p.smem_bytes, 117 * 1024);
    if (ov && ov[7] > 0) p.smem_bytes += (uint32_t)ov[7] * 1024u;  // allocation padding (layout checks)
    if (p.smem_bytes > budget) continue;
    p.grid = n_sc * c.cpg;
    p.ok = true;
    // Cost, in MMA rows of the busiest CTA of a group chunk (a CTA walks
    // whole tiles: with fewer tiles than CTAs, as in a batch-1 3D layer, the
    // time is one tile's): the rows of its tiles, plus about 1.2 tiles of
    // fill (the first copy and MMAs) and drain (the last epilogue) that no
    // other tile overlaps, plus 96 rows of fixed work per tile, all scaled
    // up when the tile has fewer units of MMA work than issuers.  Fitted to
    // tile and tap-split sweeps of ten tensor-core workloads on GB300: it
    // picks the fastest measured plan on seven and one within 3% on the
    // other three.
    const int units = G2 * np;
    const double per_cta = std::ceil((double)c.spatial_tiles / c.cpg);
    const double idle = units < tc::kIssuers ? (double)tc::kIssuers / units : 1.0;
    const double cost = ((per_cta + 1.2) * nmt * 128 + per_cta * 96) * idle;
    if (cost < best) best = cost, bestp = p;
  }
  if (best >= 1e30) return false;
  *out = bestp;
  if (cost_out) *cost_out = best;
  return true;
}

// Override slot 5: 2 = aligned copies (1 or 0 = shifted starts, the
// default).  The copies measured slower on every configuration tried on
// GB300 (ResNeXt (a) 26.7 against 23.9 us, sweep G=64 d1 s1 46.6 against
// 45.0 us): they fit only one M tile and two stages per CTA, which costs
// more than the faster MMAs save.
bool make_tc_plan(const Geometry& g, bool bf16, int num_sms, int max_smem, const int* ov, TcPlan* out) {
  const int mode = ov && ov[5] == 2 ? 2 : 1;
  TcPlan pa, pu;
  double ca = 1e30, cu = 1e30;
  const bool ok_a = mode == 2 && make_tc_plan_mode(g, bf16, num_sms, max_smem, ov, true, true, &pa, &ca);
  const bool ok_u = mode != 2 && make_tc_plan_mode(g, bf16, num_sms, max_smem, ov, true, false, &pu, &cu);
  if (ok_a || ok_u) {
    *out = (ok_a && ca <= cu) ? pa : pu;
    return true;
  }
  return mode != 2 && make_tc_plan_mode(g, bf16, num_sms, max_smem, ov, false, false, out, nullptr);
}

template <typename T>
using TcKernel = void (*)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const TcArgs);

template <typename T>
TcKernel<T> pick_tc_kernel(const TcPlan& p) {
  if (p.a.epi_off != 0) return p.sw ? tc::tc_kernel<T, true, true> : tc::tc_kernel<T, false, true>;
  return p.sw ? tc::tc_kernel<T, true, false> : tc::tc_kernel<T, false, false>;
}

template <typename T>
cudaError_t tc_launch_typed(const Geometry& g, const LaunchArgs& la, const DeviceInfo& dev) {
  struct Key {
    Geometry g;
    int tile[8];
    int num_sms, device, bf16;
  } key;
  std::memset(&key, 0, sizeof(key));
  key.g = g;
  std::memcpy(key.tile, la.tile, sizeof(key.tile));
  key.num_sms = dev.num_sms;
  key.device = dev.device;
  key.bf16 = std::is_same<T, __nv_bfloat16>::value;
  static PlanCache<TcPlan> cache;
  static SmemAttr attr[2][2];  // [swizzled rows][staged epilogue]
  TcPlan p;
  if (!cache.get(key, &p)) {
    if (!make_tc_plan(g, key.bf16, dev.num_sms, dev.max_smem_optin, la.tile, &p)) return cudaErrorNotSupported;
    const TcKernel<T> kern = pick_tc_kernel<T>(p);
    cudaError_t e = attr[p.sw][p.a.epi_off != 0].ensure(kern, dev.device, (int)p.smem_bytes);
    if (e != cudaSuccess) return e;
    // Co-resident CTAs must never need more than the SM's 512 TMEM columns,
    // or an allocation would wait for another CTA to exit.  Raise the
    // shared-memory request until occupancy x columns fits.
    for (int guard = 0; guard < 64; ++guard) {
      int occ = 0;
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, tc::kThreads, p.smem_bytes);
      if (e != cudaSuccess) return e;
      if (occ < 1) return cudaErrorNotSupported;
      if ((uint32_t)occ * p.a.tmem_cols <= 512u) break;
      p.smem_bytes += 8 * 1024;
      if (p.smem_bytes > (uint32_t)dev.max_smem_optin) return cudaErrorNotSupported;
      e = attr[p.sw][p.a.epi_off != 0].ensure(kern, dev.device, (int)p.smem_bytes);
      if (e != cudaSuccess) return e;
    }
    cache.put(key, p);
  }
  const int es = (int)sizeof(T);
  const uint64_t C = g.C();
  CUtensorMap map;
  uint64_t dims[5] = {C, (uint64_t)g.W, (uint64_t)g.H, (uint64_t)g.D, (uint64_t)g.N};
  uint64_t strides[4] = {C * es, C * es * g.W, C * es * g.W * g.H, C * es * g.W * g.H * g.D};
  const int s = p.a.s;
  uint32_t box[5] = {p.sw ? 64u : 8u, (uint32_t)(s * p.a.P), (uint32_t)(s * p.a.Hh), (uint32_t)p.a.Dh, 1u};
  uint32_t estr[5] = {1u, (uint32_t)s, (uint32_t)s, 1u, 1u};
  CUtensorMapDataType tt = std::is_same<T, __half>::value ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                          : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (encode_tiled(&map, tt, 5, la.x, dims, strides, box, estr,
                   p.sw ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  // Weights viewed as (Cg, G*Kg, taps) -- channels innermost, then output
  // channel rows, then taps -- for TMA staging of the block-diagonal B: a box
  // of 8 channels x Kg rows x (all taps when one group fills a chunk, else 1
  // tap) lands as [tap][row][8], the tap-major order of B's slabs.  Otherwise
  // the threads copy them.
  CUtensorMap wmap = map;
  int w_tma = 0;
  const uint64_t taps = (uint64_t)g.taps();
  const int box_taps = (p.a.m == 1 && taps <= 256) ? (int)taps : 1;
  if (g.Cg % 8 == 0 && g.Kg % 8 == 0 && (reinterpret_cast<uintptr_t>(la.w) & 15) == 0) {
    uint64_t wdims[3] = {(uint64_t)g.Cg, (uint64_t)g.K(), taps};
    uint64_t wstrides[2] = {taps * g.Cg * es, (uint64_t)g.Cg * es};
    uint32_t wbox[3] = {8u, (uint32_t)g.Kg, (uint32_t)box_taps};
    uint32_t westr[3] = {1u, 1u, 1u};
    if (encode_tiled(&wmap, tt, 3, la.w, wdims, wstrides, wbox, westr) == CUDA_SUCCESS) w_tma = 1;
  }
  // Output viewed as (K, Wo, Ho, Do, N) for the staged epilogue's TMA
  // stores: a box of one channel slice x TWo x TH of the tile.
  CUtensorMap ymap = map;
  if (p.a.epi_off != 0) {
    uint64_t ydims[5] = {(uint64_t)g.K(), (uint64_t)g.Wo, (uint64_t)g.Ho, (uint64_t)g.Do, (uint64_t)g.N};
    const uint64_t K = g.K();
    uint64_t ystrides[4] = {K * es, K * es * g.Wo, K * es * g.Wo * g.Ho, K * es * g.Wo * g.Ho * g.Do};
    uint32_t ybox[5] = {(uint32_t)(p.a.epi_w / es), (uint32_t)p.a.TWo, (uint32_t)p.a.TH, 1u, 1u};
    uint32_t yestr[5] = {1u, 1u, 1u, 1u, 1u};
    const CUtensorMapSwizzle ysw = p.a.epi_w == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                   : p.a.epi_w == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                      : CU_TENSOR_MAP_SWIZZLE_32B;
    if (encode_tiled(&ymap, tt, 5, la.y, ydims, ystrides, ybox, yestr, ysw) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  if (la.omap.on && p.a.epi_off != 0) return cudaErrorNotSupported;  // the TMA-store epilogue has no map
  // the stacked epilogue reads one partial and stores 16-channel runs of one phase
  if (la.omap.on == 2 && (p.a.np != 1 || la.omap.cpp % 16 != 0)) return cudaErrorNotSupported;
  TcArgs a = p.a;
  a.om = la.omap;
  a.w_tma = w_tma;
  a.w_box_taps = box_taps;
  a.w = la.w;
  a.bias = la.bias;
  a.y = la.y;
  a.status = la.status;
  a.wait_limit_ns = la.wait_limit_ns;
  a.test_flags = la.test_flags;
  const TcKernel<T> kern = pick_tc_kernel<T>(p);
  return launch_kernel(kern, dim3(p.grid), dim3(tc::kThreads), p.smem_bytes, la, map, wmap, ymap, a);
}

}  // namespace

bool tc_supported(const Geometry& g, DType dt, const LaunchArgs* a, int num_sms, int max_smem) {
  if (dt == kF32) return false;  // fp32 stays on FFMA (no TF32 rounding)
  if (merge_factor(g) == 0) return false;
  if (g.sH != g.sW || g.sH < 1 || g.sH > 2) return false;
  if (g.taps() > tc::kMaxTaps || g.Y > 16 || g.X > 16) return false;
  if (g.C() % 8 || g.K() % 8) return false;
  if ((g.Z - 1) * g.dD + 1 > 256) return false;
  if (a) {
    if ((reinterpret_cast<uintptr_t>(a->x) & 15) || (reinterpret_cast<uintptr_t>(a->y) & 15)) return false;
  }
  struct Key {
    Geometry g;
    int tile[8];
    int bf16, num_sms, max_smem;
  } key;
  std::memset(&key, 0, sizeof(key));
  key.g = g;
  if (a) std::memcpy(key.tile, a->tile, sizeof(key.tile));
  key.bf16 = dt == kBF16;
  key.num_sms = num_sms;
  key.max_smem = max_smem;
  static PlanCache<int> cache;
  int ok = 0;
  if (cache.get(key, &ok)) return ok != 0;
  TcPlan p;
  // the same planner, SM count and shared-memory limit as tc_launch_typed
  ok = make_tc_plan(g, dt == kBF16, num_sms, max_smem, a ? a->tile : nullptr, &p) ? 1 : 0;
  cache.put(key, ok);
  return ok != 0;
}

cudaError_t tc_launch(const Geometry& g, const LaunchArgs& a, const DeviceInfo& dev) {
  if (a.dt == kF16) return tc_launch_typed<__half>(g, a, dev);
  if (a.dt == kBF16) return tc_launch_typed<__nv_bfloat16>(g, a, dev);
  return cudaErrorNotSupported;
}

}  // namespace gconv
