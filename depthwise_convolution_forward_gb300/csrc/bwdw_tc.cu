// Grouped convolution backward weight on the 5th-generation tensor cores.
//
//   dw[g, k, z, yy, xx, c] = sum over (n, od, oh, ow) of dy[n, od, oh, ow, g, k]
//       * x[n, od*sD - pD + z*dD, oh*s - pH + yy*dH, ow*s - pW + xx*dW, g, c]
//
// The backward-weight variant (runner taking X and dY, partials reduced in
// two stages through an fp32 workspace) is the one the pages' CK
// grouped-convolution tile engine lists ("Grouped Convolution -- Python
// Examples", Examples and Config-options harness, two_stage).
//
// For a 64-channel chunk j of the channels (Cg == Kg, so the chunk holds the
// same groups in x and dy) and one filter row r = (z, yy), the sum is a GEMM
// over output pixels p:
//     D[k, (xx, c)] += dy[p, k] * x_shift(r, xx)[p, c]
// with k and c over the chunk's 64 channels.  Only the blocks where k and c
// belong to the same group are dw; the rest of D is computed and dropped
// (dense 64 x 64 blocks cost the tensor core the same for any group size).
//
// sm_103a design:
//  * A CTA owns (chunk j, filter row r, pixel split s) and walks the split's
//    tiles of TH full output rows.  Warp 0 copies each tile with TMA into a
//    shared-memory stage: dy as [TH * P pixels][64 channels] with the
//    128-byte swizzle (row pitch P, columns past Wo read as zeros beyond the
//    tensor's edge), and, for each stride phase px the row's taps use, the x
//    pixels s*(u + qx_min) + px of the TH input rows of filter row r, same
//    pitch.  A tap xx is then the x plane read from row offset u0(xx): the
//    same shift trick as the forward kernel, here along the contraction.
//  * Both operands are MN-major (channels contiguous, pixels along K): the
//    instruction descriptor's transpose bits.  The taps xx of the filter row
//    that share a phase and a constant offset step form one MMA with
//    N = 64 * taps, its 64-column blocks one offset step apart (the
//    descriptor's leading byte offset = step * 128 bytes): one MMA
//    (M = 64, K = 16 pixels) per K step covers a whole 3-tap row at stride 1.
//  * Warps 1-2 issue (one lane each), alternate K steps into two
//    accumulator sets in tensor memory; warps 3-6 add the two sets at the end
//    and write the group-diagonal blocks, in fp32, to the caller's workspace
//    [split][dw element].  The reduction kernel of the FFMA path adds the
//    splits in a fixed order and rounds once.
//  * All waits are bounded; on expiry a role reports a timeout and stops.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "plan_cache.h"
#include "tc_ptx.cuh"

namespace gconv {
namespace bwt {

constexpr int kMaxStages = 4;
constexpr int kIssuers = 2;
constexpr int kThreads = 32 * (1 + kIssuers + 4);  // producer, issuers, epilogue
constexpr int kMaxRuns = 4;
constexpr int kMaxX = 4;        // taps per filter row (N = 64 * taps <= 256)
constexpr int kMaxRows = 64;    // filter rows Z * Y

struct BwtArgs {
  float* ws;              // [S][E] fp32 partials
  int G, Cg, C;           // groups, channels per group (== Kg), channels
  int Ho, Wo, Do;         // output extents
  int D, X, Y, taps;      // input depth, filter width / height, taps per filter
  int sD, pD, dD;         // depth stride / pad / dilation
  int P, TH, Kp;          // pitch, output rows per tile, K rows per tile (multiple of 16)
  int tiles_h;            // tiles per output image plane (n, od)
  int64_t tiles;          // tiles in total
  int S;                  // pixel splits
  int rows, chunks;       // filter rows Z * Y, 64-channel chunks
  int stages;
  int nplane;             // x planes per stage (stride phases of the row's taps)
  int nruns;              // MMAs per K step
  int run_len[kMaxRuns];  // taps per MMA
  int run_u0[kMaxRuns];   // x-plane row offset of the run's first tap
  int run_du[kMaxRuns];   // row offset step between its taps
  int run_plane[kMaxRuns];
  int run_kx[kMaxRuns][kMaxX];
  uint32_t run_idesc[kMaxRuns];
  int plane_px[2];        // phase column of each x plane
  int qx_min;             // plane column u holds x column s * (u + qx_min) + px
  int s;                  // spatial stride (H and W)
  int row_qy[kMaxRows], row_py[kMaxRows], row_kz[kMaxRows], row_ky[kMaxRows];
  uint32_t dy_bytes, plane_bytes, stage_bytes, tx_bytes;
  uint32_t ncols, tmem_cols;  // accumulator columns per issuer (64 * X), allocation
  int64_t E;                  // dw elements
  int* status;
  uint64_t wait_limit_ns;
};

__device__ __forceinline__ uint64_t desc_mn_sw128(uint32_t saddr, uint32_t lbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;     // MN-major: stride between 64-element MN blocks
  d |= (uint64_t)((1024u >> 4) & 0x3FFFu) << 32;   // stride between 8-row K groups
  d |= (uint64_t)1u << 46;                         // fixed descriptor version bits
  d |= (uint64_t)2u << 61;                         // 128-byte swizzle
  return d;
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1) bwt_kernel(const __grid_constant__ CUtensorMap xmap,
                                                         const __grid_constant__ CUtensorMap dymap,
                                                         const __grid_constant__ BwtArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* a_full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* a_empty = a_full + kMaxStages;
  uint64_t* mma_done = a_empty + kMaxStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 256);
  uint8_t* stages = smem + 1024;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // block -> (split, chunk, filter row), filter row fastest: the CTAs of the
  // rows of one (split, chunk) read the same dy and overlapping x from L2
  const int r = blockIdx.x % a.rows;
  const int j = (blockIdx.x / a.rows) % a.chunks;
  const int split = blockIdx.x / (a.rows * a.chunks);
  const int64_t t0 = a.tiles * split / a.S, t1 = a.tiles * (split + 1) / a.S;
  const int c0 = j * 64;

  // zero every stage once: rows the copies never write (K padding, the x
  // rows past the tile) must read as finite zeros
  for (uint32_t i = tid; i < (uint32_t)a.stages * a.stage_bytes / 16u; i += kThreads)
    reinterpret_cast<uint4*>(stages)[i] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  if (tid == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(&a_full[s], 1);
      mbar_init(&a_empty[s], kIssuers);
    }
    mbar_init(mma_done, kIssuers);
    fence_mbar_init();
    tma_prefetch_desc(&xmap);
    tma_prefetch_desc(&dymap);
  }
  // x, dy and the workspace from here on.  Tensor memory is allocated only
  // after this wait, so a CTA holding it never waits on another grid.
  grid_dependency_wait();
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, a.tmem_cols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      const int qy = a.row_qy[r], py = a.row_py[r], kz = a.row_kz[r];
      int k = 0;
      for (int64_t t = t0; t < t1; ++t, ++k) {
        const int s = k % a.stages;
        if (k >= a.stages && !mbar_wait(&a_empty[s], (uint32_t)(((k / a.stages) - 1) & 1), a.wait_limit_ns)) {
          report(a.status, kDevTimeout, 21);
          break;
        }
        const int th = (int)(t % a.tiles_h);
        const int64_t img = t / a.tiles_h;
        const int od = (int)(img % a.Do), n = (int)(img / a.Do);
        const int oh0 = th * a.TH;
        const int id = od * a.sD - a.pD + kz * a.dD;
        uint8_t* st = stages + (size_t)s * a.stage_bytes;
        mbar_arrive_expect_tx(&a_full[s], a.tx_bytes);
        tma_load_5d(st, &dymap, &a_full[s], c0, 0, oh0, od, n);
        for (int pl = 0; pl < a.nplane; ++pl)
          tma_load_5d(st + a.dy_bytes + (size_t)pl * a.plane_bytes, &xmap, &a_full[s], c0,
                      a.s * a.qx_min + a.plane_px[pl], a.s * (oh0 + qy) + py, id, n);
      }
      // bounded drain: no copy may still be landing when the CTA exits
      for (int i = k > a.stages ? k - a.stages : 0; i < k; ++i)
        mbar_wait(&a_full[i % a.stages], (uint32_t)((i / a.stages) & 1), a.wait_limit_ns);
    }
  } else if (warp <= kIssuers) {
    // ---------------- MMA issuers: K steps w, w + 2, ... of every tile ----------------
    if (lane == 0) {
      const int w = warp - 1;
      const uint32_t dbase = tmem_base + (uint32_t)w * a.ncols;
      const uint32_t sbase = smem_u32(stages);
      const int ksteps = a.Kp / 16;
      bool first = true;
      int k = 0;
      for (int64_t t = t0; t < t1; ++t, ++k) {
        const int s = k % a.stages;
        if (!mbar_wait(&a_full[s], (uint32_t)((k / a.stages) & 1), a.wait_limit_ns)) {
          report(a.status, kDevTimeout, 22);
          break;
        }
        tc::fence_after_sync();
        const uint32_t st = sbase + (uint32_t)s * a.stage_bytes;
        for (int ks = w; ks < ksteps; ks += kIssuers) {
          const uint64_t adesc = desc_mn_sw128(st + (uint32_t)ks * 16u * 128u, 0u);
          uint32_t col = 0;
          for (int q = 0; q < a.nruns; ++q) {
            const uint32_t brow = (uint32_t)(ks * 16 + a.run_u0[q]);
            const uint64_t bdesc =
                desc_mn_sw128(st + a.dy_bytes + (uint32_t)a.run_plane[q] * a.plane_bytes + brow * 128u,
                              (uint32_t)a.run_du[q] * 128u);
            tc::mma_f16(dbase + col, adesc, bdesc, a.run_idesc[q], first ? 0u : 1u);
            col += 64u * (uint32_t)a.run_len[q];
          }
          first = false;
        }
        tc::commit(&a_empty[s]);  // this issuer's reads of the stage are done
      }
      tc::commit(mma_done);
    }
  } else {
    // ---------------- epilogue: warps 3..6, TMEM lane quarter q ----------------
    const int q = warp & 3;
    bool ok = true;
    if (lane == 0) ok = mbar_wait(mma_done, 0, a.wait_limit_ns);
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    if (ok && lane != 0) ok = mbar_wait(mma_done, 0, a.wait_limit_ns);
    if (!__all_sync(0xffffffffu, ok)) {
      if (lane == 0) report(a.status, kDevTimeout, 23);
    } else {
      tc::fence_after_sync();
      // An M = 64 accumulator keeps row m in lane 32 * (m / 16) + m % 16:
      // this warp's lanes 0..15 hold rows 16 q .. 16 q + 15.
      const int m = q * 16 + (lane & 15);
      const int kk = c0 + m;  // output channel of the row
      const int g = kk / a.Cg, k_in = kk - g * a.Cg;
      const int cl0 = (m / a.Cg) * a.Cg;  // the row's group block within the chunk
      const int ky_t = a.row_kz[r] * a.Y + a.row_ky[r];
      const bool has_split = t1 > t0;
      float* wsp = a.ws + (int64_t)split * a.E + ((int64_t)(g * a.Cg + k_in) * a.taps) * a.Cg;
      const uint32_t lane_addr = tmem_base + ((uint32_t)(q * 32) << 16);
      uint32_t col = 0;
      for (int qq = 0; qq < a.nruns; ++qq) {
        for (int b = 0; b < a.run_len[qq]; ++b, col += 64u) {
          const int tap = ky_t * a.X + a.run_kx[qq][b];
          for (int c16 = 0; c16 < 64; c16 += 16) {
            uint32_t p0[16], p1[16];
            tc::tmem_ld16(lane_addr + col + (uint32_t)c16, p0);
            tc::tmem_ld16(lane_addr + a.ncols + col + (uint32_t)c16, p1);
            tc::tmem_ld_wait();
            if (lane < 16 && c16 + 16 > cl0 && c16 < cl0 + a.Cg) {
              float v[16];
#pragma unroll
              for (int e = 0; e < 16; ++e)  // a split without tiles issued no MMA: its partial is zero
                v[e] = has_split ? __uint_as_float(p0[e]) + __uint_as_float(p1[e]) : 0.f;
              float* dst = wsp + (int64_t)tap * a.Cg + (c16 - cl0);
              if (a.Cg >= 16) {  // the whole piece is the row's block: 16-byte aligned stores
#pragma unroll
                for (int e = 0; e < 16; e += 4)
                  *reinterpret_cast<float4*>(dst + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
              } else {
#pragma unroll
                for (int e = 0; e < 16; ++e)
                  if (c16 + e >= cl0 && c16 + e < cl0 + a.Cg) dst[e] = v[e];
              }
            }
          }
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem_base, a.tmem_cols);
  }
}

}  // namespace bwt

namespace {

inline int mod_pos(int v, int m) { return ((v % m) + m) % m; }
inline uint32_t round_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

// Pixel splits for a 152-SM GPU: the plan (and so the workspace size)
// depends on the problem only, not on the device.
constexpr int kPlanSms = 152;

struct BwtPlan {
  bwt::BwtArgs a;
  uint32_t smem_bytes;
  int grid;
};

// The plan, or false when the shape is outside this kernel: 16-bit data,
// Cg == Kg dividing 64, C % 64 == 0, equal H / W strides of 1 or 2, filter
// rows of at most 4 taps, full output rows in one TMA box.
bool make_bwt_plan(const Geometry& g, bool half, BwtPlan* out) {
  (void)half;
  bwt::BwtArgs a;
  std::memset(&a, 0, sizeof(a));
  if (g.Cg != g.Kg || 64 % g.Cg != 0 || g.C() % 64 != 0) return false;
  if (g.sH != g.sW || g.sH < 1 || g.sH > 2) return false;
  if (g.X > bwt::kMaxX || g.Y > 16 || g.Z * g.Y > bwt::kMaxRows) return false;
  const int s = g.sH;
  a.G = g.G, a.Cg = g.Cg, a.C = g.C();
  a.Ho = g.Ho, a.Wo = g.Wo, a.Do = g.Do, a.D = g.D;
  a.X = g.X, a.Y = g.Y, a.taps = g.taps();
  a.sD = g.sD, a.pD = g.pD, a.dD = g.dD, a.s = s;
  a.rows = g.Z * g.Y;
  a.chunks = g.C() / 64;
  // columns: tap xx reads x column s * (ow + qx) + px
  int qx[bwt::kMaxX], px[bwt::kMaxX];
  int qx_min = 1 << 30, qx_max = -(1 << 30);
  for (int kx = 0; kx < g.X; ++kx) {
    const int v = kx * g.dW - g.pW;
    px[kx] = mod_pos(v, s);
    qx[kx] = (v - px[kx]) / s;
    qx_min = std::min(qx_min, qx[kx]);
    qx_max = std::max(qx_max, qx[kx]);
  }
  a.qx_min = qx_min;
  // x planes: one per phase column px in use
  a.nplane = 0;
  int plane_of[2] = {-1, -1};
  for (int kx = 0; kx < g.X; ++kx)
    if (plane_of[px[kx]] < 0) {
      plane_of[px[kx]] = a.nplane;
      a.plane_px[a.nplane++] = px[kx];
    }
  // runs: taps of one plane, in increasing offset, with a constant step
  a.nruns = 0;
  bool used[bwt::kMaxX] = {};
  for (int kx = 0; kx < g.X; ++kx) {
    if (used[kx]) continue;
    const int q = a.nruns++;
    a.run_plane[q] = plane_of[px[kx]];
    a.run_u0[q] = qx[kx] - qx_min;
    a.run_kx[q][0] = kx;
    a.run_len[q] = 1;
    used[kx] = true;
    for (int k2 = kx + 1; k2 < g.X; ++k2) {
      if (used[k2] || px[k2] != px[kx]) continue;
      const int du = qx[k2] - qx[a.run_kx[q][a.run_len[q] - 1]];
      if (a.run_len[q] == 1) a.run_du[q] = du;
      if (du != a.run_du[q] || du <= 0) continue;
      a.run_kx[q][a.run_len[q]++] = k2;
      used[k2] = true;
    }
    if (a.run_len[q] == 1) a.run_du[q] = 1;
  }
  for (int q = 0; q < a.nruns; ++q)
    a.run_idesc[q] = (1u << 4) | ((half ? 0u : 1u) << 7) | ((half ? 0u : 1u) << 10) | (1u << 15) | (1u << 16) |
                     ((uint32_t)((64 * a.run_len[q]) >> 3) << 17) | ((uint32_t)(64 >> 4) << 24);
  // filter rows: row r = (kz, ky) reads x rows s * (oh + qy) + py
  for (int kz = 0; kz < g.Z; ++kz)
    for (int ky = 0; ky < g.Y; ++ky) {
      const int r = kz * g.Y + ky;
      const int v = ky * g.dH - g.pH;
      a.row_py[r] = mod_pos(v, s);
      a.row_qy[r] = (v - a.row_py[r]) / s;
      a.row_kz[r] = kz, a.row_ky[r] = ky;
    }
  // pitch: the output row plus the columns the row's taps reach past it;
  // one TMA box (at most 256 elements per dimension) covers it
  a.P = g.Wo + (qx_max - qx_min);
  if (s * a.P > 256 || a.P > 256) return false;
  a.ncols = 64u * (uint32_t)g.X;
  a.tmem_cols = 32;
  while (a.tmem_cols < 2u * a.ncols) a.tmem_cols <<= 1;
  if (a.tmem_cols > 512) return false;
  // tile rows: about 256 K rows per stage, at least two K steps, and as many
  // stages (2..4) as shared memory holds
  const uint32_t budget = 227u * 1024u - 1024u;
  int TH = std::max(1, std::min(g.Ho, 256 / a.P));
  if (s * TH > 256) TH = 256 / s;
  for (; TH >= 1; --TH) {
    a.TH = TH;
    a.Kp = (int)round_up((uint32_t)(TH * a.P), 16);
    if (a.Kp < 32) a.Kp = 32;  // each issuer gets a K step
    const uint32_t rows_x = round_up((uint32_t)(a.Kp + (qx_max - qx_min) + 16), 8);
    a.dy_bytes = round_up((uint32_t)a.Kp * 128u, 1024);
    a.plane_bytes = round_up(rows_x * 128u, 1024);
    a.stage_bytes = a.dy_bytes + (uint32_t)a.nplane * a.plane_bytes;
    a.stages = (int)std::min<uint32_t>((uint32_t)bwt::kMaxStages, budget / a.stage_bytes);
    if (a.stages >= 2) break;
  }
  if (TH < 1 || a.stages < 2) return false;
  a.tx_bytes = (uint32_t)(1 + a.nplane) * (uint32_t)(a.TH * a.P) * 128u;
  a.tiles_h = (g.Ho + a.TH - 1) / a.TH;
  a.tiles = g.N * (int64_t)g.Do * a.tiles_h;
  const int units = a.rows * a.chunks;
  a.S = (int)std::max<int64_t>(1, std::min<int64_t>(a.tiles, kPlanSms / std::max(1, units)));
  a.E = g.w_elems();
  BwtPlan p;
  p.a = a;
  p.smem_bytes = 1024u + (uint32_t)a.stages * a.stage_bytes;
  // one CTA per SM: two could not both hold their tensor memory
  if (a.tmem_cols > 256) p.smem_bytes = std::max<uint32_t>(p.smem_bytes, 117u * 1024u);
  p.grid = units * a.S;
  *out = p;
  return true;
}

template <typename T>
cudaError_t bwt_launch_typed(const Geometry& g, const LaunchArgs& la, float* ws, const DeviceInfo& dev) {
  BwtPlan p;
  if (!make_bwt_plan(g, std::is_same<T, __half>::value, &p)) return cudaErrorNotSupported;
  if ((reinterpret_cast<uintptr_t>(la.x) | reinterpret_cast<uintptr_t>(la.w)) & 15) return cudaErrorNotSupported;
  if (p.smem_bytes > (uint32_t)dev.max_smem_optin) return cudaErrorNotSupported;
  static SmemAttr attr;
  cudaError_t e = attr.ensure(bwt::bwt_kernel<T>, dev.device, (int)p.smem_bytes);
  if (e != cudaSuccess) return e;
  const uint64_t es = sizeof(T), C = g.C();
  CUtensorMapDataType tt = std::is_same<T, __half>::value ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                          : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int s = p.a.s;
  // x as (C, W, H, D, N): 64 channels x P columns x TH rows of one phase
  CUtensorMap xmap, dymap;
  uint64_t xdims[5] = {C, (uint64_t)g.W, (uint64_t)g.H, (uint64_t)g.D, (uint64_t)g.N};
  uint64_t xstr[4] = {C * es, C * es * g.W, C * es * g.W * g.H, C * es * g.W * g.H * g.D};
  uint32_t xbox[5] = {64u, (uint32_t)(s * p.a.P), (uint32_t)(s * p.a.TH), 1u, 1u};
  uint32_t xestr[5] = {1u, (uint32_t)s, (uint32_t)s, 1u, 1u};
  if (encode_tiled(&xmap, tt, 5, la.x, xdims, xstr, xbox, xestr, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  // dy as (K, Wo, Ho, Do, N): 64 channels x P columns (past Wo: zeros) x TH rows
  uint64_t ddims[5] = {C, (uint64_t)g.Wo, (uint64_t)g.Ho, (uint64_t)g.Do, (uint64_t)g.N};
  uint64_t dstr[4] = {C * es, C * es * g.Wo, C * es * g.Wo * g.Ho, C * es * g.Wo * g.Ho * g.Do};
  uint32_t dbox[5] = {64u, (uint32_t)p.a.P, (uint32_t)p.a.TH, 1u, 1u};
  uint32_t destr[5] = {1u, 1u, 1u, 1u, 1u};
  if (encode_tiled(&dymap, tt, 5, la.w, ddims, dstr, dbox, destr, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  bwt::BwtArgs a = p.a;
  a.ws = ws;
  a.status = la.status;
  a.wait_limit_ns = la.wait_limit_ns;
  e = launch_kernel(bwt::bwt_kernel<T>, dim3(p.grid), dim3(bwt::kThreads), p.smem_bytes, la, xmap, dymap, a);
  if (e != cudaSuccess) return e;
  return bwd_weight_reduce_launch(g, la, ws, p.a.S, dev);
}

}  // namespace

bool bwd_weight_tc_supported(const Geometry& g, DType dt) {
  if (dt == kF32) return false;  // fp32 stays on FFMA (no TF32 rounding)
  BwtPlan p;
  return make_bwt_plan(g, dt == kF16, &p);
}

int64_t bwd_weight_tc_workspace_bytes(const Geometry& g, DType dt) {
  BwtPlan p;
  if (dt == kF32 || !make_bwt_plan(g, dt == kF16, &p)) return 0;
  return (int64_t)p.a.S * p.a.E * 4;
}

cudaError_t bwd_weight_tc_launch(const Geometry& g, const LaunchArgs& a, void* workspace, const DeviceInfo& dev) {
  float* ws = static_cast<float*>(workspace);
  if (a.dt == kF16) return bwt_launch_typed<__half>(g, a, ws, dev);
  if (a.dt == kBF16) return bwt_launch_typed<__nv_bfloat16>(g, a, ws, dev);
  return cudaErrorNotSupported;
}

}  // namespace gconv
