// Grouped convolution backward weight (the gradient with respect to w).
//
//   dw[g, k, z, yy, xx, c] = sum over (n, od, oh, ow) of
//       dy[n, od, oh, ow, g, k] * x[n, od*sD - pD + z*dD, oh*sH - pH + yy*dH, ow*sW - pW + xx*dW, g, c]
//
// with zero padding outside x.  The backward-weight variant, whose runner
// takes X and dY and which can reduce through an fp32 workspace in two
// stages, is listed by the pages' CK grouped-convolution tile engine and its
// Python examples (Examples; Config-options harness, two_stage).
//
// Two stages, both deterministic (fixed split and summation order):
//  1. bwd_weight_partial_kernel: the output pixels (the sum's range) are cut
//     into S equal runs ("splits").  For each split, every work item -- a
//     vector of V input channels x one output channel x a block of taps
//     (one filter row of at most 3, else up to 9) -- accumulates its
//     products in fp32 registers; items
//     that share a CTA may also share the split's pixels ("pixel lanes") and
//     are then summed through shared memory.  Each split writes its fp32
//     partial of every dw element into the caller's workspace [S][E].
//  2. bwd_weight_reduce_kernel: dw[e] = round(sum over s of partial[s][e]),
//     one round-to-nearest-even cast; 32 threads per element share its
//     splits and their sums are added in a fixed order.
// Work items: MODE 0 (grouped) takes V consecutive input channels of one
// group (Cg % V == 0) and one output channel k, lanes ordered k fastest so
// the dy reads of a warp are consecutive and its x reads are shared;
// MODE 1 (depthwise, Cg == Kg == 1) takes V consecutive groups, whose dy and
// x values are both V-element vectors.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "plan_cache.h"

namespace gconv {
namespace {

constexpr int kTapBlockMax = 9;   // most taps one work item accumulates (registers: taps x V)
constexpr int kBwwThreads = 256;  // threads per CTA of the partial kernel

struct BwwArgs {
  const void* x;
  const void* dy;
  float* ws;
  void* dw;
  int G, Cg, Kg;
  int D, H, W, Do, Ho, Wo, Z, Y, X;
  int sD, sH, sW, pD, pH, pW, dD, dH, dW;
  int taps, ntb;      // taps per filter, tap blocks
  int64_t P;          // output pixels N * Do * Ho * Wo (the sum's range)
  int S;              // splits of the pixel range
  int64_t E;          // dw elements
  int items;          // work items per split
  int ipc, lanes;     // items per CTA, pixel lanes per item (ipc * lanes <= kBwwThreads)
};

template <typename T, int V>
__device__ __forceinline__ void load_vec(const T* p, float (&v)[V]) {
  constexpr int bytes = V * (int)sizeof(T);
  if constexpr (bytes == 16) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    unpack16<T>(w, v);
  } else if constexpr (bytes == 8) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    widen_word<T>(u.x, v);
    widen_word<T>(u.y, v + 4 / (int)sizeof(T));
  } else if constexpr (bytes == 4 && sizeof(T) == 2) {
    widen_word<T>(*reinterpret_cast<const uint32_t*>(p), v);
  } else {
#pragma unroll
    for (int i = 0; i < V; ++i) v[i] = Elem<T>::to_f32(p[i]);
  }
}

// NW consecutive 32-bit words (NW = 4, 2 or 1: 16-, 8- or 4-byte aligned).
template <int NW, typename T>
__device__ __forceinline__ void load_words(const T* p, uint32_t (&w)[NW]) {
  if constexpr (NW == 4) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    w[0] = u.x, w[1] = u.y, w[2] = u.z, w[3] = u.w;
  } else if constexpr (NW == 2) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    w[0] = u.x, w[1] = u.y;
  } else {
    w[0] = *reinterpret_cast<const uint32_t*>(p);
  }
}

// Stage 1.  Grid: (CTAs per split, S).  Thread = (item, pixel lane).
template <typename T, int V, int MODE, int kTapBlock>
__global__ void __launch_bounds__(kBwwThreads) bwd_weight_partial_kernel(const BwwArgs a) {
  const T* __restrict__ x = static_cast<const T*>(a.x);
  const T* __restrict__ dy = static_cast<const T*>(a.dy);
  // pixel-lane partials for the in-CTA sum (lanes > 1 only): [tap * V + v][thread]
  extern __shared__ float red[];
  const int tid = threadIdx.x;
  const int nthr = a.ipc * a.lanes;
  const int li = tid % a.ipc, lane = tid / a.ipc;
  const int item = blockIdx.x * a.ipc + li;
  const bool active = lane < a.lanes && item < a.items;
  const int64_t C = (int64_t)a.G * a.Cg, K = (int64_t)a.G * a.Kg;

  // item -> (g, k, channel offset, tap block)
  int g = 0, k = 0, c0 = 0, tb = 0;
  if (active) {
    int f = item;
    if (MODE == 0) {
      k = f % a.Kg;
      f /= a.Kg;
      const int ncv = a.Cg / V;
      c0 = (f % ncv) * V;
      f /= ncv;
      tb = f % a.ntb;
      g = f / a.ntb;
    } else {
      const int ngv = a.G / V;
      g = (f % ngv) * V;  // first of V groups
      tb = f / ngv;
    }
  }
  const int t0 = tb * kTapBlock;
  const int nt = min(kTapBlock, a.taps - t0);

  float acc[kTapBlock][V];
#pragma unroll
  for (int t = 0; t < kTapBlock; ++t)
#pragma unroll
    for (int v = 0; v < V; ++v) acc[t][v] = 0.f;

  grid_dependency_wait();  // x, dy and the workspace are touched only from here on

  if (active) {
    const int64_t p0 = a.P * blockIdx.y / a.S, p1 = a.P * (blockIdx.y + 1) / a.S;
    int64_t p = p0 + lane;
    if (p < p1) {
      // pixel p -> (n, od, oh, ow), then walked incrementally by `lanes`
      int64_t q = p;
      int ow = (int)(q % a.Wo);
      q /= a.Wo;
      int oh = (int)(q % a.Ho);
      q /= a.Ho;
      int od = (int)(q % a.Do);
      int64_t n = q / a.Do;
      const int64_t cx = MODE == 0 ? (int64_t)g * a.Cg + c0 : (int64_t)g;  // x channel of element 0
      const int64_t cy = MODE == 0 ? (int64_t)g * a.Kg + k : (int64_t)g;   // dy channel of element 0
      // per tap of the block: its input-position offsets and its element
      // offset in x (the same for every output pixel)
      int tz[kTapBlock], ty[kTapBlock], tx[kTapBlock];
      int64_t toff[kTapBlock];
#pragma unroll
      for (int t = 0; t < kTapBlock; ++t) {
        const int tt = min(t0 + t, a.taps - 1);
        const int xx = tt % a.X, r = tt / a.X;
        const int yy = r % a.Y, z = r / a.Y;
        tz[t] = z * a.dD, ty[t] = yy * a.dH, tx[t] = xx * a.dW;
        toff[t] = (((int64_t)tz[t] * a.H + ty[t]) * a.W + tx[t]) * C;
      }
      // 16-bit data stays packed: the products are mixed-precision FMAs
      // (fp32 product and sum) of the stored halves
      constexpr bool kPacked = sizeof(T) == 2 && (V % 2) == 0;
      for (; p < p1; p += a.lanes) {
        const T* dyp = dy + p * K + cy;
        float dv[MODE == 0 ? 1 : V];
        uint32_t dw32[kPacked ? V / 2 : 1];
        if constexpr (kPacked) {
          if constexpr (MODE == 0) {
            const uint32_t h = *reinterpret_cast<const unsigned short*>(dyp);
            dw32[0] = h | (h << 16);
          } else {
            load_words<V / 2>(dyp, dw32);
          }
        } else if constexpr (MODE == 0) {
          dv[0] = Elem<T>::to_f32(*dyp);
        } else {
          load_vec<T, V>(dyp, dv);
        }
        const int ih0 = oh * a.sH - a.pH, iw0 = ow * a.sW - a.pW, id0 = od * a.sD - a.pD;
        const T* xp = x + (((n * a.D + id0) * a.H + ih0) * (int64_t)a.W + iw0) * C + cx;
#pragma unroll
        for (int t = 0; t < kTapBlock; ++t) {
          if (t < nt && (unsigned)(id0 + tz[t]) < (unsigned)a.D && (unsigned)(ih0 + ty[t]) < (unsigned)a.H &&
              (unsigned)(iw0 + tx[t]) < (unsigned)a.W) {
            if constexpr (kPacked) {
              uint32_t xw[V / 2];
              load_words<V / 2>(xp + toff[t], xw);
#pragma unroll
              for (int i = 0; i < V / 2; ++i)
                fma_mixed_pair<T>(xw[i], dw32[MODE == 0 ? 0 : i], acc[t][2 * i], acc[t][2 * i + 1]);
            } else {
              float xv[V];
              load_vec<T, V>(xp + toff[t], xv);
#pragma unroll
              for (int v = 0; v < V; ++v) acc[t][v] = fmaf(MODE == 0 ? dv[0] : dv[v], xv[v], acc[t][v]);
            }
          }
        }
        // advance the pixel by `lanes` positions
        ow += a.lanes;
        while (ow >= a.Wo) {
          ow -= a.Wo;
          if (++oh == a.Ho) {
            oh = 0;
            if (++od == a.Do) {
              od = 0;
              ++n;
            }
          }
        }
      }
    }
  }

  // Sum the pixel lanes of each item (in lane order) and write the split's
  // partial: ws[s][e], e the dw element index.
  float* ws = a.ws + (int64_t)blockIdx.y * a.E;
  if (a.lanes > 1) {
    if (active) {
#pragma unroll
      for (int t = 0; t < kTapBlock; ++t)
#pragma unroll
        for (int v = 0; v < V; ++v) red[(t * V + v) * nthr + tid] = acc[t][v];
    }
    __syncthreads();
    if (active && lane == 0) {
      for (int l = 1; l < a.lanes; ++l)
#pragma unroll
        for (int t = 0; t < kTapBlock; ++t)
#pragma unroll
          for (int v = 0; v < V; ++v) acc[t][v] += red[(t * V + v) * nthr + l * a.ipc + li];
    }
  }
  if (active && lane == 0) {
#pragma unroll
    for (int t = 0; t < kTapBlock; ++t) {
      if (t < nt) {
        const int tt = t0 + t;
#pragma unroll
        for (int v = 0; v < V; ++v) {
          const int64_t e = MODE == 0 ? ((((int64_t)g * a.Kg + k) * a.taps + tt) * a.Cg + c0 + v)
                                      : ((int64_t)(g + v) * a.taps + tt);
          ws[e] = acc[t][v];
        }
      }
    }
  }
}

// Stage 2: dw[e] = round(sum over s of ws[s][e]).  A CTA of 32 x 32
// threads takes 32 consecutive elements (coalesced reads of each split's
// row); thread (e, j) sums the splits s = j, j + 32, ... and the 32 sums of
// an element are then added in j order, so the order is fixed.
template <typename T>
__global__ void __launch_bounds__(1024) bwd_weight_reduce_kernel(const BwwArgs a) {
  T* __restrict__ dw = static_cast<T*>(a.dw);
  __shared__ float part[32][33];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  grid_dependency_wait();  // the partials are complete
  for (int64_t e0 = (int64_t)blockIdx.x * 32; e0 < a.E; e0 += (int64_t)gridDim.x * 32) {
    const int64_t e = e0 + tx;
    float s = 0.f;
    if (e < a.E) {
      int i = ty;
      for (; i + 96 < a.S; i += 128) {  // four loads in flight
        const float v0 = a.ws[(int64_t)i * a.E + e], v1 = a.ws[(int64_t)(i + 32) * a.E + e],
                    v2 = a.ws[(int64_t)(i + 64) * a.E + e], v3 = a.ws[(int64_t)(i + 96) * a.E + e];
        s += v0;
        s += v1;
        s += v2;
        s += v3;
      }
      for (; i < a.S; i += 32) s += a.ws[(int64_t)i * a.E + e];
    }
    part[ty][tx] = s;
    __syncthreads();
    if (ty == 0 && e < a.E) {
      float t = 0.f;
#pragma unroll 8
      for (int j = 0; j < 32; ++j) t += part[j][tx];
      dw[e] = epilogue_one<T>(t, 0.f);
    }
    __syncthreads();
  }
}

// Stage 2 for few splits (S <= kSmallS): each thread owns 4 consecutive
// elements and adds their S partials in split order (coalesced 16-byte
// loads; the 32 x 32 form above would leave most of its rows idle).
constexpr int kSmallS = 64;
template <typename T>
__global__ void __launch_bounds__(256) bwd_weight_reduce_few_kernel(const BwwArgs a) {
  T* __restrict__ dw = static_cast<T*>(a.dw);
  grid_dependency_wait();  // the partials are complete
  const int64_t n4 = a.E / 4;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (int64_t)gridDim.x * blockDim.x) {
    float4 acc = reinterpret_cast<const float4*>(a.ws)[i];
    for (int s = 1; s < a.S; ++s) {
      const float4 v = reinterpret_cast<const float4*>(a.ws + (int64_t)s * a.E)[i];
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    dw[4 * i] = epilogue_one<T>(acc.x, 0.f);
    dw[4 * i + 1] = epilogue_one<T>(acc.y, 0.f);
    dw[4 * i + 2] = epilogue_one<T>(acc.z, 0.f);
    dw[4 * i + 3] = epilogue_one<T>(acc.w, 0.f);
  }
}

template <typename T>
cudaError_t reduce_typed(const Geometry& g, const LaunchArgs& la, float* ws, int S, const DeviceInfo& dev);

// Tiled form for two input channels per group (Cg = 2) when every dw
// element fits one CTA's threads: a CTA stages one output row (n, od, oh)
// at a time in shared memory -- dy[n, od, oh, :, :] (Wo pixels x K channels)
// and the Z * Y input rows its taps read, each WR = (Wo-1)*sW + (X-1)*dW + 1
// pixels wide from column -pW, zeros outside x -- and thread (pair, part)
// accumulates output channel k of group g (pair = g*Kg + k) against a
// contiguous block of taps, all Cg input channels, over the row's pixels.
// The per-pixel form above issues four small global loads for six MACs on
// the 3D layers (Cg = 2, Kg = 4); here every operand comes from shared
// memory.  A CTA takes rows cta, cta + S, ... and writes one fp32 partial of
// every dw element; the reduction adds the S partials in order.
constexpr int kTileThreads = 256;
constexpr int kTileMaxTaps = 16;  // taps per thread
constexpr int kTileSplits = 304;  // CTAs (two per SM of a 152-SM GPU), fixed so the workspace is device-free

struct BwTileArgs {
  const void* x;
  const void* dy;
  float* ws;
  int G, Cg, Kg, C, K;
  int D, H, W, Do, Ho, Wo, Z, Y, X;
  int sD, sH, sW, pD, pH, pW, dD, dH, dW;
  int taps, WR;     // taps per filter, staged row width in pixels
  int tsplit, tpt;  // threads per (g, k) pair, taps per thread
  int64_t rows;     // output rows N * Do * Ho
  int S;            // CTAs = partials
  int64_t E;        // dw elements
  uint32_t x_bytes;  // staged input rows (the dy row follows)
};

// 16-byte copy global -> shared, asynchronous; src_bytes 0 writes zeros
// (the source is then not read, but is still a valid address).
__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}

// KG output channels of one group per thread (each x pair it loads feeds
// 2 * KG FMAs), at most NT taps.
template <typename T, int CG, int KG, int NT>
__global__ void __launch_bounds__(kTileThreads) bwd_weight_tile_kernel(const BwTileArgs a) {
  extern __shared__ __align__(16) uint8_t sm[];
  const uint4* __restrict__ x4 = static_cast<const uint4*>(a.x);
  const uint4* __restrict__ dy4 = static_cast<const uint4*>(a.dy);
  constexpr int kPiece = 16 / (int)sizeof(T);  // elements per 16-byte piece
  const uint32_t buf_bytes = a.x_bytes + (uint32_t)(a.Wo * a.K) * (uint32_t)sizeof(T);  // one row's staging
  const int tid = threadIdx.x;
  const int unit = tid / a.tsplit, part = tid - unit * a.tsplit;  // unit = (group, block of KG channels)
  const bool active = unit < a.G * (a.Kg / KG);
  const int pair = unit * KG;  // first (g, k) pair of the unit: g * Kg + k0
  const int g = active ? pair / a.Kg : 0;
  const int t0 = part * a.tpt;
  const int nt = active ? max(0, min(a.tpt, a.taps - t0)) : 0;
  // per tap of this thread: its element offset in the staged rows at output column 0
  int toff[NT];
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const int tt = min(t0 + t, a.taps - 1);
    const int xx = tt % a.X, r = tt / a.X;  // r = z * Y + yy
    toff[t] = (r * a.WR + xx * a.dW) * a.C + g * CG;
  }
  float acc[NT][KG][CG];
#pragma unroll
  for (int t = 0; t < NT; ++t)
#pragma unroll
    for (int k = 0; k < KG; ++k)
#pragma unroll
      for (int c = 0; c < CG; ++c) acc[t][k][c] = 0.f;
  const int colstep = a.sW * a.C;
  const int ppx = a.C / kPiece;  // pieces per input pixel
  const int row_pieces = a.WR * ppx;
  const int dy_pieces = a.Wo * a.K / kPiece;
  // the in-range pixels of an input row are contiguous in x, so staged
  // piece k of a row maps to x piece base + k; pieces outside
  // [pW * ppx, (pW + W) * ppx) are the zero padding
  const int lo = a.pW * ppx, hi = (a.pW + a.W) * ppx;

  // Copies of output row `row` into buffer b: the Z * Y input rows, then dy.
  auto stage = [&](int64_t row, int b) {
    uint8_t* base_s = sm + (size_t)b * buf_bytes;
    uint4* xs4 = reinterpret_cast<uint4*>(base_s);
    uint4* dys4 = reinterpret_cast<uint4*>(base_s + a.x_bytes);
    const int oh = (int)(row % a.Ho);
    const int64_t q = row / a.Ho;
    const int od = (int)(q % a.Do);
    const int64_t n = q / a.Do;
    for (int r = 0; r < a.Z * a.Y; ++r) {
      const int z = r / a.Y, yy = r - z * a.Y;
      const int id = od * a.sD - a.pD + z * a.dD, ih = oh * a.sH - a.pH + yy * a.dH;
      const bool rv = (unsigned)id < (unsigned)a.D && (unsigned)ih < (unsigned)a.H;
      const int64_t base = rv ? ((n * a.D + id) * a.H + ih) * (int64_t)a.W * ppx - lo : 0;
      for (int k = tid; k < row_pieces; k += kTileThreads) {
        const bool in = rv && k >= lo && k < hi;
        cp_async16(xs4 + (size_t)r * row_pieces + k, in ? x4 + base + k : x4, in ? 16u : 0u);
      }
    }
    const uint4* dsrc = dy4 + (((n * a.Do + od) * a.Ho + oh) * (int64_t)a.Wo * a.K) / kPiece;
    for (int k = tid; k < dy_pieces; k += kTileThreads) cp_async16(dys4 + k, dsrc + k, 16u);
    asm volatile("cp.async.commit_group;" ::: "memory");
  };

  grid_dependency_wait();  // x, dy and the workspace are touched only from here on

  // Two buffers: the copies of the CTA's next row are in flight while its
  // current row is summed.
  int b = 0;
  if ((int64_t)blockIdx.x < a.rows) stage(blockIdx.x, 0);
  for (int64_t row = blockIdx.x; row < a.rows; row += a.S, b ^= 1) {
    if (row + a.S < a.rows) {
      stage(row + a.S, b ^ 1);
      asm volatile("cp.async.wait_group 1;" ::: "memory");
    } else {
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    }
    __syncthreads();
    const T* xs = reinterpret_cast<const T*>(sm + (size_t)b * buf_bytes);
    const T* dys = reinterpret_cast<const T*>(sm + (size_t)b * buf_bytes + a.x_bytes);
    if (active) {
      for (int ow = 0; ow < a.Wo; ++ow) {
        const T* dyp = dys + ow * a.K + pair;  // KG consecutive output channels
        const int cb = ow * colstep;
        if constexpr (CG == 2 && sizeof(T) == 2) {
          uint32_t dpair[KG];  // each channel's dy in both halves
#pragma unroll
          for (int k = 0; k < KG; ++k) {
            const uint32_t h = *reinterpret_cast<const unsigned short*>(dyp + k);
            dpair[k] = h | (h << 16);
          }
#pragma unroll
          for (int t = 0; t < NT; ++t)
            if (t < nt) {
              const uint32_t xw = *reinterpret_cast<const uint32_t*>(xs + cb + toff[t]);
#pragma unroll
              for (int k = 0; k < KG; ++k) fma_mixed_pair<T>(xw, dpair[k], acc[t][k][0], acc[t][k][1]);
            }
        } else {
          float d[KG];
#pragma unroll
          for (int k = 0; k < KG; ++k) d[k] = Elem<T>::to_f32(dyp[k]);
#pragma unroll
          for (int t = 0; t < NT; ++t)
            if (t < nt)
#pragma unroll
              for (int c = 0; c < CG; ++c) {
                const float xv = Elem<T>::to_f32(xs[cb + toff[t] + c]);
#pragma unroll
                for (int k = 0; k < KG; ++k) acc[t][k][c] = fmaf(d[k], xv, acc[t][k][c]);
              }
        }
      }
    }
    __syncthreads();  // buffer b is free for the copies of the row after next
  }
  float* ws = a.ws + (int64_t)blockIdx.x * a.E;
#pragma unroll
  for (int t = 0; t < NT; ++t)
    if (t < nt)
#pragma unroll
      for (int k = 0; k < KG; ++k)
#pragma unroll
        for (int c = 0; c < CG; ++c) ws[((int64_t)(pair + k) * a.taps + t0 + t) * a.Cg + c] = acc[t][k][c];
}

// The tiled form's shape: threads per (g, k) pair, taps per thread, staged
// bytes; false when the problem is outside its range.
struct BwTilePlan {
  int kg, tsplit, tpt, WR, S;  // output channels per thread, threads per unit, taps per thread
  uint32_t x_bytes, smem;
};
bool plan_bw_tile(const Geometry& g, int es, BwTilePlan* p) {
  // two input channels per group: the per-pixel form's vectors serve one
  // (depthwise: 62 against 114 us on the MobileNetV2 layer) and wider groups
  if (g.Cg != 2) return false;
  if ((g.C() * es) % 16 != 0 || (g.K() * es) % 16 != 0) return false;
  // two output channels per thread where their taps per thread fit
  // (kTileMaxTaps / 2), else one: each x pair a thread loads then feeds four
  // FMAs.  (3D N=8: 67 against 69 us; four channels per thread, 77 us, had
  // eight threads of a group read eight taps' pixels on the same banks.)
  int kg = 0, tsplit = 0, tpt = 0;
  for (int k = 2; k >= 1 && kg == 0; k /= 2) {
    if (g.Kg % k != 0) continue;
    const int units = g.G * (g.Kg / k);
    if (units > kTileThreads) continue;
    const int ts = kTileThreads / units;
    const int tp = (g.taps() + ts - 1) / ts;
    if (tp <= kTileMaxTaps / k) kg = k, tsplit = ts, tpt = tp;
  }
  if (kg == 0) return false;
  const int64_t WR = (int64_t)(g.Wo - 1) * g.sW + (int64_t)(g.X - 1) * g.dW + 1;
  const int64_t xb = (int64_t)g.Z * g.Y * WR * g.C() * es, yb = (int64_t)g.Wo * g.K() * es;
  if (2 * (xb + yb) > 110 * 1024) return false;  // two buffers, two CTAs per SM
  const int64_t rows = g.N * (int64_t)g.Do * g.Ho;
  p->kg = kg, p->tsplit = tsplit, p->tpt = tpt, p->WR = (int)WR;
  p->S = (int)std::min<int64_t>(rows, kTileSplits);
  p->x_bytes = (uint32_t)xb, p->smem = (uint32_t)(2 * (xb + yb));
  return true;
}

template <typename T>
cudaError_t bwd_weight_tile_typed(const Geometry& g, const LaunchArgs& la, float* ws, const BwTilePlan& p,
                                  const DeviceInfo& dev) {
  BwTileArgs a{};
  a.x = la.x;
  a.dy = la.w;  // a.w carries dy (see kernels.h)
  a.ws = ws;
  a.G = g.G, a.Cg = g.Cg, a.Kg = g.Kg, a.C = g.C(), a.K = g.K();
  a.D = g.D, a.H = g.H, a.W = g.W, a.Do = g.Do, a.Ho = g.Ho, a.Wo = g.Wo, a.Z = g.Z, a.Y = g.Y, a.X = g.X;
  a.sD = g.sD, a.sH = g.sH, a.sW = g.sW, a.pD = g.pD, a.pH = g.pH, a.pW = g.pW, a.dD = g.dD, a.dH = g.dH,
  a.dW = g.dW;
  a.taps = g.taps(), a.WR = p.WR, a.tsplit = p.tsplit, a.tpt = p.tpt;
  a.rows = g.N * (int64_t)g.Do * g.Ho;
  a.S = p.S;
  a.E = g.w_elems();
  a.x_bytes = p.x_bytes;
  // (plan_bw_tile takes Cg = 2 only)
  cudaError_t e;
  if (p.kg == 2) {
    static SmemAttr attr;
    e = attr.ensure(bwd_weight_tile_kernel<T, 2, 2, kTileMaxTaps / 2>, dev.device, (int)p.smem);
    if (e == cudaSuccess)
      e = launch_kernel(bwd_weight_tile_kernel<T, 2, 2, kTileMaxTaps / 2>, dim3(p.S), dim3(kTileThreads), p.smem, la,
                        a);
  } else {
    static SmemAttr attr;
    e = attr.ensure(bwd_weight_tile_kernel<T, 2, 1, kTileMaxTaps>, dev.device, (int)p.smem);
    if (e == cudaSuccess)
      e = launch_kernel(bwd_weight_tile_kernel<T, 2, 1, kTileMaxTaps>, dim3(p.S), dim3(kTileThreads), p.smem, la, a);
  }
  if (e != cudaSuccess) return e;
  return reduce_typed<T>(g, la, ws, p.S, dev);
}

// Launch plan: mode, vector width, items, CTA shape and splits.  Depends on
// the problem and element size only (not on the device), so the workspace
// size can be queried without a GPU.
struct BwwPlan {
  int mode, V, tb, items, ipc, lanes, ctas_per_split, S;
  int64_t E;
};

// Items and CTA shape for vector width V.
void shape_bww(const Geometry& g, int V, BwwPlan* p) {
  const int ntb = (g.taps() + p->tb - 1) / p->tb;
  p->V = V;
  p->items = p->mode == 1 ? (g.G / V) * ntb : g.G * g.Kg * (g.Cg / V) * ntb;
  p->ipc = std::min(p->items, kBwwThreads);
  p->lanes = kBwwThreads / p->ipc;
  p->ctas_per_split = (p->items + p->ipc - 1) / p->ipc;
}

// vmax: the widest vector (elements) the buffers' alignment allows.  The
// splits S are those of the widest vector the shape allows, whatever vmax,
// so the workspace size does not depend on the pointers.
BwwPlan plan_bww(const Geometry& g, int es, int vmax) {
  BwwPlan p{};
  p.mode = (g.Cg == 1 && g.Kg == 1) ? 1 : 0;
  // taps per work item: one filter row (X taps) when that is at most 3,
  // else up to kTapBlockMax; fewer registers per thread keep more warps
  // resident to hide the load latency
  p.tb = g.X <= 3 ? g.X : kTapBlockMax;
  auto widest = [&](int cap) {
    int V = cap;
    while (V > 1 && (p.mode == 1 ? g.G % V : g.Cg % V) != 0) V /= 2;
    return V;
  };
  shape_bww(g, widest(16 / es), &p);
  p.E = (int64_t)g.K() * g.taps() * g.Cg;
  const int64_t P = g.N * (int64_t)g.Do * g.Ho * g.Wo;
  // about 1024 threads per SM of a 152-SM GPU, at least 16 pixels per
  // thread, and at most 32 MB of partials
  const int64_t want = std::max<int64_t>(1, (int64_t)152 * 1024 / ((int64_t)p.ctas_per_split * kBwwThreads));
  const int64_t by_pixels = std::max<int64_t>(1, P / ((int64_t)p.lanes * 16));
  const int64_t by_bytes = std::max<int64_t>(1, ((int64_t)32 << 20) / (p.E * 4));
  p.S = (int)std::min<int64_t>(std::min(want, by_pixels), std::min<int64_t>(by_bytes, 65535));
  shape_bww(g, widest(std::min(vmax, 16 / es)), &p);
  return p;
}

template <typename T, int V, int MODE, int TB>
cudaError_t launch_partial_tb(const BwwArgs& a, const BwwPlan& p, const LaunchArgs& la, const DeviceInfo& dev) {
  const size_t smem = p.lanes > 1 ? (size_t)TB * V * p.ipc * p.lanes * sizeof(float) : 0;
  static SmemAttr attr;
  if (smem > 48 * 1024) {
    cudaError_t e = attr.ensure(bwd_weight_partial_kernel<T, V, MODE, TB>, dev.device, (int)smem);
    if (e != cudaSuccess) return e;
  }
  return launch_kernel(bwd_weight_partial_kernel<T, V, MODE, TB>, dim3(p.ctas_per_split, p.S), dim3(kBwwThreads),
                       smem, la, a);
}
template <typename T, int V, int MODE>
cudaError_t launch_partial(const BwwArgs& a, const BwwPlan& p, const LaunchArgs& la, const DeviceInfo& dev) {
  switch (p.tb) {
    case 1: return launch_partial_tb<T, V, MODE, 1>(a, p, la, dev);
    case 2: return launch_partial_tb<T, V, MODE, 2>(a, p, la, dev);
    case 3: return launch_partial_tb<T, V, MODE, 3>(a, p, la, dev);
    default: return launch_partial_tb<T, V, MODE, kTapBlockMax>(a, p, la, dev);
  }
}

template <typename T>
cudaError_t bwd_weight_typed(const Geometry& g, const LaunchArgs& la, float* ws, const DeviceInfo& dev) {
  // the tiled form where its range and the 16-byte alignment of x and dy allow
  {
    BwTilePlan tp;
    if (plan_bw_tile(g, (int)sizeof(T), &tp) &&
        ((reinterpret_cast<uintptr_t>(la.x) | reinterpret_cast<uintptr_t>(la.w)) & 15) == 0)
      return bwd_weight_tile_typed<T>(g, la, ws, tp, dev);
  }
  // the widest vector both x and dy are aligned to
  int vmax = 16 / (int)sizeof(T);
  while (vmax > 1 && ((reinterpret_cast<uintptr_t>(la.x) | reinterpret_cast<uintptr_t>(la.w)) &
                      (uintptr_t)(vmax * sizeof(T) - 1)))
    vmax /= 2;
  const BwwPlan p = plan_bww(g, (int)sizeof(T), vmax);
  BwwArgs a{};
  a.x = la.x;
  a.dy = la.w;  // a.w carries dy (see kernels.h)
  a.ws = ws;
  a.dw = la.y;
  a.G = g.G, a.Cg = g.Cg, a.Kg = g.Kg;
  a.D = g.D, a.H = g.H, a.W = g.W, a.Do = g.Do, a.Ho = g.Ho, a.Wo = g.Wo, a.Z = g.Z, a.Y = g.Y, a.X = g.X;
  a.sD = g.sD, a.sH = g.sH, a.sW = g.sW, a.pD = g.pD, a.pH = g.pH, a.pW = g.pW, a.dD = g.dD, a.dH = g.dH,
  a.dW = g.dW;
  a.taps = g.taps();
  a.ntb = (a.taps + p.tb - 1) / p.tb;
  a.P = g.N * (int64_t)g.Do * g.Ho * g.Wo;
  a.S = p.S;
  a.E = p.E;
  a.items = p.items;
  a.ipc = p.ipc;
  a.lanes = p.lanes;
  cudaError_t e = cudaErrorNotSupported;
  // vector widths: 16 / sizeof(T) and below, as the plan's divisibility allows
#define GCONV_BWW(v_)                                                                   \
  if (p.V == v_) {                                                                      \
    e = p.mode == 1 ? launch_partial<T, v_, 1>(a, p, la, dev) : launch_partial<T, v_, 0>(a, p, la, dev); \
  }
  GCONV_BWW(1)
  GCONV_BWW(2)
  GCONV_BWW(4)
  if constexpr (sizeof(T) == 2) {
    GCONV_BWW(8)
  }
#undef GCONV_BWW
  if (e != cudaSuccess) return e;
  const int64_t blocks = std::min<int64_t>((p.E + 31) / 32, (int64_t)dev.num_sms * 2);
  return launch_kernel(bwd_weight_reduce_kernel<T>, dim3((unsigned)std::max<int64_t>(1, blocks)), dim3(1024), 0, la,
                       a);
}

template <typename T>
cudaError_t reduce_typed(const Geometry& g, const LaunchArgs& la, float* ws, int S, const DeviceInfo& dev) {
  BwwArgs a{};
  a.ws = ws;
  a.dw = la.y;
  a.S = S;
  a.E = g.w_elems();
  if (S <= kSmallS && a.E % 4 == 0) {
    const int64_t blocks = std::min<int64_t>((a.E / 4 + 255) / 256, (int64_t)dev.num_sms * 8);
    return launch_kernel(bwd_weight_reduce_few_kernel<T>, dim3((unsigned)std::max<int64_t>(1, blocks)), dim3(256),
                         0, la, a);
  }
  const int64_t blocks = std::min<int64_t>((a.E + 31) / 32, (int64_t)dev.num_sms * 2);
  return launch_kernel(bwd_weight_reduce_kernel<T>, dim3((unsigned)std::max<int64_t>(1, blocks)), dim3(1024), 0, la,
                       a);
}

}  // namespace

cudaError_t bwd_weight_reduce_launch(const Geometry& g, const LaunchArgs& a, float* ws, int S,
                                     const DeviceInfo& dev) {
  switch (a.dt) {
    case kF32: return reduce_typed<float>(g, a, ws, S, dev);
    case kF16: return reduce_typed<__half>(g, a, ws, S, dev);
    case kBF16: return reduce_typed<__nv_bfloat16>(g, a, ws, S, dev);
  }
  return cudaErrorNotSupported;
}

int64_t bwd_weight_workspace_bytes(const Geometry& g, DType dt) {
  const BwwPlan p = plan_bww(g, dtype_bytes(dt), 16 / dtype_bytes(dt));
  // any route may run (the tensor-core and tiled ones need 16-byte aligned x and dy)
  int64_t bytes = std::max<int64_t>((int64_t)p.S * p.E * 4, bwd_weight_tc_workspace_bytes(g, dt));
  BwTilePlan tp;
  if (plan_bw_tile(g, dtype_bytes(dt), &tp)) bytes = std::max<int64_t>(bytes, (int64_t)tp.S * g.w_elems() * 4);
  return bytes;
}

cudaError_t bwd_weight_launch(const Geometry& g, const LaunchArgs& a, void* workspace, const DeviceInfo& dev) {
  float* ws = static_cast<float*>(workspace);
  switch (a.dt) {
    case kF32: return bwd_weight_typed<float>(g, a, ws, dev);
    case kF16: return bwd_weight_typed<__half>(g, a, ws, dev);
    case kBF16: return bwd_weight_typed<__nv_bfloat16>(g, a, ws, dev);
  }
  return cudaErrorNotSupported;
}

}  // namespace gconv
