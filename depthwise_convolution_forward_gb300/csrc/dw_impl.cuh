// Ka: depthwise direct kernel (Cg == Kg == 1), bandwidth-bound.
//
// Design (sm_103a):
//  * Persistent CTAs walk a static list of output tiles
//    (n, od, TH x TW output pixels, TC channels).
//  * Warp 0 is a producer: for each tile one lane issues a single 5-D TMA copy
//    of the haloed input box [1 x Dh x Hh x Wh x TC] (NDHWC order) into a
//    shared-memory stage.  TMA zero-fills coordinates outside the tensor,
//    which is exactly the convolution's zero padding, so the compute loop has
//    no bounds checks.
//  * Stages form a ring with "full" (copy landed) and "empty" (consumers done)
//    mbarriers, so copies for later tiles overlap the arithmetic on this one.
//  * Each consumer thread owns one 16-byte channel vector (8 x f16/bf16 or
//    4 x f32) of a 1 x WB strip of outputs.  It reads each needed input vector
//    of an input row once (one 128-bit shared load) and reuses it across the
//    WB outputs and the K horizontal taps (register blocking), accumulates in
//    fp32, and finishes with the fused bias + round-to-nearest-even cast (Kc)
//    and a 16-byte store.  All weights of the layer stay in shared memory.
//  * Every mbarrier wait is bounded; on expiry the waiting warp reports a
//    timeout in the status word and exits, and the producer waits (bounded)
//    for the copies it still has in flight before it exits.
#pragma once

#include "common.cuh"

namespace gconv {
namespace dw {

struct DwArgs {
  const void* x;  // used by the direct-load variant only
  int D, H, W;    // input extents (direct-load variant)
  const void* w;
  const void* bias;
  void* y;
  int C;
  int Do, Ho, Wo;
  int Z, dD, sD, pD, pH, pW;
  int TH, TW, TC;
  int Dh, Hh, Wh;
  int tiles_c, tiles_w, tiles_h;
  int64_t num_tiles;
  int stages;
  uint32_t stage_bytes;   // bytes one TMA box writes
  uint32_t stage_stride;  // bytes between stages (>= stage_bytes, 1024-aligned)
  uint32_t stage_off;     // offset of stage 0 in dynamic shared memory
  int h0;                 // column form: halo rows in the first of two copies per tile (Hh: one copy)
  uint32_t bytes0;        // bytes of the first copy (bytes of the second: stage_bytes - bytes0)
  int* status;
  uint64_t wait_limit_ns;
  int test_flags;
};

struct TileCoord {
  int ct, tw, th, od, n;
};

// Tile index -> coordinates, channel tile fastest.  32-bit unsigned
// arithmetic while the tile count fits in 32 bits, 64-bit beyond.
__device__ __forceinline__ TileCoord decode_tile(const DwArgs& a, int64_t t64) {
  TileCoord c;
  if (a.num_tiles > 0xffffffffll) {  // more tiles than 32 bits count: 64-bit division
    int64_t q64 = t64 / a.tiles_c;
    c.ct = (int)(t64 - q64 * a.tiles_c);
    t64 = q64;
    q64 = t64 / a.tiles_w;
    c.tw = (int)(t64 - q64 * a.tiles_w);
    t64 = q64;
    q64 = t64 / a.tiles_h;
    c.th = (int)(t64 - q64 * a.tiles_h);
    t64 = q64;
    q64 = t64 / a.Do;
    c.od = (int)(t64 - q64 * a.Do);
    c.n = (int)q64;
    return c;
  }
  uint32_t t = (uint32_t)t64;
  uint32_t q = t / (uint32_t)a.tiles_c;
  c.ct = (int)(t - q * (uint32_t)a.tiles_c);
  t = q;
  q = t / (uint32_t)a.tiles_w;
  c.tw = (int)(t - q * (uint32_t)a.tiles_w);
  t = q;
  q = t / (uint32_t)a.tiles_h;
  c.th = (int)(t - q * (uint32_t)a.tiles_h);
  t = q;
  q = t / (uint32_t)a.Do;
  c.od = (int)(t - q * (uint32_t)a.Do);
  c.n = (int)q;
  return c;
}

// FMA forms of the inner loop.
enum DwMode : int {
  kWidenFfma = 0,   // widen inputs to fp32, scalar fp32 FMA
  kMixedFma = 1,    // PTX mixed-precision fma.rn.f32.{f16,bf16} on packed inputs
  kWidenFfma2 = 2,  // widen inputs to fp32, packed fp32x2 FMA (sm_100+)
};

constexpr int kDwMaxStages = 4;
constexpr uint32_t kDwMaxWeightBytes = 64 * 1024;

// Shared-memory layout: [full mbarriers x4][empty mbarriers x4][weights of all
// C channels][bias fp32 C] ... [stages, 1024-aligned].  Weights are fp32 in
// [tap][VEC/4][C/VEC][4] (kWidenFfma, kWidenFfma2) or storage type in
// [tap][C] (kMixedFma): either way the 16-byte piece one lane reads for a tap
// sits next to its neighbours' (conflict-free 128-bit loads).  All weights
// stay resident, so a CTA never reloads them between tiles.
__host__ __device__ inline uint32_t weight_smem_bytes(int taps, int C, int es, int mode) {
  const uint32_t b = (uint32_t)(taps * C) * (uint32_t)(mode == kMixedFma ? es : 4);
  return (b + 15u) & ~15u;
}
template <int K>
__host__ __device__ inline uint32_t fixed_smem_bytes(int Z, int C, int es, int mode) {
  return 64u + weight_smem_bytes(Z * K * K, C, es, mode) + 4u * (uint32_t)C;
}

// Warp 0 is the producer: one lane issues the TMA copy of each tile's haloed
// input box into the next free stage.  Warps 1.. are consumers: they wait for
// a stage to fill, compute their outputs from it, and release it through the
// stage's "empty" barrier (one arrival per consumer warp).  Issuing a copy can
// stall the issuing thread for about a microsecond; on its own warp that stall
// overlaps with the consumers' arithmetic.
template <typename T, int K, int S, int DL, int WB, int MODE>
__global__ void __launch_bounds__(WB >= 8 ? 288 : 512) dw_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap,
                                                                 const __grid_constant__ CUtensorMap,
                                                                 const DwArgs a) {
  constexpr int VEC = Elem<T>::kVec;
  constexpr int NCOL = (WB - 1) * S + (K - 1) * DL + 1;  // input columns per WB outputs
  static_assert(MODE != kMixedFma || sizeof(T) == 2, "mixed-precision FMA needs 16-bit storage");
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kDwMaxStages;
  const int taps = a.Z * K * K;
  uint8_t* w_raw = smem + 64;
  float* b_s = reinterpret_cast<float*>(smem + 64 + weight_smem_bytes(taps, a.C, (int)sizeof(T), MODE));
  uint8_t* stage0 = smem + a.stage_off;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int ncons = (int)blockDim.x - 32;
  const int NV = a.TC / VEC;      // channel vectors per tile
  const int NVC = a.C / VEC;      // channel vectors of the whole tensor
  const int nbw = a.TW / WB;
  const int items = NV * nbw * a.TH;
  const T* __restrict__ wg = static_cast<const T*>(a.w);
  const T* __restrict__ bg = static_cast<const T*>(a.bias);
  T* __restrict__ yg = static_cast<T*>(a.y);

  if (tid == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], (uint32_t)(ncons / 32));
    }
    fence_mbar_init();
    tma_prefetch_desc(&xmap);
  }
  grid_dependency_wait();  // x, w, bias and y are touched only from here on
  // resident weights and bias for every channel
  for (int i = tid; i < taps * a.C; i += blockDim.x) {
    const int t = i / a.C, ch = i - t * a.C;
    const T v = wg[(int64_t)ch * taps + t];
    if constexpr (MODE == kMixedFma) {
      reinterpret_cast<T*>(w_raw)[t * a.C + ch] = v;
    } else {
      const int cvv = ch / VEC, q = (ch % VEC) / 4, e = ch % 4;
      reinterpret_cast<float*>(w_raw)[((t * (VEC / 4) + q) * NVC + cvv) * 4 + e] = Elem<T>::to_f32(v);
    }
  }
  for (int i = tid; i < a.C; i += blockDim.x) b_s[i] = bg != nullptr ? Elem<T>::to_f32(bg[i]) : 0.f;
  __syncthreads();

  const bool withhold = (a.test_flags & 1) && blockIdx.x == 0;
  if (warp == 0) {
    // ---------------- producer ----------------
    if (lane == 0) {
      int k = 0;
      bool failed = false;
      for (;; ++k) {
        const int64_t tile = blockIdx.x + (int64_t)k * gridDim.x;
        if (tile >= a.num_tiles) break;
        const int s = k % a.stages;
        if (k >= a.stages &&
            !mbar_wait(&empty[s], (uint32_t)(((k / a.stages) - 1) & 1), a.wait_limit_ns)) {
          failed = true;
          break;
        }
        if (withhold && k == 0) continue;
        const TileCoord c = decode_tile(a, tile);
        const int iw0 = c.tw * a.TW * S - a.pW;
        const int ih0 = c.th * a.TH * S - a.pH;
        const int id0 = c.od * a.sD - a.pD;
        mbar_arrive_expect_tx(&full[s], a.stage_bytes);
        tma_load_5d(stage0 + (size_t)s * a.stage_stride, &xmap, &full[s], c.ct * a.TC, iw0, ih0, id0,
                    (int)c.n);
      }
      if (failed) report(a.status, kDevTimeout, 2);
      // Bounded drain of the last copies issued, so that no copy is still in
      // flight when the CTA can exit (consumers that timed out may be gone).
      for (int j = k > a.stages ? k - a.stages : 0; j < k; ++j) {
        if (withhold && j == 0) continue;
        mbar_wait(&full[j % a.stages], (uint32_t)((j / a.stages) & 1), a.wait_limit_ns);
      }
    }
    return;
  }

  // ---------------- consumers ----------------
  const int ctid = tid - 32;
  for (int k = 0;; ++k) {
    const int64_t tile = blockIdx.x + (int64_t)k * gridDim.x;
    if (tile >= a.num_tiles) break;
    const int s = k % a.stages;
    const uint32_t parity = (uint32_t)((k / a.stages) & 1);
    const TileCoord c = decode_tile(a, tile);
    const int c0 = c.ct * a.TC;

    // Lane 0 polls; after the warp agrees, every lane observes the completed
    // phase itself (acquire) before reading the stage.
    bool ok = true;
    if (lane == 0) ok = mbar_wait(&full[s], parity, a.wait_limit_ns);
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    if (ok && lane != 0) ok = mbar_wait(&full[s], parity, a.wait_limit_ns);
    if (!__all_sync(0xffffffffu, ok)) {
      if (lane == 0) report(a.status, kDevTimeout, 1);
      return;
    }

    const T* st = reinterpret_cast<const T*>(stage0 + (size_t)s * a.stage_stride);
    const int plane_elems = a.Hh * a.Wh * a.TC;
    for (int it = ctid; it < items; it += ncons) {
      const int cv = it % NV;
      const int blk = it / NV;
      const int oh_l = blk / nbw;
      const int ow_l = (blk - oh_l * nbw) * WB;
      const int oh = c.th * a.TH + oh_l;
      const int ch = c0 + cv * VEC;
      const int ow0 = c.tw * a.TW + ow_l;
      const bool row_ok = oh < a.Ho && ch < a.C;
      T* yrow = yg + ((((int64_t)c.n * a.Do + c.od) * a.Ho + oh) * (int64_t)a.Wo) * a.C + ch;
      float acc[WB][VEC];
#pragma unroll
      for (int j = 0; j < WB; ++j)
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[j][e] = 0.f;

      for (int z = 0; z < a.Z; ++z) {
        const T* plane = st + (size_t)(z * a.dD) * plane_elems;
        const bool last_z = z == a.Z - 1;
#pragma unroll
        for (int ky = 0; ky < K; ++ky) {
          const T* rowp = plane + ((size_t)(oh_l * S + ky * DL) * a.Wh + ow_l * S) * a.TC + cv * VEC;
          // In the final filter row each output is complete as soon as its K
          // taps are added: store it right away so the stores of a thread
          // spread over the row instead of bursting at the end.
          const bool store_now = last_z && ky == K - 1 && row_ok;
          uint32_t xw[NCOL][4];
#pragma unroll
          for (int cc = 0; cc < NCOL; ++cc) lds128(rowp + cc * a.TC, xw[cc]);
          if constexpr (MODE == kMixedFma) {
            const T* wz = reinterpret_cast<const T*>(w_raw) + (z * K * K + ky * K) * a.C + c0 + cv * VEC;
            uint32_t ww[K][4];
#pragma unroll
            for (int kx = 0; kx < K; ++kx) lds128(wz + kx * a.C, ww[kx]);
#pragma unroll
            for (int j = 0; j < WB; ++j) {
#pragma unroll
              for (int kx = 0; kx < K; ++kx)
#pragma unroll
                for (int q = 0; q < 4; ++q)
                  fma_mixed_pair<T>(xw[j * S + kx * DL][q], ww[kx][q], acc[j][2 * q], acc[j][2 * q + 1]);
              if (store_now && ow0 + j < a.Wo)
                epilogue_store<T, VEC>(yrow + (int64_t)(ow0 + j) * a.C, acc[j], b_s + ch);
            }
          } else {
            const float* wz =
                reinterpret_cast<const float*>(w_raw) + (z * K * K + ky * K) * a.C + (c0 / VEC + cv) * 4;
            float v[NCOL][VEC];
#pragma unroll
            for (int cc = 0; cc < NCOL; ++cc) unpack16<T>(xw[cc], v[cc]);
            float wv[K][VEC];
#pragma unroll
            for (int kx = 0; kx < K; ++kx)
#pragma unroll
              for (int q = 0; q < VEC / 4; ++q) {
                const float4 f = *reinterpret_cast<const float4*>(wz + kx * a.C + q * NVC * 4);
                wv[kx][4 * q + 0] = f.x;
                wv[kx][4 * q + 1] = f.y;
                wv[kx][4 * q + 2] = f.z;
                wv[kx][4 * q + 3] = f.w;
              }
#pragma unroll
            for (int j = 0; j < WB; ++j) {
#pragma unroll
              for (int kx = 0; kx < K; ++kx) {
                const float* xv = v[j * S + kx * DL];
                if constexpr (MODE == kWidenFfma2) {
#pragma unroll
                  for (int e = 0; e < VEC; e += 2) {
                    const float2 r = __ffma2_rn(make_float2(xv[e], xv[e + 1]), make_float2(wv[kx][e], wv[kx][e + 1]),
                                                make_float2(acc[j][e], acc[j][e + 1]));
                    acc[j][e] = r.x;
                    acc[j][e + 1] = r.y;
                  }
                } else {
#pragma unroll
                  for (int e = 0; e < VEC; ++e) acc[j][e] = fmaf(xv[e], wv[kx][e], acc[j][e]);
                }
              }
              if (store_now && ow0 + j < a.Wo)
                epilogue_store<T, VEC>(yrow + (int64_t)(ow0 + j) * a.C, acc[j], b_s + ch);
            }
          }
        }
      }
    }

    __syncwarp();  // this warp is done with stage s
    if (lane == 0) mbar_arrive(&empty[s]);
  }
}

// 128-bit read-only global load through L1.
__device__ __forceinline__ void ldg128(const void* p, uint32_t (&v)[4]) {
  asm volatile("ld.global.nc.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
               : "l"(p));
}

// Direct-load variant of Ka: one CTA per output tile, every thread reads its
// input vectors straight from global memory (L1-cached 128-bit loads; the
// halo that neighbouring threads share is served by L1), padding by
// predication.  No shared-memory staging, so many more warps fit per SM to
// hide memory latency.  Same register blocking and epilogue as dw_kernel.
template <typename T, int K, int S, int DL, int WB, int MODE>
__global__ void __launch_bounds__(256, 2) dw_ldg_kernel(const DwArgs a) {
  constexpr int VEC = Elem<T>::kVec;
  constexpr int NCOL = (WB - 1) * S + (K - 1) * DL + 1;
  static_assert(MODE != kMixedFma || sizeof(T) == 2, "mixed-precision FMA needs 16-bit storage");
  extern __shared__ __align__(1024) uint8_t smem[];
  const int taps = a.Z * K * K;
  uint8_t* w_raw = smem;
  float* b_s = reinterpret_cast<float*>(smem + weight_smem_bytes(taps, a.TC, (int)sizeof(T), MODE));
  const int tid = threadIdx.x;
  const int NV = a.TC / VEC;
  const int nbw = a.TW / WB;
  const int items = NV * nbw * a.TH;
  const T* __restrict__ xg = static_cast<const T*>(a.x);
  const T* __restrict__ wg = static_cast<const T*>(a.w);
  const T* __restrict__ bg = static_cast<const T*>(a.bias);
  T* __restrict__ yg = static_cast<T*>(a.y);
  const TileCoord c = decode_tile(a, blockIdx.x);
  const int c0 = c.ct * a.TC;
  grid_dependency_wait();  // x, w, bias and y are touched only from here on

  // this tile's channel slice of the weights and bias
  for (int i = tid; i < taps * a.TC; i += blockDim.x) {
    const int t = i / a.TC, cl = i - t * a.TC;
    const int ch = c0 + cl;
    const T v = ch < a.C ? wg[(int64_t)ch * taps + t] : Elem<T>::from_f32(0.f);
    if constexpr (MODE == kMixedFma) {
      reinterpret_cast<T*>(w_raw)[t * a.TC + cl] = v;
    } else {
      const int cvv = cl / VEC, q = (cl % VEC) / 4, e = cl % 4;
      reinterpret_cast<float*>(w_raw)[((t * (VEC / 4) + q) * NV + cvv) * 4 + e] = Elem<T>::to_f32(v);
    }
  }
  for (int i = tid; i < a.TC; i += blockDim.x) {
    const int ch = c0 + i;
    b_s[i] = (bg != nullptr && ch < a.C) ? Elem<T>::to_f32(bg[ch]) : 0.f;
  }
  __syncthreads();

  for (int it = tid; it < items; it += blockDim.x) {
    const int cv = it % NV;
    const int blk = it / NV;
    const int oh_l = blk / nbw;
    const int ow_l = (blk - oh_l * nbw) * WB;
    const int oh = c.th * a.TH + oh_l;
    const int ch = c0 + cv * VEC;
    const int ow0 = c.tw * a.TW + ow_l;
    if (oh >= a.Ho || ch >= a.C) continue;
    T* yrow = yg + ((((int64_t)c.n * a.Do + c.od) * a.Ho + oh) * (int64_t)a.Wo) * a.C + ch;
    float acc[WB][VEC];
#pragma unroll
    for (int j = 0; j < WB; ++j)
#pragma unroll
      for (int e = 0; e < VEC; ++e) acc[j][e] = 0.f;
    const int iw0 = ow0 * S - a.pW;
    for (int z = 0; z < a.Z; ++z) {
      const int id = c.od * a.sD - a.pD + z * a.dD;
      if (id < 0 || id >= a.D) continue;
#pragma unroll
      for (int ky = 0; ky < K; ++ky) {
        const int ih = oh * S - a.pH + ky * DL;
        const bool row_ok = ih >= 0 && ih < a.H;
        const T* xrow = xg + ((((int64_t)c.n * a.D + id) * a.H + (row_ok ? ih : 0)) * (int64_t)a.W) * a.C + ch;
        uint32_t xw[NCOL][4];
#pragma unroll
        for (int cc = 0; cc < NCOL; ++cc) {
          const int iw = iw0 + cc;
          if (row_ok && iw >= 0 && iw < a.W) {
            ldg128(xrow + (int64_t)iw * a.C, xw[cc]);
          } else {
            xw[cc][0] = xw[cc][1] = xw[cc][2] = xw[cc][3] = 0u;
          }
        }
        if constexpr (MODE == kMixedFma) {
          const T* wz = reinterpret_cast<const T*>(w_raw) + (z * K * K + ky * K) * a.TC + cv * VEC;
          uint32_t ww[K][4];
#pragma unroll
          for (int kx = 0; kx < K; ++kx) lds128(wz + kx * a.TC, ww[kx]);
#pragma unroll
          for (int kx = 0; kx < K; ++kx)
#pragma unroll
            for (int j = 0; j < WB; ++j)
#pragma unroll
              for (int q = 0; q < 4; ++q)
                fma_mixed_pair<T>(xw[j * S + kx * DL][q], ww[kx][q], acc[j][2 * q], acc[j][2 * q + 1]);
        } else {
          const float* wz = reinterpret_cast<const float*>(w_raw) + (z * K * K + ky * K) * a.TC + cv * 4;
          float v[NCOL][VEC];
#pragma unroll
          for (int cc = 0; cc < NCOL; ++cc) unpack16<T>(xw[cc], v[cc]);
#pragma unroll
          for (int kx = 0; kx < K; ++kx) {
            float wv[VEC];
#pragma unroll
            for (int q = 0; q < VEC / 4; ++q) {
              const float4 f = *reinterpret_cast<const float4*>(wz + kx * a.TC + q * NV * 4);
              wv[4 * q + 0] = f.x;
              wv[4 * q + 1] = f.y;
              wv[4 * q + 2] = f.z;
              wv[4 * q + 3] = f.w;
            }
#pragma unroll
            for (int j = 0; j < WB; ++j) {
              const float* xv = v[j * S + kx * DL];
              if constexpr (MODE == kWidenFfma2) {
#pragma unroll
                for (int e = 0; e < VEC; e += 2) {
                  const float2 r = __ffma2_rn(make_float2(xv[e], xv[e + 1]), make_float2(wv[e], wv[e + 1]),
                                              make_float2(acc[j][e], acc[j][e + 1]));
                  acc[j][e] = r.x;
                  acc[j][e + 1] = r.y;
                }
              } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) acc[j][e] = fmaf(xv[e], wv[e], acc[j][e]);
              }
            }
          }
        }
      }
    }
#pragma unroll
    for (int j = 0; j < WB; ++j)
      if (ow0 + j < a.Wo) epilogue_store<T, VEC>(yrow + (int64_t)(ow0 + j) * a.C, acc[j], b_s + cv * VEC);
  }
}

}  // namespace dw
}  // namespace gconv
