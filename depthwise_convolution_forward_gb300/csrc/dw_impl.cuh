// Ka: depthwise direct kernel (Cg == Kg == 1), bandwidth-bound.
//
// Design (sm_103a):
//  * Persistent CTAs walk a static list of output tiles
//    (n, od, TH x TW output pixels, TC channels).
//  * For each tile one thread issues a single 5-D TMA copy of the haloed input
//    box [1 x Dh x Hh x Wh x TC] (NDHWC order) into a shared-memory stage.
//    TMA zero-fills coordinates outside the tensor, which is exactly the
//    convolution's zero padding, so the compute loop has no bounds checks.
//  * Stages form a ring completed through mbarriers: while the CTA computes
//    tile k, the copies for tiles k+1 .. k+stages-1 are in flight.
//  * Each thread owns one 16-byte channel vector (8 x f16/bf16 or 4 x f32) of
//    a 1 x WB strip of outputs.  It reads each needed input vector of an input
//    row once into registers and reuses it across the WB outputs and the K
//    horizontal taps (register blocking), accumulates in fp32, and finishes
//    with the fused bias + round-to-nearest-even cast (Kc) and a 16-byte store.
//  * Every mbarrier wait is bounded; on expiry the CTA reports a timeout in
//    the status word, waits (bounded) for copies still in flight and exits.
#pragma once

#include "common.cuh"

namespace gconv {
namespace dw {

struct DwArgs {
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
  int* status;
  uint64_t wait_limit_ns;
  int test_flags;
};

struct TileCoord {
  int ct, tw, th, od;
  int64_t n;
};

__device__ __forceinline__ TileCoord decode_tile(const DwArgs& a, int64_t t) {
  TileCoord c;
  c.ct = (int)(t % a.tiles_c);
  t /= a.tiles_c;
  c.tw = (int)(t % a.tiles_w);
  t /= a.tiles_w;
  c.th = (int)(t % a.tiles_h);
  t /= a.tiles_h;
  c.od = (int)(t % a.Do);
  c.n = t / a.Do;
  return c;
}

// Shared-memory layout: [mbarriers 64 B][weights fp32 taps x TC][bias fp32 TC] ... [stages]
template <int K>
__host__ __device__ inline uint32_t fixed_smem_bytes(int Z, int TC) {
  return 64u + 4u * (uint32_t)(Z * K * K * TC + TC);
}

template <typename T, int K, int S, int DL, int WB>
__global__ void __launch_bounds__(WB == 8 ? 256 : 512, 1) dw_kernel(const __grid_constant__ CUtensorMap xmap,
                                                    const DwArgs a) {
  constexpr int VEC = Elem<T>::kVec;
  constexpr int NR = (K - 1) * DL + 1;               // input rows per output row
  constexpr int NCOL = (WB - 1) * S + (K - 1) * DL + 1;  // input columns per WB outputs
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  float* w_s = reinterpret_cast<float*>(smem + 64);
  const int taps = a.Z * K * K;
  float* b_s = w_s + taps * a.TC;
  uint8_t* stage0 = smem + a.stage_off;

  const int tid = threadIdx.x;
  const int NV = a.TC / VEC;
  const int nbw = a.TW / WB;
  const int items = NV * nbw * a.TH;
  const T* __restrict__ wg = static_cast<const T*>(a.w);
  const T* __restrict__ bg = static_cast<const T*>(a.bias);
  T* __restrict__ yg = static_cast<T*>(a.y);

  if (tid == 0) {
    for (int s = 0; s < a.stages; ++s) mbar_init(&full[s], 1);
    fence_mbar_init();
    tma_prefetch_desc(&xmap);
  }
  __syncthreads();

  auto issue = [&](int64_t tile, int s) {
    const TileCoord c = decode_tile(a, tile);
    const int c0 = c.ct * a.TC;
    const int iw0 = c.tw * a.TW * S - a.pW;
    const int ih0 = c.th * a.TH * S - a.pH;
    const int id0 = c.od * a.sD - a.pD;
    mbar_arrive_expect_tx(&full[s], a.stage_bytes);
    tma_load_5d(stage0 + (size_t)s * a.stage_stride, &xmap, &full[s], c0, iw0, ih0, id0, (int)c.n);
  };

  const bool withhold = (a.test_flags & 1) && blockIdx.x == 0;
  if (tid == 0) {
    for (int s = 0; s < a.stages; ++s) {
      const int64_t t = blockIdx.x + (int64_t)s * gridDim.x;
      if (t < a.num_tiles && !(withhold && s == 0)) issue(t, s);
    }
  }

  int cur_ct = -1;
  for (int64_t k = 0;; ++k) {
    const int64_t tile = blockIdx.x + k * gridDim.x;
    if (tile >= a.num_tiles) break;
    const int s = (int)(k % a.stages);
    const uint32_t parity = (uint32_t)((k / a.stages) & 1);
    const TileCoord c = decode_tile(a, tile);
    const int c0 = c.ct * a.TC;

    if (c.ct != cur_ct) {  // same decision in every thread of the CTA
      __syncthreads();
      for (int i = tid; i < taps * a.TC; i += blockDim.x) {
        const int t = i / a.TC, cl = i - t * a.TC;
        const int ch = c0 + cl;
        w_s[i] = ch < a.C ? Elem<T>::to_f32(wg[(int64_t)ch * taps + t]) : 0.f;
      }
      for (int i = tid; i < a.TC; i += blockDim.x) {
        const int ch = c0 + i;
        b_s[i] = (bg != nullptr && ch < a.C) ? Elem<T>::to_f32(bg[ch]) : 0.f;
      }
      __syncthreads();
      cur_ct = c.ct;
    }

    const bool ok = mbar_wait(&full[s], parity, a.wait_limit_ns);
    if (__syncthreads_or(!ok)) {
      if (tid == 0) {
        report(a.status, kDevTimeout, 1);
        // Bounded drain of every copy this CTA may still have in flight.
        for (int j = 0; j < a.stages; ++j) {
          const int64_t kk = k + j;
          if (blockIdx.x + kk * gridDim.x >= a.num_tiles) break;
          if (withhold && kk == 0) continue;
          mbar_wait(&full[kk % a.stages], (uint32_t)((kk / a.stages) & 1), a.wait_limit_ns);
        }
      }
      return;
    }

    const T* st = reinterpret_cast<const T*>(stage0 + (size_t)s * a.stage_stride);
    const int plane_elems = a.Hh * a.Wh * a.TC;
    for (int it = tid; it < items; it += blockDim.x) {
      const int cv = it % NV;
      const int blk = it / NV;
      const int oh_l = blk / nbw;
      const int ow_l = (blk - oh_l * nbw) * WB;
      float acc[WB][VEC];
#pragma unroll
      for (int j = 0; j < WB; ++j)
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[j][e] = 0.f;

      for (int z = 0; z < a.Z; ++z) {
        const T* plane = st + (size_t)(z * a.dD) * plane_elems;
        const float* wz = w_s + (z * K * K) * a.TC + cv * VEC;
#pragma unroll
        for (int ky = 0; ky < K; ++ky) {
          const T* rowp = plane + ((size_t)(oh_l * S + ky * DL) * a.Wh + ow_l * S) * a.TC + cv * VEC;
          float v[NCOL][VEC];
#pragma unroll
          for (int cc = 0; cc < NCOL; ++cc)
            unpack16<T>(*reinterpret_cast<const uint4*>(rowp + cc * a.TC), v[cc]);
#pragma unroll
          for (int kx = 0; kx < K; ++kx) {
            float wv[VEC];
            const float* wp = wz + (ky * K + kx) * a.TC;
#pragma unroll
            for (int q = 0; q < VEC / 4; ++q) {
              const float4 f = *reinterpret_cast<const float4*>(wp + 4 * q);
              wv[4 * q + 0] = f.x;
              wv[4 * q + 1] = f.y;
              wv[4 * q + 2] = f.z;
              wv[4 * q + 3] = f.w;
            }
#pragma unroll
            for (int j = 0; j < WB; ++j)
#pragma unroll
              for (int e = 0; e < VEC; ++e) acc[j][e] = fmaf(v[j * S + kx * DL][e], wv[e], acc[j][e]);
          }
        }
      }

      const int oh = c.th * a.TH + oh_l;
      const int ch = c0 + cv * VEC;
      if (oh < a.Ho && ch < a.C) {
        T* yrow = yg + (((c.n * a.Do + c.od) * a.Ho + oh) * (int64_t)a.Wo) * a.C + ch;
#pragma unroll
        for (int j = 0; j < WB; ++j) {
          const int ow = c.tw * a.TW + ow_l + j;
          if (ow < a.Wo) epilogue_store<T, VEC>(yrow + (int64_t)ow * a.C, acc[j], b_s + cv * VEC);
        }
      }
    }

    __syncthreads();  // every thread is done with stage s
    if (tid == 0) {
      const int64_t nt = tile + (int64_t)a.stages * gridDim.x;
      if (nt < a.num_tiles) issue(nt, s);
    }
  }
}

}  // namespace dw
}  // namespace gconv
