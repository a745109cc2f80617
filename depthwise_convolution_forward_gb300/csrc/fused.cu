// Fused block tail on sm_103a: depthwise 3x3 (+ bias, activation) on the CUDA
// cores, 1x1 projection on the tensor cores, h kept in shared memory.
//
//   h[n, o, c]  = round(act(sum_t x[n, o*s - p + t, c] * w_dw[c, t] + b_dw[c]))
//   y[n, o, k]  = round(sum_c h[n, o, c] * w_pw[k, c] + b_pw[k])
//
// The depthwise layer is the pages' MobileNetV2 benchmark layer (TileOPs PR
// #1568, the MobileNetV2 depthwise cases); the pointwise projection and the
// activation are its neighbours in that network.  Fusing them removes the
// round trip of h through HBM.  h is rounded to the storage type exactly as a
// separate depthwise layer would store it.
//
// Design:
//  * A CTA walks tiles of TH full output rows (TH * Wo <= 128 pixels).  Warp 0
//    copies each tile's input rows with TMA, 16 channels per copy (the halo
//    and the padding come from the box reaching past the tensor: zeros), 16
//    to 64 channels per copy.
//  * Warps 1-8 compute the depthwise outputs of a chunk: thread (pixel p,
//    8-channel group) takes 8 channels of one pixel, mixed-precision FMAs
//    (16-bit pairs in, fp32 products and sums) over the 9 taps,
//    bias, activation, one round-to-nearest-even, and writes the 16 bytes
//    straight into the K-major A operand of the projection (core matrices of
//    8 pixels x 8 channels, no swizzle).
//  * Once every chunk of the tile is written, one thread issues the
//    projection: per 16 channels one tcgen05.mma (M = 128 pixels, N = K
//    rounded up to 16, K = 16), accumulating in tensor memory.
//  * Warps 1-4 (one per TMEM lane quarter) read the accumulators, add the
//    projection bias, round and store K channels per pixel.
//  * All waits are bounded.  After a timeout a CTA records it in the status
//    word and stops waiting, but still takes the same path through its
//    barriers, so no warp is left behind.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <type_traits>

#include "common.cuh"
#include "fused.h"
#include "plan_cache.h"
#include "tc_ptx.cuh"

namespace gconv {
namespace fz {

constexpr int kMaxStages = 8;
constexpr int kComputeWarps = 8;
constexpr int kThreads = 32 * (1 + kComputeWarps);

struct DwPwArgs {
  const void* w_dw;
  const void* b_dw;
  const void* w_pw;
  const void* b_pw;
  void* y;
  int C, K, Np;            // channels, projection outputs, N of the MMA (K rounded up to 16)
  int Ho, Wo, s, act;      // output extents, stride, activation
  int pH, pW;              // padding
  int TH, tiles_h, tiles;  // output rows per tile, tiles per image, tiles in total
  int Win, Hin;            // copied input columns / rows per tile
  int CH, chunks, stages;  // channels per copied chunk (16..64), chunks, copy stages
  uint32_t x_stage_bytes, x_stage_stride;  // bytes one copy lands (Win * Hin * CH * 2), stage spacing
  uint32_t wdw_off, bdw_off, bpw_off, b_off, a_off, x_off;  // shared-memory offsets
  uint32_t tmem_cols, idesc;
  int* status;
  uint64_t wait_limit_ns;
};

template <typename T>
__device__ __forceinline__ float act_f(float v, int act) {
  if (act == 1) return fmaxf(v, 0.f);
  if (act == 2) return fminf(fmaxf(v, 0.f), 6.f);
  return v;
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1) dw_pw_kernel(const __grid_constant__ CUtensorMap xmap,
                                                           const __grid_constant__ DwPwArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* x_full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* x_empty = x_full + kMaxStages;
  uint64_t* mma_bar = x_empty + kMaxStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 256);
  volatile int* failed = reinterpret_cast<volatile int*>(smem + 260);
  T* wdw = reinterpret_cast<T*>(smem + a.wdw_off);          // [C/8][9 taps][8], the storage type
  float* bdw = reinterpret_cast<float*>(smem + a.bdw_off);  // [C]
  float* bpw = reinterpret_cast<float*>(smem + a.bpw_off);  // [Np]
  uint8_t* Bs = smem + a.b_off;                              // [C/8][Np rows][16 B]
  uint8_t* As = smem + a.a_off;                              // [C/8][128 rows][16 B]
  uint8_t* Xs = smem + a.x_off;                              // stages x [Hin][Win][CH channels]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const T* __restrict__ wdg = static_cast<const T*>(a.w_dw);
  const T* __restrict__ bdg = static_cast<const T*>(a.b_dw);
  const T* __restrict__ wpg = static_cast<const T*>(a.w_pw);
  const T* __restrict__ bpg = static_cast<const T*>(a.b_pw);
  T* __restrict__ yg = static_cast<T*>(a.y);

  if (tid == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(&x_full[s], 1);
      mbar_init(&x_empty[s], kComputeWarps);
    }
    mbar_init(mma_bar, 1);
    *failed = 0;
    fence_mbar_init();
    tma_prefetch_desc(&xmap);
  }
  // Weights, biases and the projection's B operand, staged once per CTA
  // after the wait on the previous grid (they are global memory).
  grid_dependency_wait();
  for (int i = tid; i < a.C * 9; i += kThreads) {
    const int c = i / 9, t = i - c * 9;
    wdw[((c >> 3) * 9 + t) * 8 + (c & 7)] = wdg[i];
  }
  for (int i = tid; i < a.C; i += kThreads) bdw[i] = bdg ? Elem<T>::to_f32(bdg[i]) : 0.f;
  for (int i = tid; i < a.Np; i += kThreads) bpw[i] = (bpg && i < a.K) ? Elem<T>::to_f32(bpg[i]) : 0.f;
  for (int i = tid; i < (a.C / 8) * a.Np; i += kThreads) {
    const int kc = i / a.Np, n = i - kc * a.Np;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (n < a.K) v = *reinterpret_cast<const uint4*>(wpg + (int64_t)n * a.C + kc * 8);
    *reinterpret_cast<uint4*>(Bs + ((size_t)kc * a.Np + n) * 16) = v;
  }
  fence_proxy_async_smem();  // B (generic-proxy writes) -> visible to the tensor core
  if (warp == 1) {           // tensor memory only after the wait on the previous grid
    tc::tmem_alloc(tmem_slot, a.tmem_cols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ---------------- TMA producer: every (tile, chunk) in order ----------------
    if (lane == 0) {
      int k = 0;
      int last[kMaxStages];  // the last copy issued into each stage
      for (int i = 0; i < kMaxStages; ++i) last[i] = -1;
      for (int tile = blockIdx.x; tile < a.tiles; tile += gridDim.x) {
        const int n = tile / a.tiles_h, oh0 = (tile - n * a.tiles_h) * a.TH;
        for (int cc = 0; cc < a.chunks; ++cc, ++k) {
          const int s = k % a.stages;
          if (k >= a.stages && !*failed &&
              !mbar_wait(&x_empty[s], (uint32_t)(((k / a.stages) - 1) & 1), a.wait_limit_ns)) {
            report(a.status, kDevTimeout, 41);
            *failed = 1;
          }
          if (*failed) continue;
          mbar_arrive_expect_tx(&x_full[s], a.x_stage_bytes);
          // CH channels x Win columns x Hin rows from (oh0 * s - pH, -pW): the
          // halo and the padding read past the tensor's edge as zeros
          tma_load_4d(Xs + (size_t)s * a.x_stage_stride, &xmap, &x_full[s], cc * a.CH, -a.pW, oh0 * a.s - a.pH, n);
          last[s] = k;
        }
      }
      // bounded drain (also after a timeout): no copy may still be landing
      // when the CTA exits
      for (int s = 0; s < a.stages; ++s)
        if (last[s] >= 0) mbar_wait(&x_full[s], (uint32_t)((last[s] / a.stages) & 1), a.wait_limit_ns);
    }
  } else {
    // ---------------- compute warps 1..8 ----------------
    const int tcid = tid - 32;
    const int p = tcid & 127;  // pixel row of the A tile this thread computes
    const uint32_t a_base = smem_u32(As), b_base = smem_u32(Bs);
    const int g8n = a.CH / 8;  // 8-channel groups per chunk; thread takes groups tcid / 128, + 2, ...
    int k = 0, tcount = 0;
    for (int tile = blockIdx.x; tile < a.tiles; tile += gridDim.x, ++tcount) {
      const int n = tile / a.tiles_h, oh0 = (tile - n * a.tiles_h) * a.TH;
      const int rows = min(a.TH, a.Ho - oh0);
      const int npx = rows * a.Wo;
      const int ohl = p / a.Wo, ow = p - ohl * a.Wo;
      for (int cc = 0; cc < a.chunks; ++cc, ++k) {
        const int s = k % a.stages;
        if (!*failed && !mbar_wait(&x_full[s], (uint32_t)((k / a.stages) & 1), a.wait_limit_ns)) {
          report(a.status, kDevTimeout, 42);
          *failed = 1;
        }
        if (p < npx && !*failed) {
          const uint8_t* px0 = Xs + (size_t)s * a.x_stage_stride + ((size_t)(ohl * a.s) * a.Win + ow * a.s) * a.CH * 2;
          for (int g8 = tcid >> 7; g8 < g8n; g8 += 2) {
            const int kc = cc * g8n + g8;  // 8-channel group of the whole C
            const uint4* wv = reinterpret_cast<const uint4*>(wdw + (size_t)kc * 72);
            float acc[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = bdw[kc * 8 + e];
#pragma unroll
            for (int ky = 0; ky < 3; ++ky)
#pragma unroll
              for (int kx = 0; kx < 3; ++kx) {
                // 8 channels of one input pixel and of one tap's weights, 16-bit
                // pairs: fp32 products and sums with one rounding per FMA
                const uint4 u = *reinterpret_cast<const uint4*>(px0 + ((size_t)ky * a.Win + kx) * a.CH * 2 + g8 * 16);
                const uint4 wq = wv[ky * 3 + kx];
                fma_mixed_pair<T>(u.x, wq.x, acc[0], acc[1]);
                fma_mixed_pair<T>(u.y, wq.y, acc[2], acc[3]);
                fma_mixed_pair<T>(u.z, wq.z, acc[4], acc[5]);
                fma_mixed_pair<T>(u.w, wq.w, acc[6], acc[7]);
              }
            uint32_t wd[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              wd[e] = epilogue_pair<T>(act_f<T>(acc[2 * e], a.act), act_f<T>(acc[2 * e + 1], a.act), 0.f, 0.f);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a_base + (uint32_t)((kc * 128 + p) * 16)),
                         "r"(wd[0]), "r"(wd[1]), "r"(wd[2]), "r"(wd[3])
                         : "memory");
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&x_empty[s]);  // this warp's reads of the stage are done
      }
      // the tile's h is complete: projection on the tensor cores
      fence_proxy_async_smem();
      tc::fence_before_sync();
      asm volatile("bar.sync 1, %0;" ::"r"(32 * kComputeWarps) : "memory");
      if (tcid == 0) {
        tc::fence_after_sync();
        for (int ks = 0; ks < a.C / 16; ++ks) {  // one K step per 16 channels
          const uint64_t ad = tc::smem_desc(a_base + (uint32_t)ks * 4096u, 2048u, 128u);
          const uint64_t bd = tc::smem_desc(b_base + (uint32_t)(2 * ks * a.Np) * 16u, (uint32_t)a.Np * 16u, 128u);
          tc::mma_f16(tmem_base, ad, bd, a.idesc, ks > 0 ? 1u : 0u);
        }
        tc::commit(mma_bar);
      }
      if (!*failed && !mbar_wait(mma_bar, (uint32_t)(tcount & 1), a.wait_limit_ns)) {
        report(a.status, kDevTimeout, 43);
        *failed = 1;
      }
      tc::fence_after_sync();
      if (warp <= 4 && !*failed) {
        // epilogue: warp w reads TMEM lanes 32 * (w & 3) .. + 31 = pixels of those A rows
        const int q = warp & 3;
        const int pe = q * 32 + lane;
        const int eh = pe / a.Wo, ew = pe - eh * a.Wo;
        T* dst = yg + (((int64_t)n * a.Ho + oh0 + eh) * a.Wo + ew) * a.K;
        for (int c0 = 0; c0 < a.Np; c0 += 16) {
          uint32_t r[16];
          tc::tmem_ld16(tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)c0, r);
          tc::tmem_ld_wait();
          if (pe < npx) {
#pragma unroll
            for (int h8 = 0; h8 < 16; h8 += 8) {
              if (c0 + h8 < a.K) {
                uint32_t wd[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                  wd[e] = epilogue_pair<T>(__uint_as_float(r[h8 + 2 * e]), __uint_as_float(r[h8 + 2 * e + 1]),
                                           bpw[c0 + h8 + 2 * e], bpw[c0 + h8 + 2 * e + 1]);
                *reinterpret_cast<uint4*>(dst + c0 + h8) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
              }
            }
          }
        }
      }
      // the accumulators and A are free for the next tile
      tc::fence_before_sync();
      asm volatile("bar.sync 1, %0;" ::"r"(32 * kComputeWarps) : "memory");
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem_base, a.tmem_cols);
  }
}

}  // namespace fz

namespace {

inline uint32_t round_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

struct DwPwPlan {
  fz::DwPwArgs a;
  uint32_t smem_bytes;
};

bool make_dw_pw_plan(const Geometry& g, bool bf16, int K, int act, int max_smem, DwPwPlan* out) {
  (void)bf16;
  if (g.ndim != 2 || g.Cg != 1 || g.Kg != 1 || g.Z != 1 || g.Y != 3 || g.X != 3) return false;
  if (g.dH != 1 || g.dW != 1 || g.sH != g.sW || g.sH < 1 || g.sH > 2) return false;
  const int C = g.C();
  if (C % 16 != 0 || C > 256 || K % 8 != 0 || K < 8 || K > 256 || act < 0 || act > 2) return false;
  if (g.Wo < 1 || g.Wo > 128 || g.Ho < 1) return false;
  fz::DwPwArgs a;
  std::memset(&a, 0, sizeof(a));
  a.C = C, a.K = K, a.Np = (K + 15) / 16 * 16;
  a.Ho = g.Ho, a.Wo = g.Wo, a.s = g.sH, a.act = act, a.pH = g.pH, a.pW = g.pW;
  a.TH = std::min(g.Ho, 128 / g.Wo);
  a.tiles_h = (g.Ho + a.TH - 1) / a.TH;
  const int64_t tiles = g.N * (int64_t)a.tiles_h;
  if (tiles >= (1ll << 31)) return false;
  a.tiles = (int)tiles;
  a.Win = (g.Wo - 1) * a.s + 3;
  a.Hin = (a.TH - 1) * a.s + 3;
  if (a.Win > 256 || a.Hin > 256) return false;
  // the largest copy chunk of 64, 48, 32 or 16 channels dividing C
  a.CH = C % 64 == 0 ? 64 : C % 48 == 0 ? 48 : C % 32 == 0 ? 32 : 16;
  a.chunks = C / a.CH;
  a.x_stage_bytes = (uint32_t)(a.Win * a.Hin * a.CH) * 2u;
  a.x_stage_stride = round_up(a.x_stage_bytes, 1024);
  a.wdw_off = 1024;
  a.bdw_off = a.wdw_off + (uint32_t)C * 9u * 2u;
  a.bpw_off = a.bdw_off + (uint32_t)C * 4u;
  a.b_off = round_up(a.bpw_off + (uint32_t)a.Np * 4u, 1024);
  a.a_off = round_up(a.b_off + (uint32_t)(C / 8) * (uint32_t)a.Np * 16u, 1024);
  a.x_off = round_up(a.a_off + (uint32_t)(C / 8) * 128u * 16u, 1024);
  const uint32_t budget = (uint32_t)std::min(max_smem, 227 * 1024);
  if (a.x_off + 2 * a.x_stage_stride > budget) return false;
  // up to 4 stages; as many as keep two CTAs on an SM (113 KB each) when two
  // fit at all, else as many as one CTA holds
  const uint32_t two = 113u * 1024u;
  a.stages = a.x_off + 2 * a.x_stage_stride <= two ? (int)((two - a.x_off) / a.x_stage_stride)
                                                    : (int)((budget - a.x_off) / a.x_stage_stride);
  a.stages = std::min(a.stages, 4);
  a.tmem_cols = 32;
  while (a.tmem_cols < (uint32_t)a.Np) a.tmem_cols <<= 1;
  a.idesc = tc::idesc_f16(bf16, 128, a.Np);
  DwPwPlan p;
  p.a = a;
  p.smem_bytes = a.x_off + (uint32_t)a.stages * a.x_stage_stride;
  *out = p;
  return true;
}

template <typename T>
cudaError_t dw_pw_launch_typed(const Geometry& g, const LaunchArgs& la, const void* w_pw, const void* b_pw, int K,
                               int act, const DeviceInfo& dev) {
  DwPwPlan p;
  if (!make_dw_pw_plan(g, std::is_same<T, __nv_bfloat16>::value, K, act, dev.max_smem_optin, &p))
    return cudaErrorNotSupported;
  const uintptr_t al = reinterpret_cast<uintptr_t>(la.x) | reinterpret_cast<uintptr_t>(la.y) |
                       reinterpret_cast<uintptr_t>(w_pw);
  if (al & 15) return cudaErrorNotSupported;
  static SmemAttr attr;
  cudaError_t e = attr.ensure(fz::dw_pw_kernel<T>, dev.device, (int)p.smem_bytes);
  if (e != cudaSuccess) return e;
  // all of the SM's unified memory as shared memory, so two CTAs fit (the
  // occupancy query below follows this preference)
  e = cudaFuncSetAttribute(fz::dw_pw_kernel<T>, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  // x as (C, W, H, N): CH channels x Win columns x Hin rows per copy
  const uint64_t es = sizeof(T), C = g.C();
  CUtensorMap xmap;
  uint64_t dims[4] = {C, (uint64_t)g.W, (uint64_t)g.H, (uint64_t)g.N};
  uint64_t strides[3] = {C * es, C * es * g.W, C * es * g.W * g.H};
  uint32_t box[4] = {(uint32_t)p.a.CH, (uint32_t)p.a.Win, (uint32_t)p.a.Hin, 1u};
  uint32_t estr[4] = {1u, 1u, 1u, 1u};
  CUtensorMapDataType tt = std::is_same<T, __half>::value ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                          : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (encode_tiled(&xmap, tt, 4, la.x, dims, strides, box, estr) != CUDA_SUCCESS) return cudaErrorInvalidValue;
  fz::DwPwArgs a = p.a;
  a.w_dw = la.w;
  a.b_dw = la.bias;
  a.w_pw = w_pw;
  a.b_pw = b_pw;
  a.y = la.y;
  a.status = la.status;
  a.wait_limit_ns = la.wait_limit_ns;
  int occ = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fz::dw_pw_kernel<T>, fz::kThreads, p.smem_bytes);
  if (e != cudaSuccess) return e;
  occ = std::max(1, std::min(occ, 512 / (int)p.a.tmem_cols));
  const int grid = std::max(1, std::min(a.tiles, dev.num_sms * occ));
  return launch_kernel(fz::dw_pw_kernel<T>, dim3(grid), dim3(fz::kThreads), p.smem_bytes, la, xmap, a);
}

}  // namespace

bool dw_pw_supported(const Geometry& g, DType dt, int K, int act) {
  if (dt == kF32) return false;
  DwPwPlan p;
  return make_dw_pw_plan(g, dt == kBF16, K, act, kDefaultSmemOptin, &p);
}

cudaError_t dw_pw_launch(const Geometry& g, const LaunchArgs& a, const void* w_pw, const void* b_pw, int K, int act,
                         const DeviceInfo& dev) {
  if (a.dt == kF16) return dw_pw_launch_typed<__half>(g, a, w_pw, b_pw, K, act, dev);
  if (a.dt == kBF16) return dw_pw_launch_typed<__nv_bfloat16>(g, a, w_pw, b_pw, K, act, dev);
  return cudaErrorNotSupported;
}

}  // namespace gconv
