// Kb: grouped implicit GEMM on the 5th-generation tensor cores.
//
// Per group chunk (m consecutive groups merged into one block-diagonal GEMM)
// and per filter tap t the convolution is the GEMM
//     D[pixel, n] += A_t[pixel, k] * B_t[n, k]
// with k over the chunk's m*Cg input channels, n over its m*Kg output
// channels, A_t the input shifted by the tap's offset and B_t the weights of
// tap t (zero outside the diagonal group blocks).  The pages describe the
// same decomposition for an implicit-GEMM convolution with grouped channel
// decode and a group grid axis (rocm-libraries PR #10064, Technical Details)
// and the merging of small groups into one tile (CK grouped-conv examples,
// Config-options harness, num_groups_to_merge).
//
// sm_103a design:
//  * A CTA owns one group chunk and walks spatial tiles of TH x TWo outputs.
//  * Warp 0 (one lane) copies the tile's haloed input with TMA into
//    "planes": for every stride phase and every 8-channel chunk, the halo
//    pixels in row-major order, 16 bytes each.  That is exactly the
//    no-swizzle K-major core-matrix layout (8 rows x 16 bytes), so the A
//    operand of tap t is the same planes read from a pixel offset: the tap's
//    shift is a descriptor start address.  Rows are flattened over the halo
//    pitch; the (pitch - TWo) wrap-around rows per output row are computed
//    and discarded.  Stride 2 uses four polyphase planes loaded with TMA
//    element strides, so every tap is again a plain shift.
//  * Warp 1 (one lane) issues tcgen05.mma (M = 128, N = m*Kg, K = 16) into
//    fp32 accumulators in tensor memory, double-buffered across tiles, and
//    signals completion with tcgen05.commit on mbarriers.
//  * Warps 2-5 read the accumulators (tcgen05.ld), apply the fused bias +
//    round-to-nearest-even epilogue and store channels-last output.
//  * All waits are bounded; on expiry every role reports a timeout, waits
//    (bounded) for its in-flight copies / MMAs, and the CTA frees its tensor
//    memory before exiting.
#pragma once

#include "tc_ptx.cuh"

namespace gconv {
namespace tc {

constexpr int kMaxTaps = 32;
constexpr int kMaxPhases = 4;
constexpr int kMaxStages = 4;
constexpr int kThreads = 192;

struct TcArgs {
  const void* w;
  const void* bias;
  void* y;
  int G, Cg, Kg, m;        // groups, channels per group, merge factor
  int Do, Ho, Wo, Ktot;    // output extents, output channels
  int sD, pD, taps_total;  // depth stride / pad, taps per filter
  int TH, TWo, P, Hh, Dh;  // tile rows / cols, halo pitch, halo rows, halo planes
  int s, qy_min, qx_min;   // spatial stride, phase-row origin offsets
  int nphase;
  int phase_py[kMaxPhases], phase_px[kMaxPhases];
  int ntaps;
  int tap_phase[kMaxTaps], tap_off[kMaxTaps];
  int nchunks, Kt, Nn, KS, nmt;
  uint32_t plane_stride, a_stage_bytes, tx_bytes;
  uint32_t a_off, b_off, bias_off;
  int stages;
  uint32_t tmem_cols, idesc;
  int n_gc, cpg, tiles_w, tiles_h;
  int spatial_tiles;
  int* status;
  uint64_t wait_limit_ns;
  int test_flags;
};

struct SpatialTile {
  int n, od, oh0, ow0;
};

__device__ __forceinline__ SpatialTile decode_spatial(const TcArgs& a, int sp) {
  SpatialTile t;
  const int tw = sp % a.tiles_w;
  sp /= a.tiles_w;
  const int th = sp % a.tiles_h;
  sp /= a.tiles_h;
  t.od = sp % a.Do;
  t.n = sp / a.Do;
  t.oh0 = th * a.TH;
  t.ow0 = tw * a.TWo;
  return t;
}

// All lanes of a warp wait on `bar`: lane 0 polls (bounded), then every lane
// observes the completed phase itself.  Returns false on timeout.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, uint64_t limit) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, limit);
  ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  if (ok && (threadIdx.x & 31) != 0) ok = mbar_wait(bar, parity, limit);
  return __all_sync(0xffffffffu, ok);
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1) tc_kernel(const __grid_constant__ CUtensorMap xmap, const TcArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* a_full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* a_empty = a_full + kMaxStages;
  uint64_t* acc_full = a_full + 2 * kMaxStages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* mma_done = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 256);
  float* bias_s = reinterpret_cast<float*>(smem + a.bias_off);
  uint8_t* Bs = smem + a.b_off;
  uint8_t* As = smem + a.a_off;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gc = blockIdx.x % a.n_gc;
  const int cta_in_gc = blockIdx.x / a.n_gc;
  const int g0 = gc * a.m;
  const T* __restrict__ wg = static_cast<const T*>(a.w);
  const T* __restrict__ bg = static_cast<const T*>(a.bias);
  T* __restrict__ yg = static_cast<T*>(a.y);

  if (tid == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(&a_full[s], 1);
      mbar_init(&a_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);
    }
    mbar_init(mma_done, 1);
    fence_mbar_init();
    tma_prefetch_desc(&xmap);
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, a.tmem_cols);
    tmem_relinquish();
  }
  // Weights of this group chunk as block-diagonal B_t[n][k], K-major core
  // matrices: byte offset ((((t*KS + ks)*2 + kc2)*Nn + n)*8 + e)*2 holds
  // k = ks*16 + kc2*8 + e.
  {
    const int per_tap = a.Kt * a.Nn;
    const int total = a.ntaps * per_tap;
    T* B = reinterpret_cast<T*>(Bs);
    for (int i = tid; i < total; i += blockDim.x) {
      const int t = i / per_tap;
      int r = i - t * per_tap;
      const int e = r & 7;
      r >>= 3;
      const int n = r % a.Nn;
      r /= a.Nn;
      const int kc2 = r & 1;
      const int ks = r >> 1;
      const int k = ks * 16 + kc2 * 8 + e;
      const int gj = k / a.Cg, cc = k - gj * a.Cg;
      const int gi = n / a.Kg, kk = n - gi * a.Kg;
      T v = Elem<T>::from_f32(0.f);
      if (gi == gj)
        v = wg[((int64_t)(g0 + gi) * a.Kg + kk) * a.taps_total * a.Cg + (int64_t)t * a.Cg + cc];
      B[i] = v;
    }
    for (int i = tid; i < a.Nn; i += blockDim.x)
      bias_s[i] = bg != nullptr ? Elem<T>::to_f32(bg[(int64_t)g0 * a.Kg + i]) : 0.f;
  }
  fence_proxy_async_smem();  // generic-proxy writes of B -> visible to the tensor core
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  const bool withhold = (a.test_flags & 1) && blockIdx.x == 0;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      int k = 0;
      bool failed = false;
      for (int sp = cta_in_gc; sp < a.spatial_tiles; sp += a.cpg, ++k) {
        const int s = k % a.stages;
        if (k >= a.stages && !mbar_wait(&a_empty[s], (uint32_t)(((k / a.stages) - 1) & 1), a.wait_limit_ns)) {
          failed = true;
          break;
        }
        if (withhold && k == 0) continue;
        const SpatialTile st = decode_spatial(a, sp);
        const int id0 = st.od * a.sD - a.pD;
        mbar_arrive_expect_tx(&a_full[s], a.tx_bytes);
        uint8_t* stage = As + (size_t)s * a.a_stage_bytes;
        for (int ph = 0; ph < a.nphase; ++ph) {
          const int ih0 = a.s * (st.oh0 + a.qy_min) + a.phase_py[ph];
          const int iw0 = a.s * (st.ow0 + a.qx_min) + a.phase_px[ph];
          for (int c = 0; c < a.nchunks; ++c)
            tma_load_5d(stage + (size_t)(ph * a.nchunks + c) * a.plane_stride, &xmap, &a_full[s],
                        g0 * a.Cg + c * 8, iw0, ih0, id0, st.n);
        }
      }
      if (failed) report(a.status, kDevTimeout, 3);
      for (int j = k > a.stages ? k - a.stages : 0; j < k; ++j) {  // bounded drain
        if (withhold && j == 0) continue;
        mbar_wait(&a_full[j % a.stages], (uint32_t)((j / a.stages) & 1), a.wait_limit_ns);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      int k = 0;
      bool failed = false;
      const uint32_t b_base = smem_u32(Bs);
      const uint32_t lbo_b = (uint32_t)a.Nn * 16u;
      for (int sp = cta_in_gc; sp < a.spatial_tiles; sp += a.cpg, ++k) {
        const int s = k % a.stages;
        const int ab = k & 1;
        if (!mbar_wait(&a_full[s], (uint32_t)((k / a.stages) & 1), a.wait_limit_ns)) {
          failed = true;
          break;
        }
        if (k >= 2 && !mbar_wait(&acc_empty[ab], (uint32_t)(((k >> 1) - 1) & 1), a.wait_limit_ns)) {
          failed = true;
          break;
        }
        fence_after_sync();
        const uint32_t a_base = smem_u32(As + (size_t)s * a.a_stage_bytes);
        for (int mt = 0; mt < a.nmt; ++mt) {
          const uint32_t d = tmem_base + (uint32_t)((ab * a.nmt + mt) * a.Nn);
          for (int t = 0; t < a.ntaps; ++t) {
            const uint32_t plane0 = a_base + (uint32_t)(a.tap_phase[t] * a.nchunks) * a.plane_stride;
            const uint32_t row0 = (uint32_t)(mt * 128 + a.tap_off[t]) * 16u;
            for (int ks = 0; ks < a.KS; ++ks) {
              const uint64_t adesc = smem_desc(plane0 + (uint32_t)(2 * ks) * a.plane_stride + row0, a.plane_stride, 128u);
              const uint64_t bdesc = smem_desc(b_base + (uint32_t)((t * a.KS + ks) * 2) * lbo_b, lbo_b, 128u);
              mma_f16(d, adesc, bdesc, a.idesc, (t | ks) != 0 ? 1u : 0u);
            }
          }
        }
        commit(&a_empty[s]);   // stage reusable once these MMAs have read it
        commit(&acc_full[ab]);  // accumulators of this tile complete
      }
      if (failed) report(a.status, kDevTimeout, 4);
      commit(mma_done);  // every MMA issued so far has completed
      mbar_wait(mma_done, 0, a.wait_limit_ns);
    }
  } else {
    // ---------------- epilogue (warps 2..5) ----------------
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;
    int k = 0;
    for (int sp = cta_in_gc; sp < a.spatial_tiles; sp += a.cpg, ++k) {
      const int ab = k & 1;
      if (!warp_wait(&acc_full[ab], (uint32_t)((k >> 1) & 1), a.wait_limit_ns)) {
        if (lane == 0) report(a.status, kDevTimeout, 5);
        break;
      }
      fence_after_sync();
      const SpatialTile st = decode_spatial(a, sp);
      for (int mt = 0; mt < a.nmt; ++mt) {
        const int f = mt * 128 + row;
        const int i = f / a.P, j = f - i * a.P;
        const int oh = st.oh0 + i, ow = st.ow0 + j;
        const bool valid = i < a.TH && j < a.TWo && oh < a.Ho && ow < a.Wo;
        T* dst = yg + ((((int64_t)st.n * a.Do + st.od) * a.Ho + oh) * (int64_t)a.Wo + ow) * a.Ktot +
                 (int64_t)g0 * a.Kg;
        const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)((ab * a.nmt + mt) * a.Nn);
        for (int c0 = 0; c0 < a.Nn; c0 += 16) {
          uint32_t r[16];
          tmem_ld16(taddr + (uint32_t)c0, r);
          tmem_ld_wait();
          if (valid) {
            float v[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] = __uint_as_float(r[e]);
            epilogue_store<T, 8>(dst + c0, v, bias_s + c0);
            epilogue_store<T, 8>(dst + c0 + 8, v + 8, bias_s + c0 + 8);
          }
        }
      }
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[ab]);
    }
  }
  __syncwarp();
  fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    fence_after_sync();
    tmem_dealloc(tmem_base, a.tmem_cols);
  }
}

}  // namespace tc
}  // namespace gconv
