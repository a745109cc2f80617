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
// Design (one persistent CTA per SM, warp-specialised):
//  * Output tiles of TH rows x TW columns (TW <= 16, TH * TW <= 128 pixels),
//    walked round-robin by the CTAs.  Warp 0 copies each tile's haloed input
//    box with TMA (all C channels in one copy, or in CH-channel chunks when
//    that keeps two tiles in flight); reads past the tensor's edge fill with
//    zeros, which is the convolution's zero padding.
//  * Compute warps 6-13: a thread owns one tile column and one 8-channel
//    group and walks down the column, loading each input row once (three
//    16-byte loads, the horizontal taps) and adding it into every output row
//    that uses it (three live rows at stride 1, two at stride 2).  Its 9 x 8
//    weights stay in registers.  Lanes run over the channel groups first, so
//    a warp's loads are consecutive 16-byte pieces of one shared-memory row.
//    Mixed-precision FMAs (16-bit operands, fp32 products and sums), bias,
//    activation, one round-to-nearest-even, and each output pixel's 8
//    channels go as one 16-byte store into the projection's A operand:
//    pixel-major rows of 128-byte-swizzled K atoms (64 channels), the layout
//    a TMA copy with 128-byte swizzle would have written, so the stores of a
//    warp spread over all banks.
//  * Warp 1 issues the projection (one tcgen05.mma per 16 channels, M = 128
//    pixel rows, N = K rounded up to 16) into one of two TMEM accumulators.
//  * Warps 2-5 (one per TMEM lane quarter) read the accumulators, add the
//    projection bias, round and store K channels per pixel.
//  * A and the accumulators are double-buffered (A single when shared memory
//    is short), so copies, depthwise math, MMAs and stores of neighbouring
//    tiles overlap.  All waits are bounded; after a timeout a CTA records it
//    in the status word, skips the remaining work and still reaches its exit.
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
constexpr int kMaxA = 3;  // A buffers (barriers: 2 x 8 stages + 2 x 3 + 2 x 2 = 26 words of the first 256 bytes)
constexpr int kMmaWarp = 1;
constexpr int kEpiWarp0 = 2, kEpiWarps = 4;
constexpr int kComputeWarp0 = 6;
// Compute warps per CTA for CP channels per compute thread: 8 channels (one
// 16-byte load per tap, 9 x 4 weight words in registers) with 8 compute
// warps, or 4 channels (8-byte loads, half the registers) with 16.
template <int CP>
struct Cfg {
  static constexpr int kComputeWarps = CP == 8 ? 8 : 16;
  static constexpr int kComputeThreads = 32 * kComputeWarps;
  static constexpr int kThreads = 32 * (kComputeWarp0 + kComputeWarps);
};
constexpr uint32_t kAtomBytes = 128u * 128u;  // one 64-channel K atom of 128 pixel rows (128-byte swizzle)
// One 8-channel group of the A tail: 128 pixel rows x 16 bytes (no swizzle),
// plus 16 bytes so consecutive groups start one bank chunk apart (the
// groups' stores from one warp then fall in different banks; the MMA reads
// the group stride as its K-direction core-matrix stride).
constexpr uint32_t kTailGroupBytes = 128u * 16u + 16u;

struct DwPwArgs {
  const void* w_dw;
  const void* b_dw;
  const void* w_pw;
  const void* b_pw;
  void* y;
  int C, K, Np, G, GT, cpt;             // channels, projection outputs, N of the MMA (K rounded up to 16), C / 8,
                                        // C / cpt (the compute threads' channel groups), channels per thread
  int Ho, Wo, act;                      // output extents, activation
  int pH, pW;                           // padding
  int TH, TW, tiles_h, tiles_w, tiles;  // tile = TH rows x TW columns; tiles down / across an image; in total
  int Win, Hin;                         // input box columns / rows per tile
  int CH, GC, chunks, stages, nA;       // channels per copy, its cpt-channel groups, copies per tile, ring, A buffers
  int NS, rps;                          // segments a column walk is split into, output rows per segment
  int inline_mma;                       // the compute warp that completes a tile's A issues its MMAs
  uint32_t x_stage_bytes, x_stage_stride, a_bytes;
  uint32_t wdw_off, bdw_off, bpw_off, b_off, a_off, x_off;  // shared-memory offsets
  uint32_t tmem_cols, idesc;
  int* status;
  uint64_t wait_limit_ns;
};

// Two values rounded to nearest-even into one word (low half = first).
template <typename T>
__device__ __forceinline__ uint32_t pack_pair(float a, float b);
template <>
__device__ __forceinline__ uint32_t pack_pair<__half>(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}
template <>
__device__ __forceinline__ uint32_t pack_pair<__nv_bfloat16>(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// The same MMA issued by one lane of the converged issuing warp (elect.sync
// picks it); every lane executes this with the same operands.
__device__ __forceinline__ void mma_f16_elect(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t.reg .b32 r;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "elect.sync r|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}
// commit() by the elected lane (the one that issued the warp's MMAs).
__device__ __forceinline__ void commit_elect(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t.reg .b32 r;\n\t"
      "elect.sync r|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}

// CP consecutive channels (CP / 2 words of 16-bit pairs) of one pixel or
// one tap, loaded from shared memory as one 8- or 16-byte access.
template <int CP>
struct Vec {
  uint32_t w[CP / 2];
};
template <int CP>
__device__ __forceinline__ Vec<CP> ld_vec(const uint8_t* p) {
  Vec<CP> v;
  if constexpr (CP == 8) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    v.w[0] = u.x, v.w[1] = u.y, v.w[2] = u.z, v.w[3] = u.w;
  } else {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    v.w[0] = u.x, v.w[1] = u.y;
  }
  return v;
}

// acc[0..CP-1] (+)= one input row's three horizontal taps xr x the filter
// row's weights wr[0..2] (16-bit pairs; fp32 products and sums).
template <typename T, int CP>
__device__ __forceinline__ void add_row(float (&acc)[CP], const Vec<CP> (&xr)[3], const Vec<CP>* wr) {
#pragma unroll
  for (int kx = 0; kx < 3; ++kx)
#pragma unroll
    for (int e = 0; e < CP / 2; ++e) fma_mixed_pair<T>(xr[kx].w[e], wr[kx].w[e], acc[2 * e], acc[2 * e + 1]);
}

// Activation and rounding of one output pixel's CP channels (the bias is
// already in acc), stored at shared address addr.  act != 0 clamps to
// [0, hi] (hi = 6 for ReLU6, infinity for ReLU).
template <typename T, int CP>
__device__ __forceinline__ void put_h(uint32_t addr, float (&acc)[CP], int act, float hi) {
  if (act) {
#pragma unroll
    for (int e = 0; e < CP; ++e) acc[e] = fminf(fmaxf(acc[e], 0.f), hi);
  }
  uint32_t wd[CP / 2];
#pragma unroll
  for (int e = 0; e < CP / 2; ++e) wd[e] = pack_pair<T>(acc[2 * e], acc[2 * e + 1]);
  if constexpr (CP == 8)
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(wd[0]), "r"(wd[1]), "r"(wd[2]),
                 "r"(wd[3])
                 : "memory");
  else
    asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(addr), "r"(wd[0]), "r"(wd[1]) : "memory");
}

// A holds the channels of whole 64-channel atoms in the 128-byte-swizzled
// K-major layout and the remaining C % 64 channels (the tail) in the plain
// K-major layout of 8-row x 16-byte core matrices, so it takes no more room
// than C channels need.  Shared address of pixel row p, 8-channel group g8,
// byte offset half (0 or 8: the second 4 channels of the group): gbase = the
// group's atom (or tail group) base, swz = whether g8 lies in a swizzled atom.
//   swizzled: 8-row block p / 8 (1024 B), row p % 8 (128 B), 16-byte chunk (g8 ^ p) % 8
//   tail:     8-row block p / 8 (128 B), row p % 8 (16 B)
__device__ __forceinline__ uint32_t a_addr(uint32_t gbase, bool swz, int p, int g8, uint32_t half) {
  return half + (swz ? gbase + (uint32_t)(p >> 3) * 1024u + (uint32_t)(p & 7) * 128u + ((uint32_t)((g8 ^ p) & 7) << 4)
                     : gbase + (uint32_t)(p >> 3) * 128u + (uint32_t)(p & 7) * 16u);
}

// Where a walk's outputs go: A row p = j * TW + w of 8-channel group g8 (at
// byte offset half inside it).
struct AOut {
  uint32_t gbase, half;
  bool swz;
  int g8, TW, w;
  __device__ __forceinline__ uint32_t at(int j) const { return a_addr(gbase, swz, j * TW + w, g8, half); }
};

// Column walk over R output rows (j0 .. j0+R-1) of one tile column and CP
// channels, fully unrolled.  xs: the thread's channels at box row 0, box
// column w * S (tap 0); rowb / pixb: bytes per box row / column.  Each input
// row is loaded once (three horizontal taps) and added into every output row
// that uses it.
template <typename T, int S, int CP, int R>
__device__ __forceinline__ void walk_fixed(const uint8_t* xs, uint32_t rowb, uint32_t pixb, const Vec<CP> (&wv)[9],
                                           const float (&bias)[CP], int j0, const AOut& o, int act, float hi) {
  float acc[R][CP];
  const uint8_t* x0 = xs + (size_t)(j0 * S) * rowb;
#pragma unroll
  for (int r = 0; r < (R - 1) * S + 3; ++r) {
    Vec<CP> xr[3];
    const uint8_t* px = x0 + (size_t)r * rowb;
#pragma unroll
    for (int kx = 0; kx < 3; ++kx) xr[kx] = ld_vec<CP>(px + kx * pixb);
#pragma unroll
    for (int ky = 0; ky < 3; ++ky) {
      // row r is filter row ky of output jj when jj * S + ky == r
      if (r - ky < 0 || (r - ky) % S != 0 || (r - ky) / S >= R) continue;
      const int jj = (r - ky) / S;
      if (ky == 0) {
#pragma unroll
        for (int e = 0; e < CP; ++e) acc[jj][e] = bias[e];
      }
      add_row<T, CP>(acc[jj], xr, &wv[3 * ky]);
      if (ky == 2) put_h<T, CP>(o.at(j0 + jj), acc[jj], act, hi);
    }
  }
}

// The same walk over R >= 2 output rows (runtime R) with a rolled loop: the
// first and last input rows are peeled, and in between every input row
// finishes one output row and starts the next (three live rows at stride
// 1, two at stride 2).  Each row is loaded one row ahead.  A fraction of the
// unrolled walk's code, which measured faster for every walk longer than one
// row (the unrolled body overflows the instruction cache and the loop around
// it misses as well).
template <typename T, int S, int CP>
__device__ __forceinline__ void walk_roll(const uint8_t* xs, uint32_t rowb, uint32_t pixb, const Vec<CP> (&wv)[9],
                                          const float (&bias)[CP], int j0, int R, const AOut& o, int act,
                                          float hi) {
  const uint8_t* px = xs + (size_t)(j0 * S) * rowb;
  auto ld = [&](Vec<CP> (&xr)[3]) {
#pragma unroll
    for (int kx = 0; kx < 3; ++kx) xr[kx] = ld_vec<CP>(px + kx * pixb);
    px += rowb;
  };
  auto start = [&](float (&acc)[CP], const Vec<CP> (&xr)[3]) {
#pragma unroll
    for (int e = 0; e < CP; ++e) acc[e] = bias[e];
    add_row<T, CP>(acc, xr, &wv[0]);
  };
  auto put = [&](int j, float (&acc)[CP]) { put_h<T, CP>(o.at(j0 + j), acc, act, hi); };
  float A[CP], B[CP];
  Vec<CP> xa[3], xb[3];  // the current input row and the next one
  if constexpr (S == 1) {
    // rows 0 and 1: outputs 0 (filter rows 0, 1) and 1 (filter row 0)
    ld(xa);
    start(A, xa);
    ld(xa);
    add_row<T, CP>(A, xa, &wv[3]);
    start(B, xa);
    // row r (r >= 2) finishes output r-2, continues r-1 and starts r.  Two
    // rows per trip: A and B swap roles every row, so no accumulator moves.
    // At the top of a trip xa holds row r, A = output r-2, B = output r-1.
    int r = 2;
    ld(xa);
#pragma unroll 1
    for (; r + 1 < R; r += 2) {
      ld(xb);  // row r+1
      add_row<T, CP>(A, xa, &wv[6]);
      put(r - 2, A);
      add_row<T, CP>(B, xa, &wv[3]);
      start(A, xa);
      ld(xa);  // row r+2 (<= R)
      add_row<T, CP>(B, xb, &wv[6]);
      put(r - 1, B);
      add_row<T, CP>(A, xb, &wv[3]);
      start(B, xb);
    }
    if (r < R) {  // r = R-1: rows R-1, R, R+1
      ld(xb);
      add_row<T, CP>(A, xa, &wv[6]);
      put(r - 2, A);
      add_row<T, CP>(B, xa, &wv[3]);
      start(A, xa);
      add_row<T, CP>(B, xb, &wv[6]);
      put(R - 2, B);
      add_row<T, CP>(A, xb, &wv[3]);
      ld(xb);
      add_row<T, CP>(A, xb, &wv[6]);
      put(R - 1, A);
    } else {  // r = R: rows R, R+1
      add_row<T, CP>(A, xa, &wv[6]);
      put(R - 2, A);
      add_row<T, CP>(B, xa, &wv[3]);
      ld(xa);
      add_row<T, CP>(B, xa, &wv[6]);
      put(R - 1, B);
    }
  } else {
    // rows 0 and 1: output 0 (filter rows 0, 1); then rows 2j (finishes
    // output j-1, starts j) and 2j+1, with xa holding row 2j at the top
    ld(xa);
    start(A, xa);
    ld(xa);
    add_row<T, CP>(A, xa, &wv[3]);
    ld(xa);
#pragma unroll 1
    for (int j = 1; j < R; ++j) {
      ld(xb);  // row 2j+1
      add_row<T, CP>(A, xa, &wv[6]);
      put(j - 1, A);
      start(A, xa);
      ld(xa);  // row 2j+2
      add_row<T, CP>(A, xb, &wv[3]);
    }
    add_row<T, CP>(A, xa, &wv[6]);  // row 2R: finishes output R-1
    put(R - 1, A);
    (void)B;
  }
}

template <typename T, int S, int CP>
__device__ __forceinline__ void walk_any(const uint8_t* xs, uint32_t rowb, uint32_t pixb, const Vec<CP> (&wv)[9],
                                         const float (&bias)[CP], int j0, int j1, const AOut& o, int act,
                                         float hi) {
  if (j1 - j0 == 1)
    walk_fixed<T, S, CP, 1>(xs, rowb, pixb, wv, bias, j0, o, act, hi);
  else
    walk_roll<T, S, CP>(xs, rowb, pixb, wv, bias, j0, j1 - j0, o, act, hi);
}

// A CTA's current tile (image n, tile row th, tile column tw), stepped by the
// grid stride with carries instead of divisions (a runtime integer division
// costs well over a hundred cycles of latency on the per-tile path).
struct TileWalk {
  int n, th, tw;     // current tile
  int dn, dth, dtw;  // the grid stride in the same units
  __device__ __forceinline__ void init(int tile, int stride, const DwPwArgs& a) {
    const int per = a.tiles_h * a.tiles_w;
    n = tile / per;
    int r = tile - n * per;
    th = r / a.tiles_w, tw = r - th * a.tiles_w;
    dn = stride / per;
    r = stride - dn * per;
    dth = r / a.tiles_w, dtw = r - dth * a.tiles_w;
  }
  __device__ __forceinline__ void next(const DwPwArgs& a) {
    tw += dtw, th += dth, n += dn;
    if (tw >= a.tiles_w) tw -= a.tiles_w, ++th;
    if (th >= a.tiles_h) th -= a.tiles_h, ++n;
  }
};

// A position in a ring of `size` slots and the parity of the number of
// times it wrapped (= the mbarrier phase parity of that use of the slot).
struct Ring {
  int pos = 0, ph = 0;
  __device__ __forceinline__ void next(int size) {
    if (++pos == size) pos = 0, ph ^= 1;
  }
};

template <typename T, int S, int CP>
__global__ void __launch_bounds__(Cfg<CP>::kThreads, 1)
    dw_pw_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ DwPwArgs a) {
  constexpr int kComputeWarps = Cfg<CP>::kComputeWarps, kComputeThreads = Cfg<CP>::kComputeThreads;
  constexpr int kThreads = Cfg<CP>::kThreads, kCPT = CP;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* x_full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* x_empty = x_full + kMaxStages;
  uint64_t* a_full = x_empty + kMaxStages;  // [nA] compute -> MMA: A written
  uint64_t* a_empty = a_full + kMaxA;       // [nA] MMA -> compute: A read
  uint64_t* acc_full = a_empty + kMaxA;     // [2] MMA -> epilogue: accumulators complete
  uint64_t* acc_empty = acc_full + 2;       // [2] epilogue -> MMA: accumulators read
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 256);
  volatile int* failed = reinterpret_cast<volatile int*>(smem + 260);
  uint32_t* a_done = reinterpret_cast<uint32_t*>(smem + 264);  // [kMaxA] compute warps done with A buffer b, ever
  const uint8_t* wdw = smem + a.wdw_off;                                // [GT][9 taps][CP], the storage type
  const uint8_t* bdw = smem + a.bdw_off;                                // [C], the storage type
  const float* bpw = reinterpret_cast<const float*>(smem + a.bpw_off);  // [Np]
  uint8_t* Xs = smem + a.x_off;                                          // stages x [Hin][Win][CH]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(&x_full[s], 1);
      mbar_init(&x_empty[s], kComputeWarps);
    }
    for (int b = 0; b < kMaxA; ++b) {
      mbar_init(&a_full[b], kComputeWarps);
      mbar_init(&a_empty[b], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], kEpiWarps);
    }
    *failed = 0;
    for (int b = 0; b < kMaxA; ++b) a_done[b] = 0u;
    fence_mbar_init();
    tma_prefetch_desc(&xmap);
  }
  const int my_tiles = (int)blockIdx.x < a.tiles ? (a.tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  const int copies = my_tiles * a.chunks;
  // Producer state (thread 0): the next copy pk is chunk pcc of tile pw, into
  // ring slot pr (the input box of CH channels x Win columns x Hin rows from
  // (oh0 * S - pH, ow0 * S - pW): the halo and the padding read as zeros).
  TileWalk pw = {};
  Ring pr;
  int pk = 0, pcc = 0;
  auto issue_next = [&]() {
    mbar_arrive_expect_tx(&x_full[pr.pos], a.x_stage_bytes);
    tma_load_4d(Xs + (size_t)pr.pos * a.x_stage_stride, &xmap, &x_full[pr.pos], pcc * a.CH,
                pw.tw * a.TW * S - a.pW, pw.th * a.TH * S - a.pH, pw.n);
    pr.next(a.stages);
    ++pk;
    if (++pcc == a.chunks) pcc = 0, pw.next(a);
  };
  // x is global memory: read only after the wait on the previous grid.  The
  // first tile's copies go out at once, while the other warps stage the
  // weights; the rest of the ring fills after that (so the first tiles of
  // all CTAs arrive first).
  grid_dependency_wait();
  if (tid == 0) {
    pw.init(blockIdx.x, gridDim.x, a);
    while (pk < min(a.chunks, copies)) issue_next();
  }
  // Weights, biases and the projection's B operand, staged once per CTA by
  // warps 1-13, every thread's global loads of a batch issued before its
  // stores so their latencies overlap.
  {
    const T* __restrict__ wdg = static_cast<const T*>(a.w_dw);
    const T* __restrict__ bdg = static_cast<const T*>(a.b_dw);
    const T* __restrict__ wpg = static_cast<const T*>(a.w_pw);
    const T* __restrict__ bpg = static_cast<const T*>(a.b_pw);
    T* wdw_s = reinterpret_cast<T*>(smem + a.wdw_off);
    T* bdw_s = reinterpret_cast<T*>(smem + a.bdw_off);
    float* bpw_s = reinterpret_cast<float*>(smem + a.bpw_off);
    uint8_t* Bs = smem + a.b_off;  // [C/8][Np rows][16 B], K-major, no swizzle
    constexpr int kB = 4, kN = kThreads - 32;
    const int t0 = tid - 32;
    for (int base = t0; t0 >= 0 && base < a.G * a.Np; base += kB * kN) {
      uint4 v[kB];
#pragma unroll
      for (int q = 0; q < kB; ++q) {
        const int i = base + q * kN, kc = i / a.Np, n = i - kc * a.Np;
        v[q] = make_uint4(0u, 0u, 0u, 0u);
        if (i < a.G * a.Np && n < a.K) v[q] = *reinterpret_cast<const uint4*>(wpg + (int64_t)n * a.C + kc * 8);
      }
#pragma unroll
      for (int q = 0; q < kB; ++q) {
        const int i = base + q * kN, kc = i / a.Np, n = i - kc * a.Np;
        if (i < a.G * a.Np) *reinterpret_cast<uint4*>(Bs + ((size_t)kc * a.Np + n) * 16) = v[q];
      }
    }
    for (int base = t0; t0 >= 0 && base < a.C * 9; base += 2 * kB * kN) {
      T v[2 * kB];
#pragma unroll
      for (int q = 0; q < 2 * kB; ++q) {
        const int i = base + q * kN;
        if (i < a.C * 9) v[q] = wdg[i];
      }
#pragma unroll
      for (int q = 0; q < 2 * kB; ++q) {
        const int i = base + q * kN, c = i / 9, t = i - c * 9;
        if (i < a.C * 9) wdw_s[((c / kCPT) * 9 + t) * kCPT + (c % kCPT)] = v[q];
      }
    }
    for (int i = t0; t0 >= 0 && i < a.C; i += kN) bdw_s[i] = bdg ? bdg[i] : Elem<T>::from_f32(0.f);
    for (int i = t0; t0 >= 0 && i < a.Np; i += kN) bpw_s[i] = (bpg && i < a.K) ? Elem<T>::to_f32(bpg[i]) : 0.f;
  }
  fence_proxy_async_smem();  // B (generic-proxy writes) -> visible to the tensor core
  if (warp == kMmaWarp) {    // tensor memory only after the wait on the previous grid
    tc::tmem_alloc(tmem_slot, a.tmem_cols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t a_base0 = smem_u32(smem + a.a_off);

  // Roles: warp 0 copies, warp 1 holds the tensor memory and issues the
  // projection (or the compute warps issue it, a.inline_mma), warps 2-5 run
  // the epilogue, warps 6.. the depthwise math.
  if (warp == 0) {
    // ---------------- TMA producer: every (tile, chunk) in order ----------------
    if (lane == 0) {
      while (pk < copies) {
        // slot pr.pos is free once the copy a ring before it was consumed
        if (pk >= a.stages && !*failed && !mbar_wait(&x_empty[pr.pos], (uint32_t)(pr.ph ^ 1), a.wait_limit_ns)) {
          report(a.status, kDevTimeout, 41);
          *failed = 1;
        }
        if (*failed) break;
        issue_next();
      }
      // bounded drain (also after a timeout): no copy may still be landing
      // when the CTA exits (copies 0 .. pk-1 were issued)
      for (int k = max(0, pk - a.stages); k < pk; ++k)
        mbar_wait(&x_full[k % a.stages], (uint32_t)((k / a.stages) & 1), a.wait_limit_ns);
    }
  } else if (warp == kMmaWarp && !a.inline_mma) {
    // ---------------- MMA issuer: the whole warp, one elected lane issues ----------------
    const uint32_t b_base = smem_u32(smem + a.b_off);
    int i = 0, issued = -1;
    Ring ra;  // A buffer of tile i and its phase parity
    for (int tile = blockIdx.x; tile < a.tiles; tile += gridDim.x, ++i, ra.next(a.nA)) {
      const int ab = ra.pos, cb = i & 1;
      if (lane == 0 && !*failed) {
        if (!mbar_wait(&a_full[ab], (uint32_t)ra.ph, a.wait_limit_ns) ||
            (i >= 2 && !mbar_wait(&acc_empty[cb], (uint32_t)(((i >> 1) - 1) & 1), a.wait_limit_ns))) {
          report(a.status, kDevTimeout, 43);
          *failed = 1;
        }
      }
      __syncwarp();
      tc::fence_after_sync();
      if (*failed) continue;
      const uint32_t d = tmem_base + (uint32_t)(cb * a.Np);
      // descriptors built once; a K step advances their start-address field
      // (bits 0-13, address / 16), which stays below 2^14 inside shared memory
      const uint32_t a_buf = a_base0 + (uint32_t)ab * a.a_bytes;
      const uint64_t ad0 = tc::smem_desc_sw128(a_buf);
      const int ks_swz = (a.C / 64) * 4;  // K steps inside the swizzled atoms
      const uint64_t at0 = tc::smem_desc(a_buf + (uint32_t)(a.C / 64) * kAtomBytes, kTailGroupBytes, 128u);
      const uint64_t bd0 = tc::smem_desc(b_base, (uint32_t)a.Np * 16u, 128u);
      for (int ks = 0; ks < a.C / 16; ++ks) {  // one K step per 16 channels
        const uint64_t ad = ks < ks_swz ? ad0 + (((uint32_t)(ks >> 2) * kAtomBytes + (uint32_t)(ks & 3) * 32u) >> 4)
                                        : at0 + ((uint32_t)(ks - ks_swz) * 2u * kTailGroupBytes >> 4);
        const uint64_t bd = bd0 + ((uint32_t)(2 * ks * a.Np) * 16u >> 4);
        mma_f16_elect(d, ad, bd, a.idesc, ks > 0 ? 1u : 0u);
      }
      commit_elect(&a_empty[ab]);
      commit_elect(&acc_full[cb]);
      issued = i;
    }
    // the last accumulators must have landed before tensor memory is freed
    if (issued >= 0 && lane == 0)
      mbar_wait(&acc_full[issued & 1], (uint32_t)((issued >> 1) & 1), a.wait_limit_ns);
    __syncwarp();
  } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + kEpiWarps) {
    // ---------------- epilogue: TMEM lane quarter q = pixel rows 32q .. 32q+31 ----------------
    T* __restrict__ yg = static_cast<T*>(a.y);
    const int q = warp & 3;
    const int p = q * 32 + lane;
    const int j = p / a.TW, w = p - j * a.TW;
    int i = 0;
    TileWalk ew;
    ew.init(blockIdx.x, gridDim.x, a);
    for (int tile = blockIdx.x; tile < a.tiles; tile += gridDim.x, ++i, ew.next(a)) {
      const int n = ew.n, oh0 = ew.th * a.TH, ow0 = ew.tw * a.TW;
      const int cb = i & 1;
      if (lane == 0 && !*failed && !mbar_wait(&acc_full[cb], (uint32_t)((i >> 1) & 1), a.wait_limit_ns)) {
        report(a.status, kDevTimeout, 44);
        *failed = 1;
      }
      __syncwarp();
      tc::fence_after_sync();
      if (!*failed) {
        const bool valid = j < min(a.TH, a.Ho - oh0) && w < min(a.TW, a.Wo - ow0);
        T* dst = yg + (((int64_t)n * a.Ho + oh0 + j) * a.Wo + ow0 + w) * a.K;
        for (int c0 = 0; c0 < a.Np; c0 += 16) {
          uint32_t rr[16];
          tc::tmem_ld16(tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(cb * a.Np + c0), rr);
          tc::tmem_ld_wait();
          if (valid) {
#pragma unroll
            for (int h8 = 0; h8 < 16; h8 += 8) {
              if (c0 + h8 < a.K) {
                uint32_t wd[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                  wd[e] = epilogue_pair<T>(__uint_as_float(rr[h8 + 2 * e]), __uint_as_float(rr[h8 + 2 * e + 1]),
                                           bpw[c0 + h8 + 2 * e], bpw[c0 + h8 + 2 * e + 1]);
                *reinterpret_cast<uint4*>(dst + c0 + h8) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
              }
            }
          }
        }
      }
      // this warp's reads of the accumulators are done
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[cb]);
    }
  } else if (warp >= kComputeWarp0) {
    // ---------------- depthwise compute: (segment, column, group) items ----------------
    // A thread's items are the same in every tile (f = tcid, tcid + 256, ...):
    // the first one's decode is kept across tiles, and the ring position of
    // the tile's copies advances by one tile per tile.
    const int tcid = tid - 32 * kComputeWarp0;
    const uint32_t b_base = smem_u32(smem + a.b_off);
    const int cols_g = a.TW * a.GT;
    const int items = a.NS * cols_g;
    const uint32_t pixb = (uint32_t)(a.CH * 2), rowb = (uint32_t)(a.Win * a.CH * 2);  // bytes per box column / row
    const float hi = a.act == 2 ? 6.f : __int_as_float(0x7f800000);                      // ReLU6 / ReLU upper clamp
    const int gfull = (a.C / 64) * 8;                                                     // groups in swizzled atoms
    auto group_off = [&](int g) -> uint32_t {  // the group's atom (or tail group) inside an A buffer
      return g < gfull ? (uint32_t)(g >> 3) * kAtomBytes
                       : (uint32_t)(gfull >> 3) * kAtomBytes + (uint32_t)(g - gfull) * kTailGroupBytes;
    };
    // decode of the first item (the common case: one item per thread)
    const int f0 = min(tcid, items - 1);
    const int seg0 = f0 / cols_g, rem0 = f0 - seg0 * cols_g;
    const int w0 = rem0 / a.GT, g0 = rem0 - w0 * a.GT;
    const int cc0 = g0 / a.GC;
    int kb_s = 0, kb_ph = 0;  // stage and phase parity of the tile's first copy
    int i = 0;
    TileWalk cw;
    cw.init(blockIdx.x, gridDim.x, a);
    Ring ca;  // A buffer of tile i and its phase parity
    for (int tile = blockIdx.x; tile < a.tiles; tile += gridDim.x, ++i, cw.next(a), ca.next(a.nA)) {
      const int rows = min(a.TH, a.Ho - cw.th * a.TH), cols = min(a.TW, a.Wo - cw.tw * a.TW);
      const int ab = ca.pos;
      // A buffer ab free: the MMAs of tile i - nA have read it
      if (i >= a.nA) {
        if (lane == 0 && !*failed && !mbar_wait(&a_empty[ab], (uint32_t)(ca.ph ^ 1), a.wait_limit_ns)) {
          report(a.status, kDevTimeout, 45);
          *failed = 1;
        }
        __syncwarp();
      }
      const uint32_t a_base = a_base0 + (uint32_t)ab * a.a_bytes;
      auto stage_of = [&](int cc, int* ph) {  // ring stage and parity of this tile's copy cc
        int st = kb_s + cc;
        *ph = kb_ph;
        if (st >= a.stages) st -= a.stages, *ph ^= 1;
        return st;
      };
      for (int f = tcid; f < items; f += kComputeThreads) {
        int seg = seg0, w = w0, g = g0, cc = cc0;
        if (f != f0) {  // further items (more (column, group) pairs than threads)
          seg = f / cols_g;
          const int rem = f - seg * cols_g;
          w = rem / a.GT, g = rem - w * a.GT;
          cc = g / a.GC;
        }
        const int j0 = seg * a.rps, j1 = min(rows, j0 + a.rps);
        if (w >= cols || j0 >= j1 || *failed) continue;
        int ph;
        const int s = stage_of(cc, &ph);
        if (!mbar_wait(&x_full[s], (uint32_t)ph, a.wait_limit_ns)) {
          report(a.status, kDevTimeout, 42);
          *failed = 1;
          continue;
        }
        Vec<kCPT> wv[9];
#pragma unroll
        for (int t = 0; t < 9; ++t) wv[t] = ld_vec<kCPT>(wdw + ((size_t)g * 9 + t) * kCPT * 2);
        float bias[kCPT];  // the group's bias, one load (consecutive groups: consecutive bytes), widened exactly
        {
          const Vec<kCPT> bq = ld_vec<kCPT>(bdw + (size_t)g * kCPT * 2);
#pragma unroll
          for (int e = 0; e < kCPT / 2; ++e) widen_word<T>(bq.w[e], &bias[2 * e]);
        }
        const int gl = g - cc * a.GC;
        const uint8_t* xs = Xs + (size_t)s * a.x_stage_stride + ((size_t)(w * S) * a.CH + gl * kCPT) * 2;
        const int g8 = (g * kCPT) >> 3;  // the 8-channel group of A the thread's channels fall in
        const AOut o{a_base + group_off(g8), (uint32_t)((g * kCPT) & 7) * 2u, g8 < gfull, g8, a.TW, w};
        walk_any<T, S, kCPT>(xs, rowb, pixb, wv, bias, j0, j1, o, a.act, hi);
      }
      // A rows of this warp written (generic proxy) -> visible to the MMAs;
      // each stage of the tile released once its copy is seen complete (so
      // an arrival can never count toward an earlier use of the stage)
      fence_proxy_async_smem();
      __syncwarp();
      uint32_t done = 0;
      if (lane == 0) {
        for (int cc = 0; cc < a.chunks; ++cc) {
          int ph;
          const int s = stage_of(cc, &ph);
          if (!*failed && !mbar_wait(&x_full[s], (uint32_t)ph, a.wait_limit_ns)) {
            report(a.status, kDevTimeout, 46);
            *failed = 1;
          }
          mbar_arrive(&x_empty[s]);
        }
        if (a.inline_mma) {
          __threadfence_block();  // this warp's A rows before its count (release)
          done = atomicAdd(&a_done[ab], 1u);
        } else {
          mbar_arrive(&a_full[ab]);
        }
      }
      done = __shfl_sync(0xffffffffu, done, 0);
      if (a.inline_mma && done % kComputeWarps == kComputeWarps - 1) {
        // This warp completed tile i's A: it issues the projection itself.  A
        // separate issuing warp shares its sub-partition with compute warps
        // and measured up to ten times slower to issue; issuing here costs
        // the compute warps that time instead, which pays when the MMAs, not
        // the depthwise math, set the pace (see the planner).
        __threadfence_block();  // the other warps' A rows (acquire)
        const int cb = i & 1;
        if (lane == 0 && i >= 2 && !*failed &&
            !mbar_wait(&acc_empty[cb], (uint32_t)(((i >> 1) - 1) & 1), a.wait_limit_ns)) {
          report(a.status, kDevTimeout, 43);
          *failed = 1;
        }
        __syncwarp();
        tc::fence_after_sync();
        if (!*failed) {
          const uint32_t d = tmem_base + (uint32_t)(cb * a.Np);
          // descriptors built once; a K step advances their start-address
          // field (bits 0-13, address / 16), below 2^14 inside shared memory
          const uint64_t ad0 = tc::smem_desc_sw128(a_base);
          const int ks_swz = (a.C / 64) * 4;  // K steps inside the swizzled atoms
          const uint64_t at0 = tc::smem_desc(a_base + (uint32_t)(a.C / 64) * kAtomBytes, kTailGroupBytes, 128u);
          const uint64_t bd0 = tc::smem_desc(b_base, (uint32_t)a.Np * 16u, 128u);
          for (int ks = 0; ks < a.C / 16; ++ks) {  // one K step per 16 channels
            const uint64_t ad = ks < ks_swz
                                    ? ad0 + (((uint32_t)(ks >> 2) * kAtomBytes + (uint32_t)(ks & 3) * 32u) >> 4)
                                    : at0 + ((uint32_t)(ks - ks_swz) * 2u * kTailGroupBytes >> 4);
            const uint64_t bd = bd0 + ((uint32_t)(2 * ks * a.Np) * 16u >> 4);
            mma_f16_elect(d, ad, bd, a.idesc, ks > 0 ? 1u : 0u);
          }
          commit_elect(&a_empty[ab]);
          commit_elect(&acc_full[cb]);
        }
      }
      kb_s += a.chunks;  // chunks <= stages: at most one wrap
      if (kb_s >= a.stages) kb_s -= a.stages, kb_ph ^= 1;
    }
  }
  // the last tile's MMAs must have completed before tensor memory is freed
  // (the epilogue waited for them too, unless a wait timed out)
  if (warp == kMmaWarp && lane == 0 && my_tiles > 0)
    mbar_wait(&acc_full[(my_tiles - 1) & 1], (uint32_t)(((my_tiles - 1) >> 1) & 1), a.wait_limit_ns);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem_base, a.tmem_cols);
  }
}

}  // namespace fz

namespace {

inline uint32_t round_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }
inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

struct DwPwPlan {
  fz::DwPwArgs a;
  uint32_t smem_bytes;
};

// Column walks: NS segments of rps output rows, as many segments as keep the
// `threads` compute threads busy.
inline void walk_split(int TH, int TW, int GT, int threads, int* NS, int* rps) {
  const int ns = std::max(1, std::min(TH, threads / (TW * GT)));
  *rps = ceil_div(TH, ns);
  *NS = ceil_div(TH, *rps);
}

inline int compute_threads(int cp) { return cp == 8 ? fz::Cfg<8>::kComputeThreads : fz::Cfg<4>::kComputeThreads; }

// Tile shape, channels per compute thread, copy chunking, buffering and the
// MMA issuer.  Candidates: 8 or 4 channels per compute thread; TW the
// balanced split of Wo into pieces of at most 16 (or 8) columns, TH the
// balanced split of Ho with TH * TW <= 128; copies of all C channels or of
// 64/48/32/16; three, two or one A buffers.  Preferred, in order: at least
// two A buffers, 8 channels per thread, more pixels per tile, two tiles of
// input in flight, fewer output rows per compute thread, more A buffers,
// fewer copies per tile.  The order follows measurements on the MobileNetV2
// layers: a tile's fixed cost (its MMA batch, barriers and loop) outweighs
// its depthwise work, so the largest tile wins (even over double-buffered
// input), and at equal tiles the 8-channel form beat the 4-channel one by
// 8-15%.  ov (may be null): {channels per thread, TH, TW, MMA issuer (1 the
// dedicated warp, 2 the compute warps)} to force, 0 = automatic.
bool make_dw_pw_plan(const Geometry& g, bool bf16, int K, int act, int max_smem, const int* ov, DwPwPlan* out) {
  if (g.ndim != 2 || g.Cg != 1 || g.Kg != 1 || g.Z != 1 || g.Y != 3 || g.X != 3) return false;
  if (g.dH != 1 || g.dW != 1 || g.sH != g.sW || g.sH < 1 || g.sH > 2) return false;
  const int C = g.C(), S = g.sH;
  if (C % 16 != 0 || C > 256 || K % 8 != 0 || K < 8 || K > 256 || act < 0 || act > 2) return false;
  if (g.Wo < 1 || g.Ho < 1) return false;
  const int ov_cp = ov ? ov[0] : 0, ov_th = ov ? ov[1] : 0, ov_tw = ov ? ov[2] : 0, ov_mma = ov ? ov[3] : 0;
  if (ov_cp != 0 && ov_cp != 4 && ov_cp != 8) return false;
  if (ov_mma < 0 || ov_mma > 2) return false;
  fz::DwPwArgs a;
  std::memset(&a, 0, sizeof(a));
  a.C = C, a.K = K, a.Np = (K + 15) / 16 * 16, a.G = C / 8;
  a.Ho = g.Ho, a.Wo = g.Wo, a.act = act, a.pH = g.pH, a.pW = g.pW;
  a.wdw_off = 1024;
  a.bdw_off = a.wdw_off + (uint32_t)C * 9u * 2u;
  a.bpw_off = a.bdw_off + (uint32_t)C * 2u;
  a.b_off = round_up(a.bpw_off + (uint32_t)a.Np * 4u, 1024);
  a.a_off = round_up(a.b_off + (uint32_t)a.G * (uint32_t)a.Np * 16u, 1024);
  a.a_bytes = round_up((uint32_t)(C / 64) * fz::kAtomBytes + (uint32_t)((C % 64) / 8) * fz::kTailGroupBytes, 1024);
  const uint32_t budget = (uint32_t)std::min(max_smem, 227 * 1024);

  bool found = false;
  int best[8] = {};  // score, compared in order (larger is better)
  for (int cp : {8, 4}) {
    if (ov_cp && cp != ov_cp) continue;
    const int GT = C / cp, threads = compute_threads(cp);
    for (int cap : {16, 8}) {
      const int TW = ov_tw ? ov_tw : ceil_div(g.Wo, ceil_div(g.Wo, cap));
      if (TW < 1 || TW > 16 || TW > g.Wo || (ov_tw && cap != 16)) continue;
      for (int nA = fz::kMaxA; nA >= 1; --nA) {
        if (a.a_off + (uint32_t)nA * a.a_bytes > budget) continue;
        const uint32_t room = budget - a.a_off - (uint32_t)nA * a.a_bytes;
        for (int thmax = std::min(g.Ho, 128 / TW); thmax >= 1; --thmax) {
          const int TH = ceil_div(g.Ho, ceil_div(g.Ho, thmax));
          if (TH != thmax) continue;  // each balanced TH once
          if (ov_th && TH != ov_th) continue;
          const int Win = (TW - 1) * S + 3, Hin = (TH - 1) * S + 3;
          if (Win > 256 || Hin > 256) continue;
          int NS, rps;
          walk_split(TH, TW, GT, threads, &NS, &rps);
          const int thread_rows = ceil_div(NS * TW * GT, threads) * rps;  // output rows a compute thread walks per tile
          for (int CH : {C, 64, 48, 32, 16}) {
            if (CH > C || C % CH != 0 || CH % cp != 0) continue;
            const int chunks = C / CH;
            const uint32_t bytes = (uint32_t)(Hin * Win * CH) * 2u, stride = round_up(bytes, 1024);
            const int stages = (int)std::min<uint32_t>(fz::kMaxStages, room / stride);
            if (stages < chunks) continue;
            const int sc[8] = {nA >= 2, cp == 8, TH * TW, stages >= 2 * chunks, -thread_rows, nA, -chunks, -TW};
            if (found && !std::lexicographical_compare(best, best + 8, sc, sc + 8)) continue;
            found = true;
            std::copy(sc, sc + 8, best);
            a.cpt = cp, a.GT = GT;
            a.TH = TH, a.TW = TW, a.Win = Win, a.Hin = Hin, a.CH = CH, a.GC = CH / cp, a.chunks = chunks;
            a.stages = stages, a.nA = nA, a.x_stage_bytes = bytes, a.x_stage_stride = stride;
          }
        }
      }
    }
  }
  if (!found) return false;
  a.x_off = a.a_off + (uint32_t)a.nA * a.a_bytes;
  a.tiles_h = ceil_div(g.Ho, a.TH);
  a.tiles_w = ceil_div(g.Wo, a.TW);
  const int64_t tiles = (int64_t)g.N * a.tiles_h * a.tiles_w;
  if (tiles >= (1ll << 31)) return false;
  a.tiles = (int)tiles;
  walk_split(a.TH, a.TW, a.GT, compute_threads(a.cpt), &a.NS, &a.rps);
  // With three A buffers the MMAs of a tile have two tiles of compute to
  // finish in, and the dedicated issuing warp keeps that time off the compute
  // warps; with fewer the MMAs set the pace and the compute warps issue them.
  a.inline_mma = ov_mma ? (ov_mma == 2) : (a.nA < 3);
  a.tmem_cols = 32;
  while (a.tmem_cols < 2u * (uint32_t)a.Np) a.tmem_cols <<= 1;
  a.idesc = tc::idesc_f16(bf16, 128, a.Np);
  DwPwPlan p;
  p.a = a;
  p.smem_bytes = a.x_off + (uint32_t)a.stages * a.x_stage_stride;
  *out = p;
  return true;
}

template <typename T, int S, int CP>
cudaError_t dw_pw_launch_cp(const DwPwPlan& p, const Geometry& g, const LaunchArgs& la, const void* w_pw,
                            const void* b_pw, const DeviceInfo& dev) {
  constexpr int kThreads = fz::Cfg<CP>::kThreads;
  static SmemAttr attr;
  cudaError_t e = attr.ensure(fz::dw_pw_kernel<T, S, CP>, dev.device, (int)p.smem_bytes);
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
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fz::dw_pw_kernel<T, S, CP>, kThreads, p.smem_bytes);
  if (e != cudaSuccess) return e;
  occ = std::max(1, std::min(occ, 512 / (int)p.a.tmem_cols));
  const int grid = std::max(1, std::min(a.tiles, dev.num_sms * occ));
  return launch_kernel(fz::dw_pw_kernel<T, S, CP>, dim3(grid), dim3(kThreads), p.smem_bytes, la, xmap, a);
}

template <typename T, int S>
cudaError_t dw_pw_launch_typed(const Geometry& g, const LaunchArgs& la, const void* w_pw, const void* b_pw, int K,
                               int act, const DeviceInfo& dev) {
  DwPwPlan p;
  if (!make_dw_pw_plan(g, std::is_same<T, __nv_bfloat16>::value, K, act, dev.max_smem_optin, la.tile, &p))
    return cudaErrorNotSupported;
  const uintptr_t al = reinterpret_cast<uintptr_t>(la.x) | reinterpret_cast<uintptr_t>(la.y) |
                       reinterpret_cast<uintptr_t>(w_pw);
  if (al & 15) return cudaErrorNotSupported;
  return p.a.cpt == 8 ? dw_pw_launch_cp<T, S, 8>(p, g, la, w_pw, b_pw, dev)
                      : dw_pw_launch_cp<T, S, 4>(p, g, la, w_pw, b_pw, dev);
}

template <typename T>
cudaError_t dw_pw_launch_stride(const Geometry& g, const LaunchArgs& la, const void* w_pw, const void* b_pw, int K,
                                int act, const DeviceInfo& dev) {
  return g.sH == 1 ? dw_pw_launch_typed<T, 1>(g, la, w_pw, b_pw, K, act, dev)
                   : dw_pw_launch_typed<T, 2>(g, la, w_pw, b_pw, K, act, dev);
}

}  // namespace

bool dw_pw_supported(const Geometry& g, DType dt, int K, int act) {
  if (dt == kF32) return false;
  DwPwPlan p;
  return make_dw_pw_plan(g, dt == kBF16, K, act, kDefaultSmemOptin, nullptr, &p);
}

cudaError_t dw_pw_launch(const Geometry& g, const LaunchArgs& a, const void* w_pw, const void* b_pw, int K, int act,
                         const DeviceInfo& dev) {
  if (a.dt == kF16) return dw_pw_launch_stride<__half>(g, a, w_pw, b_pw, K, act, dev);
  if (a.dt == kBF16) return dw_pw_launch_stride<__nv_bfloat16>(g, a, w_pw, b_pw, K, act, dev);
  return cudaErrorNotSupported;
}

}  // namespace gconv
