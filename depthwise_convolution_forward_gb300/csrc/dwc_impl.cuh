// Ka, column form: depthwise direct kernel (Cg == Kg == 1, 3x3 spatial
// filter, depth filter 1) that walks each output column down the tile with a
// rolling window of accumulator rows.
//
// Design (sm_103a):
//  * Persistent CTAs walk a static list of output tiles
//    (n, od, TH x TW output pixels, TC channels), as in the row-blocked
//    form: warp 0 is the producer and copies each tile's haloed input box
//    with 5-D TMA into a ring of shared-memory stages (zero fill at the
//    borders is the convolution's zero padding).  On request a CTA's first
//    box goes as two copies (top rows, then the rest) on two barriers, so the
//    consumers can start on the top rows while the bottom rows arrive.
//  * Consumer thread f of the tile owns output column f / NQ and the CPT
//    channels CPT (f % NQ) .. +CPT-1 (NQ = TC / CPT; CPT = 4, or 8 in the
//    kColPacked8 form).  Consecutive lanes therefore read consecutive
//    pieces of one shared-memory row (conflict-free), and every output row a
//    warp stores is one contiguous run of global memory.
//  * The thread walks the input rows of its column from top to bottom.  Each
//    input row is loaded once (three shared loads: the three horizontal taps)
//    and is added into every output row that uses it, with the filter row
//    that the row sits under; an output row is stored as soon as its last
//    filter row has been added.  For stride S and dilation DL that keeps
//    2*DL/S + 1 output rows live.
//  * The thread's 3x3xCPT weights and CPT bias values stay in registers for
//    the whole tile; the bias is the addend of each output's first fused
//    multiply-add.  16-bit inputs are multiplied with the mixed-precision
//    fma.rn.f32.{f16,bf16} (fp32 product and sum, one rounding), fp32 inputs
//    with fmaf.
//  * Fused epilogue (Kc): one round-to-nearest-even pack of the fp32 sums and
//    one vector store per output.
//  * Every mbarrier wait is bounded; a timed-out warp records the timeout in
//    the status word and exits, and the producer drains its copies first.
#pragma once

#include <type_traits>
#include <utility>

#include "dw_impl.cuh"

namespace gconv {
namespace dw {


// Operand forms of the multiply (tuning override slot 5):
//  kColPacked   16-bit storage, 4 channels per thread, pairs kept packed in
//               registers (the default for 16-bit storage);
//  kColPacked8  the same with 8 channels per thread;
//  kColSplit    16-bit storage, 4 channels, every 16-bit value in the low half
//               of its own register (weights staged split, the high half of
//               an input word shifted down once per load); fp32 storage:
//               scalar fmaf (the default for fp32);
//  kColWide     4 channels widened to fp32 once per load, multiplied in
//               channel pairs with the packed fp32x2 FMA.
//  kColGroup2   16-bit storage, groups of two channels (Cg == Kg == 2): a
//               thread's 4 channels are 2 groups; each output is the
//               two-term dot product of its group's input pair with its
//               weight pair, per tap.
enum ColForm : int { kColSplit = 0, kColPacked = 1, kColWide = 2, kColPacked8 = 3, kColGroup2 = 4 };

// Threads per CTA: a producer warp and up to 16 consumer warps (12 for the
// 8-channel form, whose threads hold twice the weights and accumulators).
__host__ __device__ constexpr int col_max_threads(int form) { return form == kColPacked8 ? 416 : 544; }

// Registers per thread the compiler may use (a cap, not a launch bound: the
// planner reads the kernel's real count).  Every form fits its
// col_max_threads at its cap.  The default 16-bit form keeps 72 when three
// output rows are live (stride 1 or 2 at dilation 1, stride 2 at dilation 2),
// so three CTAs of nine warps fit an SM when shared memory allows; five live
// rows (stride 1, dilation 2) take 88.  The other forms and fp32 hold more
// per thread (wider weights or operands) and get 96 to 152.
template <typename T, int S, int DL>
__host__ __device__ constexpr int col_reg_cap(int form) {
  return form == kColPacked8                                       ? 152
         : (form != kColPacked || sizeof(T) == 4) ? ((2 * DL) / S + 1 > 3 ? 112 : 96)
         : ((2 * DL) / S + 1 > 3)                                  ? 88
                                                                   : 72;
}
// Weight values per (tap, output channel): the group's input channels.
__host__ __device__ constexpr int col_vpc(int form) { return form == kColGroup2 ? 2 : 1; }

__device__ __forceinline__ void lds64(uint32_t addr, uint32_t (&v)[2]) {
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v[0]), "=r"(v[1]) : "r"(addr));
}
__device__ __forceinline__ void lds128a(uint32_t addr, uint32_t (&v)[4]) {
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
               : "r"(addr));
}

template <typename T>
__device__ __forceinline__ float mixed_fma(unsigned short x, unsigned short w, float c);
template <>
__device__ __forceinline__ float mixed_fma<__half>(unsigned short x, unsigned short w, float c) {
  float d;
  asm("fma.rn.f32.f16 %0, %1, %2, %3;" : "=f"(d) : "h"(x), "h"(w), "f"(c));
  return d;
}
template <>
__device__ __forceinline__ float mixed_fma<__nv_bfloat16>(unsigned short x, unsigned short w, float c) {
  float d;
  asm("fma.rn.f32.bf16 %0, %1, %2, %3;" : "=f"(d) : "h"(x), "h"(w), "f"(c));
  return d;
}

// Per (storage type, operand form): channels per thread, register operand
// type, how one thread's input piece and weight piece are read from shared
// memory, the multiply, and the bytes one staged weight takes.

struct ColOpsF32 {
  static constexpr int kCpt = 4;
  static constexpr int kOps = 4;  // registers per 4-channel piece
  using Op = float;
  static constexpr int kWeightBytes = 4;
  static constexpr int kWOps = kOps;  // registers per tap of weights
  static constexpr int kVpc = 1;
  __device__ __forceinline__ static void load_x(uint32_t addr, Op (&v)[kOps]) {
    uint32_t w[4];
    lds128a(addr, w);
#pragma unroll
    for (int e = 0; e < 4; ++e) v[e] = __uint_as_float(w[e]);
  }
  __device__ __forceinline__ static void load_w(uint32_t addr, Op (&v)[kWOps]) { load_x(addr, v); }
  __device__ __forceinline__ static void stage_w(uint8_t* dst, float v) { *reinterpret_cast<float*>(dst) = v; }
  __device__ __forceinline__ static void mac(float (&d)[kCpt], const Op (&x)[kOps], const Op (&w)[kWOps],
                                             const float (&c)[kCpt]) {
#pragma unroll
    for (int e = 0; e < kCpt; ++e) d[e] = fmaf(x[e], w[e], c[e]);
  }
};

template <typename T>
struct ColOpsWide {
  static constexpr int kCpt = 4;
  static constexpr int kOps = 4;
  using Op = float;
  static constexpr int kWeightBytes = 4;
  static constexpr int kWOps = kOps;  // registers per tap of weights
  static constexpr int kVpc = 1;
  __device__ __forceinline__ static void load_x(uint32_t addr, Op (&v)[kOps]) {
    if constexpr (sizeof(T) == 4) {
      uint32_t w[4];
      lds128a(addr, w);
#pragma unroll
      for (int e = 0; e < 4; ++e) v[e] = __uint_as_float(w[e]);
    } else {
      uint32_t w[2];
      lds64(addr, w);
      widen_word<T>(w[0], v);
      widen_word<T>(w[1], v + 2);
    }
  }
  __device__ __forceinline__ static void load_w(uint32_t addr, Op (&v)[kWOps]) {
    uint32_t w[4];
    lds128a(addr, w);
#pragma unroll
    for (int e = 0; e < 4; ++e) v[e] = __uint_as_float(w[e]);
  }
  __device__ __forceinline__ static void stage_w(uint8_t* dst, T v) {
    *reinterpret_cast<float*>(dst) = Elem<T>::to_f32(v);
  }
  __device__ __forceinline__ static void mac(float (&d)[kCpt], const Op (&x)[kOps], const Op (&w)[kWOps],
                                             const float (&c)[kCpt]) {
#pragma unroll
    for (int e = 0; e < kCpt; e += 2) {
      const float2 r = __ffma2_rn(make_float2(x[e], x[e + 1]), make_float2(w[e], w[e + 1]), make_float2(c[e], c[e + 1]));
      d[e] = r.x;
      d[e + 1] = r.y;
    }
  }
};

template <typename T>
struct ColOps16Split {
  static constexpr int kCpt = 4;
  static constexpr int kOps = 4;
  using Op = uint32_t;  // value in the low 16 bits
  static constexpr int kWeightBytes = 4;
  static constexpr int kWOps = kOps;  // registers per tap of weights
  static constexpr int kVpc = 1;
  __device__ __forceinline__ static void load_x(uint32_t addr, Op (&v)[kOps]) {
    uint32_t w[2];
    lds64(addr, w);
    v[0] = w[0], v[1] = w[0] >> 16, v[2] = w[1], v[3] = w[1] >> 16;
  }
  __device__ __forceinline__ static void load_w(uint32_t addr, Op (&v)[kWOps]) {
    uint32_t w[4];
    lds128a(addr, w);
#pragma unroll
    for (int e = 0; e < 4; ++e) v[e] = w[e];
  }
  __device__ __forceinline__ static void stage_w(uint8_t* dst, T v) {
    *reinterpret_cast<uint32_t*>(dst) = (uint32_t)(*reinterpret_cast<const unsigned short*>(&v));
  }
  __device__ __forceinline__ static void mac(float (&d)[kCpt], const Op (&x)[kOps], const Op (&w)[kWOps],
                                             const float (&c)[kCpt]) {
#pragma unroll
    for (int e = 0; e < kCpt; ++e) d[e] = mixed_fma<T>((unsigned short)x[e], (unsigned short)w[e], c[e]);
  }
};

// Two mixed-precision FMAs on the halves of packed 16-bit pairs:
// d_lo = x.lo * w.lo + c_lo, d_hi = x.hi * w.hi + c_hi.  The halves are taken
// apart inside the asm so the pairs stay packed in registers.
template <typename T>
__device__ __forceinline__ void mixed_fma_pair(uint32_t x, uint32_t w, float c_lo, float c_hi, float& d_lo,
                                               float& d_hi);
template <>
__device__ __forceinline__ void mixed_fma_pair<__half>(uint32_t x, uint32_t w, float c_lo, float c_hi, float& d_lo,
                                                       float& d_hi) {
  asm("{\n\t.reg .b16 xl, xh, wl, wh;\n\t"
      "mov.b32 {xl, xh}, %2;\n\tmov.b32 {wl, wh}, %3;\n\t"
      "fma.rn.f32.f16 %0, xl, wl, %4;\n\tfma.rn.f32.f16 %1, xh, wh, %5;\n\t}"
      : "=f"(d_lo), "=f"(d_hi)
      : "r"(x), "r"(w), "f"(c_lo), "f"(c_hi));
}
template <>
__device__ __forceinline__ void mixed_fma_pair<__nv_bfloat16>(uint32_t x, uint32_t w, float c_lo, float c_hi,
                                                              float& d_lo, float& d_hi) {
  asm("{\n\t.reg .b16 xl, xh, wl, wh;\n\t"
      "mov.b32 {xl, xh}, %2;\n\tmov.b32 {wl, wh}, %3;\n\t"
      "fma.rn.f32.bf16 %0, xl, wl, %4;\n\tfma.rn.f32.bf16 %1, xh, wh, %5;\n\t}"
      : "=f"(d_lo), "=f"(d_hi)
      : "r"(x), "r"(w), "f"(c_lo), "f"(c_hi));
}

template <typename T, int CPT>
struct ColOps16Packed {
  static constexpr int kCpt = CPT;      // 4 or 8 channels
  static constexpr int kOps = CPT / 2;  // packed pairs
  using Op = uint32_t;
  static constexpr int kWeightBytes = 2;
  static constexpr int kWOps = kOps;
  static constexpr int kVpc = 1;
  __device__ __forceinline__ static void load_x(uint32_t addr, Op (&v)[kOps]) {
    if constexpr (CPT == 8) {
      lds128a(addr, v);
    } else {
      lds64(addr, v);
    }
  }
  __device__ __forceinline__ static void load_w(uint32_t addr, Op (&v)[kWOps]) { load_x(addr, v); }
  __device__ __forceinline__ static void stage_w(uint8_t* dst, T v) { *reinterpret_cast<T*>(dst) = v; }
  __device__ __forceinline__ static void mac(float (&d)[kCpt], const Op (&x)[kOps], const Op (&w)[kWOps],
                                             const float (&c)[kCpt]) {
#pragma unroll
    for (int i = 0; i < kOps; ++i) mixed_fma_pair<T>(x[i], w[i], c[2 * i], c[2 * i + 1], d[2 * i], d[2 * i + 1]);
  }
};

// acc + x.lo * w.lo + x.hi * w.hi with mixed-precision FMAs (fp32 products
// and sums, one rounding each): the two-term dot product of a group's input
// pair with one output channel's weight pair.
template <typename T>
__device__ __forceinline__ float mixed_dot2(uint32_t x, uint32_t w, float c);
template <>
__device__ __forceinline__ float mixed_dot2<__half>(uint32_t x, uint32_t w, float c) {
  float d;
  asm("{\n\t.reg .b16 xl, xh, wl, wh;\n\t.reg .f32 t;\n\t"
      "mov.b32 {xl, xh}, %1;\n\tmov.b32 {wl, wh}, %2;\n\t"
      "fma.rn.f32.f16 t, xl, wl, %3;\n\tfma.rn.f32.f16 %0, xh, wh, t;\n\t}"
      : "=f"(d)
      : "r"(x), "r"(w), "f"(c));
  return d;
}
template <>
__device__ __forceinline__ float mixed_dot2<__nv_bfloat16>(uint32_t x, uint32_t w, float c) {
  float d;
  asm("{\n\t.reg .b16 xl, xh, wl, wh;\n\t.reg .f32 t;\n\t"
      "mov.b32 {xl, xh}, %1;\n\tmov.b32 {wl, wh}, %2;\n\t"
      "fma.rn.f32.bf16 t, xl, wl, %3;\n\tfma.rn.f32.bf16 %0, xh, wh, t;\n\t}"
      : "=f"(d)
      : "r"(x), "r"(w), "f"(c));
  return d;
}

// Groups of two channels: the thread's 4 channels are groups g, g + 1; x
// word i holds group i's input pair, weight word j = 2 * i + k the pair of
// output channel k of group i.  Staged weights are [tap][output channel][2].
template <typename T>
struct ColOps16Group2 {
  static constexpr int kCpt = 4;
  static constexpr int kOps = 2;
  using Op = uint32_t;
  static constexpr int kWeightBytes = 2;
  static constexpr int kWOps = 4;
  static constexpr int kVpc = 2;
  __device__ __forceinline__ static void load_x(uint32_t addr, Op (&v)[kOps]) { lds64(addr, v); }
  __device__ __forceinline__ static void load_w(uint32_t addr, Op (&v)[kWOps]) { lds128a(addr, v); }
  __device__ __forceinline__ static void stage_w(uint8_t* dst, T v) { *reinterpret_cast<T*>(dst) = v; }
  __device__ __forceinline__ static void mac(float (&d)[kCpt], const Op (&x)[kOps], const Op (&w)[kWOps],
                                             const float (&c)[kCpt]) {
#pragma unroll
    for (int j = 0; j < 4; ++j) d[j] = mixed_dot2<T>(x[j >> 1], w[j], c[j]);
  }
};

template <typename T, int FORM>
using ColOps = typename std::conditional<
    FORM == kColGroup2 && sizeof(T) == 2, ColOps16Group2<T>,
    typename std::conditional<
    FORM == kColWide, ColOpsWide<T>,
    typename std::conditional<
        std::is_same<T, float>::value, ColOpsF32,
        typename std::conditional<
            FORM == kColPacked8, ColOps16Packed<T, 8>,
            typename std::conditional<FORM == kColPacked, ColOps16Packed<T, 4>,
                                      ColOps16Split<T>>::type>::type>::type>::type>::type;

// Channels per thread of a (storage type, form) pair, for the host planner.
inline int col_cpt(int es, int form) { return (es == 2 && form == kColPacked8) ? 8 : 4; }

// Kc for one thread's CPT outputs: round to T, one vector store.
template <typename T, int CPT>
__device__ __forceinline__ void col_store(T* dst, const float (&acc)[CPT]) {
  if constexpr (std::is_same<T, float>::value) {
    static_assert(CPT == 4, "fp32 stores 4 channels");
    *reinterpret_cast<float4*>(dst) = make_float4(acc[0], acc[1], acc[2], acc[3]);
  } else {
    uint32_t wd[CPT / 2];
#pragma unroll
    for (int i = 0; i < CPT / 2; ++i) {
      if constexpr (std::is_same<T, __half>::value) {
        const __half2 h = __floats2half2_rn(acc[2 * i], acc[2 * i + 1]);
        wd[i] = *reinterpret_cast<const uint32_t*>(&h);
      } else {
        const __nv_bfloat162 h = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
        wd[i] = *reinterpret_cast<const uint32_t*>(&h);
      }
    }
    if constexpr (CPT == 8) {
      *reinterpret_cast<uint4*>(dst) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
    } else {
      *reinterpret_cast<uint2*>(dst) = make_uint2(wd[0], wd[1]);
    }
  }
}

// The same, stored only where `pred` holds.
template <typename T, int CPT>
__device__ __forceinline__ void col_store_if(T* dst, const float (&acc)[CPT], bool pred) {
  uint32_t wd[4];
  if constexpr (std::is_same<T, float>::value) {
    static_assert(CPT == 4, "fp32 stores 4 channels");
#pragma unroll
    for (int i = 0; i < 4; ++i) wd[i] = __float_as_uint(acc[i]);
  } else {
#pragma unroll
    for (int i = 0; i < CPT / 2; ++i) {
      if constexpr (std::is_same<T, __half>::value) {
        const __half2 h = __floats2half2_rn(acc[2 * i], acc[2 * i + 1]);
        wd[i] = *reinterpret_cast<const uint32_t*>(&h);
      } else {
        const __nv_bfloat162 h = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
        wd[i] = *reinterpret_cast<const uint32_t*>(&h);
      }
    }
  }
  // the conversion runs unconditionally and only the store is guarded, so
  // the guard compiles to a predicated store rather than a branch
  if constexpr (std::is_same<T, float>::value || CPT == 8) {
    if (pred) *reinterpret_cast<uint4*>(dst) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
  } else {
    if (pred) *reinterpret_cast<uint2*>(dst) = make_uint2(wd[0], wd[1]);
  }
}

// Per-stage tile header, written by the producer before it arms the stage's
// barrier: the output element index of the tile origin (n, od, oh0, ow0, c0)
// and the tile's first output row, rows, first column and first channel.
struct ColTile {
  int64_t y_base;
  int oh0, nrows, ow0, c0;
  int pad[2];
};
static_assert(sizeof(ColTile) == 32, "tile header is 32 bytes");

// Shared-memory layout: [full mbarriers x4][empty mbarriers x4][second-copy
// mbarriers x4][tile headers x4][weights [9][C], at most 4 bytes per
// value][bias fp32 [C]] ... [stages, 1024-aligned].
constexpr uint32_t kColHeaderOff = 128;  // after 3 x kDwMaxStages mbarriers (full, full1, empty)
constexpr uint32_t kColWeightOff = kColHeaderOff + 32u * kDwMaxStages;
__host__ __device__ inline uint32_t col_fixed_smem_bytes(int C) {
  return kColWeightOff + 36u * (uint32_t)C + 4u * (uint32_t)C;
}

// Column state shared by the per-row steps: shared-memory address of the
// thread's piece in row 0 of the stage, strides, the store window and the
// register-resident weights, bias and live accumulators.
template <typename T, int FORM, int NA>
struct ColState {
  using Ops = ColOps<T, FORM>;
  uint32_t st, row_pitch, col_step;
  int nrows;
  bool store_ok;
  int64_t y_row_step;
  const typename Ops::Op (&wr)[3][3][Ops::kWOps];
  const float (&br)[Ops::kCpt];
  float (&acc)[NA][Ops::kCpt];
};

// Filter row ky of input row u (u = row index within its block) lands on
// output row (u - ky*DL) / S of the block when the division is exact.
template <int S, int DL>
__host__ __device__ constexpr bool col_hits(int u, int ky) { return ((u - ky * DL) % S) == 0; }
template <int S, int DL>
__host__ __device__ constexpr bool col_row_used(int u) {
  return col_hits<S, DL>(u, 0) || col_hits<S, DL>(u, 1) || col_hits<S, DL>(u, 2);
}

// Add input row xv into the output row it sits under with filter row KY;
// the slot (output row mod NA) is a compile-time constant.  Output rows
// above the tile (oh < 0) or below it (oh >= rows) are accumulated like any
// other, into slots no valid row holds at that moment, and never stored, so
// the row walk needs no bounds tests.
template <typename T, int FORM, int S, int DL, int NA, int U_, int KY>
__device__ __forceinline__ void col_tap_row(ColState<T, FORM, NA>& c, const typename ColOps<T, FORM>::Op (&xv)[3][ColOps<T, FORM>::kOps],
                                            int oh_base, T* const (&yp)[NA]) {
  using Ops = ColOps<T, FORM>;
  if constexpr (col_hits<S, DL>(U_, KY)) {
    constexpr int rel = (U_ - KY * DL) / S;  // output row - oh_base (exact)
    constexpr int slot = ((rel % NA) + NA) % NA;
    if constexpr (KY == 0) {
      Ops::mac(c.acc[slot], xv[0], c.wr[KY][0], c.br);  // the bias is the first addend
    } else {
      Ops::mac(c.acc[slot], xv[0], c.wr[KY][0], c.acc[slot]);
    }
    Ops::mac(c.acc[slot], xv[1], c.wr[KY][1], c.acc[slot]);
    Ops::mac(c.acc[slot], xv[2], c.wr[KY][2], c.acc[slot]);
    if constexpr (KY == 2) {
      static_assert(rel <= 0 && rel > -NA, "a finished output row lies in this block's window");
      const bool ok = c.store_ok & ((unsigned)(oh_base + rel) < (unsigned)c.nrows);
      col_store_if<T, Ops::kCpt>(yp[-rel], c.acc[slot], ok);
    }
  }
}

// Input row r0 + U_ of the column: three shared loads (horizontal taps), then
// the filter rows it sits under.  Returns false (and does nothing) past the
// last halo row when CHECK is set.
template <typename T, int FORM, int S, int DL, int NA, bool CHECK, int U_>
__device__ __forceinline__ bool col_row(ColState<T, FORM, NA>& c, int r0, int Hh, int oh_base, T* const (&yp)[NA]) {
  using Ops = ColOps<T, FORM>;
  if constexpr (!col_row_used<S, DL>(U_)) {
    return true;
  } else {
    if (CHECK && r0 + U_ >= Hh) return false;
    typename Ops::Op xv[3][Ops::kOps];
    const uint32_t rb = c.st + (uint32_t)(r0 + U_) * c.row_pitch;
    Ops::load_x(rb, xv[0]);
    Ops::load_x(rb + c.col_step, xv[1]);
    Ops::load_x(rb + 2 * c.col_step, xv[2]);
    col_tap_row<T, FORM, S, DL, NA, U_, 0>(c, xv, oh_base, yp);
    col_tap_row<T, FORM, S, DL, NA, U_, 1>(c, xv, oh_base, yp);
    col_tap_row<T, FORM, S, DL, NA, U_, 2>(c, xv, oh_base, yp);
    return true;
  }
}

// One block of U input rows starting at r0 (a multiple of U, so every block
// starts at an output row that is a multiple of NA and the accumulator slot
// of each (row, filter row) pair is the same in every block).  Expanded at
// compile time over the U rows.
// yb points at output row oh_base of the thread's column; the rows a block
// finishes are oh_base - NA + 1 .. oh_base, whose addresses are formed once
// per block.
template <typename T, int FORM, int S, int DL, int NA, bool CHECK, int... Us>
__device__ __forceinline__ void col_block(ColState<T, FORM, NA>& c, int r0, int Hh, T* yb,
                                          std::integer_sequence<int, Us...>) {
  const int oh_base = r0 / S;
  T* yp[NA];
  yp[0] = yb;
#pragma unroll
  for (int i = 1; i < NA; ++i) yp[i] = yp[i - 1] - c.y_row_step;
  (void)(col_row<T, FORM, S, DL, NA, CHECK, Us>(c, r0, Hh, oh_base, yp) && ...);
}

template <typename T, int S, int DL, int FORM>
__global__ void __maxnreg__((col_reg_cap<T, S, DL>(FORM))) dw_col_kernel(const __grid_constant__ CUtensorMap xmap,
                                                                  const __grid_constant__ CUtensorMap xmap0,
                                                                  const __grid_constant__ CUtensorMap xmap1,
                                                                  const DwArgs a) {
  using Ops = ColOps<T, FORM>;
  using Op = typename Ops::Op;
  constexpr int CPT = Ops::kCpt;
  constexpr int es = sizeof(T);
  constexpr int NA = (2 * DL) / S + 1;  // live output rows
  constexpr int U = NA * S;             // input rows per block
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kDwMaxStages;
  uint64_t* full1 = empty + kDwMaxStages;  // second copy of each tile
  const bool split = a.h0 < a.Hh;
  ColTile* hdr = reinterpret_cast<ColTile*>(smem + kColHeaderOff);
  uint8_t* w_s = smem + kColWeightOff;
  float* b_s = reinterpret_cast<float*>(smem + kColWeightOff + 36u * (uint32_t)a.C);
  uint8_t* stage0 = smem + a.stage_off;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int ncons = (int)blockDim.x - 32;
  const T* __restrict__ wg = static_cast<const T*>(a.w);
  const T* __restrict__ bg = static_cast<const T*>(a.bias);
  T* __restrict__ yg = static_cast<T*>(a.y);

  // Stride 2 computes a quarter of the outputs per input byte, so its CTAs
  // are bandwidth-bound and let the next kernel's CTAs launch at once.  At
  // stride 1 they are issue-bound: the next kernel's CTAs, resident beside
  // them while they wait on this grid, measured about 1 us slower per
  // launch, so the dependents launch only as this grid's CTAs exit.
  if constexpr (S == 2) allow_dependent_launch();
  if (tid == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&full1[s], 1);
      mbar_init(&empty[s], (uint32_t)(ncons / 32));
    }
    fence_mbar_init();
    tma_prefetch_desc(&xmap);
    if (split) {
      tma_prefetch_desc(&xmap0);
      tma_prefetch_desc(&xmap1);
    }
  }
  __syncthreads();
  // At stride 2, where this grid's CTAs launch early and wait, the producer
  // decodes its first tile (four dependent integer divisions) before its
  // wait on the previous grid, so the first copy goes out as soon as the
  // wait ends; the empty asm keeps the decode ahead of the wait.  (At stride
  // 1 the CTAs start as the previous grid's exit, and the same code measured
  // 2-3% slower.)
  TileCoord first{};
  if constexpr (S == 2) {
    if (tid == 0 && (int64_t)blockIdx.x < a.num_tiles) {
      first = decode_tile(a, blockIdx.x);
      asm volatile("" ::"r"(first.ct), "r"(first.tw), "r"(first.th), "r"(first.od), "r"(first.n));
    }
  }
  grid_dependency_wait();  // x, w, bias and y are touched only from here on

  const bool withhold = (a.test_flags & 1) && blockIdx.x == 0;
  if (warp == 0) {
    // ---------------- producer ----------------
    // Starts copying at once; the consumers stage the weights meanwhile.
    if (lane == 0) {
      int k = 0, s = 0;
      bool failed = false;
      for (;; ++k) {
        const int64_t tile = blockIdx.x + (int64_t)k * gridDim.x;
        if (tile >= a.num_tiles) break;
        if (k >= a.stages &&
            !mbar_wait(&empty[s], (uint32_t)(((k / a.stages) - 1) & 1), a.wait_limit_ns)) {
          failed = true;
          break;
        }
        // At launch every CTA requests its first tiles at once.  Holding the
        // second copy until the first has landed lets the first tile arrive
        // (and its computation start) sooner; later copies overlap compute.
        if (k == 1 && !withhold && !mbar_wait(&full[0], 0u, a.wait_limit_ns)) {
          failed = true;
          break;
        }
        if (!(withhold && k == 0)) {
          const TileCoord c = (S == 2 && k == 0) ? first : decode_tile(a, tile);
          ColTile h;
          h.oh0 = c.th * a.TH;
          h.nrows = min(a.TH, a.Ho - h.oh0);
          h.ow0 = c.tw * a.TW;
          h.c0 = c.ct * a.TC;
          h.y_base = ((((int64_t)c.n * a.Do + c.od) * a.Ho + h.oh0) * (int64_t)a.Wo + h.ow0) * a.C + h.c0;
          hdr[s] = h;  // published to the consumers by the barrier arrive below
          uint8_t* dst = stage0 + (size_t)s * a.stage_stride;
          const int iw = h.ow0 * S - a.pW, ih = h.oh0 * S - a.pH, id = c.od * a.sD - a.pD;
          if (!(split && k == 0)) {
            mbar_arrive_expect_tx(&full[s], a.stage_bytes);
            tma_load_5d(dst, &xmap, &full[s], h.c0, iw, ih, id, (int)c.n);
          } else {
            mbar_arrive_expect_tx(&full[s], a.bytes0);
            tma_load_5d(dst, &xmap0, &full[s], h.c0, iw, ih, id, (int)c.n);
            mbar_arrive_expect_tx(&full1[s], a.stage_bytes - a.bytes0);
            tma_load_5d(dst + a.bytes0, &xmap1, &full1[s], h.c0, iw, ih + a.h0, id, (int)c.n);
          }
        }
        if (++s == a.stages) s = 0;
      }
      if (failed) report(a.status, kDevTimeout, 2);
      for (int j = k > a.stages ? k - a.stages : 0; j < k; ++j) {
        if (withhold && j == 0) continue;
        mbar_wait(&full[j % a.stages], (uint32_t)((j / a.stages) & 1), a.wait_limit_ns);
        if (split && j == 0) mbar_wait(&full1[0], 0u, a.wait_limit_ns);
      }
    }
    return;
  }

  // ---------------- consumers ----------------
  const int ctid = tid - 32;
  // weights [c][tap] in global -> [tap][c] in shared; bias -> fp32 (consumer
  // warps only, while the first copies are in flight)
  // (global reads in source order: coalesced; four loads in flight per thread)
  // (w is [output channel][tap][input channel of the group]: kVpc values per
  // tap and output channel; staged as [tap][output channel][kVpc])
  constexpr int VPC = Ops::kVpc;
  const int nw = 9 * VPC * a.C;
  for (int i0 = ctid; i0 < nw; i0 += 4 * ncons) {
    T v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * ncons;
      if (i < nw) v[u] = wg[i];
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * ncons;
      if (i < nw) {
        const int ch = i / (9 * VPC), r = i - ch * (9 * VPC);
        const int t = r / VPC, e = r - t * VPC;
        Ops::stage_w(w_s + (((size_t)t * a.C + ch) * VPC + e) * Ops::kWeightBytes, v[u]);
      }
    }
  }
  for (int i = ctid; i < a.C; i += ncons) b_s[i] = bg != nullptr ? Elem<T>::to_f32(bg[i]) : 0.f;
  asm volatile("bar.sync 1, %0;" ::"r"(ncons) : "memory");

  const int NQ = a.TC / CPT;
  const int q = ctid % NQ;
  const int wl = ctid / NQ;
  const bool active = wl < a.TW;
  const uint32_t row_pitch = (uint32_t)(a.Wh * a.TC * es);
  const uint32_t col_step = (uint32_t)(DL * a.TC * es);
  const uint32_t lane_off = (uint32_t)(((wl * S) * a.TC + q * CPT) * es);
  const int64_t y_row_step = (int64_t)a.Wo * a.C;
  const int64_t thread_off = (int64_t)wl * a.C + q * CPT;
  const int Hh = a.Hh;

  Op wr[3][3][Ops::kWOps];
  float br[CPT];
  int cur_c0 = -1;
  int s = 0;
  uint32_t parity = 0;
  for (int k = 0;; ++k) {
    const int64_t tile = blockIdx.x + (int64_t)k * gridDim.x;
    if (tile >= a.num_tiles) break;

    // Lane 0 polls; after the warp agrees, every lane observes the completed
    // phase itself (acquire) before reading the stage.
    auto warp_wait = [&](uint64_t* bar) {
      bool ok = true;
      if (lane == 0) ok = mbar_wait(bar, parity, a.wait_limit_ns);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (ok && lane != 0) ok = mbar_wait(bar, parity, a.wait_limit_ns);
      return __all_sync(0xffffffffu, ok);
    };
    if (!warp_wait(&full[s])) {
      if (lane == 0) report(a.status, kDevTimeout, 1);
      return;
    }

    const ColTile h = hdr[s];
    // Every lane of the warp walks the rows (the waits are warp-wide); lanes
    // without a column or channel of this tile read row 0 of their stage and
    // store nothing.
    const int ch = h.c0 + q * CPT;
    const bool act = active && ch < a.C;
    const int chl = act ? ch : 0;
    if (h.c0 != cur_c0) {  // weights and bias of this channel tile
      cur_c0 = h.c0;
#pragma unroll
      for (int t = 0; t < 9; ++t)
        Ops::load_w(smem_u32(w_s + ((size_t)t * a.C + chl) * VPC * Ops::kWeightBytes), wr[t / 3][t % 3]);
#pragma unroll
      for (int i = 0; i < CPT; i += 4) {
        const float4 b4 = *reinterpret_cast<const float4*>(b_s + chl + i);
        br[i] = b4.x, br[i + 1] = b4.y, br[i + 2] = b4.z, br[i + 3] = b4.w;
      }
    }
    const bool store_ok = act && h.ow0 + wl < a.Wo;
    T* yb = yg + h.y_base + thread_off;
    const uint32_t st = smem_u32(stage0 + (size_t)s * a.stage_stride) + (act ? lane_off : 0u);
    float acc[NA][CPT];
#pragma unroll
    for (int i = 0; i < NA; ++i)
#pragma unroll
      for (int e = 0; e < CPT; ++e) acc[i][e] = 0.f;
    ColState<T, FORM, NA> cs{st, row_pitch, col_step, h.nrows, store_ok, y_row_step, wr, br, acc};
    int r0 = 0;
    bool have1 = !(split && k == 0);  // first tile: rows from h0 on are in the second copy
    for (; r0 + U <= Hh; r0 += U, yb += NA * y_row_step) {
      if (!have1 && r0 + U > a.h0) {
        if (!warp_wait(&full1[s])) {
          if (lane == 0) report(a.status, kDevTimeout, 1);
          return;
        }
        have1 = true;
      }
      col_block<T, FORM, S, DL, NA, false>(cs, r0, Hh, yb, std::make_integer_sequence<int, U>{});
    }
    if (r0 < Hh) {
      if (!have1 && !warp_wait(&full1[s])) {
        if (lane == 0) report(a.status, kDevTimeout, 1);
        return;
      }
      col_block<T, FORM, S, DL, NA, true>(cs, r0, Hh, yb, std::make_integer_sequence<int, U>{});
    }

    __syncwarp();  // this warp is done with stage s
    if (lane == 0) mbar_arrive(&empty[s]);
    if (++s == a.stages) {
      s = 0;
      parity ^= 1u;
    }
  }
}

}  // namespace dw
}  // namespace gconv
