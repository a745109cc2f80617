// Shared device helpers for the grouped-convolution kernels: element traits,
// the fused bias + cast epilogue, mbarrier / TMA wrappers and the bounded
// waits that report a timeout through a status word instead of hanging.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"

namespace gconv {

// ---------------------------------------------------------------------------
// Element traits: storage type <-> fp32, 16-byte vectors.
// ---------------------------------------------------------------------------
template <typename T> struct Elem;
template <> struct Elem<float> {
  static constexpr int kVec = 4;  // elements per 16-byte vector
  __device__ __forceinline__ static float to_f32(float v) { return v; }
  __device__ __forceinline__ static float from_f32(float v) { return v; }
};
template <> struct Elem<__half> {
  static constexpr int kVec = 8;
  __device__ __forceinline__ static float to_f32(__half v) { return __half2float(v); }
  __device__ __forceinline__ static __half from_f32(float v) { return __float2half_rn(v); }
};
template <> struct Elem<__nv_bfloat16> {
  static constexpr int kVec = 8;
  __device__ __forceinline__ static float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
  __device__ __forceinline__ static __nv_bfloat16 from_f32(float v) { return __float2bfloat16_rn(v); }
};

// Widen the two 16-bit (or one 32-bit) values packed in a 32-bit word.
// Bit operations on whole words keep the compiler from splitting the
// 128-bit load that produced them into narrow loads.
template <typename T>
__device__ __forceinline__ void widen_word(uint32_t w, float* out);
template <>
__device__ __forceinline__ void widen_word<float>(uint32_t w, float* out) {
  out[0] = __uint_as_float(w);
}
template <>
__device__ __forceinline__ void widen_word<__half>(uint32_t w, float* out) {
  out[0] = __half2float(__ushort_as_half((unsigned short)(w & 0xffffu)));
  out[1] = __half2float(__ushort_as_half((unsigned short)(w >> 16)));
}
template <>
__device__ __forceinline__ void widen_word<__nv_bfloat16>(uint32_t w, float* out) {
  out[0] = __uint_as_float(w << 16);
  out[1] = __uint_as_float(w & 0xffff0000u);
}

// Unpack one 16-byte vector (as four words) into fp32 values.
template <typename T>
__device__ __forceinline__ void unpack16(const uint32_t (&v)[4], float* out) {
  constexpr int per = 4 / sizeof(T) > 0 ? (int)(4 / sizeof(T)) : 1;
#pragma unroll
  for (int i = 0; i < 4; ++i) widen_word<T>(v[i], out + i * per);
}
template <typename T>
__device__ __forceinline__ void unpack16(const uint4& v, float* out) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  unpack16<T>(w, out);
}

// 128-bit shared-memory load (always one LDS.128).
__device__ __forceinline__ void lds128(const void* p, uint32_t (&v)[4]) {
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
               : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))));
}

// acc += lo/hi half of x * lo/hi half of w, product and sum in fp32 with a
// single rounding (PTX mixed-precision fma, sm_100+).
template <typename T>
__device__ __forceinline__ void fma_mixed_pair(uint32_t x, uint32_t w, float& acc_lo, float& acc_hi);
template <>
__device__ __forceinline__ void fma_mixed_pair<__half>(uint32_t x, uint32_t w, float& lo, float& hi) {
  asm("{\n\t.reg .b16 xl, xh, wl, wh;\n\t"
      "mov.b32 {xl, xh}, %2;\n\tmov.b32 {wl, wh}, %3;\n\t"
      "fma.rn.f32.f16 %0, xl, wl, %0;\n\tfma.rn.f32.f16 %1, xh, wh, %1;\n\t}"
      : "+f"(lo), "+f"(hi)
      : "r"(x), "r"(w));
}
template <>
__device__ __forceinline__ void fma_mixed_pair<__nv_bfloat16>(uint32_t x, uint32_t w, float& lo, float& hi) {
  asm("{\n\t.reg .b16 xl, xh, wl, wh;\n\t"
      "mov.b32 {xl, xh}, %2;\n\tmov.b32 {wl, wh}, %3;\n\t"
      "fma.rn.f32.bf16 %0, xl, wl, %0;\n\tfma.rn.f32.bf16 %1, xh, wh, %1;\n\t}"
      : "+f"(lo), "+f"(hi)
      : "r"(x), "r"(w));
}

// ---------------------------------------------------------------------------
// Kc: fused epilogue.  acc (fp32) + bias (already widened to fp32), then one
// round-to-nearest-even cast to the output type.  The single rounding step is
// the only place output precision is lost.
// ---------------------------------------------------------------------------
template <typename T>
__device__ __forceinline__ T epilogue_one(float acc, float bias) {
  return Elem<T>::from_f32(acc + bias);
}

// Two consecutive outputs packed into one word (low half = first channel):
// the same round-to-nearest-even of (acc + bias) as epilogue_one, done by
// one paired conversion.
template <typename T>
__device__ __forceinline__ uint32_t epilogue_pair(float a0, float a1, float b0, float b1);
template <>
__device__ __forceinline__ uint32_t epilogue_pair<__half>(float a0, float a1, float b0, float b1) {
  const __half2 h = __floats2half2_rn(a0 + b0, a1 + b1);
  return *reinterpret_cast<const uint32_t*>(&h);
}
template <>
__device__ __forceinline__ uint32_t epilogue_pair<__nv_bfloat16>(float a0, float a1, float b0, float b1) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a0 + b0, a1 + b1);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// VEC consecutive outputs -> one aligned vector store (VEC * sizeof(T) bytes).
template <typename T, int VEC>
__device__ __forceinline__ void epilogue_store(T* dst, const float* acc, const float* bias) {
  static_assert((VEC * sizeof(T)) % 4 == 0, "vector store must be whole words");
  constexpr int kWords = VEC * sizeof(T) / 4;
  uint32_t words[kWords];
  T* e = reinterpret_cast<T*>(words);
#pragma unroll
  for (int i = 0; i < VEC; ++i) e[i] = epilogue_one<T>(acc[i], bias[i]);
  if constexpr (kWords == 4) {
    *reinterpret_cast<uint4*>(dst) = make_uint4(words[0], words[1], words[2], words[3]);
  } else if constexpr (kWords == 2) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(words[0], words[1]);
  } else if constexpr (kWords == 8) {
    uint4* d4 = reinterpret_cast<uint4*>(dst);
    d4[0] = make_uint4(words[0], words[1], words[2], words[3]);
    d4[1] = make_uint4(words[4], words[5], words[6], words[7]);
  } else {
#pragma unroll
    for (int i = 0; i < kWords; ++i) reinterpret_cast<uint32_t*>(dst)[i] = words[i];
  }
}

// ---------------------------------------------------------------------------
// Status word (two ints: code, where).  First writer wins.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void report(int* status, int code, int where) {
  if (status != nullptr && atomicCAS(status, 0, code) == 0) atomicExch(status + 1, where);
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  allow_dependent_launch() lets the next
// kernel in the stream begin launching its CTAs once every CTA of this grid
// has called it (or exited); those CTAs then occupy only resources this grid
// leaves free.  grid_dependency_wait() returns once the previous grid in the
// stream has completed and its memory operations are visible; it returns at
// once when the kernel was not launched as a dependent.  Neither is a spin
// loop in the kernel.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void allow_dependent_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait on phase `parity`.  Returns false once `limit_ns` of wall time
// (the GPU global timer) has passed without the phase completing.
// mbarrier.try_wait already suspends the thread in hardware for a while
// before it reports an incomplete phase, so the loop polls back to back and
// reads the timer only every 64 polls.  A sleep between polls (exponential
// back-off up to 256 ns) measured 1-4% slower on every kernel on GB300: a
// waiter woke up to a back-off interval after its phase completed.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// ---------------------------------------------------------------------------
// TMA (tiled tensor copies global -> shared, completion on an mbarrier)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
__device__ __forceinline__ void tma_load_5d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0,
                                            int c1, int c2, int c3, int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
      "r"(c4)
      : "memory");
}
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0,
                                            int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                                            int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
// Plain bulk copy (no tensor map): both addresses 16-byte aligned, size % 16 == 0.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// TMA tensor store shared -> global of one box (5-D coordinates, innermost
// first), tracked by the issuing thread's bulk async-group.  Out-of-range
// parts of the box are not written.
__device__ __forceinline__ void tma_store_5d(const CUtensorMap* map, const void* src, int c0, int c1, int c2, int c3,
                                             int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5, %6}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
      : "memory");
}
__device__ __forceinline__ void tma_store_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Until every committed store of this thread has finished reading shared memory.
__device__ __forceinline__ void tma_store_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Until every committed store of this thread has completed.
__device__ __forceinline__ void tma_store_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

}  // namespace gconv
