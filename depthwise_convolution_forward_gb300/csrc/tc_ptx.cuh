// Inline-PTX wrappers for the 5th-generation tensor cores (tcgen05) and
// tensor memory (TMEM) on sm_100-class GPUs, written from the PTX ISA.
#pragma once

#include "common.cuh"

namespace gconv {
namespace tc {

// --- TMEM allocation (one full warp executes each of these) ---------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// --- ordering between tcgen05 operations and thread synchronisation -------
__device__ __forceinline__ void fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// --- MMA: D(tmem, fp32) (+)= A(smem) x B(smem)^T, kind::f16 (f16 or bf16) --
// No "memory" clobber: the operands are ordered by the mbarrier waits and
// fences around the issue loop (all volatile asm with clobbers, which this
// statement is never reordered across), and leaving ordinary loads free lets
// the compiler fetch the next MMA's descriptors while this one issues.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}
// Arrive once on `bar` when every tcgen05 operation this thread issued so far
// has completed.
__device__ __forceinline__ void commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// --- TMEM -> registers: 32 lanes x 16 consecutive 32-bit columns ----------
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// --- descriptors ---------------------------------------------------------
// Shared-memory matrix descriptor, no swizzle, K-major canonical layout:
// core matrices of 8 rows x 16 bytes (rows contiguous, 128 bytes per core
// matrix); `lbo` = byte distance between the two core matrices adjacent in
// K (one MMA covers K = 2 x 8 16-bit elements), `sbo` = byte distance between
// core matrices adjacent in M (or N), i.e. between 8-row groups.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1u << 46;  // fixed descriptor version bits for tcgen05
  return d;                 // base offset 0, relative LBO, swizzle none
}

// Shared-memory matrix descriptor, 128-byte swizzle, K-major: rows of 128
// bytes (64 16-bit elements of K), 8-row atoms of 1024 bytes (SBO), the
// 16-byte chunk c of a row stored at c ^ (address bits 7..9).  The swizzle
// phase comes from the absolute shared-memory address of each row -- the same
// rule TMA applies when it writes 1024-byte-aligned atoms -- so a start
// address shifted by any whole number of rows reads those rows correctly with
// the base-offset field left at 0 (verified against the oracle for shifts
// that are and are not multiples of 8 rows).  K-steps inside a row advance
// the start by 32 bytes.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((1024u >> 4) & 0x3FFFu) << 32;  // SBO: 8 rows x 128 B
  d |= (uint64_t)1u << 46;                        // fixed descriptor version bits
  d |= (uint64_t)2u << 61;                        // layout: 128-byte swizzle
  return d;
}

// Instruction descriptor of kind::f16 with fp32 accumulation, both operands
// K-major, dense.  bf16 = true selects bf16 inputs, else f16.
__host__ __device__ constexpr uint32_t idesc_f16(bool bf16, int M, int N) {
  return (1u << 4)                          // D format: f32
         | ((bf16 ? 1u : 0u) << 7)          // A format
         | ((bf16 ? 1u : 0u) << 10)         // B format
         | ((uint32_t)(N >> 3) << 17)       // N / 8
         | ((uint32_t)(M >> 4) << 24);      // M / 16
}

}  // namespace tc
}  // namespace gconv
