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
//  * Warps 1-4 (kIssuers warps, one lane each) issue tcgen05.mma (M = 128,
//    N = m*Kg, K = 16) into fp32 accumulators in tensor memory, in two to
//    four buffers across tiles (as many as the 512 columns hold): the MMAs
//    of tile k wait only for the epilogue of tile k - nbuf.  The tile's
//    accumulators, and partial
//    accumulators that each sum a share of the taps, are dealt to the
//    issuers, so four MMA streams run at once; each issuer signals completion
//    with tcgen05.commit on mbarriers.
//  * Warps 5-8 (four epilogue warps, one per TMEM lane quarter) read the
//    accumulators (tcgen05.ld), add the partials, apply the fused bias +
//    round-to-nearest-even epilogue and store channels-last output.
//  * All waits are bounded; on expiry every role reports a timeout, waits
//    (bounded) for its in-flight copies / MMAs, and the CTA frees its tensor
//    memory before exiting.
#pragma once

#include "tc_ptx.cuh"

namespace gconv {
namespace tc {

constexpr int kMaxTaps = 32;
constexpr int kMaxPhases = 8;  // A planes per stage: stride phases (x column shift copies in aligned mode)
constexpr int kMaxStages = 4;
constexpr int kMaxAccBufs = 4;                    // accumulator buffers in tensor memory
constexpr int kMaxTab = 2048;                     // host-built MMA list entries
constexpr int kIssuers = 4;                       // MMA-issuing warps
constexpr int kThreads = 32 * (1 + kIssuers + 4);  // producer, issuers, epilogue

struct TcArgs {
  const void* w;
  const void* bias;
  void* y;
  int G, Cg, Kg, m;        // groups, channels per group, merge factor
  int Do, Ho, Wo, Ktot;    // output extents, output channels
  int sD, pD, taps_total;  // depth stride / pad, taps per filter
  int TH, TWo, P, Hh, Dh;  // tile rows / cols, halo pitch, halo rows, halo planes
  int s, qy_min, qx_min;   // spatial stride, phase-row origin offsets
  int nphase;              // A planes per stage
  int phase_py[kMaxPhases], phase_px[kMaxPhases];  // the stride phase each plane holds
  int plane_cx[kMaxPhases];  // column shift of the plane's copy (aligned mode), else 0
  int ntaps;
  int tap_phase[kMaxTaps], tap_off[kMaxTaps];
  int nchunks, Kt, Nn, KS, nmt;
  int sc;                  // group chunks per 128-byte row (swizzled layout), else 1
  int np;                  // partial accumulators per accumulator (taps split np ways)
  int shift;               // <= 0: accumulator row f holds flattened output f + shift (8-row A alignment)
  int nbuf;                // accumulator buffers (2..kMaxAccBufs): tile k uses buffer k % nbuf
  uint32_t plane_stride, a_stage_bytes, tx_bytes;
  uint32_t a_off, b_off, bias_off, tab_off;  // smem offsets (tab: MMA descriptor table)
  uint32_t epi_off;  // output-box staging for TMA tensor stores, or 0 to store straight from registers
  uint32_t epi_slice_bytes;  // staging bytes of one channel slice (1024-aligned)
  int epi_w, epi_slices;     // bytes per pixel of a slice (128, 64 or 32) and slices per CTA row
  int w_tma;         // 1: weights staged by TMA through the weight tensor map (Cg, Kg % 8 == 0)
  int w_box_taps;    // taps one weight box covers: all of them (one group per chunk) or 1
  int stages;
  uint32_t tmem_cols, idesc;
  int n_gc, cpg, tiles_w, tiles_h;
  int spatial_tiles;
  int* status;
  uint64_t wait_limit_ns;
  int test_flags;
  OutMap om;  // output placement (off: y in the plain NHWGK layout)
  // MMA lists computed on the host (ntab entries, issuer lists back to back),
  // or ntab = 0 to build them in the kernel.  Entry: x = A start offset >> 4
  // | B start offset >> 4 << 16 (bytes from the dynamic shared-memory base,
  // stage 0), y = accumulator column | flags << 16 (bit 0 accumulate, bit 1
  // skip).
  int ntab;
  uint2 tab[kMaxTab];
};

struct SpatialTile {
  int n, od, oh0, ow0;
};

// A CTA's spatial tiles sp0, sp0 + step, ... with sp = ((n * Do + od) *
// tiles_h + th) * tiles_w + tw: the digits (tw, th, od, n) of the tile index
// are advanced by the digits of the step with carries, so a tile costs no
// integer division (a runtime divide is a chain of about 150 cycles, and the
// epilogue of every tile used to wait on three).  Each digit sum stays below
// twice its radix, so one carry per digit is enough.
struct SpatialWalk {
  int tw, th, od, n;
  int dtw, dth, dod, dn;
  __device__ __forceinline__ void init(const TcArgs& a, int sp, int step) {
    tw = sp % a.tiles_w, sp /= a.tiles_w;
    th = sp % a.tiles_h, sp /= a.tiles_h;
    od = sp % a.Do, n = sp / a.Do;
    dtw = step % a.tiles_w, step /= a.tiles_w;
    dth = step % a.tiles_h, step /= a.tiles_h;
    dod = step % a.Do, dn = step / a.Do;
  }
  __device__ __forceinline__ void advance(const TcArgs& a) {
    tw += dtw;
    int c = tw >= a.tiles_w;
    if (c) tw -= a.tiles_w;
    th += dth + c;
    c = th >= a.tiles_h;
    if (c) th -= a.tiles_h;
    od += dod + c;
    c = od >= a.Do;
    if (c) od -= a.Do;
    n += dn + c;
  }
  __device__ __forceinline__ SpatialTile tile(const TcArgs& a) const {
    SpatialTile t;
    t.n = n, t.od = od, t.oh0 = th * a.TH, t.ow0 = tw * a.TWo;
    return t;
  }
};

// Position in a ring of `size` buffers and the parity of its current pass
// (the k-th use is buffer k % size, pass k / size), advanced without division.
struct Ring {
  int pos = 0, ph = 0;
  __device__ __forceinline__ void next(int size) {
    if (++pos == size) pos = 0, ph ^= 1;
  }
};

// All lanes of a warp wait on `bar`: lane 0 polls (bounded), then every lane
// observes the completed phase itself.  Returns false on timeout.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, uint64_t limit) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, limit);
  ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  if (ok && (threadIdx.x & 31) != 0) ok = mbar_wait(bar, parity, limit);
  return __all_sync(0xffffffffu, ok);
}

// Kc for 16 consecutive channels: bias add, round to T, one 32-byte store
// (a whole sector per lane).  dst must be 32-byte aligned.
template <typename T>
__device__ __forceinline__ void epilogue_store32(T* dst, const float* v, const float* bias) {
  uint32_t wd[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) wd[i] = epilogue_pair<T>(v[2 * i], v[2 * i + 1], bias[2 * i], bias[2 * i + 1]);
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(wd[0]), "r"(wd[1]),
               "r"(wd[2]), "r"(wd[3]), "r"(wd[4]), "r"(wd[5]), "r"(wd[6]), "r"(wd[7])
               : "memory");
}

// Epilogue for one output row of a tile: per batch, load kPer chunks of 16
// channels from each of the NP partial accumulators (one wait per batch),
// sum the partials, add bias, round, store.  A batch holds 64 loaded
// registers with one partial and 32 with two or four partials.  The kernel's
// nine warps cap a thread at 168 registers (three warps share one scheduler's
// 16K registers), and 64 loaded registers of two partials made the kernel
// spill; without spills (and without a division per tile) the tensor-core
// workloads measured 6-17% faster.
template <typename T, int NP>
__device__ __forceinline__ void epilogue_row(uint32_t lane_base, int mt, int G2, int sc, int Nn, bool valid, T* dst,
                                             const float* bias_s, bool v8) {
  constexpr int kPer = NP == 1 ? 4 : 1;  // chunks per batch (see epilogue_row)
  const int nchunk16 = sc * Nn / 16;
  for (int c = 0; c < nchunk16; c += kPer) {
    uint32_t r[kPer][NP][16];
#pragma unroll
    for (int b = 0; b < kPer; ++b) {
      const int cc = c + b;
      if (cc < nchunk16) {
        // chunk j = 16 cc / Nn of the row, column 16 cc % Nn in it: accumulator
        // (p * G2 + mt * sc + j), i.e. column (p * G2 + mt * sc) * Nn + 16 cc
#pragma unroll
        for (int p = 0; p < NP; ++p) tmem_ld16(lane_base + (uint32_t)((p * G2 + mt * sc) * Nn + cc * 16), r[b][p]);
      }
    }
    tmem_ld_wait();
    if (valid) {
#pragma unroll
      for (int b = 0; b < kPer; ++b) {
        const int cc = c + b;
        if (cc < nchunk16) {
          float v[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float sum = __uint_as_float(r[b][0][e]);
#pragma unroll
            for (int p = 1; p < NP; ++p) sum += __uint_as_float(r[b][p][e]);
            v[e] = sum;
          }
          if (v8) {
            epilogue_store32<T>(dst + cc * 16, v, bias_s + cc * 16);
          } else {
            epilogue_store<T, 8>(dst + cc * 16, v, bias_s + cc * 16);
            epilogue_store<T, 8>(dst + cc * 16 + 8, v + 8, bias_s + cc * 16 + 8);
          }
        }
      }
    }
  }
}

// Epilogue for one output row with one partial accumulator, when the CTA's
// channels per pixel are a multiple of 64 (groups of four 16-channel chunks)
// and y is 32-byte aligned.  Lane l holds accumulator row l, i.e. pixel l of
// the warp's 32 consecutive rows; storing each lane's own chunk writes 32 B
// to each of 32 pixels per instruction.  Instead the four lanes 4g .. 4g+3
// exchange their converted chunks (a 4 x 4 transpose of 32-byte blocks in
// two rounds of xor shuffles), after which lane 4g + c holds chunk c of
// pixels 4g .. 4g+3, and each store instruction writes 8 whole 128-byte
// pixel runs.  Removing the stores altogether measured 15-20% faster on the
// tensor-core workloads, so their request count is worth these shuffles.
template <typename T>
__device__ __forceinline__ void epilogue_row_x4(uint32_t lane_base, int mt, int sc, int Nn, bool valid, T* dst,
                                                const float* bias_s) {
  const int nchunk16 = sc * Nn / 16;
  const int lane = threadIdx.x & 31, c = lane & 3, g4 = lane & ~3;
  const bool b0 = (c & 1) != 0, b1 = (c & 2) != 0;
  // destination and validity of the group's four pixels
  T* ds[4];
  bool vs[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    ds[q] = reinterpret_cast<T*>(__shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(dst), g4 + q));
    vs[q] = __shfl_sync(0xffffffffu, valid ? 1 : 0, g4 + q) != 0;
  }
  for (int c0 = 0; c0 < nchunk16; c0 += 4) {
    uint32_t w[4][8];  // converted chunks c0 .. c0+3 of this lane's pixel, two chunks per wait
#pragma unroll
    for (int h = 0; h < 4; h += 2) {
      uint32_t r[2][16];
#pragma unroll
      for (int b = 0; b < 2; ++b) tmem_ld16(lane_base + (uint32_t)(mt * sc * Nn + (c0 + h + b) * 16), r[b]);
      tmem_ld_wait();
#pragma unroll
      for (int b = 0; b < 2; ++b)
#pragma unroll
        for (int i = 0; i < 8; ++i)
          w[h + b][i] = epilogue_pair<T>(__uint_as_float(r[b][2 * i]), __uint_as_float(r[b][2 * i + 1]),
                                         bias_s[(c0 + h + b) * 16 + 2 * i], bias_s[(c0 + h + b) * 16 + 2 * i + 1]);
    }
    // 4 x 4 block transpose over the lane group: swap the off-diagonal blocks
    // of each 2 x 2 block pair across lane bit 0, then of the 2 x 2 super-
    // blocks across lane bit 1; afterwards w[q] = chunk c0 + c of pixel g4 + q.
#pragma unroll
    for (int i = 0; i < 8; ++i) {
#pragma unroll
      for (int x = 0; x < 4; x += 2) {  // pairs (0, 1), (2, 3) on bit 0
        const uint32_t r = __shfl_xor_sync(0xffffffffu, b0 ? w[x][i] : w[x + 1][i], 1);
        if (b0) w[x][i] = r; else w[x + 1][i] = r;
      }
#pragma unroll
      for (int x = 0; x < 2; ++x) {  // pairs (0, 2), (1, 3) on bit 1
        const uint32_t r = __shfl_xor_sync(0xffffffffu, b1 ? w[x][i] : w[x + 2][i], 2);
        if (b1) w[x][i] = r; else w[x + 2][i] = r;
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (vs[q]) {
        T* d = ds[q] + (c0 + c) * 16;
        asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(d), "r"(w[q][0]),
                     "r"(w[q][1]), "r"(w[q][2]), "r"(w[q][3]), "r"(w[q][4]), "r"(w[q][5]), "r"(w[q][6]),
                     "r"(w[q][7])
                     : "memory");
      }
    }
  }
}

// Epilogue for one output row of a stacked-phase problem (OutMap mode 2,
// one partial accumulator, channels per phase a multiple of 16): output
// channel kk = k0 + column is (group, phase, channel), so each 16-column
// piece lies in one phase and lands as one 32-byte run at its dx position,
// when that position lies inside dx.  (group, phase, channel) advance by 16
// channels per piece; the residues are recomputed only when the phase
// changes.  No bias: backward data has none.
template <typename T>
__device__ __forceinline__ void epilogue_row_stacked(uint32_t lane_base, int mt, int sc, int Nn, bool valid, int n,
                                                     int od, int oh, int ow, const OutMap& om, int k0, int Kgs,
                                                     T* y) {
  const int nchunk16 = sc * Nn / 16;
  valid = valid && od >= om.lo[0] && oh >= om.lo[1] && ow >= om.lo[2];
  const int base_d = od * om.scale[0] + om.add[0], base_h = oh * om.scale[1] + om.add[1],
            base_w = ow * om.scale[2] + om.add[2];
  int g = k0 / Kgs;
  const int kp0 = k0 - g * Kgs;
  int ph = kp0 / om.cpp, ch = kp0 - ph * om.cpp;
  int rd = 0, rh = 0, rw = 0, cur = -1;
  const int64_t row = (int64_t)om.ext[1] * om.ext[2];
  for (int cc = 0; cc < nchunk16; ++cc) {
    uint32_t r[16];
    tmem_ld16(lane_base + (uint32_t)(mt * sc * Nn + cc * 16), r);
    tmem_ld_wait();
    if (valid) {
      if (ph != cur) {  // phase ph = (rd * sH + rh) * sW + rw
        cur = ph;
        rw = ph % om.scale[2];
        const int rdh = ph / om.scale[2];
        rh = rdh % om.scale[1], rd = rdh / om.scale[1];
      }
      const int md = base_d + rd, mh = base_h + rh, mw = base_w + rw;
      if (md < om.ext[0] && mh < om.ext[1] && mw < om.ext[2]) {
        T* dst = y + (((int64_t)n * om.ext[0] + md) * row + (int64_t)mh * om.ext[2] + mw) * om.ctot +
                 (int64_t)g * om.cpp + ch;
        uint32_t wd[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          wd[i] = epilogue_pair<T>(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]), 0.f, 0.f);
        asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "r"(wd[0]), "r"(wd[1]), "r"(wd[2]),
                     "r"(wd[3])
                     : "memory");
        asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(dst + 8), "r"(wd[4]), "r"(wd[5]), "r"(wd[6]),
                     "r"(wd[7])
                     : "memory");
      }
    }
    ch += 16;  // next piece: 16 channels on, carrying into the phase and the group
    if (ch == om.cpp) {
      ch = 0;
      if (++ph == om.nph) ph = 0, ++g;
    }
  }
}

// Epilogue into the shared-memory image of the tile's output box, for a
// TMA tensor store.  The box is [TH][TWo][slice of the CTA's channels] per
// channel slice of W bytes per pixel (W = 128, 64 or 32), each slice with the
// TMA swizzle of its width: the 16-byte chunk c of pixel p sits at chunk
// c ^ (bits 7.. of p * W), so the 8 consecutive pixels one warp quarter
// writes land in 8 different bank groups.  Lane = one pixel row of the
// accumulator (f = mt * 128 + row); wrap-around rows (jj >= TWo) and rows
// past the tile (i >= TH) are not part of the box and are skipped.
template <typename T, int NP>
__device__ __forceinline__ void epilogue_row_tma(uint32_t lane_base, int mt, int G2, int sc, int Nn, bool valid,
                                                 int p, const float* bias_s, uint32_t stage_base, uint32_t slice_bytes,
                                                 int W) {
  constexpr int kPer = NP == 1 ? 4 : 1;  // chunks per batch (see epilogue_row)
  const int nchunk16 = sc * Nn / 16;
  const uint32_t swz = ((uint32_t)p * (uint32_t)W >> 7) & (uint32_t)(W / 16 - 1);
  const uint32_t row_addr = stage_base + (uint32_t)p * (uint32_t)W;
  for (int c = 0; c < nchunk16; c += kPer) {
    uint32_t r[kPer][NP][16];
#pragma unroll
    for (int b = 0; b < kPer; ++b) {
      const int cc = c + b;
      if (cc < nchunk16) {
#pragma unroll
        for (int q = 0; q < NP; ++q) tmem_ld16(lane_base + (uint32_t)((q * G2 + mt * sc) * Nn + cc * 16), r[b][q]);
      }
    }
    tmem_ld_wait();
    if (valid) {
#pragma unroll
      for (int b = 0; b < kPer; ++b) {
        const int cc = c + b;
        if (cc < nchunk16) {
          uint32_t wd[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float s0 = __uint_as_float(r[b][0][2 * i]), s1 = __uint_as_float(r[b][0][2 * i + 1]);
#pragma unroll
            for (int q = 1; q < NP; ++q) {
              s0 += __uint_as_float(r[b][q][2 * i]);
              s1 += __uint_as_float(r[b][q][2 * i + 1]);
            }
            wd[i] = epilogue_pair<T>(s0, s1, bias_s[cc * 16 + 2 * i], bias_s[cc * 16 + 2 * i + 1]);
          }
          // 32 bytes of this pixel: chunks c16, c16 + 1 of its slice row
          const uint32_t byte = (uint32_t)cc * 32u;
          const uint32_t slice = byte / (uint32_t)W, c16 = (byte % (uint32_t)W) >> 4;
          const uint32_t base = row_addr + slice * slice_bytes;
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(base + ((c16 ^ swz) << 4)), "r"(wd[0]),
                       "r"(wd[1]), "r"(wd[2]), "r"(wd[3])
                       : "memory");
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(base + (((c16 + 1u) ^ swz) << 4)),
                       "r"(wd[4]), "r"(wd[5]), "r"(wd[6]), "r"(wd[7])
                       : "memory");
        }
      }
    }
  }
}

// SW = false: A planes hold one 8-channel chunk per pixel (16-byte rows,
// no swizzle), one TMA box per (phase, chunk).  SW = true: A planes hold 64
// channels per pixel (128-byte rows, 128-byte swizzle) covering `sc` group
// chunks, one TMA box per phase; each chunk is a K-offset inside the row.
template <typename T, bool SW, bool STAGED>
__global__ void __launch_bounds__(kThreads, 1) tc_kernel(const __grid_constant__ CUtensorMap xmap,
                                                        const __grid_constant__ CUtensorMap wmap,
                                                        const __grid_constant__ CUtensorMap ymap,
                                                        const __grid_constant__ TcArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* a_full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* a_empty = a_full + kMaxStages;
  uint64_t* acc_full = a_full + 2 * kMaxStages;
  uint64_t* acc_empty = acc_full + kMaxAccBufs;
  uint64_t* mma_done = acc_empty + kMaxAccBufs;
  uint64_t* w_full = mma_done + 1;  // weight copies (TMA staging)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 256);
  float* bias_s = reinterpret_cast<float*>(smem + a.bias_off);
  uint8_t* Bs = smem + a.b_off;
  uint8_t* As = smem + a.a_off;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_sc = a.n_gc / a.sc;
  const int gsc = blockIdx.x % n_sc;  // this CTA's row of sc group chunks
  const int cta_in_gc = blockIdx.x / n_sc;
  const int g0 = gsc * a.sc * a.m;
  const T* __restrict__ wg = static_cast<const T*>(a.w);
  const T* __restrict__ bg = static_cast<const T*>(a.bias);
  T* __restrict__ yg = static_cast<T*>(a.y);

  allow_dependent_launch();
  if (tid == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(&a_full[s], 1);
      mbar_init(&a_empty[s], kIssuers);
    }
    for (int b = 0; b < a.nbuf; ++b) {
      mbar_init(&acc_full[b], kIssuers);
      mbar_init(&acc_empty[b], 4);
    }
    mbar_init(mma_done, kIssuers);
    mbar_init(w_full, 1);
    fence_mbar_init();
    tma_prefetch_desc(&xmap);
    if (a.w_tma) tma_prefetch_desc(&wmap);
    if (STAGED) tma_prefetch_desc(&ymap);
  }
  // Named barrier 2 (all threads): warp 0 arrives once the barriers are
  // initialised and goes straight on to copy input tiles; warps 1.. sync on
  // it after their set-up that needs neither.  Warp 1 allocates tensor
  // memory after the wait on the previous grid in the stream: a CTA that
  // holds tensor memory never waits on another grid, so a later grid's CTA
  // waiting in its own allocation always sees it freed.
  // The producer decodes its first tile (six integer divisions, about half a
  // microsecond) before the wait on the previous grid, so its first copy
  // goes out as soon as that wait ends; the empty asm keeps the decode ahead
  // of the wait.
  SpatialWalk pwalk;
  if (warp == 0) {
    pwalk.init(a, cta_in_gc, a.cpg);
    asm volatile("" ::"r"(pwalk.tw), "r"(pwalk.th), "r"(pwalk.od), "r"(pwalk.n), "r"(pwalk.dtw), "r"(pwalk.dth),
                 "r"(pwalk.dod), "r"(pwalk.dn));
    __syncwarp();
    asm volatile("bar.arrive 2, %0;" ::"r"(kThreads) : "memory");
    grid_dependency_wait();  // x from here on
  }
  uint32_t tmem_base = 0;
  const bool withhold = (a.test_flags & 1) && blockIdx.x == 0;

  if (warp != 0) {
    // Warps 1.. build the MMA lists and stage the weights and bias while the
    // producer (warp 0) already copies the first input tiles: the A stages do
    // not depend on them.  The zero fill and the lists touch only shared
    // memory and kernel parameters, so they run before the wait on the
    // previous kernel in the stream.
    const int btid = tid - 32, bthreads = (int)blockDim.x - 32;
    // Weights of this group chunk as block-diagonal B_t[n][k], K-major core
    // matrices: byte offset (((((j*KS + ks)*2 + kc2)*ntaps + t)*Nn + n)*8 + e)*2
    // holds k = ks*16 + kc2*8 + e of tap t for group chunk j, i.e. slabs
    // [j][ks][kc2][t] of Nn rows x 16 bytes.  The two K halves of one MMA are
    // ntaps slabs apart (the descriptor's leading byte offset), and the taps
    // of one (j, ks, kc2) are consecutive, so one TMA box can fill them all.
    // The thread copy walks chunks in destination order (consecutive threads
    // fill consecutive 16-byte chunks: no bank conflicts); each chunk's
    // nonzero run (the input channels of output n's group) is one cp.async
    // when it is 16, 8 or 4 bytes and aligned, and every thread issues all its
    // copies before waiting once.  Chunks are zero-filled first when some
    // run is shorter than a chunk (merged groups).
    const int nchunk = a.sc * a.ntaps * a.KS * 2 * a.Nn;
    const uintptr_t wa = reinterpret_cast<uintptr_t>(wg);
    const bool full_runs = a.m == 1 && a.Cg % 8 == 0;
    if (!full_runs) {
      uint4* B16 = reinterpret_cast<uint4*>(Bs);
      for (int i = btid; i < nchunk; i += bthreads) B16[i] = make_uint4(0u, 0u, 0u, 0u);
      fence_proxy_async_smem();  // zeros before the copies into the same slabs (barrier 2 below)
    }
    // Per-issuer MMA lists.  The tile's work is split into units u = grp * np
    // + p (accumulator grp = mt * sc + j, partial p summing the taps t with
    // t % np == p); issuer w owns units w, w + kIssuers, ...  Its list holds,
    // in issue order (unit-local step s outer, its units inner, so consecutive
    // MMAs write different accumulators), one 32-byte entry per MMA: A
    // descriptor for stage 0, B descriptor, accumulator column, flags (bit 0:
    // accumulate, bit 1: skip).  The issuing thread then only adds the stage
    // offset, and can fetch entry i + 1 while MMA i issues.
    if (a.ntab > 0) {
      uint4* tab = reinterpret_cast<uint4*>(smem + a.tab_off);
      const uint32_t base = smem_u32(smem);
      const uint32_t lbo_b = (uint32_t)(a.ntaps * a.Nn) * 16u;
      for (int i = btid; i < a.ntab; i += bthreads) {
        const uint2 e = a.tab[i];
        uint4 e0 = make_uint4(0u, 0u, 0u, 0u);
        if (!((e.y >> 16) & 2u)) {
          const uint32_t aaddr = base + ((e.x & 0xffffu) << 4), baddr = base + ((e.x >> 16) << 4);
          uint64_t adesc;
          if constexpr (SW) {
            adesc = smem_desc_sw128(aaddr);
          } else {
            adesc = smem_desc(aaddr, a.plane_stride, 128u);
          }
          const uint64_t bdesc = smem_desc(baddr, lbo_b, 128u);
          e0 = make_uint4((uint32_t)adesc, (uint32_t)(adesc >> 32), (uint32_t)bdesc, (uint32_t)(bdesc >> 32));
        }
        tab[2 * i] = e0;
        tab[2 * i + 1] = make_uint4(e.y & 0xffffu, 0u, 0u, e.y >> 16);
      }
    } else {
      uint4* tab = reinterpret_cast<uint4*>(smem + a.tab_off);
      const int G2 = a.sc * a.nmt, NP = a.np;
      const int units = G2 * NP;
      const int steps = ((a.ntaps + NP - 1) / NP) * a.KS;
      const uint32_t a_base = smem_u32(As), b_base = smem_u32(Bs);
      const uint32_t lbo_b = (uint32_t)(a.ntaps * a.Nn) * 16u;
      int base = 0;
      for (int w = 0; w < kIssuers; ++w) {
        const int nu = units > w ? (units - w + kIssuers - 1) / kIssuers : 0;
        const int len = steps * nu;
        for (int i = btid; i < len; i += bthreads) {
          const int st = i / nu, ui = i - st * nu;
          const int u = w + kIssuers * ui;
          const int grp = u / NP, p = u - grp * NP;
          const int t = p + NP * (st / a.KS), ks = st % a.KS;
          const int mt = grp / a.sc, j = grp - mt * a.sc;
          uint4 e0 = make_uint4(0u, 0u, 0u, 0u), e1 = make_uint4(0u, 0u, 0u, 2u);  // default: skip
          if (t < a.ntaps) {
            uint64_t adesc;
            if constexpr (SW) {
              const uint32_t row = a_base + (uint32_t)a.tap_phase[t] * a.plane_stride +
                                   (uint32_t)(mt * 128 + a.shift + a.tap_off[t]) * 128u;
              adesc = smem_desc_sw128(row + (uint32_t)(j * a.Kt * 2 + ks * 32));
            } else {
              const uint32_t plane0 = a_base + (uint32_t)(a.tap_phase[t] * a.nchunks) * a.plane_stride;
              const uint32_t row0 = (uint32_t)(mt * 128 + a.shift + a.tap_off[t]) * 16u;
              adesc = smem_desc(plane0 + (uint32_t)(2 * ks) * a.plane_stride + row0, a.plane_stride, 128u);
            }
            const uint64_t bdesc =
                smem_desc(b_base + (uint32_t)(((j * a.KS + ks) * 2 * a.ntaps + t) * a.Nn) * 16u, lbo_b, 128u);
            e0 = make_uint4((uint32_t)adesc, (uint32_t)(adesc >> 32), (uint32_t)bdesc, (uint32_t)(bdesc >> 32));
            e1 = make_uint4((uint32_t)((p * G2 + grp) * a.Nn), 0u, 0u, st == 0 ? 0u : 1u);
          }
          tab[2 * (base + i)] = e0;
          tab[2 * (base + i) + 1] = e1;
        }
        base += len;
      }
    }
    grid_dependency_wait();  // w, bias (and, for the epilogue warps, y) from here on
    asm volatile("bar.sync 2, %0;" ::"r"(kThreads) : "memory");  // barriers initialised
    T* B = reinterpret_cast<T*>(Bs);
    // Bias: the first value of each thread is loaded now and stored once the
    // weight copies are issued, so its latency overlaps them.
    const int nbias = a.sc * a.Nn;
    T b_first = Elem<T>::from_f32(0.f);
    if (btid < nbias && bg != nullptr) b_first = bg[(int64_t)g0 * a.Kg + btid];
    if (a.w_tma) {
      // Cg and Kg multiples of 8: the 8 input channels of a (ks, kc2) slab lie
      // in one group gi, and for that group the slab's Kg rows n = gi*Kg + kk
      // are one TMA box {8 channels, Kg output channels, taps} of the weight
      // tensor viewed as (Cg, G*Kg, taps).  With one group per chunk (m = 1)
      // a box covers every tap (its [tap][row][8] landing order is the slabs'
      // order); otherwise one tap, at row offset gi*Kg of the slab.
      // Copies are spread over the builder threads (a single thread issuing
      // them all would serialise about 0.1 us per copy); thread 0 arms the
      // barrier with the total bytes (copies may complete before that: the
      // transaction count may go negative until then).
      const int per = a.w_box_taps, nt = a.ntaps / per;
      const int ncopy = a.sc * a.KS * 2 * nt;
      if (btid == 0) mbar_arrive_expect_tx(w_full, (uint32_t)ncopy * (uint32_t)(a.Kg * per) * 16u);
      for (int i = btid; i < ncopy; i += bthreads) {
        const int tq = i % nt, r = i / nt;  // r = (j*KS + ks)*2 + kc2
        const int kc2 = r & 1, ks = (r >> 1) % a.KS, j = (r >> 1) / a.KS;
        const int k0 = ks * 16 + kc2 * 8;
        const int gi = k0 / a.Cg, c0 = k0 - gi * a.Cg;
        const int t = tq * per;
        tma_load_3d(B + ((size_t)(r * a.ntaps + t) * a.Nn + (size_t)gi * a.Kg) * 8, &wmap, w_full, c0,
                    (g0 + j * a.m + gi) * a.Kg, t);
      }
    } else {
    // chunk index ci = ((((j*KS + ks)*2 + kc2)*ntaps + t)*Nn + n, n = gi*Kg +
    // kk, as mixed-radix digits advanced by bthreads with carries (no
    // division per chunk)
    const int rad[6] = {a.Kg, a.m, a.ntaps, 2, a.KS, a.sc};
    int dig[6], inc[6];
    {
      int v = btid, w = bthreads;
#pragma unroll
      for (int i = 0; i < 6; ++i) {
        dig[i] = v % rad[i], v /= rad[i];
        inc[i] = w % rad[i], w /= rad[i];
      }
    }
    for (int ci = btid; ci < nchunk; ci += bthreads) {
      const int kk = dig[0], gi = dig[1], t = dig[2], kc2 = dig[3], ks = dig[4], j = dig[5];
      {
        int carry = 0;
#pragma unroll
        for (int i = 0; i < 6; ++i) {
          dig[i] += inc[i] + carry;
          carry = dig[i] >= rad[i];
          if (carry) dig[i] -= rad[i];
        }
      }
      const int k0 = ks * 16 + kc2 * 8;
      const int ka = max(k0, gi * a.Cg), kb = min(k0 + 8, (gi + 1) * a.Cg);
      if (ka >= kb) continue;  // off the diagonal: zero
      const T* src = wg + ((int64_t)(g0 + j * a.m + gi) * a.Kg + kk) * a.taps_total * a.Cg + (int64_t)t * a.Cg +
                     (ka - gi * a.Cg);
      T* dst = B + (size_t)ci * 8 + (ka - k0);
      const int bytes = (kb - ka) * (int)sizeof(T);
      const uintptr_t sa = reinterpret_cast<uintptr_t>(src);
      const uint32_t da = smem_u32(dst);
      if (bytes == 16 && ((sa | da) & 15) == 0) {
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(da), "l"(src) : "memory");
      } else if (bytes == 8 && ((sa | da) & 7) == 0) {
        asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(da), "l"(src) : "memory");
      } else if (bytes == 4 && ((sa | da) & 3) == 0) {
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(da), "l"(src) : "memory");
      } else {
        for (int e = 0; e < kb - ka; ++e) dst[e] = src[e];
      }
    }
    }
    (void)wa;
    if (btid < nbias) bias_s[btid] = Elem<T>::to_f32(b_first);
    for (int i = btid + bthreads; i < nbias; i += bthreads)
      bias_s[i] = bg != nullptr ? Elem<T>::to_f32(bg[(int64_t)g0 * a.Kg + i]) : 0.f;
    if (warp == 1) {  // while the weight copies are in flight
      __syncwarp();     // the allocation is a whole-warp instruction
      tmem_alloc(tmem_slot, a.tmem_cols);
      tmem_relinquish();
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    if (a.w_tma && !mbar_wait(w_full, 0u, a.wait_limit_ns)) report(a.status, kDevTimeout, 6);
    fence_proxy_async_smem();  // generic-proxy writes of B -> visible to the tensor core
    fence_before_sync();
    asm volatile("bar.sync 1, %0;" ::"r"(bthreads) : "memory");
    fence_after_sync();
    tmem_base = *tmem_slot;
  }

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      int k = 0;
      bool failed = false;
      SpatialWalk& walk = pwalk;
      Ring sr;
      for (int sp = cta_in_gc; sp < a.spatial_tiles; sp += a.cpg, ++k, walk.advance(a), sr.next(a.stages)) {
        const int s = sr.pos;
        if (k >= a.stages && !mbar_wait(&a_empty[s], (uint32_t)(sr.ph ^ 1), a.wait_limit_ns)) {
          failed = true;
          break;
        }
        if (withhold && k == 0) continue;
        // At launch every CTA requests its stages at once.  Holding the second
        // tile's copy until the first tile and the weights have landed lets
        // the first MMAs start sooner; later copies overlap the MMAs.
        if (k == 1 && !withhold &&
            (!mbar_wait(&a_full[0], 0u, a.wait_limit_ns) || (a.w_tma && !mbar_wait(w_full, 0u, a.wait_limit_ns)))) {
          failed = true;
          break;
        }
        const SpatialTile st = walk.tile(a);
        const int id0 = st.od * a.sD - a.pD;
        mbar_arrive_expect_tx(&a_full[s], a.tx_bytes);
        uint8_t* stage = As + (size_t)s * a.a_stage_bytes;
        for (int ph = 0; ph < a.nphase; ++ph) {
          const int ih0 = a.s * (st.oh0 + a.qy_min) + a.phase_py[ph];
          const int iw0 = a.s * (st.ow0 + a.qx_min + a.plane_cx[ph]) + a.phase_px[ph];
          if constexpr (SW) {
            tma_load_5d(stage + (size_t)ph * a.plane_stride, &xmap, &a_full[s], g0 * a.Cg, iw0, ih0, id0, st.n);
          } else {
            for (int c = 0; c < a.nchunks; ++c)
              tma_load_5d(stage + (size_t)(ph * a.nchunks + c) * a.plane_stride, &xmap, &a_full[s],
                          g0 * a.Cg + c * 8, iw0, ih0, id0, st.n);
          }
        }
      }
      if (failed) report(a.status, kDevTimeout, 3);
      for (int j = k > a.stages ? k - a.stages : 0; j < k; ++j) {  // bounded drain
        if (withhold && j == 0) continue;
        mbar_wait(&a_full[j % a.stages], (uint32_t)((j / a.stages) & 1), a.wait_limit_ns);
      }
    }
  } else if (warp <= kIssuers) {
    // ---------------- MMA issuers (warps 1..kIssuers) ----------------
    // A single thread can only have one tcgen05.mma in its issue pipeline
    // at a time (about 160 cycles per instruction, whatever M and N), so
    // several warps issue in parallel.  The tile's work is split into units
    // (accumulator grp, partial p): partial p of an accumulator sums the taps
    // t with t % np == p, and the epilogue adds the np partials.  Issuer w
    // takes the units u = grp * np + p with u % kIssuers == w; within an
    // issuer, consecutive MMAs cycle over its units (no back-to-back
    // accumulation into one accumulator).  Whole warps issuing through
    // elect.sync (faster alone in a probe) measured 1.2-1.9x slower here, and
    // three issuers (eight warps, no register cap) lost on tiles of four
    // units, so four lone lanes issue.
    if (lane == 0) {
      const int w = warp - 1;
      int k = 0;
      bool failed = false;
      const int G2 = a.sc * a.nmt;
      const int NP = a.np;
      const int units = G2 * NP;
      const int steps = ((a.ntaps + NP - 1) / NP) * a.KS;
      int my_base = 0, my_len = 0;
      for (int v = 0; v <= w; ++v) {
        const int nu = units > v ? (units - v + kIssuers - 1) / kIssuers : 0;
        if (v < w) my_base += steps * nu; else my_len = steps * nu;
      }
      const uint4* my_list = reinterpret_cast<const uint4*>(smem + a.tab_off) + 2 * my_base;
      Ring sr, ar;
      for (int sp = cta_in_gc; sp < a.spatial_tiles; sp += a.cpg, ++k, sr.next(a.stages), ar.next(a.nbuf)) {
        const int s = sr.pos;
        const int ab = ar.pos;
        if (!mbar_wait(&a_full[s], (uint32_t)sr.ph, a.wait_limit_ns)) {
          failed = true;
          break;
        }
        if (k >= a.nbuf && !mbar_wait(&acc_empty[ab], (uint32_t)(ar.ph ^ 1), a.wait_limit_ns)) {
          failed = true;
          break;
        }
        fence_after_sync();
        // descriptor start addresses are in 16-byte units in the low bits
        const uint64_t stage_delta = (uint64_t)(((uint32_t)s * a.a_stage_bytes) >> 4);
        // unit (grp, p) of buffer ab sits at columns ((ab * np + p) * G2 + grp) * Nn
        const uint32_t dbuf = tmem_base + (uint32_t)(ab * NP * G2 * a.Nn);
        if (my_len > 0) {
          uint4 c0 = my_list[0], c1 = my_list[1];
          for (int i = 0; i < my_len; ++i) {
            const int nx = i + 1 < my_len ? i + 1 : i;
            const uint4 n0 = my_list[2 * nx], n1 = my_list[2 * nx + 1];
            if (!(c1.w & 2u)) {
              const uint64_t adesc = (((uint64_t)c0.y << 32) | c0.x) + stage_delta;
              const uint64_t bdesc = ((uint64_t)c0.w << 32) | c0.z;
              mma_f16(dbuf + c1.x, adesc, bdesc, a.idesc, c1.w & 1u);
            }
            c0 = n0;
            c1 = n1;
          }
        }
        commit(&a_empty[s]);    // this issuer's reads of the stage are done
        commit(&acc_full[ab]);  // this issuer's accumulations are done
      }
      if (failed) report(a.status, kDevTimeout, 4);
      commit(mma_done);  // every MMA this issuer issued has completed
      mbar_wait(mma_done, 0, a.wait_limit_ns);
    }
  } else {
    // ---------------- epilogue (warps kIssuers+1 .. kIssuers+4) ----------------
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;
    const int G2 = a.sc * a.nmt;
    const int NP = a.np;
    // 32-byte stores when every 16-channel piece starts on a 32-byte boundary
    // (each chunk row's channel offset is a multiple of 16)
    const bool v8 = (reinterpret_cast<uintptr_t>(yg) & 31) == 0 && (a.Ktot & 15) == 0;
    // whole 128-byte pixel runs per store (epilogue_row_x4): groups of four
    // 16-channel chunks, 32-byte stores, one partial accumulator
    const bool x4 = v8 && ((a.sc * a.Nn / 16) & 3) == 0;
    // STAGED (on request): the four epilogue warps write the tile's output
    // box into shared memory and one thread stores it with TMA tensor stores
    // (one per channel slice); the next tile waits until those stores have
    // read the staging buffer.
    const bool store_thread = warp == kIssuers + 1 && lane == 0;
    const uint32_t stage_base = smem_u32(smem + a.epi_off);
    // This lane's accumulator row f = mt * 128 + row is flattened output
    // f + shift, i.e. (i, jj) of the tile's rows of pitch P; the same for
    // every tile, so it is decoded once and advanced by 128 rows per M tile.
    // Rows before the first output (i < 0) are never stored.
    int i_row0 = 0, jj_row0 = row + a.shift;
    while (jj_row0 < 0) jj_row0 += a.P, --i_row0;
    i_row0 += jj_row0 / a.P;
    jj_row0 -= (jj_row0 / a.P) * a.P;
    const int di = 128 / a.P, dj = 128 - di * a.P;
    SpatialWalk walk;
    walk.init(a, cta_in_gc, a.cpg);
    Ring ar;
    for (int sp = cta_in_gc; sp < a.spatial_tiles; sp += a.cpg, walk.advance(a), ar.next(a.nbuf)) {
      const int ab = ar.pos;
      if (!warp_wait(&acc_full[ab], (uint32_t)ar.ph, a.wait_limit_ns)) {
        if (lane == 0) report(a.status, kDevTimeout, 5);
        break;
      }
      fence_after_sync();
      const SpatialTile st = walk.tile(a);
      const uint32_t lane_base = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(ab * NP * G2 * a.Nn);
      if constexpr (STAGED) {
        if (store_thread) tma_store_wait_read();  // the previous tile's stores have read the buffer
        asm volatile("bar.sync 3, 128;" ::: "memory");
      }
      int i = i_row0, jj = jj_row0;
      for (int mt = 0; mt < a.nmt; ++mt, i += di, jj += dj) {
        if (jj >= a.P) jj -= a.P, ++i;  // (i, jj) of row mt * 128 + row
        const int oh = st.oh0 + i, ow = st.ow0 + jj;
        if constexpr (STAGED) {
          // pixels past the image edge are written too; the TMA store clips them
          const bool valid = i >= 0 && i < a.TH && jj < a.TWo;
          const int p = i * a.TWo + jj;
          if (NP == 1)
            epilogue_row_tma<T, 1>(lane_base, mt, G2, a.sc, a.Nn, valid, p, bias_s, stage_base, a.epi_slice_bytes,
                                   a.epi_w);
          else if (NP == 2)
            epilogue_row_tma<T, 2>(lane_base, mt, G2, a.sc, a.Nn, valid, p, bias_s, stage_base, a.epi_slice_bytes,
                                   a.epi_w);
          else
            epilogue_row_tma<T, 4>(lane_base, mt, G2, a.sc, a.Nn, valid, p, bias_s, stage_base, a.epi_slice_bytes,
                                   a.epi_w);
        } else {
          bool valid = i >= 0 && i < a.TH && jj < a.TWo && oh < a.Ho && ow < a.Wo;
          if (a.om.on == 2) {  // stacked phases (planned with one partial accumulator)
            epilogue_row_stacked<T>(lane_base, mt, a.sc, a.Nn, valid, st.n, st.od, oh, ow, a.om, g0 * a.Kg, a.Kg,
                                    yg);
            continue;
          }
          int64_t pix;
          if (a.om.on) {  // kept outputs land at scale * v + add of the mapped tensor
            valid = valid && st.od >= a.om.lo[0] && st.od < a.om.hi[0] && oh >= a.om.lo[1] && oh < a.om.hi[1] &&
                    ow >= a.om.lo[2] && ow < a.om.hi[2];
            pix = (((int64_t)st.n * a.om.ext[0] + (st.od * a.om.scale[0] + a.om.add[0])) * a.om.ext[1] +
                   (oh * a.om.scale[1] + a.om.add[1])) * (int64_t)a.om.ext[2] + (ow * a.om.scale[2] + a.om.add[2]);
          } else {
            pix = (((int64_t)st.n * a.Do + st.od) * a.Ho + oh) * (int64_t)a.Wo + ow;
          }
          T* dst = yg + pix * a.Ktot + (int64_t)g0 * a.Kg;
          if (x4 && NP == 1) epilogue_row_x4<T>(lane_base, mt, a.sc, a.Nn, valid, dst, bias_s);
          else if (NP == 1) epilogue_row<T, 1>(lane_base, mt, G2, a.sc, a.Nn, valid, dst, bias_s, v8);
          else if (NP == 2) epilogue_row<T, 2>(lane_base, mt, G2, a.sc, a.Nn, valid, dst, bias_s, v8);
          else epilogue_row<T, 4>(lane_base, mt, G2, a.sc, a.Nn, valid, dst, bias_s, v8);
        }
      }
      // every tcgen05.ld of this tile has completed: the accumulators are free
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[ab]);
      if constexpr (STAGED) {
        fence_proxy_async_smem();  // the staging writes -> visible to the TMA engine
        asm volatile("bar.sync 3, 128;" ::: "memory");
        if (store_thread) {
          const int c0 = g0 * a.Kg;
          for (int sl = 0; sl < a.epi_slices; ++sl)
            tma_store_5d(&ymap, smem + a.epi_off + (size_t)sl * a.epi_slice_bytes, c0 + sl * (a.epi_w / 2), st.ow0,
                         st.oh0, st.od, st.n);
          tma_store_commit();
        }
      }
    }
    if constexpr (STAGED) {
      if (store_thread) tma_store_wait_all();  // the stores are complete before the CTA exits
    }
  }
  __syncwarp();
  fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    fence_after_sync();
    tmem_dealloc(tmem_base, a.tmem_cols);
  }
}

}  // namespace tc
}  // namespace gconv
