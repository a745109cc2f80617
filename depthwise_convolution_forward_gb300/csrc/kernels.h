// Internal interface between the C-ABI layer (api.cu) and the kernel
// translation units.  Not installed, not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/gconv.h"

namespace gconv {

enum DType : int { kF32 = 0, kF16 = 1, kBF16 = 2 };

inline int dtype_bytes(DType t) { return t == kF32 ? 4 : 2; }

// Validated, normalised problem.  2D problems have D = Do = Z = 1.
struct Geometry {
  int64_t N;
  int G, Cg, Kg;
  int D, H, W;
  int Do, Ho, Wo;
  int Z, Y, X;
  int sD, sH, sW;
  int pD, pH, pW;
  int dD, dH, dW;
  int ndim;
  int C() const { return G * Cg; }
  int K() const { return G * Kg; }
  int taps() const { return Z * Y * X; }
  int64_t x_elems() const { return N * D * H * W * (int64_t)C(); }
  int64_t y_elems() const { return N * Do * Ho * Wo * (int64_t)K(); }
  int64_t w_elems() const { return (int64_t)K() * taps() * Cg; }
};

// Output placement for the tensor-core kernel (backward data by stride
// phases); on = 0 keeps the plain layout.
//  on = 1: output coordinate v of dimension i (D, H, W) is kept when
//          lo[i] <= v < hi[i] and written at scale[i] * v + add[i] of a
//          tensor with extents ext[i] (same N and channel count).
//  on = 2: phases stacked as output channels: output channel
//          g * nph * cpp + ph * cpp + c goes to channel g * cpp + c (of ctot)
//          at coordinate scale[i] * v + add[i] + res[ph][i], kept when
//          v >= lo[i] and that coordinate is below ext[i].
constexpr int kMaxStackPhases = 8;
struct OutMap {
  int on;
  int scale[3], add[3], lo[3], hi[3], ext[3];
  int cpp, nph, ctot;
  int res[kMaxStackPhases][3];
};

struct LaunchArgs {
  const void* x;
  const void* w;
  const void* bias;  // may be null
  void* y;
  DType dt;
  cudaStream_t stream;
  int* status;  // device status word [code, where]
  uint64_t wait_limit_ns;
  int test_flags;
  int tile[8];  // tuning overrides, 0 = automatic
  bool pdl;     // programmatic dependent launch (the kernels wait on the grid dependency)
  OutMap omap;  // tensor-core kernel only (others refuse a map that is on)
};

// Launches kernel k on a.stream.  With a.pdl the launch carries the
// programmatic-stream-serialisation attribute: the kernel's CTAs may start
// while the previous kernel in the stream is still running, so every kernel
// launched this way calls grid_dependency_wait() before its first access to
// global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, const LaunchArgs& a,
                          Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k, std::forward<Args>(args)...);
}

// Device properties needed by the launchers (cached per device by api.cu).
struct DeviceInfo {
  int device;
  int num_sms;
  int max_smem_optin;  // bytes per block
};

// Tensor-map encoder (driver entry point resolved once by api.cu).
CUresult encode_tiled(CUtensorMap* map, CUtensorMapDataType type, uint32_t rank, const void* base,
                      const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                      const uint32_t* elem_strides, CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_NONE);

// SM count and opt-in shared memory per block assumed by the host-only
// selector (grouped_conv_select, no device at hand): those of a GB300.
constexpr int kDefaultSms = 152;
constexpr int kDefaultSmemOptin = 232448;

// ---- Ka: TMA-staged depthwise direct kernel (Cg == Kg == 1) -------------
// Returns true when the kernel supports this problem (shape, dtype, alignment)
// and its planner finds a launch plan for a device with num_sms SMs.
bool dw_supported(const Geometry& g, DType dt, const LaunchArgs* a, int num_sms);
cudaError_t dw_launch(const Geometry& g, const LaunchArgs& a, const DeviceInfo& dev);

// ---- generic direct kernel (any shape, dtype, alignment) ----------------
cudaError_t generic_launch(const Geometry& g, const LaunchArgs& a, const DeviceInfo& dev);

// ---- Kb: tcgen05 / TMEM grouped implicit GEMM ----------------------------
// Returns true when the kernel supports this problem and its planner finds a
// launch plan for a device with num_sms SMs and max_smem bytes of opt-in
// shared memory per block.
bool tc_supported(const Geometry& g, DType dt, const LaunchArgs* a, int num_sms, int max_smem);
cudaError_t tc_launch(const Geometry& g, const LaunchArgs& a, const DeviceInfo& dev);

// ---- backward data ---------------------------------------------------------
// wt[g][c][t'][k] = w[g][k][flip(t')][c] into wt (w_elems elements); a.w is w.
cudaError_t bwd_weight_flip_launch(const Geometry& g, const LaunchArgs& a, void* wt, const DeviceInfo& dev);
// Direct gather: a.x carries dy, a.w the forward weights, a.y receives dx.
cudaError_t bwd_data_direct_launch(const Geometry& g, const LaunchArgs& a, const DeviceInfo& dev);

// Stride-phase route of backward data.  One phase per (rD, rH, rW): its
// sub-filter taps per dimension (original tap indices in the order the
// phase's correlation reads them), and where its rows land in dx.
constexpr int kMaxPhaseTaps = 16;
struct PhaseTaps {
  int L[3];                    // sub-filter extent per dimension
  int t[3][kMaxPhaseTaps];     // original tap index of sub-filter position j
};
struct PhaseScatter {
  int64_t N;
  int64_t C;                   // channels per pixel of dx (and of the phase buffer)
  int in[3];                   // dx extents D, H, W
  int s[3], r[3];              // stride and phase per dimension
  int n[3];                    // phase extents: dx positions with index % s == r
  int o[3], off[3];            // phase buffer extents and the offset of the phase's first position
  int empty;                   // 1: no tap reaches this phase (write zeros)
};
// wt = the phase's sub-filter of w with channels transposed, [G][Cg][L..][Kg];
// a.w is w.
cudaError_t phase_weight_launch(const Geometry& g, const LaunchArgs& a, const PhaseTaps& pt, void* wt,
                                const DeviceInfo& dev);
// Stacked phase weights: ws[g][ph * Cg + c][qz][qy][qx][k] = w[g][k][t][c]
// for the tap t that reaches phase ph at sub-filter offset q (per dimension
// t = (r + p - s * (qmin + q)) / d when that is a whole tap index), else 0.
struct StackTaps {
  int nph;
  int s[3], p[3], d[3], k[3], Q[3], qmin[3];
};
cudaError_t phase_stack_launch(const Geometry& g, const LaunchArgs& a, const StackTaps& st, void* ws,
                               const DeviceInfo& dev);
// dx positions of one phase from the phase buffer pb (or zeros).
cudaError_t phase_scatter_launch(const PhaseScatter& ps, const void* pb, void* dx, const LaunchArgs& a,
                                 const DeviceInfo& dev);

// ---- backward weight -------------------------------------------------------
// fp32 partials of dw for a fixed number of pixel splits, then one reduction
// and rounding.  a.x carries x, a.w carries dy, a.y receives dw; the
// workspace holds bwd_weight_workspace_bytes (independent of the device).
int64_t bwd_weight_workspace_bytes(const Geometry& g, DType dt);
cudaError_t bwd_weight_launch(const Geometry& g, const LaunchArgs& a, void* workspace, const DeviceInfo& dev);
// dw = round(sum over the S splits of ws[s][e]) (stage 2 of either route).
cudaError_t bwd_weight_reduce_launch(const Geometry& g, const LaunchArgs& a, float* ws, int S,
                                     const DeviceInfo& dev);
// Tensor-core route (16-bit, Cg == Kg dividing 64, C % 64 == 0, H / W
// stride 1 or 2, at most 4 taps per filter row): shape check, workspace
// bytes (0 when unsupported), and launch (cudaErrorNotSupported when x or
// dy is not 16-byte aligned, or the plan does not fit the device).
bool bwd_weight_tc_supported(const Geometry& g, DType dt);
int64_t bwd_weight_tc_workspace_bytes(const Geometry& g, DType dt);
cudaError_t bwd_weight_tc_launch(const Geometry& g, const LaunchArgs& a, void* workspace, const DeviceInfo& dev);

// ---- Kc alone (epilogue test entry) --------------------------------------
cudaError_t epilogue_launch(const float* acc, const void* bias, void* y, int64_t rows, int cols,
                            DType dt, cudaStream_t stream);

// Records a formatted reason as the calling thread's gconv_last_error() and
// returns s (for entry points outside api.cu).
gconv_status set_last_error(gconv_status s, const char* fmt, ...);

// Status codes written into the device status word.
enum DevStatus : int { kDevOk = 0, kDevTimeout = 1 };

}  // namespace gconv
