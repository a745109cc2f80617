// Backward data for callers that cannot allocate device memory.
//
// Some callers may not call cudaMalloc (nor have anyone call it for them)
// while they run: an inference engine's plugin that is enqueued on a stream
// the engine owns and must not allocate, a runtime that reserves all device
// memory at start-up and forbids allocation on its hot path, or code that
// must not trigger the device-wide synchronisation an allocation can cause.
// grouped_conv_bwd_data asks them for a scratch workspace (the transposed,
// flipped weights of its stride-1 route); grouped_conv_bwd_data_noalloc
// takes that scratch from a fixed array in this library's device memory
// instead.  The array is a file-scope __device__ variable of
// GCONV_NOALLOC_SCRATCH_BYTES bytes: it is part of the module's static
// device memory, so every GPU that loads the library holds it until the
// process exits, and no call allocates anything.
//
// Every call shares the one array.  Its contents are whatever the last call
// left there; the weight-flip kernel rewrites every byte a call reads, so
// nothing needs clearing.  Calls whose work overlaps on the GPU (two streams,
// or two host threads without ordering) race on the array.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "../../include/gconv.h"
#include "kernels.h"

namespace gconv {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[GCONV_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch array, looked up once per device with that
// device current.  A failed look-up is not kept; the next call retries.
struct ScratchSlot {
  std::mutex mu;
  std::atomic<bool> ready{false};
  void* ptr = nullptr;
};
constexpr int kMaxScratchDevices = 64;
ScratchSlot g_scratch[kMaxScratchDevices];

cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxScratchDevices) return cudaErrorInvalidDevice;
  ScratchSlot& s = g_scratch[dev];
  if (!s.ready.load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(s.mu);
    if (!s.ready.load(std::memory_order_relaxed)) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess) return e;
      s.ptr = p;
      s.ready.store(true, std::memory_order_release);
    }
  }
  *out = s.ptr;
  return cudaSuccess;
}

}  // namespace
}  // namespace gconv

using namespace gconv;

extern "C" gconv_status grouped_conv_bwd_data_noalloc(const void* dy, const void* w, void* dx,
                                                      const gconv_problem* p, gconv_dtype dt,
                                                      struct CUstream_st* stream) {
  int64_t need = 0;
  gconv_status s = grouped_conv_bwd_data_workspace_size(p, dt, &need);
  if (s != GCONV_OK) return s;
  if (need > (int64_t)GCONV_NOALLOC_SCRATCH_BYTES && p != nullptr &&
      (p->stride[0] > 1 || p->stride[1] > 1 || p->stride[2] > 1)) {
    // the stride-phase route would need more scratch than the array holds;
    // the direct gather kernel computes the same result with none
    gconv_options o{};
    o.force_kernel = GCONV_KERNEL_BWD_DATA_DIRECT;
    return grouped_conv_bwd_data_ex(dy, w, dx, p, dt, nullptr, 0, stream, &o);
  }
  if (need > (int64_t)GCONV_NOALLOC_SCRATCH_BYTES)
    return set_last_error(GCONV_ERR_UNSUPPORTED,
                          "grouped_conv_bwd_data_noalloc: this problem needs %lld bytes of scratch, more than the "
                          "library's fixed %d bytes; call grouped_conv_bwd_data with a workspace instead",
                          (long long)need, (int)GCONV_NOALLOC_SCRATCH_BYTES);
  void* scratch = nullptr;
  if (need > 0) {
    cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess)
      return set_last_error(GCONV_ERR_CUDA, "grouped_conv_bwd_data_noalloc: scratch address: %s",
                            cudaGetErrorString(e));
  }
  return grouped_conv_bwd_data(dy, w, dx, p, dt, scratch, need, stream);
}
