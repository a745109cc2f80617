// Generic direct grouped convolution, any shape, dtype or alignment: one
// thread per output element, or one warp per output (lanes split the
// reduction) for small problems with long reductions.  It is the path for
// fp32 grouped problems (which must not use TF32 tensor cores) and for shapes
// the specialised kernels do not cover.  Also hosts the stand-alone epilogue
// (Kc) kernel.
#include <algorithm>

#include "common.cuh"

namespace gconv {
namespace {

struct GenericArgs {
  const void* x;
  const void* w;
  const void* bias;
  void* y;
  int64_t total;  // number of outputs
  int G, Cg, Kg;
  int D, H, W, Do, Ho, Wo, Z, Y, X;
  int sD, sH, sW, pD, pH, pW, dD, dH, dW;
};

template <typename T>
__global__ void __launch_bounds__(256) generic_direct_kernel(const GenericArgs a) {
  const T* __restrict__ x = static_cast<const T*>(a.x);
  const T* __restrict__ w = static_cast<const T*>(a.w);
  const T* __restrict__ bias = static_cast<const T*>(a.bias);
  T* __restrict__ y = static_cast<T*>(a.y);
  const int64_t C = (int64_t)a.G * a.Cg;
  const int taps = a.Z * a.Y * a.X;
  grid_dependency_wait();  // x, w, bias and y are touched only from here on
  for (int64_t o = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; o < a.total;
       o += (int64_t)gridDim.x * blockDim.x) {
    int64_t f = o;
    const int k = (int)(f % a.Kg);
    f /= a.Kg;
    const int g = (int)(f % a.G);
    f /= a.G;
    const int ow = (int)(f % a.Wo);
    f /= a.Wo;
    const int oh = (int)(f % a.Ho);
    f /= a.Ho;
    const int od = (int)(f % a.Do);
    const int64_t n = f / a.Do;
    float acc = 0.f;
    const T* wk = w + ((int64_t)g * a.Kg + k) * taps * a.Cg;
    for (int z = 0; z < a.Z; ++z) {
      const int id = od * a.sD - a.pD + z * a.dD;
      if (id < 0 || id >= a.D) continue;
      for (int yy = 0; yy < a.Y; ++yy) {
        const int ih = oh * a.sH - a.pH + yy * a.dH;
        if (ih < 0 || ih >= a.H) continue;
        for (int xx = 0; xx < a.X; ++xx) {
          const int iw = ow * a.sW - a.pW + xx * a.dW;
          if (iw < 0 || iw >= a.W) continue;
          const T* xp = x + (((n * a.D + id) * a.H + ih) * (int64_t)a.W + iw) * C + (int64_t)g * a.Cg;
          const T* wp = wk + ((z * a.Y + yy) * a.X + xx) * a.Cg;
          // unrolled so that several loads are in flight (same summation order)
#pragma unroll 8
          for (int cg = 0; cg < a.Cg; ++cg)
            acc = fmaf(Elem<T>::to_f32(xp[cg]), Elem<T>::to_f32(wp[cg]), acc);
        }
      }
    }
    const float b = bias ? Elem<T>::to_f32(bias[(int64_t)g * a.Kg + k]) : 0.f;
    y[o] = epilogue_one<T>(acc, b);
  }
}

// Warp per output: the warp's lanes split the (tap, input channel) reduction
// of one output and combine it with a butterfly sum.  For problems with few
// outputs and long reductions (one thread per output would leave most SMs
// idle and walk a long chain of dependent loads).
template <typename T>
__global__ void __launch_bounds__(256) generic_warp_kernel(const GenericArgs a) {
  const T* __restrict__ x = static_cast<const T*>(a.x);
  const T* __restrict__ w = static_cast<const T*>(a.w);
  const T* __restrict__ bias = static_cast<const T*>(a.bias);
  T* __restrict__ y = static_cast<T*>(a.y);
  const int lane = threadIdx.x & 31;
  const int64_t C = (int64_t)a.G * a.Cg;
  const int taps = a.Z * a.Y * a.X;
  const int red = taps * a.Cg;  // reduction length
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  grid_dependency_wait();  // x, w, bias and y are touched only from here on
  for (int64_t o = blockIdx.x * (int64_t)(blockDim.x >> 5) + (threadIdx.x >> 5); o < a.total; o += warps) {
    int64_t f = o;
    const int k = (int)(f % a.Kg);
    f /= a.Kg;
    const int g = (int)(f % a.G);
    f /= a.G;
    const int ow = (int)(f % a.Wo);
    f /= a.Wo;
    const int oh = (int)(f % a.Ho);
    f /= a.Ho;
    const int od = (int)(f % a.Do);
    const int64_t n = f / a.Do;
    const T* wk = w + ((int64_t)g * a.Kg + k) * red;
    float acc = 0.f;
    for (int i = lane; i < red; i += 32) {
      const int t = i / a.Cg, cg = i - t * a.Cg;
      const int xx = t % a.X, yy = (t / a.X) % a.Y, z = t / (a.X * a.Y);
      const int id = od * a.sD - a.pD + z * a.dD;
      const int ih = oh * a.sH - a.pH + yy * a.dH;
      const int iw = ow * a.sW - a.pW + xx * a.dW;
      if (id < 0 || id >= a.D || ih < 0 || ih >= a.H || iw < 0 || iw >= a.W) continue;
      const T* xp = x + (((n * a.D + id) * a.H + ih) * (int64_t)a.W + iw) * C + (int64_t)g * a.Cg;
      acc = fmaf(Elem<T>::to_f32(xp[cg]), Elem<T>::to_f32(wk[i]), acc);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) {
      const float b = bias ? Elem<T>::to_f32(bias[(int64_t)g * a.Kg + k]) : 0.f;
      y[o] = epilogue_one<T>(acc, b);
    }
  }
}

template <typename T>
__global__ void epilogue_kernel(const float* __restrict__ acc, const T* __restrict__ bias,
                                T* __restrict__ y, int64_t total, int cols) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int c = (int)(i % cols);
    const float b = bias ? Elem<T>::to_f32(bias[c]) : 0.f;
    y[i] = epilogue_one<T>(acc[i], b);
  }
}

int grid_for(int64_t total, int block, const DeviceInfo* dev) {
  int64_t blocks = (total + block - 1) / block;
  const int64_t cap = dev ? (int64_t)dev->num_sms * 16 : 4096;
  if (blocks > cap) blocks = cap;
  return (int)(blocks < 1 ? 1 : blocks);
}

}  // namespace

cudaError_t generic_launch(const Geometry& g, const LaunchArgs& a, const DeviceInfo& dev) {
  GenericArgs p;
  p.x = a.x;
  p.w = a.w;
  p.bias = a.bias;
  p.y = a.y;
  p.total = g.y_elems();
  p.G = g.G, p.Cg = g.Cg, p.Kg = g.Kg;
  p.D = g.D, p.H = g.H, p.W = g.W, p.Do = g.Do, p.Ho = g.Ho, p.Wo = g.Wo;
  p.Z = g.Z, p.Y = g.Y, p.X = g.X;
  p.sD = g.sD, p.sH = g.sH, p.sW = g.sW, p.pD = g.pD, p.pH = g.pH, p.pW = g.pW;
  p.dD = g.dD, p.dH = g.dH, p.dW = g.dW;
  const int block = 256;
  cudaError_t e = cudaSuccess;
  // Warp per output when one thread per output would not fill the GPU
  // (fewer than 16 threads per SM lane group) and each output sums at least
  // 64 products; otherwise thread per output.
  const int64_t red = (int64_t)g.taps() * g.Cg;
  if (p.total < (int64_t)dev.num_sms * 2048 && red >= 64) {
    const int64_t wblocks = (p.total + (block / 32) - 1) / (block / 32);
    const int grid = (int)std::min<int64_t>(wblocks, (int64_t)dev.num_sms * 16);
    switch (a.dt) {
      case kF32: e = launch_kernel(generic_warp_kernel<float>, dim3(grid), dim3(block), 0, a, p); break;
      case kF16: e = launch_kernel(generic_warp_kernel<__half>, dim3(grid), dim3(block), 0, a, p); break;
      case kBF16: e = launch_kernel(generic_warp_kernel<__nv_bfloat16>, dim3(grid), dim3(block), 0, a, p); break;
    }
    return e;
  }
  const int grid = grid_for(p.total, block, &dev);
  switch (a.dt) {
    case kF32: e = launch_kernel(generic_direct_kernel<float>, dim3(grid), dim3(block), 0, a, p); break;
    case kF16: e = launch_kernel(generic_direct_kernel<__half>, dim3(grid), dim3(block), 0, a, p); break;
    case kBF16: e = launch_kernel(generic_direct_kernel<__nv_bfloat16>, dim3(grid), dim3(block), 0, a, p); break;
  }
  return e;
}

cudaError_t epilogue_launch(const float* acc, const void* bias, void* y, int64_t rows, int cols,
                            DType dt, cudaStream_t stream) {
  const int64_t total = rows * (int64_t)cols;
  if (total == 0) return cudaSuccess;
  const int block = 256;
  const int grid = grid_for(total, block, nullptr);
  switch (dt) {
    case kF32:
      epilogue_kernel<float><<<grid, block, 0, stream>>>(acc, static_cast<const float*>(bias),
                                                         static_cast<float*>(y), total, cols);
      break;
    case kF16:
      epilogue_kernel<__half><<<grid, block, 0, stream>>>(acc, static_cast<const __half*>(bias),
                                                          static_cast<__half*>(y), total, cols);
      break;
    case kBF16:
      epilogue_kernel<__nv_bfloat16><<<grid, block, 0, stream>>>(
          acc, static_cast<const __nv_bfloat16*>(bias), static_cast<__nv_bfloat16*>(y), total, cols);
      break;
  }
  return cudaGetLastError();
}

}  // namespace gconv
