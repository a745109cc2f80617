// Grouped convolution backward data (the gradient with respect to x).
//
// dx[n, i, g, c] = sum over (o, t, k) with i = o*s - p + t*d in every
// dimension of dy[n, o, g, k] * w[g, k, t, c] -- the adjoint of the forward
// map in x.  The backward-data variant and its runner contract (dY, W) are
// listed by the pages' CK grouped-convolution tile engine and its Python
// examples; the arithmetic is that adjoint.
//
// Three routes (chosen in api.cu):
//  - stride 1 and pad <= d*(k-1) in every dimension: dx is the forward
//    convolution of dy with per-group transposed, spatially flipped weights
//    wt[g, c, t', k] = w[g, k, flip(t'), c] and padding d*(k-1) - p, so the
//    forward kernels (depthwise, tensor-core, generic) run it after
//    weight_flip_kernel has written wt into the caller's workspace;
//  - stride > 1 with grouped channels: dx is cut into its stride phases
//    (dx positions i = s*i' + r per dimension).  Phase r receives only the
//    taps t with (r + p - t*d) divisible by s, at dy offset
//    q = (r + p - t*d) / s, so it is a stride-1 forward correlation of dy
//    with that sub-filter (taps in ascending q, transposed channels) into a
//    phase buffer, which phase_scatter_kernel writes to dx's positions of
//    the phase (phases without taps write zeros);
//  - otherwise a direct kernel gathers, for each dx element, the outputs
//    whose windows cover it (fp32 accumulation, one rounding):
//    bwd_data_vec_kernel handles 16 bytes of channels per thread where they
//    share a group (or are depthwise groups), bwd_data_direct_kernel one
//    element per thread otherwise.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace gconv {
namespace {

// wt[g][c][z][y][x][k] = w[g][k][Z-1-z][Y-1-y][X-1-x][c]: consecutive threads
// write consecutive k (coalesced writes; the reads are a small gather from a
// tensor that stays in L2).
template <typename T>
__global__ void __launch_bounds__(256) weight_flip_kernel(const T* __restrict__ w, T* __restrict__ wt,
                                                          int64_t total, int Kg, int Cg, int Z, int Y, int X) {
  grid_dependency_wait();  // w and the workspace are touched only from here on
  for (int64_t o = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; o < total;
       o += (int64_t)gridDim.x * blockDim.x) {
    int64_t f = o;
    const int k = (int)(f % Kg);
    f /= Kg;
    const int xx = (int)(f % X);
    f /= X;
    const int yy = (int)(f % Y);
    f /= Y;
    const int z = (int)(f % Z);
    f /= Z;
    const int c = (int)(f % Cg);
    const int64_t g = f / Cg;
    wt[o] = w[((((g * Kg + k) * Z + (Z - 1 - z)) * Y + (Y - 1 - yy)) * (int64_t)X + (X - 1 - xx)) * Cg + c];
  }
}

struct BwdArgs {
  const void* dy;
  const void* w;
  void* dx;
  int64_t total;  // dx elements
  int G, Cg, Kg;
  int D, H, W, Do, Ho, Wo, Z, Y, X;
  int sD, sH, sW, pD, pH, pW, dD, dH, dW;
};

// One thread per dx element (channel fastest: coalesced dx writes and weight
// reads, dy reads shared by the warp).  I is the index type of the element
// decode: 32-bit unsigned when the element count fits, else 64-bit.  Output positions o along a dimension
// satisfy o*s = i + p - t*d; taps whose offset is not a multiple of the stride
// or lands outside the output contribute nothing.
template <typename T, typename I>
__global__ void __launch_bounds__(256) bwd_data_direct_kernel(const BwdArgs a) {
  const T* __restrict__ dy = static_cast<const T*>(a.dy);
  const T* __restrict__ w = static_cast<const T*>(a.w);
  T* __restrict__ dx = static_cast<T*>(a.dx);
  const int64_t K = (int64_t)a.G * a.Kg;
  const int64_t kstride = (int64_t)a.Z * a.Y * a.X * a.Cg;  // weight stride between output channels
  grid_dependency_wait();  // dy, w and dx are touched only from here on
  const I total = (I)a.total;
  for (I o = (I)blockIdx.x * (I)blockDim.x + (I)threadIdx.x; o < total; o += (I)gridDim.x * (I)blockDim.x) {
    I f = o;
    const int c = (int)(f % (I)a.Cg);
    f /= (I)a.Cg;
    const int g = (int)(f % (I)a.G);
    f /= (I)a.G;
    const int iw = (int)(f % (I)a.W);
    f /= (I)a.W;
    const int ih = (int)(f % (I)a.H);
    f /= (I)a.H;
    const int id = (int)(f % (I)a.D);
    const int64_t n = (int64_t)(f / (I)a.D);
    float acc = 0.f;
    for (int z = 0; z < a.Z; ++z) {
      const int nd = id + a.pD - z * a.dD;
      if (nd < 0 || nd % a.sD != 0) continue;
      const int od = nd / a.sD;
      if (od >= a.Do) continue;
      for (int yy = 0; yy < a.Y; ++yy) {
        const int nh = ih + a.pH - yy * a.dH;
        if (nh < 0 || nh % a.sH != 0) continue;
        const int oh = nh / a.sH;
        if (oh >= a.Ho) continue;
        for (int xx = 0; xx < a.X; ++xx) {
          const int nw = iw + a.pW - xx * a.dW;
          if (nw < 0 || nw % a.sW != 0) continue;
          const int ow = nw / a.sW;
          if (ow >= a.Wo) continue;
          const T* dyp = dy + (((n * a.Do + od) * a.Ho + oh) * (int64_t)a.Wo + ow) * K + (int64_t)g * a.Kg;
          const T* wp = w + ((((int64_t)g * a.Kg * a.Z + z) * a.Y + yy) * a.X + xx) * a.Cg + c;
#pragma unroll 4
          for (int k = 0; k < a.Kg; ++k)
            acc = fmaf(Elem<T>::to_f32(dyp[k]), Elem<T>::to_f32(wp[k * kstride]), acc);
        }
      }
    }
    dx[(int64_t)o] = epilogue_one<T>(acc, 0.f);
  }
}

// V = 16 / sizeof(T) consecutive dx channels per thread (one 16-byte store).
// MODE 0: the V channels lie in one group (Cg % V == 0): a single dy value per
//   (output, k) serves all V, and their weights are one 16-byte load.
// MODE 1: depthwise (Cg == Kg == 1, G % V == 0): the V channels are V groups;
//   their dy values are one 16-byte load, their weights V scalar loads.
// I is the index type of the element decode: 32-bit unsigned when the vector
// count fits, else 64-bit.  Same sums in the same order as the scalar kernel.
template <typename T, int MODE, typename I>
__global__ void __launch_bounds__(256) bwd_data_vec_kernel(const BwdArgs a) {
  constexpr int V = 16 / (int)sizeof(T);
  const T* __restrict__ dy = static_cast<const T*>(a.dy);
  const T* __restrict__ w = static_cast<const T*>(a.w);
  T* __restrict__ dx = static_cast<T*>(a.dx);
  const int64_t C = (int64_t)a.G * a.Cg, K = (int64_t)a.G * a.Kg;
  const int taps = a.Z * a.Y * a.X;
  const int64_t kstride = (int64_t)taps * a.Cg;
  const I per_pixel = (I)(MODE == 0 ? (a.Cg / V) * a.G : a.G / V);  // vectors per dx pixel
  const I nvec = (I)(a.total / V);
  grid_dependency_wait();  // dy, w and dx are touched only from here on
  for (I o = (I)blockIdx.x * (I)blockDim.x + (I)threadIdx.x; o < nvec; o += (I)gridDim.x * (I)blockDim.x) {
    I f = o;
    const int v = (int)(f % per_pixel);
    f /= per_pixel;
    int g, c;
    if constexpr (MODE == 0) {
      const int cvs = a.Cg / V;
      g = v / cvs;
      c = (v - g * cvs) * V;
    } else {
      g = v * V;
      c = 0;
    }
    const int iw = (int)(f % (I)a.W);
    f /= (I)a.W;
    const int ih = (int)(f % (I)a.H);
    f /= (I)a.H;
    const int id = (int)(f % (I)a.D);
    const int64_t n = (int64_t)(f / (I)a.D);
    float acc[V];
#pragma unroll
    for (int j = 0; j < V; ++j) acc[j] = 0.f;
    for (int z = 0; z < a.Z; ++z) {
      const int nd = id + a.pD - z * a.dD;
      if (nd < 0 || nd % a.sD != 0) continue;
      const int od = nd / a.sD;
      if (od >= a.Do) continue;
      for (int yy = 0; yy < a.Y; ++yy) {
        const int nh = ih + a.pH - yy * a.dH;
        if (nh < 0 || nh % a.sH != 0) continue;
        const int oh = nh / a.sH;
        if (oh >= a.Ho) continue;
        for (int xx = 0; xx < a.X; ++xx) {
          const int nw = iw + a.pW - xx * a.dW;
          if (nw < 0 || nw % a.sW != 0) continue;
          const int ow = nw / a.sW;
          if (ow >= a.Wo) continue;
          const int64_t opix = ((n * a.Do + od) * a.Ho + oh) * (int64_t)a.Wo + ow;
          if constexpr (MODE == 0) {
            const T* dyp = dy + opix * K + (int64_t)g * a.Kg;
            const T* wp = w + ((((int64_t)g * a.Kg * a.Z + z) * a.Y + yy) * a.X + xx) * a.Cg + c;
#pragma unroll 2
            for (int k = 0; k < a.Kg; ++k) {
              const float d = Elem<T>::to_f32(dyp[k]);
              float wf[V];
              unpack16<T>(*reinterpret_cast<const uint4*>(wp + k * kstride), wf);
#pragma unroll
              for (int j = 0; j < V; ++j) acc[j] = fmaf(d, wf[j], acc[j]);
            }
          } else {
            float df[V];
            unpack16<T>(*reinterpret_cast<const uint4*>(dy + opix * K + g), df);
            const int t = (z * a.Y + yy) * a.X + xx;
#pragma unroll
            for (int j = 0; j < V; ++j)
              acc[j] = fmaf(df[j], Elem<T>::to_f32(w[(int64_t)(g + j) * taps + t]), acc[j]);
          }
        }
      }
    }
    const float zero[V] = {};
    epilogue_store<T, V>(dx + (((n * a.D + id) * a.H + ih) * (int64_t)a.W + iw) * C + (int64_t)g * a.Cg + c, acc,
                         zero);
  }
}

// Phase route, weights: wt[g][c][jd][jh][jw][k] = w[g][k][td[jd]][th[jh]][tw[jw]][c]
// for the sub-filter of one stride phase (its taps in the order the phase's
// forward correlation reads them).
template <typename T>
__global__ void __launch_bounds__(256) phase_weight_kernel(const T* __restrict__ w, T* __restrict__ wt,
                                                           const PhaseTaps pt, int64_t total, int Kg, int Cg, int Z,
                                                           int Y, int X) {
  grid_dependency_wait();  // w and the workspace are touched only from here on
  for (int64_t o = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; o < total; o += (int64_t)gridDim.x * blockDim.x) {
    int64_t f = o;
    const int k = (int)(f % Kg);
    f /= Kg;
    const int jw = (int)(f % pt.L[2]);
    f /= pt.L[2];
    const int jh = (int)(f % pt.L[1]);
    f /= pt.L[1];
    const int jd = (int)(f % pt.L[0]);
    f /= pt.L[0];
    const int c = (int)(f % Cg);
    const int64_t g = f / Cg;
    wt[o] = w[((((g * Kg + k) * Z + pt.t[0][jd]) * Y + pt.t[1][jh]) * (int64_t)X + pt.t[2][jw]) * Cg + c];
  }
}

// Stacked phases: one sub-filter position q per dimension holds, for phase
// ph (residue r per dimension), the tap t with r + p - t*d = s*(qmin + q),
// if there is one; the stacked weights are zero elsewhere.
template <typename T>
__global__ void __launch_bounds__(256) phase_stack_kernel(const T* __restrict__ w, T* __restrict__ ws,
                                                          const StackTaps st, int64_t total, int G, int Kg, int Cg,
                                                          int Z, int Y, int X) {
  grid_dependency_wait();  // w and the workspace are touched only from here on
  for (int64_t o = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; o < total; o += (int64_t)gridDim.x * blockDim.x) {
    int64_t f = o;
    const int kc = (int)(f % Kg);  // dy channel = input channel of the stacked problem
    f /= Kg;
    int q[3];
    q[2] = (int)(f % st.Q[2]);
    f /= st.Q[2];
    q[1] = (int)(f % st.Q[1]);
    f /= st.Q[1];
    q[0] = (int)(f % st.Q[0]);
    f /= st.Q[0];
    const int kp = (int)(f % (st.nph * Cg));
    const int64_t g = f / (st.nph * Cg);
    const int ph = kp / Cg, c = kp - ph * Cg;
    const int r[3] = {ph / (st.s[1] * st.s[2]), (ph / st.s[2]) % st.s[1], ph % st.s[2]};
    int t[3];
    bool ok = true;
    for (int i = 0; i < 3; ++i) {
      const int num = r[i] + st.p[i] - st.s[i] * (st.qmin[i] + q[i]);
      t[i] = num >= 0 && num % st.d[i] == 0 ? num / st.d[i] : -1;
      ok = ok && t[i] >= 0 && t[i] < st.k[i];
    }
    T v = Elem<T>::from_f32(0.f);
    if (ok) v = w[((((g * Kg + kc) * Z + t[0]) * Y + t[1]) * (int64_t)X + t[2]) * Cg + c];
    ws[o] = v;
  }
}

// Phase route, output: dx[n][sD*i + rD][sH*j + rH][sW*l + rW][:] =
// pb[n][i + oD][j + oH][l + oW][:] for the phase's (i, j, l) < (nD, nH, nW),
// or 0 when the phase has no taps.  V elements (16 or fewer bytes) per
// thread.
template <typename T, int V>
__global__ void __launch_bounds__(256) phase_scatter_kernel(const T* __restrict__ pb, T* __restrict__ dx,
                                                            const PhaseScatter ps) {
  grid_dependency_wait();  // the phase buffer is complete; dx is touched only from here on
  const int64_t cv = ps.C / V;
  const int64_t total = ps.N * ps.n[0] * ps.n[1] * ps.n[2] * cv;
  for (int64_t o = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; o < total; o += (int64_t)gridDim.x * blockDim.x) {
    int64_t f = o;
    const int64_t c = (f % cv) * V;
    f /= cv;
    const int l = (int)(f % ps.n[2]);
    f /= ps.n[2];
    const int j = (int)(f % ps.n[1]);
    f /= ps.n[1];
    const int i = (int)(f % ps.n[0]);
    const int64_t n = f / ps.n[0];
    T* d = dx + (((n * ps.in[0] + (int64_t)ps.s[0] * i + ps.r[0]) * ps.in[1] + (int64_t)ps.s[1] * j + ps.r[1]) *
                     ps.in[2] + (int64_t)ps.s[2] * l + ps.r[2]) * ps.C + c;
    if (ps.empty) {
#pragma unroll
      for (int v = 0; v < V; ++v) d[v] = Elem<T>::from_f32(0.f);
      continue;
    }
    const T* src = pb + (((n * ps.o[0] + i + ps.off[0]) * ps.o[1] + j + ps.off[1]) * (int64_t)ps.o[2] + l + ps.off[2]) *
                            ps.C + c;
    if constexpr (V * sizeof(T) == 16) {
      *reinterpret_cast<uint4*>(d) = *reinterpret_cast<const uint4*>(src);
    } else {
#pragma unroll
      for (int v = 0; v < V; ++v) d[v] = src[v];
    }
  }
}

int grid_blocks(int64_t total, const DeviceInfo& dev) {
  const int64_t blocks = (total + 255) / 256;
  return (int)std::max<int64_t>(1, std::min<int64_t>(blocks, (int64_t)dev.num_sms * 16));
}

}  // namespace

cudaError_t bwd_weight_flip_launch(const Geometry& g, const LaunchArgs& a, void* wt, const DeviceInfo& dev) {
  const int64_t total = g.w_elems();
  const dim3 grid(grid_blocks(total, dev)), block(256);
  switch (a.dt) {
    case kF32:
      return launch_kernel(weight_flip_kernel<float>, grid, block, 0, a, static_cast<const float*>(a.w),
                           static_cast<float*>(wt), total, g.Kg, g.Cg, g.Z, g.Y, g.X);
    case kF16:
      return launch_kernel(weight_flip_kernel<__half>, grid, block, 0, a, static_cast<const __half*>(a.w),
                           static_cast<__half*>(wt), total, g.Kg, g.Cg, g.Z, g.Y, g.X);
    case kBF16:
      return launch_kernel(weight_flip_kernel<__nv_bfloat16>, grid, block, 0, a,
                           static_cast<const __nv_bfloat16*>(a.w), static_cast<__nv_bfloat16*>(wt), total, g.Kg,
                           g.Cg, g.Z, g.Y, g.X);
  }
  return cudaErrorNotSupported;
}

cudaError_t bwd_data_direct_launch(const Geometry& g, const LaunchArgs& a, const DeviceInfo& dev) {
  BwdArgs p;
  p.dy = a.x;  // the forward kernels' x slot carries dy
  p.w = a.w;
  p.dx = a.y;
  p.total = g.x_elems();
  p.G = g.G, p.Cg = g.Cg, p.Kg = g.Kg;
  p.D = g.D, p.H = g.H, p.W = g.W, p.Do = g.Do, p.Ho = g.Ho, p.Wo = g.Wo;
  p.Z = g.Z, p.Y = g.Y, p.X = g.X;
  p.sD = g.sD, p.sH = g.sH, p.sW = g.sW, p.pD = g.pD, p.pH = g.pH, p.pW = g.pW;
  p.dD = g.dD, p.dH = g.dH, p.dW = g.dW;
  // Vector form when 16 bytes of dx channels share a group (or are 16 bytes of
  // depthwise groups) and the vector accesses are aligned; else one element
  // per thread.
  const int V = 16 / dtype_bytes(a.dt);
  const bool a16 = ((reinterpret_cast<uintptr_t>(a.x) | reinterpret_cast<uintptr_t>(a.w) |
                     reinterpret_cast<uintptr_t>(a.y)) & 15) == 0;
  int mode = -1;
  if (a16 && g.Cg % V == 0) mode = 0;
  else if (a16 && g.Cg == 1 && g.Kg == 1 && g.G % V == 0) mode = 1;
  if (mode >= 0) {
    const bool narrow = p.total / V < ((int64_t)1 << 31);
    const dim3 grid(grid_blocks(p.total / V, dev)), block(256);
#define GCONV_BWD_VEC(TT)                                                                                  \
  if (mode == 0)                                                                                           \
    return narrow ? launch_kernel(bwd_data_vec_kernel<TT, 0, uint32_t>, grid, block, 0, a, p)              \
                  : launch_kernel(bwd_data_vec_kernel<TT, 0, int64_t>, grid, block, 0, a, p);              \
  return narrow ? launch_kernel(bwd_data_vec_kernel<TT, 1, uint32_t>, grid, block, 0, a, p)                \
                : launch_kernel(bwd_data_vec_kernel<TT, 1, int64_t>, grid, block, 0, a, p);
    switch (a.dt) {
      case kF32: GCONV_BWD_VEC(float)
      case kF16: GCONV_BWD_VEC(__half)
      case kBF16: GCONV_BWD_VEC(__nv_bfloat16)
    }
#undef GCONV_BWD_VEC
    return cudaErrorNotSupported;
  }
  const dim3 grid(grid_blocks(p.total, dev)), block(256);
  const bool narrow = p.total < ((int64_t)1 << 31);
#define GCONV_BWD_ONE(TT)                                                                   \
  return narrow ? launch_kernel(bwd_data_direct_kernel<TT, uint32_t>, grid, block, 0, a, p) \
                : launch_kernel(bwd_data_direct_kernel<TT, int64_t>, grid, block, 0, a, p);
  switch (a.dt) {
    case kF32: GCONV_BWD_ONE(float)
    case kF16: GCONV_BWD_ONE(__half)
    case kBF16: GCONV_BWD_ONE(__nv_bfloat16)
  }
#undef GCONV_BWD_ONE
  return cudaErrorNotSupported;
}

cudaError_t phase_weight_launch(const Geometry& g, const LaunchArgs& a, const PhaseTaps& pt, void* wt,
                                const DeviceInfo& dev) {
  const int64_t total = (int64_t)g.G * g.Cg * pt.L[0] * pt.L[1] * pt.L[2] * g.Kg;
  const dim3 grid(grid_blocks(total, dev)), block(256);
  switch (a.dt) {
    case kF32:
      return launch_kernel(phase_weight_kernel<float>, grid, block, 0, a, static_cast<const float*>(a.w),
                           static_cast<float*>(wt), pt, total, g.Kg, g.Cg, g.Z, g.Y, g.X);
    case kF16:
      return launch_kernel(phase_weight_kernel<__half>, grid, block, 0, a, static_cast<const __half*>(a.w),
                           static_cast<__half*>(wt), pt, total, g.Kg, g.Cg, g.Z, g.Y, g.X);
    case kBF16:
      return launch_kernel(phase_weight_kernel<__nv_bfloat16>, grid, block, 0, a,
                           static_cast<const __nv_bfloat16*>(a.w), static_cast<__nv_bfloat16*>(wt), pt, total, g.Kg,
                           g.Cg, g.Z, g.Y, g.X);
  }
  return cudaErrorNotSupported;
}

cudaError_t phase_stack_launch(const Geometry& g, const LaunchArgs& a, const StackTaps& st, void* ws,
                               const DeviceInfo& dev) {
  const int64_t total = (int64_t)g.G * st.nph * g.Cg * st.Q[0] * st.Q[1] * st.Q[2] * g.Kg;
  const dim3 grid(grid_blocks(total, dev)), block(256);
  switch (a.dt) {
    case kF16:
      return launch_kernel(phase_stack_kernel<__half>, grid, block, 0, a, static_cast<const __half*>(a.w),
                           static_cast<__half*>(ws), st, total, g.G, g.Kg, g.Cg, g.Z, g.Y, g.X);
    case kBF16:
      return launch_kernel(phase_stack_kernel<__nv_bfloat16>, grid, block, 0, a,
                           static_cast<const __nv_bfloat16*>(a.w), static_cast<__nv_bfloat16*>(ws), st, total, g.G,
                           g.Kg, g.Cg, g.Z, g.Y, g.X);
    default:
      return cudaErrorNotSupported;
  }
}

cudaError_t phase_scatter_launch(const PhaseScatter& ps, const void* pb, void* dx, const LaunchArgs& a,
                                 const DeviceInfo& dev) {
  const int es = dtype_bytes(a.dt);
  const bool v16 = (ps.C * es) % 16 == 0 &&
                   ((reinterpret_cast<uintptr_t>(pb) | reinterpret_cast<uintptr_t>(dx)) & 15) == 0;
  const int V = v16 ? 16 / es : 1;
  const int64_t total = ps.N * ps.n[0] * ps.n[1] * ps.n[2] * (ps.C / V);
  const dim3 grid(grid_blocks(total, dev)), block(256);
#define GCONV_SCATTER(TT)                                                                                          return v16 ? launch_kernel(phase_scatter_kernel<TT, 16 / sizeof(TT)>, grid, block, 0, a,                                                    static_cast<const TT*>(pb), static_cast<TT*>(dx), ps)                                           : launch_kernel(phase_scatter_kernel<TT, 1>, grid, block, 0, a, static_cast<const TT*>(pb),                                       static_cast<TT*>(dx), ps);
  switch (a.dt) {
    case kF32: GCONV_SCATTER(float)
    case kF16: GCONV_SCATTER(__half)
    case kBF16: GCONV_SCATTER(__nv_bfloat16)
  }
#undef GCONV_SCATTER
  return cudaErrorNotSupported;
}

}  // namespace gconv
