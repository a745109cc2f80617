// C ABI of the grouped-convolution library (forward pass and backward data):
// argument validation, output-shape rule, shape-based kernel selection,
// tensor-map encoding and launch.  Everything here runs on the host; the
// arithmetic runs in the kernels (dw*.cu, generic.cu, tc*.cu, bwd.cu).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/gconv.h"
#include "fused.h"
#include "kernels.h"

namespace gconv {

// Device status word: [code, where].  Kernels set it when a bounded wait
// expires; gconv_device_status / debug mode read and clear it.
__device__ int g_status_word[2];

namespace {

thread_local char t_last_error[512] = "";

gconv_status fail(gconv_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_last_error, sizeof(t_last_error), fmt, ap);
  va_end(ap);
  return s;
}

// ---------------------------------------------------------------------------
// Output extent: floor((I + 2p - d*(k-1) - 1) / s) + 1 (0 when nothing fits).
// ---------------------------------------------------------------------------
int64_t out_extent(int64_t in, int64_t k, int64_t s, int64_t p, int64_t d) {
  const int64_t span = d * (k - 1) + 1;
  const int64_t room = in + 2 * p - span;
  if (room < 0) return 0;
  return room / s + 1;
}

gconv_status validate(const gconv_problem* p, Geometry* g) {
  if (p == nullptr) return fail(GCONV_ERR_INVALID_ARG, "problem pointer is NULL");
  if (p->ndim != 2 && p->ndim != 3) return fail(GCONV_ERR_INVALID_ARG, "ndim must be 2 or 3 (got %d)", p->ndim);
  if (p->reserved != 0) return fail(GCONV_ERR_INVALID_ARG, "reserved field must be 0");
  if (p->N < 1) return fail(GCONV_ERR_INVALID_ARG, "N must be >= 1");
  if (p->G < 1 || p->C < 1 || p->K < 1) return fail(GCONV_ERR_INVALID_ARG, "G, C and K must be >= 1");
  if (p->C % p->G != 0) return fail(GCONV_ERR_INVALID_ARG, "C (%d) is not divisible by G (%d)", p->C, p->G);
  if (p->K % p->G != 0) return fail(GCONV_ERR_INVALID_ARG, "K (%d) is not divisible by G (%d)", p->K, p->G);
  for (int i = 0; i < 3; ++i) {
    if (p->in[i] < 1 || p->ker[i] < 1) return fail(GCONV_ERR_INVALID_ARG, "extents must be >= 1 (dim %d)", i);
    if (p->stride[i] < 1 || p->dil[i] < 1) return fail(GCONV_ERR_INVALID_ARG, "stride and dilation must be >= 1 (dim %d)", i);
    if (p->pad[i] < 0) return fail(GCONV_ERR_INVALID_ARG, "padding must be >= 0 (dim %d)", i);
  }
  if (p->ndim == 2 && (p->in[0] != 1 || p->ker[0] != 1 || p->stride[0] != 1 || p->dil[0] != 1 || p->pad[0] != 0))
    return fail(GCONV_ERR_INVALID_ARG, "2D problem: depth fields must be in=ker=stride=dil=1, pad=0");
  int64_t o[3];
  for (int i = 0; i < 3; ++i) {
    o[i] = out_extent(p->in[i], p->ker[i], p->stride[i], p->pad[i], p->dil[i]);
    if (o[i] < 1) return fail(GCONV_ERR_INVALID_ARG, "output extent of dim %d is empty", i);
  }
  // Element counts must fit comfortably in 63 bits.
  const double xe = (double)p->N * p->in[0] * p->in[1] * p->in[2] * p->C;
  const double ye = (double)p->N * o[0] * o[1] * o[2] * p->K;
  if (xe > 4e18 || ye > 4e18) return fail(GCONV_ERR_INVALID_ARG, "tensor too large");
  if (p->N > (int64_t)1 << 31) return fail(GCONV_ERR_INVALID_ARG, "N too large");
  g->N = p->N;
  g->G = p->G;
  g->Cg = p->C / p->G;
  g->Kg = p->K / p->G;
  g->D = p->in[0], g->H = p->in[1], g->W = p->in[2];
  g->Do = (int)o[0], g->Ho = (int)o[1], g->Wo = (int)o[2];
  g->Z = p->ker[0], g->Y = p->ker[1], g->X = p->ker[2];
  g->sD = p->stride[0], g->sH = p->stride[1], g->sW = p->stride[2];
  g->pD = p->pad[0], g->pH = p->pad[1], g->pW = p->pad[2];
  g->dD = p->dil[0], g->dH = p->dil[1], g->dW = p->dil[2];
  g->ndim = p->ndim;
  return GCONV_OK;
}

bool overlaps(const void* a, int64_t abytes, const void* b, int64_t bbytes) {
  if (a == nullptr || b == nullptr) return false;
  const uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
  return a0 < b0 + (uintptr_t)bbytes && b0 < a0 + (uintptr_t)abytes;
}

// Shape-based choice: the depthwise kernel, else the tensor-core kernel, else
// the generic kernel; each specialised kernel is taken only when its planner
// finds a launch plan for this device (dev; NULL: a GB300's SM count and
// shared memory, for the host-only query).  Groups of two channels run on
// the direct kernel at stride 1 and dilation 1 and on the tensor-core kernel
// otherwise, the faster of the two on GB300 (sweep G=256: 33.4 against 35.6
// us at stride 1 dilation 1; 38.3 against 35.4 us at dilation 2; 15.9-14.2
// against 21.8-23.6 us at stride 2).
int select_kernel(const Geometry& g, DType dt, const LaunchArgs* a, const DeviceInfo* dev) {
  const int sms = dev ? dev->num_sms : kDefaultSms;
  const int smem = dev ? dev->max_smem_optin : kDefaultSmemOptin;
  if (g.Cg == 2 && g.Kg == 2 && (g.sH > 1 || g.sW > 1 || g.dH > 1 || g.dW > 1) &&
      tc_supported(g, dt, a, sms, smem))
    return GCONV_KERNEL_IGEMM_TC;
  if (dw_supported(g, dt, a, sms)) return GCONV_KERNEL_DIRECT_DW;
  if (tc_supported(g, dt, a, sms, smem)) return GCONV_KERNEL_IGEMM_TC;
  return GCONV_KERNEL_DIRECT_GENERIC;
}

// ---------------------------------------------------------------------------
// Per-device cache: SM count, shared-memory limit, status-word address.
// ---------------------------------------------------------------------------
// The set-up makes no stream operation and no synchronisation (the status
// word starts at zero when the module is loaded), so a device's first call
// may also come inside a stream capture.  A failed set-up is not kept: the
// next call on that device tries again.
struct DevSlot {
  std::mutex mu;
  std::atomic<bool> ready{false};
  DeviceInfo info{};
  int* status = nullptr;
};
constexpr int kMaxDevices = 64;
DevSlot g_dev[kMaxDevices];

cudaError_t device_slot(DevSlot** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  DevSlot& s = g_dev[dev];
  *out = &s;
  if (s.ready.load(std::memory_order_acquire)) return cudaSuccess;
  std::lock_guard<std::mutex> lock(s.mu);
  if (s.ready.load(std::memory_order_relaxed)) return cudaSuccess;
  DeviceInfo info{};
  info.device = dev;
  int* status = nullptr;
  cudaError_t r = cudaDeviceGetAttribute(&info.num_sms, cudaDevAttrMultiProcessorCount, dev);
  if (r == cudaSuccess) r = cudaDeviceGetAttribute(&info.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (r == cudaSuccess) r = cudaGetSymbolAddress(reinterpret_cast<void**>(&status), g_status_word);
  if (r != cudaSuccess) return r;
  s.info = info;
  s.status = status;
  s.ready.store(true, std::memory_order_release);
  return cudaSuccess;
}

// ---------------------------------------------------------------------------
// cuTensorMapEncodeTiled through the runtime's driver entry point.
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
std::once_flag g_encode_once;
EncodeTiledFn g_encode = nullptr;

gconv_status read_and_clear_status(DevSlot* slot, cudaStream_t stream, int32_t* code, int32_t* where) {
  int host[2] = {0, 0};
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e == cudaSuccess) e = cudaMemcpyAsync(host, slot->status, sizeof(host), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e == cudaSuccess && host[0] != 0) {
    e = cudaMemsetAsync(slot->status, 0, sizeof(host), stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  }
  if (e != cudaSuccess) return fail(GCONV_ERR_CUDA, "status read failed: %s", cudaGetErrorString(e));
  if (code) *code = host[0];
  if (where) *where = host[1];
  return GCONV_OK;
}

LaunchArgs make_args(const void* x, const void* w, const void* bias, void* y, DType dt, struct CUstream_st* stream,
                     DevSlot* slot, const gconv_options* opt) {
  LaunchArgs a;
  a.x = x, a.w = w, a.bias = bias, a.y = y;
  a.dt = dt;
  a.stream = reinterpret_cast<cudaStream_t>(stream);
  a.status = slot->status;
  a.wait_limit_ns = (opt && opt->wait_limit_ns > 0) ? (uint64_t)opt->wait_limit_ns : 2000000000ull;
  a.test_flags = opt ? opt->test_flags : 0;
  for (int i = 0; i < 8; ++i) a.tile[i] = opt ? opt->tile[i] : 0;
  a.pdl = !(opt && opt->serial_launch);
  a.omap = OutMap{};
  return a;
}

// Forward convolution of geometry g on the buffers of a: the forced kernel
// (1..3) or the selector's choice; nothing is launched on an error.
gconv_status launch_forward(const Geometry& g, const LaunchArgs& a, const DeviceInfo& dev, int forced,
                            int32_t* selected) {
  int kernel = forced ? forced : select_kernel(g, a.dt, &a, &dev);
  if (kernel == GCONV_KERNEL_DIRECT_DW && !dw_supported(g, a.dt, &a, dev.num_sms))
    return fail(GCONV_ERR_UNSUPPORTED, "depthwise kernel cannot run this problem");
  if (kernel == GCONV_KERNEL_IGEMM_TC && !tc_supported(g, a.dt, &a, dev.num_sms, dev.max_smem_optin))
    return fail(GCONV_ERR_UNSUPPORTED, "tensor-core kernel cannot run this problem");
  if (kernel < GCONV_KERNEL_DIRECT_DW || kernel > GCONV_KERNEL_IGEMM_TC)
    return fail(GCONV_ERR_UNSUPPORTED, "unknown kernel id %d", kernel);
  cudaError_t e;
  switch (kernel) {
    case GCONV_KERNEL_DIRECT_DW: e = dw_launch(g, a, dev); break;
    case GCONV_KERNEL_IGEMM_TC: e = tc_launch(g, a, dev); break;
    default: e = generic_launch(g, a, dev); break;
  }
  // A selector's choice whose launch finds no plan on this device (the
  // occupancy or shared-memory limits of the device itself) runs on the
  // generic kernel instead; nothing was launched.
  if (e == cudaErrorNotSupported && !forced && kernel != GCONV_KERNEL_DIRECT_GENERIC) {
    kernel = GCONV_KERNEL_DIRECT_GENERIC;
    e = generic_launch(g, a, dev);
  }
  if (selected) *selected = kernel;
  if (e == cudaErrorNotSupported) return fail(GCONV_ERR_UNSUPPORTED, "no launch plan for this problem");
  if (e != cudaSuccess) return fail(GCONV_ERR_CUDA, "launch failed: %s", cudaGetErrorString(e));
  return GCONV_OK;
}

// Debug mode: wait for the stream and turn a device-side timeout into the
// return value.
gconv_status finish(DevSlot* slot, const LaunchArgs& a, const gconv_options* opt) {
  if (opt && opt->debug) {
    int32_t code = 0, where = 0;
    gconv_status st = read_and_clear_status(slot, a.stream, &code, &where);
    if (st != GCONV_OK) return st;
    if (code != 0) return fail(GCONV_ERR_TIMEOUT, "in-kernel wait timed out (site %d)", where);
  }
  return GCONV_OK;
}

// Backward data by the forward kernels: stride 1 and pad <= dil*(k-1) in
// every dimension.  Fills *fg with the forward geometry that computes dx from
// dy: Cg and Kg swapped, input extents = the forward output's, padding
// dil*(k-1) - pad, output extents = the forward input's.
bool bwd_as_forward(const Geometry& g, Geometry* fg) {
  const int k[3] = {g.Z, g.Y, g.X}, s[3] = {g.sD, g.sH, g.sW}, p[3] = {g.pD, g.pH, g.pW},
            d[3] = {g.dD, g.dH, g.dW};
  int q[3];
  for (int i = 0; i < 3; ++i) {
    if (s[i] != 1) return false;
    q[i] = d[i] * (k[i] - 1) - p[i];
    if (q[i] < 0) return false;
  }
  Geometry f = g;
  f.Cg = g.Kg, f.Kg = g.Cg;
  f.D = g.Do, f.H = g.Ho, f.W = g.Wo;
  f.Do = g.D, f.Ho = g.H, f.Wo = g.W;
  f.pD = q[0], f.pH = q[1], f.pW = q[2];
  if (out_extent(f.D, f.Z, 1, f.pD, f.dD) != g.D || out_extent(f.H, f.Y, 1, f.pH, f.dH) != g.H ||
      out_extent(f.W, f.X, 1, f.pW, f.dW) != g.W)
    return false;
  *fg = f;
  return true;
}

// Stride phases of backward data along one dimension (dx extent I, dy
// extent O, filter k, stride s, pad p, dilation d).  dx position s*i + r
// receives dy[i + q] * w[t] for the taps t with r + p - t*d = s*q; in the
// order of ascending q (descending t) those taps form a stride-1
// correlation of dy with dilation q[1] - q[0] and left padding -q[0].  The
// phase's forward problem gets symmetric padding `pad` large enough on both
// sides, so its output row `off + i` is dx's phase row i.
struct Phase1D {
  int n;      // dx positions of the phase
  int L;      // taps of the sub-filter
  int t[kMaxPhaseTaps];
  int dil, pad, out, off;
  bool empty;  // no tap reaches the phase (or it has no positions)
};

bool phase_1d(int I, int O, int k, int s, int p, int d, int r, Phase1D* ph) {
  Phase1D f{};
  f.n = r < I ? (I - r + s - 1) / s : 0;
  int q[kMaxPhaseTaps];
  for (int t = k - 1; t >= 0; --t) {
    const int v = r + p - t * d;
    if (((v % s) + s) % s != 0) continue;
    if (f.L == kMaxPhaseTaps) return false;
    q[f.L] = v / s;
    f.t[f.L++] = t;
  }
  f.empty = f.L == 0 || f.n == 0;
  if (f.empty) {
    f.L = 1, f.t[0] = 0, f.dil = 1, f.pad = 0, f.out = 1, f.off = 0;
    *ph = f;
    return true;
  }
  f.dil = f.L >= 2 ? q[1] - q[0] : 1;
  for (int j = 1; j < f.L; ++j)
    if (q[j] - q[j - 1] != f.dil) return false;
  const int qmin = q[0], qmax = q[f.L - 1];
  f.pad = std::max(0, std::max(-qmin, f.n - O + qmax));
  f.out = O + 2 * f.pad - (qmax - qmin);
  f.off = f.pad + qmin;
  if (f.off < 0 || f.off + f.n > f.out) return false;
  *ph = f;
  return true;
}

// The three dimensions of phase (rD, rH, rW); fg = its forward problem
// (valid when not empty).
struct Phase3D {
  Phase1D d[3];
  bool empty;
  Geometry fg;
};

bool phase_3d(const Geometry& g, int rd, int rh, int rw, Phase3D* ph) {
  const int I[3] = {g.D, g.H, g.W}, O[3] = {g.Do, g.Ho, g.Wo}, k[3] = {g.Z, g.Y, g.X},
            st[3] = {g.sD, g.sH, g.sW}, pd[3] = {g.pD, g.pH, g.pW}, dl[3] = {g.dD, g.dH, g.dW};
  const int r[3] = {rd, rh, rw};
  ph->empty = false;
  for (int i = 0; i < 3; ++i) {
    if (!phase_1d(I[i], O[i], k[i], st[i], pd[i], dl[i], r[i], &ph->d[i])) return false;
    ph->empty = ph->empty || ph->d[i].empty;
  }
  Geometry f = g;
  f.Cg = g.Kg, f.Kg = g.Cg;
  f.D = g.Do, f.H = g.Ho, f.W = g.Wo;
  f.Z = ph->d[0].L, f.Y = ph->d[1].L, f.X = ph->d[2].L;
  f.sD = f.sH = f.sW = 1;
  f.pD = ph->d[0].pad, f.pH = ph->d[1].pad, f.pW = ph->d[2].pad;
  f.dD = ph->d[0].dil, f.dH = ph->d[1].dil, f.dW = ph->d[2].dil;
  f.Do = ph->d[0].out, f.Ho = ph->d[1].out, f.Wo = ph->d[2].out;
  ph->fg = f;
  return true;
}

// All stride phases as one stride-1 forward problem.  For residue r of a
// dimension, dx position s*m + r takes the taps t with r + p - t*d = s*q, from
// dy row m + q.  Over every residue the offsets q span [qmin, qmax]; the
// stacked problem convolves dy with a filter of Q = qmax - qmin + 1 offsets
// per dimension whose output channels are (phase, dx channel) pairs, zero
// where a phase has no tap at an offset.  Its output v maps to phase index
// m = v - o_off (o_off = pad + qmin), written at s*m + r (OutMap mode 2).
// Phases without taps come out as zeros.  Returns false when a dimension
// has no tap reaching any residue.
struct Stacked {
  Geometry fg;
  StackTaps st;
  OutMap om;
  int64_t w_elems;  // stacked weight elements
};

bool stacked_problem(const Geometry& g, Stacked* out) {
  const int I[3] = {g.D, g.H, g.W}, O[3] = {g.Do, g.Ho, g.Wo}, k[3] = {g.Z, g.Y, g.X},
            s[3] = {g.sD, g.sH, g.sW}, p[3] = {g.pD, g.pH, g.pW}, d[3] = {g.dD, g.dH, g.dW};
  Stacked st{};
  st.st.nph = s[0] * s[1] * s[2];
  if (st.st.nph > kMaxStackPhases) return false;
  Geometry f = g;
  f.Cg = g.Kg, f.Kg = st.st.nph * g.Cg;
  f.D = g.Do, f.H = g.Ho, f.W = g.Wo;
  f.sD = f.sH = f.sW = 1;
  f.dD = f.dH = f.dW = 1;
  int fk[3], fp[3], fo[3];
  st.om.on = 2;
  for (int i = 0; i < 3; ++i) {
    int qmin = 1 << 30, qmax = -(1 << 30);
    for (int r = 0; r < s[i]; ++r)
      for (int t = 0; t < k[i]; ++t) {
        const int v = r + p[i] - t * d[i];
        if (((v % s[i]) + s[i]) % s[i] != 0) continue;
        const int q = (v - (((v % s[i]) + s[i]) % s[i])) / s[i];
        qmin = std::min(qmin, q);
        qmax = std::max(qmax, q);
      }
    if (qmin > qmax) return false;
    const int Q = qmax - qmin + 1, M = (I[i] + s[i] - 1) / s[i];
    const int pad = std::max(0, std::max(-qmin, M + qmax - O[i]));
    fk[i] = Q, fp[i] = pad, fo[i] = O[i] + 2 * pad - Q + 1;
    st.st.s[i] = s[i], st.st.p[i] = p[i], st.st.d[i] = d[i], st.st.k[i] = k[i];
    st.st.Q[i] = Q, st.st.qmin[i] = qmin;
    st.om.scale[i] = s[i];
    st.om.add[i] = -s[i] * (pad + qmin);
    st.om.lo[i] = pad + qmin;
    st.om.hi[i] = fo[i];
    st.om.ext[i] = I[i];
  }
  f.Z = fk[0], f.Y = fk[1], f.X = fk[2];
  f.pD = fp[0], f.pH = fp[1], f.pW = fp[2];
  f.Do = fo[0], f.Ho = fo[1], f.Wo = fo[2];
  st.fg = f;
  st.om.cpp = g.Cg, st.om.nph = st.st.nph, st.om.ctot = g.C();
  for (int ph = 0; ph < st.st.nph; ++ph) {
    st.om.res[ph][0] = ph / (s[1] * s[2]);
    st.om.res[ph][1] = (ph / s[2]) % s[1];
    st.om.res[ph][2] = ph % s[2];
  }
  st.w_elems = f.w_elems();
  *out = st;
  return true;
}

// The stacked phases on the tensor-core kernel (planned for a GB300), 16-bit
// grouped data with a stride above 1.
// Its epilogue stores 32-byte runs of one phase's channels (Cg a multiple of
// 16) and reads one partial accumulator (tile override slot 4 = 1 for its
// plans).
bool stacked_route(const Geometry& g, DType dt, Stacked* st) {
  if (g.sD == 1 && g.sH == 1 && g.sW == 1) return false;
  if (dt == kF32 || g.Cg % 16 != 0) return false;
  if (!stacked_problem(g, st)) return false;
  LaunchArgs plan{};  // no buffers: alignment is checked at the call
  plan.tile[4] = 1;
  return tc_supported(st->fg, dt, &plan, kDefaultSms, kDefaultSmemOptin);
}

// The stride-phase route: a stride above 1 somewhere, grouped channels (the
// depthwise case stays on the direct kernel's group vectors), 16-bit data,
// and every phase's forward problem planned on the tensor-core kernel (on a
// GB300's SM count and shared memory, so the decision, and the workspace
// size, depend on the problem only).  *pb_bytes: the largest phase buffer.
bool phase_route(const Geometry& g, DType dt, int64_t* pb_bytes) {
  if (g.sD == 1 && g.sH == 1 && g.sW == 1) return false;
  if (dt == kF32 || (g.Cg == 1 && g.Kg == 1)) return false;
  int64_t pb = 0;
  for (int rd = 0; rd < g.sD; ++rd)
    for (int rh = 0; rh < g.sH; ++rh)
      for (int rw = 0; rw < g.sW; ++rw) {
        Phase3D ph;
        if (!phase_3d(g, rd, rh, rw, &ph)) return false;
        if (ph.empty) continue;
        if (!tc_supported(ph.fg, dt, nullptr, kDefaultSms, kDefaultSmemOptin)) return false;
        pb = std::max(pb, ph.fg.y_elems() * dtype_bytes(dt));
      }
  if (pb_bytes) *pb_bytes = pb;
  return true;
}

inline int64_t align256(int64_t v) { return (v + 255) / 256 * 256; }

// Workspace of backward data: the transposed, flipped weights of the
// stride-1 route; the phase route's sub-filter weights (at most w's size)
// and its largest phase buffer; nothing for the direct kernel.
int64_t bwd_workspace_bytes(const Geometry& g, DType dt) {
  Geometry f;
  if (bwd_as_forward(g, &f)) return g.w_elems() * dtype_bytes(dt);
  int64_t pb = 0, need = 0;
  Stacked st;
  if (stacked_route(g, dt, &st)) need = st.w_elems * dtype_bytes(dt);
  if (phase_route(g, dt, &pb)) need = std::max(need, align256(g.w_elems() * dtype_bytes(dt)) + pb);
  return need;
}

}  // namespace

gconv_status set_last_error(gconv_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_last_error, sizeof(t_last_error), fmt, ap);
  va_end(ap);
  return s;
}

CUresult encode_tiled(CUtensorMap* map, CUtensorMapDataType type, uint32_t rank, const void* base,
                      const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                      const uint32_t* elem_strides, CUtensorMapSwizzle swizzle) {
  std::call_once(g_encode_once, []() {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  if (g_encode == nullptr) return CUDA_ERROR_NOT_FOUND;
  return g_encode(map, type, rank, const_cast<void*>(base), dims, strides_bytes, box, elem_strides,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace gconv

using namespace gconv;

extern "C" {

const char* gconv_status_string(gconv_status s) {
  switch (s) {
    case GCONV_OK: return "ok";
    case GCONV_ERR_INVALID_ARG: return "invalid argument";
    case GCONV_ERR_UNSUPPORTED: return "unsupported";
    case GCONV_ERR_CUDA: return "CUDA error";
    case GCONV_ERR_TIMEOUT: return "in-kernel wait timed out";
  }
  return "unknown status";
}

const char* gconv_last_error(void) { return t_last_error; }

gconv_status grouped_conv_out_shape(const gconv_problem* p, int32_t out[3]) {
  Geometry g;
  gconv_status s = validate(p, &g);
  if (s != GCONV_OK) return s;
  if (out == nullptr) return fail(GCONV_ERR_INVALID_ARG, "out pointer is NULL");
  out[0] = g.Do, out[1] = g.Ho, out[2] = g.Wo;
  return GCONV_OK;
}

gconv_status grouped_conv_select(const gconv_problem* p, gconv_dtype dt, int32_t* kernel) {
  Geometry g;
  gconv_status s = validate(p, &g);
  if (s != GCONV_OK) return s;
  if (dt != GCONV_F32 && dt != GCONV_F16 && dt != GCONV_BF16) return fail(GCONV_ERR_UNSUPPORTED, "unknown dtype %d", (int)dt);
  if (kernel == nullptr) return fail(GCONV_ERR_INVALID_ARG, "kernel pointer is NULL");
  *kernel = select_kernel(g, (DType)dt, nullptr, nullptr);
  return GCONV_OK;
}

gconv_status grouped_conv_fwd_ex(const void* x, const void* w, const void* bias, void* y, const gconv_problem* p,
                                 gconv_dtype dt, struct CUstream_st* stream, gconv_options* opt) {
  Geometry g;
  gconv_status s = validate(p, &g);
  if (s != GCONV_OK) return s;
  if (dt != GCONV_F32 && dt != GCONV_F16 && dt != GCONV_BF16) return fail(GCONV_ERR_UNSUPPORTED, "unknown dtype %d", (int)dt);
  if (x == nullptr || w == nullptr || y == nullptr) return fail(GCONV_ERR_INVALID_ARG, "x, w and y must not be NULL");
  const int es = dtype_bytes((DType)dt);
  const int64_t yb = g.y_elems() * es;
  if (overlaps(y, yb, x, g.x_elems() * es) || overlaps(y, yb, w, g.w_elems() * es) ||
      overlaps(y, yb, bias, (int64_t)g.K() * es))
    return fail(GCONV_ERR_INVALID_ARG, "y overlaps an input buffer");

  DevSlot* slot = nullptr;
  cudaError_t e = device_slot(&slot);
  if (e != cudaSuccess) return fail(GCONV_ERR_CUDA, "device query failed: %s", cudaGetErrorString(e));
  LaunchArgs a = make_args(x, w, bias, y, (DType)dt, stream, slot, opt);
  s = launch_forward(g, a, slot->info, opt ? opt->force_kernel : 0, opt ? &opt->selected : nullptr);
  if (s != GCONV_OK) return s;
  return finish(slot, a, opt);
}

gconv_status grouped_conv_bwd_data_workspace_size(const gconv_problem* p, gconv_dtype dt, int64_t* bytes) {
  Geometry g;
  gconv_status s = validate(p, &g);
  if (s != GCONV_OK) return s;
  if (dt != GCONV_F32 && dt != GCONV_F16 && dt != GCONV_BF16) return fail(GCONV_ERR_UNSUPPORTED, "unknown dtype %d", (int)dt);
  if (bytes == nullptr) return fail(GCONV_ERR_INVALID_ARG, "bytes pointer is NULL");
  *bytes = bwd_workspace_bytes(g, (DType)dt);
  return GCONV_OK;
}

gconv_status grouped_conv_bwd_data_ex(const void* dy, const void* w, void* dx, const gconv_problem* p,
                                      gconv_dtype dt, void* workspace, int64_t workspace_bytes,
                                      struct CUstream_st* stream, gconv_options* opt) {
  Geometry g;
  gconv_status s = validate(p, &g);
  if (s != GCONV_OK) return s;
  if (dt != GCONV_F32 && dt != GCONV_F16 && dt != GCONV_BF16) return fail(GCONV_ERR_UNSUPPORTED, "unknown dtype %d", (int)dt);
  if (dy == nullptr || w == nullptr || dx == nullptr) return fail(GCONV_ERR_INVALID_ARG, "dy, w and dx must not be NULL");
  const DType t = (DType)dt;
  const int es = dtype_bytes(t);
  const int64_t dxb = g.x_elems() * es;
  const int forced = opt ? opt->force_kernel : 0;
  Geometry fg;
  const bool as_fwd = forced != GCONV_KERNEL_BWD_DATA_DIRECT && bwd_as_forward(g, &fg);
  int64_t pb_bytes = 0;
  Stacked stk;
  const bool stacked = !as_fwd && forced != GCONV_KERNEL_BWD_DATA_DIRECT && stacked_route(g, t, &stk);
  const bool per_phase = !as_fwd && forced != GCONV_KERNEL_BWD_DATA_DIRECT && phase_route(g, t, &pb_bytes);
  const bool phases = stacked || per_phase;
  if (forced != 0 && forced != GCONV_KERNEL_BWD_DATA_DIRECT && !as_fwd && !phases)
    return fail(GCONV_ERR_UNSUPPORTED, "kernel %d needs a forward-kernel route (stride 1 with pad <= dil*(k-1), "
                "or stride phases of grouped 16-bit data)", forced);
  const int64_t need = as_fwd ? g.w_elems() * es : (phases ? bwd_workspace_bytes(g, t) : 0);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 15)))
    return fail(GCONV_ERR_INVALID_ARG, "workspace must be 16-byte aligned and hold %lld bytes",
                (long long)need);
  if (overlaps(dx, dxb, dy, g.y_elems() * es) || overlaps(dx, dxb, w, g.w_elems() * es) ||
      (need > 0 && overlaps(dx, dxb, workspace, need)))
    return fail(GCONV_ERR_INVALID_ARG, "dx overlaps an input buffer or the workspace");
  if (need > 0 && (overlaps(workspace, need, dy, g.y_elems() * es) || overlaps(workspace, need, w, g.w_elems() * es)))
    return fail(GCONV_ERR_INVALID_ARG, "the workspace overlaps dy or w");

  DevSlot* slot = nullptr;
  cudaError_t e = device_slot(&slot);
  if (e != cudaSuccess) return fail(GCONV_ERR_CUDA, "device query failed: %s", cudaGetErrorString(e));
  if (as_fwd) {
    // transposed, flipped weights into the workspace, then the forward pass
    LaunchArgs flip = make_args(dy, w, nullptr, workspace, t, stream, slot, opt);
    e = bwd_weight_flip_launch(g, flip, workspace, slot->info);
    if (e != cudaSuccess) return fail(GCONV_ERR_CUDA, "launch failed: %s", cudaGetErrorString(e));
    LaunchArgs a = make_args(dy, workspace, nullptr, dx, t, stream, slot, opt);
    s = launch_forward(fg, a, slot->info, forced, opt ? &opt->selected : nullptr);
    if (s != GCONV_OK) return s;
    return finish(slot, a, opt);
  }
  if (stacked && (forced == 0 || forced == GCONV_KERNEL_IGEMM_TC) && !((opt ? opt->test_flags : 0) & 2)) {
    // every phase in one launch: the stacked sub-filters into the workspace,
    // then the stacked forward problem on the tensor-core kernel, whose
    // epilogue places each (phase, channel) output at its dx position
    LaunchArgs da = make_args(dy, workspace, nullptr, dx, t, stream, slot, opt);
    da.omap = stk.om;
    da.tile[4] = 1;  // one partial accumulator
    if (tc_supported(stk.fg, t, &da, slot->info.num_sms, slot->info.max_smem_optin)) {
      LaunchArgs wa = make_args(dy, w, nullptr, workspace, t, stream, slot, opt);
      e = phase_stack_launch(g, wa, stk.st, workspace, slot->info);
      if (e == cudaSuccess) e = tc_launch(stk.fg, da, slot->info);
      if (e == cudaSuccess) {
        if (opt) opt->selected = GCONV_KERNEL_IGEMM_TC;
        return finish(slot, da, opt);
      }
      if (e != cudaErrorNotSupported) return fail(GCONV_ERR_CUDA, "launch failed: %s", cudaGetErrorString(e));
    }
  }
  if (per_phase) {
    // per stride phase: its sub-filter (transposed channels) into the
    // workspace, then its stride-1 forward correlation of dy on the
    // tensor-core kernel, whose epilogue writes the phase's outputs straight
    // to their dx positions.  Where that kernel cannot take the call (a
    // forced other kernel, pointers it cannot copy from), the correlation
    // goes to the phase buffer and a scatter kernel places it.
    uint8_t* wt = static_cast<uint8_t*>(workspace);
    uint8_t* pb = wt + align256(g.w_elems() * es);
    LaunchArgs a = make_args(dy, w, nullptr, dx, t, stream, slot, opt);
    for (int rd = 0; rd < g.sD; ++rd)
      for (int rh = 0; rh < g.sH; ++rh)
        for (int rw = 0; rw < g.sW; ++rw) {
          Phase3D ph;
          if (!phase_3d(g, rd, rh, rw, &ph)) return fail(GCONV_ERR_UNSUPPORTED, "stride phase not decomposable");
          PhaseScatter ps{};
          ps.N = g.N;
          ps.C = g.C();
          const int I3[3] = {g.D, g.H, g.W}, s3[3] = {g.sD, g.sH, g.sW}, r3[3] = {rd, rh, rw};
          for (int i = 0; i < 3; ++i) {
            ps.in[i] = I3[i], ps.s[i] = s3[i], ps.r[i] = r3[i];
            ps.n[i] = ph.d[i].n, ps.o[i] = ph.d[i].out, ps.off[i] = ph.d[i].off;
          }
          ps.empty = ph.empty ? 1 : 0;
          if (ps.n[0] == 0 || ps.n[1] == 0 || ps.n[2] == 0) continue;  // no dx positions in this phase
          if (!ph.empty) {
            PhaseTaps pt{};
            for (int i = 0; i < 3; ++i) {
              pt.L[i] = ph.d[i].L;
              for (int j = 0; j < ph.d[i].L; ++j) pt.t[i][j] = ph.d[i].t[j];
            }
            LaunchArgs wa = make_args(dy, w, nullptr, wt, t, stream, slot, opt);
            e = phase_weight_launch(g, wa, pt, wt, slot->info);
            if (e != cudaSuccess) return fail(GCONV_ERR_CUDA, "launch failed: %s", cudaGetErrorString(e));
            LaunchArgs da = make_args(dy, wt, nullptr, dx, t, stream, slot, opt);
            da.omap.on = 1;
            for (int i = 0; i < 3; ++i) {
              da.omap.scale[i] = s3[i];
              da.omap.add[i] = r3[i] - s3[i] * ph.d[i].off;
              da.omap.lo[i] = ph.d[i].off;
              da.omap.hi[i] = ph.d[i].off + ph.d[i].n;
              da.omap.ext[i] = I3[i];
            }
            if ((forced == 0 || forced == GCONV_KERNEL_IGEMM_TC) &&
                tc_supported(ph.fg, t, &da, slot->info.num_sms, slot->info.max_smem_optin)) {
              e = tc_launch(ph.fg, da, slot->info);
              if (e == cudaSuccess) {
                if (opt) opt->selected = GCONV_KERNEL_IGEMM_TC;
                continue;  // dx positions of this phase written
              }
              if (e != cudaErrorNotSupported) return fail(GCONV_ERR_CUDA, "launch failed: %s", cudaGetErrorString(e));
            }
            LaunchArgs fa = make_args(dy, wt, nullptr, pb, t, stream, slot, opt);
            s = launch_forward(ph.fg, fa, slot->info, forced, opt ? &opt->selected : nullptr);
            if (s != GCONV_OK) return s;
          }
          e = phase_scatter_launch(ps, pb, dx, a, slot->info);
          if (e != cudaSuccess) return fail(GCONV_ERR_CUDA, "launch failed: %s", cudaGetErrorString(e));
        }
    return finish(slot, a, opt);
  }
  if (forced != 0 && forced != GCONV_KERNEL_BWD_DATA_DIRECT)
    return fail(GCONV_ERR_UNSUPPORTED, "kernel %d cannot run this problem's stride phases", forced);
  LaunchArgs a = make_args(dy, w, nullptr, dx, t, stream, slot, opt);
  e = bwd_data_direct_launch(g, a, slot->info);
  if (e != cudaSuccess) return fail(GCONV_ERR_CUDA, "launch failed: %s", cudaGetErrorString(e));
  if (opt) opt->selected = GCONV_KERNEL_BWD_DATA_DIRECT;
  return finish(slot, a, opt);
}

gconv_status grouped_conv_bwd_data(const void* dy, const void* w, void* dx, const gconv_problem* p, gconv_dtype dt,
                                   void* workspace, int64_t workspace_bytes, struct CUstream_st* stream) {
  return grouped_conv_bwd_data_ex(dy, w, dx, p, dt, workspace, workspace_bytes, stream, nullptr);
}

gconv_status grouped_conv_bwd_data_route(const gconv_problem* p, gconv_dtype dt, int32_t* route, int32_t* launches) {
  Geometry g;
  gconv_status s = validate(p, &g);
  if (s != GCONV_OK) return s;
  if (dt != GCONV_F32 && dt != GCONV_F16 && dt != GCONV_BF16) return fail(GCONV_ERR_UNSUPPORTED, "unknown dtype %d", (int)dt);
  if (route == nullptr) return fail(GCONV_ERR_INVALID_ARG, "route pointer is NULL");
  Geometry f;
  int r = 0, n = 1;
  if (bwd_as_forward(g, &f)) {
    r = 1, n = 2;
  } else if (Stacked stk; stacked_route(g, (DType)dt, &stk)) {
    r = 2, n = 2;  // stacked sub-filters, one tensor-core launch
  } else if (phase_route(g, (DType)dt, nullptr)) {
    r = 2, n = 0;
    for (int rd = 0; rd < g.sD; ++rd)
      for (int rh = 0; rh < g.sH; ++rh)
        for (int rw = 0; rw < g.sW; ++rw) {
          Phase3D ph;
          phase_3d(g, rd, rh, rw, &ph);
          if (ph.d[0].n == 0 || ph.d[1].n == 0 || ph.d[2].n == 0) continue;
          n += ph.empty ? 1 : 2;  // zeros; or sub-filter + forward written into dx
        }
  }
  *route = r;
  if (launches) *launches = n;
  return GCONV_OK;
}

gconv_status grouped_conv_bwd_weight_workspace_size(const gconv_problem* p, gconv_dtype dt, int64_t* bytes) {
  Geometry g;
  gconv_status s = validate(p, &g);
  if (s != GCONV_OK) return s;
  if (dt != GCONV_F32 && dt != GCONV_F16 && dt != GCONV_BF16) return fail(GCONV_ERR_UNSUPPORTED, "unknown dtype %d", (int)dt);
  if (bytes == nullptr) return fail(GCONV_ERR_INVALID_ARG, "bytes pointer is NULL");
  *bytes = bwd_weight_workspace_bytes(g, (DType)dt);
  return GCONV_OK;
}

gconv_status grouped_conv_bwd_weight_ex(const void* x, const void* dy, void* dw, const gconv_problem* p,
                                        gconv_dtype dt, void* workspace, int64_t workspace_bytes,
                                        struct CUstream_st* stream, gconv_options* opt) {
  Geometry g;
  gconv_status s = validate(p, &g);
  if (s != GCONV_OK) return s;
  if (dt != GCONV_F32 && dt != GCONV_F16 && dt != GCONV_BF16) return fail(GCONV_ERR_UNSUPPORTED, "unknown dtype %d", (int)dt);
  if (x == nullptr || dy == nullptr || dw == nullptr) return fail(GCONV_ERR_INVALID_ARG, "x, dy and dw must not be NULL");
  const int forced = opt ? opt->force_kernel : 0;
  if (forced != 0 && forced != GCONV_KERNEL_BWD_WEIGHT && forced != GCONV_KERNEL_IGEMM_TC)
    return fail(GCONV_ERR_UNSUPPORTED, "kernel %d does not compute backward weight", forced);
  const DType t = (DType)dt;
  if (forced == GCONV_KERNEL_IGEMM_TC && !bwd_weight_tc_supported(g, t))
    return fail(GCONV_ERR_UNSUPPORTED, "tensor-core backward weight cannot run this problem");
  const int es = dtype_bytes(t);
  const int64_t dwb = g.w_elems() * es, xb = g.x_elems() * es, dyb = g.y_elems() * es;
  const int64_t need = bwd_weight_workspace_bytes(g, t);
  if (workspace == nullptr || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 15))
    return fail(GCONV_ERR_INVALID_ARG, "workspace must be 16-byte aligned and hold %lld bytes", (long long)need);
  if (overlaps(dw, dwb, x, xb) || overlaps(dw, dwb, dy, dyb) || overlaps(dw, dwb, workspace, need))
    return fail(GCONV_ERR_INVALID_ARG, "dw overlaps an input buffer or the workspace");
  if (overlaps(workspace, need, x, xb) || overlaps(workspace, need, dy, dyb))
    return fail(GCONV_ERR_INVALID_ARG, "the workspace overlaps x or dy");

  DevSlot* slot = nullptr;
  cudaError_t e = device_slot(&slot);
  if (e != cudaSuccess) return fail(GCONV_ERR_CUDA, "device query failed: %s", cudaGetErrorString(e));
  LaunchArgs a = make_args(x, dy, nullptr, dw, t, stream, slot, opt);
  // Tensor-core route where the shape allows (it declines, before launching
  // anything, when x or dy is not 16-byte aligned or its plan does not fit
  // the device); the FFMA route otherwise or when forced.
  int kernel = GCONV_KERNEL_BWD_WEIGHT;
  e = cudaErrorNotSupported;
  if (forced != GCONV_KERNEL_BWD_WEIGHT && bwd_weight_tc_supported(g, t)) {
    e = bwd_weight_tc_launch(g, a, workspace, slot->info);
    if (e == cudaSuccess) kernel = GCONV_KERNEL_IGEMM_TC;
    else if (e == cudaErrorNotSupported && forced == GCONV_KERNEL_IGEMM_TC)
      return fail(GCONV_ERR_UNSUPPORTED, "tensor-core backward weight needs 16-byte aligned x and dy");
  }
  if (e == cudaErrorNotSupported) e = bwd_weight_launch(g, a, workspace, slot->info);
  if (e != cudaSuccess) return fail(GCONV_ERR_CUDA, "launch failed: %s", cudaGetErrorString(e));
  if (opt) opt->selected = kernel;
  return finish(slot, a, opt);
}

gconv_status grouped_conv_bwd_weight(const void* x, const void* dy, void* dw, const gconv_problem* p, gconv_dtype dt,
                                     void* workspace, int64_t workspace_bytes, struct CUstream_st* stream) {
  return grouped_conv_bwd_weight_ex(x, dy, dw, p, dt, workspace, workspace_bytes, stream, nullptr);
}

gconv_status grouped_conv_fwd_dw_pw_ex(const void* x, const void* w_dw, const void* b_dw, const void* w_pw,
                                       const void* b_pw, void* y, const gconv_problem* p, int32_t K, int32_t act,
                                       gconv_dtype dt, struct CUstream_st* stream, gconv_options* opt) {
  Geometry g;
  gconv_status s = validate(p, &g);
  if (s != GCONV_OK) return s;
  if (dt != GCONV_F16 && dt != GCONV_BF16) return fail(GCONV_ERR_UNSUPPORTED, "the fused block takes f16 or bf16");
  if (x == nullptr || w_dw == nullptr || w_pw == nullptr || y == nullptr)
    return fail(GCONV_ERR_INVALID_ARG, "x, w_dw, w_pw and y must not be NULL");
  if (K < 1) return fail(GCONV_ERR_INVALID_ARG, "K must be positive");
  if (act < 0 || act > 2) return fail(GCONV_ERR_INVALID_ARG, "act must be 0, 1 or 2");
  if (opt && opt->force_kernel != 0 && opt->force_kernel != GCONV_KERNEL_DW_PW)
    return fail(GCONV_ERR_UNSUPPORTED, "kernel %d does not compute the fused block", opt->force_kernel);
  const DType t = (DType)dt;
  if (!dw_pw_supported(g, t, K, act))
    return fail(GCONV_ERR_UNSUPPORTED, "the fused block takes 2D depthwise 3x3 (dilation 1, stride 1 or 2), "
                "C %% 16 == 0 up to 256, K %% 8 == 0 up to 256");
  const int es = dtype_bytes(t);
  const int64_t yb = g.N * (int64_t)g.Ho * g.Wo * K * es, xb = g.x_elems() * es;
  if (overlaps(y, yb, x, xb) || overlaps(y, yb, w_dw, g.w_elems() * es) ||
      overlaps(y, yb, w_pw, (int64_t)K * g.C() * es) || (b_dw && overlaps(y, yb, b_dw, (int64_t)g.C() * es)) ||
      (b_pw && overlaps(y, yb, b_pw, (int64_t)K * es)))
    return fail(GCONV_ERR_INVALID_ARG, "y overlaps an input");
  DevSlot* slot = nullptr;
  cudaError_t e = device_slot(&slot);
  if (e != cudaSuccess) return fail(GCONV_ERR_CUDA, "device query failed: %s", cudaGetErrorString(e));
  LaunchArgs a = make_args(x, w_dw, b_dw, y, t, stream, slot, opt);
  e = dw_pw_launch(g, a, w_pw, b_pw, K, act, slot->info);
  if (e == cudaErrorNotSupported)
    return fail(GCONV_ERR_UNSUPPORTED, "the fused block needs 16-byte aligned x, y and w_pw, and shared memory "
                "for its tiles");
  if (e != cudaSuccess) return fail(GCONV_ERR_CUDA, "launch failed: %s", cudaGetErrorString(e));
  if (opt) opt->selected = GCONV_KERNEL_DW_PW;
  return finish(slot, a, opt);
}

gconv_status grouped_conv_fwd_dw_pw(const void* x, const void* w_dw, const void* b_dw, const void* w_pw,
                                    const void* b_pw, void* y, const gconv_problem* p, int32_t K, int32_t act,
                                    gconv_dtype dt, struct CUstream_st* stream) {
  return grouped_conv_fwd_dw_pw_ex(x, w_dw, b_dw, w_pw, b_pw, y, p, K, act, dt, stream, nullptr);
}

gconv_status grouped_conv_fwd_dw_pw_supported(const gconv_problem* p, int32_t K, int32_t act, gconv_dtype dt,
                                              int32_t* ok) {
  Geometry g;
  gconv_status s = validate(p, &g);
  if (s != GCONV_OK) return s;
  if (ok == nullptr) return fail(GCONV_ERR_INVALID_ARG, "ok pointer is NULL");
  *ok = (dt == GCONV_F16 || dt == GCONV_BF16) && act >= 0 && act <= 2 && dw_pw_supported(g, (DType)dt, K, act);
  return GCONV_OK;
}

gconv_status grouped_conv_fwd(const void* x, const void* w, const void* bias, void* y, const gconv_problem* p,
                              gconv_dtype dt, struct CUstream_st* stream) {
  return grouped_conv_fwd_ex(x, w, bias, y, p, dt, stream, nullptr);
}

gconv_status gconv_epilogue_apply(const float* acc, const void* bias, void* y, int64_t rows, int32_t cols,
                                  gconv_dtype dt, struct CUstream_st* stream) {
  if (acc == nullptr || y == nullptr) return fail(GCONV_ERR_INVALID_ARG, "acc and y must not be NULL");
  if (rows < 0 || cols < 1) return fail(GCONV_ERR_INVALID_ARG, "rows must be >= 0 and cols >= 1");
  if (dt != GCONV_F32 && dt != GCONV_F16 && dt != GCONV_BF16) return fail(GCONV_ERR_UNSUPPORTED, "unknown dtype %d", (int)dt);
  cudaError_t e = epilogue_launch(acc, bias, y, rows, cols, (DType)dt, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(GCONV_ERR_CUDA, "launch failed: %s", cudaGetErrorString(e));
  return GCONV_OK;
}

gconv_status gconv_device_status(struct CUstream_st* stream, int32_t* code, int32_t* where) {
  DevSlot* slot = nullptr;
  cudaError_t e = device_slot(&slot);
  if (e != cudaSuccess) return fail(GCONV_ERR_CUDA, "device query failed: %s", cudaGetErrorString(e));
  return read_and_clear_status(slot, reinterpret_cast<cudaStream_t>(stream), code, where);
}

}  // extern "C"
