/*
 * gconv.h -- C ABI of the GB300 grouped-convolution library: the forward
 * pass, backward data and backward weight (grouped_conv_bwd_data and
 * grouped_conv_bwd_weight, further below).
 *
 * The main operation is the grouped convolution forward pass (groups > 1,
 * including depthwise groups == C), 2D and 3D, with optional bias, stride,
 * padding and dilation:
 *
 *   y[n, od, oh, ow, g, k] = sum_{z,yy,xx} sum_{cg < Cg}
 *        x[n, od*sD - pD + z*dD, oh*sH - pH + yy*dH, ow*sW - pW + xx*dW, g, cg]
 *      * w[g, k, z, yy, xx, cg]  (+ bias[g*Kg + k])
 *
 * with Cg = C/G, Kg = K/G and zero padding outside the input.  Passages that
 * define it:
 *   - rocm-libraries PR #10064 (Rocke grouped implicit-GEMM conv), Technical
 *     Details: input channel c = g*Cg + c_in_group, weight channel extent Cg,
 *     output channel k_out = g*Kg + n, C and K divisible by G.
 *   - CK "Grouped Convolution -- Python Examples", Runner argument contract:
 *     forward input X in NHWGC, weight W in GKYXC.
 *   - CK "Grouped Convolution Tile Engine", Problem Registry: the problem
 *     record N, C, K, G, Hi, Wi[, Di], Y, X[, Z], stride_*, pad_*, dilation_*.
 *   - TileOps PR #1568 review, Code Review: bias and no-bias forward ops.
 * Readings where the pages are silent: cross-correlation (no kernel flip);
 * output extent O = floor((I + 2p - d*(k-1) - 1)/s) + 1 with symmetric zero
 * padding; output layout channels-last [N, (Do), Ho, Wo, G, Kg]; bias in the
 * tensors' dtype, added in fp32 before one round-to-nearest-even cast.
 *
 * Every function is thread-safe.  Device functions are asynchronous on the
 * caller's stream unless stated otherwise.  A device's first call only reads
 * device attributes and a symbol address (no allocation, copy or
 * synchronisation), so it may also be made inside a stream capture.
 *
 * Status word: each device has one status word that every call on that
 * device shares, whatever its stream.  A kernel whose bounded wait expires
 * writes it (the first writer wins); gconv_device_status and debug mode read
 * and clear it.  With several streams in flight, a timeout it reports may
 * therefore come from another call on the same device.
 */
#ifndef GCONV_H_
#define GCONV_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The CUDA runtime's cudaStream_t is `struct CUstream_st *`; NULL is the
 * legacy default stream. */
struct CUstream_st;

typedef enum gconv_status {
  GCONV_OK = 0,
  GCONV_ERR_INVALID_ARG = 1, /* malformed problem or pointer; nothing launched      */
  GCONV_ERR_UNSUPPORTED = 2, /* well-formed but not handled (dtype, forced kernel)   */
  GCONV_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed                    */
  GCONV_ERR_TIMEOUT = 4      /* a bounded in-kernel wait expired (debug mode only)   */
} gconv_status;

typedef enum gconv_dtype {
  GCONV_F32 = 0,  /* float32 storage, fp32 accumulation, FFMA only (no TF32) */
  GCONV_F16 = 1,  /* IEEE binary16 storage, fp32 accumulation                */
  GCONV_BF16 = 2  /* bfloat16 storage, fp32 accumulation                     */
} gconv_dtype;

/*
 * Problem record.  All extents are element counts.  Spatial arrays are
 * ordered outer to inner: [0] = depth (D / Z), [1] = height (H / Y),
 * [2] = width (W / X).  A 2D problem sets ndim = 2 and in[0] = ker[0] =
 * stride[0] = dil[0] = 1, pad[0] = 0.  Padding is symmetric per dimension.
 * Layout: 88 bytes, naturally aligned, no implicit padding.
 */
typedef struct gconv_problem {
  int32_t ndim;      /* 2 or 3                                               */
  int32_t reserved;  /* must be 0                                            */
  int64_t N;         /* batch, >= 1                                          */
  int32_t G;         /* groups, >= 1                                         */
  int32_t C;         /* input channels, C % G == 0                           */
  int32_t K;         /* output channels, K % G == 0                          */
  int32_t in[3];     /* input extents D, H, W  (>= 1)                        */
  int32_t ker[3];    /* filter extents Z, Y, X (>= 1)                        */
  int32_t stride[3]; /* >= 1                                                 */
  int32_t pad[3];    /* >= 0, applied on both sides                          */
  int32_t dil[3];    /* >= 1                                                 */
} gconv_problem;

/* Kernels the selector can pick (for options.force_kernel / options.selected). */
typedef enum gconv_kernel {
  GCONV_KERNEL_AUTO = 0,
  GCONV_KERNEL_DIRECT_DW = 1,      /* Ka: TMA-staged depthwise direct kernel        */
  GCONV_KERNEL_DIRECT_GENERIC = 2, /* direct kernel for any shape/dtype/alignment   */
  GCONV_KERNEL_IGEMM_TC = 3,       /* Kb: tcgen05/TMEM grouped implicit GEMM        */
  GCONV_KERNEL_BWD_DATA_DIRECT = 4, /* backward data: direct gather kernel          */
  GCONV_KERNEL_BWD_WEIGHT = 5,      /* backward weight: split fp32 partials + reduce */
  GCONV_KERNEL_DW_PW = 6            /* fused depthwise + activation + 1x1 projection */
} gconv_kernel;

/* Options of grouped_conv_fwd_ex.  Zero-initialise, then set what you need. */
typedef struct gconv_options {
  int32_t force_kernel;  /* gconv_kernel; AUTO (0) lets the selector choose        */
  int32_t debug;         /* 1: synchronise the stream after the launch and turn a
                            device-side status (timeout) into the return value   */
  int64_t wait_limit_ns; /* bound on each in-kernel wait; 0 = 2 s                  */
  int32_t test_flags;    /* bit 0: withhold the first input copy of CTA 0 so its
                            first wait cannot complete (timeout-path test);
                            bit 1: backward data by stride phases launches one
                            correlation per phase instead of one stacked
                            launch (tests of that placement)                   */
  int32_t selected;      /* out: the gconv_kernel that was launched               */
  int32_t tile[8];       /* tuning overrides, 0 = automatic.
                            Depthwise kernel: [0] TH, [1] TW, [2] WB (row-blocked
                            form) / 2 = first tile's input in two copies (column
                            form), [3] stages,
                            [4] CTAs per SM, [5] FMA form (row-blocked form:
                            1 = widen + fp32 FMA, 2 = mixed f16/bf16 FMA,
                            3 = widen + packed fp32x2 FMA; column form: 1 =
                            split 16-bit operands / scalar fp32, 2 = packed
                            16-bit pairs with 4 channels per thread, 3 = widen
                            + packed fp32x2 FMA, 4 = packed 16-bit pairs with 8
                            channels per thread, 0 = 2 for 16-bit storage and
                            1 for fp32), [6] form (1 =
                            row-blocked, 2 = direct loads, 3 = column form; the
                            automatic choice is the column form when the depth
                            filter is 1, else the row-blocked form).
                            Tensor-core kernel: [0] TH, [1] most accumulator
                            buffers (2-4; default as many as tensor memory
                            holds), [2] M tiles per CTA,
                            [3] stages, [4] partial accumulators, [5] 2 = one
                            copy of the tile per column shift, so every tap's
                            A operand starts on an 8-row boundary (default:
                            shifted starts), [6] 1 = force
                            16-byte chunk planes, [7] extra shared memory (KB),
                            negative: stage the tile's output box in shared
                            memory and write it with TMA tensor stores
                            (default: store from registers). */
  int32_t serial_launch; /* 0: the kernel is launched as a programmatic dependent
                            launch: its CTAs may start, and set up barriers,
                            tensor memory and tables, while the previous kernel
                            in the stream is still running; every access to
                            global memory waits until that kernel has completed
                            and its writes are visible, so stream order holds
                            for x, w, bias and y.  1: plain launch (the kernel
                            starts only after the previous one has finished). */
} gconv_options;

/*
 * grouped_conv_fwd -- y = grouped_conv(x, w) (+ bias).
 *   x    device, [N, (D), H, W, G, Cg] packed, dtype dt          (read only)
 *   w    device, [G, Kg, (Z), Y, X, Cg] packed, dtype dt         (read only)
 *   bias device, [G*Kg] in dtype dt, or NULL for no bias           (read only)
 *   y    device, [N, (Do), Ho, Wo, G, Kg] packed, dtype dt (written; must not
 *        overlap x, w or bias)
 *   p    host pointer to the problem record (read during the call only)
 *   stream  the CUDA stream the kernel is enqueued on
 * Ownership: the caller owns every buffer and the stream.  The library
 * allocates no device memory, keeps no per-call state and copies nothing
 * between host and device.  The launch is asynchronous; buffers must stay
 * valid until the stream reaches it.
 * Every well-formed problem runs: the selector takes a specialised kernel only
 * when its planner finds a launch plan on this device, and otherwise (also
 * when the device's own limits turn a plan down at launch) the generic kernel.
 * Errors: GCONV_ERR_INVALID_ARG for a malformed problem (C or K not divisible
 * by G, non-positive extents, empty output, 2D fields not neutral), NULL
 * x/w/y/p, or y overlapping an input; GCONV_ERR_UNSUPPORTED for an unknown
 * dtype; GCONV_ERR_CUDA if the launch fails.  Nothing is launched on error;
 * gconv_last_error() then describes the reason.
 */
gconv_status grouped_conv_fwd(const void *x, const void *w, const void *bias, void *y,
                              const gconv_problem *p, gconv_dtype dt, struct CUstream_st *stream);

/*
 * grouped_conv_fwd_ex -- grouped_conv_fwd with options (kernel override,
 * debug synchronisation, wait bound, timeout-path test).  `opt` may be NULL.
 * Same arguments, ownership and errors as grouped_conv_fwd, plus:
 * GCONV_ERR_UNSUPPORTED when a forced kernel cannot run this problem, and,
 * with opt->debug set, GCONV_ERR_TIMEOUT when a bounded in-kernel wait expired
 * (the kernel then returned early and y is incomplete).  With debug set the
 * call blocks until the stream has drained.
 */
gconv_status grouped_conv_fwd_ex(const void *x, const void *w, const void *bias, void *y,
                                 const gconv_problem *p, gconv_dtype dt, struct CUstream_st *stream,
                                 gconv_options *opt);

/*
 * grouped_conv_bwd_data -- dx, the gradient of y = grouped_conv(x, w) with
 * respect to x, given dy = the gradient with respect to y (the adjoint of the
 * forward map in x; the backward-data variant of the CK grouped-convolution
 * tile engine, whose runner takes dY and W):
 *   dx[n, i, g, c] = sum over (o, t, k) with i = o*s - p + t*d in every
 *                    dimension of dy[n, o, g, k] * w[g, k, t, c]
 *   dy   device, [N, (Do), Ho, Wo, G, Kg] packed, dtype dt  (the forward output
 *        layout; read only)
 *   w    device, [G, Kg, (Z), Y, X, Cg] packed, dtype dt     (read only)
 *   dx   device, [N, (D), H, W, G, Cg] packed, dtype dt      (written; must not
 *        overlap dy, w or the workspace)
 *   p    the forward problem (in[] = dx's extents; Do, Ho, Wo follow from it)
 *   workspace  device scratch of at least
 *        grouped_conv_bwd_data_workspace_size() bytes, 16-byte aligned; NULL
 *        when that size is 0.  Owned by the caller; the call uses it until the
 *        stream passes the launch.
 * Three routes (grouped_conv_bwd_data_route tells which):
 *   1. stride 1 with pad <= dil*(k-1) in every dimension: a forward
 *      convolution of dy with per-group transposed, flipped weights (written
 *      into the workspace) and padding dil*(k-1) - pad, on the forward
 *      kernels;
 *   2. a stride above 1 with grouped channels (not depthwise) in f16/bf16,
 *      when the stride phases plan on the tensor-core kernel: dx is cut
 *      into its stride phases (positions s*i + r per dimension); phase r is
 *      a stride-1 forward correlation of dy with the sub-filter of taps t
 *      that reach it (r + p - t*d divisible by s).  All phases run as one
 *      tensor-core launch: the sub-filters are stacked as output channels
 *      (phase, channel) of one filter over the union of their offsets, and
 *      the epilogue writes each (phase, channel) output to its dx position
 *      (phases with no taps come out as zeros).  Where that launch does not
 *      plan (Cg not a multiple of 16, too many stacked channels) each
 *      phase runs on its own,
 *      written straight into dx; a phase the tensor-core kernel cannot take
 *      (a forced other kernel, dy or dx not 16-byte aligned) goes through a
 *      buffer in the workspace and a copy to its dx positions instead;
 *   0. otherwise a direct gather kernel, which needs no workspace.
 * fp32 accumulation, one round-to-nearest-even cast.  Asynchronous on
 * `stream`.
 * Errors: as grouped_conv_fwd, plus GCONV_ERR_INVALID_ARG for a workspace that
 * is missing, too small or misaligned.
 */
gconv_status grouped_conv_bwd_data(const void *dy, const void *w, void *dx, const gconv_problem *p,
                                   gconv_dtype dt, void *workspace, int64_t workspace_bytes,
                                   struct CUstream_st *stream);

/*
 * grouped_conv_bwd_data_ex -- grouped_conv_bwd_data with options.
 * opt->force_kernel: GCONV_KERNEL_BWD_DATA_DIRECT forces the direct gather
 * kernel; GCONV_KERNEL_DIRECT_DW / _DIRECT_GENERIC / _IGEMM_TC force the
 * forward kernel of routes 1 and 2 (GCONV_ERR_UNSUPPORTED for a problem of
 * route 0, or when the forced kernel cannot run a phase).  opt->selected
 * reports the kernel used (for route 2, that of the last phase).
 * Other fields as for grouped_conv_fwd_ex.
 */
gconv_status grouped_conv_bwd_data_ex(const void *dy, const void *w, void *dx, const gconv_problem *p,
                                      gconv_dtype dt, void *workspace, int64_t workspace_bytes,
                                      struct CUstream_st *stream, gconv_options *opt);

/*
 * grouped_conv_bwd_data_route -- which route grouped_conv_bwd_data takes for
 * (p, dt) without a forced kernel: *route = 0 (direct gather), 1 (stride 1,
 * transposed flipped weights) or 2 (stride phases), and, if `launches` is
 * not NULL, how many kernels the call launches with 16-byte aligned
 * buffers (route 2: two for the stacked launch; else two per phase with
 * taps and one per phase without, and a phase placed through the workspace
 * buffer adds one).  Host only, no GPU
 * needed; depends on the problem only.
 */
gconv_status grouped_conv_bwd_data_route(const gconv_problem *p, gconv_dtype dt, int32_t *route, int32_t *launches);

/*
 * grouped_conv_bwd_data_workspace_size -- device workspace bytes that
 * grouped_conv_bwd_data needs for problem p in dtype dt (0 when none).  Host
 * only.  GCONV_ERR_INVALID_ARG for a malformed problem or a NULL `bytes`.
 */
gconv_status grouped_conv_bwd_data_workspace_size(const gconv_problem *p, gconv_dtype dt, int64_t *bytes);

/*
 * grouped_conv_bwd_weight -- dw, the gradient of y = grouped_conv(x, w) with
 * respect to w, given x and dy = the gradient with respect to y (the
 * backward-weight variant of the CK grouped-convolution tile engine, whose
 * runner takes X and dY and whose two_stage option reduces through an fp32
 * workspace -- "Grouped Convolution -- Python Examples", Examples and
 * Config-options harness):
 *   dw[g, k, z, yy, xx, c] = sum over (n, od, oh, ow) of dy[n, od, oh, ow, g, k]
 *        * x[n, od*sD - pD + z*dD, oh*sH - pH + yy*dH, ow*sW - pW + xx*dW, g, c]
 *   x    device, [N, (D), H, W, G, Cg] packed, dtype dt      (read only)
 *   dy   device, [N, (Do), Ho, Wo, G, Kg] packed, dtype dt  (read only)
 *   dw   device, [G, Kg, (Z), Y, X, Cg] packed, dtype dt     (written; must not
 *        overlap x, dy or the workspace)
 *   p    the forward problem
 *   workspace  device scratch of at least
 *        grouped_conv_bwd_weight_workspace_size() bytes, 16-byte aligned,
 *        owned by the caller, used until the stream passes the call.
 * Two stages: the sum over output pixels is cut into a fixed number of
 * equal runs whose fp32 partials land in the workspace, then one kernel adds
 * the partials in run order and rounds once (round-to-nearest-even).  The
 * result is deterministic: it depends on the problem only, not on the device
 * or on timing.  Asynchronous on `stream`; two launches.
 * Errors: as grouped_conv_fwd, plus GCONV_ERR_INVALID_ARG for a workspace
 * that is missing, too small or misaligned.
 */
gconv_status grouped_conv_bwd_weight(const void *x, const void *dy, void *dw, const gconv_problem *p,
                                     gconv_dtype dt, void *workspace, int64_t workspace_bytes,
                                     struct CUstream_st *stream);

/*
 * grouped_conv_bwd_weight_ex -- grouped_conv_bwd_weight with options:
 * opt->selected reports GCONV_KERNEL_BWD_WEIGHT; a force_kernel other than
 * AUTO or GCONV_KERNEL_BWD_WEIGHT returns GCONV_ERR_UNSUPPORTED; debug and
 * the other fields as for grouped_conv_fwd_ex.
 */
gconv_status grouped_conv_bwd_weight_ex(const void *x, const void *dy, void *dw, const gconv_problem *p,
                                        gconv_dtype dt, void *workspace, int64_t workspace_bytes,
                                        struct CUstream_st *stream, gconv_options *opt);

/*
 * grouped_conv_bwd_weight_workspace_size -- device workspace bytes that
 * grouped_conv_bwd_weight needs for problem p in dtype dt (never 0).  Host
 * only, no GPU needed.  GCONV_ERR_INVALID_ARG for a malformed problem or a
 * NULL `bytes`.
 */
gconv_status grouped_conv_bwd_weight_workspace_size(const gconv_problem *p, gconv_dtype dt, int64_t *bytes);

/*
 * grouped_conv_bwd_data_noalloc -- grouped_conv_bwd_data for callers that
 * cannot allocate device memory, nor have it allocated for them, while they
 * run: for example a plugin enqueued on a stream an inference engine owns, or
 * a runtime that reserves all of its memory at start-up and forbids
 * allocation (and the synchronisation an allocation can cause) later.  The
 * pages have no counterpart: this is a library convenience, not a step of the
 * method.
 * Same operation, arguments (minus the workspace), layouts, ownership and
 * errors as grouped_conv_bwd_data.  The scratch that call takes from the
 * caller (the transposed, flipped weights of its stride-1 route) comes here
 * from a fixed array of GCONV_NOALLOC_SCRATCH_BYTES bytes in the library's
 * own static device memory, which every GPU that loads the library holds
 * until the process exits.  Nothing is allocated and nothing is freed.
 *   - A problem whose scratch would exceed GCONV_NOALLOC_SCRATCH_BYTES
 *     runs on the direct gather kernel (which needs none) when it has a
 *     stride above 1, and otherwise returns GCONV_ERR_UNSUPPORTED without
 *     launching anything (grouped_conv_bwd_data_workspace_size gives the
 *     size a problem needs).
 *   - The first call on a device looks up the array's device address (once
 *     per device, with that device current); make that first call before
 *     any stream capture.
 *   - Every call shares the one array and leaves its contents behind; each
 *     call rewrites every byte it reads, so no clearing is needed.  Calls
 *     whose work overlaps on the GPU (other streams, unordered host threads)
 *     race on it: keep them ordered, e.g. on one stream.
 */
#define GCONV_NOALLOC_SCRATCH_BYTES (1 << 20)
gconv_status grouped_conv_bwd_data_noalloc(const void *dy, const void *w, void *dx, const gconv_problem *p,
                                           gconv_dtype dt, struct CUstream_st *stream);

/*
 * grouped_conv_out_shape -- output extents {Do, Ho, Wo} of problem p
 * (Do = 1 for 2D), by O = floor((I + 2p - d*(k-1) - 1)/s) + 1.  Host only,
 * no GPU needed.  GCONV_ERR_INVALID_ARG for a malformed or empty problem.
 */
gconv_status grouped_conv_out_shape(const gconv_problem *p, int32_t out[3]);

/*
 * grouped_conv_select -- which gconv_kernel grouped_conv_fwd would launch for
 * (p, dt) with 16-byte aligned buffers on a GB300 (152 SMs, 227 KB of
 * shared memory per block).  Host only, no GPU needed.
 */
gconv_status grouped_conv_select(const gconv_problem *p, gconv_dtype dt, int32_t *kernel);

/*
 * gconv_epilogue_apply -- runs the fused epilogue (Kc) alone:
 *   y[r, c] = round_to_nearest_even_dt(acc[r, c] + (bias ? float(bias[c]) : 0))
 *   acc  device fp32 [rows, cols];  bias device [cols] in dt or NULL;
 *   y    device [rows, cols] in dt.  Asynchronous on `stream`.
 * The same device code finishes every convolution kernel; this entry point
 * exists so the epilogue can be tested bit-for-bit on its own.
 * Errors: GCONV_ERR_INVALID_ARG (NULL acc/y, rows < 0, cols < 1),
 * GCONV_ERR_UNSUPPORTED (dtype), GCONV_ERR_CUDA.
 */
gconv_status gconv_epilogue_apply(const float *acc, const void *bias, void *y, int64_t rows,
                                  int32_t cols, gconv_dtype dt, struct CUstream_st *stream);

/*
 * gconv_device_status -- synchronises `stream`, then reads and clears the
 * current device's status word that kernels set when a bounded wait expires.
 * *code = 0 (none) or 1 (timeout); *where = the kernel-specific wait site.
 * Returns GCONV_ERR_CUDA if synchronisation or the read fails.
 */
gconv_status gconv_device_status(struct CUstream_st *stream, int32_t *code, int32_t *where);

/* Static description of a status code. */
const char *gconv_status_string(gconv_status s);

/* Human-readable reason for the calling thread's last non-OK status. */
const char *gconv_last_error(void);

/*
 * grouped_conv_fwd_dw_pw -- the tail of a MobileNetV2-style block in one
 * kernel: a depthwise convolution with bias and activation, then a 1x1
 * projection with bias.  The depthwise layer is the pages' MobileNetV2
 * benchmark layer (TileOPs PR #1568, Code Review: the MobileNetV2 depthwise
 * cases); the projection and the activation are its neighbours in that
 * network, and fusing them keeps the intermediate h on chip instead of
 * writing it to HBM and reading it back:
 *   h[n, oh, ow, c] = round(act(sum_{yy,xx} x[n, oh*s - pH + yy, ow*s - pW + xx, c]
 *                              * w_dw[c, 0, yy, xx, 0] + b_dw[c]))
 *   y[n, oh, ow, k] = round(sum_c h[n, oh, ow, c] * w_pw[k, c] + b_pw[k])
 * h is rounded to dt (round to nearest even) exactly as a separate depthwise
 * layer would store it; both sums are fp32.
 *   x     device, [N, H, W, C] packed, dtype dt            (read only)
 *   w_dw  device, [C, 1, 3, 3, 1] (GKYXC with G = C)        (read only)
 *   b_dw  device, [C], or NULL for no depthwise bias
 *   w_pw  device, [K, C] (GKYXC with G = 1, 1x1), 16-byte aligned
 *   b_pw  device, [K], or NULL for no projection bias
 *   y     device, [N, Ho, Wo, K] packed (Ho, Wo from p), written; must not
 *         overlap an input
 *   p     the depthwise problem: 2D, G = C (Cg = Kg = 1), 3x3 filter,
 *         dilation 1, equal H / W strides of 1 or 2, any padding
 *   act   0 none, 1 ReLU (max(v, 0)), 2 ReLU6 (min(max(v, 0), 6)) on h
 * Limits: dt f16 or bf16; C a multiple of 16 up to 256; K a multiple of 8 up
 * to 256; any H and W; x, y and w_pw 16-byte aligned.  Outside them the call
 * returns GCONV_ERR_UNSUPPORTED and launches nothing (run grouped_conv_fwd
 * and the projection separately).  Asynchronous on `stream`; one launch.
 */
gconv_status grouped_conv_fwd_dw_pw(const void *x, const void *w_dw, const void *b_dw, const void *w_pw,
                                    const void *b_pw, void *y, const gconv_problem *p, int32_t K, int32_t act,
                                    gconv_dtype dt, struct CUstream_st *stream);

/* grouped_conv_fwd_dw_pw with options (debug, wait limit, serial launch; opt->selected reports
 * GCONV_KERNEL_DW_PW; force_kernel must be AUTO or GCONV_KERNEL_DW_PW).  Tuning overrides,
 * 0 = automatic: opt->tile[0] channels per depthwise thread (8, or 4 with twice the compute
 * warps), opt->tile[1] / tile[2] the output tile's rows TH / columns TW (TW <= 16,
 * TH * TW <= 128, TH a balanced split of Ho: ceil(Ho / ceil(Ho / TH)) == TH), opt->tile[3]
 * the projection's MMA issuer (1 a dedicated warp, 2 the depthwise warp that completes a
 * tile); a choice that does not fit returns GCONV_ERR_UNSUPPORTED. */
gconv_status grouped_conv_fwd_dw_pw_ex(const void *x, const void *w_dw, const void *b_dw, const void *w_pw,
                                       const void *b_pw, void *y, const gconv_problem *p, int32_t K,
                                       int32_t act, gconv_dtype dt, struct CUstream_st *stream,
                                       gconv_options *opt);

/* Host only, no GPU needed: *ok = 1 when grouped_conv_fwd_dw_pw takes (p, K, act, dt) (its
 * shape limits above; pointer alignment is checked at the call), else 0. */
gconv_status grouped_conv_fwd_dw_pw_supported(const gconv_problem *p, int32_t K, int32_t act, gconv_dtype dt,
                                              int32_t *ok);

#ifdef __cplusplus
}
#endif

#endif /* GCONV_H_ */
