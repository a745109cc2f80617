/*
 * Grouped convolution forward, backward data and backward weight -- CPU
 * oracle (TEST INFRASTRUCTURE ONLY).
 *
 * This file is the slow, obviously-correct reference that the CUDA path is
 * checked against.  Only the test-suite, the smoke check and the benchmark's
 * CPU-baseline leg may build, load or call it; the product never does.  It
 * shares no code, header or table with the CUDA library.
 *
 * What it computes (the plain definition of grouped convolution; the two
 * gradients are defined beside their functions at the end of the file):
 *
 *   y[n, od, oh, ow, g, k] =
 *       sum_{z, yy, xx} sum_{cg < Cg}
 *           x[n, od*sD - pD + z*dD, oh*sH - pH + yy*dH, ow*sW - pW + xx*dW, g, cg]
 *         * w[g, k, z, yy, xx, cg]
 *     + (bias ? bias[g*Kg + k] : 0)
 *
 * with out-of-range input positions contributing zero (zero padding).
 *
 * Sources on the pages:
 *  - rocm-libraries PR #10064 (Rocke grouped implicit-GEMM conv), Technical
 *    Details: the input channel of group g is c = g*Cg + c_in_group, the weight
 *    channel extent is Cg (not C), and the output channel folds as
 *    k_out = g*Kg + n; C and K must be divisible by G.
 *  - CK "Grouped Convolution -- Python Examples", Runner argument contract:
 *    forward input X is NHWGC, weight W is GKYXC.
 *  - CK "Grouped Convolution Tile Engine", Problem Registry: per-dimension
 *    stride_*, pad_* and optional dilation_* fields.
 *  - TileOps PR #1568 review, Code Review: bias and no-bias forward variants.
 *
 * Readings where the pages are silent:
 *  - cross-correlation (the kernel is not flipped), as in the PyTorch
 *    baseline the TileOps review compares against;
 *  - output extent O = floor((I + 2p - d*(k-1) - 1) / s) + 1, symmetric zero
 *    padding per dimension;
 *  - output layout [N, (Do), Ho, Wo, G, Kg] (channels-last, k_out = g*Kg + k);
 *  - bias is added after the sum; everything here is float64.
 *
 * Layouts (all packed, float64): x [N][D][H][W][G][Cg], w [G][Kg][Z][Y][X][Cg],
 * bias [G*Kg] or NULL, y [N][Do][Ho][Wo][G][Kg].  A 2D problem is D = Z = 1,
 * sD = dD = 1, pD = 0.
 */
#include <stddef.h>
#include <stdint.h>

/* Output extent along one dimension; returns <= 0 when nothing fits. */
long oracle_out_extent(long in, long k, long s, long p, long d)
{
    if (s <= 0 || d <= 0 || k <= 0 || in <= 0 || p < 0)
        return 0;
    long span = d * (k - 1) + 1;
    long room = in + 2 * p - span;
    if (room < 0)
        return 0;
    return room / s + 1;
}

/* One output value, summed straight from the definition. */
static double one_output(const double *x, const double *w, const double *bias,
                         long N, long G, long Cg, long Kg,
                         const long in[3], const long ker[3], const long st[3],
                         const long pd[3], const long dl[3],
                         long n, long od, long oh, long ow, long g, long k)
{
    (void)N;
    const long D = in[0], H = in[1], W = in[2];
    const long Z = ker[0], Y = ker[1], X = ker[2];
    const long C = G * Cg;
    double acc = 0.0;
    for (long z = 0; z < Z; ++z) {
        long id = od * st[0] - pd[0] + z * dl[0];
        if (id < 0 || id >= D)
            continue;
        for (long yy = 0; yy < Y; ++yy) {
            long ih = oh * st[1] - pd[1] + yy * dl[1];
            if (ih < 0 || ih >= H)
                continue;
            for (long xx = 0; xx < X; ++xx) {
                long iw = ow * st[2] - pd[2] + xx * dl[2];
                if (iw < 0 || iw >= W)
                    continue;
                const double *xp = x + ((((n * D + id) * H + ih) * W + iw) * C + g * Cg);
                const double *wp = w + ((((g * Kg + k) * Z + z) * Y + yy) * X + xx) * Cg;
                for (long cg = 0; cg < Cg; ++cg)
                    acc += xp[cg] * wp[cg];
            }
        }
    }
    if (bias)
        acc += bias[g * Kg + k];
    return acc;
}

static int unpack(const int32_t *in3, const int32_t *ker3, const int32_t *st3,
                  const int32_t *pd3, const int32_t *dl3, long in[3], long ker[3],
                  long st[3], long pd[3], long dl[3], long out[3])
{
    for (int i = 0; i < 3; ++i) {
        in[i] = in3[i];
        ker[i] = ker3[i];
        st[i] = st3[i];
        pd[i] = pd3[i];
        dl[i] = dl3[i];
        out[i] = oracle_out_extent(in[i], ker[i], st[i], pd[i], dl[i]);
        if (out[i] <= 0)
            return -1;
    }
    return 0;
}

/*
 * Full forward pass.  Returns 0 on success, -1 if the problem is empty or
 * malformed.  Parallel over (n, od, oh) with OpenMP when built with -fopenmp.
 */
int oracle_grouped_conv_fwd(const double *x, const double *w, const double *bias, double *y,
                            long N, long G, long Cg, long Kg,
                            const int32_t *in3, const int32_t *ker3, const int32_t *st3,
                            const int32_t *pd3, const int32_t *dl3)
{
    long in[3], ker[3], st[3], pd[3], dl[3], out[3];
    if (N <= 0 || G <= 0 || Cg <= 0 || Kg <= 0)
        return -1;
    if (unpack(in3, ker3, st3, pd3, dl3, in, ker, st, pd, dl, out))
        return -1;
    const long Do = out[0], Ho = out[1], Wo = out[2];
    const long rows = N * Do * Ho;
#pragma omp parallel for schedule(dynamic, 1)
    for (long r = 0; r < rows; ++r) {
        long n = r / (Do * Ho);
        long od = (r / Ho) % Do;
        long oh = r % Ho;
        for (long ow = 0; ow < Wo; ++ow)
            for (long g = 0; g < G; ++g)
                for (long k = 0; k < Kg; ++k) {
                    long o = (((r * Wo + ow) * G + g) * Kg + k);
                    y[o] = one_output(x, w, bias, N, G, Cg, Kg, in, ker, st, pd, dl,
                                      n, od, oh, ow, g, k);
                }
    }
    return 0;
}

/*
 * Selected outputs only: idx[i] is a flat index into y's [N][Do][Ho][Wo][G][Kg]
 * layout; out[i] receives that output.  Lets large problems be checked on a
 * sample.  Returns 0, or -1 for a malformed problem or an index out of range.
 */
int oracle_grouped_conv_fwd_points(const double *x, const double *w, const double *bias,
                                   long N, long G, long Cg, long Kg,
                                   const int32_t *in3, const int32_t *ker3, const int32_t *st3,
                                   const int32_t *pd3, const int32_t *dl3,
                                   const int64_t *idx, long npts, double *out)
{
    long in[3], ker[3], st[3], pd[3], dl[3], o3[3];
    if (N <= 0 || G <= 0 || Cg <= 0 || Kg <= 0)
        return -1;
    if (unpack(in3, ker3, st3, pd3, dl3, in, ker, st, pd, dl, o3))
        return -1;
    const long Do = o3[0], Ho = o3[1], Wo = o3[2];
    const long total = N * Do * Ho * Wo * G * Kg;
    int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (long i = 0; i < npts; ++i) {
        long f = (long)idx[i];
        if (f < 0 || f >= total) {
            bad = 1;
            continue;
        }
        long k = f % Kg;
        f /= Kg;
        long g = f % G;
        f /= G;
        long ow = f % Wo;
        f /= Wo;
        long oh = f % Ho;
        f /= Ho;
        long od = f % Do;
        long n = f / Do;
        out[i] = one_output(x, w, bias, N, G, Cg, Kg, in, ker, st, pd, dl, n, od, oh, ow, g, k);
    }
    return bad ? -1 : 0;
}

/*
 * Backward data: the gradient with respect to x of a loss whose gradient
 * with respect to y is dy, i.e. the adjoint (transpose) of the forward map in
 * x.  Grouped Convolution Tile Engine and Grouped Convolution -- Python
 * Examples (Examples, Runner argument contract): a backward-data variant
 * takes dY and W.  Written as the forward definition read backwards -- every
 * product dy * w that the forward sum would have formed from input position
 * i is accumulated into dx at i:
 *
 *   dx[n, id, ih, iw, g, cg] += dy[n, od, oh, ow, g, k] * w[g, k, z, yy, xx, cg]
 *     for every (od, oh, ow, k, z, yy, xx) with
 *     id = od*sD - pD + z*dD,  ih = oh*sH - pH + yy*dH,  iw = ow*sW - pW + xx*dW
 *     inside the input; dx starts at zero.
 *
 * Layouts: dy [N][Do][Ho][Wo][G][Kg] (the forward output layout), w as in the
 * forward pass, dx [N][D][H][W][G][Cg] (the forward input layout).  Parallel
 * over (n, g): those slices of dx are disjoint.  Returns 0, or -1 for a
 * malformed or empty problem.
 */
int oracle_grouped_conv_bwd_data(const double *dy, const double *w, double *dx,
                                 long N, long G, long Cg, long Kg,
                                 const int32_t *in3, const int32_t *ker3, const int32_t *st3,
                                 const int32_t *pd3, const int32_t *dl3)
{
    long in[3], ker[3], st[3], pd[3], dl[3], out[3];
    if (N <= 0 || G <= 0 || Cg <= 0 || Kg <= 0)
        return -1;
    if (unpack(in3, ker3, st3, pd3, dl3, in, ker, st, pd, dl, out))
        return -1;
    const long D = in[0], H = in[1], W = in[2];
    const long Z = ker[0], Y = ker[1], X = ker[2];
    const long Do = out[0], Ho = out[1], Wo = out[2];
    const long C = G * Cg, K = G * Kg;
    const long nx = N * D * H * W * C;
    for (long i = 0; i < nx; ++i)
        dx[i] = 0.0;
#pragma omp parallel for schedule(dynamic, 1)
    for (long ng = 0; ng < N * G; ++ng) {
        const long n = ng / G, g = ng % G;
        for (long od = 0; od < Do; ++od)
            for (long oh = 0; oh < Ho; ++oh)
                for (long ow = 0; ow < Wo; ++ow)
                    for (long k = 0; k < Kg; ++k) {
                        const double d = dy[(((n * Do + od) * Ho + oh) * Wo + ow) * K + g * Kg + k];
                        for (long z = 0; z < Z; ++z) {
                            const long id = od * st[0] - pd[0] + z * dl[0];
                            if (id < 0 || id >= D)
                                continue;
                            for (long yy = 0; yy < Y; ++yy) {
                                const long ih = oh * st[1] - pd[1] + yy * dl[1];
                                if (ih < 0 || ih >= H)
                                    continue;
                                for (long xx = 0; xx < X; ++xx) {
                                    const long iw = ow * st[2] - pd[2] + xx * dl[2];
                                    if (iw < 0 || iw >= W)
                                        continue;
                                    double *xp = dx + ((((n * D + id) * H + ih) * W + iw) * C + g * Cg);
                                    const double *wp = w + ((((g * Kg + k) * Z + z) * Y + yy) * X + xx) * Cg;
                                    for (long cg = 0; cg < Cg; ++cg)
                                        xp[cg] += d * wp[cg];
                                }
                            }
                        }
                    }
    }
    return 0;
}

/*
 * Backward weight: the gradient with respect to w of a loss whose gradient
 * with respect to y is dy.  Grouped Convolution Tile Engine and Grouped
 * Convolution -- Python Examples (Examples, Runner argument contract): a
 * backward-weight variant takes X and dY.  Written from the forward
 * definition: each weight multiplies the input values its taps read, so
 *
 *   dw[g, k, z, yy, xx, cg] = sum over (n, od, oh, ow) of
 *       dy[n, od, oh, ow, g, k] * x[n, od*sD - pD + z*dD, oh*sH - pH + yy*dH, ow*sW - pW + xx*dW, g, cg]
 *
 * with out-of-range input positions contributing zero.  Layouts: x as in the
 * forward pass, dy [N][Do][Ho][Wo][G][Kg], dw [G][Kg][Z][Y][X][Cg].  Parallel
 * over (g, k): those slices of dw are disjoint.  Returns 0, or -1 for a
 * malformed or empty problem.
 */
int oracle_grouped_conv_bwd_weight(const double *x, const double *dy, double *dw,
                                   long N, long G, long Cg, long Kg,
                                   const int32_t *in3, const int32_t *ker3, const int32_t *st3,
                                   const int32_t *pd3, const int32_t *dl3)
{
    long in[3], ker[3], st[3], pd[3], dl[3], out[3];
    if (N <= 0 || G <= 0 || Cg <= 0 || Kg <= 0)
        return -1;
    if (unpack(in3, ker3, st3, pd3, dl3, in, ker, st, pd, dl, out))
        return -1;
    const long D = in[0], H = in[1], W = in[2];
    const long Z = ker[0], Y = ker[1], X = ker[2];
    const long Do = out[0], Ho = out[1], Wo = out[2];
    const long C = G * Cg, K = G * Kg;
#pragma omp parallel for schedule(dynamic, 1)
    for (long gk = 0; gk < G * Kg; ++gk) {
        const long g = gk / Kg, k = gk % Kg;
        for (long z = 0; z < Z; ++z)
            for (long yy = 0; yy < Y; ++yy)
                for (long xx = 0; xx < X; ++xx) {
                    double *wp = dw + ((((g * Kg + k) * Z + z) * Y + yy) * X + xx) * Cg;
                    for (long cg = 0; cg < Cg; ++cg)
                        wp[cg] = 0.0;
                    for (long n = 0; n < N; ++n)
                        for (long od = 0; od < Do; ++od) {
                            const long di = od * st[0] - pd[0] + z * dl[0];
                            if (di < 0 || di >= D)
                                continue;
                            for (long oh = 0; oh < Ho; ++oh) {
                                const long hi = oh * st[1] - pd[1] + yy * dl[1];
                                if (hi < 0 || hi >= H)
                                    continue;
                                for (long ow = 0; ow < Wo; ++ow) {
                                    const long wi = ow * st[2] - pd[2] + xx * dl[2];
                                    if (wi < 0 || wi >= W)
                                        continue;
                                    const double dyv = dy[(((n * Do + od) * Ho + oh) * Wo + ow) * K + g * Kg + k];
                                    const double *xp = x + ((((n * D + di) * H + hi) * W + wi) * C + g * Cg);
                                    for (long cg = 0; cg < Cg; ++cg)
                                        wp[cg] += dyv * xp[cg];
                                }
                            }
                        }
                }
    }
    return 0;
}
