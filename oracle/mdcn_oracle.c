/*
 * Double-precision CPU oracle for the modulated deformable convolution
 * (DCNv2) forward pass.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it. It shares no code, header or constant with the CUDA
 * library.
 *
 * Source: "TensorRT plugin walkthrough: modulatedDeformConvPlugin"
 * (trdm.cn/news/524745), the page that describes the operator:
 *   - section 2 (inputs and outputs): tensor shapes and NCHW layout; offset
 *     holds, along its channel axis, the h offset then the w offset of each
 *     sampling point; mask holds one modulation scalar per sampling point;
 *     weight is [Cout, Cin/group, kh, kw]; bias is optional.
 *   - section 3 (attributes): stride, padding, dilation, group,
 *     deformable_group; channels split into contiguous groups.
 *   - section 5 step 1 (deformable im2col): anchor ho*sh - ph, wo*sw - pw;
 *     tap (i, j) samples at anchor + i*dh + dh_off, anchor + j*dw + dw_off;
 *     bilinear sample that is 0 when the point lies outside the open range
 *     (-1, H) x (-1, W); the sample is multiplied by the mask.
 *   - section 5 step 2 (grouped GEMM): per group, m = Cout/group,
 *     n = Ho*Wo, k = Cin/group * kh * kw.
 *   - section 5 step 3: the bias is broadcast-added per output channel.
 *
 * Readings where the page is silent or garbled (each one is pinned by a test):
 *   - offset channel of tap k = i*kw + j in deformable group gd:
 *     dh at gd*2K + 2k, dw at gd*2K + 2k + 1 (K = kh*kw).
 *   - mask channel: gd*K + k.
 *   - input channel c belongs to deformable group c / (Cin/dg) and to
 *     convolution group c / (Cin/group); output channel o to group o / (Cout/group).
 *   - inside the open range, a corner outside the image reads 0, i.e. the
 *     sample is bilinear interpolation of the zero-extended image.
 *   - the mask multiplies the sample as given (no sigmoid inside the op).
 *
 * Every quantity is double; the caller passes inputs already rounded to the
 * run's storage type and widened exactly to double. No blocking, no
 * reordering: for each output element the sum runs over (c_l, i, j) in that
 * order. The column vector of one output pixel (mask * sample for every
 * input channel and tap) is computed once and reused for every output
 * channel; that is the same arithmetic, not a reordering of the sum.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Error codes of the oracle (its own, unrelated to the library's). */
#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1
#define ORACLE_NO_MEMORY 2

/* Bilinear sample of one H x W plane at real position (h, w), section 5 step 1:
 * 0 when h <= -1, h >= H, w <= -1 or w >= W; otherwise the four corners
 * around (h, w) weighted by the fractional parts, a corner outside the image
 * counting as 0. */
static double bilinear_zero(const double* plane, int64_t H, int64_t W, double h, double w)
{
    if (h <= -1.0 || h >= (double)H || w <= -1.0 || w >= (double)W) return 0.0;
    const double h0f = floor(h), w0f = floor(w);
    const int64_t h0 = (int64_t)h0f, w0 = (int64_t)w0f;
    const double lh = h - h0f, lw = w - w0f;
    double v = 0.0;
    for (int dy = 0; dy < 2; ++dy) {
        for (int dx = 0; dx < 2; ++dx) {
            const int64_t y = h0 + dy, xx = w0 + dx;
            if (y < 0 || y >= H || xx < 0 || xx >= W) continue;
            const double wy = dy ? lh : 1.0 - lh;
            const double wx = dx ? lw : 1.0 - lw;
            v += wy * wx * plane[y * W + xx];
        }
    }
    return v;
}

int mdcn_oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Forward pass. Shapes (all NCHW, contiguous):
 *   x      [N, Cin, H, W]
 *   offset [N, 2*dg*kh*kw, Ho, Wo]
 *   mask   [N, dg*kh*kw, Ho, Wo]
 *   weight [Cout, Cin/group, kh, kw]
 *   bias   [Cout] or NULL
 *   out    [N, Cout, Ho, Wo]
 * Only output rows ho in [ho_begin, ho_end) are written (lets a caller time a
 * bounded slice); pass 0, Ho for the whole output. nthreads <= 0 keeps the
 * OpenMP default.
 */
int mdcn_oracle_forward_f64(const double* x, const double* offset, const double* mask,
                            const double* weight, const double* bias, double* out,
                            int64_t N, int64_t Cin, int64_t H, int64_t W,
                            int64_t Cout, int64_t kh, int64_t kw, int64_t Ho, int64_t Wo,
                            int64_t stride_h, int64_t stride_w, int64_t pad_h, int64_t pad_w,
                            int64_t dil_h, int64_t dil_w, int64_t group, int64_t deformable_group,
                            int64_t ho_begin, int64_t ho_end, int nthreads)
{
    if (!x || !offset || !mask || !weight || !out) return ORACLE_BAD_ARG;
    if (N < 1 || Cin < 1 || H < 1 || W < 1 || Cout < 1 || kh < 1 || kw < 1 || Ho < 1 || Wo < 1)
        return ORACLE_BAD_ARG;
    if (stride_h < 1 || stride_w < 1 || dil_h < 1 || dil_w < 1 || pad_h < 0 || pad_w < 0)
        return ORACLE_BAD_ARG;
    if (group < 1 || deformable_group < 1) return ORACLE_BAD_ARG;
    if (Cin % group || Cout % group || Cin % deformable_group) return ORACLE_BAD_ARG;
    if (ho_begin < 0 || ho_end > Ho || ho_begin > ho_end) return ORACLE_BAD_ARG;

    const int64_t K = kh * kw;            /* taps */
    const int64_t Cg = Cin / group;       /* input channels per group */
    const int64_t Og = Cout / group;      /* output channels per group */
    const int64_t Cd = Cin / deformable_group; /* input channels per deformable group */
    const int64_t rows = ho_end - ho_begin;
    const int64_t work = N * rows;
    int failed = 0;

#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif

#pragma omp parallel
    {
        /* column vector of one output pixel: col[c*K + k] = mask * sample */
        double* col = (double*)malloc((size_t)(Cin * K) * sizeof(double));
        if (!col) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t t = 0; t < work; ++t) {
            if (!col) continue;
            const int64_t n = t / rows;
            const int64_t ho = ho_begin + t % rows;
            for (int64_t wo = 0; wo < Wo; ++wo) {
                /* section 5 step 1: deformable im2col with modulation */
                for (int64_t c = 0; c < Cin; ++c) {
                    const int64_t gd = c / Cd;
                    const double* plane = x + (n * Cin + c) * H * W;
                    for (int64_t i = 0; i < kh; ++i) {
                        for (int64_t j = 0; j < kw; ++j) {
                            const int64_t k = i * kw + j;
                            const int64_t och_h = gd * 2 * K + 2 * k;
                            const int64_t och_w = och_h + 1;
                            const int64_t mch = gd * K + k;
                            const double dh = offset[((n * 2 * deformable_group * K + och_h) * Ho + ho) * Wo + wo];
                            const double dw = offset[((n * 2 * deformable_group * K + och_w) * Ho + ho) * Wo + wo];
                            const double m = mask[((n * deformable_group * K + mch) * Ho + ho) * Wo + wo];
                            const double h = (double)(ho * stride_h - pad_h + i * dil_h) + dh;
                            const double w = (double)(wo * stride_w - pad_w + j * dil_w) + dw;
                            col[c * K + k] = m * bilinear_zero(plane, H, W, h, w);
                        }
                    }
                }
                /* section 5 steps 2 and 3: grouped contraction, then bias */
                for (int64_t o = 0; o < Cout; ++o) {
                    const int64_t g = o / Og;
                    double acc = 0.0;
                    for (int64_t cl = 0; cl < Cg; ++cl) {
                        const int64_t c = g * Cg + cl;
                        for (int64_t k = 0; k < K; ++k)
                            acc += weight[(o * Cg + cl) * K + k] * col[c * K + k];
                    }
                    if (bias) acc += bias[o];
                    out[((n * Cout + o) * Ho + ho) * Wo + wo] = acc;
                }
            }
        }
        free(col);
    }
    return failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}

/*
 * Backward pass: the gradients of L = sum(grad_out * out) with respect to x,
 * offset, mask, weight and bias, where out is the forward pass above. The
 * page describes the forward only; the gradient is that of the forward's
 * definition, read as follows (each point is pinned by a test):
 *   - inside the open range (-1, H) x (-1, W) the sample is the bilinear
 *     interpolation of the zero-extended image over the cell whose corner is
 *     (floor h, floor w), so its derivatives are those of that cell's
 *     bilinear polynomial (the one-sided derivative where h or w is an
 *     integer); outside the open range the sample and all of its derivatives
 *     are 0, as the forward's range test gives;
 *   - the cell is an integer decision (floor of the position), and the slope
 *     jumps across a cell edge. With positions_f32 = 0 the position is exact
 *     (double): the gradient of the forward above. With positions_f32 = 1 it
 *     is formed as the kernels form it (the integer anchor plus the offset,
 *     rounded to fp32) before its cell and fractions are taken, so that both
 *     sides take the cell decision in the same precision: a position within
 *     half an fp32 ulp of an edge (e.g. anchor 38 plus offset -1.4e-6) then
 *     lands on the edge and takes the right-hand slope;
 *   - the sample enters the output as weight * mask * sample, so with
 *     G = sum over the group's output channels of weight * grad_out (the
 *     gradient of the modulated column element) the chain rule gives
 *       grad_mask   += G * sample,
 *       grad_offset += G * mask * (d sample / dh, d sample / dw),
 *       grad_x      += G * mask * corner weight   (in-image corners only),
 *       grad_weight += grad_out * mask * sample,
 *       grad_bias    = sum of grad_out over n, ho, wo.
 * Four plain passes, each parallel over an index that owns what it writes:
 * the modulated columns and their gradients per (n, ho); grad_x per (n, c);
 * grad_offset and grad_mask per (n, ho); grad_weight per output channel.
 */

/* Sampling position anchor + offset: exact, or rounded to fp32 as the
 * kernels form it. */
static double position(int64_t anchor, double offset, int f32)
{
    const double v = (double)anchor + offset;
    return f32 ? (double)(float)v : v;
}

/* Corner weights and derivatives of one sampling point, in the cell of
 * (floor h, floor w). inside = 0 outside the open range. */
typedef struct {
    int inside;
    int64_t h0, w0;
    double lh, lw;
} cell_t;

static cell_t cell_of(int64_t H, int64_t W, double h, double w)
{
    cell_t c;
    c.inside = !(h <= -1.0 || h >= (double)H || w <= -1.0 || w >= (double)W);
    const double h0f = floor(h), w0f = floor(w);
    c.h0 = (int64_t)h0f;
    c.w0 = (int64_t)w0f;
    c.lh = h - h0f;
    c.lw = w - w0f;
    return c;
}

static double pixel_or_zero(const double* plane, int64_t H, int64_t W, int64_t y, int64_t xx)
{
    return (y < 0 || y >= H || xx < 0 || xx >= W) ? 0.0 : plane[y * W + xx];
}

/* Sample and its derivatives d/dh, d/dw at one point. */
static void sample_and_slopes(const double* plane, int64_t H, int64_t W, double h, double w,
                              double* v, double* dvdh, double* dvdw)
{
    const cell_t c = cell_of(H, W, h, w);
    *v = 0.0;
    *dvdh = 0.0;
    *dvdw = 0.0;
    if (!c.inside) return;
    for (int dy = 0; dy < 2; ++dy) {
        for (int dx = 0; dx < 2; ++dx) {
            const double X = pixel_or_zero(plane, H, W, c.h0 + dy, c.w0 + dx);
            const double wy = dy ? c.lh : 1.0 - c.lh;
            const double wx = dx ? c.lw : 1.0 - c.lw;
            *v += wy * wx * X;
            *dvdh += (dy ? 1.0 : -1.0) * wx * X;
            *dvdw += (dx ? 1.0 : -1.0) * wy * X;
        }
    }
}

int mdcn_oracle_backward_f64(const double* x, const double* offset, const double* mask,
                             const double* weight, const double* grad_out,
                             double* grad_x, double* grad_offset, double* grad_mask,
                             double* grad_weight, double* grad_bias,
                             int64_t N, int64_t Cin, int64_t H, int64_t W,
                             int64_t Cout, int64_t kh, int64_t kw, int64_t Ho, int64_t Wo,
                             int64_t stride_h, int64_t stride_w, int64_t pad_h, int64_t pad_w,
                             int64_t dil_h, int64_t dil_w, int64_t group, int64_t deformable_group,
                             int positions_f32, int nthreads)
{
    if (!x || !offset || !mask || !weight || !grad_out || !grad_x || !grad_offset || !grad_mask || !grad_weight)
        return ORACLE_BAD_ARG;
    if (N < 1 || Cin < 1 || H < 1 || W < 1 || Cout < 1 || kh < 1 || kw < 1 || Ho < 1 || Wo < 1)
        return ORACLE_BAD_ARG;
    if (stride_h < 1 || stride_w < 1 || dil_h < 1 || dil_w < 1 || pad_h < 0 || pad_w < 0)
        return ORACLE_BAD_ARG;
    if (group < 1 || deformable_group < 1) return ORACLE_BAD_ARG;
    if (Cin % group || Cout % group || Cin % deformable_group) return ORACLE_BAD_ARG;

    const int64_t K = kh * kw, Cg = Cin / group, Og = Cout / group, Cd = Cin / deformable_group;
    const int64_t P = Ho * Wo, dg = deformable_group;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    /* col[n][c][k][p] = mask * sample; gcol[n][c][k][p] = G */
    const size_t cells = (size_t)(N * Cin * K * P);
    double* col = (double*)malloc(cells * sizeof(double));
    double* gcol = (double*)malloc(cells * sizeof(double));
    if (!col || !gcol) {
        free(col);
        free(gcol);
        return ORACLE_NO_MEMORY;
    }
#define OFF_H(n, gd, k, p) offset[((n) * 2 * dg * K + (gd) * 2 * K + 2 * (k)) * P + (p)]
#define OFF_W(n, gd, k, p) offset[((n) * 2 * dg * K + (gd) * 2 * K + 2 * (k) + 1) * P + (p)]
#define MASK(n, gd, k, p) mask[((n) * dg * K + (gd) * K + (k)) * P + (p)]

    /* pass 1: the modulated columns and their gradients G */
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < N * Ho; ++t) {
        const int64_t n = t / Ho, ho = t % Ho;
        for (int64_t wo = 0; wo < Wo; ++wo) {
            const int64_t p = ho * Wo + wo;
            for (int64_t c = 0; c < Cin; ++c) {
                const int64_t gd = c / Cd, g = c / Cg, cl = c - g * Cg;
                const double* plane = x + (n * Cin + c) * H * W;
                for (int64_t i = 0; i < kh; ++i) {
                    for (int64_t j = 0; j < kw; ++j) {
                        const int64_t k = i * kw + j;
                        const double h = position(ho * stride_h - pad_h + i * dil_h, OFF_H(n, gd, k, p), positions_f32);
                        const double w = position(wo * stride_w - pad_w + j * dil_w, OFF_W(n, gd, k, p), positions_f32);
                        double v, dvdh, dvdw;
                        sample_and_slopes(plane, H, W, h, w, &v, &dvdh, &dvdw);
                        double G = 0.0;
                        for (int64_t o = g * Og; o < (g + 1) * Og; ++o)
                            G += weight[(o * Cg + cl) * K + k] * grad_out[(n * Cout + o) * P + p];
                        const size_t e = (size_t)(((n * Cin + c) * K + k) * P + p);
                        col[e] = MASK(n, gd, k, p) * v;
                        gcol[e] = G;
                    }
                }
            }
        }
    }

    /* pass 2: grad_x, the corner weights times mask times G, per (n, c) */
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < N * Cin; ++t) {
        const int64_t n = t / Cin, c = t % Cin, gd = c / Cd;
        double* gplane = grad_x + (n * Cin + c) * H * W;
        for (int64_t e = 0; e < H * W; ++e) gplane[e] = 0.0;
        for (int64_t ho = 0; ho < Ho; ++ho) {
            for (int64_t wo = 0; wo < Wo; ++wo) {
                const int64_t p = ho * Wo + wo;
                for (int64_t i = 0; i < kh; ++i) {
                    for (int64_t j = 0; j < kw; ++j) {
                        const int64_t k = i * kw + j;
                        const double h = position(ho * stride_h - pad_h + i * dil_h, OFF_H(n, gd, k, p), positions_f32);
                        const double w = position(wo * stride_w - pad_w + j * dil_w, OFF_W(n, gd, k, p), positions_f32);
                        const cell_t cc = cell_of(H, W, h, w);
                        if (!cc.inside) continue;
                        const double gm = gcol[((n * Cin + c) * K + k) * P + p] * MASK(n, gd, k, p);
                        for (int dy = 0; dy < 2; ++dy) {
                            for (int dx = 0; dx < 2; ++dx) {
                                const int64_t y = cc.h0 + dy, xx = cc.w0 + dx;
                                if (!(y >= 0 && y < H && xx >= 0 && xx < W)) continue; /* corner off the image */
                                const double wy = dy ? cc.lh : 1.0 - cc.lh;
                                const double wx = dx ? cc.lw : 1.0 - cc.lw;
                                gplane[y * W + xx] += gm * wy * wx;
                            }
                        }
                    }
                }
            }
        }
    }

    /* pass 3: grad_offset and grad_mask, summed over the deformable group's
     * channels, per (n, ho) */
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < N * Ho; ++t) {
        const int64_t n = t / Ho, ho = t % Ho;
        for (int64_t wo = 0; wo < Wo; ++wo) {
            const int64_t p = ho * Wo + wo;
            for (int64_t gd = 0; gd < dg; ++gd) {
                for (int64_t i = 0; i < kh; ++i) {
                    for (int64_t j = 0; j < kw; ++j) {
                        const int64_t k = i * kw + j;
                        const double h = position(ho * stride_h - pad_h + i * dil_h, OFF_H(n, gd, k, p), positions_f32);
                        const double w = position(wo * stride_w - pad_w + j * dil_w, OFF_W(n, gd, k, p), positions_f32);
                        const double m = MASK(n, gd, k, p);
                        double s_mask = 0.0, s_h = 0.0, s_w = 0.0;
                        for (int64_t c = gd * Cd; c < (gd + 1) * Cd; ++c) {
                            double v, dvdh, dvdw;
                            sample_and_slopes(x + (n * Cin + c) * H * W, H, W, h, w, &v, &dvdh, &dvdw);
                            const double G = gcol[((n * Cin + c) * K + k) * P + p];
                            s_mask += G * v;
                            s_h += G * m * dvdh;
                            s_w += G * m * dvdw;
                        }
                        grad_mask[((n * dg + gd) * K + k) * P + p] = s_mask;
                        grad_offset[((n * 2 * dg + gd * 2) * K + 2 * k) * P + p] = s_h;
                        grad_offset[((n * 2 * dg + gd * 2) * K + 2 * k + 1) * P + p] = s_w;
                    }
                }
            }
        }
    }

    /* pass 4: grad_weight per output channel, grad_bias */
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t o = 0; o < Cout; ++o) {
        const int64_t g = o / Og;
        for (int64_t cl = 0; cl < Cg; ++cl) {
            const int64_t c = g * Cg + cl;
            for (int64_t k = 0; k < K; ++k) {
                double s = 0.0;
                for (int64_t n = 0; n < N; ++n)
                    for (int64_t p = 0; p < P; ++p)
                        s += grad_out[(n * Cout + o) * P + p] * col[((n * Cin + c) * K + k) * P + p];
                grad_weight[(o * Cg + cl) * K + k] = s;
            }
        }
        if (grad_bias) {
            double s = 0.0;
            for (int64_t n = 0; n < N; ++n)
                for (int64_t p = 0; p < P; ++p) s += grad_out[(n * Cout + o) * P + p];
            grad_bias[o] = s;
        }
    }
#undef OFF_H
#undef OFF_W
#undef MASK
    free(col);
    free(gcol);
    return ORACLE_OK;
}
