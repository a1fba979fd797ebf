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
