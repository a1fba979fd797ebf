// Direct evaluation of the modulated deformable convolution forward
// ("TensorRT plugin walkthrough: modulatedDeformConvPlugin", section 5,
// steps 1-3) on the CUDA cores, for shapes with little contraction per output
// (Cin/group x Cout/group small, e.g. depthwise): there the implicit GEMM of
// the fused kernel pads every channel unit to a 128-byte k-tile and every
// group's output channels to an MMA's 16 columns, and its channels-last copy
// of x grows with the padding, while this kernel reads x in NCHW directly.
//
// One thread per output pixel of one image and up to 16 convolution groups
// (16 / (Cout/group) of them, 1 from 16 output channels per group on): for
// each block of up to 3 taps and each deformable group those groups' channels
// touch, it loads every offset and mask value of the block at once, computes
// the sampling points (section 5 step 1: ho*sh - ph + i*dh + dh_off,
// wo*sw - pw + j*dw + dw_off; outside (-1, H) x (-1, W) the sample is 0,
// corners outside the image read 0), the mask-weighted bilinear sample of
// each input channel of the group, and accumulates weight x sample into the
// group's output channels (fp32 registers; the sample is not rounded to the
// I/O type). The group's weights are staged in shared memory as fp32.
//
// Depthwise layers (one input and one output channel per group) take a
// channels-last form of the same sums, below: x copied to [N*H*W + 1][Cin]
// first, then 4 channels of a pixel per lane.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "mdcn_launch.h"

namespace mdcn {

namespace {

__device__ __forceinline__ float ldf(const float* p) { return __ldg(p); }
__device__ __forceinline__ float ldf(const __half* p) { return __half2float(__ldg(p)); }
__device__ __forceinline__ float ldf(const __nv_bfloat16* p) { return __bfloat162float(__ldg(p)); }

__device__ __forceinline__ void stf(float* p, float v) { *p = v; }
__device__ __forceinline__ void stf(__half* p, float v) { *p = __float2half_rn(v); }
__device__ __forceinline__ void stf(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// Four consecutive channels of one channels-last pixel, as one aligned access.
template <typename T>
struct alignas(4 * sizeof(T)) ClVec {
    T v[4];
};
__device__ __forceinline__ float cl_elem(const ClVec<float>& a, int e) { return a.v[e]; }
__device__ __forceinline__ float cl_elem(const ClVec<__half>& a, int e) { return __half2float(a.v[e]); }
__device__ __forceinline__ float cl_elem(const ClVec<__nv_bfloat16>& a, int e) { return __bfloat162float(a.v[e]); }

constexpr int kDirectThreads = 128;
constexpr int kDirectTaps = 3;  // taps whose sampling points a thread holds at once

// GPB consecutive groups per thread (GPB * OGMAX accumulators): a sampling
// point (deformable group, tap block) is computed once and reused by every
// channel of those groups that lies in its deformable group.
template <typename T, int OGMAX, int GPB>
__global__ void __launch_bounds__(kDirectThreads) direct_kernel(const T* __restrict__ x, const T* __restrict__ offset,
                                                                const T* __restrict__ mask, const T* __restrict__ weight,
                                                                const T* __restrict__ bias, T* __restrict__ out,
                                                                uint32_t* __restrict__ status, const Plan pl) {
    extern __shared__ float wsm[];  // [GPB groups][Og][Cg][K], fp32
    if (status && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && threadIdx.x == 0)
        *status = 0u;  // the call's device status word (nothing here waits)
    const int32_t g0 = blockIdx.y * GPB;
    const int32_t ng = min(GPB, pl.group - g0);
    const int64_t n = blockIdx.z;
    const int32_t Og = pl.Og, Cg = pl.Cg, K = pl.K;
    const int32_t wcount = Og * Cg * K;
    {
        const T* wg = weight + static_cast<int64_t>(g0) * wcount;
        for (int32_t i = threadIdx.x; i < ng * wcount; i += kDirectThreads) wsm[i] = ldf(wg + i);
    }
    __syncthreads();

    const int64_t P = pl.P;
    const int64_t p = static_cast<int64_t>(blockIdx.x) * kDirectThreads + threadIdx.x;
    if (p >= P) return;
    const int64_t ho = p / pl.Wo, wo = p - ho * pl.Wo;
    const int64_t H = pl.H, W = pl.W, HW = H * W;
    const float hbase = static_cast<float>(ho * pl.sh - pl.ph), wbase = static_cast<float>(wo * pl.sw - pl.pw);

    float acc[GPB][OGMAX];
#pragma unroll
    for (int q = 0; q < GPB; ++q)
#pragma unroll
        for (int o = 0; o < OGMAX; ++o) acc[q][o] = 0.f;

    // Taps in blocks of kDirectTaps: a thread has every offset and mask load of
    // a block in flight at once, then every corner load of a channel.
    for (int32_t k0 = 0; k0 < K; k0 += kDirectTaps) {
        const int32_t nk = min(kDirectTaps, K - k0);
        int32_t gd_cur = -1;
        int64_t i00[kDirectTaps];
        float wt[kDirectTaps][4];
        uint32_t vb[kDirectTaps];  // corner-valid bits: 1 (y0, x0), 2 (y0, x0+1), 4 (y0+1, x0), 8 (y0+1, x0+1)
#pragma unroll
        for (int q = 0; q < GPB; ++q) {
            if (q >= ng) break;
            const int32_t c0 = (g0 + q) * Cg;
            for (int32_t cl = 0; cl < Cg; ++cl) {
                const int32_t gd = (c0 + cl) / pl.Cd;
                if (gd != gd_cur) {
                    // the sampling points of taps k0 .. k0 + nk - 1 for deformable group gd
                    gd_cur = gd;
                    float dh[kDirectTaps], dw[kDirectTaps], mv[kDirectTaps];
#pragma unroll
                    for (int t = 0; t < kDirectTaps; ++t) {
                        dh[t] = dw[t] = 0.f;
                        mv[t] = 1.f;  // an ordinary convolution (pl.plain) reads no offset or mask
                        if (t < nk && !pl.plain) {
                            const int64_t ob = ((n * pl.dg + gd) * 2 * K + 2 * (k0 + t)) * P + p;
                            dh[t] = ldf(offset + ob);
                            dw[t] = ldf(offset + ob + P);
                            mv[t] = ldf(mask + ((n * pl.dg + gd) * K + k0 + t) * P + p);
                        }
                    }
#pragma unroll
                    for (int t = 0; t < kDirectTaps; ++t) {
                        vb[t] = 0u;
                        i00[t] = 0;
                        wt[t][0] = wt[t][1] = wt[t][2] = wt[t][3] = 0.f;
                        if (t < nk) {
                            const int32_t k = k0 + t;
                            const int32_t i = k / static_cast<int32_t>(pl.kw), j = k - i * static_cast<int32_t>(pl.kw);
                            const float hf = hbase + static_cast<float>(i * pl.dh) + dh[t];
                            const float wf = wbase + static_cast<float>(j * pl.dw) + dw[t];
                            if (hf > -1.0f && hf < static_cast<float>(H) && wf > -1.0f && wf < static_cast<float>(W)) {
                                const float h0f = floorf(hf), w0f = floorf(wf);
                                const float lh = hf - h0f, lw = wf - w0f, hh = 1.0f - lh, hw = 1.0f - lw;
                                const int64_t y0 = static_cast<int64_t>(h0f), x0 = static_cast<int64_t>(w0f);
                                vb[t] = (y0 >= 0 && x0 >= 0 ? 1u : 0u) | (y0 >= 0 && x0 + 1 < W ? 2u : 0u) |
                                        (y0 + 1 < H && x0 >= 0 ? 4u : 0u) | (y0 + 1 < H && x0 + 1 < W ? 8u : 0u);
                                wt[t][0] = hh * hw * mv[t];
                                wt[t][1] = hh * lw * mv[t];
                                wt[t][2] = lh * hw * mv[t];
                                wt[t][3] = lh * lw * mv[t];
                                i00[t] = y0 * W + x0;
                            }
                        }
                    }
                }
                const T* xc = x + (n * pl.Cin + c0 + cl) * HW;
                float xv[kDirectTaps][4];
#pragma unroll
                for (int t = 0; t < kDirectTaps; ++t) {
                    xv[t][0] = (vb[t] & 1u) ? ldf(xc + i00[t]) : 0.f;
                    xv[t][1] = (vb[t] & 2u) ? ldf(xc + i00[t] + 1) : 0.f;
                    xv[t][2] = (vb[t] & 4u) ? ldf(xc + i00[t] + W) : 0.f;
                    xv[t][3] = (vb[t] & 8u) ? ldf(xc + i00[t] + W + 1) : 0.f;
                }
                const float* wr = wsm + static_cast<int64_t>(q) * wcount + cl * K + k0;
#pragma unroll
                for (int t = 0; t < kDirectTaps; ++t) {
                    if (t < nk) {
                        float v = wt[t][0] * xv[t][0];
                        v = fmaf(wt[t][1], xv[t][1], v);
                        v = fmaf(wt[t][2], xv[t][2], v);
                        v = fmaf(wt[t][3], xv[t][3], v);
#pragma unroll
                        for (int o = 0; o < OGMAX; ++o)
                            if (o < Og) acc[q][o] = fmaf(wr[o * Cg * K + t], v, acc[q][o]);
                    }
                }
            }
        }
    }
#pragma unroll
    for (int q = 0; q < GPB; ++q) {
        if (q >= ng) break;
        const int64_t g = g0 + q;
        T* op = out + (n * pl.Cout + g * Og) * P + p;
#pragma unroll
        for (int o = 0; o < OGMAX; ++o) {
            if (o < Og) {
                const float b = bias ? ldf(bias + g * Og + o) : 0.f;
                stf(op + static_cast<int64_t>(o) * P, acc[q][o] + b);
            }
        }
    }
}

template <typename T, int OGMAX, int GPB>
cudaError_t launch_direct_gpb(const Plan& pl, const void* x, const void* offset, const void* mask, const void* weight,
                              const void* bias, void* out, uint32_t* status, cudaStream_t st) {
    const size_t smem = static_cast<size_t>(GPB) * pl.Og * pl.Cg * pl.K * sizeof(float);
    if (smem > static_cast<size_t>(kDirectMaxSmem)) return cudaErrorInvalidValue;
    auto kern = direct_kernel<T, OGMAX, GPB>;
    if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    const dim3 grid(static_cast<unsigned>((pl.P + kDirectThreads - 1) / kDirectThreads),
                    static_cast<unsigned>((pl.group + GPB - 1) / GPB), static_cast<unsigned>(pl.N));
    kern<<<grid, kDirectThreads, smem, st>>>(static_cast<const T*>(x), static_cast<const T*>(offset),
                                            static_cast<const T*>(mask), static_cast<const T*>(weight),
                                            static_cast<const T*>(bias), static_cast<T*>(out), status, pl);
    return cudaGetLastError();
}

// Several groups per thread (16 accumulators at most, direct_groups_per_thread)
// where consecutive groups share a deformable group, so their sampling points
// are computed once; one otherwise (measured on a depthwise 128-channel 80x80
// layer: with one deformable group 207 -> 96 us; with one per channel, 16
// groups per thread only cut the threads, 240 -> 324 us).
template <typename T, int OGMAX>
cudaError_t launch_direct_og(const Plan& pl, const void* x, const void* offset, const void* mask, const void* weight,
                             const void* bias, void* out, uint32_t* status, cudaStream_t st) {
    constexpr int GPB = OGMAX >= 16 ? 1 : 16 / OGMAX;
    if (GPB > 1 && pl.Cd >= 2 * pl.Cg)
        return launch_direct_gpb<T, OGMAX, GPB>(pl, x, offset, mask, weight, bias, out, status, st);
    return launch_direct_gpb<T, OGMAX, 1>(pl, x, offset, mask, weight, bias, out, status, st);
}

template <typename T>
cudaError_t launch_direct_t(const Plan& pl, const void* x, const void* offset, const void* mask, const void* weight,
                            const void* bias, void* out, uint32_t* status, cudaStream_t st) {
    if (pl.Og <= 1) return launch_direct_og<T, 1>(pl, x, offset, mask, weight, bias, out, status, st);
    if (pl.Og <= 4) return launch_direct_og<T, 4>(pl, x, offset, mask, weight, bias, out, status, st);
    if (pl.Og <= 16) return launch_direct_og<T, 16>(pl, x, offset, mask, weight, bias, out, status, st);
    return launch_direct_og<T, kDirectMaxOg>(pl, x, offset, mask, weight, bias, out, status, st);
}

// ---------------------------------------------------------------- depthwise, channels-last
// For depthwise layers (one input and one output channel per group) whose
// deformable groups hold whole 4-channel chunks: x is first made
// channels-last, so that one sampling point's 4 corners are read for 4
// channels at a time (8 bytes for 16-bit types) by each lane, and a warp
// reads a corner's 128 channels as 256 contiguous bytes instead of 128
// scattered 2-byte loads from the channel planes. (Measured on the neck
// shape as a depthwise layer, 128 channels, one deformable group.)

// x [N][C][H*W] -> xt [N*H*W + 1][C]; the last pixel is all zeros (read for
// corners outside the image). 64 x 64 tiles through shared memory; block 0
// also clears the call's status word.
template <typename T>
__global__ void __launch_bounds__(256) nhwc_zero_pixel_kernel(const T* __restrict__ x, T* __restrict__ xt,
                                                              uint32_t* __restrict__ status, int64_t C, int64_t HW,
                                                              int64_t NHW) {
    __shared__ float tile[64][65];
    if (blockIdx.x == 0 && blockIdx.y == 0) {
        if (threadIdx.x == 0 && status) *status = 0u;
        for (int64_t i = threadIdx.x; i < C; i += 256) stf(xt + NHW * C + i, 0.f);
    }
    const int64_t n = blockIdx.y;
    const int64_t ptiles = (HW + 63) / 64;
    const int64_t c0 = static_cast<int64_t>(blockIdx.x) / ptiles * 64;
    const int64_t p0 = static_cast<int64_t>(blockIdx.x) % ptiles * 64;
    const int tx = threadIdx.x % 64, ty = threadIdx.x / 64;
    float v[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const int64_t c = c0 + ty + 4 * k, pp = p0 + tx;
        v[k] = c < C && pp < HW ? ldf(x + (n * C + c) * HW + pp) : 0.f;
    }
#pragma unroll
    for (int k = 0; k < 16; ++k) tile[ty + 4 * k][tx] = v[k];
    __syncthreads();
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const int64_t pp = p0 + ty + 4 * k, c = c0 + tx;
        if (pp < HW && c < C) stf(xt + (n * HW + pp) * C + c, tile[tx][ty + 4 * k]);
    }
}

constexpr int kClPix = 32;      // output pixels per block (4 per warp)
constexpr int kClChannels = 128;  // channels per block: 4 per lane

// The block's weights, wsm[k][cc] = weight[cbase + cc][k] in fp32 (0 past Cin).
template <typename T>
__device__ __forceinline__ void cl_stage_weights(const T* __restrict__ weight, float* wsm, int32_t K, int32_t C,
                                                 int32_t cbase) {
    for (int32_t i = threadIdx.x; i < K * kClChannels; i += 256) {
        const int32_t k = i / kClChannels, c = cbase + (i - k * kClChannels);
        wsm[i] = c < C ? ldf(weight + static_cast<int64_t>(c) * K + k) : 0.f;
    }
}

// The block's output tile osm[cc][j] (+ bias) to NCHW, along pixels: warp w
// writes channels w, w + 8, ... of the block's kClPix pixels.
template <typename T>
__device__ __forceinline__ void cl_store_tile(const float* osm, const T* __restrict__ bias, T* __restrict__ out,
                                              int64_t n, int32_t C, int32_t cbase, int64_t p0, int64_t P) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t p = p0 + lane;
    for (int cc = warp; cc < kClChannels; cc += 8) {
        const int32_t co = cbase + cc;
        if (co < C && p < P) {
            const float b = bias ? ldf(bias + co) : 0.f;
            stf(out + (n * C + co) * P + p, osm[cc * (kClPix + 1) + lane] + b);
        }
    }
}

// Lane l of every warp takes channels cbase + 4l .. + 3 (one deformable group:
// one sampling point per tap) of the block's pixels, one pixel at a time, its
// taps in blocks of kDirectTaps with every offset, mask and corner load of a
// block in flight at once; the 4 channels' sums stay in fp32 registers, then
// go through a shared-memory tile so that the NCHW output is written along
// pixels.
template <typename T>
__global__ void __launch_bounds__(256) direct_cl_kernel(const T* __restrict__ xt, const T* __restrict__ offset,
                                                        const T* __restrict__ mask, const T* __restrict__ weight,
                                                        const T* __restrict__ bias, T* __restrict__ out, const Plan pl) {
    extern __shared__ float csm[];  // weights [K][128], then the output tile [128][kClPix + 1]
    const int32_t K = pl.K, C = static_cast<int32_t>(pl.Cin);
    float* wsm = csm;
    float* osm = csm + K * kClChannels;
    const int64_t n = blockIdx.z;
    const int32_t cbase = static_cast<int32_t>(blockIdx.y) * kClChannels;
    const int64_t p0 = static_cast<int64_t>(blockIdx.x) * kClPix;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    cl_stage_weights(weight, wsm, K, C, cbase);
    __syncthreads();
    const int32_t c = cbase + 4 * lane;
    const bool cval = c < C;  // C is a multiple of 4: the lane's 4 channels all exist, or none
    const int64_t gd = cval ? c / pl.Cd : 0;
    const int64_t P = pl.P, H = pl.H, W = pl.W;
    const int64_t zpix = pl.N * H * W;  // the all-zero pixel
    const float Hf = static_cast<float>(H), Wf = static_cast<float>(W);
    for (int j = warp; j < kClPix; j += 8) {
        const int64_t p = p0 + j;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        if (p < P && cval) {
            const int64_t ho = p / pl.Wo, wo = p - ho * pl.Wo;
            const float hbase = static_cast<float>(ho * pl.sh - pl.ph), wbase = static_cast<float>(wo * pl.sw - pl.pw);
            for (int32_t k0 = 0; k0 < K; k0 += kDirectTaps) {
                const int32_t nk = min(kDirectTaps, K - k0);
                float dh[kDirectTaps], dw[kDirectTaps], mv[kDirectTaps];
#pragma unroll
                for (int t = 0; t < kDirectTaps; ++t) {
                    dh[t] = dw[t] = 0.f;
                    mv[t] = t < nk ? 1.f : 0.f;  // an ordinary convolution (pl.plain) reads no offset or mask
                    if (t < nk && !pl.plain) {
                        const int64_t ob = ((n * pl.dg + gd) * 2 * K + 2 * (k0 + t)) * P + p;
                        dh[t] = ldf(offset + ob);
                        dw[t] = ldf(offset + ob + P);
                        mv[t] = ldf(mask + ((n * pl.dg + gd) * K + k0 + t) * P + p);
                    }
                }
                int64_t pix[kDirectTaps][4];
                float wq[kDirectTaps][4];
#pragma unroll
                for (int t = 0; t < kDirectTaps; ++t) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        pix[t][q] = zpix;
                        wq[t][q] = 0.f;
                    }
                    const int32_t k = k0 + t;
                    const int32_t i = k / static_cast<int32_t>(pl.kw), jj = k - i * static_cast<int32_t>(pl.kw);
                    const float hf = hbase + static_cast<float>(i * pl.dh) + dh[t];
                    const float wf = wbase + static_cast<float>(jj * pl.dw) + dw[t];
                    if (t < nk && hf > -1.0f && hf < Hf && wf > -1.0f && wf < Wf) {
                        const float h0f = floorf(hf), w0f = floorf(wf);
                        const float lh = hf - h0f, lw = wf - w0f, hh = 1.0f - lh, hw = 1.0f - lw;
                        const int64_t y0 = static_cast<int64_t>(h0f), x0 = static_cast<int64_t>(w0f);
                        const int64_t b = (n * H + y0) * W + x0;
                        if (y0 >= 0 && x0 >= 0) pix[t][0] = b;
                        if (y0 >= 0 && x0 + 1 < W) pix[t][1] = b + 1;
                        if (y0 + 1 < H && x0 >= 0) pix[t][2] = b + W;
                        if (y0 + 1 < H && x0 + 1 < W) pix[t][3] = b + W + 1;
                        wq[t][0] = hh * hw * mv[t];
                        wq[t][1] = hh * lw * mv[t];
                        wq[t][2] = lh * hw * mv[t];
                        wq[t][3] = lh * lw * mv[t];
                    }
                }
                ClVec<T> X[kDirectTaps][4];
#pragma unroll
                for (int t = 0; t < kDirectTaps; ++t)
#pragma unroll
                    for (int q = 0; q < 4; ++q) X[t][q] = *reinterpret_cast<const ClVec<T>*>(xt + pix[t][q] * C + c);
#pragma unroll
                for (int t = 0; t < kDirectTaps; ++t) {
                    if (t < nk) {
                        const float* wk = wsm + (k0 + t) * kClChannels + 4 * lane;
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            float v = wq[t][0] * cl_elem(X[t][0], e);
                            v = fmaf(wq[t][1], cl_elem(X[t][1], e), v);
                            v = fmaf(wq[t][2], cl_elem(X[t][2], e), v);
                            v = fmaf(wq[t][3], cl_elem(X[t][3], e), v);
                            acc[e] = fmaf(wk[e], v, acc[e]);
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) osm[(4 * lane + e) * (kClPix + 1) + j] = acc[e];
    }
    __syncthreads();
    cl_store_tile(osm, bias, out, n, C, cbase, p0, P);
}

// The same for 16-bit types, at most 9 taps, one deformable group per block of
// 128 channels (so every lane of a warp samples the same points) and fewer
// than 2^31 elements in the channels-last copy (32-bit offsets): a pixel's
// 3K offset and mask values are one load per lane (lane t the value t), shared
// by shuffles, and the next pixel's are loaded while this one is gathered;
// every corner load of all its taps (4K per lane) is in flight at once.
template <typename T>
__global__ void __launch_bounds__(256, 2) direct_cl9_kernel(const T* __restrict__ xt, const T* __restrict__ offset,
                                                         const T* __restrict__ mask, const T* __restrict__ weight,
                                                         const T* __restrict__ bias, T* __restrict__ out,
                                                         const Plan pl) {
    static_assert(sizeof(T) == 2, "16-bit types");
    // weights [K][128], the output tile [128][kClPix + 1], then the taps' displacements (h, then w)
    extern __shared__ float csm[];
    const int32_t K = pl.K, C = static_cast<int32_t>(pl.Cin);
    float* wsm = csm;
    float* osm = csm + K * kClChannels;
    float* tsm = osm + kClChannels * (kClPix + 1);
    const int64_t n = blockIdx.z;
    const int32_t cbase = static_cast<int32_t>(blockIdx.y) * kClChannels;
    const int64_t p0 = static_cast<int64_t>(blockIdx.x) * kClPix;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    cl_stage_weights(weight, wsm, K, C, cbase);
    if (threadIdx.x < K) {  // tap t = i * kw + j: displacement (i * dh, j * dw), once per block
        const int32_t t = threadIdx.x, i = t / static_cast<int32_t>(pl.kw), jj = t - i * static_cast<int32_t>(pl.kw);
        tsm[t] = static_cast<float>(i * pl.dh);
        tsm[kDirectClMaxTaps + t] = static_cast<float>(jj * pl.dw);
    }
    __syncthreads();
    const int32_t c = cbase + 4 * lane;
    const bool cval = c < C;
    const int64_t gd = cbase / pl.Cd;  // one deformable group for the whole block
    const int64_t P = pl.P, H = pl.H, W = pl.W;
    // pixel indices of the channels-last copy in 32 bits (its N*H*W + 1 pixels are below 2^31)
    const int32_t zpix32 = static_cast<int32_t>(pl.N * H * W), H32 = static_cast<int32_t>(H),
                  W32 = static_cast<int32_t>(W), img = static_cast<int32_t>(n * H);
    const float Hf = static_cast<float>(H), Wf = static_cast<float>(W);
    const int64_t obase = (n * pl.dg + gd) * 2 * K * P, mbase = (n * pl.dg + gd) * K * P;
    // lane t's offset / mask value of pixel p (t < 2K: offset channel t, 2K <= t < 3K: mask of tap t - 2K)
    auto om_load = [&](int64_t p) -> float {
        if (p >= P || pl.plain) return 0.f;
        if (lane < 2 * K) return ldf(offset + obase + lane * P + p);
        if (lane < 3 * K) return ldf(mask + mbase + (lane - 2 * K) * P + p);
        return 0.f;
    };
    float ov = om_load(p0 + warp);
    for (int j = warp; j < kClPix; j += 8) {
        const int64_t p = p0 + j;
        const float ov_next = om_load(p + 8);  // in flight while this pixel is gathered
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        if (p < P) {  // warp-uniform
            // 32-bit position arithmetic: pixels below 2^31, coordinates below 2^24
            const int32_t p32 = static_cast<int32_t>(p), Wo32 = static_cast<int32_t>(pl.Wo);
            const int32_t ho = p32 / Wo32, wo = p32 - ho * Wo32;
            const float hbase = static_cast<float>(ho * pl.sh - pl.ph), wbase = static_cast<float>(wo * pl.sw - pl.pw);
            ClVec<T> X[9][4];
            float lhv[9], lwv[9], mvv[9];  // the taps' cell fractions and mask (mask 0: outside)
#pragma unroll
            for (int t = 0; t < 9; ++t) {
                const float dh = __shfl_sync(0xffffffffu, ov, 2 * t), dw = __shfl_sync(0xffffffffu, ov, 2 * t + 1);
                const float mv = pl.plain ? 1.f : __shfl_sync(0xffffffffu, ov, (2 * K + t) & 31);
                int32_t pix[4] = {zpix32, zpix32, zpix32, zpix32};
                lhv[t] = lwv[t] = mvv[t] = 0.f;
                const float hf = hbase + tsm[t] + dh;
                const float wf = wbase + tsm[kDirectClMaxTaps + t] + dw;
                if (t < K && hf > -1.0f && hf < Hf && wf > -1.0f && wf < Wf) {
                    const float h0f = floorf(hf), w0f = floorf(wf);
                    lhv[t] = hf - h0f;
                    lwv[t] = wf - w0f;
                    mvv[t] = mv;
                    const int32_t y0 = static_cast<int32_t>(h0f), x0 = static_cast<int32_t>(w0f);
                    const int32_t b = (img + y0) * W32 + x0;
                    if (y0 >= 0 && x0 >= 0) pix[0] = b;
                    if (y0 >= 0 && x0 + 1 < W32) pix[1] = b + 1;
                    if (y0 + 1 < H32 && x0 >= 0) pix[2] = b + W32;
                    if (y0 + 1 < H32 && x0 + 1 < W32) pix[3] = b + W32 + 1;
                }
                if (cval) {  // element offsets in 32 bits: (N*H*W + 1) * Cin below 2^31
#pragma unroll
                    for (int q = 0; q < 4; ++q) X[t][q] = *reinterpret_cast<const ClVec<T>*>(xt + (pix[q] * C + c));
                }
            }
            if (cval) {
#pragma unroll
                for (int t = 0; t < 9; ++t) {
                    if (t < K) {
                        const float lh = lhv[t], lw = lwv[t], hh = 1.0f - lh, hw = 1.0f - lw;
                        const float wq0 = hh * hw * mvv[t], wq1 = hh * lw * mvv[t], wq2 = lh * hw * mvv[t],
                                    wq3 = lh * lw * mvv[t];
                        const float4 w4 = *reinterpret_cast<const float4*>(wsm + t * kClChannels + 4 * lane);
                        const float wk[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            float v = wq0 * cl_elem(X[t][0], e);
                            v = fmaf(wq1, cl_elem(X[t][1], e), v);
                            v = fmaf(wq2, cl_elem(X[t][2], e), v);
                            v = fmaf(wq3, cl_elem(X[t][3], e), v);
                            acc[e] = fmaf(wk[e], v, acc[e]);
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) osm[(4 * lane + e) * (kClPix + 1) + j] = acc[e];
        ov = ov_next;
    }
    __syncthreads();
    cl_store_tile(osm, bias, out, n, C, cbase, p0, P);
}

template <typename T>
cudaError_t launch_direct_cl_t(const Plan& pl, const void* x, const void* offset, const void* mask,
                               const void* weight, const void* bias, void* out, void* ws, cudaStream_t st) {
    uint32_t* status = static_cast<uint32_t*>(ws);
    T* xt = reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + pl.off_xt);
    const int64_t HW = pl.H * pl.W, NHW = pl.N * HW;
    const int64_t tiles = ((HW + 63) / 64) * ((pl.Cin + 63) / 64);
    nhwc_zero_pixel_kernel<T><<<dim3(static_cast<unsigned>(tiles), static_cast<unsigned>(pl.N)), 256, 0, st>>>(
        static_cast<const T*>(x), xt, status, pl.Cin, HW, NHW);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const size_t smem = (static_cast<size_t>(pl.K) * kClChannels + kClChannels * (kClPix + 1)) * sizeof(float);
    const dim3 grid(static_cast<unsigned>((pl.P + kClPix - 1) / kClPix),
                    static_cast<unsigned>((pl.Cin + kClChannels - 1) / kClChannels), static_cast<unsigned>(pl.N));
    // one deformable group per 128-channel block: the warp-shared sampling points
    const bool shared_points = pl.dg == 1 || pl.Cd % kClChannels == 0;
    if constexpr (sizeof(T) == 2) {
        if (shared_points && pl.K <= 9 && (pl.N * pl.H * pl.W + 1) * pl.Cin < 2147483647ll) {
            const size_t smem9 = smem + 2 * kDirectClMaxTaps * sizeof(float);
            direct_cl9_kernel<T><<<grid, 256, smem9, st>>>(xt, static_cast<const T*>(offset),
                                                          static_cast<const T*>(mask), static_cast<const T*>(weight),
                                                          static_cast<const T*>(bias), static_cast<T*>(out), pl);
            return cudaGetLastError();
        }
    }
    direct_cl_kernel<T><<<grid, 256, smem, st>>>(xt, static_cast<const T*>(offset), static_cast<const T*>(mask),
                                                 static_cast<const T*>(weight), static_cast<const T*>(bias),
                                                 static_cast<T*>(out), pl);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_direct(const Plan& pl, const void* x, const void* offset, const void* mask, const void* weight,
                          const void* bias, void* out, void* ws, cudaStream_t st) {
    if (pl.direct_cl) {
        if (pl.Cg != 1 || pl.Og != 1 || pl.Cin % 4 != 0 || pl.Cd % 4 != 0 || pl.K > kDirectClMaxTaps ||
            pl.N > 65535 || pl.Cin > 65535ll * 128 || (pl.P + kClPix - 1) / kClPix > 2147483647ll)
            return cudaErrorInvalidValue;
        switch (pl.dtype) {
            case kF32: return launch_direct_cl_t<float>(pl, x, offset, mask, weight, bias, out, ws, st);
            case kF16: return launch_direct_cl_t<__half>(pl, x, offset, mask, weight, bias, out, ws, st);
            default: return launch_direct_cl_t<__nv_bfloat16>(pl, x, offset, mask, weight, bias, out, ws, st);
        }
    }
    if (pl.Og > kDirectMaxOg || pl.P > 2147483647ll * kDirectThreads || pl.group > 65535 || pl.N > 65535 ||
        direct_groups_per_thread(pl.Og) * static_cast<int64_t>(pl.Og) * pl.Cg * pl.K * 4 > kDirectMaxSmem)
        return cudaErrorInvalidValue;
    uint32_t* status = static_cast<uint32_t*>(ws);
    switch (pl.dtype) {
        case kF32: return launch_direct_t<float>(pl, x, offset, mask, weight, bias, out, status, st);
        case kF16: return launch_direct_t<__half>(pl, x, offset, mask, weight, bias, out, status, st);
        default: return launch_direct_t<__nv_bfloat16>(pl, x, offset, mask, weight, bias, out, status, st);
    }
}

}  // namespace mdcn
