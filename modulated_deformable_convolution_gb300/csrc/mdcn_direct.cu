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

}  // namespace

cudaError_t launch_direct(const Plan& pl, const void* x, const void* offset, const void* mask, const void* weight,
                          const void* bias, void* out, void* ws, cudaStream_t st) {
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
