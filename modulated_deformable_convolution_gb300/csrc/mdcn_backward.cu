// Backward pass of the modulated deformable convolution: the gradients of
// L = sum(grad_out * y) with respect to x, offset, mask, weight and bias, for
// the forward of "TensorRT plugin walkthrough: modulatedDeformConvPlugin"
// (section 5 steps 1-3). The page has no backward; this is the gradient of its
// definition, with the right-hand slope on the edges of a bilinear cell and 0
// outside the open sampling range (-1, H) x (-1, W), as its range test gives.
//
// With G[n, c, k, p] = sum over the output channels o of c's group of
// weight[o, c_l, k] * grad_out[n, o, p] (the gradient of a modulated column
// element), and v, dv/dh, dv/dw the bilinear sample and its slopes:
//   grad_mask[n, gd*K + k, p]        = sum over c of gd: G * v
//   grad_offset[n, gd*2K + 2k (+1), p] = mask * sum over c of gd: G * dv/dh (dv/dw)
//   grad_x[n, c, corner]            += G * mask * corner weight
//   grad_weight[o, c_l, k]           = sum over n, p: grad_out[n, o, p] * mask * v
//   grad_bias[o]                     = sum over n, p: grad_out[n, o, p]
//
// Work per chunk of images (its buffers within a fixed budget):
//   1. x of the chunk -> channels-last (tiled transpose);
//   2. G = W_g^T * grad_out per group (fp32 out), laid out [n][g][p][k][c_l]
//      so that one sampling point's channels are contiguous: for float16 and
//      bfloat16 the tcgen05 GEMM of mdcn_gemm.cu (grad_out and the tap-major
//      weight read as MN-major operands, straight from their layouts), for
//      float32 one cuBLAS strided-batched GEMM per group (fp32 products);
//   3. the sampling backward: a segment of lanes per sampling point (n, p, gd,
//      k), lanes along channels; the slope sums are reduced across the
//      segment by shuffles (deterministic), grad_x goes by fp32 vector
//      reductions into a channels-last accumulator, and the modulated column
//      mask * v is written for step 4;
//   4. grad_weight += grad_out * col^T (fp32 accumulate in workspace): for
//      float16 / bfloat16 one tcgen05 GEMM over the chunk's images and all
//      groups (the contraction over images and pixels split between CTAs,
//      fp32 reductions into the zeroed accumulator); for float32, cuBLAS: for
//      group 1 one GEMM over the chunk's images, after grad_out is re-laid
//      [Cout][n][P], otherwise per image one strided-batched GEMM over the
//      groups;
//   5. the fp32 grad_x accumulator -> NCHW in the I/O type.
// Then the weight gradient to [Cout, Cg, kh, kw] and the bias reduction.
#include <cublas_v2.h>

#include <algorithm>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "mdcn_backward.h"
#include "mdcn_gemm.h"
#include "mdcn_launch.h"
#include "mdcn_plan.h"

namespace mdcn {


namespace {

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__half v) { return __half2float(v); }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T>
__device__ __forceinline__ T from_f(float v);
template <>
__device__ __forceinline__ float from_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ __half from_f<__half>(float v) { return __float2half_rn(v); }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// VEC consecutive elements of type T as one aligned access.
template <typename T, int VEC>
struct alignas(sizeof(T) * VEC) Vec {
    T v[VEC];
};

template <typename T, int VEC>
__device__ __forceinline__ void load_f(const T* p, float (&out)[VEC]) {
    const Vec<T, VEC> t = *reinterpret_cast<const Vec<T, VEC>*>(p);
#pragma unroll
    for (int i = 0; i < VEC; ++i) out[i] = to_f(t.v[i]);
}

template <typename T, int VEC>
__device__ __forceinline__ void store_f(T* p, const float (&in)[VEC]) {
    Vec<T, VEC> t;
#pragma unroll
    for (int i = 0; i < VEC; ++i) t.v[i] = from_f<T>(in[i]);
    *reinterpret_cast<Vec<T, VEC>*>(p) = t;
}

// p[0..VEC) += s * w[0..VEC) as fp32 reductions (one vector reduction for VEC = 4).
template <int VEC>
__device__ __forceinline__ void red_add(float* p, const float (&g)[VEC], float s) {
    if constexpr (VEC == 4) {
        atomicAdd(reinterpret_cast<float4*>(p), make_float4(g[0] * s, g[1] * s, g[2] * s, g[3] * s));
    } else {
#pragma unroll
        for (int i = 0; i < VEC; ++i) atomicAdd(p + i, g[i] * s);
    }
}

// out[b][c][r] = in[b][r][c] for an R x C matrix per batch entry b
// (blockIdx.y), through a 64 x 65 shared-memory tile; blockIdx.x walks the
// tiles, column tiles fastest. 256 threads as 64 x 4: each thread has its 16
// loads in flight before it stores (a 32 x 32 tile per block held too few
// bytes in flight to approach memory bandwidth).
constexpr int kTransposeTile = 64;

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(256) transpose_kernel(const Tin* __restrict__ in, Tout* __restrict__ out, int64_t R,
                                                        int64_t C) {
    constexpr int kT = kTransposeTile, kRows = kT / 4;
    __shared__ float tile[kT][kT + 1];
    const int64_t b = blockIdx.y;
    const int64_t ctiles = (C + kT - 1) / kT;
    const int64_t r0 = static_cast<int64_t>(blockIdx.x) / ctiles * kT;
    const int64_t c0 = static_cast<int64_t>(blockIdx.x) % ctiles * kT;
    const Tin* src = in + b * R * C;
    Tout* dst = out + b * R * C;
    const int tx = threadIdx.x % kT, ty = threadIdx.x / kT;
    float v[kRows];
#pragma unroll
    for (int k = 0; k < kRows; ++k) {
        const int64_t r = r0 + ty + 4 * k, c = c0 + tx;
        v[k] = r < R && c < C ? to_f(src[r * C + c]) : 0.f;
    }
#pragma unroll
    for (int k = 0; k < kRows; ++k) tile[ty + 4 * k][tx] = v[k];
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kRows; ++k) {
        const int64_t c = c0 + ty + 4 * k, r = r0 + tx;
        if (r < R && c < C) dst[c * R + r] = from_f<Tout>(tile[tx][ty + 4 * k]);
    }
}

// The same transposes with 16-byte accesses on both sides (R and C multiples
// of 16 / sizeof of each side's type): a 64 x 64 tile per block, loaded as
// 16-byte vectors along the input rows and stored as 16-byte vectors along
// the output rows, through a 64 x 65 fp32 tile. With zero != nullptr (same
// layout as out, fp32) the block also clears its tile of zero: the chunk's
// grad_x accumulator, cleared while x is transposed.
template <typename Tin, typename Tout>
__global__ void __launch_bounds__(256) transpose_vec_kernel(const Tin* __restrict__ in, Tout* __restrict__ out,
                                                            float* __restrict__ zero, int64_t R, int64_t C) {
    constexpr int kT = kTransposeTile;
    constexpr int kVi = 16 / sizeof(Tin), kVo = 16 / sizeof(Tout);
    __shared__ float tile[kT][kT + 1];
    const int64_t b = blockIdx.y;
    const int64_t ctiles = (C + kT - 1) / kT;
    const int64_t r0 = static_cast<int64_t>(blockIdx.x) / ctiles * kT;
    const int64_t c0 = static_cast<int64_t>(blockIdx.x) % ctiles * kT;
    const Tin* src = in + b * R * C;
    Tout* dst = out + b * R * C;
    // load: the tile's rows as kT / kVi vectors each
    constexpr int kVrow = kT / kVi, kLoads = kT * kVrow / 256;
    Vec<Tin, kVi> v[kLoads];
#pragma unroll
    for (int k = 0; k < kLoads; ++k) {
        const int idx = threadIdx.x + 256 * k;
        const int64_t r = r0 + idx / kVrow, c = c0 + (idx % kVrow) * kVi;
        if (r < R && c < C) {
            v[k] = *reinterpret_cast<const Vec<Tin, kVi>*>(src + r * C + c);
        } else {
#pragma unroll
            for (int e = 0; e < kVi; ++e) v[k].v[e] = Tin(0);
        }
    }
#pragma unroll
    for (int k = 0; k < kLoads; ++k) {
        const int idx = threadIdx.x + 256 * k;
#pragma unroll
        for (int e = 0; e < kVi; ++e) tile[idx / kVrow][(idx % kVrow) * kVi + e] = to_f(v[k].v[e]);
    }
    __syncthreads();
    // store: output row c0 + cc holds the tile's column cc, kT / kVo vectors each
    constexpr int kVcol = kT / kVo, kStores = kT * kVcol / 256;
#pragma unroll
    for (int k = 0; k < kStores; ++k) {
        const int cc = threadIdx.x % kT, vi = threadIdx.x / kT + (256 / kT) * k;
        const int64_t c = c0 + cc, r = r0 + vi * kVo;
        if (c < C && r < R) {
            float w[kVo];
#pragma unroll
            for (int e = 0; e < kVo; ++e) w[e] = tile[vi * kVo + e][cc];
            store_f<Tout, kVo>(dst + c * R + r, w);
            if (zero) {
#pragma unroll
                for (int e = 0; e < kVo; e += 4)
                    *reinterpret_cast<float4*>(zero + b * R * C + c * R + r + e) = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
    }
}

// out[o][n][p] = in[n][o][p] for the chunk's nb images: grad_out with the
// image index moved inside the channel index (16-byte copies along p when P
// is a multiple of 16 / sizeof(T), else element copies).
template <typename T>
__global__ void __launch_bounds__(256) swap_image_channel_kernel(const T* __restrict__ in, T* __restrict__ out,
                                                                 int64_t nb, int64_t C, int64_t P) {
    constexpr int64_t kV = 16 / sizeof(T);
    const bool vec = P % kV == 0;
    const int64_t rowlen = vec ? P / kV : P;  // units per (n, o) row
    const int64_t total = nb * C * rowlen;
    for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
         e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t row = e / rowlen, u = e - row * rowlen;
        const int64_t n = row / C, o = row - n * C;
        const int64_t dst_row = o * nb + n;
        if (vec)
            reinterpret_cast<uint4*>(out + dst_row * P)[u] = reinterpret_cast<const uint4*>(in + row * P)[u];
        else
            out[dst_row * P + u] = in[row * P + u];
    }
}

// wt[o][k][c_l] = w[o][c_l][k]
template <typename T>
__global__ void __launch_bounds__(256) weight_tap_major_kernel(const T* __restrict__ w, T* __restrict__ wt,
                                                               int64_t Cout, int64_t Cg, int64_t K,
                                                               uint32_t* __restrict__ status) {
    if (blockIdx.x == 0 && threadIdx.x == 0) *status = 0u;  // the call's device status word
    const int64_t total = Cout * Cg * K;
    for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
         e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t o = e / (K * Cg), r = e - o * (K * Cg);
        const int64_t k = r / Cg, cl = r - k * Cg;
        wt[e] = w[(o * Cg + cl) * K + k];
    }
}

// grad_weight[o][c_l][k] = gw[o][k][c_l] in the I/O type
template <typename T>
__global__ void __launch_bounds__(256) weight_grad_out_kernel(const float* __restrict__ gw, T* __restrict__ gweight,
                                                              int64_t Cout, int64_t Cg, int64_t K) {
    const int64_t total = Cout * Cg * K;
    for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
         e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t o = e / (Cg * K), r = e - o * (Cg * K);
        const int64_t cl = r / K, k = r - cl * K;
        gweight[e] = from_f<T>(gw[(o * K + k) * Cg + cl]);
    }
}

// The two weight re-layouts one output channel per block, through shared
// memory (Cg*K elements): both the read of one layout and the write of the
// other are contiguous. wt[o][k][c_l] = w[o][c_l][k]; the block of o = 0
// also clears the call's device status word.
template <typename T>
__global__ void __launch_bounds__(256) weight_tap_major_block_kernel(const T* __restrict__ w, T* __restrict__ wt,
                                                                     int32_t Cg, int32_t K,
                                                                     uint32_t* __restrict__ status) {
    extern __shared__ float wsm[];  // [c_l][k], pitch K + 1
    if (blockIdx.x == 0 && threadIdx.x == 0) *status = 0u;
    const int64_t o = blockIdx.x;
    const int32_t n = Cg * K;
    const T* src = w + o * n;
    T* dst = wt + o * n;
    // 8 loads per thread in flight per round
    for (int32_t base = 0; base < n; base += 8 * 256) {
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int32_t e = base + 256 * u + static_cast<int32_t>(threadIdx.x);
            v[u] = e < n ? to_f(src[e]) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int32_t e = base + 256 * u + static_cast<int32_t>(threadIdx.x);
            if (e < n) {
                const int32_t cl = e / K, k = e - cl * K;
                wsm[cl * (K + 1) + k] = v[u];
            }
        }
    }
    __syncthreads();
    for (int32_t e = threadIdx.x; e < n; e += blockDim.x) {
        const int32_t k = e / Cg, cl = e - k * Cg;
        dst[e] = from_f<T>(wsm[cl * (K + 1) + k]);
    }
}

// grad_weight[o][c_l][k] = gw[o][k][c_l] in the I/O type, one output channel per block.
template <typename T>
__global__ void __launch_bounds__(256) weight_grad_out_block_kernel(const float* __restrict__ gw,
                                                                    T* __restrict__ gweight, int32_t Cg, int32_t K) {
    extern __shared__ float wsm[];  // [k][c_l], pitch Cg + 1
    const int64_t o = blockIdx.x;
    const int32_t n = Cg * K;
    const float* src = gw + o * n;
    T* dst = gweight + o * n;
    // 8 loads per thread in flight per round
    for (int32_t base = 0; base < n; base += 8 * 256) {
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int32_t e = base + 256 * u + static_cast<int32_t>(threadIdx.x);
            v[u] = e < n ? src[e] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int32_t e = base + 256 * u + static_cast<int32_t>(threadIdx.x);
            if (e < n) {
                const int32_t k = e / Cg, cl = e - k * Cg;
                wsm[k * (Cg + 1) + cl] = v[u];
            }
        }
    }
    __syncthreads();
    for (int32_t e = threadIdx.x; e < n; e += blockDim.x) {
        const int32_t cl = e / K, k = e - cl * K;
        dst[e] = from_f<T>(wsm[k * (Cg + 1) + cl]);
    }
}

// grad_bias[o] with 16-byte loads (P a multiple of 16 / sizeof(T)): one block
// per output channel; each thread sums its vectors in order, then a fixed
// tree over the block.
template <typename T>
__global__ void __launch_bounds__(256) bias_grad_vec_kernel(const T* __restrict__ gout, T* __restrict__ gbias,
                                                            int64_t N, int64_t Cout, int64_t P) {
    constexpr int kV = 16 / sizeof(T);
    __shared__ float part[8];
    const int64_t o = blockIdx.x;
    const int64_t pv = P / kV;
    float s = 0.f;
    for (int64_t i = threadIdx.x; i < N * pv; i += blockDim.x) {
        const int64_t n = i / pv, v = i - n * pv;
        float x[kV];
        load_f<T, kV>(gout + (n * Cout + o) * P + v * kV, x);
#pragma unroll
        for (int e = 0; e < kV; ++e) s += x[e];
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) s += __shfl_xor_sync(0xffffffffu, s, d);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.f;
        for (int i = 0; i < 8; ++i) t += part[i];
        gbias[o] = from_f<T>(t);
    }
}

// grad_bias[o] = sum over n, p of grad_out[n][o][p]: one block per output
// channel, fixed summation order.
template <typename T>
__global__ void __launch_bounds__(256) bias_grad_kernel(const T* __restrict__ gout, T* __restrict__ gbias, int64_t N,
                                                        int64_t Cout, int64_t P) {
    __shared__ float part[8];
    const int64_t o = blockIdx.x;
    float s = 0.f;
    for (int64_t n = 0; n < N; ++n) {
        const T* row = gout + (n * Cout + o) * P;
        for (int64_t p = threadIdx.x; p < P; p += blockDim.x) s += to_f(row[p]);
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) s += __shfl_xor_sync(0xffffffffu, s, d);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.f;
        for (int i = 0; i < 8; ++i) t += part[i];
        gbias[o] = from_f<T>(t);
    }
}

// The sampling backward of one chunk. Grid (pixel blocks, dg*K, images of
// the chunk): a segment of `lanes` consecutive threads per sampling point
// (pixel p, deformable group gd, tap k of image n), each lane taking VEC
// consecutive channels of the deformable group per step. Per-point index
// arithmetic is 32-bit (the planner bounds P, Cin and the coordinates);
// element offsets are 64-bit. Reads the chunk's channels-last x and column
// gradients; writes the modulated columns, grad_offset and grad_mask of the
// point, and adds the corner terms into the fp32 channels-last grad_x. Five
// blocks per SM (48 registers) measured 1.5-2.5% faster than four (64): the
// kernel waits on its loads, and more warps hide more of that.
template <typename T, int VEC>
__global__ void __launch_bounds__(256, 5) sample_backward_kernel(const BwdPlan p, const T* __restrict__ xt,
                                                              const T* __restrict__ offset, const T* __restrict__ mask,
                                                              const float* __restrict__ gcol, T* __restrict__ col,
                                                              float* __restrict__ gx, T* __restrict__ goffset,
                                                              T* __restrict__ gmask, int64_t n0) {
    const int lanes = p.lanes;
    const int32_t K = p.K, P = static_cast<int32_t>(p.P), Cg = p.Cg;
    const int32_t pix = static_cast<int32_t>(blockIdx.x) * (256 / lanes) + static_cast<int32_t>(threadIdx.x) / lanes;
    const int32_t gd = static_cast<int32_t>(blockIdx.y) / K, k = static_cast<int32_t>(blockIdx.y) - gd * K;
    const int32_t n = static_cast<int32_t>(blockIdx.z);
    const int sub = threadIdx.x & (lanes - 1);
    const bool live = pix < P;
    const int64_t ng = n0 + n;
    const int64_t och = (ng * p.dg + gd) * 2 * K + 2 * k;  // the point's h-offset channel; w follows
    const int64_t mch = (ng * p.dg + gd) * K + k;
    float s_mask = 0.f, s_h = 0.f, s_w = 0.f, m = 0.f;
    if (live) {
        const int32_t ho = pix / static_cast<int32_t>(p.Wo), wo = pix - ho * static_cast<int32_t>(p.Wo);
        const int32_t i = k / static_cast<int32_t>(p.kw), j = k - i * static_cast<int32_t>(p.kw);
        const float offh = to_f(offset[och * P + pix]);
        const float offw = to_f(offset[(och + 1) * P + pix]);
        m = to_f(mask[mch * P + pix]);
        const float h = static_cast<float>(ho * p.sh - p.ph + i * p.dh) + offh;
        const float w = static_cast<float>(wo * p.sw - p.pw + j * p.dw) + offw;
        const bool inside = !(h <= -1.f || h >= static_cast<float>(p.H) || w <= -1.f || w >= static_cast<float>(p.W));
        const int32_t cbeg = gd * p.Cd, cend = cbeg + p.Cd;
        // column (gradient) element of channel c: ((n*group + g)*P + pix)*K*Cg + k*Cg + c_l
        const int64_t prow = static_cast<int64_t>(n) * p.group * P + pix;
        const int64_t kcg = static_cast<int64_t>(K) * Cg;
        if (inside) {
            const float h0f = floorf(h), w0f = floorf(w);
            const int32_t y0 = static_cast<int32_t>(h0f), x0 = static_cast<int32_t>(w0f);
            const float lh = h - h0f, lw = w - w0f, hh = 1.f - lh, hw = 1.f - lw;
            const float w00 = hh * hw, w01 = hh * lw, w10 = lh * hw, w11 = lh * lw;
            const bool v00 = y0 >= 0 && x0 >= 0, v01 = y0 >= 0 && x0 + 1 < p.W;
            const bool v10 = y0 + 1 < p.H && x0 >= 0, v11 = y0 + 1 < p.H && x0 + 1 < p.W;
            // corner (y0, x0) of image n, channels-last; only dereferenced when valid
            const int64_t a00 = ((static_cast<int64_t>(n) * p.H + y0) * p.W + x0) * p.Cin;
            const int64_t a01 = a00 + p.Cin, a10 = a00 + p.W * p.Cin, a11 = a10 + p.Cin;
            // channel c = g * Cg + cl, advanced by the lane stride without a division per step
            const int32_t cstep = lanes * VEC;
            int32_t c = cbeg + sub * VEC;
            int32_t g = c / Cg, cl = c - g * Cg;
            for (; c < cend; c += cstep) {
                const int64_t gi = (prow + static_cast<int64_t>(g) * P) * kcg + k * Cg + cl;
                float G[VEC], X00[VEC], X01[VEC], X10[VEC], X11[VEC], cv[VEC];
                load_f<float, VEC>(gcol + gi, G);
#pragma unroll
                for (int e = 0; e < VEC; ++e) X00[e] = X01[e] = X10[e] = X11[e] = 0.f;
                if (v00) load_f<T, VEC>(xt + a00 + c, X00);
                if (v01) load_f<T, VEC>(xt + a01 + c, X01);
                if (v10) load_f<T, VEC>(xt + a10 + c, X10);
                if (v11) load_f<T, VEC>(xt + a11 + c, X11);
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const float val = w00 * X00[e] + w01 * X01[e] + w10 * X10[e] + w11 * X11[e];
                    const float dvh = hw * (X10[e] - X00[e]) + lw * (X11[e] - X01[e]);
                    const float dvw = hh * (X01[e] - X00[e]) + lh * (X11[e] - X10[e]);
                    s_mask += G[e] * val;
                    s_h += G[e] * dvh;
                    s_w += G[e] * dvw;
                    cv[e] = m * val;
                }
                store_f<T, VEC>(col + gi, cv);
                if (v00) red_add<VEC>(gx + a00 + c, G, m * w00);
                if (v01) red_add<VEC>(gx + a01 + c, G, m * w01);
                if (v10) red_add<VEC>(gx + a10 + c, G, m * w10);
                if (v11) red_add<VEC>(gx + a11 + c, G, m * w11);
                for (cl += cstep; cl >= Cg; cl -= Cg) ++g;
            }
        } else {
            float zero[VEC];
#pragma unroll
            for (int e = 0; e < VEC; ++e) zero[e] = 0.f;
            const int32_t cstep = lanes * VEC;
            int32_t c = cbeg + sub * VEC;
            int32_t g = c / Cg, cl = c - g * Cg;
            for (; c < cend; c += cstep) {
                store_f<T, VEC>(col + (prow + static_cast<int64_t>(g) * P) * kcg + k * Cg + cl, zero);
                for (cl += cstep; cl >= Cg; cl -= Cg) ++g;
            }
        }
    }
    // segments are aligned groups of `lanes` threads inside one warp, and every
    // thread of the warp reaches this point
    for (int d = lanes >> 1; d > 0; d >>= 1) {
        s_mask += __shfl_xor_sync(0xffffffffu, s_mask, d);
        s_h += __shfl_xor_sync(0xffffffffu, s_h, d);
        s_w += __shfl_xor_sync(0xffffffffu, s_w, d);
    }
    if (live && sub == 0) {
        gmask[mch * P + pix] = from_f<T>(s_mask);
        goffset[och * P + pix] = from_f<T>(m * s_h);
        goffset[(och + 1) * P + pix] = from_f<T>(m * s_w);
    }
}

template <typename T>
constexpr cudaDataType_t blas_type();
template <>
constexpr cudaDataType_t blas_type<float>() { return CUDA_R_32F; }
template <>
constexpr cudaDataType_t blas_type<__half>() { return CUDA_R_16F; }
template <>
constexpr cudaDataType_t blas_type<__nv_bfloat16>() { return CUDA_R_16BF; }

size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

unsigned grid_for(int64_t total) {
    int64_t b = (total + 255) / 256;
    return static_cast<unsigned>(b < 1 ? 1 : (b > 8192 ? 8192 : b));
}

// out[b] = in[b]^T (R x C per batch entry); with zero != nullptr also clears zero[b] (fp32, out's layout),
// then returning whether it did (the element kernel leaves it to the caller).
template <typename Tin, typename Tout>
cudaError_t transpose(const Tin* in, Tout* out, int64_t R, int64_t C, int64_t batch, cudaStream_t st,
                      float* zero = nullptr, bool* zeroed = nullptr) {
    const int64_t tiles = ((R + kTransposeTile - 1) / kTransposeTile) * ((C + kTransposeTile - 1) / kTransposeTile);
    const dim3 grid(static_cast<unsigned>(tiles), static_cast<unsigned>(batch));
    constexpr int64_t kVi = 16 / sizeof(Tin), kVo = 16 / sizeof(Tout);
    // 16-byte vectors where a side is 16-bit (float32 on both sides is as fast element-wise, measured)
    // and the rows of both sides are whole vectors (the caller's buffers are 16-byte aligned)
    const bool vec = (sizeof(Tin) == 2 || sizeof(Tout) == 2) && C % kVi == 0 && R % kVo == 0 && (!zero || R % 4 == 0);
    if (vec) {
        transpose_vec_kernel<Tin, Tout><<<grid, 256, 0, st>>>(in, out, zero, R, C);
    } else {
        transpose_kernel<Tin, Tout><<<grid, 256, 0, st>>>(in, out, R, C);
    }
    if (zeroed) *zeroed = vec && zero;
    return cudaGetLastError();
}

cudaError_t blas_fail(cublasStatus_t s) {
    return s == CUBLAS_STATUS_SUCCESS ? cudaSuccess : cudaErrorUnknown;
}

// The column-gradient GEMM of one group for a chunk of nbc images on the
// tensor cores, computed as its transpose so that each epilogue warp writes
// 128 contiguous bytes per column: gcol[n][g][p][kc] (m = kc, n = p) = sum
// over o of wt[g][o][kc] * grad_out[n][g*Og + o][p]; A = wt (m = kc
// contiguous: MN-major, shared by the images), B = grad_out (n = p
// contiguous: MN-major, one per image), K = the group's Og output channels.
template <typename T>
cudaError_t column_grad_tc(const BwdPlan& p, const T* grad_out_chunk, const T* wt, float* gcol, int64_t nbc, int32_t g,
                           uint32_t* status, cudaStream_t st) {
    const int64_t es = sizeof(T), P = p.P, Og = p.Og, KCg = static_cast<int64_t>(p.K) * p.Cg;
    GemmOperand a{wt + static_cast<int64_t>(g) * Og * KCg, {KCg, Og, 1, 1}, {KCg * es, Og * KCg * es, Og * KCg * es}};
    GemmOperand b{grad_out_chunk + static_cast<int64_t>(g) * Og * P, {P, Og, 1, nbc},
                  {P * es, Og * P * es, p.Cout * P * es}};
    GemmArgs ga{};
    ga.M = static_cast<int32_t>(KCg);
    ga.N = static_cast<int32_t>(P);
    ga.kt_inner = static_cast<int32_t>((Og + 63) / 64);
    ga.kbatch = 1;
    ga.atomic = 0;
    ga.D = gcol + static_cast<int64_t>(g) * P * KCg;
    ga.ldm = 1;
    ga.ldn = KCg;
    ga.ldz = static_cast<int64_t>(p.group) * P * KCg;
    ga.status = status;
    // a short contraction (Og <= 128): 128-wide tiles, two stages, two CTAs per
    // SM; a longer one: 256-wide tiles (fewer operand re-reads per output byte),
    // four stages, one CTA per SM
    const int bn = Og > 128 ? 256 : 128;
    ga.stages = bn == 256 ? 4 : 2;
    ga.a_z = 0;  // batch = image: the weight shared, grad_out per image
    ga.b_z = 1;
    return launch_tc_gemm(p.dtype, a, true, b, true, bn, ga, static_cast<int>(nbc), 1, st);
}

// The weight-gradient GEMM of a chunk of nbc images, every group at once on
// the tensor cores, as its transpose: part[s][g][o][kc] (m = kc, n = o) = the
// sum over split s's share of the chunk's images and pixels of
// col[n][g][p][kc] * grad_out[n][g*Og + o][p]; A = col (m = kc contiguous:
// MN-major), B = grad_out (K-major in p). The contraction (images x pixels)
// is split between p.wsplits CTAs per tile, each writing its own fp32 slice;
// reduce_splits_kernel adds the slices in order (deterministic).
template <typename T>
cudaError_t weight_grad_tc(const BwdPlan& p, const T* grad_out_chunk, const T* col, float* part, int64_t nbc,
                           uint32_t* status, cudaStream_t st, int* splits_used) {
    const int64_t es = sizeof(T), P = p.P, Og = p.Og, KCg = static_cast<int64_t>(p.K) * p.Cg, G = p.group;
    GemmOperand a{col, {KCg, P, nbc, G}, {KCg * es, G * P * KCg * es, P * KCg * es}};
    GemmOperand b{grad_out_chunk, {P, Og, nbc, G}, {P * es, p.Cout * P * es, Og * P * es}};
    GemmArgs ga{};
    ga.M = static_cast<int32_t>(KCg);
    ga.N = static_cast<int32_t>(Og);
    ga.kt_inner = static_cast<int32_t>((P + 63) / 64);
    ga.kbatch = static_cast<int32_t>(nbc);
    ga.atomic = 0;
    ga.D = part;
    ga.ldm = 1;
    ga.ldn = KCg;
    ga.ldz = Og * KCg;
    ga.lds = G * Og * KCg;
    ga.status = status;
    ga.stages = 6;
    ga.a_z = 1;  // batch = group: both operands per group
    ga.b_z = 1;
    const int bn = Og > 128 ? 256 : 128;
    return launch_tc_gemm(p.dtype, a, true, b, false, bn, ga, static_cast<int>(G), p.wsplits, st, splits_used);
}

// gw[i] (+)= sum over s < splits of part[s][i], in order of s (first chunk: =),
// four consecutive elements per thread (count is a multiple of 4 on the
// tensor-core path: K*Cg is a multiple of 8).
__global__ void __launch_bounds__(256) reduce_splits_kernel(const float* __restrict__ part, float* __restrict__ gw,
                                                            int64_t count, int32_t splits, int32_t first) {
    const int64_t n4 = count / 4;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        float4 acc = first ? make_float4(0.f, 0.f, 0.f, 0.f) : reinterpret_cast<const float4*>(gw)[i];
        for (int32_t s = 0; s < splits; ++s) {
            const float4 v = reinterpret_cast<const float4*>(part + s * count)[i];
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        reinterpret_cast<float4*>(gw)[i] = acc;
    }
}

template <typename T>
cudaError_t run_backward(const BwdPlan& p, const T* x, const T* offset, const T* mask, const T* weight,
                         const T* grad_out, T* grad_x, T* grad_offset, T* grad_mask, T* grad_weight, T* grad_bias,
                         void* ws, cudaStream_t st) {
    uint8_t* base = static_cast<uint8_t*>(ws);
    T* wt = reinterpret_cast<T*>(base + p.off_wt);
    float* gw = reinterpret_cast<float*>(base + p.off_gw);
    T* xt = reinterpret_cast<T*>(base + p.off_xt);
    float* gx = reinterpret_cast<float*>(base + p.off_gx);
    float* gcol = reinterpret_cast<float*>(base + p.off_gcol);
    T* col = reinterpret_cast<T*>(base + p.off_col);
    const int64_t K = p.K, Cg = p.Cg, Og = p.Og, P = p.P, HW = p.H * p.W, KCg = K * Cg;
    cudaError_t e;

    uint32_t* status = reinterpret_cast<uint32_t*>(base + p.off_status);
    const bool tc = backward_uses_tc(p);
    BlasLease lease;
    cublasHandle_t h = nullptr;
    if (!tc) {
        if ((e = lease_blas(&lease, st, blas_workspace_in(base + p.off_blas), kBlasWorkspaceBytes)) != cudaSuccess)
            return e;
        h = lease.h;
    }
    const cublasComputeType_t ct = sizeof(T) == 4 ? CUBLAS_COMPUTE_32F_PEDANTIC : CUBLAS_COMPUTE_32F;
    const float one = 1.0f, zero = 0.0f;

    // one output channel per block through shared memory where its Cg*K weights (padded by a row)
    // fit 48 KB as fp32
    const int64_t wfl = KCg + std::max(Cg, K);
    const bool wblock = wfl <= 12288 && p.Cout <= 2147483647;
    const size_t wsmem = static_cast<size_t>(wfl) * sizeof(float);
    if (wblock)
        weight_tap_major_block_kernel<T><<<static_cast<unsigned>(p.Cout), 256, wsmem, st>>>(
            weight, wt, static_cast<int32_t>(Cg), static_cast<int32_t>(K), status);
    else
        weight_tap_major_kernel<T><<<grid_for(p.Cout * KCg), 256, 0, st>>>(weight, wt, p.Cout, Cg, K, status);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;

    for (int64_t n0 = 0; n0 < p.N; n0 += p.nb) {
        const int64_t nbc = p.N - n0 < p.nb ? p.N - n0 : p.nb;
        // 1. x of the chunk, channels-last, and the chunk's grad_x accumulator cleared (by the
        //    transpose where it takes 16-byte vectors, else by a memset)
        const bool clear = backward_clears_in_transpose(p);
        bool zeroed = false;
        if ((e = transpose<T, T>(x + n0 * p.Cin * HW, xt, p.Cin, HW, nbc, st, clear ? gx : nullptr, &zeroed)) !=
            cudaSuccess)
            return e;
        if (clear != zeroed) return cudaErrorInvalidValue;  // the two tests of the vector path agree
        if (!zeroed &&
            (e = cudaMemsetAsync(gx, 0, static_cast<size_t>(nbc * HW * p.Cin) * sizeof(float), st)) != cudaSuccess)
            return e;
        // 2. column gradients, per group: (K*Cg x P) = wt_g (K*Cg x Og) * grad_out_g (Og x P), column-major views
        for (int32_t g = 0; g < p.group; ++g) {
            if (tc) {
                if ((e = column_grad_tc<T>(p, grad_out + n0 * p.Cout * P, wt, gcol, nbc, g, status, st)) !=
                    cudaSuccess)
                    return e;
                continue;
            }
            e = blas_fail(cublasGemmStridedBatchedEx(
                h, CUBLAS_OP_N, CUBLAS_OP_T, static_cast<int>(KCg), static_cast<int>(P), static_cast<int>(Og), &one,
                wt + g * Og * KCg, blas_type<T>(), static_cast<int>(KCg), 0,
                grad_out + (n0 * p.Cout + g * Og) * P, blas_type<T>(), static_cast<int>(P), p.Cout * P, &zero,
                gcol + g * P * KCg, CUDA_R_32F, static_cast<int>(KCg), p.group * P * KCg, static_cast<int>(nbc), ct,
                CUBLAS_GEMM_DEFAULT));
            if (e != cudaSuccess) return e;
        }
        // 3. sampling backward
        {
            const int64_t per_block = 256 / p.lanes;
            const dim3 grid(static_cast<unsigned>((P + per_block - 1) / per_block), static_cast<unsigned>(p.dg * K),
                            static_cast<unsigned>(nbc));
            if (p.vec == 4)
                sample_backward_kernel<T, 4><<<grid, 256, 0, st>>>(p, xt, offset, mask, gcol, col, gx, grad_offset,
                                                                   grad_mask, n0);
            else
                sample_backward_kernel<T, 1><<<grid, 256, 0, st>>>(p, xt, offset, mask, gcol, col, gx, grad_offset,
                                                                   grad_mask, n0);
            if ((e = cudaGetLastError()) != cudaSuccess) return e;
        }
        // 4. weight gradient. Group 1: one GEMM over the chunk's images,
        //    (K*Cg x Cout) += col (K*Cg x nbc*P) * got (nbc*P x Cout), got = grad_out as [Cout][nbc][P];
        //    otherwise per image over the groups: (K*Cg x Og) += col (K*Cg x P) * grad_out^T (P x Og)
        if (tc) {
            float* part = reinterpret_cast<float*>(base + p.off_wpart);
            int used = 0;
            if ((e = weight_grad_tc<T>(p, grad_out + n0 * p.Cout * P, col, part, nbc, status, st, &used)) !=
                cudaSuccess)
                return e;
            reduce_splits_kernel<<<grid_for(p.Cout * KCg / 4), 256, 0, st>>>(part, gw, p.Cout * KCg, used,
                                                                           n0 == 0 ? 1 : 0);
            if ((e = cudaGetLastError()) != cudaSuccess) return e;
        } else if (p.group == 1) {
            T* got = reinterpret_cast<T*>(base + p.off_got);
            const int64_t row_units = (P * static_cast<int64_t>(sizeof(T))) % 16 == 0 ? P * sizeof(T) / 16 : P;
            const int64_t units = nbc * p.Cout * row_units;
            swap_image_channel_kernel<T><<<grid_for(units), 256, 0, st>>>(grad_out + n0 * p.Cout * P, got, nbc,
                                                                          p.Cout, P);
            if ((e = cudaGetLastError()) != cudaSuccess) return e;
            const float* beta = n0 == 0 ? &zero : &one;
            e = blas_fail(cublasGemmEx(h, CUBLAS_OP_N, CUBLAS_OP_N, static_cast<int>(KCg), static_cast<int>(p.Cout),
                                       static_cast<int>(nbc * P), &one, col, blas_type<T>(), static_cast<int>(KCg), got,
                                       blas_type<T>(), static_cast<int>(nbc * P), beta, gw, CUDA_R_32F,
                                       static_cast<int>(KCg), ct, CUBLAS_GEMM_DEFAULT));
            if (e != cudaSuccess) return e;
        } else {
            for (int64_t n = 0; n < nbc; ++n) {
                const float* beta = (n0 + n == 0) ? &zero : &one;
                e = blas_fail(cublasGemmStridedBatchedEx(
                    h, CUBLAS_OP_N, CUBLAS_OP_N, static_cast<int>(KCg), static_cast<int>(Og), static_cast<int>(P), &one,
                    col + n * p.group * P * KCg, blas_type<T>(), static_cast<int>(KCg), P * KCg,
                    grad_out + (n0 + n) * p.Cout * P, blas_type<T>(), static_cast<int>(P), Og * P, beta, gw,
                    CUDA_R_32F, static_cast<int>(KCg), Og * KCg, p.group, ct, CUBLAS_GEMM_DEFAULT));
                if (e != cudaSuccess) return e;
            }
        }
        // 5. grad_x of the chunk to NCHW
        if ((e = transpose<float, T>(gx, grad_x + n0 * p.Cin * HW, HW, p.Cin, nbc, st)) != cudaSuccess) return e;
    }
    if (wblock)
        weight_grad_out_block_kernel<T><<<static_cast<unsigned>(p.Cout), 256, wsmem, st>>>(
            gw, grad_weight, static_cast<int32_t>(Cg), static_cast<int32_t>(K));
    else
        weight_grad_out_kernel<T><<<grid_for(p.Cout * KCg), 256, 0, st>>>(gw, grad_weight, p.Cout, Cg, K);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (grad_bias) {
        if (P % (16 / static_cast<int64_t>(sizeof(T))) == 0)
            bias_grad_vec_kernel<T><<<static_cast<unsigned>(p.Cout), 256, 0, st>>>(grad_out, grad_bias, p.N, p.Cout,
                                                                                    P);
        else
            bias_grad_kernel<T><<<static_cast<unsigned>(p.Cout), 256, 0, st>>>(grad_out, grad_bias, p.N, p.Cout, P);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

void plan_backward(BwdPlan* p, size_t chunk_budget) {
    const size_t es = p->dtype == kF32 ? 4 : 2;
    p->vec = (p->Cg % 4 == 0 && p->Cd % 4 == 0 && p->Cin % 4 == 0) ? 4 : 1;
    // about four steps per lane: the per-point work (position, weights,
    // validity, the shuffle reduction) is shared by more channels
    const int64_t units = (p->Cd + p->vec - 1) / p->vec;
    int lanes = 1;
    while (lanes < 32 && lanes * 4 < units) lanes <<= 1;
    p->lanes = lanes;
    const size_t cols = static_cast<size_t>(p->P) * p->K * p->Cin;  // column elements of one image
    const size_t pix = static_cast<size_t>(p->H) * p->W * p->Cin;   // x elements of one image
    const bool tc = backward_uses_tc(*p);
    // the cuBLAS path's group-1 weight gradient wants grad_out re-laid [Cout][nb][P]
    const bool got = p->group == 1 && !tc;
    const size_t per_image = cols * (4 + es) + pix * (es + 4) + (got ? static_cast<size_t>(p->Cout) * p->P * es : 0);
    int64_t nb = static_cast<int64_t>(chunk_budget / (per_image ? per_image : 1));
    if (nb < 1) nb = 1;
    if (nb > p->N) nb = p->N;
    // the cuBLAS group-1 weight-gradient GEMM runs over nb * P columns (a 32-bit dimension)
    if (got && nb * p->P > 2147483647) nb = 2147483647 / p->P;
    if (nb > 65535) nb = 65535;
    p->nb = nb;
    const size_t wel = static_cast<size_t>(p->Cout) * p->K * p->Cg;
    size_t off = 0;
    p->off_status = off;
    off += 256;
    p->off_wt = off;
    off += align256(wel * es);
    p->off_gw = off;
    off += align256(wel * 4);
    p->off_xt = off;
    off += align256(nb * pix * es);
    p->off_gx = off;
    off += align256(nb * pix * 4);
    p->off_gcol = off;
    off += align256(nb * cols * 4);
    p->off_col = off;
    off += align256(nb * cols * es);
    p->off_got = off;
    if (got) off += align256(static_cast<size_t>(nb) * p->Cout * p->P * es);
    p->off_blas = off;
    if (!tc) off += kBlasRegionBytes;
    // tensor-core weight gradient: the contraction of each 128 x 128 output tile
    // split between about 160 / tiles CTAs, one fp32 slice each
    p->wsplits = 1;
    p->off_wpart = off;
    if (tc) {
        const int64_t KCg = static_cast<int64_t>(p->K) * p->Cg;
        const int64_t bn = p->Og > 128 ? 256 : 128;  // weight_grad_tc's tile width along Og
        const int64_t tiles = ((KCg + 127) / 128) * ((p->Og + bn - 1) / bn) * p->group;
        const int64_t kt_total = ((p->P + 63) / 64) * nb;
        int64_t sp = 160 / tiles;
        if (sp > kt_total) sp = kt_total;
        if (sp < 1) sp = 1;
        p->wsplits = static_cast<int32_t>(sp);
        off += align256(static_cast<size_t>(sp) * wel * 4);
    }
    p->ws_bytes = off;
}

bool backward_uses_tc(const BwdPlan& p) {
    // 16-bit I/O whose operand rows meet TMA's 16-byte rule: P and K*Cg
    // multiples of 8 elements (the caller's pointers are 16-byte aligned)
    const int64_t KCg = static_cast<int64_t>(p.K) * p.Cg;
    return p.dtype != kF32 && p.P % 8 == 0 && KCg % 8 == 0 && p.P < (int64_t(1) << 31) && KCg < (int64_t(1) << 31);
}

bool backward_clears_in_transpose(const BwdPlan& p) {
    // the x transpose takes 16-byte vectors on both sides: 16-bit I/O, H*W and Cin multiples of 8
    return p.dtype != kF32 && (p.H * p.W) % 8 == 0 && p.Cin % 8 == 0;
}

int backward_launch_count(const BwdPlan& p) {
    const int64_t chunks = (p.N + p.nb - 1) / p.nb;
    // per chunk: transpose (with a memset of grad_x unless the transpose clears it), one GEMM per
    // group, sampling backward, the weight-gradient GEMMs (tensor-core path: one GEMM and the
    // in-order sum of its split slices per chunk; cuBLAS path, group 1: a grad_out re-layout and
    // one GEMM; else one per image), transpose
    const int64_t wgrad = backward_uses_tc(p) ? 2 * chunks : (p.group == 1 ? 2 * chunks : p.N);
    const int64_t per_chunk = (backward_clears_in_transpose(p) ? 3 : 4) + p.group;
    return static_cast<int>(1 + chunks * per_chunk + wgrad + 1 + (p.has_bias ? 1 : 0));
}

cudaError_t launch_backward(const BwdPlan& p, const void* x, const void* offset, const void* mask, const void* weight,
                            const void* grad_out, void* grad_x, void* grad_offset, void* grad_mask, void* grad_weight,
                            void* grad_bias, void* ws, cudaStream_t st) {
#define MDCN_BWD_ARGS(T)                                                                                          \
    p, static_cast<const T*>(x), static_cast<const T*>(offset), static_cast<const T*>(mask),                     \
        static_cast<const T*>(weight), static_cast<const T*>(grad_out), static_cast<T*>(grad_x),                 \
        static_cast<T*>(grad_offset), static_cast<T*>(grad_mask), static_cast<T*>(grad_weight),                  \
        static_cast<T*>(grad_bias), ws, st
    switch (p.dtype) {
        case kF32: return run_backward<float>(MDCN_BWD_ARGS(float));
        case kF16: return run_backward<__half>(MDCN_BWD_ARGS(__half));
        default: return run_backward<__nv_bfloat16>(MDCN_BWD_ARGS(__nv_bfloat16));
    }
#undef MDCN_BWD_ARGS
}

}  // namespace mdcn
