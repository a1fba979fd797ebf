// Layout-prep kernels of the fused path:
//   x      [N, Cin, H, W]      -> xt [N, H, W, Cp]   (channels-last, units padded)
//   weight [Cout, Cg, kh, kw]  -> wp [R, KP]         (K-major in the fused K order)
// For float32 the packed weight holds two row blocks: rows [0, Cout) the
// tf32-rounded weight (hi) and rows [Cout, 2*Cout) the remainder (lo), the
// operands of the split-TF32 contraction.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "mdcn_layout.cuh"
#include "mdcn_launch.h"
#include "mdcn_ptx.cuh"

namespace mdcn {

namespace {

template <typename T>
__device__ __forceinline__ T zero_of();
template <>
__device__ __forceinline__ float zero_of<float>() { return 0.0f; }
template <>
__device__ __forceinline__ __half zero_of<__half>() { return __float2half_rn(0.0f); }
template <>
__device__ __forceinline__ __nv_bfloat16 zero_of<__nv_bfloat16>() { return __float2bfloat16_rn(0.0f); }

// One block transposes a 32 (w) x 32 (padded channel) tile of one (n, h) row;
// block (0, 0) also clears the device status word.
template <typename T>
__global__ void __launch_bounds__(256) nhwc_pad_kernel(const T* __restrict__ x, T* __restrict__ xt,
                                                       uint32_t* __restrict__ status, int64_t Cin, int64_t H,
                                                       int64_t W, int64_t Cp, int32_t U, int32_t UP, int64_t wtiles) {
    __shared__ T tile[32][33];
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0 && threadIdx.y == 0) *status = 0u;
    const int64_t bx = blockIdx.x;
    const int64_t nh = bx / wtiles;          // n*H + h
    const int64_t w0 = (bx - nh * wtiles) * 32;
    const int64_t n = nh / H;
    const int64_t h = nh - n * H;
    const int64_t pc0 = static_cast<int64_t>(blockIdx.y) * 32;
    const int tx = threadIdx.x, ty = threadIdx.y;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t pc = pc0 + ty + 8 * i;
        const int64_t w = w0 + tx;
        T v = zero_of<T>();
        if (pc < Cp && w < W) {
            const int64_t unit = pc / UP;
            const int64_t within = pc - unit * UP;
            if (within < U) {
                const int64_t c = unit * U + within;
                v = x[((n * Cin + c) * H + h) * W + w];
            }
        }
        tile[ty + 8 * i][tx] = v;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t w = w0 + ty + 8 * i;
        const int64_t pc = pc0 + tx;
        if (w < W && pc < Cp) xt[(nh * W + w) * Cp + pc] = tile[tx][ty + 8 * i];
    }
}

template <typename T>
__device__ __forceinline__ float load_f(const T* p);
template <>
__device__ __forceinline__ float load_f<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float load_f<__half>(const __half* p) { return __half2float(*p); }
template <>
__device__ __forceinline__ float load_f<__nv_bfloat16>(const __nv_bfloat16* p) { return __bfloat162float(*p); }

// Packs the weight into the fused kernel's K order (zero pad included).
template <typename T>
__global__ void __launch_bounds__(256) pack_weight_kernel(const T* __restrict__ weight, T* __restrict__ wp, Plan pl) {
    const int64_t rows = pl.Cout * (pl.dtype == kF32 ? 2 : 1);
    const int64_t total = pl.wp_rows * pl.KP;
    for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
         e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = e / pl.KP;
        const int64_t kk = e - r * pl.KP;
        const int64_t o = r % pl.Cout;
        const bool lo_half = r >= pl.Cout;
        const int32_t kt = static_cast<int32_t>(kk / pl.BKc);
        const int32_t ci = static_cast<int32_t>(kk - static_cast<int64_t>(kt) * pl.BKc);
        const KTile t = decode_ktile(kt, pl.K, pl.nch);
        const int32_t within = t.ch * pl.BKc + ci;  // channel within the unit
        T v = zero_of<T>();
        if (within < pl.U && r < rows) {
            const int64_t cl = static_cast<int64_t>(t.ul) * pl.U + within;  // channel within the group
            const T* src = weight + (o * pl.Cg + cl) * pl.K + t.tap;
            if constexpr (sizeof(T) == 4) {
                const float f = load_f<T>(src);
                const float hi = to_tf32(f);
                v = lo_half ? (f - hi) : hi;
            } else {
                v = *src;
            }
        }
        wp[e] = v;
    }
}

}  // namespace

template <typename T>
static cudaError_t prep_input_t(const Plan& pl, const void* x, void* ws, cudaStream_t st) {
    uint8_t* base = static_cast<uint8_t*>(ws);
    uint32_t* status = reinterpret_cast<uint32_t*>(base);
    T* xt = reinterpret_cast<T*>(base + pl.off_xt);
    const int64_t wtiles = (pl.W + 31) / 32;
    dim3 grid(static_cast<unsigned>(pl.N * pl.H * wtiles), static_cast<unsigned>((pl.Cp + 31) / 32));
    nhwc_pad_kernel<T><<<grid, dim3(32, 8), 0, st>>>(static_cast<const T*>(x), xt, status, pl.Cin, pl.H, pl.W, pl.Cp,
                                                     pl.U, pl.UP, wtiles);
    return cudaGetLastError();
}

template <typename T>
static cudaError_t pack_weight_t(const Plan& pl, const void* weight, void* ws, cudaStream_t st) {
    uint8_t* base = static_cast<uint8_t*>(ws);
    T* wp = reinterpret_cast<T*>(base + pl.off_wp);
    const int64_t total = pl.wp_rows * pl.KP;
    int64_t blocks = (total + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    pack_weight_kernel<T><<<static_cast<unsigned>(blocks), 256, 0, st>>>(static_cast<const T*>(weight), wp, pl);
    return cudaGetLastError();
}

cudaError_t launch_prep_input(const Plan& pl, const void* x, void* ws, cudaStream_t st) {
    switch (pl.dtype) {
        case kF32: return prep_input_t<float>(pl, x, ws, st);
        case kF16: return prep_input_t<__half>(pl, x, ws, st);
        default: return prep_input_t<__nv_bfloat16>(pl, x, ws, st);
    }
}

cudaError_t launch_pack_weight(const Plan& pl, const void* weight, void* ws, cudaStream_t st) {
    switch (pl.dtype) {
        case kF32: return pack_weight_t<float>(pl, weight, ws, st);
        case kF16: return pack_weight_t<__half>(pl, weight, ws, st);
        default: return pack_weight_t<__nv_bfloat16>(pl, weight, ws, st);
    }
}

}  // namespace mdcn
