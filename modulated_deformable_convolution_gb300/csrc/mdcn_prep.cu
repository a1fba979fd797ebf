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
// the 32 channels lie inside one unit (UP is a multiple of 32), so the source
// channel needs no per-element division. Block (0, 0) also clears the device
// status word. Grid: x = (n*H + h) * wtiles + w tile, y = padded-channel tile.
template <typename T>
__global__ void __launch_bounds__(256) nhwc_pad_kernel(const T* __restrict__ x, T* __restrict__ xt,
                                                       uint32_t* __restrict__ status, int64_t Cin, int64_t HW,
                                                       int32_t W, int64_t Cp, int32_t U, int32_t UP,
                                                       int32_t wtiles) {
    __shared__ T tile[32][33];
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0 && threadIdx.y == 0) *status = 0u;
    const uint32_t bx = blockIdx.x;
    const uint32_t nh = bx / static_cast<uint32_t>(wtiles);  // n*H + h
    const int32_t w0 = static_cast<int32_t>(bx - nh * static_cast<uint32_t>(wtiles)) * 32;
    const int64_t pc0 = static_cast<int64_t>(blockIdx.y) * 32;
    const int64_t unit = pc0 / UP;
    const int32_t within0 = static_cast<int32_t>(pc0 - unit * UP);
    const int tx = threadIdx.x, ty = threadIdx.y;
    // x[n][c][h][w] = x + (n*Cin + c)*H*W + h*W + w; with nh = n*H + h:
    const int64_t n = nh / static_cast<uint64_t>(HW / W);
    const int64_t h = nh - n * (HW / W);
    const T* src = x + n * Cin * HW + h * W + w0 + tx;
    const bool wok = w0 + tx < W;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int32_t within = within0 + ty + 8 * i;
        T v = zero_of<T>();
        if (wok && within < U) v = src[(unit * U + within) * HW];
        tile[ty + 8 * i][tx] = v;
    }
    __syncthreads();
    T* dst = xt + static_cast<int64_t>(nh) * W * Cp + pc0 + tx;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int32_t w = w0 + ty + 8 * i;
        if (w < W && pc0 + tx < Cp) dst[static_cast<int64_t>(w) * Cp] = tile[tx][ty + 8 * i];
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
// Grid: x over k-tiles of one row (blockDim.x = BKc lanes per k-tile, several
// k-tiles per block), y over rows (looping when rows exceed the grid).
template <typename T>
__global__ void __launch_bounds__(256) pack_weight_kernel(const T* __restrict__ weight, T* __restrict__ wp, Plan pl) {
    const int64_t rows = pl.Cout * (pl.dtype == kF32 ? 2 : 1);
    const int32_t ktiles_per_block = 256 / pl.BKc;
    const int32_t kt = blockIdx.x * ktiles_per_block + static_cast<int32_t>(threadIdx.x) / pl.BKc;
    const int32_t ci = static_cast<int32_t>(threadIdx.x) % pl.BKc;
    if (kt >= pl.KT) return;
    const KTile t = decode_ktile(kt, pl.K, pl.nch);
    const int32_t within = t.ch * pl.BKc + ci;  // channel within the unit
    const int64_t cl = static_cast<int64_t>(t.ul) * pl.U + within;  // channel within the group
    for (int64_t r = blockIdx.y; r < pl.wp_rows; r += gridDim.y) {
        T v = zero_of<T>();
        if (within < pl.U && r < rows) {
            const bool lo_half = r >= pl.Cout;
            const int64_t o = lo_half ? r - pl.Cout : r;
            const T* src = weight + (o * pl.Cg + cl) * pl.K + t.tap;
            if constexpr (sizeof(T) == 4) {
                const float f = load_f<T>(src);
                const float hi = to_tf32(f);
                v = lo_half ? (f - hi) : hi;
            } else {
                v = *src;
            }
        }
        wp[r * pl.KP + static_cast<int64_t>(kt) * pl.BKc + ci] = v;
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
    nhwc_pad_kernel<T><<<grid, dim3(32, 8), 0, st>>>(static_cast<const T*>(x), xt, status, pl.Cin, pl.H * pl.W,
                                                     static_cast<int32_t>(pl.W), pl.Cp, pl.U, pl.UP,
                                                     static_cast<int32_t>(wtiles));
    return cudaGetLastError();
}

template <typename T>
static cudaError_t pack_weight_t(const Plan& pl, const void* weight, void* ws, cudaStream_t st) {
    uint8_t* base = static_cast<uint8_t*>(ws);
    T* wp = reinterpret_cast<T*>(base + pl.off_wp);
    const int32_t ktiles_per_block = 256 / pl.BKc;
    const unsigned gx = static_cast<unsigned>((pl.KT + ktiles_per_block - 1) / ktiles_per_block);
    const unsigned gy = static_cast<unsigned>(pl.wp_rows < 65535 ? pl.wp_rows : 65535);
    pack_weight_kernel<T><<<dim3(gx, gy), 256, 0, st>>>(static_cast<const T*>(weight), wp, pl);
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
