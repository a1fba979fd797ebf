// Ablation path: the page's own two-stage design ("TensorRT plugin
// walkthrough: modulatedDeformConvPlugin", section 5): a deformable im2col
// kernel writes the column matrix to device memory (step 1), a GEMM per
// group contracts it with the weight (step 2, here one strided-batched
// cuBLAS call per group with fp32 accumulation), and a third kernel adds the
// bias (step 3). Kept only to compare against the fused kernel.
#include <cublas_v2.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <mutex>

#include "mdcn_launch.h"

namespace mdcn {

namespace {

__device__ __forceinline__ float ld_f(const float* p) { return *p; }
__device__ __forceinline__ float ld_f(const __half* p) { return __half2float(*p); }
__device__ __forceinline__ float ld_f(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st_f(float* p, float v) { *p = v; }
__device__ __forceinline__ void st_f(__half* p, float v) { *p = __float2half_rn(v); }
__device__ __forceinline__ void st_f(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// One thread per (n, c, output pixel); loops over the taps and writes
// cols[n][c*K + k][p] = mask * bilinear sample (fp32 math, stored as T).
template <typename T>
__global__ void __launch_bounds__(256) deform_im2col_kernel(const T* __restrict__ x, const T* __restrict__ offset,
                                                            const T* __restrict__ mask, T* __restrict__ cols, Plan pl) {
    const int64_t total = pl.N * pl.Cin * pl.P;
    for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
         e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t hw = e % pl.P;
        const int64_t nc = e / pl.P;
        const int64_t c = nc % pl.Cin;
        const int64_t n = nc / pl.Cin;
        const int64_t ho = hw / pl.Wo, wo = hw - ho * pl.Wo;
        const int64_t gd = c / pl.Cd;
        const T* plane = x + (n * pl.Cin + c) * pl.H * pl.W;
        const int64_t K = pl.K;
        T* col = cols + (n * pl.Cin + c) * K * pl.P + hw;
        for (int64_t k = 0; k < K; ++k) {
            const int64_t i = k / pl.kw, j = k - (k / pl.kw) * pl.kw;
            const int64_t och = gd * 2 * K + 2 * k;
            const float dhv = ld_f(offset + ((n * 2 * pl.dg * K + och) * pl.P + hw));
            const float dwv = ld_f(offset + ((n * 2 * pl.dg * K + och + 1) * pl.P + hw));
            const float m = ld_f(mask + ((n * pl.dg * K + gd * K + k) * pl.P + hw));
            const float h = static_cast<float>(ho * pl.sh - pl.ph + i * pl.dh) + dhv;
            const float w = static_cast<float>(wo * pl.sw - pl.pw + j * pl.dw) + dwv;
            float val = 0.0f;
            if (h > -1.0f && h < static_cast<float>(pl.H) && w > -1.0f && w < static_cast<float>(pl.W)) {
                const float h0f = floorf(h), w0f = floorf(w);
                const int64_t y0 = static_cast<int64_t>(h0f), x0 = static_cast<int64_t>(w0f);
                const float lh = h - h0f, lw = w - w0f;
                float v00 = 0.f, v01 = 0.f, v10 = 0.f, v11 = 0.f;
                if (y0 >= 0 && x0 >= 0) v00 = ld_f(plane + y0 * pl.W + x0);
                if (y0 >= 0 && x0 + 1 < pl.W) v01 = ld_f(plane + y0 * pl.W + x0 + 1);
                if (y0 + 1 < pl.H && x0 >= 0) v10 = ld_f(plane + (y0 + 1) * pl.W + x0);
                if (y0 + 1 < pl.H && x0 + 1 < pl.W) v11 = ld_f(plane + (y0 + 1) * pl.W + x0 + 1);
                val = (1.f - lh) * (1.f - lw) * v00 + (1.f - lh) * lw * v01 + lh * (1.f - lw) * v10 + lh * lw * v11;
            }
            st_f(col + k * pl.P, val * m);
        }
    }
}

template <typename T>
__global__ void __launch_bounds__(256) bias_convert_kernel(const float* __restrict__ acc, const T* __restrict__ bias,
                                                           T* __restrict__ out, int64_t total, int64_t P, int64_t Cout) {
    for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
         e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        float v = acc[e];
        if (bias) v += ld_f(bias + (e / P) % Cout);
        st_f(out + e, v);
    }
}

struct HandleCache {
    std::mutex create_mu;
    std::mutex use_mu[64];
    cublasHandle_t h[64] = {};
};

HandleCache& handle_cache() {
    static HandleCache cache;
    return cache;
}

}  // namespace

// The current device's cuBLAS handle (one per device, created on first use),
// leased for one call: the lease holds the handle's lock until it is
// destroyed, and binds the handle to the call's stream and to the call's own
// workspace region. So calls from other threads neither change the stream
// under this call's GEMMs nor share cuBLAS scratch with it on the GPU.
cudaError_t lease_blas(BlasLease* lease, cudaStream_t st, void* blas_ws, size_t blas_ws_bytes) {
    HandleCache& cache = handle_cache();
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(cache.create_mu);
        if (!cache.h[dev]) {
            cublasHandle_t h = nullptr;
            if (cublasCreate(&h) != CUBLAS_STATUS_SUCCESS) return cudaErrorNotSupported;
            cache.h[dev] = h;
        }
    }
    lease->lock = std::unique_lock<std::mutex>(cache.use_mu[dev]);
    lease->h = cache.h[dev];
    // cublasSetStream resets the workspace, so the workspace is set after it
    if (cublasSetStream(lease->h, st) != CUBLAS_STATUS_SUCCESS) return cudaErrorUnknown;
    if (cublasSetWorkspace(lease->h, blas_ws, blas_ws_bytes) != CUBLAS_STATUS_SUCCESS) return cudaErrorUnknown;
    return cudaSuccess;
}

namespace {

template <typename T>
constexpr cudaDataType_t cuda_type();
template <>
constexpr cudaDataType_t cuda_type<float>() { return CUDA_R_32F; }
template <>
constexpr cudaDataType_t cuda_type<__half>() { return CUDA_R_16F; }
template <>
constexpr cudaDataType_t cuda_type<__nv_bfloat16>() { return CUDA_R_16BF; }

size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

// Workspace of the ablation: [columns (dtype)][fp32 GEMM output][cuBLAS workspace]
size_t im2col_blas_offset(const Plan& pl) {
    const size_t el = pl.dtype == kF32 ? 4 : 2;
    return align256(static_cast<size_t>(pl.N * pl.Cin * pl.K * pl.P) * el) +
           align256(static_cast<size_t>(pl.N * pl.Cout * pl.P) * sizeof(float));
}

template <typename T>
cudaError_t run_t(const Plan& pl, const void* x, const void* offset, const void* mask, const void* weight,
                  const void* bias, void* out, void* ws, cudaStream_t st) {
    uint8_t* base = static_cast<uint8_t*>(ws);
    T* cols = reinterpret_cast<T*>(base);
    float* acc = reinterpret_cast<float*>(base + align256(static_cast<size_t>(pl.N * pl.Cin * pl.K * pl.P) * sizeof(T)));
    {
        const int64_t total = pl.N * pl.Cin * pl.P;
        int64_t blocks = (total + 255) / 256;
        if (blocks > 65536) blocks = 65536;
        deform_im2col_kernel<T><<<static_cast<unsigned>(blocks), 256, 0, st>>>(
            static_cast<const T*>(x), static_cast<const T*>(offset), static_cast<const T*>(mask), cols, pl);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    BlasLease lease;
    if (cudaError_t le = lease_blas(&lease, st, blas_workspace_in(base + im2col_blas_offset(pl)), kBlasWorkspaceBytes); le != cudaSuccess)
        return le;
    cublasHandle_t h = lease.h;
    const float one = 1.0f, zero = 0.0f;
    const int64_t CgK = static_cast<int64_t>(pl.Cg) * pl.K;
    const cublasComputeType_t ct = (sizeof(T) == 4) ? CUBLAS_COMPUTE_32F_PEDANTIC : CUBLAS_COMPUTE_32F;
    for (int32_t g = 0; g < pl.group; ++g) {
        // column-major view: out_g^T (P x Og) = cols_g^T (P x CgK) * W_g^T (CgK x Og)
        const T* A = cols + static_cast<int64_t>(g) * CgK * pl.P;
        const T* B = static_cast<const T*>(weight) + static_cast<int64_t>(g) * pl.Og * CgK;
        float* C = acc + static_cast<int64_t>(g) * pl.Og * pl.P;
        cublasStatus_t s = cublasGemmStridedBatchedEx(
            h, CUBLAS_OP_N, CUBLAS_OP_N, static_cast<int>(pl.P), pl.Og, static_cast<int>(CgK), &one, A,
            cuda_type<T>(), static_cast<int>(pl.P), pl.Cin * pl.K * pl.P, B, cuda_type<T>(), static_cast<int>(CgK), 0,
            &zero, C, CUDA_R_32F, static_cast<int>(pl.P), pl.Cout * pl.P, static_cast<int>(pl.N), ct,
            CUBLAS_GEMM_DEFAULT);
        if (s != CUBLAS_STATUS_SUCCESS) return cudaErrorUnknown;
    }
    {
        const int64_t total = pl.N * pl.Cout * pl.P;
        int64_t blocks = (total + 255) / 256;
        if (blocks > 65536) blocks = 65536;
        bias_convert_kernel<T><<<static_cast<unsigned>(blocks), 256, 0, st>>>(acc, static_cast<const T*>(bias),
                                                                            static_cast<T*>(out), total, pl.P, pl.Cout);
    }
    return cudaGetLastError();
}

}  // namespace

size_t im2col_workspace_bytes(const Plan& pl) { return im2col_blas_offset(pl) + kBlasRegionBytes; }

cudaError_t launch_im2col_gemm(const Plan& pl, const void* x, const void* offset, const void* mask,
                               const void* weight, const void* bias, void* out, void* ws, cudaStream_t st) {
    switch (pl.dtype) {
        case kF32: return run_t<float>(pl, x, offset, mask, weight, bias, out, ws, st);
        case kF16: return run_t<__half>(pl, x, offset, mask, weight, bias, out, ws, st);
        default: return run_t<__nv_bfloat16>(pl, x, offset, mask, weight, bias, out, ws, st);
    }
}

}  // namespace mdcn
