// Kernel launchers of libmdcn (internal; the public interface is include/mdcn.h).
#pragma once

#include <cublas_v2.h>
#include <cuda_runtime.h>

#include <mutex>

#include "mdcn_plan.h"

namespace mdcn {

// Layout prep of the fused path into the workspace: x -> channels-last
// (also clears the workspace status word), weight -> packed K-major.
cudaError_t launch_prep_input(const Plan& pl, const void* x, void* ws, cudaStream_t st);
cudaError_t launch_pack_weight(const Plan& pl, const void* weight, void* ws, cudaStream_t st);
// Both of the above, in one launch where the shape allows; that launch also
// prefetches offset and mask (bytes each) into L2 for the fused kernel.
cudaError_t launch_prep_both(const Plan& pl, const void* x, const void* weight, const void* offset,
                             size_t offset_bytes, const void* mask, size_t mask_bytes, void* ws, cudaStream_t st);

// The fused sampling + gather + contraction + bias kernel (reads offset, mask
// and the two workspace products of launch_prep_input and
// launch_pack_weight); tiles split between CTAs are finished inside it. A
// plan with pl.plain set is an ordinary convolution and reads no offset or
// mask (both may be null).
cudaError_t launch_fused(const Plan& pl, const void* offset, const void* mask, const void* bias, void* out, void* ws,
                         cudaStream_t st);

// The direct CUDA-core forward (mdcn_direct.cu) of plans with pl.direct: one
// launch, x read in NCHW, no workspace beyond the status word (which it
// clears). Groups of at most kDirectMaxOg output channels; a thread takes
// direct_groups_per_thread(Og) groups, whose fp32 weights (that many times
// Og * Cg * K * 4 bytes) must fit kDirectMaxSmem.
constexpr int kDirectMaxOg = 32;
// The depthwise channels-last variant (Plan::direct_cl): its weights [K][128]
// and output tile [128][33] in fp32 shared memory stay under 48 KB.
constexpr int kDirectClMaxTaps = 49;
constexpr int64_t kDirectMaxSmem = 96 * 1024;
inline int direct_og_bucket(int64_t og) { return og <= 1 ? 1 : (og <= 4 ? 4 : (og <= 16 ? 16 : kDirectMaxOg)); }
inline int direct_groups_per_thread(int64_t og) {
    const int b = direct_og_bucket(og);
    return b >= 16 ? 1 : 16 / b;
}
cudaError_t launch_direct(const Plan& pl, const void* x, const void* offset, const void* mask, const void* weight,
                          const void* bias, void* out, void* ws, cudaStream_t st);

// The pack form's split of the front end's output om [N, c_off + c_mask, P]
// (P = pl.P, N = pl.N, dtype = pl.dtype): channels [0, c_off) copied to offset
// [N, c_off, P], channels [c_off, c_off + c_mask) through the logistic sigmoid
// to mask [N, c_mask, P].
cudaError_t launch_split_offset_mask(const Plan& pl, const void* om, void* offset, void* mask, int64_t c_off,
                                     int64_t c_mask, cudaStream_t st);

// Dynamic shared memory the fused kernel may use on this device (set once).
cudaError_t prepare_fused_attributes(int dtype, int smem_bytes);

// cuBLAS workspace that every call with library GEMMs (the ablation, the
// backward) carves out of its caller's workspace; the region reserved for it
// holds 256 bytes more, so that a 256-byte aligned start (cuBLAS's rule) fits
// in a workspace that is only 16-byte aligned.
constexpr size_t kBlasWorkspaceBytes = size_t(32) << 20;
constexpr size_t kBlasRegionBytes = kBlasWorkspaceBytes + 256;
inline void* blas_workspace_in(void* region) {
    return reinterpret_cast<void*>((reinterpret_cast<uintptr_t>(region) + 255) & ~static_cast<uintptr_t>(255));
}

// The current device's cuBLAS handle, locked and bound to one call's stream
// and cuBLAS workspace (256-byte aligned) until the lease is destroyed.
struct BlasLease {
    std::unique_lock<std::mutex> lock;
    cublasHandle_t h = nullptr;
};
cudaError_t lease_blas(BlasLease* lease, cudaStream_t st, void* blas_ws, size_t blas_ws_bytes);

// Ablation: deformable im2col -> cuBLAS GEMM per group -> bias/convert.
size_t im2col_workspace_bytes(const Plan& pl);
cudaError_t launch_im2col_gemm(const Plan& pl, const void* x, const void* offset, const void* mask,
                               const void* weight, const void* bias, void* out, void* ws, cudaStream_t st);

// Bounded-wait self-test kernel.
cudaError_t launch_wait_selftest(uint32_t* status, uint64_t limit_cycles, cudaStream_t st);

}  // namespace mdcn
