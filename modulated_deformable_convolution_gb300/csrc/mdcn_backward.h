// Problem description and workspace layout of one backward call (internal;
// the public interface is include/mdcn.h). Never shared with the CPU oracle.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace mdcn {

struct BwdPlan {
    // ---- problem (section 2 layouts, section 3 attributes)
    int64_t N, Cin, H, W, Cout, kh, kw, Ho, Wo;
    int32_t sh, sw, ph, pw, dh, dw;
    int32_t group, dg;
    int32_t dtype;     // DType of every tensor
    int32_t has_bias;  // 1: grad_bias is written
    int32_t K, Cg, Og, Cd;
    int64_t P;         // Ho*Wo
    // ---- sampling-backward kernel
    int32_t vec;       // channels per lane and step: 4 when Cg, Cd and Cin are multiples of 4, else 1
    int32_t lanes;     // lanes per sampling point (power of two, <= 32)
    // ---- images per chunk: the chunk's column gradients, columns, channels-last x,
    //      fp32 grad_x accumulator (and, for group 1, grad_out as [Cout][n][P]) fit
    //      a fixed budget
    int64_t nb;
    // ---- workspace layout (byte offsets, 256-byte aligned)
    size_t off_status; // the call's device status word (bounded waits of the tensor-core GEMMs)
    size_t off_wt;    // weight, tap-major [group][Og][K][Cg] (dtype)
    size_t off_gw;    // fp32 weight gradient, same layout
    size_t off_xt;    // x of the chunk, channels-last [nb][H][W][Cin] (dtype)
    size_t off_gx;    // fp32 grad_x of the chunk, channels-last [nb][H][W][Cin]
    size_t off_gcol;  // fp32 column gradients [nb][group][P][K][Cg]
    size_t off_col;   // modulated columns [nb][group][P][K][Cg] (dtype)
    size_t off_got;   // float32, group 1 only: grad_out of the chunk as [Cout][nb][P] (dtype), so
                      // that the cuBLAS weight gradient is one GEMM over the chunk's images
    size_t off_blas;  // the call's cuBLAS workspace region (kBlasRegionBytes; float32 only)
    size_t off_wpart; // tensor-core path: fp32 weight-gradient slices [wsplits][Cout][K*Cg]
    int32_t wsplits;  // CTAs sharing one weight-gradient tile's contraction (tensor-core path)
    size_t ws_bytes;
};

// Fills nb, vec, lanes and the workspace layout of a plan whose problem
// fields are set; chunk_budget = bytes of per-chunk buffers to aim for.
void plan_backward(BwdPlan* p, size_t chunk_budget);

// Every launch of one backward call, on one stream.
cudaError_t launch_backward(const BwdPlan& p, const void* x, const void* offset, const void* mask, const void* weight,
                            const void* grad_out, void* grad_x, void* grad_offset, void* grad_mask, void* grad_weight,
                            void* grad_bias, void* ws, cudaStream_t st);

// True when the x transpose of each chunk also clears its grad_x accumulator
// (16-byte vectors: 16-bit I/O, H*W and Cin multiples of 8), so no memset is
// launched.
bool backward_clears_in_transpose(const BwdPlan& p);

// Kernel launches (and cuBLAS calls) one backward call makes.
int backward_launch_count(const BwdPlan& p);

// True when the call's contractions run on the tcgen05 GEMM (float16 and
// bfloat16 with P and K*Cg multiples of 8); false: cuBLAS (float32 products).
bool backward_uses_tc(const BwdPlan& p);

}  // namespace mdcn
