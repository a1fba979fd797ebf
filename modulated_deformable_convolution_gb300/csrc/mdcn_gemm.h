// tcgen05 GEMM of the backward pass (internal; see mdcn_gemm.cu).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "mdcn_plan.h"

namespace mdcn {

// A 16-bit operand as a 4-D strided array: dims[0] contiguous (elements),
// strides[i] = bytes between consecutive indices of dims[i + 1] (multiples of
// 16). K-major operands: dims = (k, rows, kb, z); MN-major operands: dims =
// (rows, k, kb, z); rows = m for A, n for B; kb = the contraction's second
// index (images), z = the batch.
struct GemmOperand {
    const void* base;
    int64_t dims[4];
    int64_t strides[3];
};

struct GemmArgs {
    int32_t M, N;          // extent of D along m and n
    int32_t kt_inner;      // 64-wide k-tiles per kb index (the inner k extent, rounded up)
    int32_t kbatch;        // kb indices: the contraction runs over (kb, inner k)
    int32_t atomic;        // 1: D += the product (fp32 reductions), 0: D = the product
    float* D;              // element (m, n) of batch z, split y at D + y*lds + z*ldz + m*ldm + n*ldn
    int64_t ldm, ldn, ldz, lds;
    uint32_t* status;      // device status word (a bounded wait that gave up sets bits)
    int32_t stages;        // pipeline stages (2..6)
    int32_t a_z, b_z;      // 1: the operand's dims[3] is the batch z; 0: the operand is shared by every batch
    // set by launch_tc_gemm
    int32_t fmt, mt, nt, kt_split, splits;
    int64_t items;         // work items: mt * nt * splits * batches
};

// True when the operand meets TMA's rules (16-byte aligned base and strides).
bool gemm_operand_ok(const GemmOperand& op);

// D (+)= A * B^T for every batch z < batches, the contraction split over
// `splits` CTAs, each writing (or adding into) its own slice of D at
// y * lds (lds = 0 with several splits needs atomic mode); bn = 128 or 256
// columns per tile. Float16 / bfloat16 only (dtype kF16 / kBF16).
// *splits_used (if given) receives the number of splits launched (every one
// of them has at least one k-tile): at most `splits`.
cudaError_t launch_tc_gemm(int dtype, const GemmOperand& a, bool a_mn, const GemmOperand& b, bool b_mn, int bn,
                           GemmArgs g, int batches, int splits, cudaStream_t st, int* splits_used = nullptr);

}  // namespace mdcn
