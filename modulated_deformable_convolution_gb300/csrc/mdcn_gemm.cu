// Dense contractions of the backward pass on the tcgen05 tensor cores:
//   D[z][m][n] (+)= sum over k of A(m, k) * B(n, k)
// with 16-bit operands (float16 / bfloat16) and fp32 accumulation in tensor
// memory. The contraction index k runs over (kb, inner): an optional second
// dimension of the operands (images) times their 64-element k-tiles, so that
// a sum over the pixels of several images needs no re-layout.
//
// Operands come by TMA (4-D tensor maps, 128-byte swizzle) in either
// orientation: K-major (the 64 k-elements of a row contiguous: one box of
// 64 x rows) or MN-major (64 rows of m or n contiguous per k: boxes of
// 64 x 64, 8 KB apart along m or n). The shared-memory descriptors follow:
// K-major advances 32 bytes per 16-element K-step inside the swizzle atom;
// MN-major uses a leading byte offset of 8 KB between 64-element atoms and a
// stride byte offset of 1 KB between 8-row K groups, and advances 2 KB per
// K-step.
//
// Persistent CTAs, as many as are resident at once, take the work items (m
// tile, n tile, k split, batch) in turn: 6 warps. Warp 0 issues the TMA loads
// into a ring of stages, warp 1 allocates tensor memory (two accumulators)
// and issues tcgen05.mma (128 x BN per instruction, 4 per stage), warps 2-5
// read an accumulator (each its tensor-memory lane quarter) while the MMAs
// fill the other, and store or add (fp32 vector reductions) into D, or into
// their split's own slice of D when the contraction is split between CTAs.
// Every wait is bounded (the status word records a wait that gave up).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdint>

#include "mdcn_gemm.h"
#include "mdcn_ptx.cuh"

namespace mdcn {

namespace {

constexpr int kGemmThreads = 192;
constexpr int kGemmWarpTma = 0, kGemmWarpMma = 1;

__device__ __forceinline__ void tma_load_4d_elect(uint32_t dst, const void* tmap, int32_t c0, int32_t c1, int32_t c2,
                                                  int32_t c3, uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
        "%5}], [%6];\n\t}" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
        : "memory");
}

// Shared-memory descriptor, 128-byte swizzle, with explicit byte offsets.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

__device__ __forceinline__ void red_add_v4(float* p, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

// Work item w of the persistent grid: the m tile varies fastest (consecutive
// items share their B tile), then the n tile, the k split and the batch.
struct GemmWork {
    int32_t m0, n0, z, split, k_lo, k_hi;
};

template <int BN>
__device__ __forceinline__ GemmWork gemm_work(const GemmArgs& g, int64_t w) {
    GemmWork o;
    int64_t t = w;
    const int32_t mi = static_cast<int32_t>(t % g.mt);
    t /= g.mt;
    const int32_t ni = static_cast<int32_t>(t % g.nt);
    t /= g.nt;
    o.split = static_cast<int32_t>(t % g.splits);
    o.z = static_cast<int32_t>(t / g.splits);
    o.m0 = mi * 128;
    o.n0 = ni * BN;
    const int32_t kt_total = g.kt_inner * g.kbatch;
    o.k_lo = o.split * g.kt_split;
    o.k_hi = min(o.k_lo + g.kt_split, kt_total);
    return o;
}

// Persistent: CTA c takes work items c, c + gridDim.x, ... Two accumulators
// in tensor memory (2 x BN columns): the epilogue of one item overlaps the
// MMAs of the next.
template <int BN, bool AMN, bool BMN>
__global__ void __launch_bounds__(kGemmThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tb, const GemmArgs g) {
    constexpr uint32_t kABytes = 128 * 128;  // 128 rows x 64 elements x 2 bytes
    constexpr uint32_t kBBytes = BN * 128;
    constexpr uint32_t kStageBytes = kABytes + kBBytes;
    constexpr int kEpiWarpsG = 4;
    const int S = g.stages;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (sbase - raw);
    const uint32_t bar0 = sbase + static_cast<uint32_t>(S) * kStageBytes;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
    auto accf_bar = [&](int a) { return bar0 + 8u * (2 * S + a); };
    auto acce_bar = [&](int a) { return bar0 + 8u * (2 * S + 2 + a); };
    const uint32_t drain_bar = bar0 + 8u * (2 * S + 4);
    const uint32_t slot_off = bar0 + 8u * (2 * S + 5) - sbase;
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(gbase + slot_off);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + slot_off + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == kGemmWarpTma && lane == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(accf_bar(a), 1);
            mbar_init(acce_bar(a), kEpiWarpsG);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
        tma_prefetch_desc(&ta);
        tma_prefetch_desc(&tb);
    }
    if (warp == kGemmWarpMma) {
        tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), static_cast<uint32_t>(2 * BN));
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // the operands may come from the kernel launched just before this one
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (warp == kGemmWarpTma) {
        // ---------------------------------------------------------------- TMA producer
        uint32_t st = 0, ph = 0, issued = 0;
        bool ok = true;
        for (int64_t w = blockIdx.x; w < g.items && ok; w += gridDim.x) {
            const GemmWork wk = gemm_work<BN>(g, w);
            const int32_t za = g.a_z ? wk.z : 0, zb = g.b_z ? wk.z : 0;
            for (int32_t kt = wk.k_lo; kt < wk.k_hi; ++kt) {
                if (!warp_wait_bounded(empty_bar(st), ph ^ 1u, abort_flag, g.status, kSiteTmaEmpty)) {
                    ok = false;
                    break;
                }
                const uint32_t a_s = sbase + st * kStageBytes, b_s = a_s + kABytes;
                const int32_t kb = kt / g.kt_inner;
                const int32_t kc = (kt - kb * g.kt_inner) * 64;
                mbar_arrive_expect_tx_elect(full_bar(st), kStageBytes);
                if constexpr (AMN) {
#pragma unroll
                    for (int h = 0; h < 2; ++h)
                        tma_load_4d_elect(a_s + h * 8192u, &ta, wk.m0 + 64 * h, kc, kb, za, full_bar(st));
                } else {
                    tma_load_4d_elect(a_s, &ta, kc, wk.m0, kb, za, full_bar(st));
                }
                if constexpr (BMN) {
#pragma unroll
                    for (int h = 0; h < BN / 64; ++h)
                        tma_load_4d_elect(b_s + h * 8192u, &tb, wk.n0 + 64 * h, kc, kb, zb, full_bar(st));
                } else {
                    tma_load_4d_elect(b_s, &tb, kc, wk.n0, kb, zb, full_bar(st));
                }
                ++issued;
                if (++st == static_cast<uint32_t>(S)) {
                    st = 0;
                    ph ^= 1u;
                }
            }
        }
        if (!ok && lane == 0) {
            // let the copies already issued land before the CTA exits
            volatile int never = 0;
            const uint32_t first = issued > static_cast<uint32_t>(S) ? issued - S : 0;
            for (uint32_t q = first; q < issued; ++q)
                mbar_wait_bounded(full_bar(q % S), (q / S) & 1, &never, g.status, kSiteDrain, 200000000ull);
        }
    } else if (warp == kGemmWarpMma) {
        // ---------------------------------------------------------------- MMA issuer
        const uint32_t idesc = make_idesc(static_cast<uint32_t>(g.fmt), 128u, static_cast<uint32_t>(BN)) |
                               (AMN ? (1u << 15) : 0u) | (BMN ? (1u << 16) : 0u);
        uint32_t st = 0, ph = 0, i = 0;
        bool ok = true;
        for (int64_t w = blockIdx.x; w < g.items && ok; w += gridDim.x, ++i) {
            const GemmWork wk = gemm_work<BN>(g, w);
            const uint32_t acc = i & 1u, use = i >> 1;
            // the epilogue has read this accumulator's previous item
            if (!warp_wait2(acce_bar(acc), 0u, (use & 1u) ^ 1u, abort_flag, g.status, kSiteMmaFull)) break;
            tc_fence_after();
            const uint32_t d = tmem_base + acc * static_cast<uint32_t>(BN);
            for (int32_t kt = wk.k_lo; kt < wk.k_hi; ++kt) {
                if (!warp_wait2(full_bar(st), 0u, ph, abort_flag, g.status, kSiteMmaFull)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a_s = sbase + st * kStageBytes, b_s = a_s + kABytes;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t ad =
                        AMN ? desc_sw128(a_s + 2048u * kk, 8192u, 1024u) : desc_sw128(a_s + 32u * kk, 16u, 1024u);
                    const uint64_t bd =
                        BMN ? desc_sw128(b_s + 2048u * kk, 8192u, 1024u) : desc_sw128(b_s + 32u * kk, 16u, 1024u);
                    mma_f16_elect(d, ad, bd, idesc, (kt == wk.k_lo && kk == 0) ? 0u : 1u);
                }
                mma_commit_elect(empty_bar(st));
                if (++st == static_cast<uint32_t>(S)) {
                    st = 0;
                    ph ^= 1u;
                }
            }
            mma_commit_elect(accf_bar(acc));
        }
        // every MMA issued has completed before tensor memory is released
        mma_commit_elect(drain_bar);
        volatile int never = 0;
        warp_wait2(drain_bar, 0u, 0, &never, g.status, kSiteDrain, 200000000ull);
    } else {
        // ---------------------------------------------------------------- epilogue (warps 2-5)
        const int quarter = warp & 3;
        uint32_t i = 0;
        for (int64_t w = blockIdx.x; w < g.items; w += gridDim.x, ++i) {
            const GemmWork wk = gemm_work<BN>(g, w);
            const uint32_t acc = i & 1u, use = i >> 1;
            if (!warp_wait_bounded(accf_bar(acc), use & 1u, abort_flag, g.status, kSiteEpilogue) || *abort_flag)
                break;
            tc_fence_after();
            const int32_t r = wk.m0 + quarter * 32 + lane;
            float* drow = g.D + static_cast<int64_t>(wk.split) * g.lds + static_cast<int64_t>(wk.z) * g.ldz +
                          static_cast<int64_t>(r) * g.ldm;
            const uint32_t tl = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * static_cast<uint32_t>(BN);
#pragma unroll 1
            for (int c16 = 0; c16 < BN; c16 += 16) {
                const int32_t nb = wk.n0 + c16;
                if (nb >= g.N) break;
                float v[16];
                tmem_ld16(tl + static_cast<uint32_t>(c16), v);
                if (r >= g.M) continue;
                float* dp = drow + static_cast<int64_t>(nb) * g.ldn;
                // ldm = 1: the warp's 32 rows are 32 consecutive floats of each column
                // (one 128-byte line per store); ldn = 1: 16-byte vectors along the row
                const bool vec = g.ldn == 1 && nb + 16 <= g.N && (reinterpret_cast<uintptr_t>(dp) & 15u) == 0;
                if (vec) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        if (g.atomic)
                            red_add_v4(dp + 4 * q, v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                        else
                            *reinterpret_cast<float4*>(dp + 4 * q) =
                                make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        if (nb + e < g.N) {
                            float* de = dp + static_cast<int64_t>(e) * g.ldn;
                            if (g.atomic)
                                atomicAdd(de, v[e]);
                            else
                                *de = v[e];
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acce_bar(acc));
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kGemmWarpMma) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, static_cast<uint32_t>(2 * BN));
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
    }();
    return fn;
}

// 4-D tensor map of a 16-bit operand with a 64 x rows box (128-byte swizzle).
bool encode_operand(CUtensorMap* m, const GemmOperand& op, uint32_t box_rows, int dtype) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[4], strides[3];
    for (int i = 0; i < 4; ++i) dims[i] = static_cast<cuuint64_t>(op.dims[i]);
    for (int i = 0; i < 3; ++i) strides[i] = static_cast<cuuint64_t>(op.strides[i]);
    const cuuint32_t box[4] = {64u, box_rows, 1u, 1u};
    const cuuint32_t es[4] = {1u, 1u, 1u, 1u};
    const CUtensorMapDataType t = dtype == kBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    return enc(m, t, 4, const_cast<void*>(op.base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, bool AMN, bool BMN>
cudaError_t launch_t(const CUtensorMap& ta, const CUtensorMap& tb, GemmArgs g, cudaStream_t st) {
    // as many of the requested stages as the per-CTA shared-memory limit holds
    constexpr int kStage = 128 * 128 + BN * 128, kFixed = 1024 + 256;
    const int fit = (227 * 1024 - kFixed) / kStage;
    if (g.stages > fit) g.stages = fit;
    if (g.stages < 2) return cudaErrorInvalidValue;
    int smem = g.stages * kStage + kFixed;
    cudaError_t e;
    // persistent grid: the CTAs that are resident at once, at most one per work
    // item. Each CTA holds 2 x BN tensor-memory columns of the SM's 512, so the
    // shared memory asked for is raised until no more CTAs than that fit on an
    // SM (a further CTA's allocation would wait for one of them to finish)
    int dev = 0, sms = 0, per_sm_smem = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&per_sm_smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) != cudaSuccess)
        return e;
    const int tmem_fit = 512 / (2 * BN);
    const int floor_smem = per_sm_smem / (tmem_fit + 1) + 1;  // tmem_fit + 1 CTAs (+1 KB reserve each) cannot fit
    if (smem < floor_smem && floor_smem <= 227 * 1024) smem = floor_smem;
    int per_sm = per_sm_smem / (smem + 1024);  // 1 KB reserved per CTA
    if (per_sm > tmem_fit) per_sm = tmem_fit;
    if (per_sm < 1) per_sm = 1;
    auto kern = tc_gemm_kernel<BN, AMN, BMN>;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess) return e;
    int64_t grid = static_cast<int64_t>(sms) * per_sm;
    if (grid > g.items) grid = g.items;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, ta, tb, g);
    return e == cudaSuccess ? cudaGetLastError() : e;
}

}  // namespace

bool gemm_operand_ok(const GemmOperand& op) {
    if ((reinterpret_cast<uintptr_t>(op.base) & 15u) != 0) return false;
    for (int i = 0; i < 4; ++i)
        if (op.dims[i] < 1 || op.dims[i] > (int64_t(1) << 32)) return false;
    for (int i = 0; i < 3; ++i)
        if (op.strides[i] % 16 != 0 || op.strides[i] >= (int64_t(1) << 40)) return false;
    return true;
}

cudaError_t launch_tc_gemm(int dtype, const GemmOperand& a, bool a_mn, const GemmOperand& b, bool b_mn, int bn,
                           GemmArgs g, int batches, int splits, cudaStream_t st, int* splits_used) {
    if (dtype == kF32 || !(bn == 128 || bn == 256) || !gemm_operand_ok(a) || !gemm_operand_ok(b))
        return cudaErrorInvalidValue;
    CUtensorMap ta, tb;
    // A rows: 128 (K-major box 64 x 128) or 64 (MN-major boxes 64 x 64); B likewise with BN
    if (!encode_operand(&ta, a, a_mn ? 64u : 128u, dtype)) return cudaErrorInvalidValue;
    if (!encode_operand(&tb, b, b_mn ? 64u : static_cast<uint32_t>(bn), dtype)) return cudaErrorInvalidValue;
    g.fmt = dtype == kBF16 ? 1 : 0;
    g.mt = (g.M + 127) / 128;
    g.nt = (g.N + bn - 1) / bn;
    const int64_t kt_total = static_cast<int64_t>(g.kt_inner) * g.kbatch;
    if (splits < 1) splits = 1;
    g.kt_split = static_cast<int32_t>((kt_total + splits - 1) / splits);
    splits = static_cast<int>((kt_total + g.kt_split - 1) / g.kt_split);
    if (splits > 1 && !g.atomic && g.lds == 0) return cudaErrorInvalidValue;
    if (splits_used) *splits_used = splits;
    if (batches < 1) return cudaErrorInvalidValue;
    g.splits = splits;
    g.items = static_cast<int64_t>(g.mt) * g.nt * splits * batches;
    if (g.items > (int64_t(1) << 40)) return cudaErrorInvalidValue;
    if (bn == 128) {
        if (a_mn && b_mn) return launch_t<128, true, true>(ta, tb, g, st);
        if (!a_mn && b_mn) return launch_t<128, false, true>(ta, tb, g, st);
        if (a_mn && !b_mn) return launch_t<128, true, false>(ta, tb, g, st);
        return launch_t<128, false, false>(ta, tb, g, st);
    }
    if (a_mn && b_mn) return launch_t<256, true, true>(ta, tb, g, st);
    if (!a_mn && b_mn) return launch_t<256, false, true>(ta, tb, g, st);
    if (a_mn && !b_mn) return launch_t<256, true, false>(ta, tb, g, st);
    return launch_t<256, false, false>(ta, tb, g, st);
}

}  // namespace mdcn
