// Fused implicit-GEMM kernel of the modulated deformable convolution forward
// ("TensorRT plugin walkthrough: modulatedDeformConvPlugin", section 5,
// steps 1-3, done in one kernel without the column buffer).
//
// One CTA computes a tile of 128 output pixels x (nsub*BNs) output channels
// of one convolution group:
//   warp 0     TMA: weight k-tiles (128-byte swizzled, K-major) -> smem ring
//   warp 1     allocates tensor memory; lane 0 issues tcgen05.mma
//              (A = modulated columns, B = weights, D = fp32 in TMEM)
//   warps 2-9  producers: per (pixel, tap) sample descriptor (4 corner
//              validity bits, 4 bilinear weights x mask), then per k-tile the
//              4-corner gather of 128-byte channel runs of channels-last x,
//              weighted sum, written 128-byte-swizzled into the A stage;
//              afterwards the epilogue: TMEM -> registers -> +bias -> NCHW.
// Stage hand-off uses mbarriers: full (producers), tma (transaction bytes),
// empty (tcgen05.commit). Every wait is bounded (mdcn_ptx.cuh).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <mutex>

#include "mdcn_launch.h"
#include "mdcn_layout.cuh"
#include "mdcn_ptx.cuh"

namespace mdcn {

namespace {

template <int DT>
struct Elem;
template <>
struct Elem<kF32> {
    using T = float;
    static constexpr uint32_t fmt = 2;  // tf32
    static constexpr CUtensorMapDataType tma = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
};
template <>
struct Elem<kF16> {
    using T = __half;
    static constexpr uint32_t fmt = 0;
    static constexpr CUtensorMapDataType tma = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
};
template <>
struct Elem<kBF16> {
    using T = __nv_bfloat16;
    static constexpr uint32_t fmt = 1;
    static constexpr CUtensorMapDataType tma = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
};

struct FusedParams {
    const void* xt;
    const void* offset;
    const void* mask;
    const void* bias;
    void* out;
    uint32_t* status;
    Plan pl;
};

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__half v) { return __half2float(v); }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }

__device__ __forceinline__ void from_f(float v, float* d) { *d = v; }
__device__ __forceinline__ void from_f(float v, __half* d) { *d = __float2half_rn(v); }
__device__ __forceinline__ void from_f(float v, __nv_bfloat16* d) { *d = __float2bfloat16_rn(v); }

// Bilinear weight of one corner as stored in a descriptor: fp32 bits for
// float32, the 16-bit value broadcast to both halves of a pair otherwise.
__device__ __forceinline__ uint32_t wbits(float w, float*) { return __float_as_uint(w); }
__device__ __forceinline__ uint32_t wbits(float w, __half*) {
    __half2 h = __float2half2_rn(w);
    return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t wbits(float w, __nv_bfloat16*) {
    __nv_bfloat162 h = __float2bfloat162_rn(w);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

// Sample descriptor of output pixel p (linear over N*Ho*Wo), tap `tap`,
// deformable group gd (section 5 step 1): the sampling point
// (ho*sh - ph + i*dh + dh_off, wo*sw - pw + j*dw + dw_off); outside the open
// range (-1, H) x (-1, W) every weight is 0; otherwise the four corners with
// bilinear weights times the mask, a corner outside the image disabled.
// Layout (32 bytes): int64 element offset of corner (y0, x0) in the
// channels-last x, uint32 corner-valid bits, pad, 4 x weight bits.
template <typename T>
__device__ __forceinline__ void make_desc(const Plan& pl, const T* __restrict__ offset, const T* __restrict__ mask,
                                          int64_t p, int32_t tap, int32_t gd, uint32_t dst) {
    int64_t base = 0;
    uint32_t flags = 0;
    float w00 = 0.f, w01 = 0.f, w10 = 0.f, w11 = 0.f;
    if (p < pl.NP) {
        const int64_t n = p / pl.P;
        const int64_t hw = p - n * pl.P;
        const int64_t ho = hw / pl.Wo;
        const int64_t wo = hw - ho * pl.Wo;
        const int32_t i = tap / static_cast<int32_t>(pl.kw);
        const int32_t j = tap - i * static_cast<int32_t>(pl.kw);
        const int64_t K = pl.K;
        const int64_t och = static_cast<int64_t>(gd) * 2 * K + 2 * tap;
        const int64_t ostride = pl.P;
        const int64_t obase = (n * 2 * pl.dg * K + och) * ostride + hw;
        const float dhv = to_f(offset[obase]);
        const float dwv = to_f(offset[obase + ostride]);
        const float m = to_f(mask[(n * pl.dg * K + static_cast<int64_t>(gd) * K + tap) * ostride + hw]);
        const float hf = static_cast<float>(ho * pl.sh - pl.ph + static_cast<int64_t>(i) * pl.dh) + dhv;
        const float wf = static_cast<float>(wo * pl.sw - pl.pw + static_cast<int64_t>(j) * pl.dw) + dwv;
        if (hf > -1.0f && hf < static_cast<float>(pl.H) && wf > -1.0f && wf < static_cast<float>(pl.W)) {
            const float h0f = floorf(hf), w0f = floorf(wf);
            const float lh = hf - h0f, lw = wf - w0f;
            const float hh = 1.0f - lh, hw_ = 1.0f - lw;
            const int64_t y0 = static_cast<int64_t>(h0f);
            const int64_t x0 = static_cast<int64_t>(w0f);
            w00 = hh * hw_ * m;
            w01 = hh * lw * m;
            w10 = lh * hw_ * m;
            w11 = lh * lw * m;
            const bool top = y0 >= 0, bottom = y0 + 1 < pl.H, left = x0 >= 0, right = x0 + 1 < pl.W;
            flags = (top && left ? 1u : 0u) | (top && right ? 2u : 0u) | (bottom && left ? 4u : 0u) |
                    (bottom && right ? 8u : 0u);
            base = ((n * pl.H + y0) * pl.W + x0) * pl.Cp;
        }
    }
    T* tag = nullptr;
    sts128(dst, static_cast<uint32_t>(static_cast<uint64_t>(base)), static_cast<uint32_t>(static_cast<uint64_t>(base) >> 32),
           flags, 0u);
    sts128(dst + 16, wbits(w00, tag), wbits(w01, tag), wbits(w10, tag), wbits(w11, tag));
}

// 16-bit element pairs: acc = sum_c w_c * v_c on packed halves.
__device__ __forceinline__ uint32_t combine2(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3, uint32_t v0,
                                             uint32_t v1, uint32_t v2, uint32_t v3, __half*) {
    const __half2 a0 = *reinterpret_cast<const __half2*>(&w0), a1 = *reinterpret_cast<const __half2*>(&w1);
    const __half2 a2 = *reinterpret_cast<const __half2*>(&w2), a3 = *reinterpret_cast<const __half2*>(&w3);
    const __half2 b0 = *reinterpret_cast<const __half2*>(&v0), b1 = *reinterpret_cast<const __half2*>(&v1);
    const __half2 b2 = *reinterpret_cast<const __half2*>(&v2), b3 = *reinterpret_cast<const __half2*>(&v3);
    __half2 acc = __hmul2(a0, b0);
    acc = __hfma2(a1, b1, acc);
    acc = __hfma2(a2, b2, acc);
    acc = __hfma2(a3, b3, acc);
    return *reinterpret_cast<uint32_t*>(&acc);
}

__device__ __forceinline__ uint32_t combine2(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3, uint32_t v0,
                                             uint32_t v1, uint32_t v2, uint32_t v3, __nv_bfloat16*) {
    const __nv_bfloat162 a0 = *reinterpret_cast<const __nv_bfloat162*>(&w0);
    const __nv_bfloat162 a1 = *reinterpret_cast<const __nv_bfloat162*>(&w1);
    const __nv_bfloat162 a2 = *reinterpret_cast<const __nv_bfloat162*>(&w2);
    const __nv_bfloat162 a3 = *reinterpret_cast<const __nv_bfloat162*>(&w3);
    const __nv_bfloat162 b0 = *reinterpret_cast<const __nv_bfloat162*>(&v0);
    const __nv_bfloat162 b1 = *reinterpret_cast<const __nv_bfloat162*>(&v1);
    const __nv_bfloat162 b2 = *reinterpret_cast<const __nv_bfloat162*>(&v2);
    const __nv_bfloat162 b3 = *reinterpret_cast<const __nv_bfloat162*>(&v3);
    __nv_bfloat162 acc = __hmul2(a0, b0);
    acc = __hfma2(a1, b1, acc);
    acc = __hfma2(a2, b2, acc);
    acc = __hfma2(a3, b3, acc);
    return *reinterpret_cast<uint32_t*>(&acc);
}

template <int DT>
__global__ void __launch_bounds__(kFusedThreads, 1)
    fused_kernel(const __grid_constant__ CUtensorMap tmap, const FusedParams prm) {
    using T = typename Elem<DT>::T;
    constexpr bool kF32Path = (DT == kF32);
    const Plan& pl = prm.pl;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (sbase - raw);

    const int S = pl.stages;
    const uint32_t a_bytes = static_cast<uint32_t>(pl.a_bytes);
    const uint32_t b_bytes = static_cast<uint32_t>(pl.b_bytes);
    const uint32_t a0 = sbase;
    const uint32_t b0 = sbase + S * a_bytes;
    const uint32_t d0 = b0 + S * b_bytes;
    const uint32_t bar0 = d0 + static_cast<uint32_t>(pl.desc_bytes);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto tma_bar = [&](int s) { return bar0 + 8u * (S + s); };
    auto empty_bar = [&](int s) { return bar0 + 8u * (2 * S + s); };
    const uint32_t acc_bar = bar0 + 8u * (3 * S);
    const uint32_t slot_off = (bar0 - sbase) + 8u * (3 * S + 1);
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(gbase + slot_off);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + slot_off + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t m0 = static_cast<int64_t>(blockIdx.x) * kTileM;
    const int32_t nt = blockIdx.y;
    const int32_t g = blockIdx.z;
    const int32_t ncol0 = nt * pl.nsub * pl.BNs;  // first output channel (within the group) of this tile
    const int32_t KT = pl.KT;

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), kGatherWarps);
            mbar_init(tma_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        mbar_init(acc_bar, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
        tma_prefetch_desc(&tmap);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), static_cast<uint32_t>(pl.tmem_cols));
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const int32_t row0 = g * pl.Og + ncol0;
            const uint32_t sub_bytes = static_cast<uint32_t>(pl.BNs) * 128u;
            const uint32_t half_bytes = sub_bytes * pl.nsub;
            int32_t issued = 0;
            for (int32_t kt = 0; kt < KT; ++kt) {
                const int s = kt % S;
                const uint32_t ph = (kt / S) & 1;
                if (!mbar_wait_bounded(empty_bar(s), ph ^ 1u, abort_flag, prm.status, kSiteTmaEmpty)) break;
                mbar_arrive_expect_tx(tma_bar(s), b_bytes);
                const uint32_t dst = b0 + s * b_bytes;
#pragma unroll 1
                for (int h = 0; h < (kF32Path ? 2 : 1); ++h)
#pragma unroll 1
                    for (int j = 0; j < pl.nsub; ++j)
                        tma_load_2d(dst + h * half_bytes + j * sub_bytes, &tmap, kt * pl.BKc,
                                    row0 + h * static_cast<int32_t>(pl.Cout) + j * pl.BNs, tma_bar(s));
                issued = kt + 1;
            }
            if (*abort_flag) {
                // Let the copies already issued land before the CTA exits.
                const int32_t first = issued > S ? issued - S : 0;
                for (int32_t kt = first; kt < issued; ++kt) {
                    volatile int never = 0;
                    mbar_wait_bounded(tma_bar(kt % S), (kt / S) & 1, &never, prm.status, kSiteDrain, 100000000ull);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = make_idesc(Elem<DT>::fmt, kTileM, static_cast<uint32_t>(pl.BNs));
            const uint32_t sub_bytes = static_cast<uint32_t>(pl.BNs) * 128u;
            const uint32_t half_bytes = sub_bytes * pl.nsub;
            for (int32_t kt = 0; kt < KT; ++kt) {
                const int s = kt % S;
                const uint32_t ph = (kt / S) & 1;
                if (!mbar_wait_bounded(full_bar(s), ph, abort_flag, prm.status, kSiteMmaFull)) break;
                if (!mbar_wait_bounded(tma_bar(s), ph, abort_flag, prm.status, kSiteMmaTma)) break;
                tc_fence_after();
                const uint32_t a_s = a0 + s * a_bytes;
                const uint32_t b_s = b0 + s * b_bytes;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {  // 4 MMA K-steps of 32 bytes per 128-byte k-tile
                    const uint64_t adesc = smem_desc_sw128(a_s + kk * 32);
#pragma unroll 1
                    for (int j = 0; j < pl.nsub; ++j) {
                        const uint32_t d = tmem_base + static_cast<uint32_t>(j * pl.BNs);
                        const uint64_t bdesc = smem_desc_sw128(b_s + j * sub_bytes + kk * 32);
                        const uint32_t accum = (kt > 0 || kk > 0) ? 1u : 0u;
                        if constexpr (kF32Path) {
                            const uint64_t adesc_lo = smem_desc_sw128(a_s + kTileM * 128 + kk * 32);
                            const uint64_t bdesc_lo = smem_desc_sw128(b_s + half_bytes + j * sub_bytes + kk * 32);
                            mma_tf32(d, adesc, bdesc, idesc, accum);
                            mma_tf32(d, adesc, bdesc_lo, idesc, 1u);
                            mma_tf32(d, adesc_lo, bdesc, idesc, 1u);
                        } else {
                            mma_f16(d, adesc, bdesc, idesc, accum);
                        }
                    }
                }
                mma_commit(empty_bar(s));
            }
            mma_commit(acc_bar);  // always: the epilogue waits on it
        }
    } else {
        // ------------------------------------------------------------ producers
        const int pw = warp - 2;
        const uint32_t dc = d0 + static_cast<uint32_t>(pw) * (kRowsPerWarp * kTapBlock * kDescBytes);
        const T* __restrict__ xt = static_cast<const T*>(prm.xt);
        const T* __restrict__ offset = static_cast<const T*>(prm.offset);
        const T* __restrict__ mask = static_cast<const T*>(prm.mask);
        const int q = lane & 7;       // 16-byte column chunk of the 128-byte k-tile row
        const int rsub = lane >> 3;   // row within a group of 4
        const int64_t Cp = pl.Cp;
        const int64_t coff[4] = {0, Cp, pl.W * Cp, (pl.W + 1) * Cp};
        constexpr int kVec = 16 / sizeof(T);  // elements per 16-byte vector
        bool ok = true;
        for (int32_t kt = 0; kt < KT && ok; ++kt) {
            const KTile t = decode_ktile(kt, pl.K, pl.nch);
            const int32_t unit = g * pl.Ug + t.ul;  // global unit index
            if (t.ch == 0 && t.kb == 0) {
                // sample descriptors of this warp's 16 rows for the taps of block t.b
                const int32_t gd = static_cast<int32_t>((static_cast<int64_t>(unit) * pl.U) / pl.Cd);
                __syncwarp();
                for (int e = lane; e < kRowsPerWarp * t.ntb; e += 32) {
                    const int r = e % kRowsPerWarp;
                    const int kb2 = e / kRowsPerWarp;
                    make_desc<T>(pl, offset, mask, m0 + pw * kRowsPerWarp + r, t.b * kTapBlock + kb2, gd,
                                 dc + static_cast<uint32_t>(kb2 * kRowsPerWarp + r) * kDescBytes);
                }
                __syncwarp();
            }
            const int s = kt % S;
            const uint32_t ph = (kt / S) & 1;
            // warp-uniform decision: every lane leaves together on a timeout
            const bool got = mbar_wait_bounded(empty_bar(s), ph ^ 1u, abort_flag, prm.status, kSiteGatherEmpty);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            const int64_t cbase = static_cast<int64_t>(unit) * pl.UP + static_cast<int64_t>(t.ch) * pl.BKc + q * kVec;
            const uint32_t a_s = a0 + s * a_bytes;
            uint4 v[4][4];
            uint4 wv[4];
#pragma unroll
            for (int it = 0; it < 4; ++it) {
                const int r = it * 4 + rsub;
                const uint32_t da = dc + static_cast<uint32_t>(t.kb * kRowsPerWarp + r) * kDescBytes;
                const uint4 dd = lds128(da);
                wv[it] = lds128(da + 16);
                const int64_t base = static_cast<int64_t>((static_cast<uint64_t>(dd.y) << 32) | dd.x);
                const uint32_t fl = dd.z;
                const uint4* src = reinterpret_cast<const uint4*>(xt + base + cbase);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    v[it][c] = make_uint4(0u, 0u, 0u, 0u);
                    if (fl & (1u << c)) v[it][c] = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(src) + coff[c]));
                }
            }
#pragma unroll
            for (int it = 0; it < 4; ++it) {
                const int row = pw * kRowsPerWarp + it * 4 + rsub;
                const uint32_t dst = a_s + static_cast<uint32_t>(row) * 128u + (static_cast<uint32_t>(q ^ (row & 7)) << 4);
                if constexpr (kF32Path) {
                    const float w0 = __uint_as_float(wv[it].x), w1 = __uint_as_float(wv[it].y);
                    const float w2 = __uint_as_float(wv[it].z), w3 = __uint_as_float(wv[it].w);
                    float acc[4];
                    const uint32_t* p0 = reinterpret_cast<const uint32_t*>(&v[it][0]);
                    const uint32_t* p1 = reinterpret_cast<const uint32_t*>(&v[it][1]);
                    const uint32_t* p2 = reinterpret_cast<const uint32_t*>(&v[it][2]);
                    const uint32_t* p3 = reinterpret_cast<const uint32_t*>(&v[it][3]);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        float a = w0 * __uint_as_float(p0[e]);
                        a = fmaf(w1, __uint_as_float(p1[e]), a);
                        a = fmaf(w2, __uint_as_float(p2[e]), a);
                        a = fmaf(w3, __uint_as_float(p3[e]), a);
                        acc[e] = a;
                    }
                    float hi[4], lo[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        hi[e] = to_tf32(acc[e]);
                        lo[e] = acc[e] - hi[e];
                    }
                    sts128(dst, __float_as_uint(hi[0]), __float_as_uint(hi[1]), __float_as_uint(hi[2]),
                           __float_as_uint(hi[3]));
                    sts128(dst + kTileM * 128, __float_as_uint(lo[0]), __float_as_uint(lo[1]), __float_as_uint(lo[2]),
                           __float_as_uint(lo[3]));
                } else {
                    T* tag = nullptr;
                    const uint32_t* p0 = reinterpret_cast<const uint32_t*>(&v[it][0]);
                    const uint32_t* p1 = reinterpret_cast<const uint32_t*>(&v[it][1]);
                    const uint32_t* p2 = reinterpret_cast<const uint32_t*>(&v[it][2]);
                    const uint32_t* p3 = reinterpret_cast<const uint32_t*>(&v[it][3]);
                    uint32_t o[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        o[e] = combine2(wv[it].x, wv[it].y, wv[it].z, wv[it].w, p0[e], p1[e], p2[e], p3[e], tag);
                    sts128(dst, o[0], o[1], o[2], o[3]);
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(full_bar(s));
        }

        // ------------------------------------------------------------ epilogue
        const bool acc_ok =
            __all_sync(0xffffffffu, mbar_wait_bounded(acc_bar, 0, abort_flag, prm.status, kSiteEpilogue));
        tc_fence_after();
        if (acc_ok) {
            const int quarter = warp & 3;
            const int set = pw >> 2;  // two warps per TMEM lane quarter split the columns
            const int row = quarter * 32 + lane;
            const int64_t p = m0 + row;
            const bool valid = p < pl.NP;
            const int64_t n = valid ? p / pl.P : 0;
            const int64_t hw = valid ? p - n * pl.P : 0;
            T* __restrict__ out = static_cast<T*>(prm.out);
            const T* __restrict__ bias = static_cast<const T*>(prm.bias);
            const int32_t ncols = pl.nsub * pl.BNs;
            for (int c16 = set; c16 * 16 < ncols; c16 += 2) {
                float vals[16];
                tmem_ld16(tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(c16 * 16), vals);
                if (valid) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int32_t ol = ncol0 + c16 * 16 + e;
                        if (ol < pl.Og) {
                            const int64_t o = static_cast<int64_t>(g) * pl.Og + ol;
                            float r = vals[e];
                            if (bias) r += to_f(bias[o]);
                            from_f(r, out + (n * pl.Cout + o) * pl.P + hw);
                        }
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, static_cast<uint32_t>(pl.tmem_cols));
    }
}

// Tiny kernel for the bounded-wait self-test: waits on a barrier nothing signals.
__global__ void wait_selftest_kernel(uint32_t* status, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        *status = 0u;
        fence_mbarrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const bool ok = mbar_wait_bounded(smem_u32(&bar), 0, &abort_flag, status, kSiteSelftest, limit_ns);
        if (ok) atomicOr(status, 1u << 31);  // the wait completed although nothing arrived
        // complete the phase so that no barrier is left pending at exit
        mbar_arrive(smem_u32(&bar));
    }
    __syncthreads();
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

template <int DT>
cudaError_t launch_fused_t(const Plan& pl, const void* offset, const void* mask, const void* bias, void* out, void* ws,
                           cudaStream_t st) {
    using T = typename Elem<DT>::T;
    uint8_t* base = static_cast<uint8_t*>(ws);
    const T* wp = reinterpret_cast<const T*>(base + pl.off_wp);
    auto encode = get_encode_fn();
    if (!encode) return cudaErrorNotSupported;
    CUtensorMap tmap;
    const cuuint64_t rows = static_cast<cuuint64_t>(pl.wp_rows);
    const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(pl.KP), rows};
    const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(pl.KP) * sizeof(T)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(pl.BKc), static_cast<cuuint32_t>(pl.BNs)};
    const cuuint32_t estride[2] = {1, 1};
    CUresult r = encode(&tmap, Elem<DT>::tma, 2, const_cast<T*>(wp), gdim, gstride, box, estride,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    FusedParams prm;
    prm.xt = base + pl.off_xt;
    prm.offset = offset;
    prm.mask = mask;
    prm.bias = bias;
    prm.out = out;
    prm.status = reinterpret_cast<uint32_t*>(base);
    prm.pl = pl;
    dim3 grid(static_cast<unsigned>(pl.mtiles), static_cast<unsigned>(pl.ntiles_n), static_cast<unsigned>(pl.group));
    fused_kernel<DT><<<grid, kFusedThreads, pl.smem_bytes, st>>>(tmap, prm);
    return cudaGetLastError();
}

}  // namespace

cudaError_t prepare_fused_attributes(int dtype, int smem_bytes) {
    switch (dtype) {
        case kF32:
            return cudaFuncSetAttribute(fused_kernel<kF32>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
        case kF16:
            return cudaFuncSetAttribute(fused_kernel<kF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
        default:
            return cudaFuncSetAttribute(fused_kernel<kBF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    }
}

cudaError_t launch_fused(const Plan& pl, const void* offset, const void* mask, const void* bias, void* out, void* ws,
                         cudaStream_t st) {
    switch (pl.dtype) {
        case kF32: return launch_fused_t<kF32>(pl, offset, mask, bias, out, ws, st);
        case kF16: return launch_fused_t<kF16>(pl, offset, mask, bias, out, ws, st);
        default: return launch_fused_t<kBF16>(pl, offset, mask, bias, out, ws, st);
    }
}

cudaError_t launch_wait_selftest(uint32_t* status, uint64_t limit_ns, cudaStream_t st) {
    wait_selftest_kernel<<<1, 32, 0, st>>>(status, limit_ns);
    return cudaGetLastError();
}

}  // namespace mdcn
