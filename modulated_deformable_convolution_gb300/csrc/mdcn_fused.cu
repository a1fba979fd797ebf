// Fused implicit-GEMM kernel of the modulated deformable convolution forward
// ("TensorRT plugin walkthrough: modulatedDeformConvPlugin", section 5, steps
// 1-3, without the column buffer).
//
// fused_kernel: persistent CTAs (one per SM) take equal consecutive ranges of
// the k-tiles of all output tiles (128 pixels x (nsub*BNs) output channels of
// one convolution group). Warp roles:
//   warp 0      TMA: weight k-tiles (K-major, 128-byte swizzle) -> B stages
//   warp 1      allocates tensor memory; lane 0 issues tcgen05.mma
//               (A = modulated columns, B = weights, D = fp32 in TMEM,
//               two accumulators so the epilogue overlaps the next tile)
//   warps 2-3   sampling: from offset and mask, each tile row's sampling
//               point, corner validity and bilinear weights times the mask
//               (one descriptor per row and tap) for a tap block of one
//               deformable group at a time -> two-slot ring in shared memory
//   warps 4-11  gather, as G warp groups each producing every G-th k-tile
//               (one tap, 128 bytes of channels): per row, 4 lanes x 32 bytes of
//               the 4 corners of the channels-last copy of x, weighted sum,
//               128-byte-swizzled store into the A stage
//   warps 12-15 epilogue: TMEM -> registers -> +bias -> NCHW output. A tile
//               split between CTAs (stream-K): each CTA but the one holding
//               its last k-tiles writes an fp32 partial sum to the workspace
//               and counts itself in; that last CTA (each CTA processes its
//               units last to first, so it reaches the tile last) adds the
//               partials in k order and stores the output
// Hand-offs use mbarriers; every wait is bounded (mdcn_ptx.cuh), and a wait
// that gives up raises a CTA-wide abort that every role observes.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstring>
#include <type_traits>
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
    float* part;           // fp32 partial accumulators of split tiles: one slot per CTA
    uint32_t* split_count;  // per split tile (by its owner, the CTA of its last k-tiles): contributors in
    int32_t epi_vec;        // the plan allows 16-byte output stores and out is 16-byte aligned
    Plan pl;
};

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__half v) { return __half2float(v); }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }

__device__ __forceinline__ void from_f(float v, float* d) { *d = v; }
__device__ __forceinline__ void from_f(float v, __half* d) { *d = __float2half_rn(v); }
__device__ __forceinline__ void from_f(float v, __nv_bfloat16* d) { *d = __float2bfloat16_rn(v); }

template <typename T>
__device__ __forceinline__ T ld_shared_elem(uint32_t addr) {
    if constexpr (sizeof(T) == 4) {
        uint32_t v;
        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
        return __uint_as_float(v);
    } else {
        uint16_t v;
        asm volatile("ld.shared.b16 %0, [%1];" : "=h"(v) : "r"(addr) : "memory");
        T h;
        *reinterpret_cast<uint16_t*>(&h) = v;
        return h;
    }
}

// One value converted to T, stored to shared memory.
template <typename T>
__device__ __forceinline__ void st_shared_elem(uint32_t addr, float v) {
    if constexpr (sizeof(T) == 4) {
        asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(__float_as_uint(v)) : "memory");
    } else {
        T h;
        from_f(v, &h);
        asm volatile("st.shared.b16 [%0], %1;" ::"r"(addr), "h"(*reinterpret_cast<uint16_t*>(&h)) : "memory");
    }
}

__device__ __forceinline__ uint32_t pack2(float a, float b, __half*) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack2(float a, float b, __nv_bfloat16*) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
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

// Output pixel of tile row r: returns false for rows past the edge.
struct Pixel {
    int64_t n, ho, wo;
    bool valid;
};

// Pixel indices fit in 32 bits (the planner keeps N*Ho*Wo below 2^31).
__device__ __forceinline__ Pixel tile_pixel(const Plan& pl, int64_t mt64, int r) {
    Pixel px;
    const uint32_t mt = static_cast<uint32_t>(mt64);
    if (pl.tile_mode == 0) {
        const uint32_t p = mt * kTileM + static_cast<uint32_t>(r);
        px.valid = p < static_cast<uint32_t>(pl.NP);
        const uint32_t pp = px.valid ? p : 0u;
        const uint32_t P = static_cast<uint32_t>(pl.P), Wo = static_cast<uint32_t>(pl.Wo);
        const uint32_t n = pp / P;
        const uint32_t hw = pp - n * P;
        const uint32_t ho = hw / Wo;
        px.n = n;
        px.ho = ho;
        px.wo = hw - ho * Wo;
    } else {
        const uint32_t tiles_x = static_cast<uint32_t>(pl.tiles_x);
        const uint32_t per_img = tiles_x * static_cast<uint32_t>(pl.tiles_y);
        const uint32_t n = mt / per_img;
        const uint32_t rem = mt - n * per_img;
        const uint32_t ty = rem / tiles_x;
        const uint32_t tx = rem - ty * tiles_x;
        px.n = n;
        px.ho = static_cast<int64_t>(ty * kTileH + static_cast<uint32_t>(r) / kTileW);
        px.wo = static_cast<int64_t>(tx * kTileW + static_cast<uint32_t>(r) % kTileW);
        px.valid = px.ho < pl.Ho && px.wo < pl.Wo;
    }
    return px;
}

struct TileId {
    int32_t g, nt;
    int64_t mt;
};

// Tile indices, k-tile positions and CTA indices fit in 32 bits (the planner
// keeps the k-tiles of all tiles below 2^31), so their divisions are 32-bit.
__device__ __forceinline__ TileId decode_tile(const Plan& pl, int64_t t) {
    TileId id;
    const uint32_t t32 = static_cast<uint32_t>(t);
    const uint32_t mt = static_cast<uint32_t>(pl.mtiles), nn = static_cast<uint32_t>(pl.ntiles_n);
    const uint32_t r = t32 / mt;
    id.mt = t32 - r * mt;
    const uint32_t g = r / nn;
    id.nt = static_cast<int32_t>(r - g * nn);
    id.g = static_cast<int32_t>(g);
    return id;
}

// 16-bit: out = w00*v0 + w01*v1 + w10*v2 + w11*v3 on one pair of channels;
// wa = (w00, w01), wb = (w10, w11).
__device__ __forceinline__ uint32_t blend(uint32_t wa, uint32_t wb, uint32_t v0, uint32_t v1, uint32_t v2,
                                          uint32_t v3, __half*) {
    const __half2 a = *reinterpret_cast<const __half2*>(&wa), b = *reinterpret_cast<const __half2*>(&wb);
    __half2 acc = __hmul2(__low2half2(a), *reinterpret_cast<const __half2*>(&v0));
    acc = __hfma2(__high2half2(a), *reinterpret_cast<const __half2*>(&v1), acc);
    acc = __hfma2(__low2half2(b), *reinterpret_cast<const __half2*>(&v2), acc);
    acc = __hfma2(__high2half2(b), *reinterpret_cast<const __half2*>(&v3), acc);
    return *reinterpret_cast<uint32_t*>(&acc);
}

__device__ __forceinline__ uint32_t blend(uint32_t wa, uint32_t wb, uint32_t v0, uint32_t v1, uint32_t v2,
                                          uint32_t v3, __nv_bfloat16*) {
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&wa);
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&wb);
    __nv_bfloat162 acc = __hmul2(__low2bfloat162(a), *reinterpret_cast<const __nv_bfloat162*>(&v0));
    acc = __hfma2(__high2bfloat162(a), *reinterpret_cast<const __nv_bfloat162*>(&v1), acc);
    acc = __hfma2(__low2bfloat162(b), *reinterpret_cast<const __nv_bfloat162*>(&v2), acc);
    acc = __hfma2(__high2bfloat162(b), *reinterpret_cast<const __nv_bfloat162*>(&v3), acc);
    return *reinterpret_cast<uint32_t*>(&acc);
}

// ---------------------------------------------------------------- sample descriptors
// Descriptor of (tile row, deformable group, tap): the pixel index of corner
// (y0, x0) in the channels-last x (int32), the 4 corner-valid bits, then the
// 4 bilinear weights times the mask (16-bit pairs in the last 8 bytes for
// 16-bit types; fp32 words in a second 16 bytes for fp32). Sampling point (section 5 step 1):
// (ho*sh - ph + i*dh + dh_off, wo*sw - pw + j*dw + dw_off); a point outside
// (-1, H) x (-1, W) and the corners outside the image contribute nothing.
//
// Where a tile row's sampling inputs are: its pixel, and its offset and mask
// elements of tap tap0 (taps follow at a stride of P elements).
template <typename T>
struct SampleRow {
    const T* po;   // offset channel 2*tap0 (h) of the row's pixel; w follows at +P
    const T* pm;   // mask channel tap0
    float hbase, wbase;
    int64_t nbase;
    bool valid;
};

template <typename T>
__device__ __forceinline__ SampleRow<T> sample_row_at(const Plan& pl, const T* offset, const T* mask, int64_t mt,
                                                      int64_t gd, int row, int32_t tap0) {
    const Pixel q = tile_pixel(pl, mt, row);
    const int64_t K = pl.K;
    const int64_t P = pl.P;
    const int64_t n = q.valid ? q.n : 0;
    const int64_t hw = q.valid ? q.ho * pl.Wo + q.wo : 0;
    SampleRow<T> r;
    r.po = pl.plain ? nullptr : offset + (n * 2 * pl.dg * K + gd * 2 * K + 2 * static_cast<int64_t>(tap0)) * P + hw;
    r.pm = pl.plain ? nullptr : mask + (n * pl.dg * K + gd * K + tap0) * P + hw;
    r.hbase = static_cast<float>(q.ho * pl.sh - pl.ph);
    r.wbase = static_cast<float>(q.wo * pl.sw - pl.pw);
    r.nbase = q.n * pl.H;
    r.valid = q.valid;
    return r;
}

// Descriptor of one (row, tap) from its offset pair and mask value.
template <typename T>
__device__ __forceinline__ void write_desc(const Plan& pl, const SampleRow<T>& r, int32_t i, int32_t j, float dhv,
                                           float dwv, float mv, uint8_t* dp) {
    int32_t base = 0;  // pixel index of corner (y0, x0) in the channels-last x (may be -1 - W .. )
    uint32_t flags = 0;
    float w00 = 0.f, w01 = 0.f, w10 = 0.f, w11 = 0.f;
    const float hf = r.hbase + static_cast<float>(i * pl.dh) + dhv;
    const float wf = r.wbase + static_cast<float>(j * pl.dw) + dwv;
    if (r.valid && hf > -1.0f && hf < static_cast<float>(pl.H) && wf > -1.0f && wf < static_cast<float>(pl.W)) {
        const float h0f = floorf(hf), w0f = floorf(wf);
        const float lh = hf - h0f, lw = wf - w0f;
        const float hh = 1.0f - lh, hw_ = 1.0f - lw;
        const int32_t y0 = static_cast<int32_t>(h0f);
        const int32_t x0 = static_cast<int32_t>(w0f);
        w00 = hh * hw_ * mv;
        w01 = hh * lw * mv;
        w10 = lh * hw_ * mv;
        w11 = lh * lw * mv;
        // a corner whose bilinear weight is exactly 0 (the point on a pixel row
        // or column) reads the zero pixel instead: the same sum, fewer loads
        const bool top = y0 >= 0, bottom = y0 + 1 < pl.H && lh != 0.0f;
        const bool left = x0 >= 0, right = x0 + 1 < pl.W && lw != 0.0f;
        flags = (top && left ? 1u : 0u) | (top && right ? 2u : 0u) | (bottom && left ? 4u : 0u) |
                (bottom && right ? 8u : 0u);
        base = static_cast<int32_t>((r.nbase + y0) * pl.W + x0);
    }
    uint4 d0;
    d0.x = static_cast<uint32_t>(base);
    d0.y = flags;
    if constexpr (sizeof(T) == 4) {
        d0.z = 0u;
        d0.w = 0u;
        reinterpret_cast<uint4*>(dp)[0] = d0;
        reinterpret_cast<uint4*>(dp)[1] =
            make_uint4(__float_as_uint(w00), __float_as_uint(w01), __float_as_uint(w10), __float_as_uint(w11));
    } else {
        T* tag = nullptr;
        d0.z = pack2(w00, w01, tag);
        d0.w = pack2(w10, w11, tag);
        reinterpret_cast<uint4*>(dp)[0] = d0;
    }
}

// One thread writes the descriptors of tile rows row and row + 64 for taps
// [tap0, tap0 + ntap) to dst + (kb * kTileM + row) * dsz, kb = tap - tap0;
// the offset and mask loads of kRingTaps taps of both rows are issued
// together.
constexpr int kSampleTaps = 3;   // the prologue's taps per thread (sample_row_taps)
constexpr int kRingTaps = 5;     // the sampling warps' taps per round (sample_rows): 30 loads in flight

template <typename T>
__device__ __forceinline__ void sample_rows(const Plan& pl, const T* __restrict__ offset, const T* __restrict__ mask,
                                            int64_t mt, int64_t gd, int row, int32_t tap0, int32_t ntap,
                                            uint8_t* dst, uint32_t dsz) {
    const int64_t P = pl.P;
    const SampleRow<T> ra = sample_row_at(pl, offset, mask, mt, gd, row, tap0);
    const SampleRow<T> rb = sample_row_at(pl, offset, mask, mt, gd, row + 64, tap0);
    int32_t i = tap0 / static_cast<int32_t>(pl.kw);
    int32_t j = tap0 - i * static_cast<int32_t>(pl.kw);
#pragma unroll 1
    for (int32_t kb0 = 0; kb0 < ntap; kb0 += kRingTaps) {
        float v[2][3][kRingTaps];  // [row][dh, dw, mask][tap]
        if (pl.plain) {
#pragma unroll
            for (int u = 0; u < kRingTaps; ++u) {
                v[0][0][u] = v[0][1][u] = v[1][0][u] = v[1][1][u] = 0.f;
                v[0][2][u] = v[1][2][u] = 1.f;
            }
        } else {
#pragma unroll
            for (int u = 0; u < kRingTaps; ++u) {
                const int64_t kb = kb0 + u < ntap ? kb0 + u : kb0;
                v[0][0][u] = to_f(ra.po[(2 * kb) * P]);
                v[0][1][u] = to_f(ra.po[(2 * kb + 1) * P]);
                v[0][2][u] = to_f(ra.pm[kb * P]);
                v[1][0][u] = to_f(rb.po[(2 * kb) * P]);
                v[1][1][u] = to_f(rb.po[(2 * kb + 1) * P]);
                v[1][2][u] = to_f(rb.pm[kb * P]);
            }
        }
#pragma unroll
        for (int u = 0; u < kRingTaps; ++u) {
            if (kb0 + u < ntap) {
                uint8_t* dp = dst + (static_cast<uint32_t>(kb0 + u) * kTileM + row) * dsz;
                write_desc(pl, ra, i, j, v[0][0][u], v[0][1][u], v[0][2][u], dp);
                write_desc(pl, rb, i, j, v[1][0][u], v[1][1][u], v[1][2][u], dp + 64 * dsz);
            }
            if (++j == static_cast<int32_t>(pl.kw)) {
                j = 0;
                ++i;
            }
        }
    }
}

// One tile row, taps tap0 + kb for kb = kb_first, kb_first + kb_step, ... <
// ntap (at most kSampleTaps of them): every load first, then the descriptors.
template <typename T>
__device__ __forceinline__ void sample_row_taps(const Plan& pl, const T* __restrict__ offset,
                                                const T* __restrict__ mask, int64_t mt, int64_t gd, int row,
                                                int32_t tap0, int32_t ntap, int32_t kb_first, int32_t kb_step,
                                                uint8_t* dst, uint32_t dsz) {
    const int64_t P = pl.P;
    const SampleRow<T> r = sample_row_at(pl, offset, mask, mt, gd, row, tap0);
    float v[3][kSampleTaps];
    if (pl.plain) {
#pragma unroll
        for (int u = 0; u < kSampleTaps; ++u) {
            v[0][u] = v[1][u] = 0.f;
            v[2][u] = 1.f;
        }
    } else {
#pragma unroll
        for (int u = 0; u < kSampleTaps; ++u) {
            const int32_t kb0 = kb_first + u * kb_step;
            const int64_t kb = kb0 < ntap ? kb0 : 0;
            v[0][u] = to_f(r.po[(2 * kb) * P]);
            v[1][u] = to_f(r.po[(2 * kb + 1) * P]);
            v[2][u] = to_f(r.pm[kb * P]);
        }
    }
#pragma unroll
    for (int u = 0; u < kSampleTaps; ++u) {
        const int32_t kb = kb_first + u * kb_step;
        if (kb < ntap) {
            const int32_t tap = tap0 + kb;
            const int32_t i = tap / static_cast<int32_t>(pl.kw);
            const int32_t j = tap - i * static_cast<int32_t>(pl.kw);
            write_desc(pl, r, i, j, v[0][u], v[1][u], v[2][u], dst + (static_cast<uint32_t>(kb) * kTileM + row) * dsz);
        }
    }
}

// ---------------------------------------------------------------- work split
// Stream-K: the k-tiles of all tiles form one sequence (tile t's k-tile k at
// position t*KT + k) and persistent CTA c takes the contiguous range
// [c*R, min((c+1)*R, total)), R = pl.kt_per_cta. A CTA's range covers
// "units": pieces of consecutive tiles, a whole tile or a k-range of one. A
// CTA processes its units from the last to the first (k-tiles ascending
// within each), so its first unit to finish is the piece of the tile that
// runs past its range. A tile whose k-tiles fall to several CTAs is owned by
// the CTA holding its last k-tiles (the highest of them): for that CTA the
// tile is the unit processed last, while every other contributor processes
// its piece first, writes an fp32 partial sum and counts itself in. The
// owner waits only for CTAs of lower index, which are dispatched before it,
// so no CTA waits for one that may not yet be resident.
struct Unit {
    int64_t t;        // tile
    int32_t k0, k1;   // k-tile range [k0, k1) of the tile
};

// The last unit of the range [lo, end): the piece of the tile holding
// position end - 1.
__device__ __forceinline__ Unit unit_back(const Plan& pl, int64_t lo, int64_t end) {
    Unit u;
    u.t = static_cast<uint32_t>(end - 1) / static_cast<uint32_t>(pl.KT);
    const int64_t t0 = u.t * pl.KT;
    u.k0 = static_cast<int32_t>(lo > t0 ? lo - t0 : 0);
    u.k1 = static_cast<int32_t>(end - t0);
    return u;
}

// The CTA whose range holds position pos.
__device__ __forceinline__ int64_t cta_of(const Plan& pl, int64_t pos) {
    return static_cast<uint32_t>(pos) / static_cast<uint32_t>(pl.kt_per_cta);
}

// ---------------------------------------------------------------- gather helpers
// Position in a CTA's k-tile sequence, in processing order. A tile's k-tiles
// form descriptor groups (unit ul, tap block b), in the order of the packed
// weight; each group holds its chunks x taps k-tiles.
struct Cursor {
    int64_t pos;          // position in the k-tile sequence
    int64_t ustart, uend; // the current unit [ustart, uend)
    int64_t lo;           // start of the CTA's range
    int64_t t, mt;
    int32_t g, nt;
    int32_t gi, j;        // group, k-tile within the group
    int32_t ul, b, ntbg, nktg, ch, kb, kt;  // the k-tile at that position
    uint32_t gr;          // descriptor groups entered so far
    bool live;
};

__device__ __forceinline__ void cursor_group(const Plan& pl, Cursor& c) {
    c.ul = c.gi / pl.ntb;
    c.b = c.gi - c.ul * pl.ntb;
    c.ntbg = min(kTapBlock, pl.K - c.b * kTapBlock);
    c.nktg = c.ntbg * pl.nch;
}

__device__ __forceinline__ void cursor_ktile(const Plan& pl, Cursor& c) {
    c.ch = c.j / c.ntbg;
    c.kb = c.j - c.ch * c.ntbg;
    c.kt = (c.ul * pl.K + c.b * kTapBlock) * pl.nch + c.j;  // global k-tile index (B coordinate)
}

__device__ __forceinline__ void cursor_tile(const Plan& pl, Cursor& c, int64_t t) {
    c.t = t;
    const TileId id = decode_tile(pl, t);
    c.g = id.g;
    c.nt = id.nt;
    c.mt = id.mt;
}

// Enters the unit that ends at c.uend, at its first k-tile.
__device__ __forceinline__ void cursor_enter_unit(const Plan& pl, Cursor& c) {
    const Unit un = unit_back(pl, c.lo, c.uend);
    c.ustart = un.t * pl.KT + un.k0;
    c.pos = c.ustart;
    cursor_tile(pl, c, un.t);
    int32_t k = un.k0;
    c.gi = 0;
    cursor_group(pl, c);
    while (k >= c.nktg) {
        k -= c.nktg;
        ++c.gi;
        cursor_group(pl, c);
    }
    c.j = k;
    cursor_ktile(pl, c);
}

__device__ __forceinline__ void cursor_init(const Plan& pl, Cursor& c, int64_t lo, int64_t hi) {
    c.gr = 0;
    c.lo = lo;
    c.uend = hi;
    c.live = lo < hi;
    if (!c.live) return;
    cursor_enter_unit(pl, c);
}

__device__ __forceinline__ void cursor_advance(const Plan& pl, Cursor& c) {
    if (++c.pos >= c.uend) {
        // the unit is done: on to the piece of the range before it, if any
        if (c.ustart <= c.lo) {
            c.live = false;
            return;
        }
        c.uend = c.ustart;
        ++c.gr;
        cursor_enter_unit(pl, c);
        return;
    }
    if (++c.j < c.nktg) {
        cursor_ktile(pl, c);
        return;
    }
    // the next group of the same tile (a unit never crosses a tile boundary)
    c.j = 0;
    ++c.gr;
    ++c.gi;
    cursor_group(pl, c);
    cursor_ktile(pl, c);
}

// Moves the cursor to the first k-tile of its next group.
__device__ __forceinline__ void cursor_next_group(const Plan& pl, Cursor& c) {
    c.pos += c.nktg - 1 - c.j;
    c.j = c.nktg - 1;
    cursor_advance(pl, c);
}

template <typename T>
struct GatherCtx {
    const T* xt;
    int32_t d1, dW, dW1;  // pixel deltas of corners (y0, x0+1), (y0+1, x0), (y0+1, x0+1): 1, W, W+1
    int32_t zpix;         // the all-zero pixel after the image data, read for corners outside the image
    int32_t pix_bytes;    // bytes per channels-last pixel
    uint32_t row_desc;    // this lane's descriptor within a tap block, row-iteration 0
    uint32_t row_sts;     // this lane's A-stage offset (128-byte swizzle), row-iteration 0, chunk 2*q4
    int lane, q4, rsub, row0;
    uint32_t dsz;
};

struct RowBuf {  // one row-iteration of one lane: 4 corners x 32 bytes, and the row's descriptor
    uint4 v[4][2];
    uint4 w;     // 16-bit types: .z = (w00, w01), .w = (w10, w11); fp32: the 4 weights
};

__device__ __forceinline__ uint32_t swz128(int row, int chunk) {
    return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ float blend_f32(float w00, float w01, float w10, float w11, uint32_t v0, uint32_t v1,
                                           uint32_t v2, uint32_t v3) {
    float a = w00 * __uint_as_float(v0);
    a = fmaf(w01, __uint_as_float(v1), a);
    a = fmaf(w10, __uint_as_float(v2), a);
    return fmaf(w11, __uint_as_float(v3), a);
}

// Row-iteration it of a k-tile: reads the row's descriptor (in the tap block
// at dtap) and loads its 4 corners (32 bytes per lane, chunks 2*q4, 2*q4+1)
// from cbp = the lane's channels of pixel 0. Every corner is loaded: one
// outside the image reads the zero pixel, so no load is conditional.
template <typename T, bool kF32Path>
__device__ __forceinline__ void row_issue(const GatherCtx<T>& cx, uint32_t dtap, const char* cbp, int it,
                                          RowBuf& rb) {
    const uint32_t da = dtap + cx.row_desc + static_cast<uint32_t>(it) * 8u * cx.dsz;
    const uint4 e = lds128(da);
    if constexpr (kF32Path) {
        rb.w = lds128(da + 16);
    } else {
        rb.w = e;
    }
    const int32_t base = static_cast<int32_t>(e.x);
    const uint32_t fl = e.y;
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
        const int32_t delta = cc == 0 ? 0 : (cc == 1 ? cx.d1 : (cc == 2 ? cx.dW : cx.dW1));
        const int32_t pix = (fl >> cc) & 1u ? base + delta : cx.zpix;
        ldg256(cbp + static_cast<int64_t>(pix) * cx.pix_bytes, rb.v[cc][0], rb.v[cc][1]);
    }
}

// 16-bit: the lane's 8 blended channel pairs of a row (pair m = channels
// 16*q4 + 2m, + 1 of the k-tile), m = 4*hv + j for the corner loads' half hv
// and word j.
template <typename T>
__device__ __forceinline__ void blend_row16(const RowBuf& rb, uint32_t (&v)[8]) {
    const uint4 w = rb.w;
    T* tag = nullptr;
#pragma unroll
    for (int hv = 0; hv < 2; ++hv) {
        const uint4 a = rb.v[0][hv], b = rb.v[1][hv], c = rb.v[2][hv], d = rb.v[3][hv];
        v[4 * hv + 0] = blend(w.z, w.w, a.x, b.x, c.x, d.x, tag);
        v[4 * hv + 1] = blend(w.z, w.w, a.y, b.y, c.y, d.y, tag);
        v[4 * hv + 2] = blend(w.z, w.w, a.z, b.z, c.z, d.z, tag);
        v[4 * hv + 3] = blend(w.z, w.w, a.w, b.w, c.w, d.w, tag);
    }
}

// Weighted sum of the 4 corners of row-iteration it into the A stage a_s:
// the lane's 32 bytes are 16-byte chunks 2*q4 and 2*q4 + 1 of its row
// (128-byte swizzle; channels in their natural order). Rows of a
// row-iteration are 8 apart in 128-byte lines: row & 7 == rsub.
template <typename T, bool kF32Path>
__device__ __forceinline__ void row_combine(const GatherCtx<T>& cx, uint32_t a_s, int it, const RowBuf& rb) {
    const uint32_t o0 = cx.row_sts + static_cast<uint32_t>(it) * 1024u, o1 = o0 ^ 16u;
    if constexpr (kF32Path) {
        const uint4 w = rb.w;
        const float w00 = __uint_as_float(w.x), w01 = __uint_as_float(w.y);
        const float w10 = __uint_as_float(w.z), w11 = __uint_as_float(w.w);
#pragma unroll
        for (int hv = 0; hv < 2; ++hv) {
            const uint4 a = rb.v[0][hv], b = rb.v[1][hv], c = rb.v[2][hv], d = rb.v[3][hv];
            const uint32_t o = hv ? o1 : o0;
            const float s0 = blend_f32(w00, w01, w10, w11, a.x, b.x, c.x, d.x);
            const float s1 = blend_f32(w00, w01, w10, w11, a.y, b.y, c.y, d.y);
            const float s2 = blend_f32(w00, w01, w10, w11, a.z, b.z, c.z, d.z);
            const float s3 = blend_f32(w00, w01, w10, w11, a.w, b.w, c.w, d.w);
            const float h0 = to_tf32(s0), h1 = to_tf32(s1), h2 = to_tf32(s2), h3 = to_tf32(s3);
            sts128(a_s + o, __float_as_uint(h0), __float_as_uint(h1), __float_as_uint(h2), __float_as_uint(h3));
            sts128(a_s + kTileM * 128 + o, __float_as_uint(s0 - h0), __float_as_uint(s1 - h1),
                   __float_as_uint(s2 - h2), __float_as_uint(s3 - h3));
        }
    } else {
        uint32_t v[8];
        blend_row16<T>(rb, v);
        sts128(a_s + o0, v[0], v[1], v[2], v[3]);
        sts128(a_s + o1, v[4], v[5], v[6], v[7]);
    }
}

// 16-bit, A in tensor memory: row-iterations it (rows r) and it + 1 (rows
// r + 8) of the lane, one 16-row block, stored with one 16x256b.x4 fragment
// at ta (lane = the block's first row, column = the stage's first). Fragment
// register 4k + h (h < 2: row r, else r + 8) goes to column 8k + 2*q4 + h % 2;
// it holds pair 2k + h % 2, so that column holds channels whose K position
// the tensor-memory K order (kperm16, which the packed weight follows) gives.
template <typename T>
__device__ __forceinline__ void rows_to_tmem(uint32_t ta, const RowBuf& ra, const RowBuf& rb) {
    uint32_t va[8], vb[8], r[16];
    blend_row16<T>(ra, va);
    blend_row16<T>(rb, vb);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        r[4 * k + 0] = va[2 * k];
        r[4 * k + 1] = va[2 * k + 1];
        r[4 * k + 2] = vb[2 * k];
        r[4 * k + 3] = vb[2 * k + 1];
    }
    tmem_st_16x256b_x4(ta, r);
}

// ---------------------------------------------------------------- epilogue helpers
// 32 accumulator columns from c32 (16 where fewer remain) of this thread's
// row -> the fp32 partial slot of CTA `cta` ([column][row], so each warp
// writes 128 contiguous bytes per column).
template <typename T>
__device__ __forceinline__ void write_partial32(const Plan& pl, float* part, int64_t cta, uint32_t tl, int c32,
                                                int row) {
    float vals[32];
    tmem_ld32(tl + static_cast<uint32_t>(c32), pl.acc_cols - c32 >= 32 ? 2 : 1, vals);
    float* mine = part + (cta * pl.acc_cols + c32) * kTileM + row;
#pragma unroll
    for (int c = 0; c < 32; ++c)
        if (c < pl.acc_cols - c32) mine[c * kTileM] = vals[c];
}

// After this CTA's partial slot is written by the `nthreads` threads that
// meet at named barrier `bar`: one of them counts the CTA in on the split
// tile's counter (release: the slot's writes are visible before the count).
__device__ __forceinline__ void count_in_split(uint32_t* counter, uint32_t bar, uint32_t nthreads, bool leader) {
    __threadfence();
    named_bar_sync(bar, nthreads);
    if (leader) atomicAdd(counter, 1u);
}

// The tile's bias columns -> shared memory as fp32 (0 past the group's columns).
template <typename T>
__device__ __forceinline__ void stage_bias(const Plan& pl, const T* bias, const TileId& id, uint32_t bias_s, int tid,
                                           int nthreads) {
    const int32_t ncol0 = id.nt * pl.acc_cols;
    for (int c = tid; c < pl.acc_cols; c += nthreads) {
        const int32_t ol = ncol0 + c;
        st_shared_f32(bias_s + 4u * c, ol < pl.Og ? to_f(bias[static_cast<int64_t>(id.g) * pl.Og + ol]) : 0.f);
    }
}

// The group of 16 / sizeof(T) consecutive output pixels whose 16-byte
// vectors this lane stores: group lane % (32 / that) of the 32 tile rows of
// lane quarter `quarter`, and the output index of its first pixel in the
// plane of the tile's first column.
struct OutGroup {
    int64_t base;
    bool valid;
};

template <typename T>
__device__ __forceinline__ OutGroup out_group(const Plan& pl, const TileId& id, int quarter, int lane) {
    constexpr int kVecPx = 16 / sizeof(T);
    constexpr int kGroups = 32 / kVecPx;
    const Pixel gp = tile_pixel(pl, id.mt, quarter * 32 + (lane % kGroups) * kVecPx);
    OutGroup og;
    og.base = (gp.n * pl.Cout + static_cast<int64_t>(id.g) * pl.Og + id.nt * pl.acc_cols) * pl.P + gp.ho * pl.Wo + gp.wo;
    og.valid = gp.valid;
    return og;
}

// 16 output channels (accumulator columns c16..c16+15) of the warp's 32 rows:
// + bias, converted, staged as [16 channels][32 pixels] in the warp's
// staging buffer, then stored as 16-byte vectors of consecutive pixels of
// one channel (one element per lane and channel where the layout does not
// allow vectors).
template <typename T>
__device__ __forceinline__ void store_chunk16(const Plan& pl, const FusedParams& prm, const TileId& id,
                                              const OutGroup& og, float* vals, int c16, int row, int lane,
                                              uint32_t bias_s, uint32_t stg) {
    const int32_t ncol0 = id.nt * pl.acc_cols;
    if (ncol0 + c16 >= pl.Og) return;
    T* __restrict__ out = static_cast<T*>(prm.out);
    if (prm.bias) {
#pragma unroll
        for (int e = 0; e < 16; ++e) vals[e] += ld_shared_f32(bias_s + 4u * (c16 + e));
    }
#pragma unroll
    for (int e = 0; e < 16; ++e) st_shared_elem<T>(stg + static_cast<uint32_t>((e * 32 + lane) * sizeof(T)), vals[e]);
    __syncwarp();
    if (prm.epi_vec) {
        constexpr int kVecPx = 16 / sizeof(T);
        constexpr int kGroups = 32 / kVecPx;
#pragma unroll
        for (int k = 0; k < 16 * kGroups / 32; ++k) {
            const int e = lane / kGroups + k * (32 / kGroups);  // channel of the chunk
            const uint32_t src = stg + static_cast<uint32_t>((e * 32 + (lane % kGroups) * kVecPx) * sizeof(T));
            if (og.valid && ncol0 + c16 + e < pl.Og)
                st_global_v4(out + og.base + static_cast<int64_t>(c16 + e) * pl.P, ld_shared_v4(src));
        }
    } else {
        const Pixel px = tile_pixel(pl, id.mt, row);
        if (px.valid) {
            T* o = out + (px.n * pl.Cout + static_cast<int64_t>(id.g) * pl.Og + ncol0 + c16) * pl.P +
                   px.ho * pl.Wo + px.wo;
            for (int e = 0; e < 16 && ncol0 + c16 + e < pl.Og; ++e)
                o[static_cast<int64_t>(e) * pl.P] = ld_shared_elem<T>(stg + static_cast<uint32_t>((e * 32 + lane) * sizeof(T)));
        }
    }
    __syncwarp();
}

// One kernel per (I/O type, KG = the plan's kgroups, AT = A stages in tensor
// memory): each instance holds only the gather variant it runs. The smaller
// binary reaches its first MMA sooner: start-up is dominated by instruction
// fetches of cold code.
template <int DT, int KG, bool AT>
__global__ void __launch_bounds__(kFusedThreads, 1)
    fused_kernel(const __grid_constant__ CUtensorMap tmap, const FusedParams prm) {
    using T = typename Elem<DT>::T;
    constexpr bool kF32Path = (DT == kF32);
    // tensor-memory A stages: each of a group's 4 warps writes the 32 tile rows
    // of its own lane quarter (warp % 4), two 16-row fragments per k-tile
    static_assert(!AT || (!kF32Path && KG == 2), "A in tensor memory: 16-bit types, two k-groups");
    const Plan& pl = prm.pl;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (sbase - raw);

    const int S = pl.stages;
    const uint32_t a_bytes = static_cast<uint32_t>(pl.a_bytes);
    const uint32_t b_bytes = static_cast<uint32_t>(pl.b_bytes);
    const uint32_t a0 = sbase;
    const uint32_t b0 = a0 + S * a_bytes;
    const uint32_t d0 = b0 + S * b_bytes;  // descriptor ring, 2 slots
    const uint32_t dslot = static_cast<uint32_t>(pl.desc_slot_bytes);
    const uint32_t e0s = d0 + 2 * dslot;  // epilogue staging: [16 channels][32 pixels] per warp
    const uint32_t bias_s = e0s + static_cast<uint32_t>(pl.epi_bytes);  // fp32 bias of the tile's columns
    const uint32_t bar0 = bias_s + static_cast<uint32_t>(kBiasBytes);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto tma_bar = [&](int s) { return bar0 + 8u * (S + s); };
    auto empty_bar = [&](int s) { return bar0 + 8u * (2 * S + s); };
    const uint32_t xb = bar0 + 8u * (3 * S);
    auto accf_bar = [&](int b) { return xb + 8u * b; };
    auto acce_bar = [&](int b) { return xb + 16u + 8u * b; };
    auto dfull_bar = [&](int b) { return xb + 32u + 8u * b; };
    auto dempty_bar = [&](int b) { return xb + 48u + 8u * b; };
    const uint32_t drain_bar = xb + 64u;
    // the gather warps arrive once they hold their registers: the other
    // warpgroups take their registers back (end of their roles) only after
    // that, so an early finisher cannot leave the gathers short of registers
    const uint32_t regs_bar = xb + 80u;
    const uint32_t slot_off = (xb - sbase) + 72u;
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(gbase + slot_off);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + slot_off + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int32_t KT = pl.KT;
    // this CTA's range of the k-tile sequence
    const int64_t lo = static_cast<int64_t>(blockIdx.x) * pl.kt_per_cta;
    const int64_t hi = min(lo + pl.kt_per_cta, pl.total_kt);

    if (warp == kWarpTma && lane == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), kGatherWarps / pl.kgroups);
            mbar_init(tma_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf_bar(b), 1);
            mbar_init(acce_bar(b), kEpiWarps);
            mbar_init(dfull_bar(b), 2);
            mbar_init(dempty_bar(b), kGatherWarps);
        }
        mbar_init(drain_bar, 1);
        mbar_init(regs_bar, kGatherWarps);
        *abort_flag = 0;
        fence_mbarrier_init();
        tma_prefetch_desc(&tmap);
    }
    if (warp == kWarpMma) {
        tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), static_cast<uint32_t>(pl.tmem_cols));
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    // The CTA's first descriptor group is sampled by all 512 threads together
    // (thread t: row t % 128, taps t / 128, t / 128 + 4, t / 128 + 8): the
    // first k-tiles of every role wait for it. Warps 2-3 then mark it full
    // and sample the following groups.
    {
        Cursor c0;
        cursor_init(pl, c0, lo, hi);
        if (c0.live) {
            const int64_t gd = static_cast<uint32_t>((c0.g * pl.Ug + c0.ul) * pl.U) / static_cast<uint32_t>(pl.Cd);
            sample_row_taps<T>(pl, static_cast<const T*>(prm.offset), static_cast<const T*>(prm.mask), c0.mt, gd,
                               threadIdx.x % kTileM, c0.b * kTapBlock, c0.ntbg, threadIdx.x / kTileM, 4,
                               gbase + (d0 - sbase), static_cast<uint32_t>(pl.desc_size));
        }
        // Everything so far reads only offset and mask; the channels-last x and
        // the packed weight come from the kernel launched before this one,
        // which this grid may overlap (programmatic dependent launch).
        asm volatile("griddepcontrol.wait;" ::: "memory");
        __syncthreads();
    }

    // Register split per warpgroup (launch: 128 per thread x 512 threads; the
    // host refuses to launch a build whose register count is not exactly 128):
    // TMA/MMA/sampling 88, gather 2 x 176, epilogue 72 -> 512 x 128 in total. Each
    // warpgroup's branch starts with its own setmaxnreg, so the compiler
    // allocates each role's code within that role's budget.
    const int wg = warp >> 2;
    if (wg == 0) {
    setmaxnreg_dec<kRegsCtrl>();
    if (warp == kWarpTma) {
        // ------------------------------------------------------------ TMA producer
        // The whole warp runs the loop; the elected lane issues.
        {
            const uint32_t sub_bytes = static_cast<uint32_t>(pl.BNs) * 128u;
            const uint32_t half_bytes = sub_bytes * pl.nsub;
            const int nsub = pl.nsub;
            Cursor kc;  // next weight k-tile to load
            cursor_init(pl, kc, lo, hi);
            bool ok = true;
            uint32_t s = 0, st = 0, ph = 0;
            while (kc.live && ok) {
                if (!warp_wait_bounded(empty_bar(st), ph ^ 1u, abort_flag, prm.status, kSiteTmaEmpty)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx_elect(tma_bar(st), b_bytes);
                const uint32_t dst = b0 + st * b_bytes;
                const int32_t row0 = kc.g * pl.Og + kc.nt * pl.acc_cols;
#pragma unroll
                for (int h = 0; h < (kF32Path ? 2 : 1); ++h)
#pragma unroll
                    for (int j = 0; j < 2; ++j)
                        if (j < nsub)
                            tma_load_2d_elect(dst + h * half_bytes + j * sub_bytes, &tmap, kc.kt * pl.BKc,
                                              row0 + h * static_cast<int32_t>(pl.Cout) + j * pl.BNs, tma_bar(st));
                ++s;
                if (++st == static_cast<uint32_t>(S)) {
                    st = 0;
                    ph ^= 1u;
                }
                cursor_advance(pl, kc);
            }
            if (!ok && lane == 0) {
                // let the copies already issued land before the CTA exits
                const uint32_t first = s > static_cast<uint32_t>(S) ? s - S : 0;
                volatile int never = 0;
                for (uint32_t q = first; q < s; ++q)
                    mbar_wait_bounded(tma_bar(q % S), (q / S) & 1, &never, prm.status, kSiteDrain, 200000000ull);
            }
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs the loop converged (its waits poll and vote on
        // every lane), so the descriptors stay in uniform registers; the
        // elected lane issues each tcgen05 instruction.
        {
            const uint32_t idesc = make_idesc(Elem<DT>::fmt, kTileM, static_cast<uint32_t>(pl.BNs));
            const uint32_t sub_bytes = static_cast<uint32_t>(pl.BNs) * 128u;
            const uint32_t half_bytes = sub_bytes * pl.nsub;
            const int nsub = pl.nsub;
            // Shared-memory descriptors differ only in their start-address field
            // (address >> 4, 14 bits): every descriptor of the loop is a base one
            // plus an offset. Per k-tile the warp waits, issues and commits.
            const uint64_t adesc0 = smem_desc_sw128(a0);
            const uint64_t bdesc0 = smem_desc_sw128(b0);
            const uint32_t a_step = a_bytes >> 4, b_step = b_bytes >> 4;
            const uint32_t sub_step = sub_bytes >> 4, half_step = half_bytes >> 4, alo_step = (kTileM * 128) >> 4;
            uint32_t st = 0, ph = 0, i = 0;
            bool ok = true;
            for (int64_t end = hi; end > lo && ok; ++i) {
                const Unit un = unit_back(pl, lo, end);
                end = un.t * KT + un.k0;
                const int ab = static_cast<int>(i % pl.nacc);
                const uint32_t use = i / pl.nacc;
                if (!warp_wait2(acce_bar(ab), 0u, (use & 1) ^ 1u, abort_flag, prm.status, kSiteMmaFull)) break;
                tc_fence_after();
                const uint32_t dacc = tmem_base + static_cast<uint32_t>(ab * pl.acc_cols);
                for (int32_t kt = un.k0; kt < un.k1; ++kt) {
                    // the A stage gathered and the B stage landed, polled together
                    if (!warp_wait2(full_bar(st), tma_bar(st), ph, abort_flag, prm.status, kSiteMmaFull)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = adesc0 + st * a_step;
                    const uint64_t bd = bdesc0 + st * b_step;
                    // A in tensor memory: stage st at column a_col0 + 32*st, 8 columns per K-step
                    const uint32_t at = tmem_base + static_cast<uint32_t>(pl.a_col0) + 32u * st;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {  // 4 MMA K-steps of 32 bytes per 128-byte k-tile
                        const uint32_t accum = (kt > un.k0 || kk > 0) ? 1u : 0u;
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            if (j < nsub) {
                                const uint32_t d = dacc + static_cast<uint32_t>(j * pl.BNs);
                                const uint64_t adesc = ad + 2u * kk;
                                const uint64_t bdesc = bd + j * sub_step + 2u * kk;
                                if constexpr (AT) {
                                    mma_f16_ts_elect(d, at + 8u * kk, bdesc, idesc, accum);
                                } else if constexpr (kF32Path) {
                                    mma_tf32_elect(d, adesc, bdesc, idesc, accum);
                                    mma_tf32_elect(d, adesc, bdesc + half_step, idesc, 1u);
                                    mma_tf32_elect(d, adesc + alo_step, bdesc, idesc, 1u);
                                } else {
                                    mma_f16_elect(d, adesc, bdesc, idesc, accum);
                                }
                            }
                        }
                    }
                    mma_commit_elect(empty_bar(st));
                    if (++st == static_cast<uint32_t>(S)) {
                        st = 0;
                        ph ^= 1u;
                    }
                }
                mma_commit_elect(accf_bar(ab));
            }
            // every MMA issued by the elected lane completes before TMEM is released
            mma_commit_elect(drain_bar);
            volatile int never = 0;
            warp_wait2(drain_bar, 0u, 0, &never, prm.status, kSiteDrain, 200000000ull);
        }
    } else {
        // ------------------------------------------------------------ sampling
        // Warps 2-3 fill the descriptor ring: for each descriptor group of the
        // CTA's range, in order, once every gather warp has released its slot:
        // thread t writes rows t and t + 64 for the group's taps.
        const T* offset = static_cast<const T*>(prm.offset);
        const T* mask = static_cast<const T*>(prm.mask);
        const int sid = (warp - 2) * 32 + lane;
        const uint32_t dsz = static_cast<uint32_t>(pl.desc_size);
        Cursor dc;  // first k-tile of the next group to sample
        cursor_init(pl, dc, lo, hi);
        if (dc.live) {  // the first group, sampled by every thread above
            if (lane == 0) mbar_arrive(dfull_bar(0));
            cursor_next_group(pl, dc);
        }
        while (dc.live) {
            const int slot = dc.gr & 1;
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(dempty_bar(slot), ((dc.gr >> 1) & 1) ^ 1u, abort_flag,
                                                           prm.status, kSiteTmaEmpty)))
                break;
            const int64_t unit = static_cast<int64_t>(dc.g) * pl.Ug + dc.ul;
            const int64_t gd = static_cast<uint32_t>(unit * pl.U) / static_cast<uint32_t>(pl.Cd);
            uint8_t* ring = gbase + (d0 - sbase) + slot * dslot;
            sample_rows<T>(pl, offset, mask, dc.mt, gd, sid, dc.b * kTapBlock, dc.ntbg, ring, dsz);
            __syncwarp();
            if (lane == 0) mbar_arrive(dfull_bar(slot));
            cursor_next_group(pl, dc);
        }
    }
    {
        volatile int never = 0;
        warp_wait_bounded(regs_bar, 0, &never, prm.status, kSiteDrain);
    }
    setmaxnreg_inc<kRegsLaunch>();
    } else if (wg == 1 || wg == 2) {
        setmaxnreg_inc<kRegsGather>();
        __syncwarp();
        if (lane == 0) mbar_arrive(regs_bar);
        // ------------------------------------------------------------ gather producers
        // k-tile-parallel gather: the 8 warps form G = pl.kgroups groups; group p
        // produces every G-th k-tile of the CTA's sequence (steps p, p + G, ...),
        // so G k-tiles are in production at once and a stage (stages are a
        // multiple of G) always belongs to one group. Each of a group's 8/G
        // warps handles 16*G rows as 2*G row-iterations of 8 rows, with the
        // corner loads of up to 4 row-iterations in flight (all of a k-tile's
        // for G <= 2; 4 registered buffers, the gather warps' 176 registers).
        // G is the kernel's compile-time KG.
        const int gw = warp - kWarpGather;
        auto gather = [&](auto g_const) {
            constexpr int G = decltype(g_const)::value;
            constexpr int wpg = kGatherWarps / G;  // warps per k-tile
            constexpr int nits = 2 * G;            // row-iterations per warp and k-tile
            // row-iterations whose corner loads are in flight at once (one
            // register buffer each): all of a k-tile's for G <= 2, else four
            constexpr int kDepth = nits < 4 ? nits : 4;
            const int pair = gw / wpg;
            GatherCtx<T> cx;
            cx.lane = lane;
            cx.q4 = lane & 3;     // lane's 32 bytes of the 128-byte row
            cx.rsub = lane >> 2;  // row within a group of 8
            cx.row0 = (gw % wpg) * 8 * nits;
            cx.xt = static_cast<const T*>(prm.xt);
            cx.d1 = 1;
            cx.dW = static_cast<int32_t>(pl.W);
            cx.dW1 = static_cast<int32_t>(pl.W + 1);
            cx.zpix = static_cast<int32_t>(pl.N * pl.H * pl.W);
            cx.pix_bytes = static_cast<int32_t>(pl.Cp * static_cast<int64_t>(sizeof(T)));
            cx.dsz = static_cast<uint32_t>(pl.desc_size);
            cx.row_desc = static_cast<uint32_t>(cx.row0 + cx.rsub) * cx.dsz;
            cx.row_sts = swz128(cx.row0 + cx.rsub, 2 * cx.q4);
            constexpr int kVec = 16 / sizeof(T);
            const int32_t ntb = pl.ntb, Kt = pl.K, nch = pl.nch, Ug = pl.Ug, BKc = pl.BKc;
            const int64_t UP = pl.UP;
            const int32_t ngroups = Ug * ntb;
            // this warp group's steps are pair, pair + G, ...: stage and phase advance by G
            uint32_t st = static_cast<uint32_t>(pair), phase = 0;
            uint32_t gr = 0;     // descriptor groups entered
            uint32_t sbase = 0;  // CTA step of the current unit's first k-tile
            bool ok = true;
            for (int64_t end = hi; end > lo && ok;) {
                const Unit un = unit_back(pl, lo, end);
                end = un.t * KT + un.k0;
                const TileId id = decode_tile(pl, un.t);
                int32_t q = 0;  // first k-tile (processing order) of the current group
                for (int32_t gi = 0; gi < ngroups && ok && q < un.k1; ++gi) {
                    const int32_t ul = gi / ntb;
                    const int32_t b = gi - ul * ntb;
                    const int32_t ntbg = min(kTapBlock, Kt - b * kTapBlock);
                    const int32_t nktg = ntbg * nch;
                    if (q + nktg <= un.k0) {  // group before the unit's range: not sampled
                        q += nktg;
                        continue;
                    }
                    const int slot = gr & 1;
                    if (!__all_sync(0xffffffffu, mbar_wait_bounded(dfull_bar(slot), (gr >> 1) & 1, abort_flag,
                                                                   prm.status, kSiteGatherEmpty))) {
                        ok = false;
                        break;
                    }
                    const uint32_t dbase = d0 + slot * dslot;
                    const int64_t unit = static_cast<int64_t>(id.g) * Ug + ul;
                    // k-tile j of the group is CTA step sbase + q + j - k0; this warp
                    // group takes the steps equal to pair modulo G
                    const int32_t jlo = max(un.k0 - q, 0), jhi = min(un.k1 - q, nktg);
                    const uint32_t s_lo = sbase + static_cast<uint32_t>(q + jlo - un.k0);
                    for (int32_t j = jlo + (pair - static_cast<int32_t>(s_lo % G) + G) % G; j < jhi; j += G) {
                        const int32_t ch = j / ntbg;
                        const int32_t kb = j - ch * ntbg;
                        const int64_t cb = unit * UP + static_cast<int64_t>(ch) * BKc + cx.q4 * 2 * kVec;
                        const char* cbp = reinterpret_cast<const char*>(cx.xt + cb);
                        const uint32_t dtap = dbase + static_cast<uint32_t>(kb * kTileM) * cx.dsz;
                        RowBuf rb[kDepth];
#pragma unroll
                        for (int q = 0; q < kDepth; ++q) row_issue<T, kF32Path>(cx, dtap, cbp, q, rb[q]);
                        // the stage is free once the MMAs that read it completed
                        // (tcgen05.commit); lane 0 polls, the warp follows it
                        int got = 0;
                        if (lane == 0)
                            got = mbar_wait_bounded(empty_bar(st), phase ^ 1u, abort_flag, prm.status,
                                                    kSiteGatherEmpty);
                        if (!__shfl_sync(0xffffffffu, got, 0)) {
                            ok = false;
                            break;
                        }
                        if constexpr (AT) {
                            // after the MMAs that read the stage: 16-row fragments
                            // (row-iterations 2p, 2p + 1) into the warp's lane quarter
                            static_assert(nits == kDepth && nits % 2 == 0, "every row-iteration loaded up front");
                            tc_fence_after();
                            const uint32_t ta = tmem_base + (static_cast<uint32_t>(cx.row0) << 16) +
                                                static_cast<uint32_t>(pl.a_col0) + 32u * st;
#pragma unroll
                            for (int pr = 0; pr < nits / 2; ++pr)
                                rows_to_tmem<T>(ta + ((16u * pr) << 16), rb[2 * pr], rb[2 * pr + 1]);
                            tmem_wait_st();
                            tc_fence_before();
                        } else {
                            const uint32_t a_s = a0 + st * a_bytes;
#pragma unroll
                            for (int it = 0; it < nits; ++it) {
                                row_combine<T, kF32Path>(cx, a_s, it, rb[it % kDepth]);
                                if (it + kDepth < nits)
                                    row_issue<T, kF32Path>(cx, dtap, cbp, it + kDepth, rb[it % kDepth]);
                            }
                            fence_proxy_async_smem();
                        }
                        __syncwarp();
                        if (lane == 0) mbar_arrive(full_bar(st));
                        st += G;
                        if (st >= static_cast<uint32_t>(S)) {
                            st -= S;
                            phase ^= 1u;
                        }
                    }
                    q += nktg;
                    // every gather warp releases every descriptor group, used or not
                    __syncwarp();
                    if (lane == 0) mbar_arrive(dempty_bar(slot));
                    ++gr;
                }
                sbase += static_cast<uint32_t>(un.k1 - un.k0);
            }
        };
        gather(std::integral_constant<int, KG>{});
        setmaxnreg_dec<kRegsLaunch>();
    } else {
        setmaxnreg_dec<kRegsEpi>();
        // ------------------------------------------------------------ epilogue
        // Every unit but the CTA's last (the tail below takes that one with all
        // 16 warps): a whole tile -> output, or the first unit of a tile whose
        // first k-tiles are another CTA's -> this CTA's partial slot.
        const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
        const int row = quarter * 32 + lane;
        uint32_t i = 0;
        for (int64_t end = hi; end > lo; ++i) {
            const Unit un = unit_back(pl, lo, end);
            end = un.t * KT + un.k0;
            if (end <= lo) break;  // the last unit
            const TileId id = decode_tile(pl, un.t);
            const int ab = static_cast<int>(i % pl.nacc);
            const uint32_t use = i / pl.nacc;
            // the four warps agree on going on (the named barriers below need all of them)
            if (!bar_red_and(1, kEpiWarps * 32,
                             __all_sync(0xffffffffu, mbar_wait_bounded(accf_bar(ab), use & 1, abort_flag, prm.status,
                                                                       kSiteEpilogue))))
                break;
            tc_fence_after();
            const uint32_t tl = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                static_cast<uint32_t>(ab * pl.acc_cols);
            if (un.k0 != 0 || un.k1 != KT) {
                // a split tile's first pieces: its last, and its owner, is a later CTA's
                const int64_t c_last = cta_of(pl, un.t * KT + KT - 1);
                for (int c32 = 0; c32 < pl.acc_cols; c32 += 32)
                    write_partial32<T>(pl, prm.part, blockIdx.x, tl, c32, row);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acce_bar(ab));
                count_in_split(prm.split_count + c_last, 1, kEpiWarps * 32, warp == kWarpEpi && lane == 0);
                continue;
            }
            if (prm.bias) {
                stage_bias<T>(pl, static_cast<const T*>(prm.bias), id, bias_s, row, kTileM);
                named_bar_sync(1, kEpiWarps * 32);
            }
            const OutGroup og = out_group<T>(pl, id, quarter, lane);
            for (int c16 = 0; c16 < pl.acc_cols; c16 += 16) {
                float vals[16];
                tmem_ld16(tl + static_cast<uint32_t>(c16), vals);
                store_chunk16<T>(pl, prm, id, og, vals, c16, row, lane, bias_s,
                                 e0s + static_cast<uint32_t>(quarter * 16 * 32 * sizeof(T)));
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acce_bar(ab));
        }
        {
            volatile int never = 0;
            warp_wait_bounded(regs_bar, 0, &never, prm.status, kSiteDrain);
        }
        setmaxnreg_inc<kRegsLaunch>();
    }

    // ---------------------------------------------------------------- tail
    // The pipeline has drained (the MMA warp waited for its last commit): the
    // CTA's last unit (the piece of the range's first tile) is in tensor
    // memory, and all 16 warps write it out, warp w taking lane quarter w % 4
    // and every fourth 32-column block from block w / 4. A split tile's piece
    // other than its last goes to this CTA's partial slot; the CTA holding a
    // split tile's last k-tiles (the owner) waits for the CTAs before it and
    // adds their partials, in k order, and its own accumulator last.
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (lo < hi && *abort_flag == 0) {
        int64_t end = hi;
        uint32_t nu = 0;
        Unit un;
        do {
            un = unit_back(pl, lo, end);
            end = un.t * KT + un.k0;
            ++nu;
        } while (end > lo);
        const TileId id = decode_tile(pl, un.t);
        const int ab = static_cast<int>((nu - 1) % pl.nacc);
        const int quarter = warp & 3, member = warp >> 2;
        const int row = quarter * 32 + lane;
        const uint32_t tl = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                            static_cast<uint32_t>(ab * pl.acc_cols);
        const bool split = un.k0 != 0 || un.k1 != KT;
        const int64_t me = blockIdx.x;
        const int64_t c_last = split ? cta_of(pl, un.t * KT + KT - 1) : me;
        if (c_last != me) {
            for (int c32 = 32 * member; c32 < pl.acc_cols; c32 += 128)
                write_partial32<T>(pl, prm.part, me, tl, c32, row);
            count_in_split(prm.split_count + c_last, 0, kFusedThreads, threadIdx.x == 0);
        } else {
            // the contributors: CTAs c_first .. me - 1 (none for a whole tile)
            const int64_t c_first = split ? cta_of(pl, un.t * KT) : me;
            const int32_t m = static_cast<int32_t>(me - c_first);
            if (prm.bias) stage_bias<T>(pl, static_cast<const T*>(prm.bias), id, bias_s, threadIdx.x, kFusedThreads);
            int ok = 1;
            if (m > 0 && threadIdx.x == 0) {
                ok = wait_count_bounded(prm.split_count + me, static_cast<uint32_t>(m), abort_flag, prm.status,
                                        kSiteSplitWait);
                if (ok) prm.split_count[me] = 0u;  // every contributor is in: zero again for the next call
            }
            if (__syncthreads_and(ok)) {
                const OutGroup og = out_group<T>(pl, id, quarter, lane);
                // per-warp staging in the (idle) descriptor ring
                const uint32_t stg = d0 + static_cast<uint32_t>(warp * 16 * 32 * sizeof(T));
                for (int c32 = 32 * member; c32 < pl.acc_cols; c32 += 128) {
                    const int nc = min(32, pl.acc_cols - c32);
                    float vals[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) vals[e] = 0.f;
                    for (int32_t k = 0; k < m; ++k) {
                        // one contributor's 32 columns, all loads in flight, then added
                        const float* src = prm.part + ((c_first + k) * pl.acc_cols + c32) * kTileM + row;
                        float pv[32];
#pragma unroll
                        for (int e = 0; e < 32; ++e) pv[e] = e < nc ? __ldcg(src + e * kTileM) : 0.f;
#pragma unroll
                        for (int e = 0; e < 32; ++e) vals[e] += pv[e];
                    }
                    float own[32];
                    tmem_ld32(tl + static_cast<uint32_t>(c32), nc == 32 ? 2 : 1, own);
#pragma unroll
                    for (int e = 0; e < 32; ++e) vals[e] += own[e];
                    store_chunk16<T>(pl, prm, id, og, vals, c32, row, lane, bias_s, stg);
                    if (nc > 16) store_chunk16<T>(pl, prm, id, og, vals + 16, c32 + 16, row, lane, bias_s, stg);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, static_cast<uint32_t>(pl.tmem_cols));
    }
}

// Tiny kernel for the bounded-wait self-test: waits on a barrier nothing signals.
__global__ void wait_selftest_kernel(uint32_t* status, uint64_t limit_cycles) {
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
        const bool ok = mbar_wait_bounded(smem_u32(&bar), 0, &abort_flag, status, kSiteSelftest, limit_cycles);
        if (ok) atomicOr(status, 1u << 31);  // the wait completed although nothing arrived
        mbar_arrive(smem_u32(&bar));        // complete the phase before exit
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
    const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(pl.KP), static_cast<cuuint64_t>(pl.wp_rows)};
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
    prm.part = reinterpret_cast<float*>(base + pl.off_part);
    prm.split_count = reinterpret_cast<uint32_t*>(base + kSplitCountOffset);
    prm.epi_vec = pl.epi_vec && (reinterpret_cast<uintptr_t>(out) & 15u) == 0 ? 1 : 0;
    prm.pl = pl;
    // launched dependent on the prep kernel: the prologue (barriers, tensor
    // memory, the first descriptor group) overlaps its tail
    cudaLaunchConfig_t fcfg = {};
    fcfg.gridDim = dim3(static_cast<unsigned>(pl.grid));
    fcfg.blockDim = dim3(kFusedThreads);
    fcfg.dynamicSmemBytes = static_cast<size_t>(pl.smem_bytes);
    fcfg.stream = st;
    cudaLaunchAttribute fattr[1];
    fattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    fattr[0].val.programmaticStreamSerializationAllowed = 1;
    fcfg.attrs = fattr;
    fcfg.numAttrs = 1;
    void (*kern)(CUtensorMap, FusedParams) =
        pl.kgroups == 1 ? fused_kernel<DT, 1, false>
                        : (pl.kgroups == 4 ? fused_kernel<DT, 4, false> : fused_kernel<DT, 2, false>);
    if constexpr (DT != kF32) {
        if (pl.a_tmem) kern = fused_kernel<DT, 2, true>;
    } else {
        if (pl.a_tmem) return cudaErrorInvalidValue;  // the planner never stages fp32 A in tensor memory
    }
    cudaError_t e = cudaLaunchKernelEx(&fcfg, kern, tmap, prm);
    if (e == cudaSuccess) e = cudaGetLastError();
    return e;
}

}  // namespace

// Sets the dynamic shared memory limit and checks that the build launches
// with exactly kRegsLaunch registers per thread (the warpgroup register
// split, setmaxnreg, is sized for that pool) and holds no static shared
// memory (the plan may give the whole per-CTA limit to dynamic shared
// memory); any other build is refused.
template <int DT, int KG, bool AT>
static cudaError_t prepare_variant(int smem_bytes) {
    cudaError_t e =
        cudaFuncSetAttribute(fused_kernel<DT, KG, AT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess) return e;
    cudaFuncAttributes attr;
    e = cudaFuncGetAttributes(&attr, fused_kernel<DT, KG, AT>);
    if (e != cudaSuccess) return e;
    return attr.numRegs == kRegsLaunch && attr.sharedSizeBytes == 0 ? cudaSuccess : cudaErrorInvalidDeviceFunction;
}

template <int DT>
static cudaError_t prepare_one(int smem_bytes) {
    cudaError_t e = prepare_variant<DT, 1, false>(smem_bytes);
    if (e == cudaSuccess) e = prepare_variant<DT, 2, false>(smem_bytes);
    if (e == cudaSuccess) e = prepare_variant<DT, 4, false>(smem_bytes);
    if constexpr (DT != kF32)
        if (e == cudaSuccess) e = prepare_variant<DT, 2, true>(smem_bytes);
    return e;
}

cudaError_t prepare_fused_attributes(int dtype, int smem_bytes) {
    switch (dtype) {
        case kF32: return prepare_one<kF32>(smem_bytes);
        case kF16: return prepare_one<kF16>(smem_bytes);
        default: return prepare_one<kBF16>(smem_bytes);
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

cudaError_t launch_wait_selftest(uint32_t* status, uint64_t limit_cycles, cudaStream_t st) {
    wait_selftest_kernel<<<1, 32, 0, st>>>(status, limit_cycles);
    return cudaGetLastError();
}

}  // namespace mdcn
