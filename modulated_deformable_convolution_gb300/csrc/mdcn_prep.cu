// Layout-prep kernels of the fused path:
//   x      [N, Cin, H, W]      -> xt [N*H*W + 1, Cp] (channels-last, units padded,
//                                 then one all-zero pixel;
//                                 a register-blocked kernel where H*W and the
//                                 unit are multiples of 16 bytes of elements,
//                                 a shared-memory staged one otherwise)
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

// The all-zero pixel after the image data (read for corners outside the
// image), written by one block: Cp elements, 16 bytes per thread and pass.
template <typename T>
__device__ __forceinline__ void write_zero_pixel(T* zp, int64_t Cp, int nthreads, int tid) {
    const int64_t nv = Cp * static_cast<int64_t>(sizeof(T)) / 16;
    for (int64_t v = tid; v < nv; v += nthreads) reinterpret_cast<uint4*>(zp)[v] = make_uint4(0u, 0u, 0u, 0u);
}

// One block converts a run of up to 32 pixels of one (n, h) row: it loads
// x[n, :, h, w0:w0+wc] (a warp reads 32 consecutive w of one channel) into
// shared memory as [pixel][padded channel] (pad channels zero), then writes
// the wc*Cp contiguous elements of the channels-last row with 16-byte stores.
// Block 0 also clears the device status word and writes the zero pixel. Block (32, 8); grid
// x = (n*H + h) * wchunks + chunk.
template <typename T>
__global__ void __launch_bounds__(256) nhwc_pad_kernel(const T* __restrict__ x, T* __restrict__ xt,
                                                       uint32_t* __restrict__ status, int32_t Cin, int64_t H,
                                                       int64_t W, int64_t Cp, int32_t U, int32_t UP, int32_t WC,
                                                       int64_t wchunks, int64_t zero_off) {
    extern __shared__ uint4 prep_smem[];
    T* sm = reinterpret_cast<T*>(prep_smem);
    constexpr int kVec = 16 / sizeof(T);
    const int32_t pitch = static_cast<int32_t>(Cp) + kVec;  // elements per staged pixel (16-byte multiple)
    const int tid = threadIdx.y * 32 + threadIdx.x;
    if (blockIdx.x == 0) {
        if (tid == 0) *status = 0u;
        for (int i = tid; i < kMaxCtas; i += 256) status[kSplitCountOffset / 4 + i] = 0u;
        write_zero_pixel(xt + zero_off, Cp, 256, tid);
    }
    const int64_t bx = blockIdx.x;
    const int64_t nh = bx / wchunks;
    const int64_t w0 = (bx - nh * wchunks) * WC;
    const int64_t n = nh / H;
    const int64_t h = nh - n * H;
    const int32_t wc = static_cast<int32_t>(W - w0 < WC ? W - w0 : WC);
    const int32_t nvec = wc * pitch / kVec;
    for (int32_t v = tid; v < nvec; v += 256) prep_smem[v] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
    const T* src = x + (n * Cin * H + h) * W + w0 + threadIdx.x;
    if (static_cast<int32_t>(threadIdx.x) < wc) {
        // 8 channel loads in flight per thread, then their shared-memory stores
        const int64_t cstride = H * W;
        for (int32_t c0 = threadIdx.y; c0 < Cin; c0 += 64) {
            T v[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int32_t c = c0 + 8 * k;
                if (c < Cin) v[k] = src[static_cast<int64_t>(c) * cstride];
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int32_t c = c0 + 8 * k;
                if (c < Cin) {
                    const int32_t unit = c / U;
                    sm[threadIdx.x * pitch + unit * UP + (c - unit * U)] = v[k];
                }
            }
        }
    }
    __syncthreads();
    uint4* dst = reinterpret_cast<uint4*>(xt + (nh * W + w0) * Cp);
    const int32_t cvec = static_cast<int32_t>(Cp) / kVec;
    const int32_t nout = wc * cvec;
    for (int32_t v = tid; v < nout; v += 256) {
        const int32_t w = v / cvec;
        const int32_t cv = v - w * cvec;
        dst[v] = *reinterpret_cast<const uint4*>(sm + w * pitch + cv * kVec);
    }
}

// Register-blocked conversion, for images whose pixel count H*W and channel
// unit U are multiples of kVec = 16 / sizeof(T) (8 for 16-bit types, 4 for
// fp32). Each lane moves one kVec-channel x kVec-pixel block: kVec 16-byte
// loads (kVec pixels of one channel each), a transpose in registers, and kVec
// 16-byte stores (kVec channels of one pixel each). A warp covers 8 channel
// groups x 4 pixel groups; output channels in a unit's padding are written as
// zeros. Grid (ceil(pixel blocks / 8), channel blocks, N), 8 warps per block,
// one pixel block (4 * kVec pixels) per warp. Block (0, 0, 0) also clears the
// device status word and writes the zero pixel.
template <typename T>
__device__ __forceinline__ void nhwc_block_body(const T* __restrict__ x, T* __restrict__ xt,
                                                uint32_t* __restrict__ status, int32_t Cin, int64_t P, int64_t Cp,
                                                int32_t U, int32_t UP, int64_t zero_off, uint32_t bx, uint32_t by,
                                                uint32_t bz) {
    constexpr int kVec = 16 / sizeof(T);
    if (bx == 0 && by == 0 && bz == 0) {
        if (threadIdx.x == 0) *status = 0u;
        for (int i = threadIdx.x; i < kMaxCtas; i += 256) status[kSplitCountOffset / 4 + i] = 0u;
        write_zero_pixel(xt + zero_off, Cp, 256, threadIdx.x);
    }
    const int lane = threadIdx.x & 31;
    const int cg = lane & 7, pg = lane >> 3;
    const int64_t n = bz;
    const int64_t oc0 = (static_cast<int64_t>(by) * 8 + cg) * kVec;  // output channel (padded)
    const int64_t p0 = ((static_cast<int64_t>(bx) * 8 + (threadIdx.x >> 5)) * 4 + pg) * kVec;
    if (oc0 >= Cp || p0 >= P) return;
    const int32_t unit = static_cast<int32_t>(static_cast<uint32_t>(oc0) / static_cast<uint32_t>(UP));  // Cp < 2^21
    const int32_t within = static_cast<int32_t>(oc0) - unit * UP;
    uint4 in[kVec];
    if (within < U) {
        const T* src = x + (n * Cin + static_cast<int64_t>(unit) * U + within) * P + p0;
#pragma unroll
        for (int i = 0; i < kVec; ++i) in[i] = __ldg(reinterpret_cast<const uint4*>(src + i * P));
    } else {
#pragma unroll
        for (int i = 0; i < kVec; ++i) in[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    uint4 out[kVec];
    if constexpr (kVec == 8) {
        // 8x8 halves: pair channels (c, c+1) per pixel, then pick words
        uint32_t w[8][4], t[8][4];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            w[c][0] = in[c].x;
            w[c][1] = in[c].y;
            w[c][2] = in[c].z;
            w[c][3] = in[c].w;
        }
#pragma unroll
        for (int c = 0; c < 8; c += 2)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                t[c][k] = __byte_perm(w[c][k], w[c + 1][k], 0x5410);      // (c, c+1) at pixel 2k
                t[c + 1][k] = __byte_perm(w[c][k], w[c + 1][k], 0x7632);  // (c, c+1) at pixel 2k+1
            }
#pragma unroll
        for (int q = 0; q < 8; ++q)
            out[q] = make_uint4(t[0 + (q & 1)][q >> 1], t[2 + (q & 1)][q >> 1], t[4 + (q & 1)][q >> 1],
                                t[6 + (q & 1)][q >> 1]);
    } else {
        // 4x4 words
        out[0] = make_uint4(in[0].x, in[1].x, in[2].x, in[3].x);
        out[1] = make_uint4(in[0].y, in[1].y, in[2].y, in[3].y);
        out[2] = make_uint4(in[0].z, in[1].z, in[2].z, in[3].z);
        out[3] = make_uint4(in[0].w, in[1].w, in[2].w, in[3].w);
    }
    T* dst = xt + (n * P + p0) * Cp + oc0;
#pragma unroll
    for (int q = 0; q < kVec; ++q) *reinterpret_cast<uint4*>(dst + q * Cp) = out[q];
}

template <typename T>
__global__ void __launch_bounds__(256) nhwc_block_kernel(const T* __restrict__ x, T* __restrict__ xt,
                                                         uint32_t* __restrict__ status, int32_t Cin, int64_t P,
                                                         int64_t Cp, int32_t U, int32_t UP, int64_t zero_off) {
    nhwc_block_body<T>(x, xt, status, Cin, P, Cp, U, UP, zero_off, blockIdx.x, blockIdx.y, blockIdx.z);
}

template <typename T>
__device__ __forceinline__ float load_f(const T* p);
template <>
__device__ __forceinline__ float load_f<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float load_f<__half>(const __half* p) { return __half2float(*p); }
template <>
__device__ __forceinline__ float load_f<__nv_bfloat16>(const __nv_bfloat16* p) { return __bfloat162float(*p); }

// Weight rows per pack thread and pass: 8 for 16-bit types, 4 for fp32
// (whose pass also splits each value into tf32 hi and lo; measured best).
template <typename T>
__host__ __device__ constexpr int pack_rows() { return sizeof(T) == 4 ? 4 : 8; }

// Packs the weight into the fused kernel's K order (zero pad included).
// Grid: x over k-tiles of one row (blockDim.x = BKc lanes per k-tile, several
// k-tiles per block), y over rows (looping when rows exceed the grid).
template <typename T>
__device__ __forceinline__ void pack_weight_body(const T* __restrict__ weight, T* __restrict__ wp, const Plan& pl,
                                                 uint32_t bx, uint32_t by, uint32_t gy) {
    const int64_t rows = pl.Cout * (pl.dtype == kF32 ? 2 : 1);
    const int32_t ktiles_per_block = 256 / pl.BKc;
    const int32_t kt = static_cast<int32_t>(bx) * ktiles_per_block + static_cast<int32_t>(threadIdx.x) / pl.BKc;
    const int32_t ci = static_cast<int32_t>(threadIdx.x) % pl.BKc;
    if (kt >= pl.KT) return;
    const KTile t = decode_ktile(kt, pl.K, pl.nch);
    // channel within the unit held at K position ci of the k-tile (A stages in
    // tensor memory: the order of the gather's fragments, kperm16)
    const int32_t within = t.ch * pl.BKc + (pl.a_tmem ? kperm16(ci) : ci);
    const int64_t cl = static_cast<int64_t>(t.ul) * pl.U + within;  // channel within the group
    // kRows rows per iteration: their loads are in flight together
    constexpr int kRows = pack_rows<T>();
    for (int64_t r0 = by; r0 < pl.wp_rows; r0 += kRows * static_cast<int64_t>(gy)) {
        T v[kRows];
#pragma unroll
        for (int k = 0; k < kRows; ++k) {
            const int64_t r = r0 + k * static_cast<int64_t>(gy);
            v[k] = zero_of<T>();
            if (within < pl.U && r < rows) {
                const bool lo_half = r >= pl.Cout;
                const int64_t o = lo_half ? r - pl.Cout : r;
                const T* src = weight + (o * pl.Cg + cl) * pl.K + t.tap;
                if constexpr (sizeof(T) == 4) {
                    const float f = load_f<T>(src);
                    const float hi = to_tf32(f);
                    v[k] = lo_half ? (f - hi) : hi;
                } else {
                    v[k] = *src;
                }
            }
        }
#pragma unroll
        for (int k = 0; k < kRows; ++k) {
            const int64_t r = r0 + k * static_cast<int64_t>(gy);
            if (r < pl.wp_rows) wp[r * pl.KP + static_cast<int64_t>(kt) * pl.BKc + ci] = v[k];
        }
    }
}

template <typename T>
__global__ void __launch_bounds__(256) pack_weight_kernel(const T* __restrict__ weight, T* __restrict__ wp, Plan pl) {
    pack_weight_body<T>(weight, wp, pl, blockIdx.x, blockIdx.y, gridDim.y);
}

// Both prep steps in one launch (register-blocked transpose blocks first,
// then weight-pack blocks); the fused kernel, launched dependent on it,
// may start its prologue as soon as every block of this grid has begun.
template <typename T>
__global__ void __launch_bounds__(256) prep_both_kernel(const T* __restrict__ x, const T* __restrict__ weight,
                                                        T* __restrict__ xt, T* __restrict__ wp,
                                                        uint32_t* __restrict__ status, Plan pl, uint32_t tgx,
                                                        uint32_t tgy, uint32_t nt, uint32_t pgx, uint32_t pgy,
                                                        const char* __restrict__ offset, uint32_t offset_lines,
                                                        const char* __restrict__ mask, uint32_t mask_lines) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const uint32_t b = blockIdx.x;
    // offset and mask into L2 (128-byte lines spread over the blocks): the
    // fused kernel's sampling then reads them from L2, not DRAM
    {
        const uint32_t lines = offset_lines + mask_lines;
        const uint32_t per = (lines + gridDim.x - 1) / gridDim.x;
        for (uint32_t l = b * per + threadIdx.x; l < min(lines, (b + 1) * per); l += blockDim.x)
            prefetch_l2(l < offset_lines ? offset + static_cast<size_t>(l) * 128
                                         : mask + static_cast<size_t>(l - offset_lines) * 128);
    }
    if (b < nt) {
        nhwc_block_body<T>(x, xt, status, static_cast<int32_t>(pl.Cin), pl.H * pl.W, pl.Cp, pl.U, pl.UP,
                           pl.N * pl.H * pl.W * pl.Cp, b % tgx, (b / tgx) % tgy, b / (tgx * tgy));
    } else {
        const uint32_t q = b - nt;
        pack_weight_body<T>(weight, wp, pl, q % pgx, q / pgx, pgy);
    }
}

}  // namespace

constexpr int64_t kPrepSmemBytes = 40 * 1024;

// Grid of the register-blocked transpose, or false when the shape needs the
// shared-memory staged one.
template <typename T>
static bool block_transpose_grid(const Plan& pl, dim3* grid) {
    constexpr int64_t kVec = 16 / static_cast<int64_t>(sizeof(T));
    const int64_t P = pl.H * pl.W;
    const int64_t pblocks = (P / kVec + 3) / 4;        // 4 * kVec pixels per warp
    const int64_t cblocks = (pl.Cp / kVec + 7) / 8;    // 8 * kVec output channels per warp
    if (!pl.xt_block) return false;  // the planner's check of the same conditions
    *grid = dim3(static_cast<unsigned>((pblocks + 7) / 8), static_cast<unsigned>(cblocks), static_cast<unsigned>(pl.N));
    return true;
}

template <typename T>
static void pack_grid(const Plan& pl, unsigned* gx, unsigned* gy) {
    const int32_t ktiles_per_block = 256 / pl.BKc;
    *gx = static_cast<unsigned>((pl.KT + ktiles_per_block - 1) / ktiles_per_block);
    const int64_t gyr = (pl.wp_rows + pack_rows<T>() - 1) / pack_rows<T>();
    *gy = static_cast<unsigned>(gyr < 65535 ? gyr : 65535);
}

template <typename T>
static cudaError_t prep_input_t(const Plan& pl, const void* x, void* ws, cudaStream_t st) {
    uint8_t* base = static_cast<uint8_t*>(ws);
    uint32_t* status = reinterpret_cast<uint32_t*>(base);
    T* xt = reinterpret_cast<T*>(base + pl.off_xt);
    const int64_t P = pl.H * pl.W;
    dim3 grid;
    if (block_transpose_grid<T>(pl, &grid)) {
        nhwc_block_kernel<T><<<grid, 256, 0, st>>>(static_cast<const T*>(x), xt, status,
                                                   static_cast<int32_t>(pl.Cin), P, pl.Cp, pl.U, pl.UP,
                                                   pl.N * P * pl.Cp);
        return cudaGetLastError();
    }
    const int64_t pitch_bytes = (pl.Cp + 16 / static_cast<int64_t>(sizeof(T))) * static_cast<int64_t>(sizeof(T));
    int64_t wc = kPrepSmemBytes / pitch_bytes;
    if (wc > 32) wc = 32;
    if (wc > pl.W) wc = pl.W;
    if (wc < 1) return cudaErrorInvalidConfiguration;  // a pixel's channels exceed the staging buffer
    const int64_t wchunks = (pl.W + wc - 1) / wc;
    const size_t smem = static_cast<size_t>(wc * pitch_bytes);
    nhwc_pad_kernel<T><<<static_cast<unsigned>(pl.N * pl.H * wchunks), dim3(32, 8), smem, st>>>(
        static_cast<const T*>(x), xt, status, static_cast<int32_t>(pl.Cin), pl.H, pl.W, pl.Cp, pl.U, pl.UP,
        static_cast<int32_t>(wc), wchunks, pl.N * pl.H * pl.W * pl.Cp);
    return cudaGetLastError();
}

template <typename T>
static cudaError_t pack_weight_t(const Plan& pl, const void* weight, void* ws, cudaStream_t st) {
    uint8_t* base = static_cast<uint8_t*>(ws);
    T* wp = reinterpret_cast<T*>(base + pl.off_wp);
    unsigned gx, gy;
    pack_grid<T>(pl, &gx, &gy);
    pack_weight_kernel<T><<<dim3(gx, gy), 256, 0, st>>>(static_cast<const T*>(weight), wp, pl);
    return cudaGetLastError();
}

template <typename T>
static cudaError_t prep_both_t(const Plan& pl, const void* x, const void* weight, const void* offset,
                               size_t offset_bytes, const void* mask, size_t mask_bytes, void* ws, cudaStream_t st) {
    dim3 tg;
    if (!block_transpose_grid<T>(pl, &tg)) {
        const cudaError_t e = prep_input_t<T>(pl, x, ws, st);
        return e != cudaSuccess ? e : pack_weight_t<T>(pl, weight, ws, st);
    }
    unsigned pgx, pgy;
    pack_grid<T>(pl, &pgx, &pgy);
    const uint64_t nt = static_cast<uint64_t>(tg.x) * tg.y * tg.z;
    const uint64_t np = static_cast<uint64_t>(pgx) * pgy;
    if (nt + np > 2147483647ull) {
        const cudaError_t e = prep_input_t<T>(pl, x, ws, st);
        return e != cudaSuccess ? e : pack_weight_t<T>(pl, weight, ws, st);
    }
    uint8_t* base = static_cast<uint8_t*>(ws);
    prep_both_kernel<T><<<static_cast<unsigned>(nt + np), 256, 0, st>>>(
        static_cast<const T*>(x), static_cast<const T*>(weight), reinterpret_cast<T*>(base + pl.off_xt),
        reinterpret_cast<T*>(base + pl.off_wp), reinterpret_cast<uint32_t*>(base), pl, tg.x, tg.y,
        static_cast<uint32_t>(nt), pgx, pgy, static_cast<const char*>(offset),
        static_cast<uint32_t>(offset_bytes / 128), static_cast<const char*>(mask), static_cast<uint32_t>(mask_bytes / 128));
    return cudaGetLastError();
}

namespace {

template <typename T>
__device__ __forceinline__ T store_of(float v);
template <>
__device__ __forceinline__ float store_of<float>(float v) { return v; }
template <>
__device__ __forceinline__ __half store_of<__half>(float v) { return __float2half_rn(v); }
template <>
__device__ __forceinline__ __nv_bfloat16 store_of<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// Grid (x over each plane's P elements, 4 per thread; y over the planes
// n * (c_off + c_mask) + c, looping past the grid): a plane below c_off is
// copied to the offset, a plane from c_off goes through the logistic
// sigmoid (fp32) into the mask.
template <typename T>
__global__ void __launch_bounds__(256) split_offset_mask_kernel(const T* __restrict__ om, T* __restrict__ offset,
                                                                T* __restrict__ mask, int64_t planes, int64_t c_off,
                                                                int64_t c_mask, int64_t P) {
    const int64_t ct = c_off + c_mask;
    for (int64_t pl = blockIdx.y; pl < planes; pl += gridDim.y) {
        const int64_t n = pl / ct, c = pl - n * ct;
        const T* src = om + pl * P;
        T* dst = c < c_off ? offset + (n * c_off + c) * P : mask + (n * c_mask + (c - c_off)) * P;
        const bool sig = c >= c_off;
        for (int64_t i = (static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x) * 4; i < P;
             i += static_cast<int64_t>(gridDim.x) * 256 * 4) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                if (i + k < P) {
                    const T v = src[i + k];
                    dst[i + k] = sig ? store_of<T>(1.0f / (1.0f + expf(-load_f<T>(&v)))) : v;
                }
            }
        }
    }
}

template <typename T>
cudaError_t split_t(const Plan& pl, const void* om, void* offset, void* mask, int64_t c_off, int64_t c_mask,
                    cudaStream_t st) {
    const int64_t planes = pl.N * (c_off + c_mask);
    const int64_t gx = (pl.P + 1023) / 1024;
    const unsigned gy = static_cast<unsigned>(planes < 65535 ? planes : 65535);
    split_offset_mask_kernel<T><<<dim3(static_cast<unsigned>(gx < 1024 ? gx : 1024), gy), 256, 0, st>>>(
        static_cast<const T*>(om), static_cast<T*>(offset), static_cast<T*>(mask), planes, c_off, c_mask, pl.P);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_split_offset_mask(const Plan& pl, const void* om, void* offset, void* mask, int64_t c_off,
                                     int64_t c_mask, cudaStream_t st) {
    switch (pl.dtype) {
        case kF32: return split_t<float>(pl, om, offset, mask, c_off, c_mask, st);
        case kF16: return split_t<__half>(pl, om, offset, mask, c_off, c_mask, st);
        default: return split_t<__nv_bfloat16>(pl, om, offset, mask, c_off, c_mask, st);
    }
}

cudaError_t launch_prep_both(const Plan& pl, const void* x, const void* weight, const void* offset,
                             size_t offset_bytes, const void* mask, size_t mask_bytes, void* ws, cudaStream_t st) {
    // line counts fit 32 bits for any offset/mask below 512 GB
    if (offset_bytes / 128 > 0xffffffffull / 2 || mask_bytes / 128 > 0xffffffffull / 2) offset_bytes = mask_bytes = 0;
    switch (pl.dtype) {
        case kF32: return prep_both_t<float>(pl, x, weight, offset, offset_bytes, mask, mask_bytes, ws, st);
        case kF16: return prep_both_t<__half>(pl, x, weight, offset, offset_bytes, mask, mask_bytes, ws, st);
        default: return prep_both_t<__nv_bfloat16>(pl, x, weight, offset, offset_bytes, mask, mask_bytes, ws, st);
    }
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
