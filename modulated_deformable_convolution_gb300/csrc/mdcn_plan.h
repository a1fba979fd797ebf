// Problem description and execution plan of one forward call, shared by the
// host launcher and the kernels of libmdcn (never by the CPU oracle).
#pragma once

#include <cstddef>
#include <cstdint>

namespace mdcn {

constexpr int kTileM = 128;       // output pixels per CTA tile (MMA M)
constexpr int kTapBlock = 9;      // taps whose sample descriptors are cached at once
constexpr int kGatherWarps = 8;   // producer warps (16 tile rows each); also the epilogue warps
constexpr int kRowsPerWarp = kTileM / kGatherWarps;
constexpr int kFusedThreads = 64 + 32 * kGatherWarps;  // warp 0 TMA, warp 1 MMA, 8 gather/epilogue warps
constexpr int kDescBytes = 32;    // one cached sample descriptor
constexpr int kSmemLimit = 227 * 1024;
constexpr size_t kStatusBytes = 256;  // workspace header holding the device status word

enum DType : int32_t { kF32 = 0, kF16 = 1, kBF16 = 2 };

struct Plan {
    // ---- problem (section 2 layouts, section 3 attributes)
    int64_t N, Cin, H, W, Cout, kh, kw, Ho, Wo;
    int32_t sh, sw, ph, pw, dh, dw;
    int32_t group, dg;
    int32_t dtype;
    int32_t has_bias;
    int32_t K;        // taps kh*kw
    int32_t Cg, Og, Cd;
    int64_t P;        // Ho*Wo
    int64_t NP;       // N*Ho*Wo output pixels

    // ---- channel units: U = gcd(Cin/group, Cin/dg) consecutive channels
    // share one convolution group and one deformable group. In the
    // channels-last copy of x and in the packed weight each unit is padded to
    // UP = roundup(U, BKc) channels with zeros.
    int32_t U, UP, Ug, nch;  // Ug = units per group, nch = UP / BKc
    int32_t BKc;             // channels per k-tile: 128 bytes of the element type
    int32_t ntb;             // tap blocks = ceil(K / kTapBlock)
    int32_t KT;              // k-tiles per group = Ug * K * nch
    int64_t Cp;              // padded channels of the channels-last x = (Cin/U)*UP
    int64_t KP;              // packed weight row length = KT * BKc
    int64_t wp_rows;         // packed weight rows: Cout (x2 for f32 hi/lo), at least BNs, zero-padded

    // ---- tiling of the fused kernel
    int32_t BNs;             // output channels per MMA (multiple of 16, <= 256)
    int32_t nsub;            // MMAs per k-step along N (1 or 2)
    int32_t ntiles_n;        // N tiles per group
    int64_t mtiles;          // ceil(NP / kTileM)
    int32_t stages;
    int32_t tmem_cols;
    int32_t a_bytes;         // one A stage (both tf32 halves for f32)
    int32_t b_bytes;         // one B stage
    int32_t desc_bytes;      // sample-descriptor cache
    int32_t smem_bytes;      // dynamic shared memory of the fused kernel

    // ---- workspace layout (byte offsets)
    size_t off_xt, off_wp, ws_bytes;
};

}  // namespace mdcn
