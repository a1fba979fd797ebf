// Problem description and execution plan of one forward call, shared by the
// host launcher and the kernels of libmdcn (never by the CPU oracle).
#pragma once

#include <cstddef>
#include <cstdint>

namespace mdcn {

constexpr int kTileM = 128;       // output pixels per tile (MMA M)
constexpr int kTileH = 8;         // 2-D tile: kTileH image rows x kTileW pixels
constexpr int kTileW = 16;
static_assert(kTileH * kTileW == kTileM, "2-D tile covers one tile");
constexpr int kTapBlock = 9;      // taps whose sample descriptors form one descriptor group
// Warp roles of the fused kernel (16 warps):
constexpr int kWarpTma = 0;       // TMA loads of weight k-tiles
constexpr int kWarpMma = 1;       // TMEM allocation; lane 0 issues tcgen05.mma
constexpr int kWarpGather = 4;    // 8 warps: gather + modulate into A stages
constexpr int kGatherWarps = 8;
constexpr int kWarpEpi = 12;      // 4 warps: TMEM -> +bias -> NCHW
constexpr int kEpiWarps = 4;
constexpr int kFusedThreads = 32 * 16;
// Registers per thread: at launch, and per warpgroup after setmaxnreg
// (warpgroup 0 = TMA/MMA/sampling, 1-2 = gather, 3 = epilogue).
constexpr int kRegsLaunch = 128;
constexpr int kRegsCtrl = 88;
constexpr int kRegsGather = 176;
constexpr int kRegsEpi = 72;
static_assert(kRegsCtrl + 2 * kRegsGather + kRegsEpi == 4 * kRegsLaunch, "warpgroup register split must fit");
constexpr int kSmemLimit = 227 * 1024;
constexpr int kMaxCtas = 160;         // persistent CTAs at most (one per SM; the workspace holds a partial slot each)
constexpr size_t kStatusBytes = 1024;     // workspace header: the device status word, the split-tile counters
constexpr size_t kSplitCountOffset = 64;  // uint32[kMaxCtas]: per split tile (by its first CTA), epilogue warps done
static_assert(kSplitCountOffset + 4 * kMaxCtas <= kStatusBytes, "split counters must fit the header");
constexpr int kBiasBytes = 512 * 4;  // the epilogue's fp32 copy of one tile's bias columns (up to 512)
// the tail's per-warp output staging (16 x [16 channels][32 pixels]) lives in
// the descriptor ring, which is idle by then
static_assert(kFusedThreads / 32 * 16 * 32 * 4 <= 2 * kTileM * kTapBlock * 16, "tail staging must fit the ring");

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
    int32_t tile_mode;       // 0: 128 consecutive pixels of N*Ho*Wo; 1: TH x TW block of one image
    int32_t TH, TW;          // 2-D tile shape (TH*TW = 128)
    int64_t tiles_x, tiles_y;
    int64_t mtiles;          // pixel tiles
    int64_t tiles_total;     // mtiles * ntiles_n * group
    int32_t BNs;             // output channels per MMA (multiple of 16, <= 256)
    int32_t nsub;            // MMAs per k-step along N (1 or 2)
    int32_t ntiles_n;        // N tiles per group
    int32_t acc_cols;        // TMEM columns of one accumulator = nsub * BNs
    int32_t nacc;            // accumulators in TMEM (2: epilogue overlaps the next tile)
    int32_t tmem_cols;
    int32_t direct;          // 1: the direct CUDA-core kernel (little contraction per output, e.g.
                             //    depthwise); none of the fused-path fields below is set
    int32_t direct_cl;       // 1 (with direct): its depthwise form on a channels-last copy of x at
                             //    off_xt, [N*H*W + 1][Cin] (the last pixel zero)
    int32_t a_tmem;          // 1: the A stages (modulated columns) live in tensor memory, written by the
                             //    gather with tcgen05.st and read by the MMA from there (16-bit types, 2
                             //    k-groups); 0: 128-byte-swizzled shared-memory stages
    int32_t a_col0;          // tensor-memory column of A stage 0 (after the accumulators); stage s at + 32*s
    int32_t stages;          // 2, 4, 6 or 8
    int32_t kgroups;         // k-tiles produced concurrently by the gather warps (1, 2 or 4; divides stages)
    int32_t a_bytes;         // one A stage (both tf32 halves for f32)
    int32_t b_bytes;         // one B stage
    int32_t desc_size;       // bytes per sample descriptor (16, or 32 for f32)
    int32_t desc_slot_bytes; // one descriptor group: kTileM rows x kTapBlock taps
    int32_t epi_vec;         // 1: output groups of 16 bytes of consecutive pixels stay aligned and whole
    int32_t plain;           // 1: an ordinary convolution (no offset or mask read: every offset 0, mask 1)
    int32_t epi_bytes;       // shared-memory staging of the TMA-store epilogue
    int32_t smem_bytes;      // dynamic shared memory of the fused kernel
    int32_t grid;            // persistent CTAs
    int32_t xt_block;        // 1: x goes channels-last through the register-blocked kernel, which
                             //    mdcn_forward launches together with the weight pack
    int64_t total_kt;        // k-tiles of all tiles: tiles_total * KT
    int64_t kt_per_cta;      // stream-K: consecutive k-tiles per CTA (set with grid)

    // ---- workspace layout (byte offsets)
    size_t off_xt, off_wp, off_part, ws_bytes;
};

// True when some tile's k-tiles fall to more than one CTA (the CTA ranges do
// not all end on tile boundaries), so some tile is finished from partials.
inline bool splitk_needed(const Plan& p) { return p.grid > 1 && p.kt_per_cta % p.KT != 0; }

}  // namespace mdcn
