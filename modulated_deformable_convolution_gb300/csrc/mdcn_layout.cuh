// K-order of the implicit GEMM and the padded channel layout shared by the
// layout-prep kernels and the fused kernel.
//
// Within convolution group g the contraction index runs over
//   unit ul (U consecutive channels of one deformable group)
//     tap block b (up to kTapBlock taps)
//       channel chunk ch (BKc channels = 128 bytes)
//         tap kb of the block
//           channel ci of the chunk
// so one k-tile is BKc channels of one tap, every channel of a k-tile has
// the same sampling position, and the consecutive k-tiles of a chunk revisit
// the same channels of x at neighbouring positions (cache reuse). The
// channels-last copy of x pads each unit to UP channels, so every 16-byte
// vector load of a k-tile is aligned and in bounds, and the pad reads zero.
#pragma once

#include "mdcn_plan.h"

namespace mdcn {

struct KTile {
    int32_t ul;  // unit within the group
    int32_t b;   // tap block
    int32_t ch;  // channel chunk within the unit
    int32_t kb;  // tap within the block
    int32_t tap; // tap index i*kw + j
    int32_t ntb; // taps in this block
};

// Order of the 64 channels of a 16-bit k-tile along the contraction index
// when the A stages live in tensor memory. The gather's four lanes of a tile
// row hold 16 consecutive channels each (lane q: channels 16q .. 16q+15, as 8
// pairs) and write them with the 16x256b tensor-memory store, whose fragment
// gives thread q of a row the 32-bit columns 8a + 2q and 8a + 2q + 1 (a = 0..3).
// So channel 16q + 4a + 2b + e sits at K position 16a + 4q + 2b + e (the
// two-bit fields q and a swapped), and the packed weight follows the same
// order, which leaves the contraction unchanged. The map is its own inverse.
// Shared-memory A stages keep the natural order.
__host__ __device__ __forceinline__ int32_t kperm16(int32_t ci) {
    return (ci & ~0x3c) | ((ci & 0x30) >> 2) | ((ci & 0x0c) << 2);
}

__host__ __device__ __forceinline__ KTile decode_ktile(int32_t kt, int32_t K, int32_t nch) {
    KTile t;
    const int32_t per_unit = K * nch;
    t.ul = kt / per_unit;
    const int32_t r = kt - t.ul * per_unit;
    t.b = r / (kTapBlock * nch);
    const int32_t rr = r - t.b * kTapBlock * nch;
    const int32_t rest = K - t.b * kTapBlock;
    t.ntb = rest < kTapBlock ? rest : kTapBlock;
    t.ch = rr / t.ntb;
    t.kb = rr - t.ch * t.ntb;
    t.tap = t.b * kTapBlock + t.kb;
    return t;
}

}  // namespace mdcn
