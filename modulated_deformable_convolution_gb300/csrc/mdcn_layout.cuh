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
