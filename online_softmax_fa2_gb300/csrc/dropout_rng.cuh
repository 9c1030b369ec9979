// dropout_rng.cuh -- dropout keep decisions drawn in-kernel from the counter-based generator
// Philox4x32-10 (J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw, "Parallel Random Numbers:
// As Easy as 1, 2, 3", SC'11), written from the paper's definition: ten rounds on a 128-bit
// counter under a 64-bit key; a round multiplies counter words 0 and 2 by M0 and M1 into 64-bit
// products and outputs (hi(M1 x2) ^ x1 ^ k0, lo(M1 x2), hi(M0 x0) ^ x3 ^ k1, lo(M0 x0)); the key
// is bumped by (W0, W1) between rounds.
//
// Keep convention (shared with the backward): key j of query row i of head bh = b * H + h is
// kept iff byte j % 16 of the generator at counter (i, j / 16, bh, offset) under key
// (seed_lo, seed_hi) -- the four output words in order, each little-endian -- is at least p8,
// the drop probability quantised to p8 / 256.  The same (seed, offset) gives the same decisions
// in the forward and in the backward, so no keep mask is stored anywhere.
#pragma once

#include <stdint.h>

namespace attn {
namespace rng {

constexpr uint32_t kM0 = 0xD2511F53u, kM1 = 0xCD9E8D57u;
constexpr uint32_t kW0 = 0x9E3779B9u, kW1 = 0xBB67AE85u;

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r) {
            k0 += kW0;
            k1 += kW1;
        }
        // each 64-bit product in one wide multiply
        const uint64_t p0 = (uint64_t)kM0 * c.x, p1 = (uint64_t)kM1 * c.z;
        c = make_uint4((uint32_t)(p1 >> 32) ^ c.y ^ k0, (uint32_t)p1, (uint32_t)(p0 >> 32) ^ c.w ^ k1,
                       (uint32_t)p0);
    }
    return c;
}

// 4 keep bits (bit t: byte t of w at least p8; p8x4 = p8 in each byte), compared a word at a
// time: per byte, (w | 0x80) - (p8 & 0x7f) cannot borrow from the byte above, and its top bit
// says whether the low seven bits of w reach those of p8; the two top bits decide the rest.
__device__ __forceinline__ uint32_t keep4(uint32_t w, uint32_t p8x4) {
    const uint32_t d = (w | 0x80808080u) - (p8x4 & 0x7f7f7f7fu);
    const uint32_t ge = ((w & ~p8x4) | (~(w ^ p8x4) & d)) & 0x80808080u;  // top bit per kept byte
    return ((ge >> 7) * 0x01020408u) >> 24;                                   // bytes 0..3 -> bits 0..3
}

// The 16 keep bits of keys [16 g, 16 g + 16) of row i of head bh (bit t: key 16 g + t).
__device__ __forceinline__ uint32_t keep16(uint32_t i, uint32_t g, uint32_t bh, uint32_t offset, uint32_t k0,
                                           uint32_t k1, uint32_t p8x4) {
    const uint4 w = philox4x32_10(make_uint4(i, g, bh, offset), k0, k1);
    return keep4(w.x, p8x4) | (keep4(w.y, p8x4) << 4) | (keep4(w.z, p8x4) << 8) | (keep4(w.w, p8x4) << 12);
}

// The keep bits of keys [j0, j0 + 128) of row i of head bh (j0 a multiple of 16): bit t of
// word q is key j0 + 32 q + t.  All eight groups are drawn, visible or not: skipping the
// invisible ones costs a branch per group and measured slower than drawing them.  The eight
// counters (i, g, bh, offset) differ only in word 1, so the first round's two products, the
// second round's product of word 2 and the third round's product of word 0 are the same for
// all eight and are formed once (the rounds themselves are those of philox4x32_10).
__device__ __forceinline__ uint4 keep128(uint32_t i, uint32_t j0, uint32_t bh, uint32_t offset, uint32_t k0,
                                         uint32_t k1, uint32_t p8x4) {
    // round 1: words 1-3 of the result, and word 0 up to the group number
    const uint64_t a0 = (uint64_t)kM0 * i, a1 = (uint64_t)kM1 * bh;
    const uint32_t y1 = (uint32_t)a1, w1 = (uint32_t)a0;
    const uint32_t z1 = (uint32_t)(a0 >> 32) ^ offset ^ k1;
    const uint32_t x1base = (uint32_t)(a1 >> 32) ^ k0;
    // round 2: words 0 and 1 of the result
    const uint32_t k0b = k0 + kW0, k1b = k1 + kW1;
    const uint64_t b1 = (uint64_t)kM1 * z1;
    const uint32_t x2 = (uint32_t)(b1 >> 32) ^ y1 ^ k0b, y2 = (uint32_t)b1;
    // round 3: the product of word 0
    const uint32_t k0c = k0b + kW0, k1c = k1b + kW1;
    const uint64_t c0 = (uint64_t)kM0 * x2;
    uint32_t w[8];
#pragma unroll
    for (int g = 0; g < 8; ++g) {
        const uint32_t x1 = x1base ^ ((j0 >> 4) + g);
        const uint64_t b0 = (uint64_t)kM0 * x1;
        const uint32_t z2 = (uint32_t)(b0 >> 32) ^ w1 ^ k1b, w2 = (uint32_t)b0;
        const uint64_t c1 = (uint64_t)kM1 * z2;
        uint4 c = make_uint4((uint32_t)(c1 >> 32) ^ y2 ^ k0c, (uint32_t)c1, (uint32_t)(c0 >> 32) ^ w2 ^ k1c,
                             (uint32_t)c0);
        uint32_t kk0 = k0c, kk1 = k1c;
#pragma unroll
        for (int r = 3; r < 10; ++r) {  // rounds 4 to 10
            kk0 += kW0;
            kk1 += kW1;
            const uint64_t p0 = (uint64_t)kM0 * c.x, p1 = (uint64_t)kM1 * c.z;
            c = make_uint4((uint32_t)(p1 >> 32) ^ c.y ^ kk0, (uint32_t)p1, (uint32_t)(p0 >> 32) ^ c.w ^ kk1,
                           (uint32_t)p0);
        }
        w[g] = keep4(c.x, p8x4) | (keep4(c.y, p8x4) << 4) | (keep4(c.z, p8x4) << 8) | (keep4(c.w, p8x4) << 12);
    }
    return make_uint4(w[0] | (w[1] << 16), w[2] | (w[3] << 16), w[4] | (w[5] << 16), w[6] | (w[7] << 16));
}

}  // namespace rng
}  // namespace attn
