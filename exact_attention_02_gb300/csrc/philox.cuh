// Philox-4x32-10 counter-based random bits (J. K. Salmon, M. A. Moraes, R. O. Dror,
// D. E. Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC 2011), written from the
// published definition, and the dropout keep rule built on it.
//
// One round maps the counter (c0, c1, c2, c3) with key (k0, k1) to
//   (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1, lo(M0 c0)),
// M0 = 0xD2511F53, M1 = 0xCD9E8D57; the key is bumped by (0x9E3779B9, 0xBB67AE85)
// between rounds; 10 rounds.
//
// Dropout layout: element (query i, key j) of head h takes the 16-bit half j % 2 of word
// (j % 8) / 2 of Philox(counter = (j / 8, i, h, 0), key = (seed low, seed high)); the key
// is kept iff that value is >= the threshold t = round(p * 65536), and a kept weight is
// scaled by 65536 / (65536 - t).
#pragma once

#include <stdint.h>

namespace fa {
namespace rng {

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
  }
  return c;
}

// Keep bits of the 8 keys 8*blk .. 8*blk + 7 for query i of head h: bit e = key 8*blk + e.
__device__ __forceinline__ uint32_t keep8(uint32_t blk, uint32_t i, uint32_t h, uint32_t k0, uint32_t k1,
                                          uint32_t t) {
  const uint4 w = philox4x32_10(make_uint4(blk, i, h, 0u), k0, k1);
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
  uint32_t bits = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e) bits |= (((ws[e >> 1] >> (16 * (e & 1))) & 0xFFFFu) >= t ? 1u : 0u) << e;
  return bits;
}

}  // namespace rng
}  // namespace fa
