// Philox-4x32-10 counter-based random bits (J. K. Salmon, M. A. Moraes, R. O. Dror,
// D. E. Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC 2011), written from the
// published definition, and the dropout keep rule built on it.
//
// One round maps the counter (c0, c1, c2, c3) with key (k0, k1) to
//   (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1, lo(M0 c0)),
// M0 = 0xD2511F53, M1 = 0xCD9E8D57; the key is bumped by (0x9E3779B9, 0xBB67AE85)
// between rounds; 10 rounds.
//
// Dropout layout: element (query i, key j) of head h takes byte j % 4 of word (j % 16) / 4
// of Philox(counter = (j / 16, i, h, 0), key = (seed low, seed high)), so one generator
// call serves 16 keys; the key is kept iff that byte is >= the threshold
// t = min(255, round(p * 256)), and a kept weight is scaled by 256 / (256 - t).
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

// Bit b (b < 4) is set iff byte b of a is >= byte b of tt (unsigned), for all four bytes at
// once. With H the byte sign bits: (a | H) - (tt & ~H) never borrows across bytes, and its
// sign bit says a' >= t' for the low 7 bits; a >= t then holds iff a's top bit is set and
// t's is not, or the top bits agree and a' >= t'.
__device__ __forceinline__ uint32_t bytes_ge(uint32_t a, uint32_t tt) {
  constexpr uint32_t H = 0x80808080u;
  const uint32_t d = (a | H) - (tt & ~H);
  const uint32_t r = ((a & ~tt) | (~(a ^ tt) & d)) & H;
  return ((r >> 7) & 1u) | ((r >> 14) & 2u) | ((r >> 21) & 4u) | ((r >> 28) & 8u);
}

// Keep bits of the 16 keys 16*blk .. 16*blk + 15 for query i of head h: bit e = key
// 16*blk + e. tt is the threshold t repeated in all four bytes (t * 0x01010101).
__device__ __forceinline__ uint32_t keep16(uint32_t blk, uint32_t i, uint32_t h, uint32_t k0, uint32_t k1,
                                           uint32_t tt) {
  const uint4 w = philox4x32_10(make_uint4(blk, i, h, 0u), k0, k1);
  return bytes_ge(w.x, tt) | (bytes_ge(w.y, tt) << 4) | (bytes_ge(w.z, tt) << 8) | (bytes_ge(w.w, tt) << 12);
}

}  // namespace rng
}  // namespace fa
