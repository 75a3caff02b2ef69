// philox.cuh - counter-based random bits for dropout on the attention weights.
//
// Philox-4x32-10 as defined by Salmon, Moraes, Dror and Shaw, "Parallel Random
// Numbers: As Easy as 1, 2, 3" (SC 2011), section 3.2: ten rounds over a
// counter of four 32-bit words under a two-word key; each round multiplies
// words 0 and 2 by the constants M0 = 0xD2511F53 and M1 = 0xCD9E8D57, keeps
// both halves of the 64-bit products, and permutes and xors them with the
// other two words and the round key; the key is bumped by the Weyl constants
// 0x9E3779B9 and 0xBB67AE85 between rounds.
//
// The dropout contract (the library's own: the pages name dropout as the step
// between softmax and the second matrix product but give no random numbers):
// key position j of query row i in head bh (= b * H + h) takes byte j mod 4 of
// word (j div 4) mod 4 of philox(counter = (j div 16, i, bh, offset),
// key = (seed mod 2^32, seed div 2^32)), and is kept iff that byte >= t.
#pragma once

#include <cstdint>

namespace fa {

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t hi0 = __umulhi(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c;
}

// Two counters under one key, their rounds interleaved so that the two
// independent multiply chains overlap; the same bits as two philox4x32_10
// calls.
__device__ __forceinline__ void philox4x32_10_x2(uint4& a, uint4& b, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t ahi0 = __umulhi(0xD2511F53u, a.x), alo0 = 0xD2511F53u * a.x;
    const uint32_t bhi0 = __umulhi(0xD2511F53u, b.x), blo0 = 0xD2511F53u * b.x;
    const uint32_t ahi1 = __umulhi(0xCD9E8D57u, a.z), alo1 = 0xCD9E8D57u * a.z;
    const uint32_t bhi1 = __umulhi(0xCD9E8D57u, b.z), blo1 = 0xCD9E8D57u * b.z;
    a = make_uint4(ahi1 ^ a.y ^ k0, alo1, ahi0 ^ a.w ^ k1, alo0);
    b = make_uint4(bhi1 ^ b.y ^ k0, blo1, bhi0 ^ b.w ^ k1, blo0);
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
}

// Masks for packed bf16 pairs: `keep4` = __vcmpgeu4(word, t * 0x01010101)
// holds 0xff in each kept key's byte and 0 in each dropped one; the pair of
// keys 2m, 2m+1 (m = half) of that word gets 0xffff over each kept element's
// 16 bits and 0 over a dropped one.
__device__ __forceinline__ uint32_t dropout_pair_mask(uint32_t keep4, int half) {
  return __byte_perm(keep4, 0u, half ? 0x3322u : 0x1100u);
}

}  // namespace fa
