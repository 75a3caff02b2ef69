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

// The high and low words of the 64-bit product m x, as one wide multiply.
__device__ __forceinline__ void mul_hi_lo(uint32_t m, uint32_t x, uint32_t& hi, uint32_t& lo) {
  const unsigned long long pr = (unsigned long long)m * x;
  hi = uint32_t(pr >> 32);
  lo = uint32_t(pr);
}

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    uint32_t hi0, lo0;
    mul_hi_lo(0xD2511F53u, c.x, hi0, lo0);
    uint32_t hi1, lo1;
    mul_hi_lo(0xCD9E8D57u, c.z, hi1, lo1);
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
    uint32_t ahi0, alo0;
    mul_hi_lo(0xD2511F53u, a.x, ahi0, alo0);
    uint32_t bhi0, blo0;
    mul_hi_lo(0xD2511F53u, b.x, bhi0, blo0);
    uint32_t ahi1, alo1;
    mul_hi_lo(0xCD9E8D57u, a.z, ahi1, alo1);
    uint32_t bhi1, blo1;
    mul_hi_lo(0xCD9E8D57u, b.z, bhi1, blo1);
    a = make_uint4(ahi1 ^ a.y ^ k0, alo1, ahi0 ^ a.w ^ k1, alo0);
    b = make_uint4(bhi1 ^ b.y ^ k0, blo1, bhi0 ^ b.w ^ k1, blo0);
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
}

// The dropout counter (j div 16, i, bh, offset) changes only in word 0 between
// the calls of one query row, so part of the first two rounds is the same for
// every call of the row: round 1 multiplies word 2 (bh), round 2 multiplies
// the word that round 1 made of (bh, i, key).  PhiloxRow holds those values
// (and the key) once per row; philox4x32_10_row(x, R) then returns exactly
// philox4x32_10((x, i, bh, offset), k0, k1) with two of the first four
// products and four key additions per round fewer.
struct PhiloxRow {
  uint32_t w0;    // word 0 after round 1: hi(M1 * bh) ^ i ^ k0
  uint32_t w1k;   // word 1 after round 1, xored with round 2's key 0: (M1 * bh) ^ (k0 + W0)
  uint32_t w3k;   // offset ^ k1: xored into word 2 by round 1
  uint32_t h2k;   // hi(M0 * w0) ^ (k1 + W1): round 2's word 2 before the low product of word 0
  uint32_t l2;    // lo(M0 * w0): round 2's word 3
  uint32_t k0, k1;
};

__device__ __forceinline__ PhiloxRow philox_row(uint32_t i, uint32_t bh, uint32_t offset, uint32_t k0,
                                                uint32_t k1) {
  PhiloxRow R;
  R.w0 = __umulhi(0xCD9E8D57u, bh) ^ i ^ k0;
  R.w1k = (0xCD9E8D57u * bh) ^ (k0 + 0x9E3779B9u);
  R.w3k = offset ^ k1;
  R.h2k = __umulhi(0xD2511F53u, R.w0) ^ (k1 + 0xBB67AE85u);
  R.l2 = 0xD2511F53u * R.w0;
  R.k0 = k0;
  R.k1 = k1;
  return R;
}

// The round keys of rounds 3..10 (k0 + r W0, k1 + r W1 for r = 2..9): fixed
// by the seed, so a launch computes them once (host side) and the kernels
// read them from their parameters instead of bumping the key in every call.
struct PhiloxKeys {
  uint32_t k0[8], k1[8];
};
__host__ __device__ inline PhiloxKeys philox_round_keys(uint32_t k0, uint32_t k1) {
  PhiloxKeys K;
  for (int r = 2; r < 10; ++r) {
    K.k0[r - 2] = k0 + uint32_t(r) * 0x9E3779B9u;
    K.k1[r - 2] = k1 + uint32_t(r) * 0xBB67AE85u;
  }
  return K;
}

// rounds 3..10 (r = 2..9) of philox4x32_10 on the state after round 2
__device__ __forceinline__ uint4 philox_rounds_from_3(uint4 c, const PhiloxKeys& K) {
#pragma unroll
  for (int r = 2; r < 10; ++r) {
    uint32_t hi0, lo0;
    mul_hi_lo(0xD2511F53u, c.x, hi0, lo0);
    uint32_t hi1, lo1;
    mul_hi_lo(0xCD9E8D57u, c.z, hi1, lo1);
    c = make_uint4(hi1 ^ c.y ^ K.k0[r - 2], lo1, hi0 ^ c.w ^ K.k1[r - 2], lo0);
  }
  return c;
}

// the state after rounds 1 and 2 for counter word 0 = x
__device__ __forceinline__ uint4 philox_rounds_1_2(uint32_t x, const PhiloxRow& R) {
  const uint32_t z = __umulhi(0xD2511F53u, x) ^ R.w3k;   // round 1: word 2
  const uint32_t lo = 0xD2511F53u * x;                     // round 1: word 3
  return make_uint4(__umulhi(0xCD9E8D57u, z) ^ R.w1k, 0xCD9E8D57u * z, R.h2k ^ lo, R.l2);
}

__device__ __forceinline__ uint4 philox4x32_10_row(uint32_t x, const PhiloxRow& R, const PhiloxKeys& K) {
  return philox_rounds_from_3(philox_rounds_1_2(x, R), K);
}

// two counters of one row (word 0 = xa, xb), their rounds interleaved
__device__ __forceinline__ void philox4x32_10_row_x2(uint32_t xa, uint32_t xb, const PhiloxRow& R,
                                                     const PhiloxKeys& K, uint4& a, uint4& b) {
  a = philox_rounds_1_2(xa, R);
  b = philox_rounds_1_2(xb, R);
#pragma unroll
  for (int r = 2; r < 10; ++r) {
    const uint32_t kr0 = K.k0[r - 2], kr1 = K.k1[r - 2];
    uint32_t ahi0, alo0;
    mul_hi_lo(0xD2511F53u, a.x, ahi0, alo0);
    uint32_t bhi0, blo0;
    mul_hi_lo(0xD2511F53u, b.x, bhi0, blo0);
    uint32_t ahi1, alo1;
    mul_hi_lo(0xCD9E8D57u, a.z, ahi1, alo1);
    uint32_t bhi1, blo1;
    mul_hi_lo(0xCD9E8D57u, b.z, bhi1, blo1);
    a = make_uint4(ahi1 ^ a.y ^ kr0, alo1, ahi0 ^ a.w ^ kr1, alo0);
    b = make_uint4(bhi1 ^ b.y ^ kr0, blo1, bhi0 ^ b.w ^ kr1, blo0);
  }
}

// The column form, for code that walks one key group over many query rows:
// counter words 0 (j div 16) and 2 (head) and the key are fixed, only word 1
// (the query row) changes, and round 1 leaves word 1 in word 0 only (xored
// in).  PhiloxCol holds round 1's result without word 1 and round 2's keys;
// philox4x32_10_col(i, C, K) returns exactly philox4x32_10((x, i, bh, offset),
// k0, k1).
struct PhiloxCol {
  uint32_t a, b, c, d;   // state after round 1 for row 0 (the row is xored into a)
  uint32_t k0, k1;       // round 2's keys
};

__device__ __forceinline__ PhiloxCol philox_col(uint32_t x, uint32_t bh, uint32_t offset, uint32_t k0,
                                                uint32_t k1) {
  PhiloxCol C;
  C.a = __umulhi(0xCD9E8D57u, bh) ^ k0;
  C.b = 0xCD9E8D57u * bh;
  C.c = __umulhi(0xD2511F53u, x) ^ offset ^ k1;
  C.d = 0xD2511F53u * x;
  C.k0 = k0 + 0x9E3779B9u;
  C.k1 = k1 + 0xBB67AE85u;
  return C;
}

__device__ __forceinline__ uint4 philox4x32_10_col(uint32_t i, const PhiloxCol& C, const PhiloxKeys& K) {
  uint4 c = make_uint4(C.a ^ i, C.b, C.c, C.d);
  // round 2
  uint32_t hi0, lo0;
    mul_hi_lo(0xD2511F53u, c.x, hi0, lo0);
  uint32_t hi1, lo1;
    mul_hi_lo(0xCD9E8D57u, c.z, hi1, lo1);
  c = make_uint4(hi1 ^ c.y ^ C.k0, lo1, hi0 ^ c.w ^ C.k1, lo0);
  return philox_rounds_from_3(c, K);
}

// The keep decision of four keys at once: byte b of `word` is kept iff
// b >= t.  With b = 128 h + l and t = 128 ht + lt (h, ht the top bits),
// z = (word | 0x80808080) - lt * 0x01010101 has in each byte 128 + l - lt,
// between 1 and 255 (no borrow between bytes), whose top bit is l >= lt; so
// b >= t is the top bit of (b | z) when ht = 0 and of (b & z) when ht = 1.
// Returns the word whose byte top bits are the keep bits; tl4 = lt *
// 0x01010101, hsel = all ones when t >= 128, else 0.
__host__ __device__ inline uint32_t dropout_keep_msb(uint32_t word, uint32_t tl4, uint32_t hsel) {
  const uint32_t z = (word | 0x80808080u) - tl4;
  return ((word & z) & hsel) | ((word | z) & ~hsel);
}

// Mask of a packed bf16 pair from dropout_keep_msb's word: the pair of keys
// 2m, 2m+1 (m = half) of the word gets 0xffff over each kept element's 16
// bits and 0 over a dropped one (each selected byte's top bit replicated over
// two result bytes).
__device__ __forceinline__ uint32_t dropout_pair_mask(uint32_t keep_msb, int half) {
  uint32_t m;
  asm("prmt.b32 %0, %1, 0, %2;" : "=r"(m) : "r"(keep_msb), "r"(half ? 0xBBAAu : 0x9988u));
  return m;
}

// The same keep bits as 32-bit masks, one key at a time: all ones iff the key
// of byte b (0-3) of a dropout_keep_msb word is kept (the byte's top bit
// replicated into all four bytes).
__device__ __forceinline__ uint32_t dropout_byte_mask(uint32_t keep_msb, int b) {
  uint32_t m;
  asm("prmt.b32 %0, %1, 0, %2;" : "=r"(m) : "r"(keep_msb), "r"(0x8888u + 0x1111u * uint32_t(b)));
  return m;
}

}  // namespace fa
