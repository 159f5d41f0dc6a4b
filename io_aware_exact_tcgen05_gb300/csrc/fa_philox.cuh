// fa_philox.cuh -- the counter-based generator behind attention dropout.
//
// Philox4x32-10 as published by Salmon, Moraes, Dror and Shaw ("Parallel
// random numbers: as easy as 1, 2, 3", SC 2011): a 128-bit counter and a
// 64-bit key go through ten rounds; each round multiplies two of the four
// counter words by the paper's two 32-bit multipliers, swaps in the products'
// high halves XORed with the other two words and the key, and the key is
// advanced by the paper's two Weyl increments before every round but the
// first.
//
// Dropout mapping (part of the forward/backward contract, FlashAttention_01
// page, "why the backward can recompute" and "interface and implementation
// constraints"): weight (query row i, key j) of query head bh = b * Hq + h
// is kept iff half (j mod 2) (0: low 16 bits, 1: high 16 bits) of word
// ((j mod 8) / 2) of Philox4x32-10 at counter (j / 8, i, bh, offset) under
// key (seed low, seed high) is >= floor(p * 2^16).  One call decides eight
// keys.
#pragma once

#include <cstdint>

#include "fa_internal.h"

namespace fa {

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
  constexpr uint32_t kMulA = 0xD2511F53u, kMulB = 0xCD9E8D57u;
  constexpr uint32_t kWeyl0 = 0x9E3779B9u, kWeyl1 = 0xBB67AE85u;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += kWeyl0;
      k1 += kWeyl1;
    }
    // one 32 x 32 -> 64-bit product gives both halves
    const uint64_t pa = static_cast<uint64_t>(kMulA) * c.x;
    const uint64_t pb = static_cast<uint64_t>(kMulB) * c.z;
    const uint32_t hi_a = static_cast<uint32_t>(pa >> 32), lo_a = static_cast<uint32_t>(pa);
    const uint32_t hi_b = static_cast<uint32_t>(pb >> 32), lo_b = static_cast<uint32_t>(pb);
    c = make_uint4(hi_b ^ c.y ^ k0, lo_b, hi_a ^ c.w ^ k1, lo_a);
  }
  return c;
}

// Keep bits of keys 8*j8 .. 8*j8+7 at query row i of head bh (bit t = key
// 8*j8+t).  A high half is >= the threshold iff the whole word is >= thr_hi;
// a low half iff the word shifted up by 16 is.
__device__ __forceinline__ uint32_t half_keep2(uint32_t w, uint32_t thr_hi) {
  return ((w << 16) >= thr_hi ? 1u : 0u) | (w >= thr_hi ? 2u : 0u);
}

__device__ __forceinline__ uint32_t dropout_keep8(const DropoutArgs& d, uint32_t j8, uint32_t i,
                                                  uint32_t bh) {
  const uint4 w = philox4x32_10(make_uint4(j8, i, bh, d.offset), d.seed_lo, d.seed_hi);
  return half_keep2(w.x, d.thr_hi) | (half_keep2(w.y, d.thr_hi) << 2) |
         (half_keep2(w.z, d.thr_hi) << 4) | (half_keep2(w.w, d.thr_hi) << 6);
}

}  // namespace fa
