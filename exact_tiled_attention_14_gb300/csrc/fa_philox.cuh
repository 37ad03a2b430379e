// fa_philox.cuh — the dropout mask of the attention weights, regenerated on
// the device wherever it is needed (forward P.V, backward dV and dS).
//
// The pages keep the generator's state so that the backward pass rebuilds
// the same dropout mask instead of storing a square one ("Why
// FlashAttention Can Avoid a Square Attention Array Without Making
// Attention Linear", section "Backward can recreate tiles instead of
// retaining the square").  The generator is Philox4x32 with 10 rounds
// (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2,
// 3", SC 2011): counter-based, so any element's bits come from its
// coordinates alone.  One call covers a 4 x 4 block of a head's attention
// matrix: counter (key / 4, query / 4, batch*head, offset), key = the 64-bit
// seed.  Element (i, j) takes byte j % 4 of output word i % 4 and is kept
// when that byte is below t = round((1 - p) * 256); kept weights are scaled
// by 256 / t.  A thread that walks a query row uses one word of each call,
// a thread that walks a key column one byte of each word.
#pragma once

#include <cstdint>

namespace fa {

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t hi0 = __umulhi(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
  }
  return c;
}

// Word `sel` (0..3) of a call's output.
__device__ __forceinline__ uint32_t philox_word(const uint4& r, uint32_t sel) {
  return sel == 0 ? r.x : sel == 1 ? r.y : sel == 2 ? r.z : r.w;
}

// Keep bits of the four bytes of w (bit b for byte b).
__device__ __forceinline__ uint32_t keep_bits4(uint32_t w, uint32_t t) {
  return ((w & 0xFFu) < t ? 1u : 0u) | (((w >> 8) & 0xFFu) < t ? 2u : 0u) |
         (((w >> 16) & 0xFFu) < t ? 4u : 0u) | ((w >> 24) < t ? 8u : 0u);
}

// 64 keep bits of query row `qrow` over keys key0 .. key0 + 63 (key0 a
// multiple of 4): bit e for key key0 + e.
__device__ __forceinline__ uint64_t keep_row64(uint32_t qrow, uint32_t key0, uint32_t bh,
                                               uint32_t off, uint32_t k0, uint32_t k1,
                                               uint32_t t) {
  uint64_t bits = 0;
  const uint32_t sel = qrow & 3u;
#pragma unroll
  for (int g = 0; g < 16; ++g) {
    const uint4 r = philox4x32_10(make_uint4((key0 >> 2) + g, qrow >> 2, bh, off), k0, k1);
    bits |= static_cast<uint64_t>(keep_bits4(philox_word(r, sel), t)) << (4 * g);
  }
  return bits;
}

// 64 keep bits of key column `key` over queries q0 .. q0 + 63 (q0 a multiple
// of 4): bit e for query q0 + e.
__device__ __forceinline__ uint64_t keep_col64(uint32_t key, uint32_t q0, uint32_t bh,
                                               uint32_t off, uint32_t k0, uint32_t k1,
                                               uint32_t t) {
  uint64_t bits = 0;
  const uint32_t sh = (key & 3u) * 8u;
#pragma unroll
  for (int g = 0; g < 16; ++g) {
    const uint4 r = philox4x32_10(make_uint4(key >> 2, (q0 >> 2) + g, bh, off), k0, k1);
    const uint32_t b = (((r.x >> sh) & 0xFFu) < t ? 1u : 0u) | (((r.y >> sh) & 0xFFu) < t ? 2u : 0u) |
                       (((r.z >> sh) & 0xFFu) < t ? 4u : 0u) | (((r.w >> sh) & 0xFFu) < t ? 8u : 0u);
    bits |= static_cast<uint64_t>(b) << (4 * g);
  }
  return bits;
}

// The 16-bit pair mask of keep bits b0 (low half) and b1 (high half).
__device__ __forceinline__ uint32_t pair_mask(uint64_t bits, int e) {
  return (((bits >> e) & 1ull) ? 0x0000FFFFu : 0u) | (((bits >> (e + 1)) & 1ull) ? 0xFFFF0000u : 0u);
}

}  // namespace fa
