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
// by 256 / t.  A quad of lanes shares the calls of a block row (or block
// column); see keep_row_quad.
#pragma once

#include <cstdint>

namespace fa {

// High word of a 32 x 32-bit product (the device's multiply-high; the host
// form lets the mask code below be checked on the CPU).
__host__ __device__ __forceinline__ uint32_t mul_hi32(uint32_t a, uint32_t b) {
#ifdef __CUDA_ARCH__
  return __umulhi(a, b);
#else
  return static_cast<uint32_t>((static_cast<uint64_t>(a) * b) >> 32);
#endif
}

__host__ __device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t hi0 = mul_hi32(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
    const uint32_t hi1 = mul_hi32(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
  }
  return c;
}

// Word `sel` (0..3) of a call's output.
__device__ __forceinline__ uint32_t philox_word(const uint4& r, uint32_t sel) {
  return sel == 0 ? r.x : sel == 1 ? r.y : sel == 2 ? r.z : r.w;
}

// Keep bits of the four bytes of w (bit b for byte b), 1 <= t <= 255, given
// c4 = (256 - t) in every byte (t = 256 keeps everything and never reaches
// the kernels that draw a mask): byte < t exactly when byte + (256 - t) does not carry out of
// the byte.  The low seven bits are added without reaching the next byte;
// a byte's carry out is then the majority of its top bit, the complement's
// top bit and the carry into bit 7, and one multiply gathers the four top
// bits (7, 15, 23, 31 -> 28 .. 31; the other partial products stay below
// bit 28 and never overlap, so nothing carries into them).
__host__ __device__ __forceinline__ uint32_t keep_bits4_swar(uint32_t w, uint32_t c4) {
  const uint32_t lo = (w & 0x7F7F7F7Fu) + (c4 & 0x7F7F7F7Fu);
  const uint32_t carry = (w & c4) | ((w ^ c4) & lo);
  const uint32_t keep = ~carry & 0x80808080u;
  return (keep * 0x00204081u) >> 28;
}

// Keep bits of a whole 4 x 4 block: bit 4 w + c for row w, column c.
__device__ __forceinline__ uint32_t keep16(const uint4& r, uint32_t c4) {
  return keep_bits4_swar(r.x, c4) | (keep_bits4_swar(r.y, c4) << 4) |
         (keep_bits4_swar(r.z, c4) << 8) | (keep_bits4_swar(r.w, c4) << 12);
}

// The same masks with the generator work shared by a quad of lanes (lanes
// 4m .. 4m+3 hold four consecutive rows, or columns, of one block row, or
// block column): lane k of the quad draws the blocks b = k, k + 4, ...,
// two blocks' 16 bits per register, and the quad exchanges the registers
// with broadcast shuffles; every lane then keeps its own row's (column's)
// bits.  NB blocks (NB / 4 calls per lane).  All 32 lanes must call it.
//
// Row walk: bit 4 b + c of `out` (NB = 16 fills one word, 32 two) is key
// key0 + 4 b + c of query row qrow.
template <int NB>
__device__ __forceinline__ void keep_row_quad(uint32_t qrow, uint32_t key0, uint32_t bh,
                                              uint32_t off, uint32_t k0, uint32_t k1, uint32_t t,
                                              uint64_t (&out)[NB / 16]) {
  const uint32_t lane = threadIdx.x & 31u, k = lane & 3u, r = qrow & 3u;
  const uint32_t c4 = (256u - t) * 0x01010101u;
  uint32_t v[NB / 8];
#pragma unroll
  for (int a = 0; a < NB / 4; ++a) {
    const uint4 w = philox4x32_10(make_uint4((key0 >> 2) + 4u * a + k, qrow >> 2, bh, off), k0, k1);
    const uint32_t bits = keep16(w, c4);
    if (a & 1) v[a >> 1] |= bits << 16; else v[a >> 1] = bits;
  }
#pragma unroll
  for (int i = 0; i < NB / 16; ++i) out[i] = 0;
#pragma unroll
  for (int k2 = 0; k2 < 4; ++k2) {
#pragma unroll
    for (int m = 0; m < NB / 8; ++m) {
      const uint32_t y = __shfl_sync(0xffffffffu, v[m], (lane & ~3u) | k2);
      const int b0 = 4 * (2 * m) + k2, b1 = b0 + 4;   // blocks of the two halves
      out[b0 / 16] |= static_cast<uint64_t>((y >> (4 * r)) & 0xFu) << (4 * (b0 % 16));
      out[b1 / 16] |= static_cast<uint64_t>((y >> (16 + 4 * r)) & 0xFu) << (4 * (b1 % 16));
    }
  }
}

// prmt.b32 in its default mode: each selector nibble picks a byte of
// {b, a} (low three bits) and, with its top bit set, replicates that byte's
// sign bit over all eight bits instead of copying it.  The host form spells
// that rule out for the CPU check of the mask code.
__host__ __device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
#ifdef __CUDA_ARCH__
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
#else
  const uint64_t bytes = (static_cast<uint64_t>(b) << 32) | a;
  uint32_t d = 0;
  for (int i = 0; i < 4; ++i) {
    const uint32_t n = (sel >> (4 * i)) & 0xFu;
    uint32_t byte = static_cast<uint32_t>(bytes >> (8 * (n & 7u))) & 0xFFu;
    if (n & 8u) byte = (byte & 0x80u) ? 0xFFu : 0u;
    d |= byte << (8 * i);
  }
  return d;
#endif
}

// Bits of a where m is set, bits of b elsewhere.
__host__ __device__ __forceinline__ uint32_t sel_bits(uint32_t m, uint32_t a, uint32_t b) {
  return (a & m) | (b & ~m);
}

// Bit 7 of byte c of the result is set when byte c of w is kept (below t),
// given c4 = (256 - t) in every byte: the no-carry-out test of
// keep_bits4_swar, left unmasked (the other bits are not meaningful).
__host__ __device__ __forceinline__ uint32_t keep_top(uint32_t w, uint32_t c4) {
  const uint32_t lo = (w & 0x7F7F7F7Fu) + (c4 & 0x7F7F7F7Fu);
  return ~((w & c4) | ((w ^ c4) & lo));
}

// Keep bits of a 4 x 4 block laid out by key: bit 7 - r of byte c is row r
// against key c (bits 3 .. 0 of each byte are not meaningful).  Each row's
// top bits are moved down by r and merged under a byte mask.
__host__ __device__ __forceinline__ uint32_t keep_by_key(const uint4& r, uint32_t c4) {
  const uint32_t t01 = sel_bits(0x80808080u, keep_top(r.x, c4), keep_top(r.y, c4) >> 1);
  const uint32_t t23 = sel_bits(0x80808080u, keep_top(r.z, c4), keep_top(r.w, c4) >> 1);
  return sel_bits(0xC0C0C0C0u, t01, t23 >> 2);
}

// The forward pass at d = 128 draws its masks in a warpgroup of their own
// and hands them to the softmax through shared memory, 2 KB per 128 x 128
// tile; at d = 64 each softmax quad draws its own (drop_row128):
//
// drop_words: the four words lane k of a quad (k = 0 .. 3) draws for the
// four query rows qrow0 .. qrow0 + 3 (qrow0 a multiple of 4) against keys
// key0 .. key0 + 127: blocks k, k + 4, ..., k + 28 of the row (8 Philox
// calls), word m holding blocks 8m + k (bits 7 .. 4 of each byte) and
// 8m + 4 + k (bits 3 .. 0) laid out by key (keep_by_key).  The calls run
// two at a time in a loop (one copy of the generator's code, two
// independent chains in flight), the words passed down a four-register
// queue.
__host__ __device__ __forceinline__ uint4 drop_words(uint32_t qrow0, uint32_t key0, uint32_t k, uint32_t bh,
                                            uint32_t off, uint32_t k0, uint32_t k1, uint32_t t) {
  const uint32_t c4 = (256u - t) * 0x01010101u;
  uint32_t v0 = 0, v1 = 0, v2 = 0, v3 = 0;
#pragma unroll 1
  for (int a = 0; a < 8; a += 2) {
    const uint4 wa = philox4x32_10(make_uint4((key0 >> 2) + 4u * a + k, qrow0 >> 2, bh, off), k0, k1);
    const uint4 wb =
        philox4x32_10(make_uint4((key0 >> 2) + 4u * (a + 1) + k, qrow0 >> 2, bh, off), k0, k1);
    const uint32_t word = sel_bits(0xF0F0F0F0u, keep_by_key(wa, c4), keep_by_key(wb, c4) >> 4);
    v3 = v2; v2 = v1; v1 = v0; v0 = word;
  }
  return make_uint4(v3, v2, v1, v0);
}

// drop_apply: clears, in the 16-bit weights pk of a query row (pk[i] holds
// keys 2i and 2i + 1 of the tile), every weight the mask drops, given the
// words y[k] = drop_words(.., k, ..) of the row's quad and the row's place
// r (0 .. 3) in it.  One shift brings row r's bit of each key to the top of
// the key's byte, and two byte permutes with sign replication turn those
// top bits into the 0x0000FFFF / 0xFFFF0000 halves of pk[2b] and
// pk[2b + 1] for block b.  The result is the same as applying
// keep_row_quad<32>'s bits pair by pair.
__host__ __device__ __forceinline__ void drop_apply(uint32_t (&pk)[64], const uint4 (&y)[4], uint32_t r) {
#pragma unroll
  for (int k2 = 0; k2 < 4; ++k2) {
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const uint32_t word = m == 0 ? y[k2].x : m == 1 ? y[k2].y : m == 2 ? y[k2].z : y[k2].w;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int b = 4 * (2 * m + h) + k2;            // block of keys 4b .. 4b + 3
        const uint32_t spread = word << (r + 4u * h);  // row r's bit of key c at bit 8c + 7
        pk[2 * b] &= prmt(spread, 0u, 0x9988u);
        pk[2 * b + 1] &= prmt(spread, 0u, 0xBBAAu);
      }
    }
  }
}

// drop_row128: drop_words and drop_apply within one quad of softmax lanes:
// lane k draws its words, and each word of each other lane arrives by a
// broadcast shuffle just before the two blocks it holds are applied.  All
// 32 lanes must call it.
__device__ __forceinline__ void drop_row128(uint32_t (&pk)[64], uint32_t qrow, uint32_t key0,
                                            uint32_t bh, uint32_t off, uint32_t k0, uint32_t k1,
                                            uint32_t t) {
  const uint32_t lane = threadIdx.x & 31u, r = qrow & 3u;
  const uint4 mine = drop_words(qrow & ~3u, key0, lane & 3u, bh, off, k0, k1, t);
  const uint32_t v[4] = {mine.x, mine.y, mine.z, mine.w};
#pragma unroll
  for (int k2 = 0; k2 < 4; ++k2) {
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const uint32_t word = __shfl_sync(0xffffffffu, v[m], (lane & ~3u) | static_cast<uint32_t>(k2));
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int b = 4 * (2 * m + h) + k2;            // block of keys 4b .. 4b + 3
        const uint32_t spread = word << (r + 4u * h);  // row r's bit of key c at bit 8c + 7
        pk[2 * b] &= prmt(spread, 0u, 0x9988u);
        pk[2 * b + 1] &= prmt(spread, 0u, 0xBBAAu);
      }
    }
  }
}

// Column walk over 64 queries: bit 4 b + w of the result is query
// q0 + 4 b + w against key column `key`.
__device__ __forceinline__ uint64_t keep_col_quad64(uint32_t key, uint32_t q0, uint32_t bh,
                                                    uint32_t off, uint32_t k0, uint32_t k1,
                                                    uint32_t t) {
  const uint32_t lane = threadIdx.x & 31u, k = lane & 3u, c = key & 3u;
  const uint32_t c4 = (256u - t) * 0x01010101u;
  uint32_t v[2];
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const uint4 w = philox4x32_10(make_uint4(key >> 2, (q0 >> 2) + 4u * a + k, bh, off), k0, k1);
    const uint32_t bits = keep16(w, c4);
    if (a & 1) v[a >> 1] |= bits << 16; else v[a >> 1] = bits;
  }
  uint64_t out = 0;
  // column c of a block's 16 bits (bits c, 4 + c, 8 + c, 12 + c) as a nibble
  auto col = [&](uint32_t h) -> uint32_t {
    const uint32_t x = (h >> c) & 0x1111u;
    return (x | (x >> 3) | (x >> 6) | (x >> 9)) & 0xFu;
  };
#pragma unroll
  for (int k2 = 0; k2 < 4; ++k2) {
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      const uint32_t y = __shfl_sync(0xffffffffu, v[m], (lane & ~3u) | k2);
      const int b0 = 4 * (2 * m) + k2, b1 = b0 + 4;
      out |= static_cast<uint64_t>(col(y & 0xFFFFu)) << (4 * b0);
      out |= static_cast<uint64_t>(col(y >> 16)) << (4 * b1);
    }
  }
  return out;
}

// The 16-bit pair mask of keep bits b0 (low half) and b1 (high half).
__device__ __forceinline__ uint32_t pair_mask(uint64_t bits, int e) {
  return (((bits >> e) & 1ull) ? 0x0000FFFFu : 0u) | (((bits >> (e + 1)) & 1ull) ? 0xFFFF0000u : 0u);
}

}  // namespace fa
