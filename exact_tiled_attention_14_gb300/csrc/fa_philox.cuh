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
// column); see drop_words and drop_words16.
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

// Bit 7 of byte c of the result is set when byte c of w is kept (below t,
// 1 <= t <= 255), given c4 = (256 - t) in every byte: byte < t exactly when
// byte + (256 - t) does not carry out of the byte.  The low seven bits are
// added without reaching the next byte, and the carry out of bit 7 is the
// majority of the byte's top bit, the complement's top bit and the carry
// into bit 7.  The other bits of the result are not meaningful.
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
// pk[2b + 1] for block b: each 16-bit half of pk is cleared exactly when
// its key's byte is not below t.
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

// The backward pass walks 64 keys of a query row (dQ pass) or 64 queries of
// a key column (dK/dV pass) per thread and tile, sixteen 4 x 4 blocks.
// drop_words16: the two words lane k (0 .. 3) of a quad draws for those
// blocks: blocks k, k + 4, k + 8, k + 12 of the walk, word m holding blocks
// 8m + k (bits 7 .. 4 of each byte) and 8m + 4 + k (bits 3 .. 0), laid out
// by key (keep_by_key).  Row walk (kCol = false): block i is (key block
// kb0 + i, query block qb0) and the quad's lanes are the block row's four
// queries; column walk (kCol = true): block i is (kb0, qb0 + i) and the
// quad's lanes are the block column's four keys.
template <bool kCol>
__host__ __device__ __forceinline__ uint2 drop_words16(uint32_t kb0, uint32_t qb0, uint32_t k,
                                                       uint32_t bh, uint32_t off, uint32_t k0,
                                                       uint32_t k1, uint32_t t) {
  const uint32_t c4 = (256u - t) * 0x01010101u;
  uint32_t w[2];
#pragma unroll
  for (int m = 0; m < 2; ++m) {
    const uint32_t i0 = 8u * m + k, i1 = i0 + 4u;
    const uint4 ra = philox4x32_10(kCol ? make_uint4(kb0, qb0 + i0, bh, off)
                                        : make_uint4(kb0 + i0, qb0, bh, off), k0, k1);
    const uint4 rb = philox4x32_10(kCol ? make_uint4(kb0, qb0 + i1, bh, off)
                                        : make_uint4(kb0 + i1, qb0, bh, off), k0, k1);
    w[m] = sel_bits(0xF0F0F0F0u, keep_by_key(ra, c4), keep_by_key(rb, c4) >> 4);
  }
  return make_uint2(w[0], w[1]);
}

// The one-pass backward walks 32 queries of a key column per thread and
// tile, eight 4 x 4 blocks.  drop_words8: the word lane k (0 .. 3) of a
// quad, whose four lanes are the block column's four keys, draws for those
// blocks: blocks k (bits 7 .. 4 of each byte) and k + 4 (bits 3 .. 0) of
// the walk, laid out by key.  kb0 is the key block, qb0 the first query
// block; block i is (kb0, qb0 + i), as in drop_words16's column walk.
__host__ __device__ __forceinline__ uint32_t drop_words8(uint32_t kb0, uint32_t qb0, uint32_t k,
                                                         uint32_t bh, uint32_t off, uint32_t k0,
                                                         uint32_t k1, uint32_t t) {
  const uint32_t c4 = (256u - t) * 0x01010101u;
  const uint4 ra = philox4x32_10(make_uint4(kb0, qb0 + k, bh, off), k0, k1);
  const uint4 rb = philox4x32_10(make_uint4(kb0, qb0 + k + 4u, bh, off), k0, k1);
  return sel_bits(0xF0F0F0F0u, keep_by_key(ra, c4), keep_by_key(rb, c4) >> 4);
}

// Row walk: with y the word holding block 8m + 4h + k2 (word m of quad
// lane k2), the mask (all ones or zero) of key c (0 .. 3) of that block for
// query row r (0 .. 3) of the quad.
__host__ __device__ __forceinline__ uint32_t row_key_mask(uint32_t y, uint32_t r, int h, int c) {
  return prmt(y << (r + 4u * static_cast<uint32_t>(h)), 0u, 0x8888u + 0x1111u * c);
}

// Column walk: with y as above and csel = 0x4440 + c for key column c of
// the quad, a word whose byte r has its top bit set when query r of the
// block is kept (byte c of y moved to byte 0, then one multiply sends bit
// 7 - r, or 3 - r for the block in the low nibbles, to bit 8r + 7; the
// partial products fall on distinct bits, so nothing carries).
__host__ __device__ __forceinline__ uint32_t col_query_bits(uint32_t y, uint32_t csel, int h) {
  return prmt(y, 0u, csel) * (h ? 0x80402010u : 0x08040201u);
}

}  // namespace fa
