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
// sign bit over all eight bits instead of copying it.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Clears, in the 16-bit weights pk of query row `qrow` against keys key0 ..
// key0 + 127 (pk[i] holds keys 2i and 2i + 1), every weight the mask drops.
// The generator work is shared by the quad exactly as in keep_row_quad
// (lane k draws blocks k, k + 4, ...; broadcast shuffles hand each lane the
// other blocks), and the row's four keep bits of block b become the masks
// of pk[2b] and pk[2b + 1] directly: one multiply moves bit i of the
// nibble to the top bit of byte i (the partial products fall on distinct
// bits, so nothing carries), and two byte permutes with sign replication
// turn those top bits into 0x0000FFFF / 0xFFFF0000 halves.  All 32 lanes
// must call it; the result is the same as applying keep_row_quad<32>'s bits
// pair by pair.
__device__ __forceinline__ void drop_row128(uint32_t (&pk)[64], uint32_t qrow, uint32_t key0,
                                            uint32_t bh, uint32_t off, uint32_t k0, uint32_t k1,
                                            uint32_t t) {
  const uint32_t lane = threadIdx.x & 31u, k = lane & 3u, sh = 4u * (qrow & 3u);
  const uint32_t c4 = (256u - t) * 0x01010101u;
  // The eight generator calls run as a loop (one copy of the generator's
  // code in the instruction stream instead of eight), their 16-bit keep
  // words collected in a small per-thread array.
  uint16_t v16[8];
#pragma unroll 1
  for (int a = 0; a < 8; ++a) {
    const uint4 w = philox4x32_10(make_uint4((key0 >> 2) + 4u * a + k, qrow >> 2, bh, off), k0, k1);
    v16[a] = static_cast<uint16_t>(keep16(w, c4));
  }
  uint32_t v[4];
#pragma unroll
  for (int m = 0; m < 4; ++m) v[m] = v16[2 * m] | (static_cast<uint32_t>(v16[2 * m + 1]) << 16);
#pragma unroll
  for (int k2 = 0; k2 < 4; ++k2) {
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const uint32_t y = __shfl_sync(0xffffffffu, v[m], (lane & ~3u) | k2);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int b = 4 * (2 * m + h) + k2;          // block of keys 4b .. 4b + 3
        const uint32_t spread = ((y >> (sh + 16u * h)) & 0xFu) * 0x10204080u;
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
