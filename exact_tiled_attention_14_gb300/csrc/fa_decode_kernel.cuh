// fa_decode_kernel.cuh — split-KV attention for a few queries against a long
// key/value cache (decoding), on the CUDA cores.
//
// With Nq <= 16 queries per head there is no square score matrix to avoid;
// the work is bound by reading K and V from HBM, and a head alone cannot keep
// every SM busy.  So the key axis is split across CTAs, each CTA streams its
// key range tile by tile through shared memory (TMA, 128 keys per tile) and
// keeps, per query, the online softmax state of its range: a running
// maximum m, a running sum l and an unnormalised output.  A second kernel
// combines the parts with the same rescale identity the online softmax
// rests on — scale every part to the largest m, add, divide once ("FlashAttention:
// The Matrix You Never Have to Write Down", section "What it doesn't solve":
// decoding reads one query against a cached history, and Flash-Decoding
// splits the key axis across parallel workers and combines partial results).
//
// Causal masking uses the decoding convention: query i of Nq sits at
// position Nk - Nq + i, after the cached keys, and sees keys j <= that
// position (first page, section "Build it", note on non-square causal
// alignment: incremental decoding offsets the query positions by the cache
// length).
#pragma once

#include <cuda.h>
#include <cstdint>

#include "ptx_sm103.cuh"

namespace fa {

constexpr int kDecThreads = 512;
constexpr int kDecTile = 128;       // keys per tile
constexpr int kDecMaxQ = 16;        // queries per head
enum DecWaitSite : uint32_t { kSiteDecFull = 30 };

struct DecodeParams {
  CUtensorMap tm_k;     // [BH, Nk, d], boxes of 128 rows x 64 columns, 128-byte swizzle
  CUtensorMap tm_v;
  const void* q;        // [BH, Nq, d]
  float* part_o;        // [BH, splits, Nq, d] unnormalised partial outputs
  float2* part_ml;      // [BH, splits, Nq] (m in log2 units, l) of each part
  unsigned int* status;
  unsigned long long watchdog_cycles;
  int BH;
  int Nq;
  int Nk;
  int splits;           // CTAs per head
  int tiles_per_split;  // key tiles of one split (the last may have fewer)
  int causal;
  float scale_log2;     // scale * log2(e)
};

// NQ: query slots compiled in (1, 2, 4, 8 or 16 >= Nq; the extra slots idle).
template <int D, int NQ>
struct DecSmem {
  static constexpr int kChunks = D / 64;
  static constexpr int kTile = kDecTile * D * 2;        // one K or V tile
  static constexpr int kChunkBytes = kDecTile * 128;
  static constexpr int kStages = (D == 128) ? 3 : 6;
  static constexpr int kRing = 0;                         // [stage][K, V]; reused for the final sum
  static constexpr int kQRow = D + 16;                    // padded query row, floats (see q_index)
  static constexpr int kQ = kRing + kStages * 2 * kTile;  // fp32 [NQ][kQRow]
  static constexpr int kS = kQ + NQ * kQRow * 4;          // fp32 scores [NQ][128]
  static constexpr int kBar = (kS + NQ * kDecTile * 4 + 15) / 16 * 16;
  static constexpr int kMisc = kBar + 8 * kStages;        // abort flag
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;
  static_assert(kAlloc <= 232448, "shared memory budget");
  static_assert(kDecThreads * 8 * 4 <= kStages * 2 * kTile, "final sum fits in the ring");
};

// 8 consecutive values of row r, 16-byte piece j (of D/8) of a tile stored as
// 64-column chunks with the 128-byte swizzle.
template <bool kBf16>
__device__ __forceinline__ void load8(const uint8_t* tile, int r, int j, float* out) {
  const int chunk = j >> 3, pc = j & 7;
  const uint4 v = *reinterpret_cast<const uint4*>(tile + chunk * (kDecTile * 128) + r * 128 +
                                                  ((pc ^ (r & 7)) << 4));
  ptx::unpack2<kBf16>(v.x, out[0], out[1]);
  ptx::unpack2<kBf16>(v.y, out[2], out[3]);
  ptx::unpack2<kBf16>(v.z, out[4], out[5]);
  ptx::unpack2<kBf16>(v.w, out[6], out[7]);
}

// Shared-memory index of column `col` of query q: each quarter of the row
// is shifted by 16 bytes, so the four threads that share a key (one quarter
// each) read their query values from different banks.
template <int D>
__device__ __forceinline__ int q_index(int q, int col) {
  return q * (D + 16) + col + (col / (D / 4)) * 4;
}

// One CTA per (split, batch*head): the online softmax over keys
// [split * tiles_per_split * 128, ...) for every query of the head.
//   phase A  scores: four consecutive threads share key r, each dotting a
//            quarter of its columns with every query (two-lane fp32 FMAs),
//            summed with two shuffles.
//   phase B  P V: thread (query, 8-column piece, key group) works for one
//            query, the same for a whole warp; every warp of a query takes
//            the tile's maximum and sum itself (new reference, rescale
//            factor, running sum), then accumulates P V over the keys of its
//            group.  Groups are summed once at the end.
template <int D, int NQ, bool kBf16>
__global__ void __launch_bounds__(kDecThreads, 1)
    fa_decode_partial_kernel(const __grid_constant__ DecodeParams p) {
  using L = DecSmem<D, NQ>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = ptx::smem_u32(smem_raw);
  const uint32_t sbase = (raw_base + 1023u) & ~1023u;
  uint8_t* sgen = smem_raw + (sbase - raw_base);
  auto bar = [&](int i) -> uint32_t { return sbase + L::kBar + 8u * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sgen + L::kMisc);
  const ptx::Watchdog wd{p.watchdog_cycles, abort_flag, p.status};

  // the combine kernel may be scheduled once every CTA has started (it waits
  // for this grid to complete before reading the parts)
  ptx::griddep_launch_dependents();
  const int tid = threadIdx.x, lane = tid & 31;
  const int split = blockIdx.x % p.splits, bh = blockIdx.x / p.splits;
  const int Nq = p.Nq;
  const int n_tiles_all = (p.Nk + kDecTile - 1) / kDecTile;
  const int t0 = split * p.tiles_per_split;
  const int nt = max(0, min(p.tiles_per_split, n_tiles_all - t0));
  float* q_s = reinterpret_cast<float*>(sgen + L::kQ);
  float* s_s = reinterpret_cast<float*>(sgen + L::kS);
  const float c = p.scale_log2;

  if (tid == 0) {
    *abort_flag = 0;
    for (int s = 0; s < L::kStages; ++s) ptx::mbar_init(bar(s), 1);
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
  }
  // queries of this head, as fp32 (slots past Nq are zero)
  {
    const uint32_t* qg = reinterpret_cast<const uint32_t*>(static_cast<const uint16_t*>(p.q) +
                                                           static_cast<size_t>(bh) * Nq * D);
    for (int i = tid; i < NQ * D / 2; i += kDecThreads) {
      float a = 0.f, b = 0.f;
      if (i < Nq * D / 2) ptx::unpack2<kBf16>(qg[i], a, b);
      const int q = (2 * i) / D, col = (2 * i) % D;
      q_s[q_index<D>(q, col)] = a;
      q_s[q_index<D>(q, col + 1)] = b;
    }
  }
  __syncthreads();
  auto issue = [&](int it) {   // TMA loads of tile t0 + it into slot it % kStages
    const int slot = it % L::kStages;
    const uint32_t dst = sbase + L::kRing + slot * 2 * L::kTile;
    ptx::mbar_arrive_expect_tx(bar(slot), 2 * L::kTile);
    for (int ch = 0; ch < L::kChunks; ++ch) {
      ptx::tma_load_3d(dst + ch * L::kChunkBytes, &p.tm_k, bar(slot), ch * 64, (t0 + it) * kDecTile, bh);
      ptx::tma_load_3d(dst + L::kTile + ch * L::kChunkBytes, &p.tm_v, bar(slot), ch * 64,
                       (t0 + it) * kDecTile, bh);
    }
  };
  int issued = 0;   // tiles whose loads thread 0 has issued
  if (tid == 0)
    for (; issued < nt && issued < L::kStages; ++issued) issue(issued);

  // phase-A mapping: key row r, column quarter qd
  const int r = tid >> 2, qd = tid & 3;
  constexpr int kPieces = D / 8;              // 16-byte pieces per row
  constexpr int kMyPieces = kPieces / 4;
  // phase-B mapping: 8-column piece, query, key group
  constexpr int kGroupsAll = kDecThreads / kPieces;
  constexpr int kGroups = kGroupsAll / NQ;    // key groups per query
  static_assert((kGroups * kPieces) % 32 == 0, "a warp serves one query");
  const int piece = tid % kPieces;
  const int qc = (tid / kPieces) / kGroups;
  const int kg = (tid / kPieces) % kGroups;
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  // softmax state of query qc (kept alike by every warp serving it)
  float m2 = -INFINITY, l = 0.f;

  bool alive = true;
  for (int it = 0; it < nt; ++it) {
    const int slot = it % L::kStages;
    alive = ptx::wait_bounded(bar(slot), (it / L::kStages) & 1, wd, kSiteDecFull) && alive;
    const uint8_t* kt = sgen + L::kRing + slot * 2 * L::kTile;
    const uint8_t* vt = kt + L::kTile;
    const int key0 = (t0 + it) * kDecTile;
    // ---- phase A
    {
      uint64_t sacc[NQ];
#pragma unroll
      for (int q = 0; q < NQ; ++q) sacc[q] = ptx::f2_pack(0.f, 0.f);
#pragma unroll
      for (int jj = 0; jj < kMyPieces; ++jj) {
        const int j = qd * kMyPieces + jj;
        float kv[8];
        load8<kBf16>(kt, r, j, kv);
        const uint64_t k01 = ptx::f2_pack(kv[0], kv[1]), k23 = ptx::f2_pack(kv[2], kv[3]);
        const uint64_t k45 = ptx::f2_pack(kv[4], kv[5]), k67 = ptx::f2_pack(kv[6], kv[7]);
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          const uint64_t* qp = reinterpret_cast<const uint64_t*>(q_s + q_index<D>(q, j * 8));
          sacc[q] = ptx::ffma2(k01, qp[0], sacc[q]);
          sacc[q] = ptx::ffma2(k23, qp[1], sacc[q]);
          sacc[q] = ptx::ffma2(k45, qp[2], sacc[q]);
          sacc[q] = ptx::ffma2(k67, qp[3], sacc[q]);
        }
      }
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        float a, b;
        ptx::f2_unpack(sacc[q], a, b);
        float sum = a + b;
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        if (qd == 0) s_s[q * kDecTile + r] = sum;
      }
    }
    __syncthreads();
    // ---- phase B: this warp's query qc: tile maximum and sum, then P V
    if (qc < Nq) {
      const long long pos = static_cast<long long>(p.Nk) - Nq + qc;   // causal: last keys visible
      const float* srow = s_s + qc * kDecTile;
      float sv[4];
      float tmax = -INFINITY;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int kr = lane + 32 * e;
        const long long key = key0 + kr;
        const bool vis = key < p.Nk && (!p.causal || key <= pos);
        sv[e] = vis ? srow[kr] * c : -INFINITY;
        tmax = fmaxf(tmax, sv[e]);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
      const float mnew = fmaxf(m2, tmax);
      // no visible key yet: keep the reference at 0 so -inf - (-inf) never occurs
      const float ref = (mnew == -INFINITY) ? 0.f : mnew;
      const float alpha = (m2 == -INFINITY) ? 0.f : ptx::ex2(m2 - ref);
      float lsum = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) lsum += ptx::ex2(sv[e] - ref);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
      l = l * alpha + lsum;
      m2 = mnew;
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] *= alpha;
#pragma unroll
      for (int kr = kg; kr < kDecTile; kr += kGroups) {
        const long long key = key0 + kr;
        const bool vis = key < p.Nk && (!p.causal || key <= pos);
        const float pv = vis ? ptx::ex2(srow[kr] * c - ref) : 0.f;
        float vv[8];
        load8<kBf16>(vt, kr, piece, vv);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = fmaf(pv, vv[e], acc[e]);
      }
    }
    __syncthreads();   // the slot and the score buffer are free again
    if (tid == 0 && alive && it + L::kStages < nt) issue(issued++);
  }
  // After an aborted wait, loads may still be in flight: let them land
  // before the ring is reused and the CTA exits (bounded).
  if (tid == 0 && !alive)
    for (int it = 0; it < issued; ++it)
      ptx::wait_drain(bar(it % L::kStages), (it / L::kStages) & 1, 200000000ull);
  __syncthreads();

  // ---- sum the key groups (in the now idle ring) and write this part
  float* red = reinterpret_cast<float*>(sgen + L::kRing);
#pragma unroll
  for (int e = 0; e < 8; ++e) red[tid * 8 + e] = acc[e];
  __syncthreads();
  const size_t part = (static_cast<size_t>(bh) * p.splits + split) * Nq;
  if (qc < Nq && kg == 0) {
    float o[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) o[e] = 0.f;
    for (int g = 0; g < kGroups; ++g) {
      const int src = (qc * kGroups + g) * kPieces + piece;
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] += red[src * 8 + e];
    }
    float4* dst = reinterpret_cast<float4*>(p.part_o + (part + qc) * D + piece * 8);
    dst[0] = make_float4(o[0], o[1], o[2], o[3]);
    dst[1] = make_float4(o[4], o[5], o[6], o[7]);
  }
  if (qc < Nq && kg == 0 && piece == 0) p.part_ml[part + qc] = make_float2(m2, l);
}

// One block of D threads per (batch*head, query): combine the parts, thread
// c owning output column c.  Parts with no visible key (l = 0) are skipped;
// a query with none at all gets O = 0 and LSE = -inf.
constexpr int kCombineFast = 32;   // parts merged from registers in one pass

template <int D, bool kBf16>
__global__ void __launch_bounds__(D, 1) fa_decode_combine_kernel(const float* __restrict__ part_o,
                                                              const float2* __restrict__ part_ml,
                                                              void* o, float* lse, int splits,
                                                              int Nq) {
  // launched while the partial kernel finishes: its parts must be complete
  ptx::griddep_wait();
  // Merge of the parts of one (head, query) row by the rescale identity:
  // with m* the largest part maximum (log2 units), O = sum_s 2^(m_s - m*) O_s
  // / sum_s 2^(m_s - m*) l_s.  Thread c owns output column c.  First m*
  // (block reduction), then the scaled sums, eight parts per step so their
  // loads are in flight together (up to 32 parts: all loads at once).  Parts with l = 0 (no visible key) carry
  // no weight and their partial row is never read into the sum.
  __shared__ float red[D / 32];
  const int c = threadIdx.x;
  const int q = blockIdx.x % Nq, bh = blockIdx.x / Nq;
  const size_t base = static_cast<size_t>(bh) * splits * Nq + q;   // part of split s: base + s*Nq
  float m = -INFINITY, acc = 0.f, lt = 0.f;
  if (splits <= kCombineFast) {
    // Up to 32 parts: every thread loads all (m, l) pairs and its column of
    // every part at once (one round trip), then takes m* and the sums from
    // registers.
    float2 ml[kCombineFast];
    float ov[kCombineFast];
#pragma unroll
    for (int i = 0; i < kCombineFast; ++i) {
      const size_t part = base + static_cast<size_t>(i) * Nq;
      ml[i] = i < splits ? part_ml[part] : make_float2(0.f, 0.f);
      ov[i] = i < splits ? part_o[part * D + c] : 0.f;
    }
#pragma unroll
    for (int i = 0; i < kCombineFast; ++i)
      if (ml[i].y > 0.f) m = fmaxf(m, ml[i].x);
#pragma unroll
    for (int i = 0; i < kCombineFast; ++i) {
      const bool live = ml[i].y > 0.f;
      const float f = live ? ptx::ex2(ml[i].x - m) : 0.f;
      acc = live ? fmaf(f, ov[i], acc) : acc;
      lt = live ? fmaf(f, ml[i].y, lt) : lt;
    }
  } else {
    for (int s = c; s < splits; s += D) {
      const float2 ml = part_ml[base + static_cast<size_t>(s) * Nq];
      if (ml.y > 0.f) m = fmaxf(m, ml.x);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if ((c & 31) == 0) red[c >> 5] = m;
    __syncthreads();
    m = red[0];
#pragma unroll
    for (int i = 1; i < D / 32; ++i) m = fmaxf(m, red[i]);
    int s = 0;
    for (; s + 8 <= splits; s += 8) {
      float2 ml[8];
      float ov[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const size_t part = base + static_cast<size_t>(s + i) * Nq;
        ml[i] = part_ml[part];
        ov[i] = part_o[part * D + c];
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const bool live = ml[i].y > 0.f;
        const float f = live ? ptx::ex2(ml[i].x - m) : 0.f;
        acc = live ? fmaf(f, ov[i], acc) : acc;
        lt = live ? fmaf(f, ml[i].y, lt) : lt;
      }
    }
    for (; s < splits; ++s) {
      const size_t part = base + static_cast<size_t>(s) * Nq;
      const float2 ml = part_ml[part];
      if (ml.y > 0.f) {
        const float f = ptx::ex2(ml.x - m);
        acc = fmaf(f, part_o[part * D + c], acc);
        lt = fmaf(f, ml.y, lt);
      }
    }
  }
  const size_t row = static_cast<size_t>(bh) * Nq + q;
  const float out = lt > 0.f ? acc / lt : 0.f;
  const uint32_t pk = ptx::pack2<kBf16>(out, 0.f);   // the value in the low half
  static_cast<uint16_t*>(o)[row * D + c] = static_cast<uint16_t>(pk & 0xffffu);
  if (c == 0) lse[row] = lt > 0.f ? (m + ptx::lg2(lt)) * 0.693147180559945309f : -INFINITY;
}

}  // namespace fa
