// fa_bwd_kernel.cuh — gradients of exact attention for sm_103a (tcgen05 + TMEM + TMA).
//
// What it computes: dQ, dK, dV of sum(dO * O) for O = softmax(scale Q K^T) V
// (causal or not).  Like the forward pass, no N x N matrix is stored: the
// score and probability tiles are rebuilt from Q, K and the per-row LSE the
// forward pass emitted ("FlashAttention: The Matrix You Never Have to Write
// Down", section "The forward pass is only half of it"; "Why FlashAttention
// Can Avoid a Square Attention Array Without Making Attention Linear",
// section "Backward can recreate tiles instead of retaining the square").
// With P = exp(scale S - LSE) and D = rowsum(dO * O), the chain rule through
// the softmax gives, per (query tile i, key tile j):
//   dV_j += P^T dO_i,   dP = dO_i V_j^T,   dS = P * (dP - D),
//   dK_j += scale dS^T Q_i,   dQ_i += scale dS K_j.
//
// Three kernels, launched in this order on one stream:
//   fa_bwd_delta_kernel  D = rowsum(dO * O), memory-bound, one pass over O, dO.
//   fa_bwd_dkdv_kernel   one CTA per (batch*head, key tile j): K_j, V_j stay in
//                        shared memory while (Q_i, dO_i) stream past; rebuilds
//                        S^T = K_j Q_i^T and dP^T = V_j dO_i^T on the tensor
//                        core, forms P^T and dS^T in registers, accumulates
//                        dV_j and dK_j in TMEM.
//   fa_bwd_dq_kernel     one CTA per (batch*head, query tile i): Q_i, dO_i stay
//                        while (K_j, V_j) stream past; rebuilds S and dP, forms
//                        dS, accumulates dQ_i in TMEM.
// Each gradient row is written by exactly one CTA, so there are no atomics
// and the result is deterministic; the price is that S and dP are formed
// twice (seven tile GEMMs per (i, j) instead of five).
//
// CTA layout (both tensor-core kernels): warps 0-7 do the element-wise
// work, warp w on TMEM lanes 32*(w%4) .. +31 (key rows in dkdv, query rows
// in dq) and on column half w/4 of each 128-column tile, so a row's 128
// scores are shared by two threads; warp 8 issues the tcgen05 MMAs from one
// thread; warp 9 issues the TMA loads from one thread.  TMEM: S (or S^T) in
// columns 0-127, dP (dP^T) in 128-255, the fp32 accumulators from 256.  The 16-bit P^T and dS^T (dS)
// overwrite the first 64 columns of S^T and dP^T (S) once those are read.
#pragma once

#include <cuda.h>
#include <cstdint>

#include "ptx_sm103.cuh"

namespace fa {

constexpr int kBwdThreads = 320;
constexpr int kBwdEwThreads = 256;       // element-wise warps 0-7
constexpr int kBwdMmaWarp = 8;
constexpr int kBwdLoadWarp = 9;
constexpr int kBwdTile = 128;            // rows of a query or key tile = TMEM lanes
constexpr uint32_t kBwdTmemCols = 512;

// Sites recorded in the status word when a wait of a backward kernel runs out.
enum BwdWaitSite : uint32_t {
  kSiteBwdEmpty = 20, kSiteBwdRes = 21, kSiteBwdFull = 22, kSiteBwdSFull = 23,
  kSiteBwdPFull = 24, kSiteBwdDone = 25
};

struct BwdParams {
  CUtensorMap tm_q;    // [BH, N, d], boxes of 128 rows x 64 columns, 128-byte swizzle
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  CUtensorMap tm_do;
  const float* lse;    // [BH, N] natural-log LSE of the scaled scores (forward output)
  const float* delta;  // [BH, N] rowsum(dO * O)
  void* dq;            // [BH, N, d]
  void* dk;
  void* dv;
  unsigned int* status;
  unsigned long long watchdog_cycles;
  int BH;
  int N;
  int n_tiles;         // ceil(N / 128)
  float scale;
  float scale_log2;    // scale * log2(e)
};

// Shared memory of the two tensor-core kernels: a resident pair of tiles (K_j,
// V_j or Q_i, dO_i), a ring of streamed pairs, the per-query LSE and D of the
// current query tile (dkdv only, double-buffered), and the barriers.
template <int D>
struct BwdSmem {
  static constexpr int kChunks = D / 64;
  static constexpr int kTile = kBwdTile * D * 2;
  static constexpr int kChunkBytes = kBwdTile * 128;
  static constexpr int kStages = (D == 128) ? 2 : 4;
  static constexpr int kRes = 0;
  static constexpr int kRing = kRes + 2 * kTile;
  static constexpr int kVec = kRing + kStages * 2 * kTile;   // [2 buffers][2 vectors][128] floats
  static constexpr int kBar = kVec + 2 * 2 * kBwdTile * 4;
  static constexpr int bFull = 0, bEmpty = kStages, bRes = 2 * kStages, bSFull = bRes + 1,
                       bPFull = bSFull + 1, bDone = bPFull + 1, kNumBars = bDone + 1;
  static constexpr int kMisc = kBar + 8 * kNumBars;   // tmem base, abort flag
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;
  static_assert(kAlloc <= 232448, "shared memory budget");
};

// ---------------------------------------------------------------- D = rowsum(dO * O)
// Each row is read as 16-byte pieces (8 values), D/8 consecutive threads per
// row, reduced with shuffles.  The loop runs warp-uniformly so every lane
// takes part in every shuffle.
template <int D, bool kBf16>
__global__ void __launch_bounds__(256) fa_bwd_delta_kernel(const uint4* __restrict__ o,
                                                           const uint4* __restrict__ dout,
                                                           float* __restrict__ delta,
                                                           long long rows) {
  constexpr int kPer = D / 8;   // threads per row
  const long long total = rows * kPer;
  const int lane = threadIdx.x & 31;
  const long long warp_id = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  for (long long base = warp_id * 32; base < total; base += nwarps * 32) {
    const long long idx = base + lane;
    float acc = 0.f;
    if (idx < total) {
      const uint4 a = o[idx], b = dout[idx];
      const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float a0, a1, b0, b1;
        ptx::unpack2<kBf16>(av[e], a0, a1);
        ptx::unpack2<kBf16>(bv[e], b0, b1);
        acc = fmaf(a0, b0, acc);
        acc = fmaf(a1, b1, acc);
      }
    }
#pragma unroll
    for (int off = kPer / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (idx < total && (lane % kPer) == 0) delta[idx / kPer] = acc;
  }
}

// ---------------------------------------------------------------- shared pieces
// TMEM columns.
constexpr uint32_t kColS = 0, kColDp = 128, kColAcc = 256;

// Issue A (K-major, resident) x B^T (K-major) over the head width into d_tmem:
// M = N = 128, K = D in steps of 16 columns.
template <int D, int Chunk>
__device__ __forceinline__ void issue_kmajor(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo,
                                             uint32_t idesc) {
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = static_cast<uint32_t>((kk >> 2) * Chunk + (kk & 3) * 32) >> 4;
    ptx::mma_ss(d_tmem, ptx::desc_sw128(a_lo + off), ptx::desc_sw128(b_lo + off), idesc, kk > 0);
  }
}

// Issue A (16-bit, in TMEM, 128 rows x 128 along K) x B (MN-major tile of 128
// rows along K, D columns) into d_tmem (N = D).
__device__ __forceinline__ void issue_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo,
                                             uint32_t idesc, uint32_t acc) {
#pragma unroll
  for (int kk = 0; kk < kBwdTile / 16; ++kk)
    ptx::mma_ts(d_tmem, a_tmem + kk * 8, ptx::desc_sw128(b_lo + kk * (2048 >> 4)), idesc,
                kk > 0 ? 1u : acc);
}

// Write columns [c0, c0 + NC) of one row of a TMEM accumulator (fp32), times
// `mul`, to global memory in the storage dtype (rows past N are skipped).
template <int D, int NC, bool kBf16>
__device__ __forceinline__ void store_acc_cols(uint32_t t_acc, int c0, float mul, void* base,
                                               long long row, bool in_range) {
  uint4* out = reinterpret_cast<uint4*>(static_cast<uint8_t*>(base) + row * (D * 2) + c0 * 2);
#pragma unroll 1
  for (int q4 = 0; q4 < NC / 32; ++q4) {
    uint32_t r[32];
    ptx::tmem_ld32(t_acc + c0 + q4 * 32, r);
    ptx::tmem_wait_ld();
    uint32_t pk[16];
#pragma unroll
    for (int e = 0; e < 16; ++e)
      pk[e] = ptx::pack2<kBf16>(__uint_as_float(r[2 * e]) * mul, __uint_as_float(r[2 * e + 1]) * mul);
    if (in_range) {
#pragma unroll
      for (int v = 0; v < 4; ++v)
        out[q4 * 4 + v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
    }
  }
}

// Shared setup of the two tensor-core kernels: TMEM allocation by the MMA
// warp, barrier initialisation by the load thread.
template <int D>
__device__ __forceinline__ uint32_t bwd_setup(uint32_t sbase, uint8_t* sgen, int warp,
                                              uint32_t pfull_count) {
  using L = BwdSmem<D>;
  uint32_t* tmem_base_ptr = reinterpret_cast<uint32_t*>(sgen + L::kMisc);
  if (warp == kBwdMmaWarp) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_base_ptr), kBwdTmemCols);
    ptx::tmem_relinquish();
  }
  if (threadIdx.x == kBwdLoadWarp * 32) {
    *reinterpret_cast<volatile int*>(sgen + L::kMisc + 4) = 0;
    auto bar = [&](int i) -> uint32_t { return sbase + L::kBar + 8u * i; };
    for (int s = 0; s < L::kStages; ++s) {
      ptx::mbar_init(bar(L::bFull + s), 1);
      ptx::mbar_init(bar(L::bEmpty + s), 1);
    }
    ptx::mbar_init(bar(L::bRes), 1);
    ptx::mbar_init(bar(L::bSFull), 1);
    ptx::mbar_init(bar(L::bPFull), pfull_count);
    ptx::mbar_init(bar(L::bDone), 1);
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  return *tmem_base_ptr;
}

// The load thread: the resident pair (res_a, res_b at tile `res_tile`), then
// the streamed pairs (str_a, str_b) of tiles first .. first + count - 1.
template <int D>
__device__ __forceinline__ void bwd_producer(uint32_t sbase, const CUtensorMap* res_a,
                                             const CUtensorMap* res_b, int res_tile,
                                             const CUtensorMap* str_a, const CUtensorMap* str_b,
                                             int first, int count, int bh,
                                             const ptx::Watchdog& wd) {
  using L = BwdSmem<D>;
  auto bar = [&](int i) -> uint32_t { return sbase + L::kBar + 8u * i; };
  bool alive = true;
  ptx::mbar_arrive_expect_tx(bar(L::bRes), 2 * L::kTile);
  for (int c = 0; c < L::kChunks; ++c) {
    ptx::tma_load_3d(sbase + L::kRes + c * L::kChunkBytes, res_a, bar(L::bRes), c * 64,
                     res_tile * kBwdTile, bh);
    ptx::tma_load_3d(sbase + L::kRes + L::kTile + c * L::kChunkBytes, res_b, bar(L::bRes), c * 64,
                     res_tile * kBwdTile, bh);
  }
  int loads = 0;
  for (int it = 0; it < count; ++it) {
    const int slot = it % L::kStages, use = it / L::kStages;
    if (use > 0)
      alive = ptx::wait_bounded(bar(L::bEmpty + slot), (use - 1) & 1, wd, kSiteBwdEmpty) && alive;
    if (!alive) break;
    const uint32_t dst = sbase + L::kRing + slot * 2 * L::kTile;
    ptx::mbar_arrive_expect_tx(bar(L::bFull + slot), 2 * L::kTile);
    for (int c = 0; c < L::kChunks; ++c) {
      ptx::tma_load_3d(dst + c * L::kChunkBytes, str_a, bar(L::bFull + slot), c * 64,
                       (first + it) * kBwdTile, bh);
      ptx::tma_load_3d(dst + L::kTile + c * L::kChunkBytes, str_b, bar(L::bFull + slot), c * 64,
                       (first + it) * kBwdTile, bh);
    }
    ++loads;
  }
  // Drain: every issued copy has landed before the CTA can exit.
  const unsigned long long drain = 200000000ull;
  ptx::wait_drain(bar(L::bRes), 0, drain);
  for (int l = loads > L::kStages ? loads - L::kStages : 0; l < loads; ++l)
    ptx::wait_drain(bar(L::bFull + l % L::kStages), (l / L::kStages) & 1, drain);
}

// ---------------------------------------------------------------- dK, dV
template <int D, bool kBf16, bool kCausal>
__global__ void __launch_bounds__(kBwdThreads, 1)
    fa_bwd_dkdv_kernel(const __grid_constant__ BwdParams p) {
  using L = BwdSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = ptx::smem_u32(smem_raw);
  const uint32_t sbase = (raw_base + 1023u) & ~1023u;
  uint8_t* sgen = smem_raw + (sbase - raw_base);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto bar = [&](int i) -> uint32_t { return sbase + L::kBar + 8u * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sgen + L::kMisc + 4);

  // Key tile kt of head bh; for causal runs the first key tiles (the most
  // query tiles to visit) are dealt first.
  const int kt = blockIdx.x / p.BH;
  const int bh = blockIdx.x - kt * p.BH;
  const int i0 = kCausal ? kt : 0;           // query tiles i >= kt see this key tile
  const int nq = p.n_tiles - i0;

  const uint32_t tmem_base = bwd_setup<D>(sbase, sgen, warp, kBwdEwThreads);
  const ptx::Watchdog wd{p.watchdog_cycles, abort_flag, p.status};

  if (warp == kBwdLoadWarp) {
    if (lane == 0) bwd_producer<D>(sbase, &p.tm_k, &p.tm_v, kt, &p.tm_q, &p.tm_do, i0, nq, bh, wd);
    __syncwarp();
  } else if (warp == kBwdMmaWarp) {
    if (lane == 0) {
      constexpr int fmt = kBf16 ? 1 : 0;
      constexpr uint32_t idesc_s = ptx::idesc_f16(kBwdTile, kBwdTile, fmt, 0);
      constexpr uint32_t idesc_o = ptx::idesc_f16(kBwdTile, D, fmt, 1);
      const uint32_t k_lo = ptx::desc_lo(sbase + L::kRes, 16);
      const uint32_t v_lo = ptx::desc_lo(sbase + L::kRes + L::kTile, 16);
      const uint32_t q_lo0 = ptx::desc_lo(sbase + L::kRing, 16);                  // K-major use
      const uint32_t do_lo0 = ptx::desc_lo(sbase + L::kRing + L::kTile, 16);
      const uint32_t q_mn0 = ptx::desc_lo(sbase + L::kRing, L::kChunkBytes);      // MN-major use
      const uint32_t do_mn0 = ptx::desc_lo(sbase + L::kRing + L::kTile, L::kChunkBytes);
      constexpr uint32_t kSlotLo = (2 * L::kTile) >> 4;
      const uint32_t tS = tmem_base + kColS, tDp = tmem_base + kColDp;
      const uint32_t tDv = tmem_base + kColAcc, tDk = tmem_base + kColAcc + D;
      bool alive = ptx::wait_bounded(bar(L::bRes), 0, wd, kSiteBwdRes);
      for (int it = 0; it < nq; ++it) {
        const uint32_t slot = it % L::kStages;
        alive = ptx::wait_bounded(bar(L::bFull + slot), (it / L::kStages) & 1, wd, kSiteBwdFull) && alive;
        ptx::tc_fence_after();
        if (!alive) break;
        // S^T = K_j Q_i^T and dP^T = V_j dO_i^T (keys on the TMEM lanes)
        issue_kmajor<D, L::kChunkBytes>(tS, k_lo, q_lo0 + slot * kSlotLo, idesc_s);
        issue_kmajor<D, L::kChunkBytes>(tDp, v_lo, do_lo0 + slot * kSlotLo, idesc_s);
        ptx::mma_commit(bar(L::bSFull));
        alive = ptx::wait_bounded(bar(L::bPFull), it & 1, wd, kSiteBwdPFull) && alive;
        ptx::tc_fence_after();
        if (!alive) break;
        // dV_j += P^T dO_i and dK_j += dS^T Q_i (scale applied at the end)
        issue_tmem_a(tDv, tS, do_mn0 + slot * kSlotLo, idesc_o, it > 0 ? 1u : 0u);
        issue_tmem_a(tDk, tDp, q_mn0 + slot * kSlotLo, idesc_o, it > 0 ? 1u : 0u);
        ptx::mma_commit(bar(L::bEmpty + slot));
      }
      ptx::mma_commit(bar(L::bDone));
      ptx::wait_drain(bar(L::bDone), 0, 200000000ull);
    }
    __syncwarp();
  } else {
    // ============================================================ element-wise
    const int quarter = warp & 3, half = warp >> 2;
    const int t = quarter * 32 + lane;                    // key row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem_base + lane_off + kColS, tDp = tmem_base + lane_off + kColDp;
    const long long key = static_cast<long long>(kt) * kBwdTile + t;
    const float c = p.scale_log2;
    float* vec = reinterpret_cast<float*>(sgen + L::kVec);   // [2][2][128]
    const float* lse_h = p.lse + static_cast<long long>(bh) * p.N;
    const float* del_h = p.delta + static_cast<long long>(bh) * p.N;
    for (int it = 0; it < nq; ++it) {
      const int i = i0 + it;
      // LSE (in log2 units) and D of the 128 queries of tile i; a query past
      // N gets LSE = +inf, so its P is 0.
      float* lv = vec + (it & 1) * 256;
      if (half == 0) {
        const int qrow = i * kBwdTile + t;
        lv[t] = qrow < p.N ? lse_h[qrow] * 1.4426950408889634f : INFINITY;
        lv[128 + t] = qrow < p.N ? del_h[qrow] : 0.f;
      }
      ptx::named_bar_sync(1, kBwdEwThreads);
      ptx::wait_bounded(bar(L::bSFull), it & 1, wd, kSiteBwdSFull);
      __syncwarp();
      ptx::tc_fence_after();
      // this thread's 64 query columns of S^T and dP^T, 32 at a time
      const bool diag = kCausal && i == kt;
      uint32_t pk[32], dk[32];
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        uint32_t sr[32], dpr[32];
        ptx::tmem_ld32(tS + half * 64 + ch * 32, sr);
        ptx::tmem_ld32(tDp + half * 64 + ch * 32, dpr);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int qc = half * 64 + ch * 32 + e;         // query column within the tile
          float p0 = ptx::ex2(fmaf(__uint_as_float(sr[e]), c, -lv[qc]));
          float p1 = ptx::ex2(fmaf(__uint_as_float(sr[e + 1]), c, -lv[qc + 1]));
          if (diag) {                                     // key after the query: masked
            if (i * kBwdTile + qc < key) p0 = 0.f;
            if (i * kBwdTile + qc + 1 < key) p1 = 0.f;
          }
          const float d0 = p0 * (__uint_as_float(dpr[e]) - lv[128 + qc]);
          const float d1 = p1 * (__uint_as_float(dpr[e + 1]) - lv[128 + qc + 1]);
          pk[ch * 16 + e / 2] = ptx::pack2<kBf16>(p0, p1);
          dk[ch * 16 + e / 2] = ptx::pack2<kBf16>(d0, d1);
        }
      }
      // P^T and dS^T go to the first 64 columns of S^T and dP^T, which the
      // other half's warps read: every load is done before any store.
      ptx::named_bar_sync(2, kBwdEwThreads);
      ptx::tmem_st16(tS + half * 32, pk);
      ptx::tmem_st16(tS + half * 32 + 16, pk + 16);
      ptx::tmem_st16(tDp + half * 32, dk);
      ptx::tmem_st16(tDp + half * 32 + 16, dk + 16);
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar(L::bPFull));
    }
    // dV_j rows (warps 0-3) and dK_j = scale * (dS^T Q) rows (warps 4-7)
    ptx::wait_bounded(bar(L::bDone), 0, wd, kSiteBwdDone);
    __syncwarp();
    ptx::tc_fence_after();
    const long long row = static_cast<long long>(bh) * p.N + key;
    if (half == 0)
      store_acc_cols<D, D, kBf16>(tmem_base + lane_off + kColAcc, 0, 1.f, p.dv, row, key < p.N);
    else
      store_acc_cols<D, D, kBf16>(tmem_base + lane_off + kColAcc + D, 0, p.scale, p.dk, row,
                                  key < p.N);
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kBwdMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, kBwdTmemCols);
  }
}

// ---------------------------------------------------------------- dQ
template <int D, bool kBf16, bool kCausal>
__global__ void __launch_bounds__(kBwdThreads, 1)
    fa_bwd_dq_kernel(const __grid_constant__ BwdParams p) {
  using L = BwdSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = ptx::smem_u32(smem_raw);
  const uint32_t sbase = (raw_base + 1023u) & ~1023u;
  uint8_t* sgen = smem_raw + (sbase - raw_base);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto bar = [&](int i) -> uint32_t { return sbase + L::kBar + 8u * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sgen + L::kMisc + 4);

  // Query tile qt of head bh; for causal runs the last query tiles (the most
  // key tiles to visit) are dealt first.
  const int r = blockIdx.x / p.BH;
  const int bh = blockIdx.x - r * p.BH;
  const int qt = kCausal ? p.n_tiles - 1 - r : r;
  const int nk = kCausal ? qt + 1 : p.n_tiles;   // key tiles j <= qt are visible

  const uint32_t tmem_base = bwd_setup<D>(sbase, sgen, warp, kBwdEwThreads);
  const ptx::Watchdog wd{p.watchdog_cycles, abort_flag, p.status};

  if (warp == kBwdLoadWarp) {
    if (lane == 0) bwd_producer<D>(sbase, &p.tm_q, &p.tm_do, qt, &p.tm_k, &p.tm_v, 0, nk, bh, wd);
    __syncwarp();
  } else if (warp == kBwdMmaWarp) {
    if (lane == 0) {
      constexpr int fmt = kBf16 ? 1 : 0;
      constexpr uint32_t idesc_s = ptx::idesc_f16(kBwdTile, kBwdTile, fmt, 0);
      constexpr uint32_t idesc_o = ptx::idesc_f16(kBwdTile, D, fmt, 1);
      const uint32_t q_lo = ptx::desc_lo(sbase + L::kRes, 16);
      const uint32_t do_lo = ptx::desc_lo(sbase + L::kRes + L::kTile, 16);
      const uint32_t k_lo0 = ptx::desc_lo(sbase + L::kRing, 16);                 // K-major use
      const uint32_t v_lo0 = ptx::desc_lo(sbase + L::kRing + L::kTile, 16);
      const uint32_t k_mn0 = ptx::desc_lo(sbase + L::kRing, L::kChunkBytes);     // MN-major use
      constexpr uint32_t kSlotLo = (2 * L::kTile) >> 4;
      const uint32_t tS = tmem_base + kColS, tDp = tmem_base + kColDp;
      const uint32_t tDq = tmem_base + kColAcc;
      bool alive = ptx::wait_bounded(bar(L::bRes), 0, wd, kSiteBwdRes);
      for (int it = 0; it < nk; ++it) {
        const uint32_t slot = it % L::kStages;
        alive = ptx::wait_bounded(bar(L::bFull + slot), (it / L::kStages) & 1, wd, kSiteBwdFull) && alive;
        ptx::tc_fence_after();
        if (!alive) break;
        // S = Q_i K_j^T and dP = dO_i V_j^T (queries on the TMEM lanes)
        issue_kmajor<D, L::kChunkBytes>(tS, q_lo, k_lo0 + slot * kSlotLo, idesc_s);
        issue_kmajor<D, L::kChunkBytes>(tDp, do_lo, v_lo0 + slot * kSlotLo, idesc_s);
        ptx::mma_commit(bar(L::bSFull));
        alive = ptx::wait_bounded(bar(L::bPFull), it & 1, wd, kSiteBwdPFull) && alive;
        ptx::tc_fence_after();
        if (!alive) break;
        // dQ_i += dS K_j (scale applied at the end)
        issue_tmem_a(tDq, tS, k_mn0 + slot * kSlotLo, idesc_o, it > 0 ? 1u : 0u);
        ptx::mma_commit(bar(L::bEmpty + slot));
      }
      ptx::mma_commit(bar(L::bDone));
      ptx::wait_drain(bar(L::bDone), 0, 200000000ull);
    }
    __syncwarp();
  } else {
    // ============================================================ element-wise
    const int quarter = warp & 3, half = warp >> 2;
    const int t = quarter * 32 + lane;                    // query row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem_base + lane_off + kColS, tDp = tmem_base + lane_off + kColDp;
    const long long qrow = static_cast<long long>(qt) * kBwdTile + t;
    const bool q_in = qrow < p.N;
    const long long grow = static_cast<long long>(bh) * p.N + qrow;
    const float lse2 = q_in ? p.lse[grow] * 1.4426950408889634f : INFINITY;
    const float dl = q_in ? p.delta[grow] : 0.f;
    const float c = p.scale_log2;
    for (int j = 0; j < nk; ++j) {
      ptx::wait_bounded(bar(L::bSFull), j & 1, wd, kSiteBwdSFull);
      __syncwarp();
      ptx::tc_fence_after();
      // keys past N, and on the diagonal tile keys after this query, are masked
      int lim = p.N - j * kBwdTile;
      if (kCausal && j == qt) lim = min(lim, t + 1);
      uint32_t dk[32];
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        uint32_t sr[32], dpr[32];
        ptx::tmem_ld32(tS + half * 64 + ch * 32, sr);
        ptx::tmem_ld32(tDp + half * 64 + ch * 32, dpr);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int kc = half * 64 + ch * 32 + e;         // key column within the tile
          float p0 = ptx::ex2(fmaf(__uint_as_float(sr[e]), c, -lse2));
          float p1 = ptx::ex2(fmaf(__uint_as_float(sr[e + 1]), c, -lse2));
          if (kc >= lim) p0 = 0.f;
          if (kc + 1 >= lim) p1 = 0.f;
          dk[ch * 16 + e / 2] = ptx::pack2<kBf16>(p0 * (__uint_as_float(dpr[e]) - dl),
                                                  p1 * (__uint_as_float(dpr[e + 1]) - dl));
        }
      }
      // dS goes to the first 64 columns of S, which the other half's warps
      // read: every load is done before any store.
      ptx::named_bar_sync(1, kBwdEwThreads);
      ptx::tmem_st16(tS + half * 32, dk);
      ptx::tmem_st16(tS + half * 32 + 16, dk + 16);
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar(L::bPFull));
    }
    // dQ = scale * (dS K): each half of the warps writes half of the columns
    ptx::wait_bounded(bar(L::bDone), 0, wd, kSiteBwdDone);
    __syncwarp();
    ptx::tc_fence_after();
    store_acc_cols<D, D / 2, kBf16>(tmem_base + lane_off + kColAcc, half * (D / 2), p.scale, p.dq,
                                    grow, q_in);
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kBwdMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, kBwdTmemCols);
  }
}

}  // namespace fa
