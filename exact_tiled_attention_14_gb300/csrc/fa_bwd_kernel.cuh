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
// Two kernels, launched in this order on one stream:
//   fa_bwd_delta_kernel  D = rowsum(dO * O), memory-bound, one pass over O, dO.
//   fa_bwd_kernel        both tensor-core passes in one grid:
//   - dK/dV CTAs         one per (batch*head, key tile j): K_j, V_j stay in
//                        shared memory while Q_i and dO_i stream past; rebuilds
//                        S^T = K_j Q_i^T and dP^T = V_j dO_i^T on the tensor
//                        core, forms P^T and dS^T in registers, accumulates
//                        dV_j and dK_j in TMEM.
//   - dQ CTAs            one per (batch*head, query tile i): Q_i, dO_i stay
//                        while K_j and V_j stream past; rebuilds S and dP, forms
//                        dS, accumulates dQ_i in TMEM.
// Each gradient row is written by exactly one CTA, so there are no atomics
// and the result is deterministic; the price is that S and dP are formed
// twice (seven tile GEMMs per (i, j) instead of five).  fa_bwd_onepass.cuh
// holds the other trade: five tile GEMMs per pair, dQ summed in fp32 by the
// TMA engine in no fixed order.
//
// CTA layout (both tensor-core kernels): warps 0-7 do the element-wise
// work, warp w on TMEM lanes 32*(w%4) .. +31 (key rows in dkdv, query rows
// in dq) and on column half w/4 of each 128-column tile, so a row's 128
// scores are shared by two threads; warp 8 issues the tcgen05 MMAs from one
// thread; warp 9 issues the TMA loads from one thread.  TMEM: S (or S^T) in
// columns 0-127, dP (dP^T) in 128-255, the fp32 accumulators from 256.  The
// streamed operands come through two rings: ring A holds the operand the
// last product of a tile still reads (Q_i in dkdv, K_j in dq), ring B the
// other one (dO_i, V_j), so B's slots free up earlier.
//
// Overlap.  The tensor core is kept busy while the element-wise warps work:
//   dkdv  the element-wise pass runs in two phases.  Phase 1 turns S^T_i into
//         P^T_i and writes it, 16-bit, over the S^T columns the same warp has
//         just read (columns 0-31 and 64-95); phase 2 does the same with
//         dP^T_i and dS^T_i (columns 128-159 and 192-223).  The MMA thread
//         issues dV_j += P^T_i dO_i as soon as phase 1 is done, then S^T_{i+1},
//         then dK_j += dS^T_i Q_i once phase 2 is done, then dP^T_{i+1}: each
//         product that overwrites a 16-bit operand follows the one that reads
//         it in the thread's order.  Phase 1 of tile i+1 runs while the
//         tensor core works on dK_j and dP^T_{i+1}.
//   dq    dS goes to TMEM columns of its own (two buffers after dQ), so
//         S_{j+1} and dP_{j+1} are issued as soon as the element-wise warps
//         have read S_j and dP_j, and dQ_i += dS_j K_j when dS_j is written.
#pragma once

#include <cuda.h>
#include <cstdint>

#include "fa_philox.cuh"
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
  kSiteBwdPFull = 24, kSiteBwdDone = 25, kSiteBwdDpFull = 26, kSiteBwdDsReady = 27,
  kSiteBwdDsFree = 28, kSiteBwdSFree = 29, kSiteBwdDqFull = 32, kSiteBwdDqFree = 33
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
  // Dropout of the forward pass (kDrop variants only): keep threshold t,
  // seed words, offset and 256 / t.  The mask is regenerated from them:
  // dV += (P Z)^T dO and dS = P (Z dP 256/t - D), dV scaled by 256 / t.
  uint32_t drop_t;
  uint32_t drop_k0, drop_k1;
  uint32_t drop_off;
  float drop_scale;
  // Queries against a key set of another length (kKv variants; N and
  // n_tiles then count queries): Nk keys per head in n_ktiles tiles (K, V,
  // dK, dV are [BH, Nk, d]), per-batch key counts seqlens_k[b] (NULL: all
  // Nk; batch b = bh / H), and the causal alignment: align_br = 0 puts
  // query i at position i, 1 at len_b - N + i.  Square calls set
  // Nk = N, n_ktiles = n_tiles.
  int Nk;
  int n_ktiles;
  int H;
  const int* seqlens_k;
  int align_br;
  // Widths (kKv variants; square calls set both to D): width_qk of Q, K,
  // dQ, dK and width_v of V, dO, O, dV, each 64 or 128 with D the larger.
  // Each tensor map has its tensor's own width and only those 64-column
  // chunks are loaded; products over the head width take width_qk / 16 (S)
  // or width_v / 16 (dP) K steps, and dV is accumulated over width_v
  // columns, dK and dQ over width_qk.
  int width_qk;
  int width_v;
  // Packed variable-length batches (kKv variants with varlen = 1): Q, dO, O,
  // dQ token-major [total_q, H, d], K, V, dK, dV [Nk = total_k, H, d], LSE
  // [H, total_q] (as the forward writes it), D [total_q, H]; sequence b owns
  // query tokens cu_q[b] .. cu_q[b+1] - 1 and key tokens cu_k[b] ..
  // cu_k[b+1] - 1 (clamped to the totals).  N and n_tiles are then the
  // longest query count and its tiles, n_ktiles the longest key count's.
  // The tensor maps are (column, head, token).
  const int* cu_q;
  const int* cu_k;
  int varlen;
  int total_q;
  // One-pass kernel: dQ is accumulated, unscaled, in fp32 in blocks of 32
  // queries x 16 columns: block (bh, query tile qt, column block cb, row
  // quarter rq) holds element (column cc, row rr) at
  // dq_acc[((((bh * n_tiles + qt) * (width_qk / 16) + cb) * 4 + rq) * 16 + cc) * 32 + rr]
  // (dq_pad = n_tiles * 128 rows per head).  Zeroed before the launch and
  // converted to dQ by fa_bwd_dq_convert_kernel afterwards.
  float* dq_acc;
  int dq_pad;
  // Work items (key tiles of dK/dV or one-pass CTAs, query tiles of dQ
  // CTAs) are dealt in groups of item_group heads, tile by tile within a
  // group, so the CTAs at work share a few heads' streamed tiles in L2.
  int item_group;
};

// Tile index and head of work item `blk` among BH * n_tiles items dealt in
// groups of p.item_group heads (the last group may be smaller).
__host__ __device__ __forceinline__ void bwd_item(const BwdParams& p, int blk, int n_tiles,
                                                  int& tile, int& bh) {
  const int per_group = p.item_group * n_tiles;
  const int g = blk / per_group, r = blk - g * per_group;
  const int left = p.BH - g * p.item_group;
  const int gh = p.item_group < left ? p.item_group : left;
  tile = r / gh;
  bh = g * p.item_group + (r - tile * gh);
}

// Where head bh's rows sit in a kKv call: its key count len and query
// offset off (query i at position i + off), its query count lenq, and with
// packed batches the first query and key token q0, k0.
struct BwdHead {
  int len, off, lenq, q0, k0;
};
__device__ __forceinline__ BwdHead bwd_kv_head(const BwdParams& p, int bh, bool causal) {
  BwdHead h;
  const int b = bh / p.H;
  h.lenq = p.N;
  h.q0 = 0;
  h.k0 = 0;
  if (p.varlen) {
    h.q0 = min(max(p.cu_q[b], 0), p.total_q);
    h.lenq = min(max(p.cu_q[b + 1], h.q0), p.total_q) - h.q0;
    h.k0 = min(max(p.cu_k[b], 0), p.Nk);
    h.len = min(max(p.cu_k[b + 1], h.k0), p.Nk) - h.k0;
  } else {
    h.len = p.seqlens_k ? p.seqlens_k[b] : p.Nk;
    h.len = min(max(h.len, 0), p.Nk);
  }
  h.off = (causal && p.align_br) ? h.len - h.lenq : 0;
  return h;
}

// Row indices of head bh (h = bh % H): of query row qrow in Q, dO, dQ (rows
// of d values), of key row key in K, V, dK, dV, and of the query's LSE and D.
__device__ __forceinline__ long long bwd_qrow(const BwdParams& p, bool tok, const BwdHead& hd,
                                              int bh, long long qrow) {
  return tok ? (hd.q0 + qrow) * p.H + bh % p.H : static_cast<long long>(bh) * p.N + qrow;
}
__device__ __forceinline__ long long bwd_krow(const BwdParams& p, bool tok, const BwdHead& hd,
                                              int bh, long long key) {
  return tok ? (hd.k0 + key) * p.H + bh % p.H : static_cast<long long>(bh) * p.Nk + key;
}
__device__ __forceinline__ long long bwd_lse_at(const BwdParams& p, bool tok, const BwdHead& hd,
                                                int bh, long long qrow) {
  return tok ? static_cast<long long>(bh % p.H) * p.total_q + hd.q0 + qrow
             : static_cast<long long>(bh) * p.N + qrow;
}

// Shared memory of the tensor-core kernels: the resident pair of tiles
// (K_j, V_j or Q_i, dO_i), ring A and ring B of streamed tiles, in the
// one-pass kernel (kOne, fa_bwd_onepass.cuh) a 128 x 128 tile of dS and
// 32 KB of dQ staging blocks, kVecBytes of per-query vectors (dkdv: -LSE in
// log2 units and D of the current query tile), the ring barriers and ten
// kernel-specific barriers.  The dS tile and the staging blocks take the
// room of ring stages.
template <int D, int kVecBytes, bool kOne = false>
struct BwdSmem {
  static constexpr int kChunks = D / 64;
  static constexpr int kTile = kBwdTile * D * 2;
  static constexpr int kChunkBytes = kBwdTile * 128;
  static constexpr int kStagesA = (D == 128) ? (kOne ? 2 : 3) : (kOne ? 4 : 6);
  static constexpr int kStagesB = (D == 128) ? (kOne ? 1 : 2) : (kOne ? 3 : 4);
  static constexpr int kRes = 0;
  static constexpr int kRingA = kRes + 2 * kTile;
  static constexpr int kRingB = kRingA + kStagesA * kTile;
  static constexpr int kDs = kRingB + kStagesB * kTile;   // 1024-aligned like the tiles
  static constexpr int kStg = kDs + (kOne ? kBwdTile * kBwdTile * 2 : 0);
  static constexpr int kStgBytes = 32 * 1024;
  static constexpr int kVec = kStg + (kOne ? kStgBytes : 0);
  static constexpr int kBar = kVec + kVecBytes;
  static constexpr int bFullA = 0, bEmptyA = kStagesA, bFullB = 2 * kStagesA,
                       bEmptyB = bFullB + kStagesB, bRes = bEmptyB + kStagesB, bX = bRes + 1,
                       kNumBars = bX + 10;
  static constexpr int kMisc = kBar + 8 * kNumBars;   // tmem base, abort flag
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;
  static_assert(kAlloc <= 232448, "shared memory budget");
};

// Kernel-specific barriers (offsets from bX).
struct DkdvBars {
  static constexpr int kSFull = 0, kDpFull = 1, kPReady = 2, kDsReady = 3, kDone = 4;
  static constexpr int kDqFull = 5, kDqFree = 7;   // one-pass kernel: two each (per dQ buffer)
};
struct DqBars {
  static constexpr int kSFull = 0, kSFree = 1, kPFull = 2, kDsFree = 4, kDone = 6;   // PFull, DsFree: 2 each
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
  // the tensor-core grid may be scheduled once every CTA here has started:
  // its prologue and first loads overlap this pass, and its element-wise
  // warps wait for D before reading it
  ptx::griddep_launch_dependents();
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

// ---------------------------------------------------------------- dQ = scale * accumulator
// The one-pass kernel leaves dQ unscaled in fp32 in blocks of 32 queries x
// 16 columns, column by column within a block (BwdParams::dq_acc); the
// blocks of one (batch*head, 128-query tile) are contiguous, 128 x W floats.
// One CTA per (batch*head, query tile) moves them, 64 columns at a time,
// through a shared-memory tile with 16-byte loads and writes the rows in
// the storage dtype, scaled, with 16-byte stores.  Blocks: bh * n_tiles +
// query tile.
template <bool kBf16>
__global__ void __launch_bounds__(256) fa_bwd_dq_convert_kernel(const float* __restrict__ acc,
                                                                uint32_t* __restrict__ dq,
                                                                int N, int W, int pad,
                                                                float scale) {
  __shared__ float tile[kBwdTile][65];
  const int n_tiles = pad / kBwdTile;
  const int bh = blockIdx.x / n_tiles;
  const int qt = blockIdx.x - bh * n_tiles;
  const float4* src = reinterpret_cast<const float4*>(
      acc + (static_cast<long long>(bh) * n_tiles + qt) * kBwdTile * W);
  for (int h = 0; h < W / 64; ++h) {
    // blocks cb = 4h .. 4h + 3 of the tile: 4 x 4 blocks of 512 floats
    const float4* s4 = src + h * (4 * 4 * 512 / 4);
    for (int idx = threadIdx.x; idx < 4 * 4 * 512 / 4; idx += 256) {
      const float4 v = s4[idx];
      const int e = idx * 4;                          // float index within the half
      const int blk = e >> 9, in = e & 511;           // block (cb - 4h) * 4 + rq, offset
      const int cc = in >> 5, rr = in & 31;           // column within the block, row
      const int row = (blk & 3) * 32 + rr, col = (blk >> 2) * 16 + cc;
      tile[row][col] = v.x;
      tile[row + 1][col] = v.y;
      tile[row + 2][col] = v.z;
      tile[row + 3][col] = v.w;
    }
    __syncthreads();
    // 128 rows x 8 pieces of 8 columns
    for (int idx = threadIdx.x; idx < kBwdTile * 8; idx += 256) {
      const int r = idx >> 3, c8 = (idx & 7) * 8;
      const int q = qt * kBwdTile + r;
      if (q < N) {
        uint4 out;
        out.x = ptx::pack2<kBf16>(tile[r][c8] * scale, tile[r][c8 + 1] * scale);
        out.y = ptx::pack2<kBf16>(tile[r][c8 + 2] * scale, tile[r][c8 + 3] * scale);
        out.z = ptx::pack2<kBf16>(tile[r][c8 + 4] * scale, tile[r][c8 + 5] * scale);
        out.w = ptx::pack2<kBf16>(tile[r][c8 + 6] * scale, tile[r][c8 + 7] * scale);
        *reinterpret_cast<uint4*>(dq + (static_cast<long long>(bh) * N + q) * (W / 2) +
                                  (h * 64 + c8) / 2) = out;
      }
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------- shared pieces
// TMEM columns.
constexpr uint32_t kColS = 0, kColDp = 128, kColAcc = 256;

// Issue A (K-major, shared memory) x B^T (K-major) over the head width into
// d_tmem: M = N = 128, K = D in steps of 16 columns.
template <int D, int Chunk>
__device__ __forceinline__ void issue_kmajor(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo,
                                             uint32_t idesc, int steps = D / 16) {
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    if (kk >= steps) break;
    const uint32_t off = static_cast<uint32_t>((kk >> 2) * Chunk + (kk & 3) * 32) >> 4;
    ptx::mma_ss(d_tmem, ptx::desc_sw128(a_lo + off), ptx::desc_sw128(b_lo + off), idesc, kk > 0);
  }
}

// Issue A (16-bit, in TMEM, 128 rows x 128 along K) x B (MN-major tile of 128
// rows along K, D columns) into d_tmem (N = D).  kSplitA: A's 64 packed
// columns sit in two blocks of 32 at a_tmem and a_tmem + 64 (a 16-bit tile
// written over the fp32 columns each half of the warps read).
template <bool kSplitA>
__device__ __forceinline__ void issue_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo,
                                             uint32_t idesc, uint32_t acc) {
#pragma unroll
  for (int kk = 0; kk < kBwdTile / 16; ++kk) {
    const uint32_t acol = kSplitA ? (kk >> 2) * 64 + (kk & 3) * 8 : kk * 8;
    ptx::mma_ts(d_tmem, a_tmem + acol, ptx::desc_sw128(b_lo + kk * (2048 >> 4)), idesc,
                kk > 0 ? 1u : acc);
  }
}

// Issue A (K-major, shared memory, 128 rows x 128 along K in two 64-column
// chunks) x B (MN-major tile of 128 rows along K) into d_tmem.
template <int Chunk>
__device__ __forceinline__ void issue_smem_a(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo,
                                             uint32_t idesc, uint32_t acc) {
#pragma unroll
  for (int kk = 0; kk < kBwdTile / 16; ++kk) {
    const uint32_t aoff = static_cast<uint32_t>((kk >> 2) * Chunk + (kk & 3) * 32) >> 4;
    ptx::mma_ss(d_tmem, ptx::desc_sw128(a_lo + aoff), ptx::desc_sw128(b_lo + kk * (2048 >> 4)),
                idesc, kk > 0 ? 1u : acc);
  }
}

// Issue A x B with both operands MN-major in shared memory (128 rows along
// K each, 16 rows = 2 KB per K step) into a fresh accumulator at d_tmem.
__device__ __forceinline__ void issue_mn_mn(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo,
                                            uint32_t idesc) {
#pragma unroll
  for (int kk = 0; kk < kBwdTile / 16; ++kk)
    ptx::mma_ss(d_tmem, ptx::desc_sw128(a_lo + kk * (2048 >> 4)),
                ptx::desc_sw128(b_lo + kk * (2048 >> 4)), idesc, kk > 0 ? 1u : 0u);
}

// Instruction-descriptor bit that marks A as MN-major (kind::f16).
constexpr uint32_t kIdescAMnMajor = 1u << 15;

// Element-wise fp32 addition of `bytes` (a multiple of 16) of shared memory
// into global memory by the TMA engine, in this thread's bulk group.
__device__ __forceinline__ void bulk_reduce_add_f32(float* gdst, uint32_t ssrc, uint32_t bytes) {
  asm volatile(
      "cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;\n\t"
      "cp.async.bulk.commit_group;" ::"l"(gdst),
      "r"(ssrc), "r"(bytes)
      : "memory");
}
// Wait until this thread's bulk groups have finished reading shared memory
// (the source may be overwritten), or have completed entirely.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// One-pass kernel: TMEM column of dQ buffer b.  At d = 128 TMEM holds S^T,
// dP^T, dV and dK (512 columns), so the single dQ buffer takes the dP^T
// columns once the element-wise warps have read them; at d = 64 two
// buffers of 64 columns follow dV and dK.
template <int D>
struct DqBuf {
  static constexpr int kBufs = (D == 128) ? 1 : 2;
  static __device__ __forceinline__ uint32_t col(int b) {
    return D == 128 ? kColDp : kColAcc + 2u * D + 64u * b;
  }
};

// Write columns [c0, c0 + nc) (nc a multiple of 32) of one row of a TMEM
// accumulator (fp32), times `mul`, to global memory in the storage dtype, in
// rows of `width` values (rows past N are skipped).
template <bool kBf16>
__device__ __forceinline__ void store_acc_cols(uint32_t t_acc, int c0, int nc, int width, float mul,
                                               void* base, long long row, bool in_range) {
  uint4* out = reinterpret_cast<uint4*>(static_cast<uint8_t*>(base) + row * (width * 2) + c0 * 2);
#pragma unroll 1
  for (int q4 = 0; q4 < nc / 32; ++q4) {
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

// Shared setup of one work item of the tensor-core grid: the ring barriers
// and, through `init_x(bar)`, the item's own barriers, initialised by the
// load thread.  The CTA's TMEM is allocated once for all its items.
template <class L, class InitX>
__device__ __forceinline__ void bwd_setup(uint32_t sbase, uint8_t* sgen, InitX init_x) {
  if (threadIdx.x == kBwdLoadWarp * 32) {
    *reinterpret_cast<volatile int*>(sgen + L::kMisc + 4) = 0;
    auto bar = [&](int i) -> uint32_t { return sbase + L::kBar + 8u * i; };
    for (int s = 0; s < L::kStagesA; ++s) {
      ptx::mbar_init(bar(L::bFullA + s), 1);
      ptx::mbar_init(bar(L::bEmptyA + s), 1);
    }
    for (int s = 0; s < L::kStagesB; ++s) {
      ptx::mbar_init(bar(L::bFullB + s), 1);
      ptx::mbar_init(bar(L::bEmptyB + s), 1);
    }
    ptx::mbar_init(bar(L::bRes), 1);
    init_x(bar);
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
}

// End of one work item: every role is done (the MMA thread has seen its
// last commit, the load thread its last copy), so the load thread
// invalidates the item's barriers; the next item, whose layout may put
// other data there, initialises its own.
template <class L>
__device__ __forceinline__ void bwd_teardown(uint32_t sbase) {
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (threadIdx.x == kBwdLoadWarp * 32)
    for (int i = 0; i < L::kNumBars; ++i) ptx::mbar_inval(sbase + L::kBar + 8u * i);
}

// The load thread: the resident pair (res_a, res_b at tile `res_tile`), then
// tiles first .. first + count - 1 of str_a into ring A and of str_b into
// ring B, in the order A_0, B_0, A_1, B_1, ...  The "a" tensors (K and Q)
// have chunks_a 64-column chunks, the "b" tensors (V and dO) chunks_b; only
// those are loaded.
template <class L>
__device__ __forceinline__ void bwd_producer(uint32_t sbase, const CUtensorMap* res_a,
                                             const CUtensorMap* res_b, int res_tile,
                                             const CUtensorMap* str_a, const CUtensorMap* str_b,
                                             int first, int count, int bh,
                                             const ptx::Watchdog& wd, int tok_h = -1,
                                             int res_tok0 = 0, int str_tok0 = 0,
                                             int chunks_a = L::kChunks, int chunks_b = L::kChunks) {
  auto bar = [&](int i) -> uint32_t { return sbase + L::kBar + 8u * i; };
  bool alive = true;
  // tile `tile` of a [BH, rows, d] map: (column, row, batch*head); with
  // packed batches (tok_h = head) of a (column, head, token) map from token
  // tok0 on
  auto y_of = [&](int tile, int tok0) { return tok_h < 0 ? tile * kBwdTile : tok_h; };
  auto z_of = [&](int tile, int tok0) { return tok_h < 0 ? bh : tok0 + tile * kBwdTile; };
  ptx::mbar_arrive_expect_tx(bar(L::bRes), (chunks_a + chunks_b) * L::kChunkBytes);
  for (int c = 0; c < chunks_a; ++c)
    ptx::tma_load_3d(sbase + L::kRes + c * L::kChunkBytes, res_a, bar(L::bRes), c * 64,
                     y_of(res_tile, res_tok0), z_of(res_tile, res_tok0));
  for (int c = 0; c < chunks_b; ++c)
    ptx::tma_load_3d(sbase + L::kRes + L::kTile + c * L::kChunkBytes, res_b, bar(L::bRes), c * 64,
                     y_of(res_tile, res_tok0), z_of(res_tile, res_tok0));
  // one tile of `tm` into slot `slot` of a ring, once its previous use is over
  auto load = [&](const CUtensorMap* tm, int ring, int full0, int empty0, int stages, int it,
                  int chunks) {
    const int slot = it % stages, use = it / stages;
    if (use > 0)
      alive = ptx::wait_bounded(bar(empty0 + slot), (use - 1) & 1, wd, kSiteBwdEmpty) && alive;
    if (!alive) return;
    const uint32_t dst = sbase + ring + slot * L::kTile;
    ptx::mbar_arrive_expect_tx(bar(full0 + slot), chunks * L::kChunkBytes);
    for (int c = 0; c < chunks; ++c)
      ptx::tma_load_3d(dst + c * L::kChunkBytes, tm, bar(full0 + slot), c * 64,
                       y_of(first + it, str_tok0), z_of(first + it, str_tok0));
  };
  int loads = 0;
  for (int it = 0; it < count && alive; ++it) {
    load(str_a, L::kRingA, L::bFullA, L::bEmptyA, L::kStagesA, it, chunks_a);
    if (!alive) break;
    load(str_b, L::kRingB, L::bFullB, L::bEmptyB, L::kStagesB, it, chunks_b);
    if (!alive) {   // tile `it` of ring A was issued: drain it too
      ptx::wait_drain(bar(L::bFullA + it % L::kStagesA), (it / L::kStagesA) & 1, 200000000ull);
      break;
    }
    ++loads;
  }
  // Drain: every issued copy has landed before the CTA can exit.
  const unsigned long long drain = 200000000ull;
  ptx::wait_drain(bar(L::bRes), 0, drain);
  for (int l = loads > L::kStagesA ? loads - L::kStagesA : 0; l < loads; ++l)
    ptx::wait_drain(bar(L::bFullA + l % L::kStagesA), (l / L::kStagesA) & 1, drain);
  for (int l = loads > L::kStagesB ? loads - L::kStagesB : 0; l < loads; ++l)
    ptx::wait_drain(bar(L::bFullB + l % L::kStagesB), (l / L::kStagesB) & 1, drain);
}

// ---------------------------------------------------------------- dK, dV
// Per-query vectors of the dkdv kernel: one buffer at d = 128 (shared memory
// is full), two at d = 64.
template <int D>
struct DkdvVec {
  static constexpr int kBufs = (D == 128) ? 1 : 2;
  static constexpr int kBytes = kBufs * 2 * kBwdTile * 4;
};

// One CTA of the dK/dV pass: block `blk` of BH * n_tiles.
template <int D, bool kBf16, bool kCausal, bool kDrop, bool kKv>
__device__ __forceinline__ void bwd_dkdv_cta(const BwdParams& p, int blk, uint32_t tmem_base) {
  using L = BwdSmem<D, DkdvVec<D>::kBytes>;
  using X = DkdvBars;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = ptx::smem_u32(smem_raw);
  const uint32_t sbase = (raw_base + 1023u) & ~1023u;
  uint8_t* sgen = smem_raw + (sbase - raw_base);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto bar = [&](int i) -> uint32_t { return sbase + L::kBar + 8u * i; };
  auto xbar = [&](int i) -> uint32_t { return bar(L::bX + i); };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sgen + L::kMisc + 4);

  // Key tile kt of head bh; for causal runs the first key tiles of a group
  // of heads (the most query tiles to visit) are dealt first.
  int kt, bh;
  bwd_item(p, blk, p.n_ktiles, kt, bh);
  int i0 = kCausal ? kt : 0;                 // query tiles i >= kt see this key tile
  int len = p.N, off = 0;                    // keys of this head, query offset (kKv)
  int n_q = p.n_tiles;                       // query tiles of this head
  const bool tok = kKv && p.varlen;          // packed batch: token-major rows
  BwdHead hd{p.N, 0, p.N, 0, 0};
  if constexpr (kKv) {
    // the first query that sees key kt * 128 sits at row kt * 128 - off
    hd = bwd_kv_head(p, bh, kCausal);
    len = hd.len;
    off = hd.off;
    if (tok) n_q = (hd.lenq + kBwdTile - 1) / kBwdTile;
    const int first = kt * kBwdTile - off;
    i0 = !kCausal || first <= 0 ? 0 : first / kBwdTile;
    if (kt * kBwdTile >= len) i0 = n_q;      // padding: no query sees these keys
  }
  // key rows this CTA owns: padded keys are written (as zeros); a packed
  // sequence's rows end at its key count
  const int key_rows = tok ? len : p.Nk;
  const int q_rows = tok ? hd.lenq : p.N;
  const int nq = n_q - i0;
  if (kKv && nq <= 0) {
    // no query sees this key tile: its dK and dV rows are zero
    if (threadIdx.x < kBwdEwThreads) {
      const int t = threadIdx.x & 127;
      const long long key = static_cast<long long>(kt) * kBwdTile + t;
      if (key < key_rows) {
        const int width = threadIdx.x < 128 ? p.width_v : p.width_qk;
        uint4* row = reinterpret_cast<uint4*>(static_cast<uint8_t*>(threadIdx.x < 128 ? p.dv : p.dk) +
                                              bwd_krow(p, tok, hd, bh, key) * (width * 2));
        for (int c = 0; c < width / 8; ++c) row[c] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    return;
  }

  bwd_setup<L>(sbase, sgen, [&](auto b) {
    ptx::mbar_init(b(L::bX + X::kSFull), 1);
    ptx::mbar_init(b(L::bX + X::kDpFull), 1);
    ptx::mbar_init(b(L::bX + X::kPReady), kBwdEwThreads);
    ptx::mbar_init(b(L::bX + X::kDsReady), kBwdEwThreads);
    ptx::mbar_init(b(L::bX + X::kDone), 1);
  });
  const ptx::Watchdog wd{p.watchdog_cycles, abort_flag, p.status};

  if (warp == kBwdLoadWarp) {
    if (lane == 0)
      bwd_producer<L>(sbase, &p.tm_k, &p.tm_v, kt, &p.tm_q, &p.tm_do, i0, nq, bh, wd,
                      tok ? bh % p.H : -1, hd.k0, hd.q0, p.width_qk / 64, p.width_v / 64);
    __syncwarp();
  } else if (warp == kBwdMmaWarp) {
    if (lane == 0) {
      constexpr int fmt = kBf16 ? 1 : 0;
      constexpr uint32_t idesc_s = ptx::idesc_f16(kBwdTile, kBwdTile, fmt, 0);
      // dV has width_v columns, dK width_qk
      const uint32_t idesc_dv = ptx::idesc_f16(kBwdTile, p.width_v, fmt, 1);
      const uint32_t idesc_dk = ptx::idesc_f16(kBwdTile, p.width_qk, fmt, 1);
      const int steps_s = p.width_qk / 16, steps_dp = p.width_v / 16;
      constexpr uint32_t kSlotLo = L::kTile >> 4;
      const uint32_t k_lo = ptx::desc_lo(sbase + L::kRes, 16);
      const uint32_t v_lo = ptx::desc_lo(sbase + L::kRes + L::kTile, 16);
      const uint32_t q_lo0 = ptx::desc_lo(sbase + L::kRingA, 16);                  // K-major use
      const uint32_t do_lo0 = ptx::desc_lo(sbase + L::kRingB, 16);
      const uint32_t q_mn0 = ptx::desc_lo(sbase + L::kRingA, L::kChunkBytes);      // MN-major use
      const uint32_t do_mn0 = ptx::desc_lo(sbase + L::kRingB, L::kChunkBytes);
      const uint32_t tS = tmem_base + kColS, tDp = tmem_base + kColDp;
      const uint32_t tDv = tmem_base + kColAcc, tDk = tmem_base + kColAcc + D;
      auto full_a = [&](int it) {
        return ptx::wait_bounded(bar(L::bFullA + it % L::kStagesA), (it / L::kStagesA) & 1, wd,
                                 kSiteBwdFull);
      };
      auto full_b = [&](int it) {
        return ptx::wait_bounded(bar(L::bFullB + it % L::kStagesB), (it / L::kStagesB) & 1, wd,
                                 kSiteBwdFull);
      };
      // S^T = K_j Q_i^T and dP^T = V_j dO_i^T (keys on the TMEM lanes)
      auto issue_s = [&](int it) {
        issue_kmajor<D, L::kChunkBytes>(tS, k_lo, q_lo0 + (it % L::kStagesA) * kSlotLo, idesc_s,
                                        steps_s);
        ptx::mma_commit(xbar(X::kSFull));
      };
      auto issue_dp = [&](int it) {
        issue_kmajor<D, L::kChunkBytes>(tDp, v_lo, do_lo0 + (it % L::kStagesB) * kSlotLo, idesc_s,
                                        steps_dp);
        ptx::mma_commit(xbar(X::kDpFull));
      };
      bool alive = ptx::wait_bounded(bar(L::bRes), 0, wd, kSiteBwdRes);
      alive = alive && full_a(0) && full_b(0);
      ptx::tc_fence_after();
      if (alive) {
        issue_s(0);
        issue_dp(0);
      }
      for (int it = 0; alive && it < nq; ++it) {
        const bool more = it + 1 < nq;
        alive = ptx::wait_bounded(xbar(X::kPReady), it & 1, wd, kSiteBwdPFull);
        ptx::tc_fence_after();
        if (!alive) break;
        // dV_j += P^T dO_i; P^T sits in TMEM columns 0-31 and 64-95
        issue_tmem_a<true>(tDv, tS, do_mn0 + (it % L::kStagesB) * kSlotLo, idesc_dv,
                           it > 0 ? 1u : 0u);
        ptx::mma_commit(bar(L::bEmptyB + it % L::kStagesB));
        if (more) {
          alive = full_a(it + 1);
          ptx::tc_fence_after();
          if (!alive) break;
          issue_s(it + 1);   // after dV in this thread's order: P^T has been read
        }
        alive = ptx::wait_bounded(xbar(X::kDsReady), it & 1, wd, kSiteBwdDsReady);
        ptx::tc_fence_after();
        if (!alive) break;
        // dK_j += dS^T Q_i (scale applied at the end); dS^T in columns 128-159 and 192-223
        issue_tmem_a<true>(tDk, tDp, q_mn0 + (it % L::kStagesA) * kSlotLo, idesc_dk,
                           it > 0 ? 1u : 0u);
        ptx::mma_commit(bar(L::bEmptyA + it % L::kStagesA));
        if (more) {
          alive = full_b(it + 1);
          ptx::tc_fence_after();
          if (!alive) break;
          issue_dp(it + 1);  // after dK: dS^T has been read
        }
      }
      ptx::mma_commit(xbar(X::kDone));
      ptx::wait_drain(xbar(X::kDone), 0, 200000000ull);
    }
    __syncwarp();
  } else {
    // ============================================================ element-wise
    ptx::griddep_wait();   // D of the pass launched just before this grid
    const int quarter = warp & 3, half = warp >> 2;
    const int t = quarter * 32 + lane;                    // key row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    // this thread's 64 query columns of S^T and dP^T
    const uint32_t tS = tmem_base + lane_off + kColS + half * 64;
    const uint32_t tDp = tmem_base + lane_off + kColDp + half * 64;
    const long long key = static_cast<long long>(kt) * kBwdTile + t;
    const uint64_t c2 = ptx::f2_pack(p.scale_log2, p.scale_log2);

    // LSE and D of query row t of tile i, fetched one tile ahead by the
    // first half of the warps.  The loads are unconditional (a row past the
    // queries reads row 0) and nothing uses their values until the tile is
    // staged, so the warps do not wait for them; a query past N then gets
    // -LSE = -inf, so its P is 0, and D = 0.
    bool in_next = false;
    auto fetch = [&](int i, float& lse, float& dd) {
      const int qrow = i * kBwdTile + t;
      in_next = qrow < q_rows;
      const int qr = in_next ? qrow : 0;
      const long long qi = bwd_lse_at(p, tok, hd, bh, qr);
      lse = p.lse[qi];
      dd = p.delta[tok ? bwd_qrow(p, tok, hd, bh, qr) : qi];
    };
    float lse_next = 0.f, d_next = 0.f;
    if (half == 0) fetch(i0, lse_next, d_next);
    float pf[64];          // P^T of the current tile, from phase 1 to phase 2
    // dropout: keep bits of this key against the thread's 64 queries, from
    // the quad's words (zw[2 k2 + m]: word m of lane k2, blocks 8m + 4h + k2
    // of 4 queries each), from phase 1 to phase 2
    uint32_t zw[8] = {};
    const uint32_t csel = 0x4440u + (static_cast<uint32_t>(lane) & 3u);   // this key's byte
    // query bits of block b (queries 4b .. 4b + 3 of the thread's 64)
    auto zq = [&](int b) -> uint32_t {
      return col_query_bits(zw[2 * (b & 3) + (b >> 3)], csel, (b >> 2) & 1);
    };
    // vectors of query tile i0 + it: [0,128) -LSE, [128,256) D
    auto vec_of = [&](int it) {
      return reinterpret_cast<float*>(sgen + L::kVec) + (it % DkdvVec<D>::kBufs) * 256;
    };
    auto stage_vec = [&](int it) {
      float* vec = vec_of(it);
      // with one buffer, every thread must be done with the previous tile's
      if (DkdvVec<D>::kBufs == 1 && it > 0) ptx::named_bar_sync(1, kBwdEwThreads);
      if (half == 0) {
        vec[t] = in_next ? -lse_next * 1.4426950408889634f : -INFINITY;   // -LSE, log2 units
        vec[128 + t] = in_next ? d_next : 0.f;
        if (it + 1 < nq) fetch(i0 + it + 1, lse_next, d_next);
      }
      ptx::named_bar_sync(2, kBwdEwThreads);
    };

    // ---- phase 1: P^T = 2^(S^T c - LSE) over this thread's 64 queries
    auto phase1 = [&](int it) {
      const int i = i0 + it;
      const float4* nl4 = reinterpret_cast<const float4*>(vec_of(it)) + half * 16;
      ptx::wait_bounded(xbar(X::kSFull), it & 1, wd, kSiteBwdSFull);
      __syncwarp();
      ptx::tc_fence_after();
      {
        uint32_t sr[64];
        ptx::tmem_ld32(tS, sr);
        ptx::tmem_ld32(tS + 32, sr + 32);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 64; e += 4) {
          const float4 nl = nl4[e / 4];
          float x0, x1, x2, x3;
          ptx::f2_unpack(ptx::ffma2(ptx::f2_pack(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])),
                                    c2, ptx::f2_pack(nl.x, nl.y)), x0, x1);
          ptx::f2_unpack(ptx::ffma2(ptx::f2_pack(__uint_as_float(sr[e + 2]), __uint_as_float(sr[e + 3])),
                                    c2, ptx::f2_pack(nl.z, nl.w)), x2, x3);
          pf[e] = ptx::ex2(x0);
          pf[e + 1] = ptx::ex2(x1);
          pf[e + 2] = ptx::ex2(x2);
          pf[e + 3] = ptx::ex2(x3);
        }
      }
      if constexpr (kKv) {
        // padding keys see nothing; with causal masking query q sees this
        // key once q + off >= key
        const int qb = i * kBwdTile + half * 64;
        const int lo = key >= len ? 64 : (kCausal ? static_cast<int>(key) - off - qb : 0);
#pragma unroll
        for (int e = 0; e < 64; ++e)
          if (e < lo) pf[e] = 0.f;
      } else if (kCausal && i == kt) {   // diagonal tile: a key after the query is masked
#pragma unroll
        for (int e = 0; e < 64; ++e)
          if (i * kBwdTile + half * 64 + e < key) pf[e] = 0.f;
      }
      // dropout: keep bits of this key against the thread's 64 queries, from
      // the quad's words (zw[2 k2 + m]: word m of lane k2, blocks 8m + 4h + k2
      // of 4 queries each); the dV product reads P with the dropped weights
      // zeroed
      if constexpr (kDrop) {
        const uint2 mine = drop_words16<true>(static_cast<uint32_t>(key >> 2),
                                              static_cast<uint32_t>(i * kBwdTile + half * 64) >> 2,
                                              static_cast<uint32_t>(lane) & 3u,
                                              static_cast<uint32_t>(bh), p.drop_off, p.drop_k0,
                                              p.drop_k1, p.drop_t);
#pragma unroll
        for (int k2 = 0; k2 < 4; ++k2) {
          const int src = (lane & ~3) | k2;
          zw[2 * k2] = __shfl_sync(0xffffffffu, mine.x, src);
          zw[2 * k2 + 1] = __shfl_sync(0xffffffffu, mine.y, src);
        }
      }
      {
        uint32_t pk[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          pk[e] = ptx::pack2<kBf16>(pf[2 * e], pf[2 * e + 1]);
          if constexpr (kDrop) pk[e] &= prmt(zq(e >> 1), 0u, (e & 1) ? 0xBBAAu : 0x9988u);
        }
        ptx::tmem_st16(tS, pk);          // over S^T columns this warp has read
        ptx::tmem_st16(tS + 16, pk + 16);
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(xbar(X::kPReady));
    };

    // ---- phase 2: dS^T = P^T * (dP^T - D)
    auto phase2 = [&](int it) {
      const float4* dl4 = reinterpret_cast<const float4*>(vec_of(it) + 128) + half * 16;
      ptx::wait_bounded(xbar(X::kDpFull), it & 1, wd, kSiteBwdDpFull);
      __syncwarp();
      ptx::tc_fence_after();
      uint32_t dk[32];
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        uint32_t dpr[32];
        ptx::tmem_ld32(tDp + ch * 32, dpr);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const float4 dd = dl4[(ch * 32 + e) / 4];
          const int f = ch * 32 + e;
          // dP^T, with dropout Z dP^T (the 256 / t joins in the subtraction of D)
          uint32_t zx = 0;
          if constexpr (kDrop) zx = zq(f >> 2);   // f is a multiple of 4: one block
          auto dpv = [&](int x) -> float {
            if constexpr (kDrop)
              return __uint_as_float(dpr[e + x] & prmt(zx, 0u, 0x8888u + 0x1111u * x));
            return __uint_as_float(dpr[e + x]);
          };
          auto dmd = [&](float a, float b, float da, float db) -> uint64_t {
            if constexpr (kDrop)
              return ptx::ffma2(ptx::f2_pack(a, b), ptx::f2_pack(p.drop_scale, p.drop_scale),
                                ptx::f2_pack(-da, -db));
            return ptx::fadd2(ptx::f2_pack(a, b), ptx::f2_pack(-da, -db));
          };
          float d0, d1, d2, d3;
          ptx::f2_unpack(ptx::fmul2(ptx::f2_pack(pf[f], pf[f + 1]), dmd(dpv(0), dpv(1), dd.x, dd.y)),
                         d0, d1);
          ptx::f2_unpack(ptx::fmul2(ptx::f2_pack(pf[f + 2], pf[f + 3]),
                                    dmd(dpv(2), dpv(3), dd.z, dd.w)), d2, d3);
          dk[f / 2] = ptx::pack2<kBf16>(d0, d1);
          dk[f / 2 + 1] = ptx::pack2<kBf16>(d2, d3);
        }
      }
      ptx::tmem_st16(tDp, dk);           // over dP^T columns this warp has read
      ptx::tmem_st16(tDp + 16, dk + 16);
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(xbar(X::kDsReady));
    };

    for (int it = 0; it < nq; ++it) {
      stage_vec(it);
      phase1(it);
      phase2(it);
    }
    // dV_j rows (warps 0-3) and dK_j = scale * (dS^T Q) rows (warps 4-7)
    ptx::wait_bounded(xbar(X::kDone), 0, wd, kSiteBwdDone);
    __syncwarp();
    ptx::tc_fence_after();
    const long long row = bwd_krow(p, tok, hd, bh, key);
    if (half == 0)
      store_acc_cols<kBf16>(tmem_base + lane_off + kColAcc, 0, p.width_v, p.width_v,
                            kDrop ? p.drop_scale : 1.f, p.dv, row, key < key_rows);
    else
      store_acc_cols<kBf16>(tmem_base + lane_off + kColAcc + D, 0, p.width_qk, p.width_qk,
                            p.scale, p.dk, row, key < key_rows);
  }
  bwd_teardown<L>(sbase);
}

// ---------------------------------------------------------------- dQ
// TMEM columns of the two dS buffers (16-bit, 64 packed columns each), after dQ.
template <int D>
__device__ __forceinline__ uint32_t dq_ds_col(int b) {
  return kColAcc + D + 64u * b;
}

// One CTA of the dQ pass: block `blk` of BH * n_tiles.
template <int D, bool kBf16, bool kCausal, bool kDrop, bool kKv>
__device__ __forceinline__ void bwd_dq_cta(const BwdParams& p, int blk, uint32_t tmem_base) {
  using L = BwdSmem<D, 0>;
  using X = DqBars;
  static_assert(kColAcc + D + 128 <= kBwdTmemCols, "dS buffers fit in TMEM");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = ptx::smem_u32(smem_raw);
  const uint32_t sbase = (raw_base + 1023u) & ~1023u;
  uint8_t* sgen = smem_raw + (sbase - raw_base);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto bar = [&](int i) -> uint32_t { return sbase + L::kBar + 8u * i; };
  auto xbar = [&](int i) -> uint32_t { return bar(L::bX + i); };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sgen + L::kMisc + 4);

  // Query tile qt of head bh; for causal runs the last query tiles (the most
  // key tiles to visit) are dealt first.
  int r, bh;
  bwd_item(p, blk, p.n_tiles, r, bh);
  const int qt = kCausal ? p.n_tiles - 1 - r : r;
  int nk = kCausal ? qt + 1 : p.n_tiles;   // key tiles j <= qt are visible
  int len = p.N, off = 0;                  // keys of this head, query offset (kKv)
  const bool tok = kKv && p.varlen;        // packed batch: token-major rows
  BwdHead hd{p.N, 0, p.N, 0, 0};
  if constexpr (kKv) {
    // key tiles up to the position of the tile's last query row
    hd = bwd_kv_head(p, bh, kCausal);
    len = hd.len;
    off = hd.off;
    if (qt * kBwdTile >= hd.lenq) return;   // past this sequence's queries: no rows
    const int nkv = (len + kBwdTile - 1) / kBwdTile;
    const int last = min(qt * kBwdTile + kBwdTile, hd.lenq) - 1 + off;
    nk = !kCausal ? nkv : (last < 0 ? 0 : min(last / kBwdTile + 1, nkv));
  }
  const int q_rows = tok ? hd.lenq : p.N;
  if (kKv && nk <= 0) {
    // no query of this tile sees a key: its dQ rows are zero
    if (threadIdx.x < kBwdEwThreads) {
      const int t = threadIdx.x & 127, hf = threadIdx.x >> 7;
      const long long qrow = static_cast<long long>(qt) * kBwdTile + t;
      if (qrow < q_rows) {
        // each half of the threads clears half of the row's width_qk columns
        uint4* row = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.dq) +
                                              bwd_qrow(p, tok, hd, bh, qrow) * (p.width_qk * 2) +
                                              hf * p.width_qk);
        for (int c = 0; c < p.width_qk / 16; ++c) row[c] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    return;
  }

  bwd_setup<L>(sbase, sgen, [&](auto b) {
    ptx::mbar_init(b(L::bX + X::kSFull), 1);
    ptx::mbar_init(b(L::bX + X::kSFree), kBwdEwThreads);
    for (int k = 0; k < 2; ++k) {
      ptx::mbar_init(b(L::bX + X::kPFull + k), kBwdEwThreads);
      ptx::mbar_init(b(L::bX + X::kDsFree + k), 1);
    }
    ptx::mbar_init(b(L::bX + X::kDone), 1);
  });
  const ptx::Watchdog wd{p.watchdog_cycles, abort_flag, p.status};

  if (warp == kBwdLoadWarp) {
    if (lane == 0)
      bwd_producer<L>(sbase, &p.tm_q, &p.tm_do, qt, &p.tm_k, &p.tm_v, 0, nk, bh, wd,
                      tok ? bh % p.H : -1, hd.q0, hd.k0, p.width_qk / 64, p.width_v / 64);
    __syncwarp();
  } else if (warp == kBwdMmaWarp) {
    if (lane == 0) {
      constexpr int fmt = kBf16 ? 1 : 0;
      constexpr uint32_t idesc_s = ptx::idesc_f16(kBwdTile, kBwdTile, fmt, 0);
      const uint32_t idesc_dq = ptx::idesc_f16(kBwdTile, p.width_qk, fmt, 1);   // dQ: width_qk columns
      const int steps_s = p.width_qk / 16, steps_dp = p.width_v / 16;
      constexpr uint32_t kSlotLo = L::kTile >> 4;
      const uint32_t q_lo = ptx::desc_lo(sbase + L::kRes, 16);
      const uint32_t do_lo = ptx::desc_lo(sbase + L::kRes + L::kTile, 16);
      const uint32_t k_lo0 = ptx::desc_lo(sbase + L::kRingA, 16);                 // K-major use
      const uint32_t v_lo0 = ptx::desc_lo(sbase + L::kRingB, 16);
      const uint32_t k_mn0 = ptx::desc_lo(sbase + L::kRingA, L::kChunkBytes);     // MN-major use
      const uint32_t tS = tmem_base + kColS, tDp = tmem_base + kColDp;
      const uint32_t tDq = tmem_base + kColAcc;
      // dQ_i += dS_j K_j for key tile j (scale applied at the end)
      auto issue_dq = [&](int j) -> bool {
        const bool ok = ptx::wait_bounded(xbar(X::kPFull + (j & 1)), (j >> 1) & 1, wd, kSiteBwdPFull);
        ptx::tc_fence_after();
        if (!ok) return false;
        const int slot = j % L::kStagesA;
        issue_tmem_a<false>(tDq, tmem_base + dq_ds_col<D>(j & 1), k_mn0 + slot * kSlotLo, idesc_dq,
                            j > 0 ? 1u : 0u);
        ptx::mma_commit(bar(L::bEmptyA + slot));
        ptx::mma_commit(xbar(X::kDsFree + (j & 1)));
        return true;
      };
      bool alive = ptx::wait_bounded(bar(L::bRes), 0, wd, kSiteBwdRes);
      for (int it = 0; alive && it < nk; ++it) {
        const int sa = it % L::kStagesA, sb = it % L::kStagesB;
        alive = ptx::wait_bounded(bar(L::bFullA + sa), (it / L::kStagesA) & 1, wd, kSiteBwdFull);
        alive = alive && ptx::wait_bounded(bar(L::bFullB + sb), (it / L::kStagesB) & 1, wd, kSiteBwdFull);
        // the element-wise warps have read S and dP of the previous key tile
        if (it > 0) alive = alive && ptx::wait_bounded(xbar(X::kSFree), (it - 1) & 1, wd, kSiteBwdSFree);
        ptx::tc_fence_after();
        if (!alive) break;
        // S = Q_i K_j^T and dP = dO_i V_j^T (queries on the TMEM lanes)
        issue_kmajor<D, L::kChunkBytes>(tS, q_lo, k_lo0 + sa * kSlotLo, idesc_s, steps_s);
        issue_kmajor<D, L::kChunkBytes>(tDp, do_lo, v_lo0 + sb * kSlotLo, idesc_s, steps_dp);
        ptx::mma_commit(xbar(X::kSFull));
        ptx::mma_commit(bar(L::bEmptyB + sb));   // V_j is not read again
        if (it > 0) alive = issue_dq(it - 1);
      }
      if (alive) issue_dq(nk - 1);
      ptx::mma_commit(xbar(X::kDone));
      ptx::wait_drain(xbar(X::kDone), 0, 200000000ull);
    }
    __syncwarp();
  } else {
    // ============================================================ element-wise
    ptx::griddep_wait();   // D of the pass launched just before this grid
    const int quarter = warp & 3, half = warp >> 2;
    const int t = quarter * 32 + lane;                    // query row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    // this thread's 64 key columns of S and dP
    const uint32_t tS = tmem_base + lane_off + kColS + half * 64;
    const uint32_t tDp = tmem_base + lane_off + kColDp + half * 64;
    const long long qrow = static_cast<long long>(qt) * kBwdTile + t;
    const bool q_in = qrow < q_rows;
    const long long grow = bwd_qrow(p, tok, hd, bh, qrow);
    const long long li = bwd_lse_at(p, tok, hd, bh, qrow);
    const float nl = q_in ? -p.lse[li] * 1.4426950408889634f : -INFINITY;
    const float dl = q_in ? p.delta[tok ? grow : li] : 0.f;
    const uint64_t c2 = ptx::f2_pack(p.scale_log2, p.scale_log2);
    const uint64_t nl2 = ptx::f2_pack(nl, nl);
    const uint64_t ndl2 = ptx::f2_pack(-dl, -dl);
    for (int j = 0; j < nk; ++j) {
      ptx::wait_bounded(xbar(X::kSFull), j & 1, wd, kSiteBwdSFull);
      __syncwarp();
      ptx::tc_fence_after();
      // keys past N, and on the diagonal tile keys after this query, are
      // masked (limits relative to this thread's first key column)
      int lim = p.N - j * kBwdTile - half * 64;
      if constexpr (kKv) {
        // keys past this head's count, and with causal masking keys after
        // this query's position
        lim = len - j * kBwdTile - half * 64;
        if (kCausal) lim = min(lim, static_cast<int>(qrow) + off + 1 - j * kBwdTile - half * 64);
      } else if (kCausal && j == qt) {
        lim = min(lim, t + 1 - half * 64);
      }
      // all of S and dP into registers first: the next products wait for this
      uint32_t sr[64], dpr[64];
      ptx::tmem_ld32(tS, sr);
      ptx::tmem_ld32(tS + 32, sr + 32);
      ptx::tmem_ld32(tDp, dpr);
      ptx::tmem_ld32(tDp + 32, dpr + 32);
      ptx::tmem_wait_ld();
      ptx::tc_fence_before();
      ptx::mbar_arrive(xbar(X::kSFree));     // S and dP may be overwritten now
      // dropout: keep bits of this query against the thread's 64 keys, from
      // the quad's words (zw[2 k2 + m]: word m of lane k2, blocks 8m + 4h + k2
      // of 4 keys each)
      uint32_t zw[8] = {};
      if constexpr (kDrop) {
        const uint2 mine = drop_words16<false>(static_cast<uint32_t>(j * kBwdTile + half * 64) >> 2,
                                               static_cast<uint32_t>(qrow >> 2),
                                               static_cast<uint32_t>(lane) & 3u,
                                               static_cast<uint32_t>(bh), p.drop_off, p.drop_k0,
                                               p.drop_k1, p.drop_t);
#pragma unroll
        for (int k2 = 0; k2 < 4; ++k2) {
          const int src = (lane & ~3) | k2;
          zw[2 * k2] = __shfl_sync(0xffffffffu, mine.x, src);
          zw[2 * k2 + 1] = __shfl_sync(0xffffffffu, mine.y, src);
        }
      }
      uint32_t dk[32];
#pragma unroll
      for (int kc = 0; kc < 64; kc += 2) {
        float x0, x1;
        ptx::f2_unpack(ptx::ffma2(ptx::f2_pack(__uint_as_float(sr[kc]), __uint_as_float(sr[kc + 1])),
                                  c2, nl2), x0, x1);
        float p0 = ptx::ex2(x0), p1 = ptx::ex2(x1);
        if (kc >= lim) p0 = 0.f;
        if (kc + 1 >= lim) p1 = 0.f;
        float g0 = __uint_as_float(dpr[kc]), g1 = __uint_as_float(dpr[kc + 1]);
        uint64_t gd;
        if constexpr (kDrop) {   // Z dP 256 / t - D
          const int b = kc >> 2;                       // block of keys 4b .. 4b + 3
          const uint32_t y = zw[2 * (b & 3) + (b >> 3)], r = static_cast<uint32_t>(qrow) & 3u;
          g0 = __uint_as_float(dpr[kc] & row_key_mask(y, r, (b >> 2) & 1, kc & 3));
          g1 = __uint_as_float(dpr[kc + 1] & row_key_mask(y, r, (b >> 2) & 1, (kc + 1) & 3));
          gd = ptx::ffma2(ptx::f2_pack(g0, g1), ptx::f2_pack(p.drop_scale, p.drop_scale), ndl2);
        } else {
          gd = ptx::fadd2(ptx::f2_pack(g0, g1), ndl2);
        }
        float d0, d1;
        ptx::f2_unpack(ptx::fmul2(ptx::f2_pack(p0, p1), gd), d0, d1);
        dk[kc / 2] = ptx::pack2<kBf16>(d0, d1);
      }
      // dS to its TMEM buffer once the tensor core has read what it held
      // (dQ of key tile j - 2)
      const int b = j & 1;
      if (j >= 2) ptx::wait_bounded(xbar(X::kDsFree + b), ((j >> 1) - 1) & 1, wd, kSiteBwdDsFree);
      __syncwarp();
      ptx::tc_fence_after();
      const uint32_t tDs = tmem_base + lane_off + dq_ds_col<D>(b) + half * 32;
      ptx::tmem_st16(tDs, dk);
      ptx::tmem_st16(tDs + 16, dk + 16);
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(xbar(X::kPFull + b));
    }
    // dQ = scale * (dS K): each half of the warps writes half of the columns
    ptx::wait_bounded(xbar(X::kDone), 0, wd, kSiteBwdDone);
    __syncwarp();
    ptx::tc_fence_after();
    store_acc_cols<kBf16>(tmem_base + lane_off + kColAcc, half * (p.width_qk / 2), p.width_qk / 2,
                          p.width_qk, p.scale, p.dq, grow, q_in);
  }
  bwd_teardown<L>(sbase);
}

// ---------------------------------------------------------------- entry point
// Both tensor-core passes in one persistent grid of at most one CTA per SM.
// The work items are [0, BH * n_ktiles) dK/dV items (the ones with the most
// query tiles first), then the dQ items (most key tiles first); CTA c takes
// items c, c + grid, c + 2 grid, ...  (A snake order, c then grid - 1 - c,
// measured no better.)  One grid lets SMs that finish their dK/dV items
// take dQ items at once, so the two passes share one partial last round,
// and a CTA that stays resident across items skips the relaunch and the
// TMEM allocation of every item after its first.  Shared memory is sized
// for the larger layout.
template <int D, bool kBf16, bool kCausal, bool kDrop = false, bool kKv = false>
__global__ void __launch_bounds__(kBwdThreads, 1)
    fa_bwd_kernel(const __grid_constant__ BwdParams p) {
  __shared__ uint32_t s_tmem_base;
  const int warp = threadIdx.x >> 5;
  if (warp == kBwdMmaWarp) {
    ptx::tmem_alloc(ptx::smem_u32(&s_tmem_base), kBwdTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = s_tmem_base;
  const int per_pass = p.BH * p.n_ktiles;   // dK/dV items, one per key tile
  const int total = per_pass + p.BH * p.n_tiles;
  for (int item = blockIdx.x; item < total; item += gridDim.x) {
    if (item < per_pass)
      bwd_dkdv_cta<D, kBf16, kCausal, kDrop, kKv>(p, item, tmem_base);
    else
      bwd_dq_cta<D, kBf16, kCausal, kDrop, kKv>(p, item - per_pass, tmem_base);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kBwdMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, kBwdTmemCols);
  }
}

}  // namespace fa
