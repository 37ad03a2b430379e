// fa_fwd_kernel.cuh — exact attention forward for sm_103a (tcgen05 + TMEM + TMA).
//
// What it computes ("FlashAttention: The Matrix You Never Have to Write
// Down", section "From softmax to attention: rescale the output too"): for
// each query row, key/value tiles stream past a resident query tile; the
// kernel keeps a running maximum m, a running exp-sum l and an unnormalised
// output accumulator O, rescales l and O by exp(m_old - m_new) when a tile
// raises the maximum, and divides O by l once after the last tile (section
// "Build it"; the deferred division).  LSE = m + ln l is written per row.
//
// Rescaling is lazy: the reference maximum is only moved when a tile's
// maximum exceeds it by more than kTau in log2 units (a factor of 2^8);
// otherwise the tile is accumulated against the stale reference.  Because l
// and O always share one reference, the final O / l and m + ln l are exact
// for any threshold (section "What it doesn't solve", the FA4 paragraph on
// deferring the correction while tracking it).
//
// Causal runs skip key tiles that lie wholly in a query tile's future and
// mask only the diagonal tile (section "Causal masking: half the score tiles
// disappear").
//
// Structure of one CTA (persistent; one CTA per SM):
//   warps 0-3  softmax warpgroup 0  -> query tile 0 of the unit (TMEM lanes 0-127)
//   warps 4-7  softmax warpgroup 1  -> query tile 1 of the unit
//   warp  8    MMA issuer (one thread): S = Q K^T
//   warp  9    TMA producer (one thread): Q tiles and a ring of K/V tiles
//   warp  10   MMA issuer (one thread): O += P V
//   warp  11   idle (it completes the third warpgroup, which lets the issue
//              warps give their registers to the softmax warpgroups)
// A work unit is (batch*head, block of 256 query rows) = two 128-row query
// tiles.  TMEM holds S0, S1 (128 fp32 columns each) and O0, O1 (d fp32
// columns each).  P (16-bit) has 64 TMEM columns of its own at d = 64 and a
// shared-memory tile at d = 128 (see OwnP).
//
// The two query tiles ping-pong, so one tile's softmax runs while the tensor
// core works on the other tile.  S_w_{j+1} = Q_w K_{j+1}^T is issued as soon
// as the softmax has read S_w_j into registers (barrier SFree), one key tile
// ahead of the softmax; P_w_j V_j as soon as the softmax has written P_w_j.
// The softmax waits for P_w_{j-1} V_{j-1} (barrier PvDone) before it writes
// P_w_j or rescales O_w.  The two products have an issuing thread each:
// a thread that waits on a barrier stalls until the tensor core has taken
// every MMA it queued before, and with two issuers one thread's waits
// overlap the other's queued work.
#pragma once

#include <cuda.h>
#include <cstdint>

#include "fa_philox.cuh"
#include "ptx_sm103.cuh"

namespace fa {

constexpr int kBM = 128;              // query rows per tile = TMEM lanes
constexpr int kBN = 128;              // keys per K/V tile
constexpr int kThreads = 384;         // three warpgroups
constexpr int kMmaWarp = 8;
constexpr int kLoadWarp = 9;
constexpr int kPvWarp = 10;           // second MMA issuer (own-P layout only)
// Dropout at d = 128 adds a fourth warpgroup (warps 12 .. 15) that draws the
// mask of each key tile ahead of the softmax; at d = 64 (a shorter key step
// than the generator's work) the softmax warps draw their own.
constexpr int kGenWarp0 = 12;
template <int D, bool kDrop>
constexpr bool has_gen() { return kDrop && D == 128; }
template <int D, bool kDrop>
constexpr int threads_of() { return has_gen<D, kDrop>() ? 512 : kThreads; }
// Registers per thread after the split: the launch gives every thread 168
// (64512 per CTA); the issue warpgroup drops to 88 so the two softmax
// warpgroups can hold a whole 128-column score row plus its packed P.
// 2 * 128 * kSoftmaxRegs + 128 * kIssueRegs must not exceed 168 * 384.
constexpr uint32_t kSoftmaxRegs = 208;
constexpr uint32_t kIssueRegs = 88;
static_assert(2 * 128 * kSoftmaxRegs + 128 * kIssueRegs <= 168 * kThreads, "register split");
// With the mask generator, 512 threads launch with 128 registers each (65536
// per CTA): softmax 200, issue 64, mask generator 48.
constexpr uint32_t kSoftmaxRegsDrop = 200;
constexpr uint32_t kIssueRegsDrop = 64;
constexpr uint32_t kGenRegs = 48;
static_assert(2 * 128 * kSoftmaxRegsDrop + 128 * kIssueRegsDrop + 128 * kGenRegs <= 128 * 512,
              "register split with dropout");
constexpr uint32_t kTmemCols = 512;
constexpr float kTau = 8.0f;          // lazy-rescale threshold, log2 units
constexpr float kLn2 = 0.693147180559945309f;

// Sites recorded in the status word when a wait runs out.
enum WaitSite : uint32_t {
  kSiteQEmpty = 1, kSiteKvEmpty = 2, kSiteQFull = 3, kSiteKvFull = 4, kSitePFull = 5,
  kSiteOFree = 6, kSiteSFull = 7, kSiteSFree = 9, kSitePvDone = 10, kSiteMaskFull = 11,
  kSiteMaskEmpty = 12
};

struct FwdParams {
  CUtensorMap tm_q;  // [BH, N, d] boxes of 128 rows x 64 columns, 128-byte swizzle
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  CUtensorMap tm_o;
  void* o;                 // [BH, N, d] (direct-store epilogue)
  float* lse;              // [BH, N]
  unsigned int* status;    // device status word
  unsigned long long watchdog_cycles;  // budget of one bounded wait, SM cycles
  int BH;                  // batch * heads
  int N;                   // sequence length
  int n_qblk;              // ceil(N / 256): units per head
  int n_kv;                // ceil(N / 128): key tiles per head
  int num_units;           // BH * n_qblk
  int hgroup;              // unit order: heads per group, 1 .. BH (see unit_at)
  // Split tail (unmasked only, see next_piece): after full_rounds rounds of
  // whole units, the last tail_units units are cut along the key axis so
  // every CTA gets the same number of key tiles.  Partial results go to
  // ws_part; ws_count counts, per (tail unit, query tile), pieces finished.
  int split;               // 0: whole units only
  int full_rounds;
  int tail_units;
  float* ws_part;          // 2 * grid slots of kSlotFloats(D) floats
  int* ws_count;           // 2 * tail_units counters, zero at launch
  float scale_log2;        // scale * log2(e)
  unsigned long long* trace;  // event trace buffer (only read in FA_TRACE builds)
  // Queries against a key set of another length (kKv variants only; N is
  // then the number of queries): keys per head Nk (tm_k / tm_v have Nk
  // rows), per-batch key counts seqlens_k[b] (NULL: all Nk; batch b = bh / H),
  // and the causal alignment: align_br = 0 puts query i at position i,
  // align_br = 1 at position len_b - N + i (the queries are the last N
  // positions of the batch's keys).
  int Nk;
  int H;
  const int* seqlens_k;
  int align_br;
  // Widths (kKv variants only): dqk of Q and K, dv of V and O, each 64 or
  // 128 with D = max(dqk, dv).  Each tensor map has its tensor's own width
  // and only those 64-column chunks are loaded; S takes only dqk / 16 K
  // steps and O += P V computes only dv columns, so the chunks not loaded
  // are never read.
  int dqk;
  int dv;
  // Packed variable-length batches (kKv variants with varlen = 1): Q, O
  // token-major [total_q, H, d|dv], K, V [Nk = total_k, H, d|dv], LSE
  // [H, total_q]; sequence b owns query tokens cu_q[b] .. cu_q[b+1] - 1 and
  // key tokens cu_k[b] .. cu_k[b+1] - 1 (clamped to the totals); N is then
  // the longest query count the call was sized for.  The tensor maps are
  // (column, head, token), so a TMA box of 128 tokens of one head lands in
  // the same shared-memory layout as a tile of the [B, H, N, d] layout.
  const int* cu_q;
  const int* cu_k;
  int varlen;
  int total_q;
  // Dropout on the attention weights (kDrop variants only): keep threshold
  // t (1 .. 255), the seed as two words, the caller's offset, and 256 / t.
  uint32_t drop_t;
  uint32_t drop_k0, drop_k1;
  uint32_t drop_off;
  float drop_scale;
};

// ---------------------------------------------------------------- tracing
// Builds compiled with -DFA_TRACE record timestamped events of each role of
// each CTA (SM clock, clock64) into p.trace: kTraceCap events of two 64-bit
// words (time, event << 32 | argument) per (CTA, role).  Roles: 0/1 softmax
// warpgroups (their first thread), 2 MMA issuer, 3 TMA producer.  Normal
// builds compile every trace point away.
constexpr int kTraceCap = 4096;
enum TraceEvent : uint32_t {
  kEvSReady = 1, kEvPArrive = 2, kEvRescale = 3, kEvEpiStart = 4, kEvEpiEnd = 5,
  kEvUnit = 10, kEvPvIssue = 11, kEvSIssue = 12, kEvKvWaited = 13, kEvPWaited = 14,
  kEvLoadK = 20, kEvLoadV = 21, kEvLoadQ = 22
};
// Builds compiled with -DFA_PROFILE instead accumulate, per role, the SM
// cycles spent in each wait and work phase, and write the totals once at the
// end (kProfSlots 32-bit counters per role per CTA, into p.trace).
constexpr int kProfSlots = 20;
struct Prof {
#ifdef FA_PROFILE
  uint32_t acc[kProfSlots];
  long long t_mark;
  __device__ __forceinline__ Prof() : t_mark(ptx::clk64()) {
#pragma unroll
    for (int i = 0; i < kProfSlots; ++i) acc[i] = 0;
  }
  // Charge the cycles since the previous mark to counter i.
  __device__ __forceinline__ void lap(int i) {
    const long long t = ptx::clk64();
    acc[i] += static_cast<uint32_t>(t - t_mark);
    t_mark = t;
  }
  __device__ __forceinline__ void count(int i) { acc[i] += 1; }
  __device__ __forceinline__ void flush(const FwdParams& p, int role) {
    if (p.trace == nullptr) return;
    unsigned long long* dst = p.trace + (static_cast<size_t>(blockIdx.x) * 4 + role) * kProfSlots;
#pragma unroll
    for (int i = 0; i < kProfSlots; ++i) dst[i] = acc[i];
  }
#else
  __device__ __forceinline__ void lap(int) {}
  __device__ __forceinline__ void count(int) {}
  __device__ __forceinline__ void flush(const FwdParams&, int) {}
#endif
};

__device__ __forceinline__ void trace_event(const FwdParams& p, int role, uint32_t& cnt,
                                            uint32_t ev, uint32_t arg) {
#ifdef FA_TRACE
  if (p.trace != nullptr && cnt < static_cast<uint32_t>(kTraceCap)) {
    const size_t i = (static_cast<size_t>(blockIdx.x) * 4 + role) * kTraceCap + cnt;
    p.trace[2 * i] = ptx::clk64();
    p.trace[2 * i + 1] = (static_cast<unsigned long long>(ev) << 32) | arg;
  }
  ++cnt;
#else
  (void)p; (void)role; (void)cnt; (void)ev; (void)arg;
#endif
}

// Where P lives.  P has storage of its own, so the next S of a query tile
// can be computed as soon as the softmax has read the current S into
// registers, which takes the tensor-core work of the next tile off the
// softmax's critical path.  At d = 64 the last 128 TMEM columns are free and
// each query tile gets a P buffer there (64 columns: 128 16-bit values per
// row).  At d = 128, S0, S1, O0 and O1 fill all 512 TMEM columns, so P goes
// to shared memory (one 128 x 128 tile per query tile, laid out like a Q
// tile) and the P.V product reads both operands from there.
template <int D>
struct OwnP {
  static constexpr bool kTmem = (2 * 128 + 2 * D + 2 * 64) <= static_cast<int>(kTmemCols);
  static constexpr bool kSmem = !kTmem;
};

// Shared-memory plan.  At d = 128 the two output staging tiles would cost two
// K/V ring stages (the ring then cannot cover L2 latency), so O is written
// straight from registers; at d = 64 there is room for both, and O goes out
// through a staging tile and a TMA store.  With the dropout mask generator
// (d = 128), each query tile's keep bits come over in a ring of kMaskStages
// buffers of kMaskBytes (128 rows x 128 keys, one bit each); they take the
// room of one K/V stage, and the ring keeps two (a key step with dropout
// lasts several microseconds, longer than a tile's load).
template <int D, bool kDrop = false>
struct Smem {
  static constexpr bool kGen = has_gen<D, kDrop>();
  static constexpr int kChunks = D / 64;             // 128-byte swizzle columns per row
  static constexpr int kTile = kBM * D * 2;          // one 128 x D tile of 16-bit values
  static constexpr int kChunkBytes = kBM * 128;      // 128 rows x 128 bytes
  static constexpr bool kTmaStore = (D == 64);       // epilogue through smem + TMA store
  // K/V ring depth (at d = 128 with P in shared memory the two P tiles take
  // two of the five stages)
  static constexpr int kStages = (D == 128) ? (OwnP<D>::kSmem ? (kGen ? 2 : 3) : 5) : 8;
  static constexpr int kMaskStages = 2;
  static constexpr int kMaskBytes = kBM * kBN / 8;
  // Q buffers (two query tiles each): at d = 64 two, so a unit's Q tiles
  // load while the previous unit still runs (units of a few key tiles
  // otherwise waited for them); at d = 128 one (no room).
  static constexpr int kQBufs = (D == 64) ? 2 : 1;
  static constexpr int kQ = 0;
  static constexpr int kKV = kQ + kQBufs * 2 * kTile;   // ring of K or V tiles
  static constexpr int kO = kKV + kStages * kTile;   // two output staging tiles (if any)
  static constexpr int kP = kO + (kTmaStore ? 2 * kTile : 0);   // two P tiles (if in smem)
  static constexpr int kMask = kP + (OwnP<D>::kSmem ? 2 * kBM * kBN * 2 : 0);  // mask rings
  static constexpr int kBar = kMask + (kGen ? 2 * kMaskStages * kMaskBytes : 0);
  // barrier indices (the mask barriers, [query tile][stage], only with the generator)
  static constexpr int bQFull = 0, bQEmpty = kQBufs, bKvFull = 2 * kQBufs,
                       bKvEmpty = bKvFull + kStages, bSFull = bKvFull + 2 * kStages,
                       bPFull = bSFull + 2,
                       bOFree = bPFull + 2, bSFree = bOFree + 2, bPvDone = bSFree + 2,
                       bFinal = bPvDone + 2, bFinalPv = bFinal + 1, bMaskFull = bFinalPv + 1,
                       bMaskEmpty = bMaskFull + 2 * kMaskStages,
                       kNumBars = kGen ? bMaskEmpty + 2 * kMaskStages : bFinalPv + 1;
  static constexpr int kMisc = kBar + 8 * kNumBars;  // tmem base, abort flag, 2 merge flags
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;       // slack to align the base to 1024
  static_assert(kAlloc <= 232448, "shared memory budget");
};

// TMEM column of S / O for query tile w.
template <int D>
__device__ __forceinline__ uint32_t s_col(int w) { return w ? 128u : 0u; }
template <int D>
__device__ __forceinline__ uint32_t o_col(int w) { return 256u + (w ? D : 0); }
// TMEM column of P (d = 64, where P is in TMEM).
template <int D>
__device__ __forceinline__ uint32_t p_col(int w) { return 256u + 2u * D + (w ? 64u : 0u); }

struct Unit {
  int bh, mblk, n0, n1;
  int len, off;   // keys of this head; position of query row r is r + off (kKv)
  int lenq, q0, k0;   // queries of this head; first query and key token (varlen)
};

// A piece of work: key tiles [kb, kb + n_w) of query tile w of one unit.
// tail >= 0 marks a partial piece of tail unit `tail` whose results go to
// workspace slot `slot` and are merged by whichever piece finishes last.
struct Piece {
  int bh, mblk, kb, n0, n1, tail, slot;
  int len, off, lenq, q0, k0;   // as in Unit
};

// Floats of one workspace slot: unnormalised O of both query tiles stored
// column by column (element (col, row) of tile w at (w*D + col)*128 + row,
// so a warp's rows are contiguous), then (-m*c, l) per row.
template <int D>
__host__ __device__ constexpr int kSlotFloats() { return 2 * kBM * (D + 2); }

// Static persistent schedule, deterministic so every role of a CTA walks the
// same list without communicating.  Units are dealt to CTAs in a snake
// (boustrophedon) order, round by round, from one ordering: heads in groups
// of `hgroup`, one group after the other, and inside a group level by level
// (the heaviest query block of each of its heads first; for causal masking
// the last blocks).  hgroup = BH is plain level order, which balances best
// when the K/V of all heads fit in L2; hgroup = 1 walks one head at a time,
// so the units in flight share a few heads' K/V in L2.  The host picks the
// group from the L2 budget and the balance of the deal (fa_fwd_api.cu).
__device__ __forceinline__ int unit_at(int round, int cta, int grid) {
  return round * grid + ((round & 1) ? (grid - 1 - cta) : cta);
}

__host__ __device__ __forceinline__ int imin(int a, int b) { return a < b ? a : b; }
__host__ __device__ __forceinline__ int imax(int a, int b) { return a > b ? a : b; }

// Unit s of the schedule: its (batch*head, query block) and the number of key
// tiles each of its two query tiles streams.  Host code calls it too
// (fa_work_tiles counts the tile pairs of a head with it), so the count the
// host reports is the loop bound the kernel runs.
template <bool kCausal, bool kKv = false>
__host__ __device__ __forceinline__ Unit decode_unit(int s, const FwdParams& p) {
  Unit u;
  {
    const int per_group = p.hgroup * p.n_qblk;
    const int g = s / per_group;
    const int r = s - g * per_group;
    const int gl = imin(p.hgroup, p.BH - g * p.hgroup);   // heads in this group (the last may be short)
    const int level = r / gl;
    u.bh = g * p.hgroup + (r - level * gl);
    u.mblk = p.n_qblk - 1 - level;
  }
  const int t0 = 2 * u.mblk;
  if constexpr (kKv) {
    // keys and queries of this batch, and the key tiles each query tile can
    // see: with causal masking, keys up to the position of its last row
    const int b = u.bh / p.H;
    int len, lenq = p.N, q0 = 0, k0 = 0;
    if (p.varlen) {
      q0 = imin(imax(p.cu_q[b], 0), p.total_q);
      lenq = imin(imax(p.cu_q[b + 1], q0), p.total_q) - q0;
      k0 = imin(imax(p.cu_k[b], 0), p.Nk);
      len = imin(imax(p.cu_k[b + 1], k0), p.Nk) - k0;
    } else {
      len = p.seqlens_k ? p.seqlens_k[b] : p.Nk;
      len = imin(imax(len, 0), p.Nk);
    }
    u.len = len;
    u.lenq = lenq;
    u.q0 = q0;
    u.k0 = k0;
    u.off = (kCausal && p.align_br) ? len - lenq : 0;
    const int nkv = (len + kBN - 1) / kBN;
    int n[2];
#pragma unroll
    for (int w = 0; w < 2; ++w) {
      const int first = (t0 + w) * kBM;                       // the tile's first row
      const int last = imin(first + kBM, lenq) - 1 + u.off;   // position of its last row
      n[w] = first >= lenq ? 0 : !kCausal ? nkv : (last < 0 ? 0 : imin(last / kBN + 1, nkv));
    }
    u.n0 = n[0];
    u.n1 = n[1];
  } else {
    u.len = p.N;
    u.off = 0;
    u.lenq = p.N;
    u.q0 = 0;
    u.k0 = 0;
    // causal: key tiles 0 .. t of query tile t (the last one is the diagonal
    // tile, the only one masked); tiles wholly in the future are never visited
    if (kCausal) {
      u.n0 = imin(t0 + 1, p.n_kv);
      u.n1 = imin(t0 + 2, p.n_kv);
    } else {
      u.n0 = p.n_kv;
      u.n1 = p.n_kv;
    }
  }
  if ((t0 + 1) * kBM >= p.N) u.n1 = 0;  // second query tile lies wholly past N
  return u;
}

// Per-CTA walk over its pieces.  Whole units first (round by round as
// above); with a split tail, CTA c then takes tail key tiles
// [c*W/grid, (c+1)*W/grid) of the W = tail_units * n_kv tail key tiles, in
// unit order, so every CTA does the same number of key tiles and at most two
// pieces of the tail.
struct Cursor {
  int r;                 // next round of whole units
  long long pos, end;    // tail key tiles left to this CTA
  int first_t;           // tail unit of this CTA's first tail piece
};
__device__ __forceinline__ long long tail_start(const FwdParams& p, int c, int grid) {
  return static_cast<long long>(p.tail_units) * p.n_kv * c / grid;
}
template <bool kSplit>
__device__ __forceinline__ void cursor_init(const FwdParams& p, int cta, int grid, Cursor& cu) {
  cu.r = 0;
  cu.pos = kSplit ? tail_start(p, cta, grid) : 0;
  cu.end = kSplit ? tail_start(p, cta + 1, grid) : 0;
  cu.first_t = kSplit ? static_cast<int>(cu.pos / p.n_kv) : 0;
}
template <bool kCausal, bool kSplit, bool kKv = false>
__device__ __forceinline__ bool next_piece(const FwdParams& p, int cta, int grid, Cursor& cu,
                                           Piece& pc) {
  if (!kSplit || cu.r < p.full_rounds) {
    const int s = unit_at(cu.r, cta, grid);
    if (!kSplit && s >= p.num_units) return false;
    ++cu.r;
    const Unit u = decode_unit<kCausal, kKv>(s, p);
    pc.bh = u.bh; pc.mblk = u.mblk; pc.kb = 0; pc.n0 = u.n0; pc.n1 = u.n1;
    pc.tail = -1; pc.slot = 0; pc.len = u.len; pc.off = u.off;
    pc.lenq = u.lenq; pc.q0 = u.q0; pc.k0 = u.k0;
    return true;
  }
  if (cu.pos >= cu.end) return false;
  const int t = static_cast<int>(cu.pos / p.n_kv);
  const long long ubeg = static_cast<long long>(t) * p.n_kv;
  const int kb = static_cast<int>(cu.pos - ubeg);
  const int ke = static_cast<int>((cu.end < ubeg + p.n_kv ? cu.end : ubeg + p.n_kv) - ubeg);
  cu.pos = ubeg + ke;
  const Unit u = decode_unit<kCausal>(p.full_rounds * grid + t, p);
  pc.bh = u.bh; pc.mblk = u.mblk; pc.kb = kb;
  pc.n0 = ke - kb;
  pc.n1 = u.n1 > 0 ? ke - kb : 0;
  pc.tail = (kb == 0 && ke == p.n_kv) ? -1 : t;
  pc.slot = 2 * cta + (t == cu.first_t ? 0 : 1);
  pc.len = u.len; pc.off = u.off;
  pc.lenq = u.lenq; pc.q0 = u.q0; pc.k0 = u.k0;
  return true;
}

// Walks the CTAs holding pieces of one tail unit, in CTA order, without a
// division per step: CTA c's tail range starts at c*q + floor(c*r/grid)
// with q = W / grid, r = W mod grid (W = tail_units * n_kv), so consecutive
// starts differ by q or q + 1.  Each CTA holds at most one piece of a unit.
struct TailWalk {
  int c;            // current CTA
  long long st;     // its tail range start
  int frac;         // c * r mod grid
  long long q;
  int r, grid;
  __device__ __forceinline__ void init(const FwdParams& p, int grid_, int t) {
    grid = grid_;
    const long long W = static_cast<long long>(p.tail_units) * p.n_kv;
    q = W / grid;
    r = static_cast<int>(W - q * grid);
    const long long ua = static_cast<long long>(t) * p.n_kv;
    // first CTA whose range starts at or before ua (its range then covers ua)
    long long c0 = ((ua + 1) * grid + W - 1) / W - 1;
    c = static_cast<int>(c0 < 0 ? 0 : (c0 > grid - 1 ? grid - 1 : c0));
    st = static_cast<long long>(c) * q + (static_cast<long long>(c) * r) / grid;
    frac = static_cast<int>((static_cast<long long>(c) * r) % grid);
  }
  __device__ __forceinline__ long long next_start() const {
    return st + q + ((frac + r >= grid) ? 1 : 0);
  }
  __device__ __forceinline__ void step() {
    st += q;
    frac += r;
    if (frac >= grid) { ++st; frac -= grid; }
    ++c;
  }
};

// Output row of query row `row` of piece u (O is addressed in rows of the
// value width) and its LSE element: [B, H, N, .] and [B, H, N], or with
// packed batches [total_q, H, .] and [H, total_q].
template <bool kKv>
__device__ __forceinline__ size_t out_row(const FwdParams& p, const Piece& u, int row) {
  if constexpr (kKv) {
    if (p.varlen) return static_cast<size_t>(u.q0 + row) * p.H + (u.bh % p.H);
  }
  return static_cast<size_t>(u.bh) * p.N + row;
}
template <bool kKv>
__device__ __forceinline__ size_t lse_at(const FwdParams& p, const Piece& u, int row) {
  if constexpr (kKv) {
    if (p.varlen) return static_cast<size_t>(u.bh % p.H) * p.total_q + u.q0 + row;
  }
  return static_cast<size_t>(u.bh) * p.N + row;
}

// kSplit: compile the split-tail path (unmasked calls with a workspace only);
// the other variants carry none of its code.
// kKv: queries against a key set of their own length, per-batch key counts
// and a causal alignment (see FwdParams); square calls compile none of it.
// kDrop: dropout on the attention weights (with kKv on square shapes).
template <int D, bool kBf16, bool kCausal, bool kSplit, bool kKv = false, bool kDrop = false>
__global__ void __launch_bounds__(threads_of<D, kDrop>(), 1)
    fa_fwd_kernel(const __grid_constant__ FwdParams p) {
  using L = Smem<D, kDrop>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = ptx::smem_u32(smem_raw);
  const uint32_t sbase = (raw_base + 1023u) & ~1023u;
  uint8_t* sgen = smem_raw + (sbase - raw_base);  // generic pointer to the aligned base

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  auto bar = [&](int i) -> uint32_t { return sbase + L::kBar + 8u * i; };
  uint32_t* tmem_base_ptr = reinterpret_cast<uint32_t*>(sgen + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sgen + L::kMisc + 4);
  volatile int* merge_flag = reinterpret_cast<volatile int*>(sgen + L::kMisc + 8);  // [2]

  // ---------------------------------------------------------------- setup
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_base_ptr), kTmemCols);
    ptx::tmem_relinquish();
  }
  if (threadIdx.x == kLoadWarp * 32) {
    *abort_flag = 0;
    for (int qb = 0; qb < L::kQBufs; ++qb) {
      ptx::mbar_init(bar(L::bQFull + qb), 1);
      ptx::mbar_init(bar(L::bQEmpty + qb), 1);
    }
    for (int s = 0; s < L::kStages; ++s) {
      ptx::mbar_init(bar(L::bKvFull + s), 1);
      ptx::mbar_init(bar(L::bKvEmpty + s), 1);
    }
    for (int w = 0; w < 2; ++w) {
      ptx::mbar_init(bar(L::bSFull + w), 1);
      ptx::mbar_init(bar(L::bPFull + w), 128);
      ptx::mbar_init(bar(L::bOFree + w), 128);
      ptx::mbar_init(bar(L::bSFree + w), 128);
      ptx::mbar_init(bar(L::bPvDone + w), 1);
    }
    ptx::mbar_init(bar(L::bFinal), 1);
    ptx::mbar_init(bar(L::bFinalPv), 1);
    if constexpr (L::kGen) {
      for (int i = 0; i < 2 * L::kMaskStages; ++i) {
        ptx::mbar_init(bar(L::bMaskFull + i), 128);    // every generator thread
        ptx::mbar_init(bar(L::bMaskEmpty + i), 128);   // every softmax thread of the tile
      }
    }
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
    ptx::prefetch_tmap(&p.tm_q);
    ptx::prefetch_tmap(&p.tm_k);
    ptx::prefetch_tmap(&p.tm_v);
    ptx::prefetch_tmap(&p.tm_o);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_base_ptr;
  const ptx::Watchdog wd{p.watchdog_cycles, abort_flag, p.status};
  const int grid = gridDim.x;
  const int cta = blockIdx.x;
  // Each role's code sits inside the branch that set its register budget.
  bool gen_role = false;
  if constexpr (L::kGen) gen_role = (warp >= kGenWarp0);
  if (gen_role) {
    ptx::setmaxnreg_dec<kGenRegs>();
    if constexpr (L::kGen) {
      // ============================================================ dropout mask generator
      // Thread g draws, for every (query tile, key tile) the softmax will
      // process, the words of lane g % 4 of row quad g / 4 (drop_words) and
      // stores them at [lane][quad] of the tile's mask buffer; the softmax
      // thread of row 4 * quad + r reads the quad's four words back.  The
      // order (key tile, then query tile) is the order the issuers serve
      // the two query tiles in, so neither softmax waits on masks the
      // generator holds back for the other.
      const int g = threadIdx.x - kGenWarp0 * 32;
      const uint32_t quad = static_cast<uint32_t>(g) >> 2, kq = static_cast<uint32_t>(g) & 3u;
      uint32_t mc0 = 0, mc1 = 0;    // masks produced for query tile 0 / 1
      bool alive = true;
      Cursor cu;
      cursor_init<kSplit>(p, cta, grid, cu);
      Piece u;
      while (next_piece<kCausal, kSplit, kKv>(p, cta, grid, cu, u)) {
        const int nkv = max(u.n0, u.n1);
        for (int j = 0; j < nkv; ++j) {
          for (int w = 0; w < 2; ++w) {
            if (j >= (w ? u.n1 : u.n0)) continue;
            uint32_t& mc = w ? mc1 : mc0;
            const uint32_t use = mc / L::kMaskStages;
            const int bi = w * L::kMaskStages + static_cast<int>(mc % L::kMaskStages);
            if (use > 0)
              alive = ptx::wait_bounded(bar(L::bMaskEmpty + bi), (use - 1) & 1, wd,
                                        kSiteMaskEmpty) && alive;
            if (alive) {
              const uint32_t qrow0 = static_cast<uint32_t>((2 * u.mblk + w) * kBM) + 4u * quad;
              const uint4 words = drop_words(qrow0, static_cast<uint32_t>((u.kb + j) * kBN), kq,
                                             u.bh, p.drop_off, p.drop_k0, p.drop_k1, p.drop_t);
              *reinterpret_cast<uint4*>(sgen + L::kMask + bi * L::kMaskBytes +
                                        (kq * 32 + quad) * 16) = words;
            }
            ptx::mbar_arrive(bar(L::bMaskFull + bi));
            ++mc;
          }
        }
      }
    }
  } else if (warp >= 8) {
  ptx::setmaxnreg_dec<L::kGen ? kIssueRegsDrop : kIssueRegs>();
  if (warp == kLoadWarp) {
    // ============================================================ TMA producer
    if (lane == 0) {
      uint32_t tr = 0;          // trace events recorded
      uint32_t loads = 0;       // K/V tiles issued (ring position)
      uint32_t q_issued = 0;    // units whose Q load was issued
      uint32_t k_units = 0;     // pieces walked
      bool alive = true;
      Cursor cu;
      cursor_init<kSplit>(p, cta, grid, cu);
      Piece u;
      while (next_piece<kCausal, kSplit, kKv>(p, cta, grid, cu, u)) {
        const int nkv = max(u.n0, u.n1);
        if (kKv && nkv == 0) continue;   // no visible key: the softmax warps write the rows
        // Q of this piece may only overwrite the buffer once the previous
        // piece's last S MMA has read it; the first K tile does not wait for
        // that, so it is requested first.
        auto load_q = [&]() {
          const uint32_t qb = k_units % L::kQBufs, quse = k_units / L::kQBufs;
          if (quse > 0)
            alive = ptx::wait_bounded(bar(L::bQEmpty + qb), (quse - 1) & 1, wd, kSiteQEmpty) &&
                    alive;
          if (alive) {
            const int ntile = u.n1 > 0 ? 2 : 1;
            // kKv with d < D: only the chunks of Q's own columns are loaded
            // (the S products never read the others)
            const int qc = kKv ? p.dqk / 64 : L::kChunks;
            ptx::mbar_arrive_expect_tx(bar(L::bQFull + qb), ntile * qc * L::kChunkBytes);
            for (int w = 0; w < ntile; ++w) {
              int y = (2 * u.mblk + w) * kBM, z = u.bh;      // row, batch*head
              if (kKv && p.varlen) { z = u.q0 + y; y = u.bh % p.H; }   // head, token
              for (int c = 0; c < qc; ++c)
                ptx::tma_load_3d(sbase + L::kQ + (qb * 2 + w) * L::kTile + c * L::kChunkBytes,
                                 &p.tm_q, bar(L::bQFull + qb), c * 64, y, z);
            }
            q_issued = k_units + 1;
            trace_event(p, 3, tr, kEvLoadQ, k_units);
          }
        };
        auto load_kv = [&](int kv, int j) {
          const uint32_t slot = loads % L::kStages, use = loads / L::kStages;
          if (use > 0)
            alive = ptx::wait_bounded(bar(L::bKvEmpty + slot), (use - 1) & 1, wd, kSiteKvEmpty) &&
                    alive;
          if (alive) {
            // kKv: only the chunks of the tensor's own width (d for K, dv for V)
            const int nc = kKv ? (kv ? p.dv : p.dqk) / 64 : L::kChunks;
            ptx::mbar_arrive_expect_tx(bar(L::bKvFull + slot), nc * L::kChunkBytes);
            const CUtensorMap* tm = kv ? &p.tm_v : &p.tm_k;
            int y = (u.kb + j) * kBN, z = u.bh;              // row, batch*head
            if (kKv && p.varlen) { z = u.k0 + y; y = u.bh % p.H; }   // head, token
            for (int c = 0; c < nc; ++c)
              ptx::tma_load_3d(sbase + L::kKV + slot * L::kTile + c * L::kChunkBytes, tm,
                               bar(L::bKvFull + slot), c * 64, y, z);
            trace_event(p, 3, tr, kv ? kEvLoadV : kEvLoadK, j);
            ++loads;
          }
        };
        // The ring is filled in the order the two MMA issuers need the tiles:
        // K0 K1 V0 K2 V1 ... K_{n-1} V_{n-2} V_{n-1} (S_{j+1} before P_j V_j).
        load_kv(0, 0);
        load_q();
        for (int j = 0; j < nkv; ++j) {
          if (j + 1 < nkv) load_kv(0, j + 1);
          load_kv(1, j);
        }
        ++k_units;
      }
      // Drain: make sure every issued copy has landed before the CTA can exit.
      const unsigned long long drain = 200000000ull;   // cycles (~0.1 s)
      const uint32_t first = loads > (uint32_t)L::kStages ? loads - L::kStages : 0;
      for (uint32_t l = first; l < loads; ++l)
        ptx::wait_drain(bar(L::bKvFull + l % L::kStages), (l / L::kStages) & 1, drain);
      for (uint32_t q = q_issued > (uint32_t)L::kQBufs ? q_issued - L::kQBufs : 0; q < q_issued; ++q)
        ptx::wait_drain(bar(L::bQFull + q % L::kQBufs), (q / L::kQBufs) & 1, drain);
    }
    __syncwarp();
  } else if (warp == kMmaWarp || warp == kPvWarp) {
    // ============================================================ MMA issuers
    // The issue loop has to keep up with the tensor core (an M128 x N128 x
    // K16 MMA lasts ~64 cycles), so descriptors are precomputed: per MMA only
    // the 32-bit address word changes, by a compile-time offset.
    // Warp 8 issues the S = Q K^T products, warp 10 the O += P V products.
    if (lane == 0) {
      constexpr int fmt = kBf16 ? 1 : 0;
      constexpr uint32_t idesc_s = ptx::idesc_f16(kBM, kBN, fmt, 0);  // Q (K-major) x K (K-major)
      constexpr uint32_t idesc_o_full = ptx::idesc_f16(kBM, D, fmt, 1);  // P x V (MN-major)
      // a value width below D (kKv) computes only dv columns of O
      const uint32_t idesc_o =
          (kKv && p.dv < D) ? ptx::idesc_f16(kBM, 64, fmt, 1) : idesc_o_full;
      // Address words of the shared-memory descriptors (start >> 4 | LBO >> 4 << 16).
      const uint32_t q_lo0 = ptx::desc_lo(sbase + L::kQ, 16);
      const uint32_t q_lo1 = ptx::desc_lo(sbase + L::kQ + L::kTile, 16);
      const uint32_t k_lo0 = ptx::desc_lo(sbase + L::kKV, 16);
      const uint32_t v_lo0 = ptx::desc_lo(sbase + L::kKV, L::kChunkBytes);
      constexpr uint32_t kSlotLo = L::kTile >> 4;
      const uint32_t tS0 = tmem_base + s_col<D>(0), tS1 = tmem_base + s_col<D>(1);
      const uint32_t tO0 = tmem_base + o_col<D>(0), tO1 = tmem_base + o_col<D>(1);

      // S = Q_w K^T over the head width: K-major operands, 128-byte swizzle;
      // a K step of 16 columns moves 32 bytes inside a swizzle row, and every
      // 64 columns start a new chunk.
      const int s_steps = kKv ? p.dqk / 16 : D / 16;   // K steps of S (columns of Q, K / 16)
      auto issue_s = [&](uint32_t d_tmem, uint32_t q_lo, uint32_t k_lo) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          if (kKv && kk >= s_steps) break;
          const uint32_t off = static_cast<uint32_t>((kk >> 2) * L::kChunkBytes + (kk & 3) * 32) >> 4;
          ptx::mma_ss(d_tmem, ptx::desc_sw128(q_lo + off), ptx::desc_sw128(k_lo + off), idesc_s,
                      kk > 0);
        }
      };
      // O_w (+)= P_w V over 128 keys: P from TMEM (two 16-bit values per
      // column, 8 columns per 16 keys); V MN-major (d contiguous): 8-key
      // groups 1024 bytes apart (SBO), 64-column chunks kChunkBytes apart (LBO).
      // P in shared memory: the A operand is a K-major tile laid out like Q
      // (128 keys along K in two 64-column chunks), so its K steps advance as
      // in issue_s.
      auto issue_pv = [&](uint32_t o_tmem, uint32_t p_addr, uint32_t v_lo, uint32_t acc) {
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          if constexpr (OwnP<D>::kSmem) {
            const uint32_t off = static_cast<uint32_t>((kk >> 2) * L::kChunkBytes + (kk & 3) * 32) >> 4;
            ptx::mma_ss(o_tmem, ptx::desc_sw128(p_addr + off),
                        ptx::desc_sw128(v_lo + kk * (2048 >> 4)), idesc_o, kk > 0 ? 1u : acc);
          } else {
            ptx::mma_ts(o_tmem, p_addr + kk * 8, ptx::desc_sw128(v_lo + kk * (2048 >> 4)), idesc_o,
                        kk > 0 ? 1u : acc);
          }
        }
      };

      Prof pf;                         // FA_PROFILE: 0 kv wait, 1 p wait, 2 q wait, 3 o_free wait,
                                       // 4 S issue, 5 PV issue, 6 other, 7 groups issued,
                                       // 16 S-free wait
      uint32_t k_units = 0;            // units walked
      uint32_t ucnt0 = 0, ucnt1 = 0;   // units in which query tile 0 / 1 was active
      uint32_t pph0 = 0, pph1 = 0;     // p_full phase parity of tile 0 / 1
      bool alive = true;
      bool issued_any = false;
      Cursor cu;
      cursor_init<kSplit>(p, cta, grid, cu);
      Piece u;
      // With a P buffer per query tile, S_w_{j+1} waits only until the
      // softmax has read S_w_j, and P_w_j V_j only for P_w_j.
      // P_w: TMEM column address, or the address word of its shared-memory descriptor
      const uint32_t tP0 = OwnP<D>::kSmem ? ptx::desc_lo(sbase + L::kP, 16) : tmem_base + p_col<D>(0);
      const uint32_t tP1 = OwnP<D>::kSmem ? ptx::desc_lo(sbase + L::kP + kBM * kBN * 2, 16)
                                          : tmem_base + p_col<D>(1);
      uint32_t sc0 = 0, sc1 = 0;     // S issued into S0 / S1 so far
      uint32_t q_add = 0;            // address-word offset of the current unit's Q buffer
      auto issue_s_own = [&](int w, uint32_t kslot_) {
        uint32_t& sc = w ? sc1 : sc0;
        pf.lap(6);
        if (sc > 0)   // the softmax has read the previous S of this tile
          alive = ptx::wait_bounded(bar(L::bSFree + w), (sc - 1) & 1, wd, kSiteSFree) && alive;
        pf.lap(16);
        ptx::tc_fence_after();
        if (alive) {
          issue_s(w ? tS1 : tS0, (w ? q_lo1 : q_lo0) + q_add, k_lo0 + kslot_ * kSlotLo);
          ptx::mma_commit(bar(L::bSFull + w));
        }
        ++sc;
        pf.lap(4);
        pf.count(7);
      };
      auto issue_pv_own = [&](int w, int j, uint32_t v_lo) {
        uint32_t& pph = w ? pph1 : pph0;
        const uint32_t ucnt = w ? ucnt1 : ucnt0;
        pf.lap(6);
        if (j == 0 && ucnt > 0)   // O_w of the previous piece must have been read out
          alive = ptx::wait_bounded(bar(L::bOFree + w), (ucnt - 1) & 1, wd, kSiteOFree) && alive;
        pf.lap(3);
        alive = ptx::wait_bounded(bar(L::bPFull + w), pph, wd, kSitePFull) && alive;
        pf.lap(1);
        pph ^= 1u;
        ptx::tc_fence_after();
        if (alive) {
          issue_pv(w ? tO1 : tO0, w ? tP1 : tP0, v_lo, j > 0 ? 1u : 0u);
          ptx::mma_commit(bar(L::bPvDone + w));
        }
        pf.lap(5);
        pf.count(7);
      };
      // The producer fills the ring with K0 K1 V0 K2 V1 ... K_{n-1} V_{n-2}
      // V_{n-1} for a piece of n key tiles: 2n loads from ring position
      // `base`; each issuer waits only for the tiles it reads.
      auto ring_wait = [&](uint32_t pos) -> uint32_t {
        const uint32_t sl = pos % L::kStages;
        pf.lap(6);
        alive = ptx::wait_bounded(bar(L::bKvFull + sl), (pos / L::kStages) & 1, wd, kSiteKvFull) &&
                alive;
        pf.lap(0);
        ptx::tc_fence_after();
        return sl;
      };
      uint32_t base = 0;
      if (warp == kMmaWarp) {
        // S = Q K^T for both query tiles, one key tile ahead of the softmax
        while (next_piece<kCausal, kSplit, kKv>(p, cta, grid, cu, u)) {
          const int nkv = max(u.n0, u.n1);
          if (kKv && nkv == 0) continue;
          pf.lap(6);
          const uint32_t qb = k_units % L::kQBufs;
          alive = ptx::wait_bounded(bar(L::bQFull + qb), (k_units / L::kQBufs) & 1, wd, kSiteQFull) &&
                  alive;
          q_add = qb * static_cast<uint32_t>((2 * L::kTile) >> 4);
          pf.lap(2);
          ptx::tc_fence_after();
          for (int j = 0; j < nkv; ++j) {
            const uint32_t kslot = ring_wait(base + (j == 0 ? 0u : 2u * j - 1u));
            if (j < u.n0) issue_s_own(0, kslot);
            if (j < u.n1) issue_s_own(1, kslot);
            if (alive) {
              ptx::mma_commit(bar(L::bKvEmpty + kslot));
              if (j + 1 == nkv) ptx::mma_commit(bar(L::bQEmpty + qb));  // last use of Q
            }
            issued_any = true;
          }
          base += 2u * nkv;
          ++k_units;
        }
      } else {
        // O += P V for both query tiles, as soon as the softmax has written P
        while (next_piece<kCausal, kSplit, kKv>(p, cta, grid, cu, u)) {
          const int nkv = max(u.n0, u.n1);
          if (kKv && nkv == 0) continue;
          for (int j = 0; j < nkv; ++j) {
            const uint32_t vslot =
                ring_wait(base + (j + 1 < nkv ? 2u * j + 2u : 2u * nkv - 1u));
            const uint32_t v_lo = v_lo0 + vslot * kSlotLo;
            if (j < u.n0) issue_pv_own(0, j, v_lo);
            if (j < u.n1) issue_pv_own(1, j, v_lo);
            if (alive) ptx::mma_commit(bar(L::bKvEmpty + vslot));
            issued_any = true;
          }
          if (u.n0 > 0) ++ucnt0;
          if (u.n1 > 0) ++ucnt1;
          base += 2u * nkv;
        }
      }
      pf.lap(6);
      const bool pv_thread = (warp == kPvWarp);
      pf.flush(p, pv_thread ? 3 : 2);
      // Drain: every MMA issued by this thread has completed before TMEM is freed.
      if (issued_any) {
        const uint32_t fb = bar(pv_thread ? L::bFinalPv : L::bFinal);
        ptx::mma_commit(fb);
        ptx::wait_drain(fb, 0, 200000000ull);
      }
    }
    __syncwarp();
  }
  } else {
    ptx::setmaxnreg_inc<L::kGen ? kSoftmaxRegsDrop : kSoftmaxRegs>();
    // ============================================================ softmax + epilogue
    const int w = warp >> 2;                 // query tile of the unit
    const int t = threadIdx.x & 127;         // row within the tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem_base + lane_off + s_col<D>(w);
    const uint32_t tO = tmem_base + lane_off + o_col<D>(w);
    const uint32_t tP = tmem_base + lane_off + p_col<D>(w);
    const uint32_t stage = sbase + L::kO + w * L::kTile;   // used when kTmaStore
    const float c = p.scale_log2;
    uint32_t scnt = 0, ucnt = 0;
    uint32_t pvcnt = 0;                       // P.V products of this tile waited for
    uint32_t mcnt = 0;                        // dropout masks of this tile consumed
    uint32_t tr = 0;                          // trace events recorded (thread t == 0)
    const bool tracer = (t == 0);
    Prof pf;   // FA_PROFILE: 0 s wait, 1 load S, 2 max + rescale, 3 exp/sum/pack, 4 store P + arrive,
               // 5 o_done wait, 6 epilogue, 7 other, 8 tiles, 9 rescales, 16 P.V-done wait,
               // 18 dropout mask wait, 19 dropout mask load and apply

    Cursor cu;
    cursor_init<kSplit>(p, cta, grid, cu);
    Piece u;
    while (next_piece<kCausal, kSplit, kKv>(p, cta, grid, cu, u)) {
      const int n = w ? u.n1 : u.n0;
      const int tile = 2 * u.mblk + w;
      const int row = tile * kBM + t;
      if (n == 0) {
        if constexpr (kKv) {
          // a query tile that sees no key: O = 0 and LSE = -inf (the policy
          // for an empty key set)
          if (row < u.lenq) {
            uint4* orow = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.o) +
                                                   out_row<kKv>(p, u, row) * (p.dv * 2));
            for (int v = 0; v < p.dv / 8; ++v) orow[v] = make_uint4(0u, 0u, 0u, 0u);
            p.lse[lse_at<kKv>(p, u, row)] = -INFINITY;
          }
        }
        continue;
      }

      float m_ref = -INFINITY;  // reference maximum of the raw scores q.k
      float neg_m = 0.f;        // -m_ref * c (0 while m_ref is -inf)
      float l = 0.f;            // running sum of 2^(s*c + neg_m)
      for (int j = 0; j < n; ++j) {
        pf.lap(7);
        ptx::wait_bounded(bar(L::bSFull + w), scnt & 1, wd, kSiteSFull);
        pf.lap(0);
        pf.count(8);
        ++scnt;
        if (tracer) trace_event(p, w, tr, kEvSReady, j);
        __syncwarp();
        ptx::tc_fence_after();
        uint32_t sr[kBN];
#pragma unroll
        for (int q4 = 0; q4 < kBN / 32; ++q4) ptx::tmem_ld32(tS + q4 * 32, sr + q4 * 32);
        ptx::tmem_wait_ld();
        float sv[kBN];
#pragma unroll
        for (int i = 0; i < kBN; ++i) sv[i] = __uint_as_float(sr[i]);
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(L::bSFree + w));     // S_w may be overwritten now
        pf.lap(1);

        // mask: keys past N, and on the diagonal tile keys after this row
        const int kj = u.kb + j;                 // key tile index
        if constexpr (kKv) {
          // keys past this batch's count, and keys after this row's position
          int lim = min(kBN, u.len - kj * kBN);
          if (kCausal) lim = min(lim, row + u.off - kj * kBN + 1);
          if (lim < kBN) {
#pragma unroll
            for (int i = 0; i < kBN; ++i)
              if (i >= lim) sv[i] = -INFINITY;
          }
        } else {
          const int rem = p.N - kj * kBN;
          const bool diag = kCausal && kj == tile;
          if (diag || rem < kBN) {
            int lim = rem < kBN ? rem : kBN;
            if (diag) lim = min(lim, t + 1);
#pragma unroll
            for (int i = 0; i < kBN; ++i)
              if (i >= lim) sv[i] = -INFINITY;
          }
        }

        // row maximum.  At d = 64 (the softmax bounds the key step) a tree:
        // sixteen chains of three three-input maxima, then two levels; at
        // d = 128 four chains of sixteen (measured faster there).
        float mx;
        if constexpr (D == 64) {
          static_assert(kBN == 128, "the tree covers 16 x 8 keys");
          float a[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) a[c] = ptx::max3(sv[8 * c], sv[8 * c + 1], sv[8 * c + 2]);
#pragma unroll
          for (int c = 0; c < 16; ++c) a[c] = ptx::max3(a[c], sv[8 * c + 3], sv[8 * c + 4]);
#pragma unroll
          for (int c = 0; c < 16; ++c)
            a[c] = ptx::max3(a[c], sv[8 * c + 5], fmaxf(sv[8 * c + 6], sv[8 * c + 7]));
          const float b0 = ptx::max3(a[0], a[1], a[2]), b1 = ptx::max3(a[3], a[4], a[5]);
          const float b2 = ptx::max3(a[6], a[7], a[8]), b3 = ptx::max3(a[9], a[10], a[11]);
          const float b4 = ptx::max3(a[12], a[13], a[14]);
          mx = fmaxf(ptx::max3(b0, b1, b2), ptx::max3(b3, b4, a[15]));
        } else {
          float a0 = -INFINITY, a1 = -INFINITY, a2 = -INFINITY, a3 = -INFINITY;
#pragma unroll
          for (int i = 0; i < kBN; i += 8) {
            a0 = ptx::max3(a0, sv[i + 0], sv[i + 1]);
            a1 = ptx::max3(a1, sv[i + 2], sv[i + 3]);
            a2 = ptx::max3(a2, sv[i + 4], sv[i + 5]);
            a3 = ptx::max3(a3, sv[i + 6], sv[i + 7]);
          }
          mx = fmaxf(fmaxf(a0, a1), fmaxf(a2, a3));
        }

        // lazy rescale: move the reference only when the tile max exceeds it
        // by more than kTau (always on the first finite tile; never for -inf)
        const bool grow = (mx - m_ref) * c > kTau;
        float alpha = 1.f;
        if (grow) {
          const float nm = -mx * c;
          alpha = (m_ref == -INFINITY) ? 0.f : ptx::ex2(nm - neg_m);
          l *= alpha;
          m_ref = mx;
          neg_m = nm;
        }
        const bool rescale = j > 0 && __any_sync(0xffffffffu, grow);
        // O_w *= alpha.  PV_w_{j-1} must be complete (waited for below) and
        // PV_w_j cannot start before this warpgroup arrives on p_full.
        auto rescale_o = [&]() {
          if (tracer) trace_event(p, w, tr, kEvRescale, j);
          pf.count(9);
#pragma unroll 1
          for (int q4 = 0; q4 < D / 32; ++q4) {
            uint32_t orr[32];
            ptx::tmem_ld32(tO + q4 * 32, orr);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) orr[i] = __float_as_uint(__uint_as_float(orr[i]) * alpha);
            ptx::tmem_st32(tO + q4 * 32, orr);
          }
        };

        // P_w and O_w are still in use by PV_w_{j-1} until it completes
        // (the wait of the early stores below).
        auto wait_pv = [&]() {
          if (j > 0) {
            pf.lap(3);
            ptx::wait_bounded(bar(L::bPvDone + w), pvcnt & 1, wd, kSitePvDone);
            ++pvcnt;
            pf.lap(16);
            __syncwarp();
            ptx::tc_fence_after();
          }
        };
        // Without dropout (no mask to apply after the exponentials) the
        // first half of P is stored as soon as it is packed, once
        // PV_w_{j-1} has completed, so the store overlaps the second half's
        // exponentials: into TMEM at d = 64; into shared memory (the first
        // 64-key chunk) at d = 128 for unmasked calls (measured slower on
        // the causal workload, which runs power-capped).
        constexpr bool kEarlyP = !kDrop && OwnP<D>::kTmem;
        constexpr bool kEarlyS = !kDrop && OwnP<D>::kSmem && !kCausal;

        pf.lap(2);
        // P = 2^(s*c - m_ref*c), summed into l, packed to 16 bits into TMEM.
        // The exponent argument and the row sum use two-lane fp32 instructions.
        const uint64_t c2 = ptx::f2_pack(c, c);
        const uint64_t nm2 = ptx::f2_pack(neg_m, neg_m);
        uint64_t acc0 = ptx::f2_pack(0.f, 0.f), acc1 = acc0;
        uint32_t pk[kBN / 2];
#pragma unroll
        for (int i = 0; i < kBN / 2; i += 2) {
          if constexpr (kEarlyS) {
            if (i == kBN / 4) {   // keys 0 .. 63 (chunk 0) are packed
              wait_pv();
              if (rescale) rescale_o();
              uint8_t* prow0 = sgen + L::kP + w * (kBM * kBN * 2) + t * 128;
#pragma unroll
              for (int k = 0; k < 8; ++k)
                *reinterpret_cast<uint4*>(prow0 + (((k & 7) ^ (t & 7)) << 4)) =
                    make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
            }
          }
          if constexpr (kEarlyP) {
            if (i == kBN / 4) {   // pk[0 .. 31] are packed
              wait_pv();
              if (rescale) rescale_o();
              ptx::tmem_st32(tP, pk);
            }
          }
          float x0, x1, x2, x3;
          ptx::f2_unpack(ptx::ffma2(ptx::f2_pack(sv[2 * i + 0], sv[2 * i + 1]), c2, nm2), x0, x1);
          ptx::f2_unpack(ptx::ffma2(ptx::f2_pack(sv[2 * i + 2], sv[2 * i + 3]), c2, nm2), x2, x3);
          const float p0 = ptx::ex2(x0), p1 = ptx::ex2(x1), p2 = ptx::ex2(x2), p3 = ptx::ex2(x3);
          acc0 = ptx::fadd2(acc0, ptx::f2_pack(p0, p1));
          acc1 = ptx::fadd2(acc1, ptx::f2_pack(p2, p3));
          pk[i] = ptx::pack2<kBf16>(p0, p1);
          pk[i + 1] = ptx::pack2<kBf16>(p2, p3);
        }
        {
          float a, b, cc, dd;
          ptx::f2_unpack(acc0, a, b);
          ptx::f2_unpack(acc1, cc, dd);
          l += (a + b) + (cc + dd);
        }
        if constexpr (kDrop) {
          // dropout: the weights of dropped keys leave P (l keeps them: the
          // normalisation is the softmax's); 256 / t is applied with 1 / l.
          pf.lap(3);
          if constexpr (L::kGen) {
            // the keep bits of this tile come from the generator's ring
            const int bi = w * L::kMaskStages + static_cast<int>(mcnt % L::kMaskStages);
            ptx::wait_bounded(bar(L::bMaskFull + bi), (mcnt / L::kMaskStages) & 1, wd,
                              kSiteMaskFull);
            pf.lap(18);
            ++mcnt;
            const uint8_t* mrow = sgen + L::kMask + bi * L::kMaskBytes + (t >> 2) * 16;
            uint4 yq[4];
#pragma unroll
            for (int k2 = 0; k2 < 4; ++k2)
              yq[k2] = *reinterpret_cast<const uint4*>(mrow + k2 * 512);
            ptx::mbar_arrive(bar(L::bMaskEmpty + bi));   // the buffer may be refilled
            drop_apply(pk, yq, static_cast<uint32_t>(t & 3));
          } else {
            drop_row128(pk, static_cast<uint32_t>(row), static_cast<uint32_t>(kj * kBN), u.bh,
                        p.drop_off, p.drop_k0, p.drop_k1, p.drop_t);
          }
          pf.lap(19);
        }
        pf.lap(3);
        if constexpr (!kEarlyP && !kEarlyS) {
          // P_w and O_w are still in use by PV_w_{j-1} until it completes.
          if (j > 0) {
            pf.lap(3);
            ptx::wait_bounded(bar(L::bPvDone + w), pvcnt & 1, wd, kSitePvDone);
            ++pvcnt;
            pf.lap(16);
            __syncwarp();
            ptx::tc_fence_after();
          }
          if (rescale) rescale_o();
        }
        if constexpr (OwnP<D>::kSmem) {
          // row t of the P_w tile: 16 pieces of 8 keys, 128-byte swizzle
          uint8_t* prow = sgen + L::kP + w * (kBM * kBN * 2) + t * 128;
#pragma unroll
          for (int k = kEarlyS ? 8 : 0; k < kBN / 8; ++k)
            *reinterpret_cast<uint4*>(prow + (k >> 3) * L::kChunkBytes + (((k & 7) ^ (t & 7)) << 4)) =
                make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
          ptx::fence_proxy_async_smem();   // visible to the tensor core's reads
        } else {
          if constexpr (!kEarlyP) ptx::tmem_st32(tP, pk);
          ptx::tmem_st32(tP + 32, pk + 32);
        }
        ptx::tmem_wait_st();               // P (in TMEM) and a rescaled O are written
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(L::bPFull + w));
        pf.lap(4);
        if (tracer) trace_event(p, w, tr, kEvPArrive, j);
      }

      // ---- epilogue: O / l in the storage dtype, and LSE = m + ln l per row
      pf.lap(7);
      ptx::wait_bounded(bar(L::bPvDone + w), pvcnt & 1, wd, kSitePvDone);   // last PV_w
      ++pvcnt;
      pf.lap(5);
      ++ucnt;
      if (tracer) trace_event(p, w, tr, kEvEpiStart, ucnt - 1);
      __syncwarp();
      ptx::tc_fence_after();
      // a row that saw no key (kKv masks) keeps l = 0: O = 0, LSE = -inf
      const float inv_l = (l > 0.f ? 1.0f / l : 0.f) * (kDrop ? p.drop_scale : 1.f);
      if (kSplit && u.tail >= 0) {
        // Partial piece of a split unit: unnormalised O rows and (-m*c, l)
        // go to this piece's workspace slot; the piece that finishes last
        // (counted per tail unit and query tile) merges all of them with
        // the combining identity: with m* the largest m, each piece is
        // scaled by 2^((m_p - m*) c), l = sum of scaled l_p, O = sum of
        // scaled O_p / l, LSE = m* + ln l.
        pf.lap(6);
        float* slot = p.ws_part + static_cast<size_t>(u.slot) * kSlotFloats<D>();
        float* so = slot + static_cast<size_t>(w) * D * kBM + t;
#pragma unroll 1
        for (int q4 = 0; q4 < D / 32; ++q4) {
          uint32_t orr[32];
          ptx::tmem_ld32(tO + q4 * 32, orr);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) so[(q4 * 32 + e) * kBM] = __uint_as_float(orr[e]);
        }
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(L::bOFree + w));        // O_w may be overwritten now
        reinterpret_cast<float2*>(slot + 2 * kBM * D)[w * kBM + t] = make_float2(neg_m, l);
        pf.lap(10);
        __threadfence();
        pf.lap(11);
        ptx::named_bar_sync(1 + w, 128);
        const long long ua = static_cast<long long>(u.tail) * p.n_kv, ub = ua + p.n_kv;
        int npieces = 0;
        {
          TailWalk tw;
          tw.init(p, grid, u.tail);
          for (; tw.c < grid && tw.st < ub; tw.step()) {
            const long long en = tw.next_start();
            if (tw.st < en && en > ua) ++npieces;
          }
        }
        if (t == 0) {
          const int done = atomicAdd(p.ws_count + 2 * u.tail + w, 1);
          merge_flag[w] = (done == npieces - 1) ? 1 : 0;
        }
        ptx::named_bar_sync(1 + w, 128);
        pf.lap(12);
        if (merge_flag[w]) {
          __threadfence();
          pf.count(14);
          // One pass over the pieces with the online rescale: a running
          // reference nm_run = -m*c, running l and an O row accumulator.
          float nm_run = INFINITY, l_run = 0.f;
          float acc[D];
#pragma unroll
          for (int e = 0; e < D; ++e) acc[e] = 0.f;
          TailWalk tw;
          tw.init(p, grid, u.tail);
          for (; tw.c < grid && tw.st < ub; tw.step()) {
            const long long en = tw.next_start();
            if (!(tw.st < en && en > ua)) continue;          // no piece of this unit
            const int first_t = static_cast<int>(tw.st / p.n_kv);
            const float* sp = p.ws_part +
                              static_cast<size_t>(2 * tw.c + (u.tail == first_t ? 0 : 1)) * kSlotFloats<D>();
            const float2 ml = reinterpret_cast<const float2*>(sp + 2 * kBM * D)[w * kBM + t];
            if (!(ml.y > 0.f)) continue;
            float f = 1.f;
            if (ml.x < nm_run) {                              // larger maximum: move the reference
              const float a = (nm_run == INFINITY) ? 0.f : ptx::ex2(ml.x - nm_run);
#pragma unroll
              for (int e = 0; e < D; ++e) acc[e] *= a;
              l_run *= a;
              nm_run = ml.x;
            } else {
              f = ptx::ex2(nm_run - ml.x);
            }
            l_run += f * ml.y;
            const float* src = sp + static_cast<size_t>(w) * D * kBM + t;
#pragma unroll
            for (int e = 0; e < D; ++e) acc[e] += f * src[e * kBM];
          }
          const float inv_lt = 1.0f / l_run;
          if (row < p.N) {
            uint4* orow = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.o) +
                                                   (static_cast<size_t>(u.bh) * p.N + row) * (D * 2));
#pragma unroll
            for (int v = 0; v < D / 8; ++v)
              orow[v] = make_uint4(ptx::pack2<kBf16>(acc[8 * v] * inv_lt, acc[8 * v + 1] * inv_lt),
                                   ptx::pack2<kBf16>(acc[8 * v + 2] * inv_lt, acc[8 * v + 3] * inv_lt),
                                   ptx::pack2<kBf16>(acc[8 * v + 4] * inv_lt, acc[8 * v + 5] * inv_lt),
                                   ptx::pack2<kBf16>(acc[8 * v + 6] * inv_lt, acc[8 * v + 7] * inv_lt));
            p.lse[static_cast<size_t>(u.bh) * p.N + row] = (ptx::lg2(l_run) - nm_run) * kLn2;
          }
          if (t == 0) p.ws_count[2 * u.tail + w] = 0;   // ready for the next call
          pf.lap(13);
        }
        pf.count(15);
      } else if (L::kTmaStore && !(kKv && p.varlen)) {
        // through a swizzled staging tile and a TMA store (rows past N
        // clipped; packed batches, whose tiles end mid-tensor, store directly)
        if (t == 0) ptx::bulk_wait_group_read0();   // staging tile free again
        ptx::named_bar_sync(1 + w, 128);
#pragma unroll 1
        for (int q4 = 0; q4 < D / 32; ++q4) {
          uint32_t orr[32];
          ptx::tmem_ld32(tO + q4 * 32, orr);
          ptx::tmem_wait_ld();
          const int chunk = q4 >> 1;
#pragma unroll
          for (int pc4 = 0; pc4 < 4; ++pc4) {
            const int pc = (q4 & 1) * 4 + pc4;   // 16-byte piece within the 128-byte row
            uint32_t v4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              v4[e] = ptx::pack2<kBf16>(__uint_as_float(orr[pc4 * 8 + 2 * e]) * inv_l,
                                        __uint_as_float(orr[pc4 * 8 + 2 * e + 1]) * inv_l);
            const uint32_t addr =
                stage + chunk * L::kChunkBytes + t * 128 + ((pc ^ (t & 7)) << 4);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v4[0]),
                         "r"(v4[1]), "r"(v4[2]), "r"(v4[3])
                         : "memory");
          }
        }
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(L::bOFree + w));        // O_w may be overwritten now
        ptx::fence_proxy_async_smem();
        ptx::named_bar_sync(1 + w, 128);
        if (t == 0) {
          for (int ch = 0; ch < L::kChunks; ++ch)
            ptx::tma_store_3d(&p.tm_o, stage + ch * L::kChunkBytes, ch * 64, tile * kBM, u.bh);
          ptx::bulk_commit_group();
        }
      } else {
        // straight from registers: each thread writes its own row (of dv
        // columns in the kKv variants)
        const int ocols = kKv ? p.dv : D;
        uint4* orow = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.o) +
                                               out_row<kKv>(p, u, row) * (ocols * 2));
        const int nrows = kKv ? u.lenq : p.N;
#pragma unroll 1
        for (int q4 = 0; q4 < ocols / 32; ++q4) {
          uint32_t orr[32];
          ptx::tmem_ld32(tO + q4 * 32, orr);
          ptx::tmem_wait_ld();
          const uint64_t il2 = ptx::f2_pack(inv_l, inv_l);
          uint32_t pk16[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float a, b;
            ptx::f2_unpack(ptx::fmul2(ptx::f2_pack(__uint_as_float(orr[2 * e]),
                                                   __uint_as_float(orr[2 * e + 1])), il2), a, b);
            pk16[e] = ptx::pack2<kBf16>(a, b);
          }
          if (row < nrows) {
#pragma unroll
            for (int v = 0; v < 4; ++v)
              orow[q4 * 4 + v] = make_uint4(pk16[4 * v], pk16[4 * v + 1], pk16[4 * v + 2],
                                            pk16[4 * v + 3]);
          }
        }
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(L::bOFree + w));        // O_w may be overwritten now
      }
      if ((!kSplit || u.tail < 0) && row < (kKv ? u.lenq : p.N))
        p.lse[lse_at<kKv>(p, u, row)] = l > 0.f ? (ptx::lg2(l) - neg_m) * kLn2 : -INFINITY;
      if (tracer) trace_event(p, w, tr, kEvEpiEnd, ucnt - 1);
      pf.lap(6);
    }
    pf.lap(7);
    if (tracer) pf.flush(p, w);
    if constexpr (L::kTmaStore) {
      if (t == 0) ptx::bulk_wait_group0();
    }
  }

  // ---------------------------------------------------------------- teardown
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace fa
