// fa_fwd_api.cu — the forward entry points of the C ABI declared in
// include/fa.h: argument checks, TMA descriptors, the unit order and the
// launch of the forward kernels (square, balanced, kv, packed, dropout).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <vector>

#include "fa.h"
#include "fa_host.cuh"
#include "fa_launch.cuh"

using namespace fa::host;

namespace {

// ---------------------------------------------------------------- unit order
// The kernels deal (batch*head, 256-row query block) units to the CTAs in a
// snake order over groups of `hgroup` heads (level by level inside a group).
// Small groups keep the units in flight on few heads, whose K/V tiles the
// CTAs then share in L2 (measured: head by head is best for the long causal
// and prefill workloads, 10-15 % over larger groups); larger groups balance
// causal work better when there are few heads (B1 H8 N32768: level order 29 %
// faster than head by head).  So the group is capped by an L2 budget, and
// for causal calls of known lengths the host simulates the deal of each
// group size and takes the smallest one within 1 % of the most even deal.
// Results do not depend on the choice.

std::atomic<int> g_unit_group{0};   // fa_set_unit_group override (0 = automatic)

constexpr long long kL2GroupBudget = 64ll << 20;   // K/V bytes of the heads of one group

int group_cap(long long bh, long long kv_head_bytes) {
  if (kv_head_bytes <= 0) return static_cast<int>(bh);
  const long long g = kL2GroupBudget / kv_head_bytes;
  return static_cast<int>(g < 1 ? 1 : (g > bh ? bh : g));
}

// Mean over largest CTA load of the snake deal with group size g, every head
// alike: a unit costs its key tiles (both query tiles) plus 2 for its fixed
// work; `cost[m]` is that cost for query block m.
double deal_balance(int g, int BH, int n_qblk, int grid, const std::vector<double>& cost,
                    std::vector<double>& load) {
  load.assign(grid, 0.0);
  const int per_group = g * n_qblk;
  const long long units = static_cast<long long>(BH) * n_qblk;
  for (long long s = 0; s < units; ++s) {
    const long long grp = s / per_group;
    const long long r = s - grp * per_group;
    const long long gl = std::min<long long>(g, BH - grp * g);
    const int mblk = n_qblk - 1 - static_cast<int>(r / gl);
    const long long round = s / grid, c = s - round * grid;
    load[(round & 1) ? grid - 1 - c : c] += cost[mblk];
  }
  double mx = 0.0, sum = 0.0;
  for (double x : load) { mx = std::max(mx, x); sum += x; }
  return mx > 0.0 ? sum / grid / mx : 1.0;
}

struct GroupKey {
  long long bh;
  int n_qblk, Nq, Nk, off, causal, grid, cap;
  bool operator==(const GroupKey& o) const {
    return bh == o.bh && n_qblk == o.n_qblk && Nq == o.Nq && Nk == o.Nk && off == o.off &&
           causal == o.causal && grid == o.grid && cap == o.cap;
  }
};

// Group size for heads of equal shape: Nq queries (query i at position
// i + off) against Nk keys each.
int choose_group(long long bh, int n_qblk, int Nq, int Nk, int off, bool causal, int grid,
                 long long kv_head_bytes) {
  const int forced = g_unit_group.load();
  if (forced > 0) return static_cast<int>(std::min<long long>(forced, bh));
  const int cap = group_cap(bh, kv_head_bytes);
  const long long units = bh * n_qblk;
  // Without a mask every unit costs the same (only the last block may be
  // short) and any order deals the same loads: level order while all K/V
  // are small, else head by head for L2 reuse.
  if (!causal) return bh * kv_head_bytes <= (32ll << 20) ? static_cast<int>(bh) : 1;
  // Past ~64K units the deal is even anyway, and simulating it would cost
  // milliseconds.
  if (cap == 1 || units <= grid || units > (1 << 16)) return cap;

  static std::mutex mu;
  static GroupKey keys[32];
  static int vals[32];
  static int used = 0, next = 0;
  const GroupKey key{bh, n_qblk, Nq, Nk, off, causal ? 1 : 0, grid, cap};
  {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
      if (keys[i] == key) return vals[i];
  }
  std::vector<double> cost(n_qblk), load;
  const int nkv = (Nk + fa::kBN - 1) / fa::kBN;
  for (int m = 0; m < n_qblk; ++m) {
    int c = 0;
    for (int w = 0; w < 2; ++w) {
      const int first = (2 * m + w) * fa::kBM;
      if (first >= Nq) continue;
      const int last = std::min(first + fa::kBM, Nq) - 1 + off;
      c += last < 0 ? 0 : std::min(last / fa::kBN + 1, nkv);
    }
    cost[m] = c > 0 ? c + 2.0 : 0.1;
  }
  const int top = cap < 32 ? cap : 32;
  std::vector<double> bal(top + 1, 0.0);
  double best_bal = 0.0;
  for (int g = 1; g <= top; ++g) {
    bal[g] = deal_balance(g, static_cast<int>(bh), n_qblk, grid, cost, load);
    best_bal = std::max(best_bal, bal[g]);
  }
  int best = 1;
  while (bal[best] < best_bal - 0.01) ++best;   // the smallest group within 1 %
  std::lock_guard<std::mutex> lock(mu);
  keys[next] = key;
  vals[next] = best;
  next = (next + 1) % 32;
  if (used < 32) ++used;
  return best;
}

// Heads of different lengths (per-batch key counts or packed sequences that
// only the device knows): without a mask as choose_group; with one, groups
// of whole batches (the H heads of a sequence share a shape, so a group's
// levels cost alike) as far as the L2 budget allows (measured on a packed
// batch of 16 causal sequences of 618-3993 tokens: 2 sequences per group
// 21 % faster than head by head).
int choose_group_ragged(long long bh, int H, long long kv_head_bytes, bool causal) {
  const int forced = g_unit_group.load();
  if (forced > 0) return static_cast<int>(std::min<long long>(forced, bh));
  if (!causal) return bh * kv_head_bytes <= (32ll << 20) ? static_cast<int>(bh) : 1;
  const int cap = group_cap(bh, kv_head_bytes);
  if (cap >= H) return (cap / H) * H;
  for (int g = cap; g > 1; --g)
    if (H % g == 0) return g;   // a divisor of H: groups never straddle two batches
  return 1;
}

}  // namespace

extern "C" {

int fa_set_unit_group(int heads) {
  if (heads < 0) return FA_ERR_SHAPE;
  g_unit_group.store(heads);
  return FA_OK;
}

}  // extern "C"

namespace {

// Size of one split schedule: units, persistent grid, tail.
struct SplitPlan {
  long long units = 0;
  int grid = 0;
  int full_rounds = 0;
  int tail_units = 0;
  bool split = false;
  size_t counter_bytes = 0;   // 2 * tail_units ints, rounded up to 256 bytes
  size_t slot_bytes = 0;      // one workspace slot
  size_t bytes = 0;           // whole workspace (0 when the tail is not split)
};

// The tail is split when the call is unmasked, the units do not fill whole
// rounds of the persistent grid, and there is more than one key tile to
// split.  `sms` is the device's SM count.
SplitPlan plan_split(long long bh, int N, int d, int causal, int sms) {
  SplitPlan sp;
  const long long n_qblk = (static_cast<long long>(N) + 2 * fa::kBM - 1) / (2 * fa::kBM);
  const int n_kv = (N + fa::kBN - 1) / fa::kBN;
  sp.units = bh * n_qblk;
  sp.grid = static_cast<int>(sp.units < sms ? sp.units : sms);
  if (sp.grid <= 0) return sp;
  sp.full_rounds = static_cast<int>(sp.units / sp.grid);
  sp.tail_units = static_cast<int>(sp.units - static_cast<long long>(sp.full_rounds) * sp.grid);
  sp.split = !causal && sp.tail_units > 0 && n_kv >= 2;
  if (sp.split) {
    sp.counter_bytes = ((2 * static_cast<size_t>(sp.tail_units) * sizeof(int)) + 255) / 256 * 256;
    const int slot_floats = (d == 64) ? fa::kSlotFloats<64>() : fa::kSlotFloats<128>();
    sp.slot_bytes = static_cast<size_t>(slot_floats) * sizeof(float);
    sp.bytes = sp.counter_bytes + 2 * static_cast<size_t>(sp.grid) * sp.slot_bytes;
  }
  return sp;
}

}  // namespace

namespace fa {
namespace host {

int check_forward_args(const void* q, const void* k, const void* v, const void* o,
                       const float* lse, int B, int H, int N, int d, float scale, int dtype,
                       bool* empty) {
  *empty = false;
  if (B < 0 || H < 0 || N < 0 || d <= 0) return FA_ERR_SHAPE;
  const long long bh = static_cast<long long>(B) * H;
  const long long n_qblk = (static_cast<long long>(N) + 2 * fa::kBM - 1) / (2 * fa::kBM);
  if (bh > INT_MAX || bh * n_qblk > INT_MAX) return FA_ERR_SHAPE;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED_D;
  if (dtype != FA_BF16 && dtype != FA_FP16) return FA_ERR_DTYPE;
  if (!std::isfinite(scale) || !(scale > 0.0f)) return FA_ERR_SCALE;
  if (bh == 0 || N == 0) {  // nothing to write
    *empty = true;
    return FA_OK;
  }
  if (!q || !k || !v || !o || !lse) return FA_ERR_NULLPTR;
  const uintptr_t a16 = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                        reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o);
  if ((a16 & 15u) || (reinterpret_cast<uintptr_t>(lse) & 3u)) return FA_ERR_ALIGN;
  return FA_OK;
}

}  // namespace host
}  // namespace fa

namespace {

// Shared by fa_fwd (no workspace) and fa_fwd_ws.
int launch_forward(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                   int N, int d, int causal, float scale, int dtype, void* workspace,
                   size_t workspace_bytes, cudaStream_t stream) {
  bool empty = false;
  const int arg_rc = check_forward_args(q, k, v, o, lse, B, H, N, d, scale, dtype, &empty);
  if (arg_rc != FA_OK || empty) return arg_rc;
  const long long bh = static_cast<long long>(B) * H;
  const long long n_qblk = (static_cast<long long>(N) + 2 * fa::kBM - 1) / (2 * fa::kBM);

  int dev = 0;
  const DeviceInfo* info = device_info(&dev);
  if (!info || !info->supported) return FA_ERR_DEVICE;
  if (info->err != FA_OK) return info->err;

  SplitPlan sp = plan_split(bh, N, d, causal, info->sms);
  if (workspace != nullptr && sp.split) {
    if (workspace_bytes < sp.bytes) return FA_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return FA_ERR_ALIGN;
  } else {
    sp.split = false;   // no workspace (fa_fwd), or nothing to split
  }

  const bool bf16 = dtype == FA_BF16;
  fa::FwdParams p;
  if (!make_tmap(&p.tm_q, q, static_cast<int>(bh), N, d, bf16) ||
      !make_tmap(&p.tm_k, k, static_cast<int>(bh), N, d, bf16) ||
      !make_tmap(&p.tm_v, v, static_cast<int>(bh), N, d, bf16) ||
      !make_tmap(&p.tm_o, o, static_cast<int>(bh), N, d, bf16))
    return FA_ERR_TENSORMAP;
  p.o = o;
  p.lse = lse;
  p.trace = g_trace.load();
  p.status = info->status;
  // The kernels count the budget in SM cycles; converting at the highest SM
  // clock of the part (2.1 GHz) makes the real-time budget at least the one
  // asked for, whatever clock the GPU runs at.
  const unsigned long long wd = g_watchdog_ns.load();
  p.watchdog_cycles = (wd ? wd : kDefaultWatchdogNs) * 21ull / 10ull;
  p.BH = static_cast<int>(bh);
  p.N = N;
  p.n_qblk = static_cast<int>(n_qblk);
  p.n_kv = (N + fa::kBN - 1) / fa::kBN;
  p.num_units = static_cast<int>(bh * n_qblk);
  // Head-by-head unit order when the K and V of all heads would take more
  // than half of L2 (so concurrent units re-read K/V from L2, not HBM).
  p.hgroup = choose_group(bh, static_cast<int>(n_qblk), N, N, 0, causal != 0, sp.grid,
                          2ll * N * d * 2ll);
  p.scale_log2 = scale * 1.4426950408889634f;
  p.split = sp.split ? 1 : 0;
  p.full_rounds = sp.full_rounds;
  p.tail_units = sp.split ? sp.tail_units : 0;
  p.Nk = N;
  p.H = H;
  p.seqlens_k = nullptr;
  p.align_br = 0;
  p.dqk = d;
  p.dv = d;
  set_dropout(&p, 256, 0, 0);
  p.cu_q = nullptr;
  p.cu_k = nullptr;
  p.varlen = 0;
  p.total_q = 0;
  p.ws_count = sp.split ? static_cast<int*>(workspace) : nullptr;
  p.ws_part = sp.split ? reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + sp.counter_bytes)
                       : nullptr;
  if (sp.split && cudaMemsetAsync(workspace, 0, sp.counter_bytes, stream) != cudaSuccess)
    return FA_ERR_LAUNCH;

  const cudaError_t e = (d == 64) ? fa::launch_fwd_d64(p, sp.grid, bf16, causal != 0, stream)
                                  : fa::launch_fwd_d128(p, sp.grid, bf16, causal != 0, stream);
  return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

}  // namespace

extern "C" {

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
           int d, int causal, float scale, int dtype, cudaStream_t stream) {
  return launch_forward(q, k, v, o, lse, B, H, N, d, causal, scale, dtype, nullptr, 0, stream);
}

int fa_fwd_workspace_size(int B, int H, int N, int d, int causal, size_t* bytes) {
  if (!bytes) return FA_ERR_NULLPTR;
  if (B < 0 || H < 0 || N < 0 || d <= 0) return FA_ERR_SHAPE;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED_D;
  *bytes = 0;
  const long long bh = static_cast<long long>(B) * H;
  if (bh == 0 || N == 0) return FA_OK;
  int dev = 0;
  const DeviceInfo* info = device_info(&dev);
  if (!info || !info->supported) return FA_ERR_DEVICE;
  *bytes = plan_split(bh, N, d, causal, info->sms).bytes;
  return FA_OK;
}

int fa_fwd_ws(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
              int d, int causal, float scale, int dtype, void* workspace, size_t workspace_bytes,
              cudaStream_t stream) {
  return launch_forward(q, k, v, o, lse, B, H, N, d, causal, scale, dtype, workspace,
                        workspace_bytes, stream);
}

// fa_fwd_kv, and fa_fwd_dropout when drop_t < 256 (square shapes, no key
// counts; the caller checks that).
static int forward_kv(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                      int H, int Nq, int Nk, int d, int dv, int causal, const int* seqlens_k,
                      float scale, int dtype, int drop_t, unsigned long long seed,
                      unsigned int drop_off, cudaStream_t stream) {
  if (B < 0 || H < 0 || Nq < 0 || Nk < 0 || d <= 0 || dv <= 0) return FA_ERR_SHAPE;
  if (causal < 0 || causal > 2) return FA_ERR_SHAPE;
  const long long bh = static_cast<long long>(B) * H;
  const long long n_qblk = (static_cast<long long>(Nq) + 2 * fa::kBM - 1) / (2 * fa::kBM);
  if (bh > INT_MAX || bh * n_qblk > INT_MAX) return FA_ERR_SHAPE;
  if ((d != 64 && d != 128) || (dv != 64 && dv != 128)) return FA_ERR_UNSUPPORTED_D;
  if (dtype != FA_BF16 && dtype != FA_FP16) return FA_ERR_DTYPE;
  if (!std::isfinite(scale) || !(scale > 0.0f)) return FA_ERR_SCALE;
  if (bh == 0 || Nq == 0) return FA_OK;  // nothing to write
  if (!q || !o || !lse || (Nk > 0 && (!k || !v))) return FA_ERR_NULLPTR;
  const uintptr_t a16 = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                        reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o);
  const uintptr_t a4 = reinterpret_cast<uintptr_t>(lse) | reinterpret_cast<uintptr_t>(seqlens_k);
  if ((a16 & 15u) || (a4 & 3u)) return FA_ERR_ALIGN;

  int dev = 0;
  const DeviceInfo* info = device_info(&dev);
  if (!info || !info->supported) return FA_ERR_DEVICE;
  if (info->err != FA_OK) return info->err;

  const bool bf16 = dtype == FA_BF16;
  fa::FwdParams p;
  // With no keys no key tile is ever loaded; the maps still need a row and
  // an address (k, v may then be NULL: q stands in).
  const int nk_rows = Nk > 0 ? Nk : 1;
  const void* kp = Nk > 0 ? k : q;
  const void* vp = Nk > 0 ? v : q;
  // Each map has its tensor's own width: with d != dv the kernel of width
  // max(d, dv) loads only the narrower tensors' own columns.
  if (!make_tmap(&p.tm_q, q, static_cast<int>(bh), Nq, d, bf16) ||
      !make_tmap(&p.tm_k, kp, static_cast<int>(bh), nk_rows, d, bf16) ||
      !make_tmap(&p.tm_v, vp, static_cast<int>(bh), nk_rows, dv, bf16) ||
      !make_tmap(&p.tm_o, o, static_cast<int>(bh), Nq, dv, bf16))
    return FA_ERR_TENSORMAP;
  p.o = o;
  p.lse = lse;
  p.trace = g_trace.load();
  p.status = info->status;
  const unsigned long long wd = g_watchdog_ns.load();
  p.watchdog_cycles = (wd ? wd : kDefaultWatchdogNs) * 21ull / 10ull;
  p.BH = static_cast<int>(bh);
  p.N = Nq;
  p.n_qblk = static_cast<int>(n_qblk);
  p.n_kv = (Nk + fa::kBN - 1) / fa::kBN;
  p.num_units = static_cast<int>(bh * n_qblk);
  const int grid = p.num_units < info->sms ? p.num_units : info->sms;
  const long long kv_head = static_cast<long long>(Nk) * (d + dv) * 2ll;
  p.hgroup = seqlens_k ? choose_group_ragged(bh, H, kv_head, causal != 0)
                       : choose_group(bh, static_cast<int>(n_qblk), Nq, Nk,
                                      causal == 2 ? Nk - Nq : 0, causal != 0, grid, kv_head);
  p.scale_log2 = scale * 1.4426950408889634f;
  p.split = 0;
  p.full_rounds = 0;
  p.tail_units = 0;
  p.ws_count = nullptr;
  p.ws_part = nullptr;
  p.Nk = Nk;
  p.H = H;
  p.seqlens_k = seqlens_k;
  p.align_br = causal == 2 ? 1 : 0;
  p.dqk = d;
  p.dv = dv;
  p.cu_q = nullptr;
  p.cu_k = nullptr;
  p.varlen = 0;
  p.total_q = 0;
  set_dropout(&p, drop_t, seed, drop_off);
  const bool w64 = d == 64 && dv == 64;   // else the kernel of width 128
  cudaError_t e;
  if (drop_t < 256)
    e = w64 ? fa::launch_fwd_drop_d64(p, grid, bf16, causal != 0, stream)
            : fa::launch_fwd_drop_d128(p, grid, bf16, causal != 0, stream);
  else
    e = w64 ? fa::launch_fwd_kv_d64(p, grid, bf16, causal != 0, stream)
            : fa::launch_fwd_kv_d128(p, grid, bf16, causal != 0, stream);
  return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

int fa_fwd_kv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
              int Nq, int Nk, int d, int dv, int causal, const int* seqlens_k, float scale,
              int dtype, cudaStream_t stream) {
  return forward_kv(q, k, v, o, lse, B, H, Nq, Nk, d, dv, causal, seqlens_k, scale, dtype, 256, 0,
                    0, stream);
}

int fa_fwd_kv_dropout(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                      int H, int Nq, int Nk, int d, int dv, int causal, const int* seqlens_k,
                      float scale, float dropout_p, unsigned long long seed, unsigned int offset,
                      int dtype, cudaStream_t stream) {
  const int t = drop_threshold(dropout_p);
  if (t < 0) return FA_ERR_DROPOUT;
  return forward_kv(q, k, v, o, lse, B, H, Nq, Nk, d, dv, causal, seqlens_k, scale, dtype, t, seed,
                    offset, stream);
}

int fa_fwd_dropout(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                   int H, int N, int d, int causal, float scale, float dropout_p,
                   unsigned long long seed, unsigned int offset, int dtype,
                   cudaStream_t stream) {
  if (causal < 0 || causal > 1) return FA_ERR_SHAPE;
  const int t = drop_threshold(dropout_p);
  if (t < 0) return FA_ERR_DROPOUT;
  if (t == 256) return fa_fwd(q, k, v, o, lse, B, H, N, d, causal, scale, dtype, stream);
  return forward_kv(q, k, v, o, lse, B, H, N, N, d, d, causal, nullptr, scale, dtype, t, seed,
                    offset, stream);
}

// fa_fwd_varlen, and fa_fwd_varlen_dropout when drop_t < 256.
static int forward_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                          const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int H,
                          int max_seqlen_q, int total_q, int total_k, int d, int dv, int causal,
                          float scale, int dtype, int drop_t, unsigned long long seed,
                          unsigned int drop_off, cudaStream_t stream) {
  if (B < 0 || H < 0 || max_seqlen_q < 0 || total_q < 0 || total_k < 0 || d <= 0 || dv <= 0)
    return FA_ERR_SHAPE;
  if (causal < 0 || causal > 2) return FA_ERR_SHAPE;
  const long long bh = static_cast<long long>(B) * H;
  const long long n_qblk = (static_cast<long long>(max_seqlen_q) + 2 * fa::kBM - 1) / (2 * fa::kBM);
  if (bh > INT_MAX || bh * n_qblk > INT_MAX ||
      static_cast<long long>(total_q) * H > INT_MAX || static_cast<long long>(total_k) * H > INT_MAX)
    return FA_ERR_SHAPE;
  if ((d != 64 && d != 128) || (dv != 64 && dv != 128)) return FA_ERR_UNSUPPORTED_D;
  if (dtype != FA_BF16 && dtype != FA_FP16) return FA_ERR_DTYPE;
  if (!std::isfinite(scale) || !(scale > 0.0f)) return FA_ERR_SCALE;
  if (bh == 0 || max_seqlen_q == 0 || total_q == 0) return FA_OK;  // nothing to write
  if (!q || !o || !lse || !cu_seqlens_q || !cu_seqlens_k || (total_k > 0 && (!k || !v)))
    return FA_ERR_NULLPTR;
  const uintptr_t a16 = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                        reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o);
  const uintptr_t a4 = reinterpret_cast<uintptr_t>(lse) |
                       reinterpret_cast<uintptr_t>(cu_seqlens_q) |
                       reinterpret_cast<uintptr_t>(cu_seqlens_k);
  if ((a16 & 15u) || (a4 & 3u)) return FA_ERR_ALIGN;

  int dev = 0;
  const DeviceInfo* info = device_info(&dev);
  if (!info || !info->supported) return FA_ERR_DEVICE;
  if (info->err != FA_OK) return info->err;

  const bool bf16 = dtype == FA_BF16;
  fa::FwdParams p;
  const int nk_tok = total_k > 0 ? total_k : 1;   // no key tile is loaded without keys
  const void* kp = total_k > 0 ? k : q;
  const void* vp = total_k > 0 ? v : q;
  if (!make_tmap_tokens(&p.tm_q, q, H, total_q, d, bf16) ||
      !make_tmap_tokens(&p.tm_k, kp, H, nk_tok, d, bf16) ||
      !make_tmap_tokens(&p.tm_v, vp, H, nk_tok, dv, bf16) ||
      !make_tmap_tokens(&p.tm_o, o, H, total_q, dv, bf16))   // unused: rows are stored directly
    return FA_ERR_TENSORMAP;
  p.o = o;
  p.lse = lse;
  p.trace = g_trace.load();
  p.status = info->status;
  const unsigned long long wd = g_watchdog_ns.load();
  p.watchdog_cycles = (wd ? wd : kDefaultWatchdogNs) * 21ull / 10ull;
  p.BH = static_cast<int>(bh);
  p.N = max_seqlen_q;
  p.n_qblk = static_cast<int>(n_qblk);
  p.n_kv = 0;   // per sequence, from cu_seqlens_k
  p.num_units = static_cast<int>(bh * n_qblk);
  // K/V bytes of an average (sequence, head)
  p.hgroup = choose_group_ragged(bh, H, static_cast<long long>(total_k) * (d + dv) * 2ll / B,
                                 causal != 0);
  p.scale_log2 = scale * 1.4426950408889634f;
  p.split = 0;
  p.full_rounds = 0;
  p.tail_units = 0;
  p.ws_count = nullptr;
  p.ws_part = nullptr;
  p.Nk = total_k;
  p.H = H;
  p.seqlens_k = nullptr;
  p.align_br = causal == 2 ? 1 : 0;
  p.dqk = d;
  p.dv = dv;
  p.cu_q = cu_seqlens_q;
  p.cu_k = cu_seqlens_k;
  p.varlen = 1;
  p.total_q = total_q;
  set_dropout(&p, drop_t, seed, drop_off);
  const int grid = p.num_units < info->sms ? p.num_units : info->sms;
  const bool w64 = d == 64 && dv == 64;
  cudaError_t e;
  if (drop_t < 256)
    e = w64 ? fa::launch_fwd_drop_d64(p, grid, bf16, causal != 0, stream)
            : fa::launch_fwd_drop_d128(p, grid, bf16, causal != 0, stream);
  else
    e = w64 ? fa::launch_fwd_kv_d64(p, grid, bf16, causal != 0, stream)
            : fa::launch_fwd_kv_d128(p, grid, bf16, causal != 0, stream);
  return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

int fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                  const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int H,
                  int max_seqlen_q, int total_q, int total_k, int d, int dv, int causal,
                  float scale, int dtype, cudaStream_t stream) {
  return forward_varlen(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, B, H, max_seqlen_q, total_q,
                        total_k, d, dv, causal, scale, dtype, 256, 0, 0, stream);
}

int fa_fwd_varlen_dropout(const void* q, const void* k, const void* v, void* o, float* lse,
                          const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int H,
                          int max_seqlen_q, int total_q, int total_k, int d, int dv, int causal,
                          float scale, float dropout_p, unsigned long long seed,
                          unsigned int offset, int dtype, cudaStream_t stream) {
  const int t = drop_threshold(dropout_p);
  if (t < 0) return FA_ERR_DROPOUT;
  return forward_varlen(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, B, H, max_seqlen_q, total_q,
                        total_k, d, dv, causal, scale, dtype, t, seed, offset, stream);
}

}  // extern "C"
