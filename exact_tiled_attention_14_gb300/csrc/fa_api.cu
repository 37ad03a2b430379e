// fa_api.cu — the C ABI declared in include/fa.h: argument checks, TMA
// descriptors, per-device setup and the launch of the forward kernel.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <vector>

#include "fa.h"
#include "fa_bwd_launch.cuh"
#include "fa_decode_kernel.cuh"
#include "fa_launch.cuh"

namespace {

// Device status word written by the kernels' bounded waits (bit 0 = a wait
// ran out, bits 8..15 = where).  One per device; read and cleared by fa_status.
__device__ unsigned int g_fa_status = 0;

constexpr unsigned long long kDefaultWatchdogNs = 2000000000ull;

// Site recorded by the watchdog self-test's wait.
constexpr unsigned int kSiteSelfTest = 31;

// One thread waits, through the same bounded wait every kernel uses, on a
// barrier that nothing ever completes; the wait runs out after the budget
// and records the timeout in the status word, and the kernel returns.
__global__ void fa_watchdog_selftest_kernel(unsigned long long budget_cycles,
                                            unsigned int* status) {
  __shared__ __align__(8) unsigned long long never;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  abort_flag = 0;
  const uint32_t bar = fa::ptx::smem_u32(&never);
  fa::ptx::mbar_init(bar, 1);
  fa::ptx::fence_mbar_init();
  const fa::ptx::Watchdog wd{budget_cycles, &abort_flag, status};
  fa::ptx::wait_bounded(bar, 0, wd, kSiteSelfTest);
}
std::atomic<unsigned long long> g_watchdog_ns{0};
std::atomic<unsigned long long*> g_trace{nullptr};  // FA_TRACE builds only

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

struct DeviceInfo {
  int sms = 0;
  bool supported = false;
  unsigned int* status = nullptr;
  int err = FA_ERR_DEVICE;
};

constexpr int kMaxDevices = 64;
std::mutex g_dev_mutex;
bool g_dev_ready[kMaxDevices] = {};
DeviceInfo g_dev[kMaxDevices];

// Per-device facts, queried once with that device current.
const DeviceInfo* device_info(int* dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  *dev_out = dev;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  if (!g_dev_ready[dev]) {
    DeviceInfo info;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&info.sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess) {
      info.supported = (major == 10 && minor == 3);
      void* addr = nullptr;
      if (info.supported && cudaGetSymbolAddress(&addr, g_fa_status) == cudaSuccess) {
        info.status = static_cast<unsigned int*>(addr);
        info.err = FA_OK;
      }
    }
    g_dev[dev] = info;
    g_dev_ready[dev] = true;
  }
  return &g_dev[dev];
}

// 3-D view [BH, N, d] of a contiguous [B, H, N, d] tensor; boxes of 128 rows x
// 64 columns (128 bytes), 128-byte swizzle, zero fill past N.
bool make_tmap(CUtensorMap* m, const void* ptr, int BH, int N, int d, bool bf16) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                                 static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(d) * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(fa::kBM), 1};
  const cuuint32_t elem_strides[3] = {1, 1, 1};
  const CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                        3, const_cast<void*>(ptr), dims, strides, box, elem_strides,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// A packed token-major tensor [tokens, H, width] as a (column, head, token)
// map: a box of 64 columns x 1 head x 128 tokens fills shared memory exactly
// like a 128 x 64 tile of the [B, H, N, d] layout.
bool make_tmap_tokens(CUtensorMap* m, const void* ptr, int H, int tokens, int width, bool bf16) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(width), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(tokens)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(width) * 2,
                                 static_cast<cuuint64_t>(H) * static_cast<cuuint64_t>(width) * 2};
  const cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(fa::kBM)};
  const cuuint32_t elem_strides[3] = {1, 1, 1};
  const CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                        3, const_cast<void*>(ptr), dims, strides, box, elem_strides,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// ---------------------------------------------------------------- dropout
// Keep threshold of the dropout rule: an element is kept when its random
// byte is below t = floor((1 - p) * 256 + 1/2), computed in double from the
// float p; kept weights are scaled by 256 / t.  -1 when p is not in [0, 1)
// or leaves t = 0.  t = 256 keeps everything (no dropout).
int drop_threshold(float p) {
  if (!(p >= 0.0f) || !(p < 1.0f)) return -1;
  const int t = static_cast<int>(std::floor((1.0 - static_cast<double>(p)) * 256.0 + 0.5));
  return t >= 1 ? t : -1;
}

template <class Params>
void set_dropout(Params* p, int t, unsigned long long seed, unsigned int off) {
  p->drop_t = static_cast<uint32_t>(t);
  p->drop_k0 = static_cast<uint32_t>(seed);
  p->drop_k1 = static_cast<uint32_t>(seed >> 32);
  p->drop_off = off;
  p->drop_scale = 256.0f / static_cast<float>(t);
}

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

int fa_version(void) { return 103; }

const char* fa_strerror(int code) {
  switch (code) {
    case FA_OK: return "ok";
    case FA_ERR_NULLPTR: return "a required pointer is NULL";
    case FA_ERR_SHAPE: return "bad shape (negative size, d <= 0, or sizes overflow)";
    case FA_ERR_UNSUPPORTED_D: return "head width d must be 64 or 128";
    case FA_ERR_DTYPE: return "dtype must be FA_BF16 or FA_FP16";
    case FA_ERR_ALIGN: return "q/k/v/o must be 16-byte aligned and lse 4-byte aligned";
    case FA_ERR_SCALE: return "scale must be finite and > 0";
    case FA_ERR_DEVICE: return "current device is not a compute capability 10.3 GPU";
    case FA_ERR_TENSORMAP: return "TMA descriptor creation failed";
    case FA_ERR_LAUNCH: return "kernel launch failed";
    case FA_ERR_TIMEOUT: return "a bounded wait in a kernel ran out (watchdog)";
    case FA_ERR_CUDA: return "CUDA runtime error";
    case FA_ERR_WORKSPACE: return "workspace smaller than fa_fwd_workspace_size reports";
    case FA_ERR_DROPOUT: return "dropout probability must be in [0, 1) and keep at least 1/256";
    default: return "unknown error code";
  }
}

void fa_set_watchdog_ns(unsigned long long ns) {
  const unsigned long long kMaxNs = 1000000000000ull;  // 1000 s keeps the cycle count in range
  g_watchdog_ns.store(ns > kMaxNs ? kMaxNs : ns);
}

int fa_set_unit_group(int heads) {
  if (heads < 0) return FA_ERR_SHAPE;
  g_unit_group.store(heads);
  return FA_OK;
}

#if defined(FA_TRACE) || defined(FA_PROFILE)
// Trace / profile builds only (not part of the ABI in fa.h): device buffer that
// kernels launched afterwards record events into, or NULL to stop.  It must
// hold grid * 4 * kTraceCap * 16 bytes.
int fa_debug_set_trace(void* buf) {
  g_trace.store(static_cast<unsigned long long*>(buf));
  return FA_OK;
}
int fa_debug_trace_cap(void) { return fa::kTraceCap; }
int fa_debug_prof_slots(void) { return fa::kProfSlots; }
#endif

int fa_work_tiles(int N, int causal, long long* pairs) {
  if (!pairs) return FA_ERR_NULLPTR;
  if (N < 0) return FA_ERR_SHAPE;
  const long long n = (static_cast<long long>(N) + fa::kBN - 1) / fa::kBN;
  *pairs = causal ? n * (n + 1) / 2 : n * n;
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

// Shared by fa_fwd (no workspace) and fa_fwd_ws.
int launch_forward(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                   int N, int d, int causal, float scale, int dtype, void* workspace,
                   size_t workspace_bytes, cudaStream_t stream) {
  if (B < 0 || H < 0 || N < 0 || d <= 0) return FA_ERR_SHAPE;
  const long long bh = static_cast<long long>(B) * H;
  const long long n_qblk = (static_cast<long long>(N) + 2 * fa::kBM - 1) / (2 * fa::kBM);
  if (bh > INT_MAX || bh * n_qblk > INT_MAX) return FA_ERR_SHAPE;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED_D;
  if (dtype != FA_BF16 && dtype != FA_FP16) return FA_ERR_DTYPE;
  if (!std::isfinite(scale) || !(scale > 0.0f)) return FA_ERR_SCALE;
  if (bh == 0 || N == 0) return FA_OK;  // nothing to write
  if (!q || !k || !v || !o || !lse) return FA_ERR_NULLPTR;
  const uintptr_t a16 = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                        reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o);
  if ((a16 & 15u) || (reinterpret_cast<uintptr_t>(lse) & 3u)) return FA_ERR_ALIGN;

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

int fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                  const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int H,
                  int max_seqlen_q, int total_q, int total_k, int d, int dv, int causal,
                  float scale, int dtype, cudaStream_t stream) {
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
  set_dropout(&p, 256, 0, 0);
  const int grid = p.num_units < info->sms ? p.num_units : info->sms;
  const bool w64 = d == 64 && dv == 64;
  const cudaError_t e = w64 ? fa::launch_fwd_kv_d64(p, grid, bf16, causal != 0, stream)
                            : fa::launch_fwd_kv_d128(p, grid, bf16, causal != 0, stream);
  return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

// fa_bwd, fa_bwd_dropout when drop_t < 256, and fa_bwd_kv when kv (Nq
// queries against Nk keys with per-batch key counts; causal 2 bottom-right).
static int backward(const void* q, const void* k, const void* v, const void* o, const float* lse,
                    const void* dout, void* dq, void* dk, void* dv, float* delta, int B, int H,
                    int Nq, int Nk, int d, int causal, bool kv, const int* seqlens_k, float scale,
                    int dtype, int drop_t, unsigned long long seed, unsigned int drop_off,
                    cudaStream_t stream) {
  if (B < 0 || H < 0 || Nq < 0 || Nk < 0 || d <= 0) return FA_ERR_SHAPE;
  if (causal < 0 || causal > (kv ? 2 : 1)) return FA_ERR_SHAPE;
  const long long bh = static_cast<long long>(B) * H;
  const long long n_qtiles = (static_cast<long long>(Nq) + fa::kBwdTile - 1) / fa::kBwdTile;
  const long long n_ktiles = (static_cast<long long>(Nk) + fa::kBwdTile - 1) / fa::kBwdTile;
  if (bh > INT_MAX || bh * (n_qtiles + n_ktiles) > INT_MAX) return FA_ERR_SHAPE;   // one grid
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED_D;
  if (dtype != FA_BF16 && dtype != FA_FP16) return FA_ERR_DTYPE;
  if (!std::isfinite(scale) || !(scale > 0.0f)) return FA_ERR_SCALE;
  if (bh == 0 || (Nq == 0 && Nk == 0)) return FA_OK;  // nothing to write
  if (Nq > 0 && (!q || !o || !lse || !dout || !dq || !delta)) return FA_ERR_NULLPTR;
  if (Nk > 0 && (!k || !v || !dk || !dv)) return FA_ERR_NULLPTR;
  const uintptr_t a16 = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                        reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o) |
                        reinterpret_cast<uintptr_t>(dout) | reinterpret_cast<uintptr_t>(dq) |
                        reinterpret_cast<uintptr_t>(dk) | reinterpret_cast<uintptr_t>(dv);
  const uintptr_t a4 = reinterpret_cast<uintptr_t>(lse) | reinterpret_cast<uintptr_t>(delta) |
                       reinterpret_cast<uintptr_t>(seqlens_k);
  if ((a16 & 15u) || (a4 & 3u)) return FA_ERR_ALIGN;

  int dev = 0;
  const DeviceInfo* info = device_info(&dev);
  if (!info || !info->supported) return FA_ERR_DEVICE;
  if (info->err != FA_OK) return info->err;

  const bool bf16 = dtype == FA_BF16;
  fa::BwdParams p;
  // Without queries or keys no tile of them is ever loaded; the maps still
  // need a row and an address.
  const int nq_rows = Nq > 0 ? Nq : 1, nk_rows = Nk > 0 ? Nk : 1;
  const void* qa = Nq > 0 ? q : k;
  const void* ka = Nk > 0 ? k : q;
  const void* va = Nk > 0 ? v : q;
  const void* da = Nq > 0 ? dout : k;
  if (!make_tmap(&p.tm_q, qa, static_cast<int>(bh), nq_rows, d, bf16) ||
      !make_tmap(&p.tm_k, ka, static_cast<int>(bh), nk_rows, d, bf16) ||
      !make_tmap(&p.tm_v, va, static_cast<int>(bh), nk_rows, d, bf16) ||
      !make_tmap(&p.tm_do, da, static_cast<int>(bh), nq_rows, d, bf16))
    return FA_ERR_TENSORMAP;
  p.lse = lse;
  p.delta = delta;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.status = info->status;
  const unsigned long long wd = g_watchdog_ns.load();
  p.watchdog_cycles = (wd ? wd : kDefaultWatchdogNs) * 21ull / 10ull;
  p.BH = static_cast<int>(bh);
  p.N = Nq;
  p.n_tiles = static_cast<int>(n_qtiles);
  p.Nk = Nk;
  p.n_ktiles = static_cast<int>(n_ktiles);
  p.H = H;
  p.seqlens_k = seqlens_k;
  p.align_br = causal == 2 ? 1 : 0;
  p.cu_q = nullptr;
  p.cu_k = nullptr;
  p.varlen = 0;
  p.total_q = 0;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  set_dropout(&p, drop_t, seed, drop_off);
  const bool c = causal != 0;
  cudaError_t e;
  if (kv)
    e = (d == 64) ? fa::launch_bwd_kv_d64(p, o, dout, delta, bf16, c, info->sms, stream)
                  : fa::launch_bwd_kv_d128(p, o, dout, delta, bf16, c, info->sms, stream);
  else if (drop_t < 256)
    e = (d == 64) ? fa::launch_bwd_drop_d64(p, o, dout, delta, bf16, c, info->sms, stream)
                  : fa::launch_bwd_drop_d128(p, o, dout, delta, bf16, c, info->sms, stream);
  else
    e = (d == 64) ? fa::launch_bwd_d64(p, o, dout, delta, bf16, c, info->sms, stream)
                  : fa::launch_bwd_d128(p, o, dout, delta, bf16, c, info->sms, stream);
  return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
           const void* dout, void* dq, void* dk, void* dv, float* delta, int B, int H, int N,
           int d, int causal, float scale, int dtype, cudaStream_t stream) {
  return backward(q, k, v, o, lse, dout, dq, dk, dv, delta, B, H, N, N, d, causal, false, nullptr,
                  scale, dtype, 256, 0, 0, stream);
}

int fa_bwd_kv(const void* q, const void* k, const void* v, const void* o, const float* lse,
              const void* dout, void* dq, void* dk, void* dv, float* delta, int B, int H, int Nq,
              int Nk, int d, int causal, const int* seqlens_k, float scale, int dtype,
              cudaStream_t stream) {
  return backward(q, k, v, o, lse, dout, dq, dk, dv, delta, B, H, Nq, Nk, d, causal, true,
                  seqlens_k, scale, dtype, 256, 0, 0, stream);
}

int fa_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const float* lse,
                  const void* dout, void* dq, void* dk, void* dv, float* delta,
                  const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int H,
                  int max_seqlen_q, int max_seqlen_k, int total_q, int total_k, int d,
                  int causal, float scale, int dtype, cudaStream_t stream) {
  if (B < 0 || H < 0 || max_seqlen_q < 0 || max_seqlen_k < 0 || total_q < 0 || total_k < 0 ||
      d <= 0)
    return FA_ERR_SHAPE;
  if (causal < 0 || causal > 2) return FA_ERR_SHAPE;
  const long long bh = static_cast<long long>(B) * H;
  const long long n_qtiles = (static_cast<long long>(max_seqlen_q) + fa::kBwdTile - 1) / fa::kBwdTile;
  const long long n_ktiles = (static_cast<long long>(max_seqlen_k) + fa::kBwdTile - 1) / fa::kBwdTile;
  if (bh > INT_MAX || bh * (n_qtiles + n_ktiles) > INT_MAX ||
      static_cast<long long>(total_q) * H > INT_MAX || static_cast<long long>(total_k) * H > INT_MAX)
    return FA_ERR_SHAPE;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED_D;
  if (dtype != FA_BF16 && dtype != FA_FP16) return FA_ERR_DTYPE;
  if (!std::isfinite(scale) || !(scale > 0.0f)) return FA_ERR_SCALE;
  if (bh == 0 || (total_q == 0 && total_k == 0) || (n_qtiles == 0 && n_ktiles == 0)) return FA_OK;
  if (!cu_seqlens_q || !cu_seqlens_k) return FA_ERR_NULLPTR;
  if (total_q > 0 && (!q || !o || !lse || !dout || !dq || !delta)) return FA_ERR_NULLPTR;
  if (total_k > 0 && (!k || !v || !dk || !dv)) return FA_ERR_NULLPTR;
  const uintptr_t a16 = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                        reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o) |
                        reinterpret_cast<uintptr_t>(dout) | reinterpret_cast<uintptr_t>(dq) |
                        reinterpret_cast<uintptr_t>(dk) | reinterpret_cast<uintptr_t>(dv);
  const uintptr_t a4 = reinterpret_cast<uintptr_t>(lse) | reinterpret_cast<uintptr_t>(delta) |
                       reinterpret_cast<uintptr_t>(cu_seqlens_q) |
                       reinterpret_cast<uintptr_t>(cu_seqlens_k);
  if ((a16 & 15u) || (a4 & 3u)) return FA_ERR_ALIGN;

  int dev = 0;
  const DeviceInfo* info = device_info(&dev);
  if (!info || !info->supported) return FA_ERR_DEVICE;
  if (info->err != FA_OK) return info->err;

  const bool bf16 = dtype == FA_BF16;
  fa::BwdParams p;
  const int q_tok = total_q > 0 ? total_q : 1, k_tok = total_k > 0 ? total_k : 1;
  const void* qa = total_q > 0 ? q : k;
  const void* da = total_q > 0 ? dout : k;
  const void* ka = total_k > 0 ? k : q;
  const void* va = total_k > 0 ? v : q;
  if (!make_tmap_tokens(&p.tm_q, qa, H, q_tok, d, bf16) ||
      !make_tmap_tokens(&p.tm_k, ka, H, k_tok, d, bf16) ||
      !make_tmap_tokens(&p.tm_v, va, H, k_tok, d, bf16) ||
      !make_tmap_tokens(&p.tm_do, da, H, q_tok, d, bf16))
    return FA_ERR_TENSORMAP;
  p.lse = lse;
  p.delta = delta;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.status = info->status;
  const unsigned long long wd = g_watchdog_ns.load();
  p.watchdog_cycles = (wd ? wd : kDefaultWatchdogNs) * 21ull / 10ull;
  p.BH = static_cast<int>(bh);
  p.N = max_seqlen_q;
  p.n_tiles = static_cast<int>(n_qtiles);
  p.Nk = total_k;
  p.n_ktiles = static_cast<int>(n_ktiles);
  p.H = H;
  p.seqlens_k = nullptr;
  p.align_br = causal == 2 ? 1 : 0;
  p.cu_q = cu_seqlens_q;
  p.cu_k = cu_seqlens_k;
  p.varlen = 1;
  p.total_q = total_q;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  set_dropout(&p, 256, 0, 0);
  const bool c = causal != 0;
  const cudaError_t e = (d == 64) ? fa::launch_bwd_kv_d64(p, o, dout, delta, bf16, c, info->sms, stream)
                                  : fa::launch_bwd_kv_d128(p, o, dout, delta, bf16, c, info->sms, stream);
  return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

int fa_bwd_dropout(const void* q, const void* k, const void* v, const void* o, const float* lse,
                   const void* dout, void* dq, void* dk, void* dv, float* delta, int B, int H,
                   int N, int d, int causal, float scale, float dropout_p,
                   unsigned long long seed, unsigned int offset, int dtype,
                   cudaStream_t stream) {
  const int t = drop_threshold(dropout_p);
  if (t < 0) return FA_ERR_DROPOUT;
  return backward(q, k, v, o, lse, dout, dq, dk, dv, delta, B, H, N, N, d, causal, false, nullptr,
                  scale, dtype, t, seed, offset, stream);
}

}  // extern "C"

namespace fa {
cudaError_t launch_decode(const DecodeParams& p, void* o, float* lse, int d, bool bf16,
                          cudaStream_t stream);
}

namespace {

// Split of the key axis for fa_decode.  One CTA per SM at a time (its ring
// takes most of the shared memory), so a call takes ceil(CTAs / SMs) waves,
// each as long as a split plus a fixed cost per CTA (query load, pipeline
// fill, partial write; about three tiles' worth).  The plan takes the
// number of splits per head, 1 .. ceil(tiles / 4), that minimises
// waves x (tiles per split + 3) (measured on a 67 MB cache over 8 heads:
// one wave of 19 splits, 39 us, against 47 us for 32 splits in two waves).
struct DecodePlan {
  int splits = 0;
  int tiles_per_split = 0;
  size_t o_bytes = 0;     // partial outputs
  size_t bytes = 0;       // whole workspace (partial outputs, then (m, l) pairs)
};

DecodePlan plan_decode(long long bh, int Nq, int Nk, int d, int sms) {
  DecodePlan dp;
  const int tiles = (Nk + fa::kDecTile - 1) / fa::kDecTile;
  if (tiles == 0 || bh == 0) return dp;
  // Within a number of waves more splits never cost more, so only the
  // largest split count of each wave count (and the cap itself) is tried.
  const long long max_splits = (tiles + 3) / 4;
  long long want = 1, best = -1;
  auto consider = [&](long long sp) {
    if (sp < 1) sp = 1;
    if (sp > max_splits) sp = max_splits;
    const long long per = (tiles + sp - 1) / sp;
    const long long cost = ((bh * sp + sms - 1) / sms) * (per + 3);
    if (best < 0 || cost < best || (cost == best && sp < want)) {
      best = cost;
      want = sp;
    }
  };
  const long long max_waves = (bh * max_splits + sms - 1) / sms;
  for (long long w = 1; w <= max_waves; ++w) consider(w * sms / bh);
  consider(max_splits);
  dp.tiles_per_split = static_cast<int>((tiles + want - 1) / want);
  dp.splits = (tiles + dp.tiles_per_split - 1) / dp.tiles_per_split;
  const size_t parts = static_cast<size_t>(bh) * dp.splits * Nq;
  dp.o_bytes = (parts * d * sizeof(float) + 255) / 256 * 256;
  dp.bytes = dp.o_bytes + (parts * 2 * sizeof(float) + 255) / 256 * 256;
  return dp;
}

int decode_checks(int B, int H, int Nq, int Nk, int d, long long* bh) {
  if (B < 0 || H < 0 || Nk < 0 || d <= 0) return FA_ERR_SHAPE;
  if (Nq < 1 || Nq > fa::kDecMaxQ) return FA_ERR_SHAPE;
  *bh = static_cast<long long>(B) * H;
  if (*bh * Nq > INT_MAX || *bh * ((static_cast<long long>(Nk) + 127) / 128) > INT_MAX)
    return FA_ERR_SHAPE;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED_D;
  return FA_OK;
}

}  // namespace

extern "C" {

int fa_decode_workspace_size(int B, int H, int Nq, int Nk, int d, size_t* bytes) {
  if (!bytes) return FA_ERR_NULLPTR;
  long long bh = 0;
  const int rc = decode_checks(B, H, Nq, Nk, d, &bh);
  if (rc != FA_OK) return rc;
  *bytes = 0;
  if (bh == 0 || Nk == 0) return FA_OK;
  int dev = 0;
  const DeviceInfo* info = device_info(&dev);
  if (!info || !info->supported) return FA_ERR_DEVICE;
  *bytes = plan_decode(bh, Nq, Nk, d, info->sms).bytes;
  return FA_OK;
}

int fa_decode(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
              int Nq, int Nk, int d, int causal, float scale, int dtype, void* workspace,
              size_t workspace_bytes, cudaStream_t stream) {
  long long bh = 0;
  const int rc = decode_checks(B, H, Nq, Nk, d, &bh);
  if (rc != FA_OK) return rc;
  if (dtype != FA_BF16 && dtype != FA_FP16) return FA_ERR_DTYPE;
  if (!std::isfinite(scale) || !(scale > 0.0f)) return FA_ERR_SCALE;
  if (bh == 0) return FA_OK;  // nothing to write
  if (!q || !o || !lse || (Nk > 0 && (!k || !v))) return FA_ERR_NULLPTR;
  const uintptr_t a16 = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                        reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o);
  if ((a16 & 15u) || (reinterpret_cast<uintptr_t>(lse) & 3u)) return FA_ERR_ALIGN;

  int dev = 0;
  const DeviceInfo* info = device_info(&dev);
  if (!info || !info->supported) return FA_ERR_DEVICE;
  if (info->err != FA_OK) return info->err;
  const DecodePlan dp = plan_decode(bh, Nq, Nk, d, info->sms);
  if (dp.bytes > 0) {
    if (!workspace || workspace_bytes < dp.bytes) return FA_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return FA_ERR_ALIGN;
  }
  const bool bf16 = dtype == FA_BF16;
  fa::DecodeParams p;
  if (Nk > 0 && (!make_tmap(&p.tm_k, k, static_cast<int>(bh), Nk, d, bf16) ||
                 !make_tmap(&p.tm_v, v, static_cast<int>(bh), Nk, d, bf16)))
    return FA_ERR_TENSORMAP;
  p.q = q;
  p.part_o = static_cast<float*>(workspace);
  p.part_ml = dp.bytes ? reinterpret_cast<float2*>(static_cast<uint8_t*>(workspace) + dp.o_bytes)
                       : nullptr;
  p.status = info->status;
  const unsigned long long wd = g_watchdog_ns.load();
  p.watchdog_cycles = (wd ? wd : kDefaultWatchdogNs) * 21ull / 10ull;
  p.BH = static_cast<int>(bh);
  p.Nq = Nq;
  p.Nk = Nk;
  p.splits = dp.splits;
  p.tiles_per_split = dp.tiles_per_split;
  p.causal = causal ? 1 : 0;
  p.scale_log2 = scale * 1.4426950408889634f;
  const cudaError_t e = fa::launch_decode(p, o, lse, d, bf16, stream);
  return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

int fa_watchdog_selftest(unsigned long long budget_ns, cudaStream_t stream) {
  if (budget_ns == 0 || budget_ns > 1000000000ull) return FA_ERR_SHAPE;
  int dev = 0;
  const DeviceInfo* info = device_info(&dev);
  if (!info || !info->supported) return FA_ERR_DEVICE;
  if (info->err != FA_OK) return info->err;
  fa_watchdog_selftest_kernel<<<1, 32, 0, stream>>>(budget_ns * 21ull / 10ull, info->status);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

int fa_status(cudaStream_t stream, unsigned int* detail) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return FA_ERR_CUDA;
  unsigned int word = 0;
  if (cudaMemcpyFromSymbol(&word, g_fa_status, sizeof(word)) != cudaSuccess) return FA_ERR_CUDA;
  if (word) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_fa_status, &zero, sizeof(zero)) != cudaSuccess) return FA_ERR_CUDA;
  }
  if (detail) *detail = word;
  return word ? FA_ERR_TIMEOUT : FA_OK;
}

}  // extern "C"
