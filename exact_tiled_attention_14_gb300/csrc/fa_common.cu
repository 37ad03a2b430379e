// fa_common.cu — the parts of the C ABI declared in include/fa.h that every
// entry point shares: per-device setup, TMA descriptors, error strings, the
// status word and its self-test, and the process-wide settings.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "fa.h"
#include "fa_host.cuh"
#include "fa_launch.cuh"

using namespace fa::host;

namespace {

// Device status word written by the kernels' bounded waits (bit 0 = a wait
// ran out, bits 8..15 = where).  One per device; read and cleared by fa_status.
__device__ unsigned int g_fa_status = 0;

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

// cuCtxGetCurrent and cuCtxGetId through the runtime's driver entry points
// (the library links no driver library).
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
struct CtxFns {
  CtxGetCurrentFn get_current = nullptr;
  CtxGetIdFn get_id = nullptr;
};
const CtxFns& ctx_fns() {
  static CtxFns fns;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fns.get_current = reinterpret_cast<CtxGetCurrentFn>(ptr);
    ptr = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fns.get_id = reinterpret_cast<CtxGetIdFn>(ptr);
  });
  return fns;
}

constexpr int kMaxDevices = 64;
std::mutex g_dev_mutex;
bool g_dev_ready[kMaxDevices] = {};
unsigned long long g_dev_ctx[kMaxDevices] = {};   // context the entry was set up in
DeviceInfo g_dev[kMaxDevices];

}  // namespace

namespace fa {
namespace host {

std::atomic<unsigned long long> g_watchdog_ns{0};
std::atomic<unsigned long long*> g_trace{nullptr};  // FA_TRACE builds only

unsigned long long current_context_id() {
  const CtxFns& f = ctx_fns();
  if (!f.get_current || !f.get_id) return 0;
  CUcontext ctx = nullptr;
  if (f.get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  unsigned long long id = 0;
  return f.get_id(ctx, &id) == CUDA_SUCCESS ? id : 0;
}

const DeviceInfo* device_info(int* dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  *dev_out = dev;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  // A device reset replaces the context, and with it the addresses of this
  // library's device symbols: set the entry up again in the new context.
  const unsigned long long ctx = current_context_id();
  if (g_dev_ready[dev] && ctx != 0 && ctx != g_dev_ctx[dev]) g_dev_ready[dev] = false;
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
    // the symbol lookup above made the device's primary context current if
    // no context was
    g_dev_ctx[dev] = ctx != 0 ? ctx : current_context_id();
  }
  return &g_dev[dev];
}

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

int drop_threshold(float p) {
  if (!(p >= 0.0f) || !(p < 1.0f)) return -1;
  const int t = static_cast<int>(std::floor((1.0 - static_cast<double>(p)) * 256.0 + 0.5));
  return t >= 1 ? t : -1;
}

}  // namespace host
}  // namespace fa

extern "C" {

int fa_version(void) { return 104; }

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
  // One head's schedule, walked unit by unit with the kernel's own decode:
  // the sum of the key tiles its query tiles stream.
  fa::FwdParams p{};
  p.BH = 1;
  p.H = 1;
  p.N = N;
  p.Nk = N;
  p.n_qblk = (N + 2 * fa::kBM - 1) / (2 * fa::kBM);
  p.n_kv = (N + fa::kBN - 1) / fa::kBN;
  p.num_units = p.n_qblk;
  p.hgroup = 1;
  long long total = 0;
  for (int s = 0; s < p.num_units; ++s) {
    const fa::Unit u = causal ? fa::decode_unit<true>(s, p) : fa::decode_unit<false>(s, p);
    total += u.n0 + u.n1;
  }
  *pairs = total;
  return FA_OK;
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
