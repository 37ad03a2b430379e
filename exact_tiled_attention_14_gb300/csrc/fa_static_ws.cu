// fa_static_ws.cu — fa_fwd_static: the balanced forward pass (fa_fwd_ws) with
// its scratch held in a fixed device array of this library, for callers that
// cannot allocate device memory themselves.
#include <cuda_runtime.h>

#include <mutex>

#include "fa.h"
#include "fa_host.cuh"

namespace {

// Scratch of fa_fwd_static.  Every GPU that loads this library holds these
// 40 MiB from the moment the library's code is loaded on it until the
// process exits.  That covers the balancing workspace of every supported
// shape on a GPU with up to 152 SMs (at most 38.6 MiB, at head width 128);
// a shape that would need more is rejected with FA_ERR_WORKSPACE.
constexpr size_t kStaticScratchBytes = 40ull << 20;
static __device__ __align__(256) unsigned char g_fa_static_scratch[kStaticScratchBytes];

// Device address of the array, looked up once per device (and again when a
// device reset has replaced that device's context: the library's code is
// then loaded anew and the array may sit elsewhere).  In host code the
// array's name only stands in for the symbol; the address a kernel can use
// comes from cudaGetSymbolAddress with that device current.
constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};

}  // namespace

extern "C" int fa_fwd_static(const void* q, const void* k, const void* v, void* o, float* lse,
                             int B, int H, int N, int d, int causal, float scale, int dtype,
                             cudaStream_t stream) {
  // the argument checks of fa_fwd_ws, in its order, before the size check
  bool empty = false;
  const int arg_rc =
      fa::host::check_forward_args(q, k, v, o, lse, B, H, N, d, scale, dtype, &empty);
  if (arg_rc != FA_OK || empty) return arg_rc;
  size_t need = 0;
  const int rc = fa_fwd_workspace_size(B, H, N, d, causal, &need);
  if (rc != FA_OK) return rc;
  if (need > kStaticScratchBytes) return FA_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (need > 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_mutex);
    const unsigned long long ctx = fa::host::current_context_id();
    if (g_scratch_addr[dev] == nullptr || (ctx != 0 && ctx != g_scratch_ctx[dev])) {
      void* addr = nullptr;
      if (cudaGetSymbolAddress(&addr, g_fa_static_scratch) != cudaSuccess || addr == nullptr)
        return FA_ERR_CUDA;
      g_scratch_addr[dev] = addr;
      g_scratch_ctx[dev] = ctx != 0 ? ctx : fa::host::current_context_id();
    }
    scratch = g_scratch_addr[dev];
  }
  // fa_fwd_ws clears the counters it needs at zero before its kernel runs.
  return fa_fwd_ws(q, k, v, o, lse, B, H, N, d, causal, scale, dtype, scratch,
                   scratch ? kStaticScratchBytes : 0, stream);
}
