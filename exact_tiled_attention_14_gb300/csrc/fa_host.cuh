// fa_host.cuh — host-side pieces shared by the translation units of the C
// ABI (defined in fa_common.cu): per-device facts, TMA descriptors, the
// bounded-wait budget and trace buffer, and the dropout keep rule.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "fa.h"

namespace fa {
namespace host {

constexpr unsigned long long kDefaultWatchdogNs = 2000000000ull;

struct DeviceInfo {
  int sms = 0;
  bool supported = false;
  unsigned int* status = nullptr;
  int err = FA_ERR_DEVICE;
};

// Per-device facts, queried with that device current once per CUDA context
// on it (again after a device reset has replaced the context, since the
// library's device symbols then have new addresses); NULL when no device is
// current.
const DeviceInfo* device_info(int* dev_out);

// Unique id of the calling thread's current CUDA context (cuCtxGetId), 0 when
// none is current or the driver cannot tell.
unsigned long long current_context_id();

// Argument checks of the square forward entry points, in their documented
// order: shape, head width, dtype, scale, then (unless the call is empty,
// which sets *empty and returns FA_OK) null pointers and alignment.
int check_forward_args(const void* q, const void* k, const void* v, const void* o,
                       const float* lse, int B, int H, int N, int d, float scale, int dtype,
                       bool* empty);

// 3-D view [BH, N, d] of a contiguous [B, H, N, d] tensor; boxes of 128 rows x
// 64 columns (128 bytes), 128-byte swizzle, zero fill past N.
bool make_tmap(CUtensorMap* m, const void* ptr, int BH, int N, int d, bool bf16);
// A packed token-major tensor [tokens, H, width] as a (column, head, token)
// map: a box of 64 columns x 1 head x 128 tokens fills shared memory exactly
// like a 128 x 64 tile of the [B, H, N, d] layout.
bool make_tmap_tokens(CUtensorMap* m, const void* ptr, int H, int tokens, int width, bool bf16);

// Budget of the kernels' bounded waits in ns (fa_set_watchdog_ns; 0 means
// kDefaultWatchdogNs), and the event-trace buffer of FA_TRACE builds.
extern std::atomic<unsigned long long> g_watchdog_ns;
extern std::atomic<unsigned long long*> g_trace;

// Keep threshold of the dropout rule: an element is kept when its random
// byte is below t = floor((1 - p) * 256 + 1/2), computed in double from the
// float p; kept weights are scaled by 256 / t.  -1 when p is not in [0, 1)
// or leaves t = 0.  t = 256 keeps everything (no dropout).
int drop_threshold(float p);

template <class Params>
void set_dropout(Params* p, int t, unsigned long long seed, unsigned int off) {
  p->drop_t = static_cast<uint32_t>(t);
  p->drop_k0 = static_cast<uint32_t>(seed);
  p->drop_k1 = static_cast<uint32_t>(seed >> 32);
  p->drop_off = off;
  p->drop_scale = 256.0f / static_cast<float>(t);
}

}  // namespace host
}  // namespace fa
