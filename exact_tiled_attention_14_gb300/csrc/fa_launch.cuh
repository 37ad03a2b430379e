// fa_launch.cuh — host-side launch of one compiled variant of the forward kernel.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "fa_fwd_kernel.cuh"

namespace fa {

// Launch fa_fwd_kernel<D, kBf16, kCausal, kSplit, kKv, kDrop> with `grid` persistent CTAs.
template <int D, bool kBf16, bool kCausal, bool kSplit, bool kKv = false, bool kDrop = false>
cudaError_t launch_variant(const FwdParams& p, int grid, cudaStream_t stream) {
  static std::atomic<uint64_t> attr_done{0};  // devices on which the smem limit was raised
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_done.load() & bit)) {
    e = cudaFuncSetAttribute(fa_fwd_kernel<D, kBf16, kCausal, kSplit, kKv, kDrop>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, Smem<D, kDrop>::kAlloc);
    if (e != cudaSuccess) return e;
    attr_done.fetch_or(bit);
  }
  fa_fwd_kernel<D, kBf16, kCausal, kSplit, kKv, kDrop><<<grid, threads_of<D, kDrop>(), Smem<D, kDrop>::kAlloc,
                                                         stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_fwd_d64(const FwdParams& p, int grid, bool bf16, bool causal,
                           cudaStream_t stream);
cudaError_t launch_fwd_d128(const FwdParams& p, int grid, bool bf16, bool causal,
                            cudaStream_t stream);
// Queries against a key set of their own length (the kKv variants).
cudaError_t launch_fwd_kv_d64(const FwdParams& p, int grid, bool bf16, bool causal,
                              cudaStream_t stream);
cudaError_t launch_fwd_kv_d128(const FwdParams& p, int grid, bool bf16, bool causal,
                               cudaStream_t stream);
// Square calls with dropout on the attention weights (the kKv, kDrop variants).
cudaError_t launch_fwd_drop_d64(const FwdParams& p, int grid, bool bf16, bool causal,
                                cudaStream_t stream);
cudaError_t launch_fwd_drop_d128(const FwdParams& p, int grid, bool bf16, bool causal,
                                 cudaStream_t stream);

}  // namespace fa
