// fa_bwd_launch.cuh — host-side launches of the backward kernels.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "fa_bwd_kernel.cuh"

namespace fa {

// Raise the dynamic shared-memory limit of `fn` once per device.
template <typename Fn>
cudaError_t bwd_smem_attr(Fn fn, std::atomic<uint64_t>& done, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(done.load() & bit)) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    done.fetch_or(bit);
  }
  return cudaSuccess;
}

// D = rowsum(dO * O), then one grid of dK/dV CTAs (one per key tile) and dQ
// CTAs (one per query tile), all on `stream`.  `o`, `dout` are [BH, N, D] in the storage dtype.
template <int D, bool kBf16, bool kCausal, bool kDrop = false, bool kKv = false>
cudaError_t launch_bwd_variant(const BwdParams& p, const void* o, const void* dout, float* delta,
                               int sms, cudaStream_t stream) {
  // rows of O and dO: every (batch*head, query), or the packed tokens x H
  const long long rows = p.varlen ? static_cast<long long>(p.total_q) * p.H
                                  : static_cast<long long>(p.BH) * p.N;
  // D = rowsum(dO * O) over the value width
  const long long threads = rows * (p.width_v / 8);
  long long blocks = (threads + 255) / 256;
  const long long cap = 8ll * sms;
  if (blocks > cap) blocks = cap;
  cudaError_t e = cudaSuccess;
  if (blocks > 0) {   // no queries (a kv call with Nq = 0): no D to form
    if (p.width_v == 64)
      fa_bwd_delta_kernel<64, kBf16><<<static_cast<int>(blocks), 256, 0, stream>>>(
          static_cast<const uint4*>(o), static_cast<const uint4*>(dout), delta, rows);
    else
      fa_bwd_delta_kernel<128, kBf16><<<static_cast<int>(blocks), 256, 0, stream>>>(
          static_cast<const uint4*>(o), static_cast<const uint4*>(dout), delta, rows);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }

  static std::atomic<uint64_t> done{0};
  constexpr int kAllocKv = BwdSmem<D, DkdvVec<D>::kBytes>::kAlloc;
  constexpr int kAllocQ = BwdSmem<D, 0>::kAlloc;
  constexpr int kAlloc = kAllocKv > kAllocQ ? kAllocKv : kAllocQ;
  e = bwd_smem_attr(fa_bwd_kernel<D, kBf16, kCausal, kDrop, kKv>, done, kAlloc);
  if (e != cudaSuccess) return e;
  // dK/dV items (one per key tile) then dQ items (one per query tile), on
  // at most one persistent CTA per SM, with programmatic dependent launch:
  // CTAs start their setup and loads while the D pass ends, and wait on the
  // device before reading D.
  const long long items = static_cast<long long>(p.BH) * (p.n_ktiles + p.n_tiles);
  const long long grid = items < sms ? items : sms;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kBwdThreads);
  cfg.dynamicSmemBytes = kAlloc;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fa_bwd_kernel<D, kBf16, kCausal, kDrop, kKv>, p);
}

cudaError_t launch_bwd_d64(const BwdParams& p, const void* o, const void* dout, float* delta,
                           bool bf16, bool causal, int sms, cudaStream_t stream);
cudaError_t launch_bwd_d128(const BwdParams& p, const void* o, const void* dout, float* delta,
                            bool bf16, bool causal, int sms, cudaStream_t stream);
// With dropout in the forward pass (the kDrop variants).
cudaError_t launch_bwd_drop_d64(const BwdParams& p, const void* o, const void* dout, float* delta,
                                bool bf16, bool causal, int sms, cudaStream_t stream);
cudaError_t launch_bwd_drop_d128(const BwdParams& p, const void* o, const void* dout, float* delta,
                                 bool bf16, bool causal, int sms, cudaStream_t stream);
// Queries against a key set of another length, or packed batches, with
// dropout in the forward pass (the kKv, kDrop variants).
cudaError_t launch_bwd_kv_drop_d64(const BwdParams& p, const void* o, const void* dout,
                                   float* delta, bool bf16, bool causal, int sms,
                                   cudaStream_t stream);
cudaError_t launch_bwd_kv_drop_d128(const BwdParams& p, const void* o, const void* dout,
                                    float* delta, bool bf16, bool causal, int sms,
                                    cudaStream_t stream);
// Queries against a key set of another length (the kKv variants).
cudaError_t launch_bwd_kv_d64(const BwdParams& p, const void* o, const void* dout, float* delta,
                              bool bf16, bool causal, int sms, cudaStream_t stream);
cudaError_t launch_bwd_kv_d128(const BwdParams& p, const void* o, const void* dout, float* delta,
                               bool bf16, bool causal, int sms, cudaStream_t stream);

}  // namespace fa
