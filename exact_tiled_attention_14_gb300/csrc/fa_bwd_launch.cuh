// fa_bwd_launch.cuh — host-side launches of the backward kernels.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "fa_bwd_kernel.cuh"
#include "fa_bwd_onepass.cuh"

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

// D = rowsum(dO * O) over the value width on `stream`.  `o`, `dout` are
// [BH, N, width_v] (or the packed tokens x H) in the storage dtype.
template <bool kBf16>
cudaError_t launch_bwd_delta(const BwdParams& p, const void* o, const void* dout, float* delta,
                             int sms, cudaStream_t stream) {
  // rows of O and dO: every (batch*head, query), or the packed tokens x H
  const long long rows = p.varlen ? static_cast<long long>(p.total_q) * p.H
                                  : static_cast<long long>(p.BH) * p.N;
  const long long threads = rows * (p.width_v / 8);
  long long blocks = (threads + 255) / 256;
  const long long cap = 8ll * sms;
  if (blocks > cap) blocks = cap;
  if (blocks <= 0) return cudaSuccess;   // no queries (a kv call with Nq = 0): no D to form
  if (p.width_v == 64)
    fa_bwd_delta_kernel<64, kBf16><<<static_cast<int>(blocks), 256, 0, stream>>>(
        static_cast<const uint4*>(o), static_cast<const uint4*>(dout), delta, rows);
  else
    fa_bwd_delta_kernel<128, kBf16><<<static_cast<int>(blocks), 256, 0, stream>>>(
        static_cast<const uint4*>(o), static_cast<const uint4*>(dout), delta, rows);
  return cudaGetLastError();
}

// The tensor-core grid of `kernel` on at most one CTA per SM, with
// programmatic dependent launch: CTAs start their setup and loads while the
// D pass ends, and wait on the device before reading D.
template <typename Kernel>
cudaError_t launch_bwd_grid(Kernel kernel, const BwdParams& p, long long items, int smem, int sms,
                            cudaStream_t stream, int threads = kBwdThreads) {
  const long long grid = items < sms ? items : sms;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

// D = rowsum(dO * O), then one grid of dK/dV CTAs (one per key tile) and dQ
// CTAs (one per query tile), all on `stream`.  `o`, `dout` are [BH, N, D] in the storage dtype.
template <int D, bool kBf16, bool kCausal, bool kDrop = false, bool kKv = false>
cudaError_t launch_bwd_variant(const BwdParams& p, const void* o, const void* dout, float* delta,
                               int sms, cudaStream_t stream) {
  cudaError_t e = launch_bwd_delta<kBf16>(p, o, dout, delta, sms, stream);
  if (e != cudaSuccess) return e;

  static std::atomic<uint64_t> done{0};
  constexpr int kAllocKv = BwdSmem<D, DkdvVec<D>::kBytes>::kAlloc;
  constexpr int kAllocQ = BwdSmem<D, 0>::kAlloc;
  constexpr int kAlloc = kAllocKv > kAllocQ ? kAllocKv : kAllocQ;
  e = bwd_smem_attr(fa_bwd_kernel<D, kBf16, kCausal, kDrop, kKv>, done, kAlloc);
  if (e != cudaSuccess) return e;
  // dK/dV items (one per key tile) then dQ items (one per query tile)
  const long long items = static_cast<long long>(p.BH) * (p.n_ktiles + p.n_tiles);
  return launch_bwd_grid(fa_bwd_kernel<D, kBf16, kCausal, kDrop, kKv>, p, items, kAlloc, sms,
                         stream);
}

// The one-pass backward (square calls): the fp32 dQ accumulator p.dq_acc
// ([BH, width_qk, dq_pad]) is zeroed, D formed, one grid of dK/dV CTAs adds
// every dQ_i = dS K_j into the accumulator, and a last kernel writes
// dQ = scale * accumulator in the storage dtype, all on `stream`.
template <int D, bool kBf16, bool kCausal, bool kDrop = false>
cudaError_t launch_bwd_onepass_variant(const BwdParams& p, const void* o, const void* dout,
                                       float* delta, int sms, cudaStream_t stream) {
  const size_t acc_bytes =
      static_cast<size_t>(p.BH) * p.width_qk * static_cast<size_t>(p.dq_pad) * sizeof(float);
  cudaError_t e = cudaMemsetAsync(p.dq_acc, 0, acc_bytes, stream);
  if (e != cudaSuccess) return e;
  e = launch_bwd_delta<kBf16>(p, o, dout, delta, sms, stream);
  if (e != cudaSuccess) return e;
  static std::atomic<uint64_t> done{0};
  constexpr int kAlloc = BwdSmem<D, DkdvVec<D>::kBytes, true>::kAlloc;
  auto kernel = fa_bwd_onepass_kernel<D, kBf16, kCausal, kDrop>;
  e = bwd_smem_attr(kernel, done, kAlloc);
  if (e != cudaSuccess) return e;
  e = launch_bwd_grid(kernel, p, static_cast<long long>(p.BH) * p.n_ktiles, kAlloc, sms, stream,
                      kOneThreads);
  if (e != cudaSuccess) return e;
  const long long blocks = static_cast<long long>(p.BH) * p.n_tiles;
  fa_bwd_dq_convert_kernel<kBf16><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      p.dq_acc, static_cast<uint32_t*>(p.dq), p.N, p.width_qk, p.dq_pad, p.scale);
  return cudaGetLastError();
}

cudaError_t launch_bwd_d64(const BwdParams& p, const void* o, const void* dout, float* delta,
                           bool bf16, bool causal, int sms, cudaStream_t stream);
cudaError_t launch_bwd_d128(const BwdParams& p, const void* o, const void* dout, float* delta,
                            bool bf16, bool causal, int sms, cudaStream_t stream);
// The one-pass backward (square calls, dQ accumulated in p.dq_acc), and
// with dropout in the forward pass.
cudaError_t launch_bwd_onepass_d64(const BwdParams& p, const void* o, const void* dout,
                                   float* delta, bool bf16, bool causal, int sms,
                                   cudaStream_t stream);
cudaError_t launch_bwd_onepass_d128(const BwdParams& p, const void* o, const void* dout,
                                    float* delta, bool bf16, bool causal, int sms,
                                    cudaStream_t stream);
cudaError_t launch_bwd_onepass_drop_d64(const BwdParams& p, const void* o, const void* dout,
                                        float* delta, bool bf16, bool causal, int sms,
                                        cudaStream_t stream);
cudaError_t launch_bwd_onepass_drop_d128(const BwdParams& p, const void* o, const void* dout,
                                         float* delta, bool bf16, bool causal, int sms,
                                         cudaStream_t stream);
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
