// fa_decode.cu — launches of the split-KV decoding kernels (both head widths).
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "fa_decode_kernel.cuh"

namespace fa {

namespace {

template <int D, int NQ, bool kBf16>
cudaError_t launch_partial(const DecodeParams& p, cudaStream_t stream) {
  static std::atomic<uint64_t> done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(done.load() & bit)) {
    e = cudaFuncSetAttribute(fa_decode_partial_kernel<D, NQ, kBf16>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, DecSmem<D, NQ>::kAlloc);
    if (e != cudaSuccess) return e;
    done.fetch_or(bit);
  }
  fa_decode_partial_kernel<D, NQ, kBf16>
      <<<p.BH * p.splits, kDecThreads, DecSmem<D, NQ>::kAlloc, stream>>>(p);
  return cudaGetLastError();
}

// The partial kernel compiled for the smallest query-slot count >= Nq.
template <int D, bool kBf16>
cudaError_t launch_decode_variant(const DecodeParams& p, void* o, float* lse, cudaStream_t stream) {
  if (p.splits > 0) {
    cudaError_t e;
    if (p.Nq <= 1) e = launch_partial<D, 1, kBf16>(p, stream);
    else if (p.Nq <= 2) e = launch_partial<D, 2, kBf16>(p, stream);
    else if (p.Nq <= 4) e = launch_partial<D, 4, kBf16>(p, stream);
    else if (p.Nq <= 8) e = launch_partial<D, 8, kBf16>(p, stream);
    else e = launch_partial<D, 16, kBf16>(p, stream);
    if (e != cudaSuccess) return e;
  }
  // Programmatic dependent launch: the combine grid is set up while the
  // partial kernel runs its last CTAs and waits on the device for its parts.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.BH * p.Nq));
  cfg.blockDim = dim3(D);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fa_decode_combine_kernel<D, kBf16>, p.part_o, p.part_ml, o, lse,
                            p.splits, p.Nq);
}

}  // namespace

cudaError_t launch_decode(const DecodeParams& p, void* o, float* lse, int d, bool bf16,
                          cudaStream_t stream) {
  if (d == 64)
    return bf16 ? launch_decode_variant<64, true>(p, o, lse, stream)
                : launch_decode_variant<64, false>(p, o, lse, stream);
  return bf16 ? launch_decode_variant<128, true>(p, o, lse, stream)
              : launch_decode_variant<128, false>(p, o, lse, stream);
}

}  // namespace fa
