// fa_fwd_drop.cu — the forward variants with dropout on the attention
// weights: widths 64 and 128 x bf16/fp16 x causal/unmasked.
#include "fa_launch.cuh"

namespace fa {

cudaError_t launch_fwd_drop_d64(const FwdParams& p, int grid, bool bf16, bool causal,
                                cudaStream_t stream) {
  if (causal)
    return bf16 ? launch_variant<64, true, true, false, true, true>(p, grid, stream)
                : launch_variant<64, false, true, false, true, true>(p, grid, stream);
  return bf16 ? launch_variant<64, true, false, false, true, true>(p, grid, stream)
              : launch_variant<64, false, false, false, true, true>(p, grid, stream);
}

cudaError_t launch_fwd_drop_d128(const FwdParams& p, int grid, bool bf16, bool causal,
                                 cudaStream_t stream) {
  if (causal)
    return bf16 ? launch_variant<128, true, true, false, true, true>(p, grid, stream)
                : launch_variant<128, false, true, false, true, true>(p, grid, stream);
  return bf16 ? launch_variant<128, true, false, false, true, true>(p, grid, stream)
              : launch_variant<128, false, false, false, true, true>(p, grid, stream);
}

}  // namespace fa
