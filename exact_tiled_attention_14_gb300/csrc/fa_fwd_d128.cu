// fa_fwd_d128.cu — the four variants (bf16/fp16 x causal/unmasked) for head width 128.
#include "fa_launch.cuh"

namespace fa {

cudaError_t launch_fwd_d128(const FwdParams& p, int grid, bool bf16, bool causal,
                           cudaStream_t stream) {
  if (bf16)
    return causal ? launch_variant<128, true, true>(p, grid, stream)
                  : launch_variant<128, true, false>(p, grid, stream);
  return causal ? launch_variant<128, false, true>(p, grid, stream)
                : launch_variant<128, false, false>(p, grid, stream);
}

}  // namespace fa
