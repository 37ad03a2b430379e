// fa_fwd_d64.cu — the four variants (bf16/fp16 x causal/unmasked) for head width 64.
#include "fa_launch.cuh"

namespace fa {

cudaError_t launch_fwd_d64(const FwdParams& p, int grid, bool bf16, bool causal,
                           cudaStream_t stream) {
  if (bf16)
    return causal ? launch_variant<64, true, true>(p, grid, stream)
                  : launch_variant<64, true, false>(p, grid, stream);
  return causal ? launch_variant<64, false, true>(p, grid, stream)
                : launch_variant<64, false, false>(p, grid, stream);
}

}  // namespace fa
