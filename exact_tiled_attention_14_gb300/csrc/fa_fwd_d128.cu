// fa_fwd_d128.cu — the variants for head width 128: bf16/fp16 x (causal, unmasked,
// unmasked with a split tail), and the variants for a key set of another length
// (causal or not).
#include "fa_launch.cuh"

namespace fa {

cudaError_t launch_fwd_d128(const FwdParams& p, int grid, bool bf16, bool causal,
                           cudaStream_t stream) {
  if (causal)
    return bf16 ? launch_variant<128, true, true, false>(p, grid, stream)
                : launch_variant<128, false, true, false>(p, grid, stream);
  if (p.split)
    return bf16 ? launch_variant<128, true, false, true>(p, grid, stream)
                : launch_variant<128, false, false, true>(p, grid, stream);
  return bf16 ? launch_variant<128, true, false, false>(p, grid, stream)
              : launch_variant<128, false, false, false>(p, grid, stream);
}

cudaError_t launch_fwd_kv_d128(const FwdParams& p, int grid, bool bf16, bool causal,
                               cudaStream_t stream) {
  if (causal)
    return bf16 ? launch_variant<128, true, true, false, true>(p, grid, stream)
                : launch_variant<128, false, true, false, true>(p, grid, stream);
  return bf16 ? launch_variant<128, true, false, false, true>(p, grid, stream)
              : launch_variant<128, false, false, false, true>(p, grid, stream);
}

}  // namespace fa
