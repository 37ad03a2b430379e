// fa_bwd_one_drop_d64.cu — the one-pass backward with dropout for head width 64: bf16/fp16 x causal/unmasked.
#include "fa_bwd_launch.cuh"

namespace fa {

cudaError_t launch_bwd_onepass_drop_d64(const BwdParams& p, const void* o, const void* dout,
                                        float* delta, bool bf16, bool causal, int sms,
                                        cudaStream_t stream) {
  if (causal)
    return bf16 ? launch_bwd_onepass_variant<64, true, true, true>(p, o, dout, delta, sms, stream)
                : launch_bwd_onepass_variant<64, false, true, true>(p, o, dout, delta, sms, stream);
  return bf16 ? launch_bwd_onepass_variant<64, true, false, true>(p, o, dout, delta, sms, stream)
              : launch_bwd_onepass_variant<64, false, false, true>(p, o, dout, delta, sms, stream);
}

}  // namespace fa
