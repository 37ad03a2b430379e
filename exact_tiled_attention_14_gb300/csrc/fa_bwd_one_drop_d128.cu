// fa_bwd_one_drop_d128.cu — the one-pass backward with dropout for head width 128: bf16/fp16 x causal/unmasked.
#include "fa_bwd_launch.cuh"

namespace fa {

cudaError_t launch_bwd_onepass_drop_d128(const BwdParams& p, const void* o, const void* dout,
                                         float* delta, bool bf16, bool causal, int sms,
                                         cudaStream_t stream) {
  if (causal)
    return bf16 ? launch_bwd_onepass_variant<128, true, true, true>(p, o, dout, delta, sms, stream)
                : launch_bwd_onepass_variant<128, false, true, true>(p, o, dout, delta, sms, stream);
  return bf16 ? launch_bwd_onepass_variant<128, true, false, true>(p, o, dout, delta, sms, stream)
              : launch_bwd_onepass_variant<128, false, false, true>(p, o, dout, delta, sms, stream);
}

}  // namespace fa
