// fa_bwd_kv_drop.cu — the backward variants for queries against a key set of
// another length (and packed batches) with dropout in the forward pass:
// widths 64 and 128 x bf16/fp16 x causal/unmasked.
#include "fa_bwd_launch.cuh"

namespace fa {

cudaError_t launch_bwd_kv_drop_d64(const BwdParams& p, const void* o, const void* dout,
                                   float* delta, bool bf16, bool causal, int sms,
                                   cudaStream_t stream) {
  if (causal)
    return bf16 ? launch_bwd_variant<64, true, true, true, true>(p, o, dout, delta, sms, stream)
                : launch_bwd_variant<64, false, true, true, true>(p, o, dout, delta, sms, stream);
  return bf16 ? launch_bwd_variant<64, true, false, true, true>(p, o, dout, delta, sms, stream)
              : launch_bwd_variant<64, false, false, true, true>(p, o, dout, delta, sms, stream);
}

cudaError_t launch_bwd_kv_drop_d128(const BwdParams& p, const void* o, const void* dout,
                                    float* delta, bool bf16, bool causal, int sms,
                                    cudaStream_t stream) {
  if (causal)
    return bf16 ? launch_bwd_variant<128, true, true, true, true>(p, o, dout, delta, sms, stream)
                : launch_bwd_variant<128, false, true, true, true>(p, o, dout, delta, sms, stream);
  return bf16 ? launch_bwd_variant<128, true, false, true, true>(p, o, dout, delta, sms, stream)
              : launch_bwd_variant<128, false, false, true, true>(p, o, dout, delta, sms, stream);
}

}  // namespace fa
