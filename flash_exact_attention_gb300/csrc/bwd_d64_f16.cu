// Backward kernels for head dim 64, fp16 inputs and gradients (causal and non-causal).
#include "bwd_launch.cuh"

namespace attn {
cudaError_t launch_bwd_d64_f16(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const CUtensorMap& tdo, const BwdParams& p, const void* o,
                          const void* dout, const float* lse, void* dq, bool causal,
                          cudaStream_t stream) {
  return causal ? launch_bwd_impl<64, true, true>(tq, tk, tv, tdo, p, o, dout, lse, dq, stream)
                : launch_bwd_impl<64, false, true>(tq, tk, tv, tdo, p, o, dout, lse, dq, stream);
}
}  // namespace attn
