// Packed variable-length backward kernels for head dim 128 (fp16, causal and not).
#include "bwd_launch.cuh"

namespace attn {
cudaError_t launch_bwd_varlen_d128_f16(const CUtensorMap& tq, const CUtensorMap& tk,
                                      const CUtensorMap& tv, const CUtensorMap& tdo,
                                      const CUtensorMap& tdq, const BwdParams& p, const void* o,
                                      const void* dout, const float* lse, void* dq, bool causal,
                                      cudaStream_t stream) {
  return causal
      ? launch_bwd_varlen_impl<128, true, true>(tq, tk, tv, tdo, tdq, p, o, dout, lse, dq, stream)
      : launch_bwd_varlen_impl<128, false, true>(tq, tk, tv, tdo, tdq, p, o, dout, lse, dq, stream);
}
}  // namespace attn
