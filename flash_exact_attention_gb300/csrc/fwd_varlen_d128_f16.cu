// Packed variable-length forward kernels for head dim 128 (fp16, causal and not).
#include "fwd_launch.cuh"

namespace attn {
cudaError_t launch_fwd_varlen_d128_f16(const CUtensorMap& tq, const CUtensorMap& tk,
                                      const CUtensorMap& tv, const FwdParams& p, bool causal,
                                      cudaStream_t stream) {
  return causal ? launch_fwd_impl<128, true, true, true>(tq, tk, tv, p, stream)
                : launch_fwd_impl<128, false, true, true>(tq, tk, tv, p, stream);
}
}  // namespace attn
