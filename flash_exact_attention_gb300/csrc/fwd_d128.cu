// Forward kernels for head dim 128 (causal and non-causal).
#include "fwd_launch.cuh"

namespace attn {
cudaError_t launch_fwd_d128(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const FwdParams& p, bool causal, cudaStream_t stream) {
  return causal ? launch_fwd_impl<128, true>(tq, tk, tv, p, stream)
                : launch_fwd_impl<128, false>(tq, tk, tv, p, stream);
}
}  // namespace attn
