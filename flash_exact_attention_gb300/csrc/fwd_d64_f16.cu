// Forward kernels for head dim 64, fp16 inputs and output (causal and non-causal).
#include "fwd_launch.cuh"

namespace attn {
cudaError_t launch_fwd_d64_f16(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const FwdParams& p, bool causal, cudaStream_t stream) {
  // A causal grid of less than one wave (zigzag pairs) is bound by the
  // latency of one K/V step: P in columns of its own shortens it.
  if (causal && p.zigzag) return launch_fwd_impl<64, true, true, false, true>(tq, tk, tv, p, stream);
  return causal ? launch_fwd_impl<64, true, true>(tq, tk, tv, p, stream)
                : launch_fwd_impl<64, false, true>(tq, tk, tv, p, stream);
}
}  // namespace attn
