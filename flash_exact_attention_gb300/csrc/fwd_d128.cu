// Forward kernels for head dim 128, bf16 inputs and output (causal and non-causal).
#include "fwd_launch.cuh"

namespace attn {
cudaError_t launch_fwd_d128(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const FwdParams& p, bool causal, cudaStream_t stream) {
  // Grids of less than one wave: one query tile per CTA with its key range
  // split over the two slots.
  if (p.kvsplit)
    return causal ? launch_fwd_impl<128, true, false, false, true>(tq, tk, tv, p, stream)
                  : launch_fwd_impl<128, false, false, false, true>(tq, tk, tv, p, stream);
  return causal ? launch_fwd_impl<128, true, false>(tq, tk, tv, p, stream)
                : launch_fwd_impl<128, false, false>(tq, tk, tv, p, stream);
}
}  // namespace attn
