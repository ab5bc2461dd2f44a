// Deterministic backward kernels for head dim 128, bf16 (dK/dV without the dQ
// reduce-adds, then dQ per query tile in a fixed order).
#include "bwd_launch.cuh"

namespace attn {
cudaError_t launch_bwd_det_d128(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const CUtensorMap& tdo, const BwdParams& p, const void* o,
                              const void* dout, const float* lse, void* dq, bool causal,
                              cudaStream_t stream) {
  return causal ? launch_bwd_impl<128, true, false, false>(tq, tk, tv, tdo, p, o, dout, lse, dq, stream)
                : launch_bwd_impl<128, false, false, false>(tq, tk, tv, tdo, p, o, dout, lse, dq, stream);
}
}  // namespace attn
