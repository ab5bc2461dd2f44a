// Stieltjes attention forward kernels for head dim 128 (orders 2 and 4, causal and not).
#include "stj_kernel.cuh"

namespace attn {
namespace {
template <bool CAUSAL, int ORDER>
cudaError_t launch_one(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const FwdParams& p, cudaStream_t stream) {
  using Cfg = StjCfg<128>;
  auto kern = stj_kernel<128, CAUSAL, ORDER>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Cfg::kSmemBytes);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)p.num_qblocks * (unsigned)p.B * (unsigned)p.Hq;
  kern<<<grid, Cfg::kThreads, Cfg::kSmemBytes, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_stj_d128(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const FwdParams& p, bool causal, int order, cudaStream_t stream) {
  if (order == 2)
    return causal ? launch_one<true, 2>(tq, tk, tv, p, stream)
                  : launch_one<false, 2>(tq, tk, tv, p, stream);
  return causal ? launch_one<true, 4>(tq, tk, tv, p, stream)
                : launch_one<false, 4>(tq, tk, tv, p, stream);
}
}  // namespace attn
