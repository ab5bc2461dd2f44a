// fwd_launch.cuh -- host-side launch of fwd_kernel (one grid per call).
#pragma once
#include "fwd_kernel.cuh"

namespace attn {

template <int D, bool CAUSAL, bool F16, bool VARLEN = false, bool KVSPLIT = false>
cudaError_t launch_fwd_impl(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const FwdParams& p, cudaStream_t stream) {
  using Cfg = FwdCfg<D>;
  const unsigned per_head = KVSPLIT ? (unsigned)p.num_kv_tiles : (unsigned)p.num_qblocks;
  const unsigned units = per_head * (unsigned)p.B * (unsigned)p.Hq;
  // The split-key mode with more units than SMs: persistent CTAs (one per SM,
  // each walking its units); otherwise one CTA per unit.
  const bool persist = KVSPLIT && p.ctas > 0 && (unsigned)p.ctas < units;
  auto kern = persist ? fwd_kernel<D, CAUSAL, F16, VARLEN, KVSPLIT, KVSPLIT>
                      : fwd_kernel<D, CAUSAL, F16, VARLEN, KVSPLIT, false>;
  // Attributes are per device; setting them on every call is cheap and keeps
  // multi-device processes correct.
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Cfg::kSmemBytes);
  if (e != cudaSuccess) return e;
  const unsigned grid = persist ? (unsigned)p.ctas : units;
  kern<<<grid, Cfg::kThreads, Cfg::kSmemBytes, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace attn
