// bwd_launch.cuh -- host-side launch of the three backward kernels for one head dim.
#pragma once
#include "bwd_kernel.cuh"
#include "bwd_dq_kernel.cuh"

namespace attn {

// DQ = false: the deterministic backward (dK/dV kernel, then bwd_dq_kernel).
template <int D, bool CAUSAL, bool F16, bool DQ = true>
cudaError_t launch_bwd_impl(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const BwdParams& p, const void* o,
                            const void* dout, const float* lse, void* dq, cudaStream_t stream) {
  using Cfg = BwdCfg<D>;
  // The fp32 dQ accumulator, target of the TMA reduce-add (none without DQ: the
  // kernel then never touches the map, which is left a copy of a valid one).
  CUtensorMap tdq = tq;
  if (DQ && encode_f32_rows_map(&tdq, p.dq_acc, D, p.Npad, p.B * p.Hq) != 0)
    return cudaErrorInvalidValue;
  // Group split: the fp32 dK/dV accumulators (else unused: any valid map).
  CUtensorMap tdk = tdq, tdv = tdq;
  const bool split = p.gsplit > 1;
  if (split && (encode_f32_rows_map(&tdk, p.dk_acc, D, p.Npad, p.B * p.Hkv) != 0 ||
                encode_f32_rows_map(&tdv, p.dv_acc, D, p.Npad, p.B * p.Hkv) != 0))
    return cudaErrorInvalidValue;
  const long long prow = (long long)p.B * p.Hq * p.Npad;  // padded rows
  const long long kv_rows = split ? (long long)p.B * p.Hkv * p.Npad : 0;
  constexpr long long kPreRows = pre_rows_per_cta<D>();
  bwd_preprocess<D, F16><<<(unsigned)((prow + kPreRows - 1) / kPreRows), 256, 0, stream>>>(
      static_cast<const uint16_t*>(o), static_cast<const uint16_t*>(dout), lse,
      const_cast<float*>(p.lse2), const_cast<float*>(p.delta), p.dq_acc, prow, p.N, p.Npad,
      p.dk_acc, p.dv_acc, kv_rows);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  auto kern = bwd_kernel<D, CAUSAL, F16, DQ>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)p.num_kv_tiles * (unsigned)(p.B * p.Hkv) * (unsigned)p.gsplit;
  kern<<<grid, Cfg::kThreads, Cfg::kSmemBytes, stream>>>(tq, tk, tv, tdo, tdq, tdk, tdv, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long orow = (long long)p.B * p.Hq * p.N;
  if (DQ) {
    const long long groups = orow * (D / 8);
    bwd_postprocess<D, F16><<<(unsigned)((groups + 255) / 256), 256, 0, stream>>>(
        p.dq_acc, static_cast<uint16_t*>(dq), orow, p.N, p.Npad, p.scale);
  } else {
    using DCfg = DqCfg<D>;
    auto dkern = bwd_dq_kernel<D, CAUSAL, F16>;
    e = cudaFuncSetAttribute(dkern, cudaFuncAttributeMaxDynamicSharedMemorySize, DCfg::kSmemBytes);
    if (e != cudaSuccess) return e;
    const unsigned dgrid = (unsigned)p.num_kv_tiles * (unsigned)(p.B * p.Hq);
    dkern<<<dgrid, DCfg::kThreads, DCfg::kSmemBytes, stream>>>(tq, tk, tv, tdo, p,
                                                               static_cast<uint16_t*>(dq));
  }
  if (split) {
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const long long kvrow = (long long)p.B * p.Hkv * p.N;
    const long long kvgroups = kvrow * (D / 8);
    bwd_post_kv<D, F16><<<(unsigned)((kvgroups + 255) / 256), 256, 0, stream>>>(
        p.dk_acc, p.dv_acc, static_cast<uint16_t*>(p.dk), static_cast<uint16_t*>(p.dv),
        kvrow, p.N, p.Npad, p.scale);
  }
  return cudaGetLastError();
}

// Packed variable-length backward: LSE2/Delta into padded rows, the main
// kernel (dQ partials reduce-added into the packed fp32 accumulator p.dq_acc,
// zeroed here), then dQ = scale * dQacc.  p.N is max_seqlen.
template <int D, bool CAUSAL, bool F16 = false>
cudaError_t launch_bwd_varlen_impl(const CUtensorMap& tq, const CUtensorMap& tk,
                                   const CUtensorMap& tv, const CUtensorMap& tdo,
                                   const CUtensorMap& tdq, const BwdParams& p, const void* o,
                                   const void* dout, const float* lse, void* dq,
                                   cudaStream_t stream) {
  using Cfg = BwdCfg<D>;
  const long long qrows = (long long)p.total * p.Hq;  // packed dQ rows
  cudaError_t e = cudaMemsetAsync(p.dq_acc, 0, (size_t)qrows * D * 4, stream);
  if (e != cudaSuccess) return e;
  const long long prow = (long long)p.B * p.Hq * p.Npad;
  constexpr long long kPreRows = pre_rows_per_cta<D>();
  bwd_preprocess_varlen<D, F16><<<(unsigned)((prow + kPreRows - 1) / kPreRows), 256, 0,
                                  stream>>>(
      static_cast<const uint16_t*>(o), static_cast<const uint16_t*>(dout), lse, p.cu_seqlens,
      const_cast<float*>(p.lse2), const_cast<float*>(p.delta), prow, p.Hq, p.Npad, p.N, p.total);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  auto kern = bwd_kernel<D, CAUSAL, F16, true, true>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)p.num_kv_tiles * (unsigned)(p.B * p.Hkv);
  // No group split: the dK/dV accumulator maps are never read (any valid map).
  kern<<<grid, Cfg::kThreads, Cfg::kSmemBytes, stream>>>(tq, tk, tv, tdo, tdq, tdq, tdq, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // dQacc and dq have the same packed row order: one "row" of length 1 per
  // (token, head).
  const long long groups = qrows * (D / 8);
  bwd_postprocess<D, F16><<<(unsigned)((groups + 255) / 256), 256, 0, stream>>>(
      p.dq_acc, static_cast<uint16_t*>(dq), qrows, 1, 1, p.scale);
  return cudaGetLastError();
}

}  // namespace attn
