// Nystrom attention forward kernels for head dim 128.
#include "nys_kernel.cuh"

namespace attn {

cudaError_t launch_nys_d128(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const CUtensorMap& tqt, const CUtensorMap& tkt, const CUtensorMap& ty,
                          const CUtensorMap& to, const NysParams& p, cudaStream_t stream) {
  constexpr int D = 128;
  const int BH = p.B * p.Hq;
  cudaError_t e;
  nys_pool_kernel<D><<<dim3(p.pool_splits, p.m, BH), 256, 0, stream>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // Qt: four columns per thread for a few splits, one for many
  if (p.pool_splits < 8)
    nys_qt_kernel<D, 4><<<dim3(128 * D / 4 / kNysSmallThreads, BH), kNysSmallThreads, 0,
                          stream>>>(p);
  else
    nys_qt_kernel<D, 1><<<dim3(128, BH), D, 0, stream>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  e = cudaFuncSetAttribute(nys_kv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           NysKvCfg<D>::kSmemBytes);
  if (e != cudaSuccess) return e;
  nys_kv_kernel<D><<<dim3(p.kv_chunks, BH), NysKvCfg<D>::kThreads, NysKvCfg<D>::kSmemBytes,
                     stream>>>(tqt, tk, tv, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  // merge: one chunk group per thread for a few chunks, four for many
  if (p.kv_chunks <= 4)
    nys_merge_kernel<D, 1><<<dim3((p.m * D / 4 + kNysSmallThreads - 1) / kNysSmallThreads, BH),
                             kNysSmallThreads, 0, stream>>>(p);
  else
    nys_merge_kernel<D, 4><<<dim3((p.m * D + kNysSmallThreads - 1) / kNysSmallThreads, BH),
                             kNysSmallThreads, 0, stream>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  e = cudaFuncSetAttribute(nys_lmy_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           NysLyCfg<D>::kSmemBytes);
  if (e != cudaSuccess) return e;
  nys_lmy_kernel<D><<<BH, NysLyCfg<D>::kThreads, NysLyCfg<D>::kSmemBytes, stream>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  e = cudaFuncSetAttribute(nys_out_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           NysOutCfg<D>::kSmemBytes);
  if (e != cudaSuccess) return e;
  nys_out_kernel<D><<<p.out_ctas, NysOutCfg<D>::kThreads, NysOutCfg<D>::kSmemBytes, stream>>>(
      tq, tkt, ty, to, p);
  return cudaGetLastError();
}

}  // namespace attn
