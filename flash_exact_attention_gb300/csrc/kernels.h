// kernels.h -- internal interface between the C-ABI layer (attn_api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace attn {

// Forward kernel parameters (everything but the tensor maps).
struct FwdParams {
  void* o;              // bf16 [B, Hq, N, D]
  float* lse;           // fp32 [B, Hq, N]
  int B, Hq, Hkv, N;
  int G;                // Hq / Hkv
  int num_qblocks;      // ceil(N / 256): CTAs per (batch, head)
  int num_kv_tiles;     // ceil(N / 128)
  float scale_log2;     // scale * log2(e)
  uint64_t timeout_ns;  // limit of every device-side wait
  unsigned int* err;    // device error word
};

// Each launcher enqueues one forward kernel; returns the launch's cudaError_t.
cudaError_t launch_fwd_d64(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const FwdParams& p, bool causal, cudaStream_t stream);
cudaError_t launch_fwd_d128(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const FwdParams& p, bool causal, cudaStream_t stream);

// Entry points behind the C ABI (attn_api.cu, bwd.cu).
int bwd_entry(const void* q, const void* k, const void* v, const void* o, const float* lse, int B,
              int Hq, int Hkv, int N, int D, int causal, float scale, void* stream,
              const void* dout, void* dq, void* dk, void* dv);

}  // namespace attn
