// bwd.cu -- backward entry (validation and dispatch).
#include <cuda_runtime.h>
#include "../../include/attn.h"
#include "kernels.h"

namespace attn {

int bwd_entry(const void* q, const void* k, const void* v, const void* o, const float* lse, int B,
              int Hq, int Hkv, int N, int D, int causal, float scale, void* stream,
              const void* dout, void* dq, void* dk, void* dv) {
  (void)q; (void)k; (void)v; (void)o; (void)lse; (void)B; (void)Hq; (void)Hkv; (void)N;
  (void)D; (void)causal; (void)scale; (void)stream; (void)dout; (void)dq; (void)dk; (void)dv;
  return ATTN_ERR_UNSUPPORTED;
}

}  // namespace attn
