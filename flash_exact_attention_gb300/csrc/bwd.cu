// bwd.cu -- the backward entry point: validation, stream-ordered fp32 scratch,
// tensor maps and the three kernel launches.
#include <cuda_runtime.h>
#include "../../include/attn.h"
#include "kernels.h"

namespace attn {

size_t bwd_scratch_bytes(int B, int Hq, int N, int D) {
  const size_t npad = ((size_t)N + 127) / 128 * 128;
  const size_t rows = (size_t)B * Hq * npad;
  return rows * (size_t)D * 4 + 2 * rows * 4;  // dQ accumulator, LSE2, Delta
}

BwdScratch carve_scratch(void* base, int B, int Hq, int N, int D) {
  const size_t npad = ((size_t)N + 127) / 128 * 128;
  const size_t rows = (size_t)B * Hq * npad;
  BwdScratch s;
  s.dq_acc = static_cast<float*>(base);
  s.lse2 = s.dq_acc + rows * D;
  s.delta = s.lse2 + rows;
  return s;
}

// Validates everything that can be checked on the host; returns ATTN_OK and
// fills *params (except scratch pointers) and the tensor maps.
int bwd_prepare(const void* q, const void* k, const void* v, const void* o,
                       const float* lse, int B, int Hq, int Hkv, int N, int D, float scale,
                       const void* dout, void* dq, void* dk, void* dv, BwdParams* p,
                       CUtensorMap* tq, CUtensorMap* tk, CUtensorMap* tv, CUtensorMap* tdo) {
  int st = validate_shape(B, Hq, Hkv, N, D, scale);
  if (st != ATTN_OK) return st;
  if ((long long)B * Hq * N == 0) return -1;  // nothing to do
  const void* ptrs[] = {q, k, v, o, lse, dout, dq, dk, dv};
  for (const void* ptr : ptrs)
    if (!ptr || !aligned16(ptr)) return ATTN_ERR_INVALID_ARG;
  int dev = 0;
  unsigned int* err = nullptr;
  st = device_setup(&dev, &err);
  if (st != ATTN_OK) return st;
  if (encode_tile_map(tq, q, D, N, B * Hq) != ATTN_OK ||
      encode_tile_map(tk, k, D, N, B * Hkv) != ATTN_OK ||
      encode_tile_map(tv, v, D, N, B * Hkv) != ATTN_OK ||
      encode_tile_map(tdo, dout, D, N, B * Hq) != ATTN_OK)
    return ATTN_ERR_CUDA;
  p->dk = dk;
  p->dv = dv;
  p->B = B;
  p->Hq = Hq;
  p->Hkv = Hkv;
  p->N = N;
  p->Npad = (N + 127) / 128 * 128;
  p->G = Hq / Hkv;
  p->num_kv_tiles = (N + 127) / 128;
  p->scale = scale;
  p->scale_log2 = scale * 1.4426950408889634f;
  p->timeout_ns = wait_timeout_ns();
  p->err = err;
  return ATTN_OK;
}

int bwd_launch(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                      const CUtensorMap& tdo, const BwdParams& p, const void* o, const void* dout,
                      const float* lse, void* dq, int D, int causal, cudaStream_t s) {
  cudaError_t e = (D == 64) ? launch_bwd_d64(tq, tk, tv, tdo, p, o, dout, lse, dq, causal != 0, s)
                            : launch_bwd_d128(tq, tk, tv, tdo, p, o, dout, lse, dq, causal != 0, s);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int bwd_entry(const void* q, const void* k, const void* v, const void* o, const float* lse, int B,
              int Hq, int Hkv, int N, int D, int causal, float scale, void* stream,
              const void* dout, void* dq, void* dk, void* dv) {
  BwdParams p;
  CUtensorMap tq, tk, tv, tdo;
  int st = bwd_prepare(q, k, v, o, lse, B, Hq, Hkv, N, D, scale, dout, dq, dk, dv, &p, &tq, &tk,
                       &tv, &tdo);
  if (st == -1) return ATTN_OK;
  if (st != ATTN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* ws = nullptr;
  if (cudaMallocAsync(&ws, bwd_scratch_bytes(B, Hq, N, D), s) != cudaSuccess) return ATTN_ERR_CUDA;
  const BwdScratch sc = carve_scratch(ws, B, Hq, N, D);
  p.dq_acc = sc.dq_acc;
  p.lse2 = sc.lse2;
  p.delta = sc.delta;
  st = bwd_launch(tq, tk, tv, tdo, p, o, dout, lse, dq, D, causal, s);
  if (cudaFreeAsync(ws, s) != cudaSuccess && st == ATTN_OK) st = ATTN_ERR_CUDA;
  return st;
}

}  // namespace attn
