// bwd.cu -- the backward entry point: validation, stream-ordered fp32 scratch,
// tensor maps and the three kernel launches.
#include <cuda_runtime.h>
#include "../../include/attn.h"
#include "kernels.h"

namespace attn {

void bwd_order(BwdParams* p, long long units, int tiles, double unit_bytes, int sms) {
  // Plain j order while the units are few: the ~sms/units CTAs of a unit that
  // are resident together walk its query tiles a step apart, so each Q, dO
  // and dQ tile is used several times while it is in L2.
  p->band = units < 1 ? 1 : (int)units;
  p->jchunks = 1;
  const double budget = 80.0 * 1024 * 1024;  // query-side bytes kept in L2 (of 126 MB)
  if (units * 4 <= sms || (double)units * unit_bytes <= budget) return;
  const long long want = (2LL * sms + tiles - 1) / tiles;  // about two waves of CTAs
  long long b = (long long)(budget / unit_bytes);
  if (b > want) b = want;
  if (b < 1) b = 1;
  if (b > units) b = units;
  p->band = (int)b;
  p->jchunks = tiles >= 2 ? 2 : 1;
}

size_t bwd_scratch_bytes(int B, int Hq, int N, int D) {
  const size_t npad = ((size_t)N + 127) / 128 * 128;
  const size_t rows = (size_t)B * Hq * npad;
  return rows * (size_t)D * 4 + 2 * rows * 4;  // dQ accumulator, LSE2, Delta
}

size_t bwd_scratch_bytes_split(int B, int Hq, int Hkv, int N, int D, int gsplit) {
  const size_t npad = ((size_t)N + 127) / 128 * 128;
  const size_t kv = gsplit > 1 ? 2 * (size_t)B * Hkv * npad * (size_t)D * 4 : 0;
  return bwd_scratch_bytes(B, Hq, N, D) + kv;
}

BwdScratch carve_scratch_split(void* base, int B, int Hq, int Hkv, int N, int D, int gsplit) {
  BwdScratch s = carve_scratch(base, B, Hq, N, D);
  if (gsplit > 1) {
    const size_t npad = ((size_t)N + 127) / 128 * 128;
    s.dk_acc = s.delta + (size_t)B * Hq * npad;
    s.dv_acc = s.dk_acc + (size_t)B * Hkv * npad * D;
  }
  return s;
}

BwdScratch carve_scratch(void* base, int B, int Hq, int N, int D) {
  const size_t npad = ((size_t)N + 127) / 128 * 128;
  const size_t rows = (size_t)B * Hq * npad;
  BwdScratch s;
  s.dq_acc = static_cast<float*>(base);
  s.lse2 = s.dq_acc + rows * D;
  s.delta = s.lse2 + rows;
  s.dk_acc = nullptr;
  s.dv_acc = nullptr;
  return s;
}

// Validates everything that can be checked on the host; returns ATTN_OK and
// fills *params (except scratch pointers) and the tensor maps.
int bwd_prepare(const void* q, const void* k, const void* v, const void* o,
                       const float* lse, int B, int Hq, int Hkv, int N, int D, float scale,
                       const void* dout, void* dq, void* dk, void* dv, BwdParams* p,
                       CUtensorMap* tq, CUtensorMap* tk, CUtensorMap* tv, CUtensorMap* tdo,
                       bool allow_split, bool f16) {
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
  if (encode_tile_map(tq, q, D, N, B * Hq, f16) != ATTN_OK ||
      encode_tile_map(tk, k, D, N, B * Hkv, f16) != ATTN_OK ||
      encode_tile_map(tv, v, D, N, B * Hkv, f16) != ATTN_OK ||
      encode_tile_map(tdo, dout, D, N, B * Hq, f16) != ATTN_OK)
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
  // One CTA per (key tile, batch, kv head) keeps a whole GQA group's dK/dV in
  // TMEM.  When that grid is shorter than one wave, split the group's query
  // heads over gsplit CTAs (the smallest divisor of G that fills the GPU).
  p->gsplit = 1;
  p->dk_acc = nullptr;
  p->dv_acc = nullptr;
  p->cu_seqlens = nullptr;
  p->total = 0;
  const long long ctas = (long long)p->num_kv_tiles * B * Hkv;
  const int sms = device_sm_count(dev);
  if (allow_split && p->G > 1 && ctas < sms) {
    int g = p->G;
    for (int d = 2; d <= p->G; ++d)
      if (p->G % d == 0 && ctas * d >= sms) {
        g = d;
        break;
      }
    p->gsplit = g;
  }
  // Per unit: Gs query heads of N rows of Q and dO (bf16) and the fp32 dQ
  // accumulator.
  bwd_order(p, (long long)B * Hkv * p->gsplit, p->num_kv_tiles,
            (double)(p->G / p->gsplit) * N * D * 8.0, sms);
  return ATTN_OK;
}

int bwd_launch(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                      const CUtensorMap& tdo, const BwdParams& p, const void* o, const void* dout,
                      const float* lse, void* dq, int D, int causal, cudaStream_t s, bool f16,
                      bool det) {
  const bool c = causal != 0;
  cudaError_t e =
      det ? ((D == 64) ? launch_bwd_det_d64(tq, tk, tv, tdo, p, o, dout, lse, dq, c, s)
                       : launch_bwd_det_d128(tq, tk, tv, tdo, p, o, dout, lse, dq, c, s)) :
      f16 ? ((D == 64) ? launch_bwd_d64_f16(tq, tk, tv, tdo, p, o, dout, lse, dq, c, s)
                       : launch_bwd_d128_f16(tq, tk, tv, tdo, p, o, dout, lse, dq, c, s))
          : ((D == 64) ? launch_bwd_d64(tq, tk, tv, tdo, p, o, dout, lse, dq, c, s)
                       : launch_bwd_d128(tq, tk, tv, tdo, p, o, dout, lse, dq, c, s));
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int bwd_entry(const void* q, const void* k, const void* v, const void* o, const float* lse, int B,
              int Hq, int Hkv, int N, int D, int causal, float scale, void* stream,
              const void* dout, void* dq, void* dk, void* dv, bool f16, bool det) {
  BwdParams p;
  CUtensorMap tq, tk, tv, tdo;
  int st = bwd_prepare(q, k, v, o, lse, B, Hq, Hkv, N, D, scale, dout, dq, dk, dv, &p, &tq, &tk,
                       &tv, &tdo, /*allow_split=*/!det, f16);
  if (st == -1) return ATTN_OK;
  if (st != ATTN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* ws = nullptr;
  // The deterministic backward needs only LSE2 and Delta (no dQ accumulator).
  const size_t rows = (size_t)B * Hq * (size_t)p.Npad;
  const size_t bytes = det ? 2 * rows * 4 : bwd_scratch_bytes_split(B, Hq, Hkv, N, D, p.gsplit);
  if (cudaMallocAsync(&ws, bytes, s) != cudaSuccess) return ATTN_ERR_CUDA;
  BwdScratch sc = carve_scratch_split(ws, B, Hq, Hkv, N, D, p.gsplit);
  if (det) {
    sc.dq_acc = nullptr;
    sc.lse2 = static_cast<float*>(ws);
    sc.delta = sc.lse2 + rows;
  }
  p.dq_acc = sc.dq_acc;
  p.lse2 = sc.lse2;
  p.delta = sc.delta;
  p.dk_acc = sc.dk_acc;
  p.dv_acc = sc.dv_acc;
  st = bwd_launch(tq, tk, tv, tdo, p, o, dout, lse, dq, D, causal, s, f16, det);
  if (cudaFreeAsync(ws, s) != cudaSuccess && st == ATTN_OK) st = ATTN_ERR_CUDA;
  return st;
}

int bwd_varlen_entry(const void* q, const void* k, const void* v, const void* o,
                     const float* lse, const int* cu_seqlens, int B, int Hq, int Hkv, int total,
                     int max_seqlen, int D, int causal, float scale, void* stream,
                     const void* dout, void* dq, void* dk, void* dv, bool f16) {
  if (total < 0 || max_seqlen < 0) return ATTN_ERR_INVALID_ARG;
  int st = validate_shape(B, Hq, Hkv, max_seqlen, D, scale);
  if (st != ATTN_OK) return st;
  if (B == 0 || total == 0 || max_seqlen == 0) return ATTN_OK;
  const void* ptrs[] = {q, k, v, o, lse, dout, dq, dk, dv};
  for (const void* ptr : ptrs)
    if (!ptr || !aligned16(ptr)) return ATTN_ERR_INVALID_ARG;
  if (!cu_seqlens || (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u) != 0)
    return ATTN_ERR_INVALID_ARG;
  int dev = 0;
  unsigned int* err = nullptr;
  st = device_setup(&dev, &err);
  if (st != ATTN_OK) return st;
  CUtensorMap tq, tk, tv, tdo, tdq;
  if (encode_packed_map(&tq, q, D, Hq, total) != ATTN_OK ||
      encode_packed_map(&tk, k, D, Hkv, total) != ATTN_OK ||
      encode_packed_map(&tv, v, D, Hkv, total) != ATTN_OK ||
      encode_packed_map(&tdo, dout, D, Hq, total) != ATTN_OK)
    return ATTN_ERR_CUDA;
  BwdParams p;
  p.dk = dk;
  p.dv = dv;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.N = max_seqlen;
  p.Npad = (max_seqlen + 127) / 128 * 128;
  p.G = Hq / Hkv;
  p.num_kv_tiles = (max_seqlen + 127) / 128;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.timeout_ns = wait_timeout_ns();
  p.err = err;
  p.gsplit = 1;
  p.dk_acc = nullptr;
  p.dv_acc = nullptr;
  p.cu_seqlens = cu_seqlens;
  p.total = total;
  {
    // Bands sized for the mean sequence length.
    const double mean_len = (double)total / B > 1.0 ? (double)total / B : 1.0;
    const int mean_tiles = (int)((mean_len + 127.0) / 128.0);
    bwd_order(&p, (long long)B * Hkv, mean_tiles, (double)p.G * mean_len * D * 8.0,
              device_sm_count(dev));
    // The grid walks max_seqlen's key tiles: at most one range per tile.
    if (p.jchunks > p.num_kv_tiles) p.jchunks = p.num_kv_tiles;
  }
  // Scratch: the packed fp32 dQ accumulator [total, Hq, D], then LSE2 and
  // Delta [B*Hq, Npad] (every part a multiple of 512 bytes long).
  const size_t acc = (size_t)total * Hq * D * 4;
  const size_t rows = (size_t)B * Hq * (size_t)p.Npad;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* ws = nullptr;
  if (cudaMallocAsync(&ws, acc + 2 * rows * 4, s) != cudaSuccess) return ATTN_ERR_CUDA;
  p.dq_acc = static_cast<float*>(ws);
  p.lse2 = reinterpret_cast<float*>(static_cast<char*>(ws) + acc);
  p.delta = p.lse2 + rows;
  if (encode_packed_map(&tdq, p.dq_acc, D, Hq, total, /*f32=*/true) != ATTN_OK) {
    cudaFreeAsync(ws, s);
    return ATTN_ERR_CUDA;
  }
  const bool c = causal != 0;
  // (the packed maps only copy 16-bit elements: the same for bf16 and fp16)
  cudaError_t e =
      f16 ? ((D == 64) ? launch_bwd_varlen_d64_f16(tq, tk, tv, tdo, tdq, p, o, dout, lse, dq, c, s)
                       : launch_bwd_varlen_d128_f16(tq, tk, tv, tdo, tdq, p, o, dout, lse, dq, c, s))
          : ((D == 64) ? launch_bwd_varlen_d64(tq, tk, tv, tdo, tdq, p, o, dout, lse, dq, c, s)
                       : launch_bwd_varlen_d128(tq, tk, tv, tdo, tdq, p, o, dout, lse, dq, c, s));
  st = e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
  if (cudaFreeAsync(ws, s) != cudaSuccess && st == ATTN_OK) st = ATTN_ERR_CUDA;
  return st;
}

}  // namespace attn
