// nys.cu -- host side of the Nystrom attention forward (attn_nystrom_fwd):
// validation, work split, stream-ordered scratch and the tensor maps of the
// six kernels in nys_kernel.cuh.
#include <cmath>
#include <cstdint>

#include "../../include/attn.h"
#include "kernels.h"

namespace attn {
namespace {
size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
}  // namespace

int nys_entry(const void* q, const void* k, const void* v, void* o, int B, int Hq, int Hkv, int N,
              int D, int m, int iters, float kappa, float scale, void* stream) {
  int st = validate_shape(B, Hq, Hkv, N, D, scale);
  if (st != ATTN_OK) return st;
  if (m < 1 || iters < 0 || iters > 100 || !std::isfinite(kappa) || kappa < 0.f)
    return ATTN_ERR_INVALID_ARG;
  if (m > 64) return ATTN_ERR_UNSUPPORTED;
  if ((long long)B * Hq == 0) return ATTN_OK;
  if (N < m) return ATTN_ERR_INVALID_ARG;
  if ((long long)B * (Hq + Hkv) > 65535) return ATTN_ERR_INVALID_ARG;
  if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
    return ATTN_ERR_INVALID_ARG;
  int dev = 0;
  unsigned int* err = nullptr;
  st = device_setup(&dev, &err);
  if (st != ATTN_OK) return st;
  const int sms = device_sm_count(dev);

  NysParams p;
  p.q = q;
  p.k = k;
  p.o = o;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.N = N;
  p.G = Hq / Hkv;
  p.m = m;
  p.mp = m <= 16 ? 16 : (m + 15) / 16 * 16;
  p.iters = iters;
  p.kappa = kappa;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.num_kv_tiles = (N + 127) / 128;
  const long long BH = (long long)B * Hq, BHk = (long long)B * Hkv, T = p.num_kv_tiles;
  // Q pooling: at least four full waves of 256-thread CTAs (eight per SM),
  // splits of at least 128 rows, at most 64 splits.
  {
    const long long units = BH * m;
    long long s = (32LL * sms + units - 1) / units;
    const long long cap = (long long)(N / m) / 128;
    if (s > cap) s = cap;
    if (s > 64) s = 64;
    if (s < 1) s = 1;
    p.pool_splits = (int)s;
  }
  // Split-key pass (one CTA per SM): the chunk count C that minimises the
  // tiles on the critical path, waves(C) * (ceil(T / C) + 2), two tiles being
  // about a CTA's start-up and drain; ties go to fewer chunks.
  {
    long long best_c = 1, best = -1;
    for (long long c = 1; c <= T && c <= 4096; ++c) {
      const long long waves = (BH * c + sms - 1) / sms;
      const long long cost = waves * ((T + c - 1) / c + 2);
      if (best < 0 || cost < best) {
        best = cost;
        best_c = c;
      }
    }
    const long long tpc = (T + best_c - 1) / best_c;
    p.kv_tpc = (int)tpc;
    p.kv_chunks = (int)((T + tpc - 1) / tpc);
  }
  // K-sum slots of a segment: the chunks one landmark segment meets, at most,
  // times the row shares of a key tile (4 at D = 64, 2 at D = 128).
  {
    const long long rows = (long long)p.kv_tpc * 128;
    long long parts = 1;
    for (int i = 0; i < m; ++i) {
      const long long lo = (long long)i * N / m, hi = (long long)(i + 1) * N / m;
      const long long c = (hi - 1) / rows - lo / rows + 1;
      if (c > parts) parts = c;
    }
    p.kparts = (int)parts * (D == 64 ? 4 : 2);
  }
  p.out_ctas = (int)(BH * T < sms ? BH * T : sms);
  p.timeout_ns = wait_timeout_ns();
  p.err = err;

  const size_t b_pool = align256((size_t)BH * m * p.pool_splits * D * 4);
  const size_t b_qt32 = align256((size_t)BH * m * D * 4);
  const size_t b_kpart = align256((size_t)BHk * m * p.kparts * D * 4);
  const size_t b_qt = align256((size_t)BH * 2 * 128 * D * 2);
  const size_t b_kt = align256((size_t)BHk * 2 * p.mp * D * 2);
  const size_t b_y = align256((size_t)BH * 2 * p.mp * D * 2);
  const size_t b_kvo = align256((size_t)BH * p.kv_chunks * m * D * 4);
  const size_t b_kvml = align256((size_t)BH * p.kv_chunks * m * 2 * 4);
  const size_t b_w = align256((size_t)BH * m * D * 4);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* ws = nullptr;
  if (cudaMallocAsync(&ws, b_pool + b_qt32 + b_kpart + b_qt + b_kt + b_y + b_kvo + b_kvml + b_w,
                      s) != cudaSuccess)
    return ATTN_ERR_CUDA;
  uint8_t* w = static_cast<uint8_t*>(ws);
  p.pool_part = reinterpret_cast<float*>(w);
  w += b_pool;
  p.qt32 = reinterpret_cast<float*>(w);
  w += b_qt32;
  p.kpart = reinterpret_cast<float*>(w);
  w += b_kpart;
  p.qt16 = reinterpret_cast<uint16_t*>(w);
  w += b_qt;
  p.kt16 = reinterpret_cast<uint16_t*>(w);
  w += b_kt;
  p.y16 = reinterpret_cast<uint16_t*>(w);
  w += b_y;
  p.kv_o = reinterpret_cast<float*>(w);
  w += b_kvo;
  p.kv_ml = reinterpret_cast<float*>(w);
  w += b_kvml;
  p.w = reinterpret_cast<float*>(w);

  CUtensorMap tq, tk, tv, tqt, tkt, ty, to;
  if (encode_tile_map(&tq, q, D, N, (int)BH) != ATTN_OK ||
      encode_tile_map(&to, o, D, N, (int)BH) != ATTN_OK ||
      encode_tile_map(&tk, k, D, N, (int)BHk) != ATTN_OK ||
      encode_tile_map(&tv, v, D, N, (int)BHk) != ATTN_OK ||
      encode_tile_map(&tqt, p.qt16, D, 256, (int)BH) != ATTN_OK ||
      encode_tile_map(&tkt, p.kt16, D, 2 * p.mp, (int)BHk, false, p.mp) != ATTN_OK ||
      encode_tile_map(&ty, p.y16, D, 2 * p.mp, (int)BH, false, p.mp) != ATTN_OK) {
    st = ATTN_ERR_CUDA;
  } else {
    // K-sum slots that no (chunk, share) pair writes must read as zero
    cudaError_t e = cudaMemsetAsync(p.kpart, 0, b_kpart, s);
    if (e == cudaSuccess)
      e = (D == 64) ? launch_nys_d64(tq, tk, tv, tqt, tkt, ty, to, p, s)
                              : launch_nys_d128(tq, tk, tv, tqt, tkt, ty, to, p, s);
    st = e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
  }
  if (cudaFreeAsync(ws, s) != cudaSuccess && st == ATTN_OK) st = ATTN_ERR_CUDA;
  return st;
}

}  // namespace attn

extern "C" int attn_nystrom_fwd(const void* q, const void* k, const void* v, void* o, int B,
                                int Hq, int Hkv, int N, int D, int num_landmarks,
                                int newton_iters, float kappa, float scale, void* stream) {
  return attn::nys_entry(q, k, v, o, B, Hq, Hkv, N, D, num_landmarks, newton_iters, kappa, scale,
                         stream);
}
