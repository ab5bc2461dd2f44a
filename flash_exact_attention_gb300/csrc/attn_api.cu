// attn_api.cu -- the C ABI of libattn.so (declared in include/attn.h): argument
// validation, TMA tensor-map encoding, kernel dispatch and device status.
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/attn.h"
#include "kernels.h"
#include "ptx.cuh"

namespace attn {

// One error word per device that loads this library.  Kernels receive its
// address as a parameter; the host reads and clears it in attn_device_status.
__device__ unsigned int g_error_word;

namespace {

constexpr int kMaxDevices = 64;

// Signature of the driver's cuTensorMapEncodeTiled (fetched at run time so
// that the library does not link against libcuda directly).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

std::mutex g_mu;
EncodeTiledFn g_encode = nullptr;
unsigned int* g_err_ptr[kMaxDevices] = {};
int g_arch_ok[kMaxDevices] = {};  // 0 unknown, 1 ok, -1 wrong arch
int g_num_sms[kMaxDevices] = {};
uint64_t g_timeout_ns = 2000ull * 1000ull * 1000ull;

}  // namespace

uint64_t wait_timeout_ns() {
  std::lock_guard<std::mutex> lock(g_mu);
  return g_timeout_ns;
}

// Per-device setup: architecture check and the address of the error word.
int device_setup(int* dev_out, unsigned int** err_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_arch_ok[dev] == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return ATTN_ERR_CUDA;
    g_arch_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return ATTN_ERR_CUDA;
    g_num_sms[dev] = sms;
  }
  if (g_arch_ok[dev] < 0) return ATTN_ERR_ARCH;
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return ATTN_ERR_CUDA;
    g_err_ptr[dev] = static_cast<unsigned int*>(p);
  }
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return ATTN_ERR_CUDA;
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  *dev_out = dev;
  *err_out = g_err_ptr[dev];
  return ATTN_OK;
}

int device_sm_count(int dev) {
  std::lock_guard<std::mutex> lock(g_mu);
  return (dev >= 0 && dev < kMaxDevices) ? g_num_sms[dev] : 0;
}

// 3-D map over a contiguous bf16 (or fp16) [BH, N, D] tensor: dims (D, N, BH), box
// (64, box_rows, 1) (128 rows unless a caller asks for fewer), 128-byte swizzle.  Rows past N inside a (batch, head) plane
// read as zero, so a ragged tail never reads the next head.
int encode_tile_map(CUtensorMap* map, const void* base, int D, int N, int BH, bool f16,
                    int box_rows) {
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)N * D * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                        3, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

// 3-D map over a packed token-major bf16 [total, H, D] tensor: dims
// (D, H, total), box (64, 1, 128) -- 128 tokens of one head, 128-byte rows --
// with 128-byte swizzle, so a tile lands in shared memory exactly as a tile of
// the dense map does.  Tokens past `total` read as zero (and are not written
// by a store or reduce-add).  f32: an fp32 [total, H, D] tensor, box
// (32, 1, 128) -- the packed dQ accumulator of the variable-length backward.
int encode_packed_map(CUtensorMap* map, const void* base, int D, int H, int total, bool f32) {
  const cuuint64_t es = f32 ? 4 : 2;  // element bytes; a box row is 128 bytes either way
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)total};
  cuuint64_t strides[2] = {(cuuint64_t)D * es, (cuuint64_t)H * D * es};
  cuuint32_t box[3] = {f32 ? 32u : 64u, 1, 128};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                        3, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

// 3-D map over a contiguous fp32 [BH, rows, D] array: dims (D, rows, BH), box
// (32, 128, 1) (128-byte rows), 128-byte swizzle.  Used for the dQ reduce-add.
int encode_f32_rows_map(CUtensorMap* map, const void* base, int D, int rows, int BH) {
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)rows, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)D * 4, (cuuint64_t)rows * D * 4};
  cuuint32_t box[3] = {32, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

// Shape / scale checks shared by the forward and backward.
int validate_shape(int B, int Hq, int Hkv, int N, int D, float scale) {
  if (B < 0 || N < 0 || Hq <= 0 || Hkv <= 0) return ATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (!(std::isfinite(scale) && scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  // Element offsets use 64-bit arithmetic; grid size and TMA plane counts are
  // 32-bit.  (B*Hq) * ceil(N/256) CTAs must fit the grid's x dimension.
  const long long bh = (long long)B * Hq;
  const long long qblocks = ((long long)N + 255) / 256;
  if (bh * qblocks * 2 > 0x7FFFFFFFll || bh > 0x7FFFFFFFll) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}


int fwd_entry(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
              int Hkv, int N, int D, int causal, float scale, void* stream, bool f16) {
  int st = validate_shape(B, Hq, Hkv, N, D, scale);
  if (st != ATTN_OK) return st;
  if ((long long)B * Hq * N == 0) return ATTN_OK;
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return ATTN_ERR_INVALID_ARG;
  int dev = 0;
  unsigned int* err = nullptr;
  st = device_setup(&dev, &err);
  if (st != ATTN_OK) return st;

  CUtensorMap tq, tk, tv;
  if (encode_tile_map(&tq, q, D, N, B * Hq, f16) != ATTN_OK ||
      encode_tile_map(&tk, k, D, N, B * Hkv, f16) != ATTN_OK ||
      encode_tile_map(&tv, v, D, N, B * Hkv, f16) != ATTN_OK)
    return ATTN_ERR_CUDA;

  FwdParams p;
  p.o = o;
  p.lse = lse;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.N = N;
  p.G = Hq / Hkv;
  p.num_qblocks = ((N + 127) / 128 + 1) / 2;
  // Less than one wave of tile pairs: one query tile per CTA, its key range
  // split over the two slots -- when causal (LPT over single tiles of about
  // half the steps) and when one tile per CTA still fits in a wave.
  {
    const long long tiles = (long long)((N + 127) / 128) * B * Hq;
    const int sms = device_sm_count(dev);
    p.kvsplit = ((long long)p.num_qblocks * B * Hq < sms) && (causal != 0 || tiles <= sms);
    p.ctas = sms;
  }
  p.num_kv_tiles = (N + 127) / 128;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.timeout_ns = wait_timeout_ns();
  p.err = err;
  p.scale = scale;
  p.steps = 0;
  p.cu_seqlens = nullptr;
  p.total = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool c = causal != 0;
  cudaError_t e = f16 ? ((D == 64) ? launch_fwd_d64_f16(tq, tk, tv, p, c, s)
                                   : launch_fwd_d128_f16(tq, tk, tv, p, c, s))
                      : ((D == 64) ? launch_fwd_d64(tq, tk, tv, p, c, s)
                                   : launch_fwd_d128(tq, tk, tv, p, c, s));
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int fwd_varlen_entry(const void* q, const void* k, const void* v, void* o, float* lse,
                     const int* cu_seqlens, int B, int Hq, int Hkv, int total, int max_seqlen,
                     int D, int causal, float scale, void* stream, bool f16) {
  if (total < 0 || max_seqlen < 0) return ATTN_ERR_INVALID_ARG;
  int st = validate_shape(B, Hq, Hkv, max_seqlen, D, scale);
  if (st != ATTN_OK) return st;
  if (B == 0 || total == 0 || max_seqlen == 0) return ATTN_OK;
  if (!q || !k || !v || !o || !lse || !cu_seqlens) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(cu_seqlens) & 3u) != 0) return ATTN_ERR_INVALID_ARG;
  int dev = 0;
  unsigned int* err = nullptr;
  st = device_setup(&dev, &err);
  if (st != ATTN_OK) return st;
  CUtensorMap tq, tk, tv;
  if (encode_packed_map(&tq, q, D, Hq, total) != ATTN_OK ||
      encode_packed_map(&tk, k, D, Hkv, total) != ATTN_OK ||
      encode_packed_map(&tv, v, D, Hkv, total) != ATTN_OK)
    return ATTN_ERR_CUDA;
  FwdParams p;
  p.o = o;
  p.lse = lse;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.N = max_seqlen;
  p.G = Hq / Hkv;
  p.num_qblocks = ((max_seqlen + 127) / 128 + 1) / 2;
  p.kvsplit = 0;
  p.num_kv_tiles = (max_seqlen + 127) / 128;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.timeout_ns = wait_timeout_ns();
  p.err = err;
  p.scale = scale;
  p.steps = 0;
  p.cu_seqlens = cu_seqlens;
  p.total = total;
  p.ctas = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool c = causal != 0;
  // (the packed maps only copy 16-bit elements: the same for bf16 and fp16)
  cudaError_t e = f16 ? ((D == 64) ? launch_fwd_varlen_d64_f16(tq, tk, tv, p, c, s)
                                   : launch_fwd_varlen_d128_f16(tq, tk, tv, p, c, s))
                      : ((D == 64) ? launch_fwd_varlen_d64(tq, tk, tv, p, c, s)
                                   : launch_fwd_varlen_d128(tq, tk, tv, p, c, s));
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int stj_entry(const void* q, const void* k, const void* v, void* o, float* pole, int B, int Hq,
              int Hkv, int N, int D, int causal, float scale, int order, int steps,
              void* stream) {
  int st = validate_shape(B, Hq, Hkv, N, D, scale);
  if (st != ATTN_OK) return st;
  if (order != 2 && order != 4) return ATTN_ERR_UNSUPPORTED;
  if (steps < 1 || steps > 64) return ATTN_ERR_INVALID_ARG;
  if ((long long)B * Hq * N == 0) return ATTN_OK;
  if (!q || !k || !v || !o || !pole) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(pole))
    return ATTN_ERR_INVALID_ARG;
  int dev = 0;
  unsigned int* err = nullptr;
  st = device_setup(&dev, &err);
  if (st != ATTN_OK) return st;
  CUtensorMap tq, tk, tv;
  if (encode_tile_map(&tq, q, D, N, B * Hq) != ATTN_OK ||
      encode_tile_map(&tk, k, D, N, B * Hkv) != ATTN_OK ||
      encode_tile_map(&tv, v, D, N, B * Hkv) != ATTN_OK)
    return ATTN_ERR_CUDA;
  FwdParams p;
  p.o = o;
  p.lse = pole;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.N = N;
  p.G = Hq / Hkv;
  p.num_qblocks = ((N + 127) / 128 + 1) / 2;
  p.kvsplit = 0;
  p.num_kv_tiles = (N + 127) / 128;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.timeout_ns = wait_timeout_ns();
  p.err = err;
  p.scale = scale;
  p.steps = steps;
  p.cu_seqlens = nullptr;
  p.total = 0;
  p.ctas = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = (D == 64) ? launch_stj_d64(tq, tk, tv, p, causal != 0, order, s)
                            : launch_stj_d128(tq, tk, tv, p, causal != 0, order, s);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int device_status(void* stream) {
  int dev = 0;
  unsigned int* err = nullptr;
  int st = device_setup(&dev, &err);
  if (st != ATTN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return ATTN_ERR_CUDA;
  unsigned int word = 0;
  if (cudaMemcpyAsync(&word, err, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaMemsetAsync(err, 0, sizeof(word), s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (word & kErrTimeout) return ATTN_ERR_DEVICE_TIMEOUT;
  return word ? ATTN_ERR_INVALID_ARG : ATTN_OK;  // kErrSeqlen: bad cu_seqlens / max_seqlen
}

int set_wait_timeout_ms(int ms) {
  if (ms < 1) return ATTN_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mu);
  g_timeout_ns = (uint64_t)ms * 1000000ull;
  return ATTN_OK;
}

}  // namespace attn

extern "C" {

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
             int Hkv, int N, int D, int causal, float scale, void* stream) {
  return attn::fwd_entry(q, k, v, o, lse, B, Hq, Hkv, N, D, causal, scale, stream);
}

int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, int B,
             int Hq, int Hkv, int N, int D, int causal, float scale, void* stream,
             const void* dout, void* dq, void* dk, void* dv) {
  return attn::bwd_entry(q, k, v, o, lse, B, Hq, Hkv, N, D, causal, scale, stream, dout, dq, dk,
                         dv);
}

int attn_fwd_f16(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                 int Hkv, int N, int D, int causal, float scale, void* stream) {
  return attn::fwd_entry(q, k, v, o, lse, B, Hq, Hkv, N, D, causal, scale, stream, true);
}

int attn_bwd_f16(const void* q, const void* k, const void* v, const void* o, const float* lse,
                 int B, int Hq, int Hkv, int N, int D, int causal, float scale, void* stream,
                 const void* dout, void* dq, void* dk, void* dv) {
  return attn::bwd_entry(q, k, v, o, lse, B, Hq, Hkv, N, D, causal, scale, stream, dout, dq, dk,
                         dv, true);
}

int attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                    const int* cu_seqlens, int B, int Hq, int Hkv, int total, int max_seqlen,
                    int D, int causal, float scale, void* stream) {
  return attn::fwd_varlen_entry(q, k, v, o, lse, cu_seqlens, B, Hq, Hkv, total, max_seqlen, D,
                                causal, scale, stream);
}

int attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const float* lse,
                    const int* cu_seqlens, int B, int Hq, int Hkv, int total, int max_seqlen,
                    int D, int causal, float scale, void* stream, const void* dout, void* dq,
                    void* dk, void* dv) {
  return attn::bwd_varlen_entry(q, k, v, o, lse, cu_seqlens, B, Hq, Hkv, total, max_seqlen, D,
                                causal, scale, stream, dout, dq, dk, dv);
}

int attn_fwd_varlen_f16(const void* q, const void* k, const void* v, void* o, float* lse,
                        const int* cu_seqlens, int B, int Hq, int Hkv, int total, int max_seqlen,
                        int D, int causal, float scale, void* stream) {
  return attn::fwd_varlen_entry(q, k, v, o, lse, cu_seqlens, B, Hq, Hkv, total, max_seqlen, D,
                                causal, scale, stream, true);
}

int attn_bwd_varlen_f16(const void* q, const void* k, const void* v, const void* o,
                        const float* lse, const int* cu_seqlens, int B, int Hq, int Hkv,
                        int total, int max_seqlen, int D, int causal, float scale, void* stream,
                        const void* dout, void* dq, void* dk, void* dv) {
  return attn::bwd_varlen_entry(q, k, v, o, lse, cu_seqlens, B, Hq, Hkv, total, max_seqlen, D,
                                causal, scale, stream, dout, dq, dk, dv, true);
}

int attn_stieltjes_fwd(const void* q, const void* k, const void* v, void* o, float* pole, int B,
                       int Hq, int Hkv, int N, int D, int causal, float scale, int order,
                       int newton_steps, void* stream) {
  return attn::stj_entry(q, k, v, o, pole, B, Hq, Hkv, N, D, causal, scale, order, newton_steps,
                         stream);
}

int attn_bwd_deterministic(const void* q, const void* k, const void* v, const void* o,
                           const float* lse, int B, int Hq, int Hkv, int N, int D, int causal,
                           float scale, void* stream, const void* dout, void* dq, void* dk,
                           void* dv) {
  return attn::bwd_entry(q, k, v, o, lse, B, Hq, Hkv, N, D, causal, scale, stream, dout, dq, dk,
                         dv, false, true);
}

const char* attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported configuration (head dim must be 64 or 128)";
    case ATTN_ERR_CUDA: return "CUDA call or kernel launch failed";
    case ATTN_ERR_DEVICE_TIMEOUT: return "a bounded device-side wait ran out";
    case ATTN_ERR_ARCH: return "device is not compute capability 10.3 (GB300)";
    case ATTN_ERR_SCRATCH_LIMIT:
      return "problem needs more scratch than attn_bwd_noalloc's fixed array holds";
    default: return "unknown status";
  }
}

int attn_device_status(void* stream) { return attn::device_status(stream); }

int attn_set_wait_timeout_ms(int ms) { return attn::set_wait_timeout_ms(ms); }

int attn_version(void) { return (1 << 16) | 0; }

}  // extern "C"
