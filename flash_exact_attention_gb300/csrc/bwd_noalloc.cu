// bwd_noalloc.cu -- a backward entry point that allocates no device memory.
//
// attn_bwd takes its fp32 scratch (the dQ accumulator and the per-row LSE2 and
// Delta vectors) from the stream-ordered allocator on every call.  Some callers
// cannot allow that: a process that has handed (nearly) all device memory to
// its own pool at start-up, or a serving loop that forbids any allocation after
// initialisation so that its latency never depends on the CUDA allocator.  For
// them, attn_bwd_noalloc runs the very same kernels with the scratch placed in
// one fixed array in device global memory, declared below.
//
// Consequences of a single fixed array:
//   - Problems whose scratch exceeds kNoAllocScratchBytes are rejected with
//     ATTN_ERR_SCRATCH_LIMIT before any device work.
//   - Every call on a device shares the array, and the array keeps whatever the
//     previous call left in it.  The preprocess kernel rewrites every word the
//     call reads (it zeroes the dQ accumulator and writes LSE2 and Delta) before
//     the main kernel runs, so stale contents never leak into results.
//   - Calls that can overlap on the GPU (different streams, or different host
//     threads without ordering) race on the array and give wrong gradients.
//     Order them on one stream, or synchronise between them.
//   - The array occupies device memory on every device where this library's
//     module is loaded, until the process exits.  With lazy module loading
//     (the CUDA default) that happens at the first call into the library on
//     a device; with CUDA_MODULE_LOADING=EAGER the array is reserved when the
//     context is created, whether or not attn_bwd_noalloc is ever called.
//   - The cached address (below) belongs to the device's current context.
//     cudaDeviceReset destroys that context: do not use this library across
//     a cudaDeviceReset (the error word of attn_api.cu is cached the same way).
//   - In host code the array's name is only a host-side stand-in, never a
//     device address.  The first call on each device (with that device current)
//     looks the real address up once with cudaGetSymbolAddress and caches it;
//     make that first call before any stream capture begins on that device.
#include <cstddef>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/attn.h"
#include "kernels.h"

namespace attn {
namespace {

// 32 MiB: enough for B*Hq*roundup(N,128)*(D+2)*4 bytes, e.g. B=1, H=16,
// N=4096, D=64 (17.3 MB) or B=1, H=8, N=8192, D=128 (34.1 MB does NOT fit).
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device (set up once).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr)
      return ATTN_ERR_CUDA;
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return ATTN_OK;
}

}  // namespace

size_t bwd_noalloc_scratch_limit() { return kNoAllocScratchBytes; }

int bwd_noalloc_entry(const void* q, const void* k, const void* v, const void* o,
                      const float* lse, int B, int Hq, int Hkv, int N, int D, int causal,
                      float scale, void* stream, const void* dout, void* dq, void* dk, void* dv) {
  int st = validate_shape(B, Hq, Hkv, N, D, scale);
  if (st != ATTN_OK) return st;
  if ((long long)B * Hq * N == 0) return ATTN_OK;
  if (bwd_scratch_bytes(B, Hq, N, D) > kNoAllocScratchBytes) return ATTN_ERR_SCRATCH_LIMIT;
  BwdParams p;
  CUtensorMap tq, tk, tv, tdo;
  st = bwd_prepare(q, k, v, o, lse, B, Hq, Hkv, N, D, scale, dout, dq, dk, dv, &p, &tq, &tk, &tv,
                   &tdo);
  if (st == -1) return ATTN_OK;
  if (st != ATTN_OK) return st;
  void* ws = nullptr;
  st = scratch_address(&ws);
  if (st != ATTN_OK) return st;
  const BwdScratch sc = carve_scratch(ws, B, Hq, N, D);
  p.dq_acc = sc.dq_acc;
  p.lse2 = sc.lse2;
  p.delta = sc.delta;
  return bwd_launch(tq, tk, tv, tdo, p, o, dout, lse, dq, D, causal,
                    static_cast<cudaStream_t>(stream));
}

}  // namespace attn

extern "C" int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                                const float* lse, int B, int Hq, int Hkv, int N, int D,
                                int causal, float scale, void* stream, const void* dout, void* dq,
                                void* dk, void* dv) {
  return attn::bwd_noalloc_entry(q, k, v, o, lse, B, Hq, Hkv, N, D, causal, scale, stream, dout,
                                 dq, dk, dv);
}

extern "C" long long attn_bwd_noalloc_scratch_limit(void) {
  return (long long)attn::bwd_noalloc_scratch_limit();
}
