// selftest.cu -- exercises the failure-detection path of the bounded waits.
//
// Every kernel of this library waits on mbarriers with a wall-clock limit; a
// wait that runs out sets the device error word, the kernel leaves cleanly and
// attn_device_status() reports ATTN_ERR_DEVICE_TIMEOUT.  The probe below makes
// exactly that happen on purpose: one thread waits for the first phase of an
// mbarrier that nothing ever arrives on.  No fault, trap or unbounded loop is
// involved: the wait gives up after `timeout_ns`.
#include <cuda_runtime.h>

#include "../../include/attn.h"
#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace {

__global__ void wait_timeout_probe(uint64_t timeout_ns, unsigned int* err) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 1);
  abort_flag = 0;
  fence_barrier_init();
  const WaitCtl wc{timeout_ns, err, &abort_flag};
  // Phase 0 of a fresh barrier completes only after one arrival: never here.
  mbar_wait(b, 0, wc);
}

}  // namespace

int selftest_wait_timeout(int timeout_ms, void* stream) {
  if (timeout_ms < 1 || timeout_ms > 10000) return ATTN_ERR_INVALID_ARG;
  int dev = 0;
  unsigned int* err = nullptr;
  int st = device_setup(&dev, &err);
  if (st != ATTN_OK) return st;
  wait_timeout_probe<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(
      (uint64_t)timeout_ms * 1000000ull, err);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace attn

extern "C" int attn_selftest_wait_timeout(int timeout_ms, void* stream) {
  return attn::selftest_wait_timeout(timeout_ms, stream);
}
