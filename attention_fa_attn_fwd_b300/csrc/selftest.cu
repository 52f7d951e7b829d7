// attn_selftest_wait_timeout: exercises the bounded-wait path every kernel of
// this library relies on, without faulting or hanging the GPU.
//
// One warp initialises an mbarrier that nothing will ever arrive at and waits
// on it with the same bounded wait the kernels use (mbar_wait_limit), but with
// a short limit.  The wait gives up, raises the CTA's abort flag and records
// kErrTimeoutSelftest in a device error word; the kernel then returns.  The
// host call reads the word back: finding the code proves that an expired wait
// is detected, reported and survived (the context stays usable).

#include <cstdio>

#include "attn_b300.h"
#include "attn_internal.h"
#include "ptx.cuh"

namespace attn {

__device__ int g_selftest_error[2];  // see ErrSink

namespace {

__global__ void __launch_bounds__(32) wait_timeout_selftest_kernel(uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar_storage;
  __shared__ int abort_flag;
  const uint32_t bar = smem_u32(&bar_storage);
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncwarp();
  // Nothing arrives on `bar`: this wait must give up after limit_ns.
  const ErrSink err{g_selftest_error, 1u};
  const bool ok = mbar_wait_limit(bar, 0, &abort_flag, err, kErrTimeoutSelftest, limit_ns);
  if (ok && threadIdx.x == 0) atomicExch(&g_selftest_error[0], -1);  // must not happen
}

}  // namespace
}  // namespace attn

extern "C" attn_status attn_selftest_wait_timeout(unsigned limit_us, attn_stream_t stream) {
  if (limit_us < 1 || limit_us > 1000000u) {
    attn::set_last_error("attn_selftest_wait_timeout: limit_us must be in [1, 1e6]");
    return ATTN_EINVAL;
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int zero = 0;
  cudaError_t e = cudaMemcpyToSymbolAsync(attn::g_selftest_error, &zero, sizeof(int), 0,
                                          cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) {
    attn::wait_timeout_selftest_kernel<<<1, 32, 0, st>>>(uint64_t(limit_us) * 1000ull);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  int word = 0;
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&word, attn::g_selftest_error, sizeof(int));
  if (e != cudaSuccess) {
    attn::set_last_error("attn_selftest_wait_timeout: %s", cudaGetErrorString(e));
    return ATTN_ECUDA;
  }
  if (word != attn::kErrTimeoutSelftest) {
    attn::set_last_error("attn_selftest_wait_timeout: device word 0x%x, expected 0x%x", word,
                         attn::kErrTimeoutSelftest);
    return ATTN_EDEVICE;
  }
  return ATTN_OK;
}
