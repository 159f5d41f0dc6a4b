// fa_selftest.cu -- a check of the bounded-wait machinery every kernel uses.
//
// One CTA of two warps waits on mbarriers that nothing ever arrives on, with
// the same helpers the attention kernels use for their pipeline waits:
//   warp 0 waits on barrier A until its time limit (1 s) runs out; it records
//          the timeout with its site id in the status word and raises the
//          CTA's abort flag;
//   warp 1 starts its wait on barrier B a little later and gives up as soon as
//          it sees the abort flag, without a second timeout.
// The kernel then returns normally, so the context stays usable.  The host
// reads the status word through fa_device_status().
#include <cuda_runtime.h>

#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

constexpr unsigned int kSiteSelfTestA = 0x7e;
constexpr unsigned int kSiteSelfTestB = 0x7f;

__global__ void __launch_bounds__(64) fa_selftest_wait_kernel(unsigned int* result) {
  __shared__ uint64_t bar_a, bar_b;
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(&bar_a, 1);
    mbar_init(&bar_b, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  volatile int* abort = &abort_flag;
  bool ok;
  if (warp == 0) {
    ok = mbar_wait_warp(&bar_a, 0, abort, kSiteSelfTestA);
  } else {
    // let warp 0's limit run out first (100 ms of global time, with a spin cap)
    const unsigned long long t0 = global_timer_ns();
    for (uint32_t i = 0; i < (1u << 24) && global_timer_ns() - t0 < 100ull * 1000ull * 1000ull; ++i) {
    }
    ok = mbar_wait_warp(&bar_b, 0, abort, kSiteSelfTestB);
  }
  // result[w] = 1 if warp w's wait reported failure (as it must)
  if ((threadIdx.x & 31) == 0) result[warp] = ok ? 0u : 1u;
}

}  // namespace

cudaError_t launch_selftest_wait(unsigned int* result, cudaStream_t stream) {
  fa_selftest_wait_kernel<<<1, 64, 0, stream>>>(result);
  return cudaGetLastError();
}

unsigned int read_selftest_status(bool clear) {
  unsigned int v = 0;
  cudaMemcpyFromSymbol(&v, g_status, sizeof v);
  if (clear) {
    const unsigned int z = 0;
    cudaMemcpyToSymbol(g_status, &z, sizeof z);
  }
  return v;
}

}  // namespace fa
