// Self-test of the bounded wait that every kernel's mbarrier waits go through.
// The pages define no such operation: it exists so that the give-up path
// (DUSTIN_DEV_TIMEOUT, the CTA-wide abort flag) runs on a GPU without any
// copy, MMA or peer being left in flight.
//
// One CTA of two warps and one mbarrier that expects one arrival which never
// comes.  Thread 0 waits with the caller's limit and gives up; thread 32 waits
// with the kernels' own limit and must return as soon as thread 0 raises the
// abort flag.  Each records how long it waited.
#include "common.cuh"
#include "kernels.h"

namespace dustin {

namespace {

__global__ void __launch_bounds__(64) wait_selftest_kernel(int* err, long long* waited,
                                                           unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_word;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_word = 0;
    fence_barrier_init();
  }
  __syncthreads();
  volatile int* abort_flag = &abort_word;
  const unsigned long long t0 = globaltimer();
  if (threadIdx.x == 0) {
    const bool ok = mbar_wait(&bar, 0, err, abort_flag, limit_ns);
    waited[0] = ok ? -1 : (long long)(globaltimer() - t0);
  } else if (threadIdx.x == 32) {
    const bool ok = mbar_wait(&bar, 0, err, abort_flag);
    waited[1] = ok ? -1 : (long long)(globaltimer() - t0);
  }
}

}  // namespace

cudaError_t wait_selftest_launch(int* err, long long* waited, unsigned long long limit_ns,
                                 cudaStream_t stream) {
  wait_selftest_kernel<<<1, 64, 0, stream>>>(err, waited, limit_ns);
  return cudaGetLastError();
}

}  // namespace dustin
