// Self-test of the library's failure path: a kernel whose mbarrier wait can
// never complete.  The wait is the same bounded wait every tensor-core kernel
// uses; it gives up after its bound, sets the timeout bit of the device error
// word and returns, so the host sees SEMMOE_ERR_DEVICE_TIMEOUT from
// semmoe_check_errors() and the context stays usable.
#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace semmoe {
namespace {

__device__ int g_err;

__global__ void bounded_wait_kernel() {
  __shared__ uint64_t bar;
  __shared__ int abort_s;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);
    tc::mbar_init_fence();
    abort_s = 0;
  }
  __syncthreads();
  if (threadIdx.x == 0) tc::mbar_wait(&bar, 0, &abort_s, &g_err);  // nothing ever arrives
  __syncthreads();
}

}  // namespace

int selftest_take_errors(cudaStream_t s, int* bits) { return take_error_word(g_err, s, bits); }

cudaError_t launch_selftest_bounded_wait(cudaStream_t s) {
  bounded_wait_kernel<<<1, 32, 0, s>>>();
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace semmoe
