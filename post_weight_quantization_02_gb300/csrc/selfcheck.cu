// gptq_check_wait_timeout: a self-check of the failure path that every bounded device
// wait of the library takes.
//
// The tensor-core kernels wait on mbarriers with tc::mbar_wait, which gives up after a
// time limit, records GPTQ_ERR_TIMEOUT in the call's status word and lets the kernel
// return, so that a wait that can never be satisfied ends the call with an error instead
// of hanging the device.  Making a real kernel's wait run out would leave its copies and
// matrix operations in flight; this check instead runs the same wait on an mbarrier that
// nothing ever arrives on, in a kernel that has nothing else in flight, and reports what
// the wait did through the same status word and host path as every other call.
#include <cuda_runtime.h>

#include "common.cuh"
#include "tc_common.cuh"

namespace gptq {
namespace {

__global__ void wait_timeout_kernel(DevStatus* st, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);  // one arrival completes phase 0; none ever comes
    abort_flag = 0;
    tc::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !tc::mbar_wait(&bar, 0, &abort_flag, limit_ns)) {
    dev_fail(st, GPTQ_ERR_TIMEOUT, 0);
    atomicAdd(&st->timeouts, 1);
  }
}

}  // namespace

void launch_wait_timeout(DevStatus* st, uint64_t limit_ns, cudaStream_t s) {
  GPTQ_LAUNCH(GPTQ_K_SELFCHECK, s, wait_timeout_kernel, 1, 32, 0, st, limit_ns);
}

}  // namespace gptq
