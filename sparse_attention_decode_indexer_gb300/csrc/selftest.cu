// selftest.cu -- ssa_selftest_bounded_wait: proof that a lost mbarrier
// arrival ends in a status bit, not a hang.
//
// One CTA initialises an mbarrier that expects one arrival, never arrives on
// it, and waits with the same bounded wait every kernel of the library uses
// (wall-clock limit kWaitLimitNs).  The wait gives up, the kernel records
// SSA_ST_TIMEOUT in the caller's status word and returns normally, leaving
// the context usable.
#include "common.cuh"
#include "internal.h"

namespace ssa {
namespace {

__global__ void bounded_wait_kernel(int32_t* status) {
  __shared__ uint64_t bar;
  __shared__ int never;                 // the abort flag nothing sets
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    never = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait(&bar, 0, &never)) set_status(status, SSA_ST_TIMEOUT);
}

}  // namespace
}  // namespace ssa

extern "C" int ssa_selftest_bounded_wait(int32_t* status, ssa_stream_t stream) {
  if (!status) return SSA_ERR_INVALID_ARG;
  ssa::bounded_wait_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(status);
  ssa::count_launch();
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? SSA_OK : ssa::record_cuda_error(e);
}
