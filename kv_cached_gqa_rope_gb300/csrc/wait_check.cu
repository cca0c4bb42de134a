// A check of the library's bounded waits on the GPU: one CTA holds tensor
// memory and waits on an mbarrier that nothing ever arrives on, with the same
// wait primitive the kernels use (mbar_wait_bounded).  The wait gives up after
// its bound, sets KVGQA_FLAG_TIMEOUT in the status word and the CTA's abort
// flag; the other warp, waiting on the same barrier, sees the abort flag and
// gives up too; the CTA frees its tensor memory and returns.  Nothing faults
// and nothing spins without limit, so the context stays usable: this is how a
// kernel of this library ends when a copy or an MMA it waits for never
// completes.
#include <cuda_runtime.h>

#include "kvgqa_internal.h"
#include "tcgen05.cuh"

namespace kvgqa {
namespace {

__global__ void __launch_bounds__(64, 1) bounded_wait_check_kernel(int32_t* status) {
  __shared__ __align__(8) uint64_t never;  // no thread or copy ever arrives on it
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(&never, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_slot, 32);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  volatile int* abort = &abort_flag;
  // Warp 0 runs into the limit; warp 1 polls with a long suspend hint and
  // leaves once warp 0 has flagged the abort.
  const bool ok = warp == 0 ? mbar_wait_bounded(&never, 0, abort, status)
                            : mbar_wait_bounded(&never, 0, abort, status, 1000);
  (void)ok;  // false on every thread: nothing arrives
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 32);
}

}  // namespace

cudaError_t launch_bounded_wait_check(int32_t* status, cudaStream_t stream) {
  bounded_wait_check_kernel<<<1, 64, 0, stream>>>(status);
  return cudaGetLastError();
}

}  // namespace kvgqa
