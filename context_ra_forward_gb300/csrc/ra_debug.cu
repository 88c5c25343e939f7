// ra_debug.cu — failure-detection self test for the bounded waits.
//
// One block initialises an mbarrier that expects one arrival and then waits on
// it with the same bounded wait the attention kernels use.  Nothing ever
// arrives, so the wait gives up after `limit_us`, records RA_ERR_TIMEOUT in the
// status word and the kernel returns normally: no trap, no fault, no hang.
#include "ra_common.cuh"
#include "ra_kernels.h"

namespace ra {

namespace {

__global__ void debug_wait_kernel(int32_t limit_us, int32_t* status) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  mbar_wait(b, 0, status, kKernDebug, kSiteDebug, (uint64_t)limit_us * 1000ull);
  __syncthreads();
}

}  // namespace

cudaError_t launch_debug_wait(int32_t limit_us, int32_t* status, cudaStream_t st) {
  debug_wait_kernel<<<1, 32, 0, st>>>(limit_us, status);
  note_launch();
  return cudaGetLastError();
}

}  // namespace ra
