// k_debug.cu -- check of the bounded device-side waits: one thread waits on a
// shared-memory barrier that nothing ever arrives at.  The wait gives up after
// the limit, records TP_ERR_TIMEOUT in the status word, and the kernel returns.
#include "ptx.cuh"
#include "tp_internal.h"

namespace tp {

__global__ void debug_wait_kernel(int64_t limit_ns, int *status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // Phase 0 never completes: the single expected arrival never happens.
    mbar_wait(smem_u32(&bar), 0, (uint64_t)limit_ns, status, &abort_flag);
  }
  __syncthreads();
}

int launch_debug_wait(int64_t limit_ns, int *status, cudaStream_t s) {
  debug_wait_kernel<<<1, 32, 0, s>>>(limit_ns, status);
  note_launch();
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? TP_OK : cuda_error(e, "debug_wait_kernel launch");
}

}  // namespace tp
