// diag.cu -- self-check of the bounded wait the attention kernels use: one CTA waits on
// an mbarrier that nothing ever arrives at, so the wait must give up after its limit,
// record REC_ATTN_ERR_TIMEOUT in a status word and return, leaving the context usable.
#include <cuda_runtime.h>

#include "launchers.cuh"
#include "wait.cuh"

namespace recattn {

namespace {

__global__ void k_wait_timeout(int* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    abort_flag = 0;
    ptx::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) bounded_wait(&bar, 0, &abort_flag, status, limit_ns);  // no arrival ever comes
}

}  // namespace

cudaError_t launch_wait_timeout(int* status, unsigned long long limit_ns, cudaStream_t st) {
  k_wait_timeout<<<1, 32, 0, st>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace recattn
