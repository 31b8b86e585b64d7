// selftest.cu -- exercises the failure path of the bounded device-side waits.
//
// Every wait of the fused forward (sm100.cuh: mbar_wait) gives up after about a second, records
// its code in the workspace's error word and returns, so that a lost hand-off becomes
// MLSTM_ERR_TIMEOUT on the host instead of a hung GPU.  This kernel runs that same wait on a
// barrier that nothing ever completes, on one thread of one CTA: it gives up, writes its code
// into the given error word and returns.  Nothing faults, traps or hangs.
#include "common.cuh"
#include "kernels.cuh"
#include "sm100.cuh"

namespace mlstm {

__global__ void wait_selftest_kernel(int *err, int code) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    *(volatile int *)err = 0;
    sm100::mbar_init(&bar, 1);
    sm100::fence_barrier_init();
  }
  __syncthreads();
  // no thread arrives on `bar`: phase 0 never completes
  if (threadIdx.x == 0) sm100::mbar_wait(&bar, 0, err, code);
}

cudaError_t launch_wait_selftest(int *err, int code, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(err, code);
  return cudaGetLastError();
}

}  // namespace mlstm
