// Self-test of the kernels' bounded waits: one warp waits, through the same
// mbarrier helper the attention kernels use, on a barrier that nothing ever
// arrives on.  The wait must give up after its time limit, record
// kErrWaitTimeout in the error word and return, leaving the context usable.
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "pst_internal.h"

namespace pst {

namespace {

__global__ void __launch_bounds__(32) bounded_wait_kernel(int32_t* err, int32_t* gave_up) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    ptx::fence_mbar_init();
  }
  __syncwarp();
  // phase 0 of a fresh barrier completes only after one arrival, and none comes
  const bool completed = ptx::mbar_wait(&bar, 0, nullptr, err);
  if (!completed) atomicAdd(gave_up, 1);
}

}  // namespace

cudaError_t run_bounded_wait_selftest(int device, int32_t* err_word, int32_t* lanes_gave_up) {
  cudaError_t e = cudaSetDevice(device);
  if (e != cudaSuccess) return e;
  int32_t* d = nullptr;
  if ((e = cudaMalloc(&d, 2 * sizeof(int32_t))) != cudaSuccess) return e;
  cudaStream_t s = nullptr;
  if ((e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking)) == cudaSuccess) {
    int32_t h[2] = {0, 0};
    if ((e = cudaMemsetAsync(d, 0, 2 * sizeof(int32_t), s)) == cudaSuccess) {
      bounded_wait_kernel<<<1, 32, 0, s>>>(d, d + 1);
      if ((e = cudaGetLastError()) == cudaSuccess &&
          (e = cudaMemcpyAsync(h, d, sizeof(h), cudaMemcpyDeviceToHost, s)) == cudaSuccess &&
          (e = cudaStreamSynchronize(s)) == cudaSuccess) {
        *err_word = h[0];
        *lanes_gave_up = h[1];
      }
    }
    cudaStreamDestroy(s);
  }
  cudaFree(d);
  return e;
}

}  // namespace pst
