// Self-test of the bounded wait that every kernel of the library uses on its
// own asynchronous work (TMA copies, tensor-core commits): a wait on an
// mbarrier that nothing arrives on gives up after `polls` polls, records
// kDevErrTimeout in the device error word and returns.  That is the path a
// kernel takes, instead of spinning forever, if its copies or MMAs never
// complete; the test shows the status reaches the host and the context stays
// usable, without faulting or hanging the GPU.
// Self-test of the bounds guard: one guard on element 1 of a one-element
// buffer, and no memory access at all.  In the bounds-checked build it
// records kDevErrBounds; in the normal build the guard is compiled out and the
// kernel does nothing, so the test tells which build is loaded.
#include <cuda_runtime.h>

#include "kda_internal.h"
#include "kda_sm100.cuh"

namespace kda {

namespace {

__global__ void bounded_wait_kernel(uint32_t polls, int* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    sm100::mbar_init(&bar, 1);  // one arrival expected; none is made
    sm100::mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !sm100::mbar_wait(&bar, 0, polls)) atomicOr(err, kDevErrTimeout);
}

__global__ void bounds_guard_kernel(int* err) {
  if (threadIdx.x == 0) (void)kda_guard(1, 1, 1, err);
}

}  // namespace

cudaError_t launch_bounds_guard_selftest(int* err, cudaStream_t s) {
  bounds_guard_kernel<<<1, 32, 0, s>>>(err);
  return cudaGetLastError();
}

cudaError_t launch_bounded_wait_selftest(uint32_t polls, int* err, cudaStream_t s) {
  bounded_wait_kernel<<<1, 32, 0, s>>>(polls, err);
  return cudaGetLastError();
}

}  // namespace kda
