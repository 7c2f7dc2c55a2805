// Check of the bounded-wait path that every kernel of this library relies on: one block waits on
// an mbarrier that nothing arrives on. The wait gives up after the library's limit (2 s of
// %globaltimer), sets the timeout bit in the given error word and the kernel returns, so the
// context stays usable. No fault, trap or unbounded loop is involved.
#include "internal.h"
#include "ptx.cuh"

namespace mlora {
namespace {

__global__ void wait_check_kernel(uint32_t* __restrict__ err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    ptx::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) (void)ptx::mbar_wait(&bar, 0, err);   // phase 0 never completes
}

}  // namespace

cudaError_t launch_wait_check(uint32_t* err, cudaStream_t s) {
  note_launch_begin(kKindSlot, s);
  wait_check_kernel<<<1, 32, 0, s>>>(err);
  cudaError_t e = cudaGetLastError();
  note_launch_end(kKindSlot, s);
  return e;
}

}  // namespace mlora
