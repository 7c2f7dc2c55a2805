// Expand after the small-batch fused GEMM, which leaves v of every token against every active
// slot in vfull[t][a][q] ("Multi-LoRA Serving Explained", batched serving: each token's side
// path added to the shared base product; "[RFC] Per-request activation of multiple LoRA
// adapters": k slots per token with per-adapter scales). These kernels are programmatic
// dependents of that GEMM: everything that does not depend on it (the step's metadata, the B
// rows, which are prefetched into L2) is done before griddepcontrol.wait, and only v and y are
// touched after it. The work items are in expand_vfull.cuh.
#include "expand_vfull.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace mlora {
namespace {

constexpr int kExpandThreads = 256;      // one output column per thread, coalesced B rows and y

// One slot per token: item = (pair-block, 512-column range): B rows of the slot read once per block.
__global__ void __launch_bounds__(kExpandThreads)
lora_expand_vfull_segment_kernel(float* __restrict__ y, PoolView pool, MetaView m, int n_dchunk) {
  __shared__ ExpandSmem es;
  const int items = m.counts[2] * n_dchunk;
  bool waited = false;
  for (int item = blockIdx.x; item < items; item += gridDim.x)
    expand_vfull_segment_item<kExpandThreads>(y, pool, m, item, n_dchunk, es, &waited);
  if (!waited) {
    ptx::grid_dependency_wait();
    ptx::grid_dependents_launch();
  }
}

// Several slots per token: item = (token, 512-column range), slots added in order j = 0..J-1.
__global__ void __launch_bounds__(kExpandThreads)
lora_expand_vfull_token_kernel(float* __restrict__ y, PoolView pool, MetaView m, int n_dchunk) {
  __shared__ ExpandSmem es;
  const int items = m.T * n_dchunk;
  bool waited = false;
  for (int item = blockIdx.x; item < items; item += gridDim.x)
    expand_vfull_token_item<kExpandThreads>(y, pool, m, item, n_dchunk, es, &waited);
  if (!waited) {
    ptx::grid_dependency_wait();
    ptx::grid_dependents_launch();
  }
}

}  // namespace

cudaError_t launch_lora_expand_vfull(float* y, const PoolView& pool, const MetaView& m, int num_sms,
                                     cudaStream_t s) {
  if (m.n == 0 || pool.D == 0) return cudaSuccess;
  const int n_dchunk = (pool.D + kExpandVfullCols - 1) / kExpandVfullCols;
  const int max_items = (m.J == 1 ? m.n : m.T) * n_dchunk;
  int grid = num_sms * 8;
  if (grid > max_items) grid = max_items;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kExpandThreads, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  note_launch_begin(kKindExpand, s);
  cudaError_t e = (m.J == 1) ? cudaLaunchKernelEx(&cfg, lora_expand_vfull_segment_kernel, y, pool, m, n_dchunk)
                             : cudaLaunchKernelEx(&cfg, lora_expand_vfull_token_kernel, y, pool, m, n_dchunk);
  note_launch_end(kKindExpand, s);
  return e;
}

}  // namespace mlora
