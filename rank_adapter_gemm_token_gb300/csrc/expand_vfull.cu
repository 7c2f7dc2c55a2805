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
constexpr size_t kRowsMaxSmem = 64 * 1024;   // the output-row form's per-pair rows and tables

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

// Output-row form for a one-class pool: item = kRowsPerItem (16) consecutive output columns o of y for
// every token. B [D, C] is read a row range at a time (each CTA touches rows o0 .. o0 + 15 of the
// active slots' columns, through L1), so its rows are streamed once in address order instead of
// as 16- to 128-byte pieces per (pair-block, column range). Before griddepcontrol.wait the CTA
// stages, per pair, the slot's first column, its rank and the factor s c (metadata and pool
// only); after it, every pair's scaled v row (shared memory, rows padded by 4 floats so the
// tokens of a warp hit different banks); then thread (token, row) adds, for each of the
// token's slots in order j, sum_q B[o][off + q] v[q] to y[t][o].
constexpr int kRowsPerItem = 16;

__global__ void __launch_bounds__(kExpandThreads, 2)
lora_expand_vfull_rows_kernel(float* __restrict__ y, PoolView pool, MetaView m) {
  extern __shared__ __align__(16) float vrows[];           // [T * J][R + 4] scaled v, then pair info
  const int R = pool.R, D = pool.D, C = pool.C, n = m.n;
  const int ld = R + 4;
  int* poff = reinterpret_cast<int*>(vrows + static_cast<size_t>(n) * ld);   // [n] first column (-1: none)
  int* prank = poff + n;                                                    // [n]
  int* pact = prank + n;                                                    // [n] active-slot index
  float* pcoef = reinterpret_cast<float*>(pact + n);                        // [n] s c
  for (int p = threadIdx.x; p < n; p += kExpandThreads) {
    const int s = m.pair_slot[p];
    poff[p] = s >= 0 ? pool.slot_off[s] : -1;
    prank[p] = s >= 0 ? pool.slot_rank[s] : 0;
    pact[p] = m.pair_act[p];
    pcoef[p] = s >= 0 ? m.pair_scale[p] * pool.slot_scale[s] : 0.f;
  }
  __syncthreads();
  ptx::grid_dependency_wait();                             // v and y of the fused GEMM are complete
  ptx::grid_dependents_launch();
  // one pair's row per thread, four 16-byte loads in flight at a time
  for (int p = threadIdx.x; p < n; p += kExpandThreads) {
    const int rank = prank[p], act = pact[p];
    const float coef = pcoef[p];
    const float4* src = reinterpret_cast<const float4*>(m.vfull + static_cast<size_t>(p / m.J) * m.vfull_ld +
                                                        static_cast<size_t>(act < 0 ? 0 : act) * R);
    float* dst = vrows + static_cast<size_t>(p) * ld;
    for (int c = 0; c < R / 4; c += 4) {
      float4 v[4];
#pragma unroll
      for (int k = 0; k < 4; ++k)
        v[k] = (c + k < R / 4 && 4 * (c + k) < rank) ? src[c + k] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (c + k < R / 4) {
          const int q = 4 * (c + k);
          dst[q] = q < rank ? coef * v[k].x : 0.f;
          dst[q + 1] = q + 1 < rank ? coef * v[k].y : 0.f;
          dst[q + 2] = q + 2 < rank ? coef * v[k].z : 0.f;
          dst[q + 3] = q + 3 < rank ? coef * v[k].w : 0.f;
        }
      }
    }
  }
  __syncthreads();
  const int o = blockIdx.x * kRowsPerItem + (threadIdx.x % kRowsPerItem);
  if (o >= D) return;
  const uint16_t* brow = pool.B + static_cast<size_t>(o) * C;
  constexpr int kStep = kExpandThreads / kRowsPerItem;      // token lanes of the CTA
  constexpr int kTok = 8;                                    // tokens in flight per thread
  for (int t0 = threadIdx.x / kRowsPerItem; t0 < m.T; t0 += kTok * kStep) {
    float acc[kTok];
#pragma unroll
    for (int i = 0; i < kTok; ++i) {
      const int t = t0 + i * kStep;
      acc[i] = t < m.T ? y[static_cast<size_t>(t) * D + o] : 0.f;
    }
    for (int j = 0; j < m.J; ++j) {
      int off[kTok], nu[kTok], pp[kTok], nu_max = 0;
#pragma unroll
      for (int i = 0; i < kTok; ++i) {
        const int t = t0 + i * kStep;
        pp[i] = t * m.J + j;
        off[i] = t < m.T ? poff[pp[i]] : -1;
        nu[i] = off[i] >= 0 ? (prank[pp[i]] + 7) / 8 : 0;
        nu_max = max(nu_max, nu[i]);
      }
      float d[kTok];
#pragma unroll
      for (int i = 0; i < kTok; ++i) d[i] = 0.f;
      for (int u = 0; u < nu_max; ++u) {
        uint4 bv[kTok];
#pragma unroll
        for (int i = 0; i < kTok; ++i)
          bv[i] = u < nu[i] ? __ldg(reinterpret_cast<const uint4*>(brow + off[i]) + u) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int i = 0; i < kTok; ++i)
          if (u < nu[i]) d[i] += ev_dot8(bv[i], vrows + static_cast<size_t>(pp[i]) * ld + 8 * u);
      }
#pragma unroll
      for (int i = 0; i < kTok; ++i)
        if (off[i] >= 0) acc[i] += d[i];
    }
#pragma unroll
    for (int i = 0; i < kTok; ++i) {
      const int t = t0 + i * kStep;
      if (t < m.T) y[static_cast<size_t>(t) * D + o] = acc[i];
    }
  }
}

}  // namespace

static size_t expand_vfull_rows_smem(const PoolView& pool, const MetaView& m) {
  return static_cast<size_t>(m.n) * ((pool.R + 4) * sizeof(float) + 4 * sizeof(int));
}

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
  // a one-class pool whose pairs' v rows fit in shared memory takes the output-row form
  const size_t rows_smem = expand_vfull_rows_smem(pool, m);
  const bool rows = pool.uniform && rows_smem <= kRowsMaxSmem;
  if (rows) {
    static int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
      cudaError_t e = cudaFuncSetAttribute(lora_expand_vfull_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(kRowsMaxSmem));
      if (e != cudaSuccess) return e;
      configured_device = dev;
    }
    cfg.gridDim = dim3((pool.D + kRowsPerItem - 1) / kRowsPerItem, 1, 1);
    cfg.dynamicSmemBytes = rows_smem;
  }
  note_launch_begin(kKindExpand, s);
  cudaError_t e = rows ? cudaLaunchKernelEx(&cfg, lora_expand_vfull_rows_kernel, y, pool, m)
                  : (m.J == 1) ? cudaLaunchKernelEx(&cfg, lora_expand_vfull_segment_kernel, y, pool, m, n_dchunk)
                               : cudaLaunchKernelEx(&cfg, lora_expand_vfull_token_kernel, y, pool, m, n_dchunk);
  note_launch_end(kKindExpand, s);
  return e;
}

}  // namespace mlora
