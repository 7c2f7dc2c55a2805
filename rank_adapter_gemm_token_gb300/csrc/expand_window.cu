// Expand for the overflow window of a large batch: the tokens of the one or two 128-token tiles
// whose pairs use more than kTileSlots slots (decode-like parts of a mixed batch). The skinny
// kernel in shrink-only mode has left v of those tokens against every active slot in
// MetaView::vfull, row w = window row (tile counts[6] first, then tile counts[7]); here
//
//   y[t][o] += sum over t's pairs not handled on the tensor cores of  s c sum_q B_slot[o][q] v[w(t)][slot][q]
//
// ("Multi-LoRA Serving Explained", batched serving: each token's side path added to the shared
// base product; "[RFC] Per-request activation of multiple LoRA adapters": k slots per token).
// One slot per token: item = (pair-block still to do, 512-column range), B rows read once per
// block; several slots per token: item = (window row, 512-column range), slots added in order j.
// Programmatic dependents of the shrink: metadata and the L2 prefetch of B rows come before
// griddepcontrol.wait, v and y after it; every block waits before it leaves.
#include "expand_vfull.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace mlora {
namespace {

constexpr int kWinThreads = 256;

__device__ __forceinline__ int window_row(int t, int tile_a, int tile_b) {
  const int tile = t >> 7;
  return tile == tile_a ? (t & 127) : (tile == tile_b ? 128 + (t & 127) : -1);
}

__global__ void __launch_bounds__(kWinThreads)
lora_expand_window_segment_kernel(float* __restrict__ y, PoolView pool, MetaView m, int n_dchunk) {
  __shared__ ExpandSmem es;
  const int tile_a = m.counts[6], tile_b = m.counts[7];     // the metadata is complete: read early
  const int items = tile_a >= 0 ? m.counts[5] * n_dchunk : 0;
  const int R = pool.R, D = pool.D;
  bool waited = false;
  for (int item = blockIdx.x; item < items; item += gridDim.x) {
    const int b = m.todo_blk[item / n_dchunk], dc = item % n_dchunk;
    const int slot = m.blk_slot[b], start = m.blk_start[b], cnt = m.blk_count[b];
    const int rank = pool.slot_rank[slot];
    const int rpad = (rank + 7) & ~7;
    const int oa = dc * kExpandVfullCols, ob = min(D, oa + kExpandVfullCols);
    __syncthreads();
    if (threadIdx.x < cnt) {
      const int p = m.order[start + threadIdx.x];          // one slot per token: token == pair
      const int w = window_row(p, tile_a, tile_b);
      const bool done = m.pair_fused[p] || w < 0;          // added inside the base GEMM
      es.tok[threadIdx.x] = done ? -1 : p;
      es.act[threadIdx.x] = done ? 0 : w * m.vfull_ld + m.pair_act[p] * R;   // v row of the pair
      es.coef[threadIdx.x] = done ? 0.f : pool.slot_scale[slot] * m.pair_scale[p];
    }
    if (!waited && rpad == R) {                            // a prefetch brings whole 128-byte lines:
      for (int o = oa + threadIdx.x; o < ob; o += kWinThreads)   // only when the rank fills the row
        for (int u = 0; u < rpad; u += 32) prefetch_l2(pool.B + (static_cast<size_t>(slot) * D + o) * R + u);
    }
    __syncthreads();
    if (!waited) {
      ptx::grid_dependency_wait();                         // v of the window shrink is complete
      ptx::grid_dependents_launch();
      waited = true;
    }
    for (int i = threadIdx.x; i < cnt * rpad; i += kWinThreads) {
      const int pi = i / rpad, q = i - pi * rpad;
      es.vs[pi][q] = (q < rank && es.tok[pi] >= 0) ? es.coef[pi] * m.vfull[es.act[pi] + q] : 0.f;
    }
    __syncthreads();
    for (int o = oa + threadIdx.x; o < ob; o += kWinThreads) {
      const uint4* brow = reinterpret_cast<const uint4*>(pool.B + (static_cast<size_t>(slot) * D + o) * R);
      for (int g = 0; g < cnt; g += 4) {                   // pairs in groups of four
        float yv[4], d[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int t = g + i < cnt ? es.tok[g + i] : -1;
          yv[i] = t >= 0 ? y[static_cast<size_t>(t) * D + o] : 0.f;
          d[i] = 0.f;
        }
        for (int u = 0; u < rpad / 8; ++u) {
          const uint4 bv = __ldg(brow + u);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (g + i < cnt) d[i] += ev_dot8(bv, &es.vs[g + i][8 * u]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int t = g + i < cnt ? es.tok[g + i] : -1;
          if (t >= 0) y[static_cast<size_t>(t) * D + o] = yv[i] + d[i];
        }
      }
    }
  }
  if (!waited) {
    ptx::grid_dependency_wait();
    ptx::grid_dependents_launch();
  }
}

// Several slots per token: item = (window row, 512-column range); the token's slots are added in
// order j (all of them: a token of an overflow tile has no pair on the tensor cores).
__global__ void __launch_bounds__(kWinThreads)
lora_expand_window_token_kernel(float* __restrict__ y, PoolView pool, MetaView m, int n_dchunk) {
  __shared__ ExpandSmem es;
  const int tile_a = m.counts[6], tile_b = m.counts[7];
  const int items = tile_a >= 0 ? 2 * 128 * n_dchunk : 0;
  const int J = m.J, R = pool.R, D = pool.D;
  bool waited = false;
  for (int item = blockIdx.x; item < items; item += gridDim.x) {
    const int w = item / n_dchunk, dc = item % n_dchunk;
    const int tile = w < 128 ? tile_a : tile_b;
    const int t = tile * 128 + (w & 127);
    if (tile < 0 || t >= m.T) continue;                    // uniform across the block
    __syncthreads();
    if (threadIdx.x < J) {
      const int p = t * J + threadIdx.x;
      const int s = m.pair_fused[p] ? -1 : m.pair_slot[p];
      es.ss[threadIdx.x] = s;
      es.rs[threadIdx.x] = s >= 0 ? pool.slot_rank[s] : 0;
      es.coef[threadIdx.x] = s >= 0 ? m.pair_scale[p] * pool.slot_scale[s] : 0.f;
      es.act[threadIdx.x] = s >= 0 ? m.pair_act[p] : 0;
    }
    __syncthreads();
    const int oa = dc * kExpandVfullCols, ob = min(D, oa + kExpandVfullCols);
    if (!waited) {
      for (int j = 0; j < J; ++j)
        if (es.ss[j] >= 0 && ((es.rs[j] + 7) & ~7) == R)    // whole rows only (see above)
          for (int o = oa + threadIdx.x; o < ob; o += kWinThreads)
            for (int u = 0; u < es.rs[j]; u += 32)
              prefetch_l2(pool.B + (static_cast<size_t>(es.ss[j]) * D + o) * R + u);
      ptx::grid_dependency_wait();                         // v of the window shrink is complete
      ptx::grid_dependents_launch();
      waited = true;
    }
    for (int i = threadIdx.x; i < J * R; i += kWinThreads) {
      const int j = i / R, q = i - j * R;
      es.vs[j][q] = (es.ss[j] >= 0 && q < es.rs[j])
                        ? es.coef[j] * m.vfull[static_cast<size_t>(w) * m.vfull_ld + es.act[j] * R + q]
                        : 0.f;
    }
    __syncthreads();
    for (int o = oa + threadIdx.x; o < ob; o += kWinThreads) {
      float acc = y[static_cast<size_t>(t) * D + o];
      for (int j = 0; j < J; ++j) {
        const int s = es.ss[j];
        if (s < 0) continue;
        const uint4* brow = reinterpret_cast<const uint4*>(pool.B + (static_cast<size_t>(s) * D + o) * R);
        float d = 0.f;
        for (int u = 0; u < (es.rs[j] + 7) / 8; ++u) d += ev_dot8(__ldg(brow + u), &es.vs[j][8 * u]);
        acc += d;
      }
      y[static_cast<size_t>(t) * D + o] = acc;
    }
  }
  if (!waited) {
    ptx::grid_dependency_wait();
    ptx::grid_dependents_launch();
  }
}

}  // namespace

cudaError_t launch_lora_expand_window(float* y, const PoolView& pool, const MetaView& m, int num_sms,
                                      cudaStream_t s) {
  if (m.n == 0 || pool.D == 0) return cudaSuccess;
  const int n_dchunk = (pool.D + kExpandVfullCols - 1) / kExpandVfullCols;
  const int max_items = (m.J == 1 ? m.n : 2 * 128) * n_dchunk;
  int grid = num_sms * 8;
  if (grid > max_items) grid = max_items;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kWinThreads, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  note_launch_begin(kKindExpand, s);
  cudaError_t e = (m.J == 1) ? cudaLaunchKernelEx(&cfg, lora_expand_window_segment_kernel, y, pool, m, n_dchunk)
                             : cudaLaunchKernelEx(&cfg, lora_expand_window_token_kernel, y, pool, m, n_dchunk);
  note_launch_end(kKindExpand, s);
  return e;
}

}  // namespace mlora
