// Expand work items after the small-batch fused GEMM, which leaves v of every token against every
// active slot in MetaView::vfull. Used by the vfull expand kernels (programmatic dependents of
// the GEMM); the B-row prefetch helper is also called by the GEMM's epilogue warps.
//
// y[t][o] += sum_j s c sum_q B_slot[o][q] v[t][slot][q]  ("Multi-LoRA Serving Explained", batched
// serving: each token's side path added to the shared base product; "[RFC] Per-request
// activation of multiple LoRA adapters": k slots per token with per-adapter scales).
// One slot per token: item = (pair-block, 512-column range): B rows of the slot are read once
// per block (thread = output column: B rows and y accessed coalesced), each y element gets one
// update. Several slots per token: item = (token, 512-column range), slots added in order j.
#pragma once
#include "internal.h"
#include "ptx.cuh"

namespace mlora {

constexpr int kExpandVfullCols = 512;

struct ExpandSmem {
  float vs[kPairBlock][kMaxRank];   // scaled v rows of the item's pairs (kMaxJ <= kPairBlock)
  int tok[kPairBlock], act[kPairBlock];
  float coef[kPairBlock];
  int ss[kMaxJ], rs[kMaxJ];
};

__device__ __forceinline__ void prefetch_l2(const void* p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }

__device__ __forceinline__ float ev_dot8(const uint4& b, const float* v) {
  float a = ptx::bf16_lo(b.x) * v[0];
  a = fmaf(ptx::bf16_hi(b.x), v[1], a);
  a = fmaf(ptx::bf16_lo(b.y), v[2], a);
  a = fmaf(ptx::bf16_hi(b.y), v[3], a);
  a = fmaf(ptx::bf16_lo(b.z), v[4], a);
  a = fmaf(ptx::bf16_hi(b.z), v[5], a);
  a = fmaf(ptx::bf16_lo(b.w), v[6], a);
  a = fmaf(ptx::bf16_hi(b.w), v[7], a);
  return a;
}

// Prefetches into L2 the B rows an item will read (a hint; no ordering needed).
__device__ __forceinline__ void expand_vfull_prefetch(const PoolView& pool, const MetaView& m, int item,
                                                      int n_dchunk, int tid, int nthreads) {
  const int D = pool.D;
  const int dc = item % n_dchunk, key = item / n_dchunk;
  const int oa = dc * kExpandVfullCols, ob = min(D, oa + kExpandVfullCols);
  if (m.J == 1) {
    const int slot = m.blk_slot[key];
    const int rpad = (pool.slot_rank[slot] + 7) & ~7;
    for (int o = oa + tid; o < ob; o += nthreads)
      for (int u = 0; u < rpad; u += 32) prefetch_l2(pool.B + static_cast<size_t>(o) * pool.C + pool.slot_off[slot] + u);
  } else {
    for (int j = 0; j < m.J; ++j) {
      const int s = m.pair_slot[key * m.J + j];
      if (s < 0) continue;
      const int rpad = (pool.slot_rank[s] + 7) & ~7;
      for (int o = oa + tid; o < ob; o += nthreads)
        for (int u = 0; u < rpad; u += 32) prefetch_l2(pool.B + static_cast<size_t>(o) * pool.C + pool.slot_off[s] + u);
    }
  }
}

// *waited: whether this block has passed griddepcontrol.wait (set on the first item; a caller
// that has already synchronised with the producer passes true).
template <int NT>
__device__ __forceinline__ void expand_vfull_segment_item(float* __restrict__ y, const PoolView& pool,
                                                          const MetaView& m, int item, int n_dchunk, ExpandSmem& es,
                                                          bool* waited) {
  const int R = pool.R, D = pool.D;
  const int b = item / n_dchunk, dc = item - b * n_dchunk;
  const int slot = m.blk_slot[b];
  const int start = m.blk_start[b];
  const int cnt = m.blk_count[b];
  const int rank = pool.slot_rank[slot];
  const int rpad = (rank + 7) & ~7;
  const int oa = dc * kExpandVfullCols;
  const int ob = min(D, oa + kExpandVfullCols);
  __syncthreads();
  if (threadIdx.x < cnt) {                         // the step's metadata: ready before the GEMM
    const int p = m.order[start + threadIdx.x];
    es.tok[threadIdx.x] = p;                       // one slot per token: token index == pair index
    es.act[threadIdx.x] = m.pair_act[p];
    es.coef[threadIdx.x] = pool.slot_scale[slot] * m.pair_scale[p];
  }
  const int boff = pool.slot_off[slot];
  if (!*waited) {
    for (int o = oa + threadIdx.x; o < ob; o += NT)
      for (int u = 0; u < rpad; u += 32) prefetch_l2(pool.B + static_cast<size_t>(o) * pool.C + boff + u);
  }
  __syncthreads();
  if (!*waited) {
    ptx::grid_dependency_wait();                   // v and y of the fused GEMM are complete
    ptx::grid_dependents_launch();                 // dependents start only after this wait
    *waited = true;
  }
  for (int i = threadIdx.x; i < cnt * rpad; i += NT) {
    const int pi = i / rpad, q = i - pi * rpad;
    es.vs[pi][q] =
        q < rank ? es.coef[pi] * m.vfull[static_cast<size_t>(es.tok[pi]) * m.vfull_ld + es.act[pi] * R + q] : 0.f;
  }
  __syncthreads();
  for (int o = oa + threadIdx.x; o < ob; o += NT) {
    const uint4* brow = reinterpret_cast<const uint4*>(pool.B + static_cast<size_t>(o) * pool.C + boff);
    for (int g = 0; g < cnt; g += 4) {               // pairs in groups of four (few registers)
      float yv[4], d[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        yv[i] = g + i < cnt ? y[static_cast<size_t>(es.tok[g + i]) * D + o] : 0.f;
        d[i] = 0.f;
      }
      for (int u = 0; u < rpad / 8; ++u) {
        const uint4 bv = __ldg(brow + u);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (g + i < cnt) d[i] += ev_dot8(bv, &es.vs[g + i][8 * u]);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (g + i < cnt) y[static_cast<size_t>(es.tok[g + i]) * D + o] = yv[i] + d[i];
    }
  }
}

template <int NT>
__device__ __forceinline__ void expand_vfull_token_item(float* __restrict__ y, const PoolView& pool,
                                                        const MetaView& m, int item, int n_dchunk, ExpandSmem& es,
                                                        bool* waited) {
  const int J = m.J, R = pool.R, D = pool.D;
  const int t = item / n_dchunk, dc = item - t * n_dchunk;
  bool any = false;
  for (int j = 0; j < J; ++j) any |= m.pair_slot[t * J + j] >= 0;
  if (!any) return;                                // uniform across the block
  __syncthreads();
  if (threadIdx.x < J) {
    const int p = t * J + threadIdx.x;
    const int s = m.pair_slot[p];
    es.ss[threadIdx.x] = s;
    es.rs[threadIdx.x] = s >= 0 ? pool.slot_rank[s] : 0;
    es.coef[threadIdx.x] = s >= 0 ? m.pair_scale[p] * pool.slot_scale[s] : 0.f;
    es.act[threadIdx.x] = m.pair_act[p];
  }
  __syncthreads();
  const int oa = dc * kExpandVfullCols;
  const int ob = min(D, oa + kExpandVfullCols);
  if (!*waited) {
    for (int j = 0; j < J; ++j)
      if (es.ss[j] >= 0)
        for (int o = oa + threadIdx.x; o < ob; o += NT)
          for (int u = 0; u < es.rs[j]; u += 32)
            prefetch_l2(pool.B + static_cast<size_t>(o) * pool.C + pool.slot_off[es.ss[j]] + u);
    ptx::grid_dependency_wait();
    ptx::grid_dependents_launch();
    *waited = true;
  }
  for (int i = threadIdx.x; i < J * R; i += NT) {
    const int j = i / R, q = i - j * R;
    es.vs[j][q] = (es.ss[j] >= 0 && q < es.rs[j])
                      ? es.coef[j] * m.vfull[static_cast<size_t>(t) * m.vfull_ld + es.act[j] * R + q]
                      : 0.f;
  }
  __syncthreads();
  for (int o = oa + threadIdx.x; o < ob; o += NT) {
    float acc = y[static_cast<size_t>(t) * D + o];
    for (int j = 0; j < J; ++j) {
      const int s = es.ss[j];
      if (s < 0) continue;
      const uint4* brow = reinterpret_cast<const uint4*>(pool.B + static_cast<size_t>(o) * pool.C + pool.slot_off[s]);
      float d = 0.f;
      for (int u = 0; u < (es.rs[j] + 7) / 8; ++u) d += ev_dot8(__ldg(brow + u), &es.vs[j][8 * u]);
      acc += d;
    }
    y[static_cast<size_t>(t) * D + o] = acc;
  }
}

}  // namespace mlora
