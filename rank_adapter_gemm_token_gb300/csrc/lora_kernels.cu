// The low-rank side path: shrink (K -> r) and expand (r -> D) with the slot gathered per pair.
//
// "Multi-LoRA Serving Explained" (sevydevy.com), batched-serving section: each token finds
// its A and B through its slot; gathering reads an adapter per token, grouping a slot's
// tokens reads it once per group; the two steps are named shrink (full width down to the
// rank) and expand (rank back up). "[RFC] Per-request activation of multiple LoRA adapters"
// (vLLM issue 51940), Proposed Change items 3-4: up to k slots per token with the sentinel
// -1 skipped, each weighted by its own scale, iterated inside one fused pass. "[vLLM] LoRA"
// (secrett2633 blog), PEFTHelper: the slot factor is alpha/r, alpha/sqrt(r) under rsLoRA.
//
// Shrink works per pair-block (at most 16 pairs of one slot, from the sorted metadata) and K
// split: each lane streams its share of A[slot] once with 16-byte loads, reusing each vector
// for the pairs of the block, and writes unscaled fp32 partial sums per split. Expand adds the
// splits in a fixed order and multiplies by the pair's scale times the slot factor. With one
// slot per token it works per pair-block and column range (512 columns, more when there are
// enough items): B[slot] rows are read once per block (thread = output column, so both
// the B rows and y are accessed coalesced) and each y element receives exactly one update.
// With several slots per token it works per token, adding the slots in order j = 0..J-1.
// Either way every output is a fixed sequence of fp32 operations (deterministic), tokens
// whose slots are all -1 are never touched, and with no active pair no block does any work.
#include "internal.h"
#include "ptx.cuh"

namespace mlora {
namespace {

constexpr int kShrinkThreads = 256;      // 8 warps; warp w owns adapter rows w, w + 8, ...
constexpr int kExpandThreads = 256;      // one output column per thread, coalesced B rows and y
constexpr int kExpandColsPerItem = 512;  // output columns per item (two per thread) ...
constexpr int kExpandMaxColsPerItem = 4096;   // ... doubled up to this while the items still fill the SMs

__device__ __forceinline__ float dot8_bf16(const uint4& a, const uint4& b) {
  float s = ptx::bf16_lo(a.x) * ptx::bf16_lo(b.x);
  s = fmaf(ptx::bf16_hi(a.x), ptx::bf16_hi(b.x), s);
  s = fmaf(ptx::bf16_lo(a.y), ptx::bf16_lo(b.y), s);
  s = fmaf(ptx::bf16_hi(a.y), ptx::bf16_hi(b.y), s);
  s = fmaf(ptx::bf16_lo(a.z), ptx::bf16_lo(b.z), s);
  s = fmaf(ptx::bf16_hi(a.z), ptx::bf16_hi(b.z), s);
  s = fmaf(ptx::bf16_lo(a.w), ptx::bf16_lo(b.w), s);
  s = fmaf(ptx::bf16_hi(a.w), ptx::bf16_hi(b.w), s);
  return s;
}

__device__ __forceinline__ float dot8_bf16_f32(const uint4& b, const float* v) {
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

// Item = (pair-block, K split). Warp w owns adapter rows w, w + 8, ... (RPW of them per group of
// rows); lane l covers 8-element vectors l, l + 32, ... of the split. Each lane loads its A
// vectors once (eight 16-byte loads in flight) and reuses them for every pair of the block, so
// the dot products need only warp shuffles. The split's fp32 partial sums go to
// vpart[split][p][q]; a consumer adds the splits in order 0, 1, ... . Items are spread over
// every SM, and the kernel lets a dependent kernel (programmatic launch) start right away.
template <int RPW>
__global__ void __launch_bounds__(kShrinkThreads)
lora_shrink_kernel(const uint16_t* __restrict__ x, PoolView pool, MetaView m, int kc_len, int n_ks, int skip_fused) {
  constexpr int G = 4;                                        // pairs per register group
  constexpr int V = 8 / RPW;                                  // vectors per lane per row
  ptx::grid_dependents_launch();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int items = m.counts[skip_fused ? 5 : 2] * n_ks;
  const int K = pool.K, R = pool.R;
  for (int item = blockIdx.x; item < items; item += gridDim.x) {
    const int bi = item / n_ks, ks = item - bi * n_ks;
    const int b = skip_fused ? m.todo_blk[bi] : bi;
    const int slot = m.blk_slot[b];
    const int start = m.blk_start[b];
    const int cnt = m.blk_count[b];
    const int rank = pool.slot_rank[slot];
    const int aoff = pool.slot_off[slot];
    const int k0 = ks * kc_len;
    const int nv = (min(K, k0 + kc_len) - k0) / 8;            // vectors in this split
    for (int qg = warp; qg < rank; qg += 8 * RPW) {           // rows qg + 8 i, i < RPW
      for (int g0 = 0; g0 < cnt; g0 += G) {
        const int gc = min(G, cnt - g0);
        int pr[G];
        const uint4* xv[G];
#pragma unroll
        for (int i = 0; i < G; ++i) {
          pr[i] = m.order[start + g0 + (i < gc ? i : 0)];
          xv[i] = reinterpret_cast<const uint4*>(x + static_cast<size_t>(pr[i] / m.J) * K + k0);
        }
        float acc[RPW][G];
#pragma unroll
        for (int r = 0; r < RPW; ++r)
#pragma unroll
          for (int i = 0; i < G; ++i) acc[r][i] = 0.f;
        for (int u0 = lane; u0 < nv; u0 += 32 * V) {
          uint4 a[RPW][V];
#pragma unroll
          for (int r = 0; r < RPW; ++r) {
            const int q = qg + 8 * r;
            const uint4* arow = reinterpret_cast<const uint4*>(pool.A + (static_cast<size_t>(aoff) + q) * K + k0);
#pragma unroll
            for (int v = 0; v < V; ++v) {
              const int u = u0 + 32 * v;
              a[r][v] = (q < rank && u < nv) ? __ldg(arow + u) : make_uint4(0u, 0u, 0u, 0u);
            }
          }
#pragma unroll
          for (int i = 0; i < G; ++i) {
            if (i < gc) {
#pragma unroll
              for (int v = 0; v < V; ++v) {
                const int u = u0 + 32 * v;
                if (u < nv) {
                  const uint4 xx = __ldg(xv[i] + u);
#pragma unroll
                  for (int r = 0; r < RPW; ++r) acc[r][i] += dot8_bf16(a[r][v], xx);
                }
              }
            }
          }
        }
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
#pragma unroll
          for (int i = 0; i < G; ++i) {
            float v = acc[r][i];
#pragma unroll
            for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
            const int q = qg + 8 * r;
            if (lane == 0 && i < gc && q < rank) m.vpart[(static_cast<size_t>(ks) * m.n + pr[i]) * R + q] = v;
          }
        }
      }
    }
  }
}

// v of pair p: the K-split partials added in order, times coef; zero beyond the rank.
__device__ __forceinline__ float pair_v(const MetaView& m, int R, int n_ks, int p, int q, int rank, float coef) {
  if (q >= rank) return 0.f;
  float v = 0.f;
  for (int ks = 0; ks < n_ks; ++ks) v += m.vpart[(static_cast<size_t>(ks) * m.n + p) * R + q];
  return coef * v;
}

// J == 1: item = (pair-block, 512-column range). The block's scaled v rows sit in shared memory;
// thread c reads B[slot] row o (consecutive threads -> consecutive rows, coalesced) once and
// updates y[t][o] for every token of the block (consecutive o, coalesced). Each y element is
// updated by exactly one pair, so the result is deterministic.
__global__ void __launch_bounds__(kExpandThreads)
lora_expand_segment_kernel(float* __restrict__ y, PoolView pool, MetaView m, int n_ks, int n_dchunk, int cols,
                           int skip_fused) {
  __shared__ __align__(16) float vs[kPairBlock][kMaxRank];
  __shared__ int tok[kPairBlock];
  // skip_fused: only todo_blk's blocks
  const int items = m.counts[skip_fused ? 5 : 2] * n_dchunk;
  const int R = pool.R, D = pool.D;
  for (int item = blockIdx.x; item < items; item += gridDim.x) {
    const int bi = item / n_dchunk, dc = item - bi * n_dchunk;
    const int b = skip_fused ? m.todo_blk[bi] : bi;
    const int slot = m.blk_slot[b];
    const int start = m.blk_start[b];
    const int cnt = m.blk_count[b];
    const int rank = pool.slot_rank[slot];
    const float c = pool.slot_scale[slot];
    const int rpad = (rank + 7) & ~7;
    __syncthreads();
    for (int i = threadIdx.x; i < cnt * rpad; i += kExpandThreads) {
      const int pi = i / rpad, q = i - pi * rpad;
      const int p = m.order[start + pi];
      const bool done = skip_fused && m.pair_fused[p];        // added inside the base GEMM
      vs[pi][q] = done ? 0.f : pair_v(m, R, n_ks, p, q, rank, c * m.pair_scale[p]);
      if (q == 0) tok[pi] = done ? -1 : p;          // J == 1: token index == pair index
    }
    __syncthreads();
    for (int o = dc * cols + threadIdx.x; o < min(D, (dc + 1) * cols);
         o += kExpandThreads) {
      const uint4* brow = reinterpret_cast<const uint4*>(pool.B + static_cast<size_t>(o) * pool.C + pool.slot_off[slot]);
      float d[kPairBlock];
#pragma unroll
      for (int i = 0; i < kPairBlock; ++i) d[i] = 0.f;
      for (int u = 0; u < rpad / 8; ++u) {
        const uint4 bv = __ldg(brow + u);
#pragma unroll
        for (int i = 0; i < kPairBlock; ++i)
          if (i < cnt) d[i] += dot8_bf16_f32(bv, &vs[i][8 * u]);
      }
#pragma unroll
      for (int i = 0; i < kPairBlock; ++i)
        if (i < cnt && tok[i] >= 0) y[static_cast<size_t>(tok[i]) * D + o] += d[i];
    }
  }
}

// J > 1: item = (token, 512-column range); slots are added in order j = 0..J-1 so every output
// is a fixed sequence of fp32 additions. Thread c owns column o: B rows and y coalesced.
__global__ void __launch_bounds__(kExpandThreads)
lora_expand_token_kernel(float* __restrict__ y, PoolView pool, MetaView m, int n_ks, int n_dchunk, int cols,
                         int skip_fused) {
  __shared__ __align__(16) float vs[kMaxJ][kMaxRank];
  __shared__ float cs[kMaxJ];
  __shared__ int ss[kMaxJ], rs[kMaxJ];
  const int J = m.J, R = pool.R, D = pool.D;
  const bool none = skip_fused && m.counts[5] == 0;
  const int items = none ? 0 : m.T * n_dchunk;          // nothing left off the tensor cores
  for (int item = blockIdx.x; item < items; item += gridDim.x) {
    const int t = item / n_dchunk, dc = item - t * n_dchunk;
    bool any = false;
    for (int j = 0; j < J; ++j) any |= m.pair_slot[t * J + j] >= 0 && !(skip_fused && m.pair_fused[t * J + j]);
    if (!any) continue;                                // uniform across the block
    __syncthreads();
    if (threadIdx.x < J) {
      const int p = t * J + threadIdx.x;
      const int s = (skip_fused && m.pair_fused[p]) ? -1 : m.pair_slot[p];
      ss[threadIdx.x] = s;
      rs[threadIdx.x] = s >= 0 ? pool.slot_rank[s] : 0;
      cs[threadIdx.x] = s >= 0 ? m.pair_scale[p] * pool.slot_scale[s] : 0.f;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < J * R; i += kExpandThreads) {
      const int j = i / R, q = i - j * R;
      vs[j][q] = ss[j] >= 0 ? pair_v(m, R, n_ks, t * J + j, q, rs[j], cs[j]) : 0.f;
    }
    __syncthreads();
    for (int o = dc * cols + threadIdx.x; o < min(D, (dc + 1) * cols);
         o += kExpandThreads) {
      float acc = y[static_cast<size_t>(t) * D + o];
      for (int j = 0; j < J; ++j) {
        const int s = ss[j];
        if (s < 0) continue;
        const uint4* brow = reinterpret_cast<const uint4*>(pool.B + static_cast<size_t>(o) * pool.C + pool.slot_off[s]);
        float d = 0.f;
        for (int u = 0; u < (rs[j] + 7) / 8; ++u) d += dot8_bf16_f32(__ldg(brow + u), &vs[j][8 * u]);
        acc += d;
      }
      y[static_cast<size_t>(t) * D + o] = acc;
    }
  }
}

}  // namespace

int shrink_rows_per_warp(int R) { return R <= 8 ? 1 : R <= 16 ? 2 : R <= 32 ? 4 : 8; }

void shrink_split(int K, int R, int* kc_len, int* n_ks) {
  int kc = 256 * (8 / shrink_rows_per_warp(R));             // eight A vectors per lane
  if ((K + kc - 1) / kc > kMaxShrinkSplits) kc = ((K + kMaxShrinkSplits - 1) / kMaxShrinkSplits + 255) / 256 * 256;
  *kc_len = kc;
  *n_ks = (K + kc - 1) / kc;
}

cudaError_t launch_lora_shrink(const uint16_t* x, const PoolView& pool, const MetaView& m, int num_sms,
                               cudaStream_t s, bool skip_fused) {
  const int skip = skip_fused ? 1 : 0;
  if (m.n == 0) return cudaSuccess;
  int kc, n_ks;
  shrink_split(pool.K, pool.R, &kc, &n_ks);
  const int max_items = m.n * n_ks;                     // pair-blocks <= pairs
  int grid = num_sms * 2;
  if (grid > max_items) grid = max_items;
  note_launch_begin(kKindShrink, s);
  switch (shrink_rows_per_warp(pool.R)) {
    case 1: lora_shrink_kernel<1><<<grid, kShrinkThreads, 0, s>>>(x, pool, m, kc, n_ks, skip); break;
    case 2: lora_shrink_kernel<2><<<grid, kShrinkThreads, 0, s>>>(x, pool, m, kc, n_ks, skip); break;
    case 4: lora_shrink_kernel<4><<<grid, kShrinkThreads, 0, s>>>(x, pool, m, kc, n_ks, skip); break;
    default: lora_shrink_kernel<8><<<grid, kShrinkThreads, 0, s>>>(x, pool, m, kc, n_ks, skip); break;
  }
  cudaError_t e = cudaGetLastError();
  note_launch_end(kKindShrink, s);
  return e;
}

cudaError_t launch_lora_expand(float* y, const PoolView& pool, const MetaView& m, int num_sms, cudaStream_t s,
                               bool skip_fused) {
  const int skip = skip_fused ? 1 : 0;
  if (m.n == 0 || pool.D == 0) return cudaSuccess;
  int kc, n_ks;
  shrink_split(pool.K, pool.R, &kc, &n_ks);
  // Wider column ranges per item amortise an item's set-up (its pairs, their v) over more columns;
  // they are used while the items still number at least eight per SM (pair-blocks counted as
  // full, a lower bound, for one slot per token).
  const long lo_rows = m.J == 1 ? (m.n + kPairBlock - 1) / kPairBlock : m.T;
  int cols = kExpandColsPerItem;
  while (cols < kExpandMaxColsPerItem && lo_rows * ((pool.D + 2 * cols - 1) / (2 * cols)) >= 8L * num_sms) cols *= 2;
  const int n_dchunk = (pool.D + cols - 1) / cols;
  const int max_items = (m.J == 1 ? m.n : m.T) * n_dchunk;
  int grid = num_sms * 8;
  if (grid > max_items) grid = max_items;
  note_launch_begin(kKindExpand, s);
  if (m.J == 1)
    lora_expand_segment_kernel<<<grid, kExpandThreads, 0, s>>>(y, pool, m, n_ks, n_dchunk, cols, skip);
  else
    lora_expand_token_kernel<<<grid, kExpandThreads, 0, s>>>(y, pool, m, n_ks, n_dchunk, cols, skip);
  cudaError_t e = cudaGetLastError();
  note_launch_end(kKindExpand, s);
  return e;
}

}  // namespace mlora
