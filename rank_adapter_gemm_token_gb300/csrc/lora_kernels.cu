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
// Shrink works per pair-block (at most 16 pairs of one slot, from the sorted metadata) and
// per K chunk: a warp owns one adapter row q, streams A[slot][q][chunk] once with 16-byte
// loads and reuses it for every pair of the block, writing fp32 partial sums
// vpart[chunk][p][q] (unscaled). Expand works per token and D range: it sums the chunk
// partials in a fixed order, multiplies by pair scale * slot factor, and adds the slot's
// B rows (16-byte loads, zero padding beyond the true rank skipped) into y in slot order
// j = 0..J-1, so every output is deterministic. Tokens whose slots are all -1 are never
// touched, and when the step has no active pair no block does any work.
#include "internal.h"
#include "ptx.cuh"

namespace mlora {
namespace {

constexpr int kShrinkThreads = 256;
constexpr int kExpandThreads = 256;
constexpr int kExpandCols = 8;            // outputs per thread

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

__global__ void __launch_bounds__(kShrinkThreads)
lora_shrink_kernel(const uint16_t* __restrict__ x, PoolView pool, MetaView m, int kc_len, int n_kc) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_blocks = m.counts[2];
  const int items = n_blocks * n_kc;
  const int K = pool.K, R = pool.R;
  for (int item = blockIdx.x; item < items; item += gridDim.x) {
    const int b = item / n_kc, kc = item - b * n_kc;
    const int slot = m.blk_slot[b];
    const int start = m.blk_start[b];
    const int cnt = m.blk_count[b];
    const int rank = pool.slot_rank[slot];
    const int k0 = kc * kc_len;
    const int k1 = min(K, k0 + kc_len);
    int tok[kPairBlock];
    int pr[kPairBlock];
#pragma unroll
    for (int i = 0; i < kPairBlock; ++i) {
      pr[i] = i < cnt ? m.order[start + i] : 0;
      tok[i] = pr[i] / m.J;
    }
    for (int q = warp; q < rank; q += kShrinkThreads / 32) {
      const uint16_t* arow = pool.A + (static_cast<size_t>(slot) * R + q) * K;
      float acc[kPairBlock];
#pragma unroll
      for (int i = 0; i < kPairBlock; ++i) acc[i] = 0.f;
      for (int k = k0 + lane * 8; k < k1; k += 256) {
        const uint4 av = *reinterpret_cast<const uint4*>(arow + k);
#pragma unroll
        for (int i = 0; i < kPairBlock; ++i) {
          if (i < cnt) {
            const uint4 xv = *reinterpret_cast<const uint4*>(x + static_cast<size_t>(tok[i]) * K + k);
            acc[i] += dot8_bf16(av, xv);
          }
        }
      }
#pragma unroll
      for (int i = 0; i < kPairBlock; ++i) {
        float v = acc[i];
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
        if (lane == 0 && i < cnt) m.vpart[(static_cast<size_t>(kc) * m.n + pr[i]) * R + q] = v;
      }
    }
  }
}

__global__ void __launch_bounds__(kExpandThreads)
lora_expand_kernel(float* __restrict__ y, PoolView pool, MetaView m, int n_kc) {
  __shared__ float vs[kMaxJ][kMaxRank];
  __shared__ float cs[kMaxJ];
  __shared__ int ss[kMaxJ], rs[kMaxJ];
  const int t = blockIdx.y;
  const int J = m.J, R = pool.R, D = pool.D;
  bool any = false;
  for (int j = 0; j < J; ++j) any |= m.pair_slot[t * J + j] >= 0;
  if (!any) return;
  if (threadIdx.x < J) {
    const int p = t * J + threadIdx.x;
    const int s = m.pair_slot[p];
    ss[threadIdx.x] = s;
    rs[threadIdx.x] = s >= 0 ? pool.slot_rank[s] : 0;
    cs[threadIdx.x] = s >= 0 ? m.pair_scale[p] * pool.slot_scale[s] : 0.f;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < J * R; i += kExpandThreads) {
    const int j = i / R, q = i - j * R;
    float v = 0.f;
    if (ss[j] >= 0 && q < rs[j]) {
      const size_t p = static_cast<size_t>(t) * J + j;
      for (int kc = 0; kc < n_kc; ++kc) v += m.vpart[(static_cast<size_t>(kc) * m.n + p) * R + q];
    }
    vs[j][q] = v;
  }
  __syncthreads();
  const int o0 = (blockIdx.x * kExpandThreads + threadIdx.x) * kExpandCols;
  if (o0 >= D) return;
  const int ncol = min(kExpandCols, D - o0);
  float acc[kExpandCols];
  float* yrow = y + static_cast<size_t>(t) * D + o0;
#pragma unroll
  for (int c = 0; c < kExpandCols; ++c) acc[c] = c < ncol ? yrow[c] : 0.f;
  for (int j = 0; j < J; ++j) {
    const int s = ss[j];
    if (s < 0) continue;
    const int nvec = (rs[j] + 7) / 8;                  // 16-byte vectors covering the true rank
    float d[kExpandCols];
#pragma unroll
    for (int c = 0; c < kExpandCols; ++c) {
      d[c] = 0.f;
      if (c < ncol) {
        const uint16_t* brow = pool.B + (static_cast<size_t>(s) * D + o0 + c) * R;
        for (int u = 0; u < nvec; ++u) {
          const uint4 bv = *reinterpret_cast<const uint4*>(brow + 8 * u);
          const float* v = &vs[j][8 * u];
          float a = d[c];
          a = fmaf(ptx::bf16_lo(bv.x), v[0], a);
          a = fmaf(ptx::bf16_hi(bv.x), v[1], a);
          a = fmaf(ptx::bf16_lo(bv.y), v[2], a);
          a = fmaf(ptx::bf16_hi(bv.y), v[3], a);
          a = fmaf(ptx::bf16_lo(bv.z), v[4], a);
          a = fmaf(ptx::bf16_hi(bv.z), v[5], a);
          a = fmaf(ptx::bf16_lo(bv.w), v[6], a);
          a = fmaf(ptx::bf16_hi(bv.w), v[7], a);
          d[c] = a;
        }
      }
    }
#pragma unroll
    for (int c = 0; c < kExpandCols; ++c) acc[c] = fmaf(cs[j], d[c], acc[c]);
  }
#pragma unroll
  for (int c = 0; c < kExpandCols; ++c)
    if (c < ncol) yrow[c] = acc[c];
}

}  // namespace

int shrink_k_chunk(int K) {
  int per = (K + kShrinkSplits - 1) / kShrinkSplits;
  return ((per + 255) / 256) * 256;
}

cudaError_t launch_lora_shrink(const uint16_t* x, const PoolView& pool, const MetaView& m, int num_sms,
                               cudaStream_t s) {
  if (m.n == 0) return cudaSuccess;
  const int kc = shrink_k_chunk(pool.K);
  const int n_kc = (pool.K + kc - 1) / kc;
  const int max_items = m.n * n_kc;                     // blocks <= pairs
  int grid = num_sms * 8;
  if (grid > max_items) grid = max_items;
  note_launch_begin(kKindShrink, s);
  lora_shrink_kernel<<<grid, kShrinkThreads, 0, s>>>(x, pool, m, kc, n_kc);
  cudaError_t e = cudaGetLastError();
  note_launch_end(kKindShrink, s);
  return e;
}

cudaError_t launch_lora_expand(float* y, const PoolView& pool, const MetaView& m, cudaStream_t s) {
  if (m.n == 0 || pool.D == 0) return cudaSuccess;
  const int kc = shrink_k_chunk(pool.K);
  const int n_kc = (pool.K + kc - 1) / kc;
  dim3 grid((pool.D + kExpandThreads * kExpandCols - 1) / (kExpandThreads * kExpandCols), m.T);
  note_launch_begin(kKindExpand, s);
  lora_expand_kernel<<<grid, kExpandThreads, 0, s>>>(y, pool, m, n_kc);
  cudaError_t e = cudaGetLastError();
  note_launch_end(kKindExpand, s);
  return e;
}

}  // namespace mlora
