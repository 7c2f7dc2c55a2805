// LoRA on the token embedding lookup:
//
//     y[t, :] = E[id_t, :] + sum_{j : slot[t,j] != -1} s[t,j] c(slot) B_slot A_slot[:, id_t]
//
// "[vLLM] LoRA" (secrett2633 blog), layer-implementation section: the embedding is one of the
// LoRA layer variants (VocabParallelEmbeddingWithLoRA); "LoRA Serving" (vLLM learning book
// ch. 09-04), sections 2 and 6: it is served through the same per-token slot mapping as the
// linear variants. The lookup of id i is the linear map of the one-hot vector e_i with weight
// E^T, so an adapter (A [r, V], B [D, r]) adds c B A[:, i] ("Multi-LoRA Serving Explained",
// LoRA basics; "[vLLM] LoRA", PEFTHelper for c): the shrink is a gather of one column of A and
// the expand is the linear layer's.
//
// An embedding pool keeps A token-major: A^T [V, C], row i holding column i of every slot's A
// (slot s at columns off_s .. off_s + width_s - 1 of the slot space), so a token's shrink is
// one contiguous read of its r values; B is [D, C] as for the linear pools. Work is HBM-bound
// (the table rows and y dominate), so it runs on the CUDA cores with coalesced rows:
//   - one slot per token: item = (group of at most 16 pairs of one slot, column range), the
//     groups being the metadata's pair-blocks plus groups of the sentinel pairs (which take the
//     table row alone). The block's scaled A columns sit in shared memory; each thread owns two
//     adjacent output columns, reads their B row segments once for the whole group and writes
//     each token's y once (no read-modify-write).
//   - several slots per token: item = (token, column range), slots added in order j.
// Every output is a fixed sequence of fp32 operations. A token id outside [0, V) gives a zero
// row and sets ptx::kErrBadId in the metadata's error word.
#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace mlora {
namespace {

constexpr int kEmbThreads = 256;
constexpr int kEmbCpt = 2;                  // adjacent output columns per thread
constexpr int kEmbColsPerItem = 512;        // columns per item ...
constexpr int kEmbMaxColsPerItem = 4096;    // ... doubled up to this while items still fill the SMs

__device__ __forceinline__ float bf16_f32(uint16_t h) { return __uint_as_float(static_cast<uint32_t>(h) << 16); }

// sum_e b[e] v[e] over 8 bf16 values of b (one 16-byte vector) in a fixed order.
__device__ __forceinline__ float dot8(const uint4& b, const float* v) {
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

// Two adjacent bf16 table entries as floats (0 for a rejected id).
__device__ __forceinline__ float2 table_pair(const uint16_t* E, int row, int D, int o) {
  if (row < 0) return make_float2(0.f, 0.f);
  const uint32_t w = __ldg(reinterpret_cast<const unsigned int*>(E + static_cast<size_t>(row) * D + o));
  return make_float2(ptx::bf16_lo(w), ptx::bf16_hi(w));
}

// The 8 bf16 values of a 16-byte vector as floats.
__device__ __forceinline__ void unpack8(const uint4& w, float* f) {
  f[0] = ptx::bf16_lo(w.x);
  f[1] = ptx::bf16_hi(w.x);
  f[2] = ptx::bf16_lo(w.y);
  f[3] = ptx::bf16_hi(w.y);
  f[4] = ptx::bf16_lo(w.z);
  f[5] = ptx::bf16_hi(w.z);
  f[6] = ptx::bf16_lo(w.w);
  f[7] = ptx::bf16_hi(w.w);
}

__global__ void __launch_bounds__(kEmbThreads, 3)
embedding_segment_kernel(const int32_t* __restrict__ ids, const uint16_t* __restrict__ E, float* __restrict__ y,
                         PoolView pool, MetaView m, int n_dchunk, int cols) {
  __shared__ __align__(16) float vs[kPairBlock][kMaxRank];
  __shared__ int tok[kPairBlock], row[kPairBlock];
  const int n_sent = m.n - m.counts[1];                        // sentinel pairs lead the order
  const int n_sg = (n_sent + kPairBlock - 1) / kPairBlock;
  const int items = (n_sg + m.counts[2]) * n_dchunk;
  const int V = pool.K, D = pool.D, C = pool.C;
  for (int item = blockIdx.x; item < items; item += gridDim.x) {
    const int g = item / n_dchunk, dc = item - g * n_dchunk;
    int slot = -1, start, cnt;
    if (g < n_sg) {
      start = g * kPairBlock;
      cnt = min(kPairBlock, n_sent - start);
    } else {
      const int b = g - n_sg;
      slot = m.blk_slot[b];
      start = m.blk_start[b];
      cnt = m.blk_count[b];
    }
    const int rank = slot >= 0 ? pool.slot_rank[slot] : 0;
    const int off = slot >= 0 ? pool.slot_off[slot] : 0;
    const float c = slot >= 0 ? pool.slot_scale[slot] : 0.f;
    const int rpad = (rank + 7) & ~7;
    __syncthreads();                                           // previous item's tables are read
    if (threadIdx.x < cnt) {
      const int p = m.order[start + threadIdx.x];              // one slot per token: token = pair
      const int id = ids[p];
      const bool ok = id >= 0 && id < V;
      if (!ok && dc == 0) atomicOr(m.err, ptx::kErrBadId);
      tok[threadIdx.x] = p;
      row[threadIdx.x] = ok ? id : -1;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < cnt * rpad; i += kEmbThreads) {
      const int pi = i / rpad, q = i - pi * rpad;
      const int id = row[pi];
      const float coef = c * m.pair_scale[tok[pi]];
      vs[pi][q] = (q < rank && id >= 0) ? coef * bf16_f32(pool.A[static_cast<size_t>(id) * C + off + q]) : 0.f;
    }
    __syncthreads();
    const int nu = rpad / 8;
    for (int o = dc * cols + threadIdx.x * kEmbCpt; o < min(D, (dc + 1) * cols); o += kEmbThreads * kEmbCpt) {
      // B rows o and o + 1 of the slot, 8 columns per step, the next step's vectors loaded
      // while this one is multiplied
      const uint4* b0 = reinterpret_cast<const uint4*>(pool.B + static_cast<size_t>(o) * C + off);
      const uint4* b1 = reinterpret_cast<const uint4*>(pool.B + static_cast<size_t>(o + 1) * C + off);
      uint4 n0 = make_uint4(0u, 0u, 0u, 0u), n1 = n0;
      if (nu > 0) {
        n0 = __ldg(b0);
        n1 = __ldg(b1);
      }
      float d[kPairBlock][kEmbCpt];
#pragma unroll
      for (int i = 0; i < kPairBlock; ++i) {
        d[i][0] = 0.f;
        d[i][1] = 0.f;
      }
      for (int u = 0; u < nu; ++u) {
        float f0[8], f1[8];
        unpack8(n0, f0);
        unpack8(n1, f1);
        if (u + 1 < nu) {
          n0 = __ldg(b0 + u + 1);
          n1 = __ldg(b1 + u + 1);
        }
#pragma unroll
        for (int i = 0; i < kPairBlock; ++i) {
          if (i < cnt) {
            const float4 va = *reinterpret_cast<const float4*>(&vs[i][8 * u]);
            const float4 vb = *reinterpret_cast<const float4*>(&vs[i][8 * u + 4]);
            const float v[8] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              d[i][0] = fmaf(f0[k], v[k], d[i][0]);
              d[i][1] = fmaf(f1[k], v[k], d[i][1]);
            }
          }
        }
      }
#pragma unroll
      for (int i = 0; i < kPairBlock; ++i) {
        if (i < cnt) {
          const float2 ev = table_pair(E, row[i], D, o);
          *reinterpret_cast<float2*>(y + static_cast<size_t>(tok[i]) * D + o) = make_float2(ev.x + d[i][0], ev.y + d[i][1]);
        }
      }
    }
  }
}

__global__ void __launch_bounds__(kEmbThreads)
embedding_token_kernel(const int32_t* __restrict__ ids, const uint16_t* __restrict__ E, float* __restrict__ y,
                       PoolView pool, MetaView m, int n_dchunk, int cols) {
  __shared__ __align__(16) float vs[kMaxJ][kMaxRank];
  __shared__ int ss[kMaxJ], rs[kMaxJ], os[kMaxJ];
  __shared__ float cs[kMaxJ];
  __shared__ int s_row;
  const int J = m.J, R = pool.R, V = pool.K, D = pool.D, C = pool.C;
  const int items = m.T * n_dchunk;
  for (int item = blockIdx.x; item < items; item += gridDim.x) {
    const int t = item / n_dchunk, dc = item - t * n_dchunk;
    __syncthreads();
    if (threadIdx.x == 0) {
      const int id = ids[t];
      const bool ok = id >= 0 && id < V;
      if (!ok && dc == 0) atomicOr(m.err, ptx::kErrBadId);
      s_row = ok ? id : -1;
    }
    if (threadIdx.x < J) {
      const int p = t * J + threadIdx.x;
      const int s = m.pair_slot[p];
      ss[threadIdx.x] = s;
      rs[threadIdx.x] = s >= 0 ? pool.slot_rank[s] : 0;
      os[threadIdx.x] = s >= 0 ? pool.slot_off[s] : 0;
      cs[threadIdx.x] = s >= 0 ? pool.slot_scale[s] * m.pair_scale[p] : 0.f;
    }
    __syncthreads();
    const int id = s_row;
    for (int i = threadIdx.x; i < J * R; i += kEmbThreads) {
      const int j = i / R, q = i - j * R;
      vs[j][q] = (ss[j] >= 0 && q < rs[j] && id >= 0)
                     ? cs[j] * bf16_f32(pool.A[static_cast<size_t>(id) * C + os[j] + q]) : 0.f;
    }
    __syncthreads();
    for (int o = dc * cols + threadIdx.x * kEmbCpt; o < min(D, (dc + 1) * cols); o += kEmbThreads * kEmbCpt) {
      const float2 ev = table_pair(E, id, D, o);
      float acc[kEmbCpt] = {ev.x, ev.y};
      for (int j = 0; j < J; ++j) {
        if (ss[j] < 0) continue;
        const int nu = (rs[j] + 7) / 8;
#pragma unroll
        for (int e = 0; e < kEmbCpt; ++e) {
          const uint4* brow = reinterpret_cast<const uint4*>(pool.B + static_cast<size_t>(o + e) * C + os[j]);
          float dd = 0.f;
          for (int u = 0; u < nu; ++u) dd += dot8(__ldg(brow + u), &vs[j][8 * u]);
          acc[e] += dd;
        }
      }
      *reinterpret_cast<float2*>(y + static_cast<size_t>(t) * D + o) = make_float2(acc[0], acc[1]);
    }
  }
}

// A^T[v][off + q] = stage[q][v] (an adapter's A [r, V] staged whole) for q < r, 0 for r <= q <
// width: item = (8-column group g, id v), v fastest, so a warp reads each staged row
// coalesced and writes one 16-byte segment per id.
__global__ void scatter_slot_at_kernel(uint16_t* __restrict__ At, int C, int off, int width, int V,
                                       const uint16_t* __restrict__ stage, int r) {
  const long items = static_cast<long>(width / 8) * V;
  for (long item = blockIdx.x * static_cast<long>(blockDim.x) + threadIdx.x; item < items;
       item += static_cast<long>(gridDim.x) * blockDim.x) {
    const int g = static_cast<int>(item / V), v = static_cast<int>(item - static_cast<long>(g) * V);
    uint32_t w[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const int q0 = 8 * g + 2 * h, q1 = q0 + 1;
      const uint32_t lo = q0 < r ? stage[static_cast<size_t>(q0) * V + v] : 0u;
      const uint32_t hi = q1 < r ? stage[static_cast<size_t>(q1) * V + v] : 0u;
      w[h] = lo | (hi << 16);
    }
    *reinterpret_cast<uint4*>(At + static_cast<size_t>(v) * C + off + 8 * g) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

}  // namespace

cudaError_t launch_embedding(const int32_t* ids, const uint16_t* E, float* y, const PoolView& pool, const MetaView& m,
                             int num_sms, cudaStream_t s) {
  if (m.T == 0 || pool.D == 0) return cudaSuccess;
  // groups of one slot per token: at most ceil(n / 16) sentinel groups plus n pair-blocks
  const long lo_rows = m.J == 1 ? (m.n + kPairBlock - 1) / kPairBlock : m.T;
  int cols = kEmbColsPerItem;
  while (cols < kEmbMaxColsPerItem && lo_rows * ((pool.D + 2 * cols - 1) / (2 * cols)) >= 8L * num_sms) cols *= 2;
  const int n_dchunk = (pool.D + cols - 1) / cols;
  const long max_items = (m.J == 1 ? (m.n + kPairBlock - 1) / kPairBlock + m.n : static_cast<long>(m.T)) * n_dchunk;
  const int grid = static_cast<int>(std::min<long>(max_items, 8L * num_sms));
  note_launch_begin(kKindEmbed, s);
  if (m.J == 1)
    embedding_segment_kernel<<<grid, kEmbThreads, 0, s>>>(ids, E, y, pool, m, n_dchunk, cols);
  else
    embedding_token_kernel<<<grid, kEmbThreads, 0, s>>>(ids, E, y, pool, m, n_dchunk, cols);
  cudaError_t e = cudaGetLastError();
  note_launch_end(kKindEmbed, s);
  return e;
}

cudaError_t launch_scatter_slot_at(uint16_t* At, int C, int off, int width, int V, const uint16_t* stage, int r,
                                   cudaStream_t s) {
  const long items = static_cast<long>(width / 8) * V;
  const int grid = static_cast<int>(std::min<long>((items + 255) / 256, 4096));
  scatter_slot_at_kernel<<<grid, 256, 0, s>>>(At, C, off, width, V, stage, r);
  return cudaGetLastError();
}

}  // namespace mlora
