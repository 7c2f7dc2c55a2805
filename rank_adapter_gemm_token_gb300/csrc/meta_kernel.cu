// Per-step slot metadata: a stable counting sort of the step's (token, slot) pairs by slot.
//
// "Multi-LoRA Serving Explained" (sevydevy.com), batched-serving section: the segmented
// method orders tokens with a stable argsort of their slot ids and runs one small product
// per group, so each adapter is read once per group; the same page reports that the vLLM
// kernel path sorts the batch by slot before shrink and expand, and skips the LoRA kernels
// when no token uses an adapter. "[RFC] Per-request activation of multiple LoRA adapters"
// (vLLM issue 51940), Proposed Change item 2: k slots per token, unused ones the sentinel.
//
// One CTA of 1024 threads does the whole sort: a shared-memory histogram over the S + 1
// bins (bin 0 = sentinel), one block-wide exclusive scan (bin starts, segment numbers and
// pair-block numbers at once), then a scatter in chunks of 1024 pairs in which each pair's
// rank inside its bin is (pairs of the same bin in earlier chunks) + (in earlier warps of
// this chunk) + (in earlier lanes of its warp, from __match_any_sync). The result is
// exactly the stable order; it does not depend on thread timing.
#include <climits>

#include "internal.h"
#include "ptx.cuh"

namespace mlora {
namespace {

// Dynamic shared memory of the metadata kernel: the per-bin arrays (80 B per slot bin, up to
// 164 KB at 2048 slots) plus, when they fit, four int arrays over the pairs (16 B per pair).
// The kernel's static arrays (~11 KB) come on top, within the 227 KB a block may use.
constexpr size_t kMetaMaxDynSmem = 200 * 1024;

__device__ __forceinline__ void block_exclusive_scan3(int a, int b, int c, int& pa, int& pb, int& pc,
                                                      int* warp_sums /* [3][32] */) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int sa = a, sb = b, sc = c;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    int ta = __shfl_up_sync(0xffffffffu, sa, d), tb = __shfl_up_sync(0xffffffffu, sb, d),
        tc = __shfl_up_sync(0xffffffffu, sc, d);
    if (lane >= d) { sa += ta; sb += tb; sc += tc; }
  }
  if (lane == 31) { warp_sums[warp] = sa; warp_sums[32 + warp] = sb; warp_sums[64 + warp] = sc; }
  __syncthreads();
  if (warp == 0) {
    int wa = warp_sums[lane], wb = warp_sums[32 + lane], wc = warp_sums[64 + lane];
    int xa = wa, xb = wb, xc = wc;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      int ta = __shfl_up_sync(0xffffffffu, xa, d), tb = __shfl_up_sync(0xffffffffu, xb, d),
          tc = __shfl_up_sync(0xffffffffu, xc, d);
      if (lane >= d) { xa += ta; xb += tb; xc += tc; }
    }
    warp_sums[lane] = xa - wa; warp_sums[32 + lane] = xb - wb; warp_sums[64 + lane] = xc - wc;
  }
  __syncthreads();
  pa = warp_sums[warp] + sa - a;
  pb = warp_sums[32 + warp] + sb - b;
  pc = warp_sums[64 + warp] + sc - c;
  __syncthreads();
}

__global__ void __launch_bounds__(kMetaThreads, 1)
build_meta_kernel(const int32_t* __restrict__ token_slots, const float* __restrict__ scales, int n, int S,
                  const int32_t* __restrict__ slot_rank, MetaView m, int cache) {
  extern __shared__ int smem[];
  const int nb = S + 1;
  int* hist = smem;                          // [nb] pairs per bin
  int* cursor = hist + nb;                   // [nb] next free position of each bin
  int* chunk_tot = cursor + nb;              // [nb] pairs per bin in the current chunk
  int* actidx = chunk_tot + nb;              // [nb] index among the active slots (-1: none)
  uint16_t* wcnt = reinterpret_cast<uint16_t*>(actidx + nb);   // [32][nb]
  // small steps keep their pair slots, order and pair-blocks in shared memory as well, so the
  // later steps read them there instead of going back to global memory
  int* c_base = reinterpret_cast<int*>(wcnt + 32 * nb);
  int* pslot = cache ? c_base : m.pair_slot;            // [n] validated slot per pair
  int* ord = cache ? c_base + n : m.order;              // [n] sorted pair order
  int* bstart = cache ? c_base + 2 * n : m.blk_start;   // [n] pair-block starts
  int* bcount = cache ? c_base + 3 * n : m.blk_count;   // [n] pair-block sizes
  __shared__ int warp_sums[96];
  __shared__ int first_bad;
  __shared__ int n_blk_sh;                               // pair-blocks in total
  __shared__ int ovf_n, ovf_a, ovf_b;                    // overflow tiles: count, first two
  __shared__ int tile_cnt[kMaxTiles];                    // distinct slots per 128-token M-tile
  __shared__ int tile_list[kMaxTiles * kTileSlots];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  ptx::grid_dependents_launch();             // the first linear's GEMM may start its set-up
  // the first chunk's inputs are loaded while the slot table is staged
  const int s_first = tid < n ? token_slots[tid] : -1;
  const float c_first = tid < n && scales ? scales[tid] : 1.0f;
  // 0. which slots hold an adapter (staged once, so pair validation needs no dependent load);
  //    `cursor` is free until step 2
  for (int b = tid; b < nb; b += kMetaThreads) {
    hist[b] = 0;
    if (b < S) cursor[b] = slot_rank[b] > 0;
  }
  if (tid == 0) first_bad = INT_MAX;
  __syncthreads();

  // 1. validate, histogram, per-pair slot and scale; the first chunk's bins stay in registers
  int first_bin = nb;
  for (int p = tid; p < n; p += kMetaThreads) {
    int s = p < kMetaThreads ? s_first : token_slots[p];
    const bool ok = (s == -1) || (s >= 0 && s < S && cursor[s]);
    if (!ok) {
      atomicMin(&first_bad, p);
      s = -1;
    }
    m.pair_slot[p] = s;
    if (cache) pslot[p] = s;
    m.pair_scale[p] = (s < 0) ? 0.0f : (p < kMetaThreads ? c_first : (scales ? scales[p] : 1.0f));
    atomicAdd(&hist[s + 1], 1);
    if (p < kMetaThreads) first_bin = s + 1;
  }
  __syncthreads();

  // 2. one scan for bin starts, segment numbers and pair-block numbers
  const int per = (nb + kMetaThreads - 1) / kMetaThreads;
  const int b0 = min(tid * per, nb), b1 = min(b0 + per, nb);
  int h = 0, f = 0, k = 0;
  for (int b = b0; b < b1; ++b) {
    const int c = hist[b];
    h += c;
    f += c > 0;
    if (b > 0) k += (c + kPairBlock - 1) / kPairBlock;
  }
  int ph, pf, pk;
  block_exclusive_scan3(h, f, k, ph, pf, pk, warp_sums);
  const int has_sentinel = hist[0] > 0;
  for (int b = b0; b < b1; ++b) {
    const int c = hist[b];
    cursor[b] = ph;
    actidx[b] = -1;
    if (c > 0) {
      m.seg_slot[pf] = b - 1;
      m.seg_off[pf] = ph;
      if (b > 0) {
        actidx[b] = pf - has_sentinel;
        m.act_slot[pf - has_sentinel] = b - 1;
      }
      ++pf;
      if (b > 0) {
        for (int i = 0; i * kPairBlock < c; ++i, ++pk) {
          m.blk_slot[pk] = b - 1;
          m.blk_start[pk] = ph + i * kPairBlock;
          m.blk_count[pk] = min(kPairBlock, c - i * kPairBlock);
          if (cache) {
            bstart[pk] = ph + i * kPairBlock;
            bcount[pk] = min(kPairBlock, c - i * kPairBlock);
          }
        }
      }
    }
    ph += c;
  }
  if (b1 == nb && b0 < b1) {                 // the thread owning the last bin holds the totals
    m.seg_off[pf] = n;
    m.counts[0] = pf;
    m.counts[1] = n - hist[0];
    m.counts[2] = pk;
    m.counts[4] = pf - has_sentinel;
    n_blk_sh = pk;
  }
  __syncthreads();

  // 3. stable scatter, 1024 pairs per chunk
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int base = 0; base < n; base += kMetaThreads) {
    for (int i = tid; i < 32 * nb; i += kMetaThreads) wcnt[i] = 0;
    __syncthreads();
    const int p = base + tid;
    const bool valid = p < n;
    const int bin = !valid ? nb : (base == 0 ? first_bin : pslot[p] + 1);   // nb = "no pair"
    const unsigned peers = __match_any_sync(0xffffffffu, bin);
    const int rank_in_warp = __popc(peers & lt_mask);
    if (valid && lane == __ffs(peers) - 1) wcnt[warp * nb + bin] = static_cast<uint16_t>(__popc(peers));
    __syncthreads();
    for (int b = tid; b < nb; b += kMetaThreads) {
      int run = 0;
      for (int w = 0; w < 32; ++w) {
        const int c = wcnt[w * nb + b];
        wcnt[w * nb + b] = static_cast<uint16_t>(run);
        run += c;
      }
      chunk_tot[b] = run;
    }
    __syncthreads();
    if (valid) {
      const int pos = cursor[bin] + wcnt[warp * nb + bin] + rank_in_warp;
      m.order[pos] = p;
      if (cache) ord[pos] = p;
      m.pair_act[p] = actidx[bin];
    }
    __syncthreads();
    for (int b = tid; b < nb; b += kMetaThreads) cursor[b] += chunk_tot[b];
    __syncthreads();
  }

  // Steps 4 and 5 serve only the tensor-core prefill path, which batches of at most
  // kSkinnyMaxT tokens never take (they use the small-batch path or the CUDA-core kernels).
  if (m.T <= kSkinnyMaxT) {
    if (tid == 0) {
      m.counts[3] = first_bad;
      m.counts[5] = 0;
      m.counts[6] = -1;
      m.counts[7] = -1;
      if (first_bad != INT_MAX) atomicOr(m.err, ptx::kErrBadSlot);
    }
    return;
  }

  // 4. slots of each 128-token M-tile (x order), for the tensor-core prefill path: within a
  //    segment the pairs are in token order, so the first pair of each (slot, tile) run adds the
  //    slot to that tile's list; a tile with more than kTileSlots slots overflows.
  const int n_tiles = (m.T + 127) / 128;
  for (int i = tid; i < n_tiles; i += kMetaThreads) tile_cnt[i] = 0;
  __syncthreads();
  for (int i = tid; i < n; i += kMetaThreads) {
    const int p = ord[i];
    const int s = pslot[p];
    if (s < 0) continue;
    const int tile = (p / m.J) >> 7;
    bool first = true;
    if (i > 0) {
      const int q = ord[i - 1];
      first = pslot[q] != s || ((q / m.J) >> 7) != tile;
    }
    if (first) {
      const int k = atomicAdd(&tile_cnt[tile], 1);
      if (k < kTileSlots) tile_list[tile * kTileSlots + k] = s;
    }
  }
  __syncthreads();
  for (int tile = tid; tile < n_tiles; tile += kMetaThreads) {   // ascending slot order per tile
    const int c = tile_cnt[tile];
    int* l = &tile_list[tile * kTileSlots];
    const int k = c < kTileSlots ? c : kTileSlots;
    for (int a = 1; a < k; ++a)
      for (int b = a; b > 0 && l[b - 1] > l[b]; --b) {
        const int t = l[b];
        l[b] = l[b - 1];
        l[b - 1] = t;
      }
    m.tile_info[tile * (kTileSlots + 1)] = c;
    for (int a = 0; a < kTileSlots; ++a) m.tile_info[tile * (kTileSlots + 1) + 1 + a] = a < k ? l[a] : -1;
  }
  __syncthreads();
  for (int p = tid; p < n; p += kMetaThreads)
    m.pair_fused[p] = pslot[p] >= 0 && tile_cnt[(p / m.J) >> 7] <= kTileSlots;

  // the overflow window: with one or two overflow tiles, counts[6] and counts[7] name them in
  // ascending order (counts[7] = -1 for one); otherwise both are -1 (none, or too many)
  if (tid == 0) {
    ovf_n = 0;
    ovf_a = INT_MAX;
    ovf_b = INT_MAX;
  }
  __syncthreads();
  for (int tile = tid; tile < n_tiles; tile += kMetaThreads)
    if (tile_cnt[tile] > kTileSlots) {
      atomicAdd(&ovf_n, 1);
      atomicMin(&ovf_a, tile);
    }
  __syncthreads();
  for (int tile = tid; tile < n_tiles; tile += kMetaThreads)
    if (tile_cnt[tile] > kTileSlots && tile != ovf_a) atomicMin(&ovf_b, tile);
  __syncthreads();
  if (tid == 0) {
    const bool win = ovf_n == 1 || ovf_n == 2;
    m.counts[6] = win ? ovf_a : -1;
    m.counts[7] = win && ovf_n == 2 ? ovf_b : -1;
  }

  // 5. the pair-blocks that still need the CUDA-core shrink/expand (a pair in an overflow tile),
  //    in ascending order, so those kernels skip the fused blocks without looking at them
  {
    auto todo = [&](int b) {
      const int start = bstart[b], cnt = bcount[b];
      bool t = false;
      for (int i = 0; i < cnt; ++i) t |= tile_cnt[(ord[start + i] / m.J) >> 7] > kTileSlots;
      return t;
    };
    const int nblk = n_blk_sh;
    const int per_b = (nblk + kMetaThreads - 1) / kMetaThreads;
    const int c0 = min(tid * per_b, nblk), c1 = min(c0 + per_b, nblk);
    int mine = 0;
    for (int b = c0; b < c1; ++b) mine += todo(b);
    int pos, unused0, unused1;
    block_exclusive_scan3(mine, 0, 0, pos, unused0, unused1, warp_sums);
    if (tid == kMetaThreads - 1) m.counts[5] = pos + mine;
    for (int b = c0; b < c1; ++b)
      if (todo(b)) m.todo_blk[pos++] = b;
  }

  if (tid == 0) {
    m.counts[3] = first_bad;
    if (first_bad != INT_MAX) atomicOr(m.err, ptx::kErrBadSlot);
  }
}

}  // namespace

cudaError_t launch_build_meta(const int32_t* token_slots, const float* scales, int T, int J, int S,
                              const int32_t* slot_rank, const MetaView& m, cudaStream_t s) {
  const int nb = S + 1;
  const int n = T * J;
  const size_t bins = static_cast<size_t>(nb) * (4 * sizeof(int) + 32 * sizeof(uint16_t));
  const int cache = bins + static_cast<size_t>(n) * 4 * sizeof(int) <= kMetaMaxDynSmem ? 1 : 0;
  const size_t smem = bins + (cache ? static_cast<size_t>(n) * 4 * sizeof(int) : 0);
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(build_meta_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kMetaMaxDynSmem));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  note_launch_begin(kKindMeta, s);
  build_meta_kernel<<<1, kMetaThreads, smem, s>>>(token_slots, scales, n, S, slot_rank, m, cache);
  cudaError_t e = cudaGetLastError();
  note_launch_end(kKindMeta, s);
  return e;
}

}  // namespace mlora
