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
#include <algorithm>
#include <climits>

#include "internal.h"
#include "ptx.cuh"

namespace mlora {
namespace {

// Dynamic shared memory of the metadata kernel: the per-bin arrays (80 B per slot bin, up to
// 164 KB at 2048 slots; later reused for two column-block bitmaps per warp) plus, when they fit,
// four int arrays over the pairs (16 B per pair). The kernel's static arrays (~10 KB) come on
// top, within the 227 KB a block may use.
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

// Bitmap (n_words words) of the column blocks owned by the slots of M-tile `tile`'s active pairs,
// built by one warp without atomics. slot_blk[s] holds the first block of slot s in its low 16
// bits and the last in its high 16 bits (a slot of width w at column offset off covers blocks
// off / 64 .. (off + w - 1) / 64). Per round of 32 pairs and per block of their slots, the lanes
// OR their bits word by word (one warp reduction per distinct word in the round).
__device__ __forceinline__ void tile_block_bitmap(uint32_t* bm, int n_words, int tile, int T, int J,
                                                  const int* pslot, const uint32_t* slot_blk) {
  const int lane = threadIdx.x & 31;
  for (int k = lane; k < n_words; k += 32) bm[k] = 0u;
  __syncwarp();
  const int p0 = tile * 128 * J, p1 = min(T, tile * 128 + 128) * J;
  for (int pb = p0; pb < p1; pb += 32) {
    const int p = pb + lane;
    const int s = p < p1 ? pslot[p] : -1;
    const uint32_t sb = s >= 0 ? slot_blk[s] : 0u;
    const int b0 = static_cast<int>(sb & 0xFFFFu);
    const int nblk = s >= 0 ? static_cast<int>(sb >> 16) - b0 + 1 : 0;
    int more = __reduce_max_sync(0xffffffffu, nblk);
    for (int i = 0; i < more; ++i) {
      const bool has = i < nblk;
      const int b = b0 + i;
      const uint32_t w = has ? static_cast<uint32_t>(b >> 5) : 0xFFFFFFFFu;
      unsigned todo = __ballot_sync(0xffffffffu, has);
      while (todo) {
        const uint32_t ww = __shfl_sync(0xffffffffu, w, __ffs(todo) - 1);
        const bool mine = has && w == ww;
        const uint32_t bits = __reduce_or_sync(0xffffffffu, mine ? (1u << (b & 31)) : 0u);
        todo &= ~__ballot_sync(0xffffffffu, mine);
        if (lane == 0) bm[ww] |= bits;
      }
    }
  }
  __syncwarp();
}

// Writes the positions of the set bits of a warp's bitmap in ascending order: bit b of the map
// goes to out[base + rank of b]; one word per step, the lanes taking its 32 bits.
template <typename F>
__device__ __forceinline__ void emit_bits(const uint32_t* bm, int n_words, F&& put) {
  const int lane = threadIdx.x & 31;
  int run = 0;
  for (int k = 0; k < n_words; ++k) {
    const uint32_t w = bm[k];
    if (w == 0u) continue;                               // uniform: every lane reads the same word
    if ((w >> lane) & 1u) put(k * 32 + lane, run + __popc(w & ((1u << lane) - 1u)));
    run += __popc(w);
  }
}

__global__ void __launch_bounds__(kMetaThreads, 1)
build_meta_kernel(const int32_t* __restrict__ token_slots, const float* __restrict__ scales, int n, PoolView pool,
                  MetaView m, int cache, int keep, int mode) {
  extern __shared__ int smem[];
  const int S = pool.S;
  const int nb = S + 1;
  int* hist = smem;                          // [nb] pairs per bin
  int* cursor = hist + nb;                   // [nb] next free position of each bin
  int* chunk_tot = cursor + nb;              // [nb] pairs per bin in the current chunk
  int* actidx = chunk_tot + nb;              // [nb] index among the active slots (-1: none)
  uint16_t* wcnt = reinterpret_cast<uint16_t*>(actidx + nb);   // [32][nb]
  const int n_blocks = (pool.C + kBlockCols - 1) / kBlockCols;  // column blocks of the slot space
  const int n_words = (n_blocks + 31) / 32;
  // after the sort the bins' area holds block bitmaps: with `keep`, one per M-tile, built once and
  // read by every later step; otherwise two per warp, rebuilt where needed (the host sized it)
  uint32_t* bitmaps = reinterpret_cast<uint32_t*>(smem);
  const size_t bins_bytes = static_cast<size_t>(nb) * (4 * sizeof(int) + 32 * sizeof(uint16_t));
  const int n_tiles_all = (m.T + 127) / 128;
  const size_t bm_bytes = (keep ? static_cast<size_t>(n_tiles_all) : static_cast<size_t>(32) * 2) * n_words * sizeof(uint32_t);
  const size_t front = ((bins_bytes > bm_bytes ? bins_bytes : bm_bytes) + 15) / 16 * 16;
  uint32_t* slot_blk = reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(smem) + front);   // [S]
  // small steps keep their pair slots, order and pair-blocks in shared memory as well, so the
  // later steps read them there instead of going back to global memory
  int* c_base = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(smem) + front + (static_cast<size_t>(S) * 4 + 15) / 16 * 16);
  int* pslot = cache ? c_base : m.pair_slot;            // [n] validated slot per pair
  int* ord = cache ? c_base + n : m.order;              // [n] sorted pair order
  int* bstart = cache ? c_base + 2 * n : m.blk_start;   // [n] pair-block starts
  int* bcount = cache ? c_base + 3 * n : m.blk_count;   // [n] pair-block sizes
  __shared__ int warp_sums[96];
  __shared__ int first_bad;
  __shared__ int n_blk_sh;                               // pair-blocks in total
  __shared__ int tile_cnt[kMaxTiles];                    // units per 128-token M-tile (0 if it overflows)
  __shared__ int tile_off[kMaxTiles + 1];                // first unit of each M-tile
  __shared__ uint8_t tile_ovf[kMaxTiles];                // 1: the tile's pairs take the CUDA-core kernels
  __shared__ int ptile_cnt[kMaxTiles / 2];               // entries per pair tile

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  ptx::grid_dependents_launch();             // the first linear's kernels may start their set-up
  // the first chunk's inputs are loaded while the slot table is staged
  const bool sort = mode != kMetaUnitsOnly, units = mode != kMetaSortOnly;
  const int s_first = sort && tid < n ? token_slots[tid] : -1;
  const float c_first = sort && tid < n && scales ? scales[tid] : 1.0f;
  // 0. which slots hold an adapter (staged once, so pair validation needs no dependent load);
  //    `cursor` is free until step 2
  for (int b = tid; b < nb; b += kMetaThreads) {
    hist[b] = 0;
    if (b < S) {
      cursor[b] = pool.slot_rank[b] > 0;
      const int off = pool.slot_off[b];
      slot_blk[b] = static_cast<uint32_t>(off / kBlockCols) |
                    (static_cast<uint32_t>((off + pool.slot_width[b] - 1) / kBlockCols) << 16);
    }
  }
  if (tid == 0) first_bad = INT_MAX;
  __syncthreads();

  if (sort) {
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
  } else {
    if (tid == 0) n_blk_sh = m.counts[2];           // the sort of this step ran in an earlier launch
    __syncthreads();
  }

  if (units) {
  // 4. units of the tensor-core side path: for each 128-token M-tile the column blocks its active
  //    pairs' slots own (warp per tile, bitmap over the blocks), counted, capped, numbered.
  const int n_tiles = (m.T + 127) / 128;
  const int n_ptiles = (n_tiles + 1) / 2;
  uint32_t* scratchA = bitmaps + warp * 2 * n_words;     // without `keep`
  uint32_t* scratchB = scratchA + n_words;
  auto tile_map = [&](int i, uint32_t* scratch) -> const uint32_t* {
    if (keep) return bitmaps + static_cast<size_t>(i) * n_words;
    tile_block_bitmap(scratch, n_words, i, m.T, m.J, pslot, slot_blk);
    return scratch;
  };
  for (int i = warp; i < n_tiles; i += 32) {
    uint32_t* bm = keep ? bitmaps + static_cast<size_t>(i) * n_words : scratchA;
    tile_block_bitmap(bm, n_words, i, m.T, m.J, pslot, slot_blk);
    int c = 0;
    for (int w = lane; w < n_words; w += 32) c += __popc(bm[w]);
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) c += __shfl_xor_sync(0xffffffffu, c, d);
    if (lane == 0) tile_cnt[i] = c;
    __syncwarp();
  }
  __syncthreads();
  {
    // a tile with too many units, or whose units would pass the capacity, overflows (every later
    // tile with units then overflows as well, since the units are numbered in tile order)
    const int c = tid < n_tiles ? tile_cnt[tid] : 0;
    const int capped = c <= kMaxTileUnits ? c : 0;
    int off, unused0, unused1;
    block_exclusive_scan3(capped, 0, 0, off, unused0, unused1, warp_sums);
    const bool ovf = c > kMaxTileUnits || off + capped > m.unit_cap;
    const int fin = ovf ? 0 : c;
    int uoff;
    block_exclusive_scan3(fin, 0, 0, uoff, unused0, unused1, warp_sums);
    if (tid < n_tiles) {
      tile_cnt[tid] = fin;
      tile_off[tid] = uoff;
      tile_ovf[tid] = ovf ? 1 : 0;
      m.tile_unit_off[tid] = uoff;
    }
    if (tid == n_tiles - 1) {
      tile_off[n_tiles] = uoff + fin;
      m.tile_unit_off[n_tiles] = uoff + fin;
      m.counts[6] = uoff + fin;
    }
    if (n_tiles == 0 && tid == 0) {
      m.tile_unit_off[0] = 0;
      m.counts[6] = 0;
      m.counts[7] = 0;
    }
  }
  __syncthreads();
  // units in ascending block order per tile
  for (int i = warp; i < n_tiles; i += 32) {
    if (tile_cnt[i] == 0) continue;
    const uint32_t* bm = tile_map(i, scratchA);
    const int ubase = tile_off[i];
    emit_bits(bm, n_words, [&](int b, int r) {
      m.unit_blk[ubase + r] = b;
      m.unit_tile[ubase + r] = i;
    });
  }
  // pair tiles (M-tiles 2 mp and 2 mp + 1): the union of both tiles' blocks, each entry with the
  // unit of either tile on that block (-1 where the tile does not use it)
  for (int mp = warp; mp < n_ptiles; mp += 32) {
    const int ta = 2 * mp, tb = 2 * mp + 1;
    const bool ha = tile_cnt[ta] > 0, hb = tb < n_tiles && tile_cnt[tb] > 0;
    const uint32_t* bmA = ha ? tile_map(ta, scratchA) : nullptr;
    const uint32_t* bmB = hb ? tile_map(tb, scratchB) : nullptr;
    int c = 0;
    for (int w = lane; w < n_words; w += 32) c += __popc((ha ? bmA[w] : 0u) | (hb ? bmB[w] : 0u));
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) c += __shfl_xor_sync(0xffffffffu, c, d);
    if (lane == 0) ptile_cnt[mp] = c;
    __syncwarp();
  }
  __syncthreads();
  {
    // entries of each pair tile, and the shrink's groups of kGroupUnits consecutive entries
    const int c = tid < n_ptiles ? ptile_cnt[tid] : 0;
    const int ng = (c + kGroupUnits - 1) / kGroupUnits;
    int off, goff, unused1;
    block_exclusive_scan3(c, ng, 0, off, goff, unused1, warp_sums);
    if (tid < n_ptiles) m.ptile_off[tid] = off;
    if (tid == n_ptiles - 1) {
      m.ptile_off[n_ptiles] = off + c;
      m.counts[7] = goff + ng;
    }
    if (n_ptiles == 0 && tid == 0) m.ptile_off[0] = 0;
    for (int g = 0; g < ng; ++g) {
      m.grp_mp[goff + g] = tid;
      m.grp_ent[goff + g] = off + g * kGroupUnits;
      m.grp_cnt[goff + g] = min(kGroupUnits, c - g * kGroupUnits);
    }
    // the pair tiles with the most entries first (the pair GEMM hands out their tiles first)
    if (tid < n_ptiles) {
      int r = 0;
      for (int q = 0; q < n_ptiles; ++q) {
        const int cq = ptile_cnt[q];
        r += (cq > c || (cq == c && q < tid)) ? 1 : 0;
      }
      m.ptile_order[r] = tid;
    }
    for (int i = tid; i < n_ptiles + 2; i += kMetaThreads) m.sync[i] = 0u;
    __syncthreads();                                   // every count read before it is replaced
    if (tid < n_ptiles) ptile_cnt[tid] = off;          // from here: first entry of the pair tile
  }
  __syncthreads();
  for (int mp = warp; mp < n_ptiles; mp += 32) {
    const int ta = 2 * mp, tb = 2 * mp + 1;
    const bool ha = tile_cnt[ta] > 0, hb = tb < n_tiles && tile_cnt[tb] > 0;
    if (!ha && !hb) continue;
    const uint32_t* bmA = ha ? tile_map(ta, scratchA) : nullptr;
    const uint32_t* bmB = hb ? tile_map(tb, scratchB) : nullptr;
    const int ua = tile_off[ta], ub = hb ? tile_off[tb] : 0, ebase = ptile_cnt[mp];
    int ra = 0, rb = 0, ru = 0;                          // set bits of earlier words
    for (int k = 0; k < n_words; ++k) {
      const uint32_t wa = ha ? bmA[k] : 0u, wb = hb ? bmB[k] : 0u, wu = wa | wb;
      if (wu == 0u) continue;                              // uniform across the warp
      if ((wu >> lane) & 1u) {
        const uint32_t below = (1u << lane) - 1u;
        const int e = ebase + ru + __popc(wu & below);
        m.pent_blk[e] = k * 32 + lane;
        m.pent_u0[e] = (wa >> lane) & 1u ? ua + ra + __popc(wa & below) : -1;
        m.pent_u1[e] = (wb >> lane) & 1u ? ub + rb + __popc(wb & below) : -1;
      }
      ra += __popc(wa);
      rb += __popc(wb);
      ru += __popc(wu);
    }
  }
  for (int p = tid; p < n; p += kMetaThreads) m.pair_fused[p] = pslot[p] >= 0 && !tile_ovf[(p / m.J) >> 7];

  // 5. the pair-blocks that still need the CUDA-core shrink/expand (a pair in an overflow tile),
  //    in ascending order, so those kernels skip the fused blocks without looking at them
  {
    auto todo = [&](int b) {
      const int start = bstart[b], cnt = bcount[b];
      bool t = false;
      for (int i = 0; i < cnt; ++i) t |= tile_ovf[(ord[start + i] / m.J) >> 7] != 0;
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
  }

  if (sort && tid == 0) {
    m.counts[3] = first_bad;
    if (first_bad != INT_MAX) atomicOr(m.err, ptx::kErrBadSlot);
  }
}

}  // namespace

cudaError_t launch_build_meta(const int32_t* token_slots, const float* scales, int T, int J, const PoolView& pool,
                              const MetaView& m, cudaStream_t s, int mode) {
  const int nb = pool.S + 1;
  const int n = T * J;
  const size_t bins = static_cast<size_t>(nb) * (4 * sizeof(int) + 32 * sizeof(uint16_t));
  const size_t n_words = (static_cast<size_t>(pool.C) + kBlockCols * 32 - 1) / (kBlockCols * 32);
  const size_t n_tiles = (static_cast<size_t>(T) + 127) / 128;
  const size_t slots_bytes = (static_cast<size_t>(pool.S) * 4 + 15) / 16 * 16;
  // keep every tile's bitmap when they fit beside the rest, else two scratch bitmaps per warp
  const size_t kept = n_tiles * n_words * sizeof(uint32_t);
  const size_t scratch = 32 * 2 * n_words * sizeof(uint32_t);
  const int keep = ((std::max(bins, kept) + 15) / 16 * 16 + slots_bytes <= kMetaMaxDynSmem) ? 1 : 0;
  const size_t bitmaps = keep ? kept : scratch;
  const size_t front = ((bins > bitmaps ? bins : bitmaps) + 15) / 16 * 16 + slots_bytes;
  if (front > kMetaMaxDynSmem) return cudaErrorInvalidValue;
  // the units-only pass reads the sort's arrays from global memory
  const int cache = mode != kMetaUnitsOnly && front + static_cast<size_t>(n) * 4 * sizeof(int) <= kMetaMaxDynSmem ? 1 : 0;
  const size_t smem = front + (cache ? static_cast<size_t>(n) * 4 * sizeof(int) : 0);
  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(build_meta_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kMetaMaxDynSmem));
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  note_launch_begin(kKindMeta, s);
  build_meta_kernel<<<1, kMetaThreads, smem, s>>>(token_slots, scales, n, pool, m, cache, keep, mode);
  cudaError_t e = cudaGetLastError();
  note_launch_end(kKindMeta, s);
  return e;
}

}  // namespace mlora
