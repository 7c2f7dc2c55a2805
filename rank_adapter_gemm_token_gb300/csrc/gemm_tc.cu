// Base product of the layer: y[T, D] (fp32) = x[T, K] * W[D, K]^T, bf16 operands.
//
// "Multi-LoRA Serving Explained" (sevydevy.com), batched-serving section: every token of
// the mixed-tenant batch is multiplied by the one shared base weight in a single large
// matrix product; only the thin side path differs per token. "LoRA Serving" (vLLM
// learning book, ch. 09-04), section 3: the batch still runs x * W once as one GEMM.
//
// sm_103a design: a persistent, warp-specialised kernel on the 5th-generation tensor cores.
//   warp 0      TMA producer: 128 x 64 tiles of x and BN x 64 tiles of W into a ring of
//               STAGES shared-memory stages (128-byte swizzle), one mbarrier per stage;
//   warp 1      allocates 2*BN TMEM columns and issues tcgen05.mma (M=128, N=BN, K=16)
//               from one thread, committing each stage back to the producer;
//   warps 2..5  epilogue: tcgen05.ld of the fp32 accumulator (one row per thread) and
//               stores to y. Two accumulators in TMEM let the epilogue of one tile overlap
//               the main loop of the next.
// Tiles are visited M-fastest so that the CTAs working on one W column block run together
// and W is read from HBM once. Every wait is bounded (2 s): on a timeout the kernel sets
// an error bit and leaves instead of hanging.
#include <cooperative_groups.h>
#include <cuda.h>

#include <algorithm>
#include <cstdio>

#include "expand_vfull.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace mlora {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;                    // 64 bf16 = one 128-byte swizzle row
constexpr int kGemmThreads = 192;

template <int BN, int STAGES>
struct GemmSmem {
  static constexpr int kABytes = BM * BK * 2;
  static constexpr int kBBytes = BN * BK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kBarrierOffset = STAGES * kStageBytes;
  static constexpr int kBytes = kBarrierOffset + 256 + 1024;   // + barriers, + alignment slack
};

// Extra K blocks of the fused side path: one per unit of the M-tile (a 64-column block of the slot
// space used by its tokens) with A operand = the unit's scaled v tile (tensor-core shrink output)
// and B operand = the block's 64 columns of B for the N tile, both fetched by TMA into the same
// stage layout.
__device__ __forceinline__ int extra_kblocks(const int32_t* tile_unit_off, int m_blk) {
  return tile_unit_off ? tile_unit_off[m_blk + 1] - tile_unit_off[m_blk] : 0;
}

// M-tile of the tile with sequence number `tile`: M fastest, rotated by the column index (each
// column's rows stay a permutation), so that M-tiles with many extra K blocks are spread over the
// persistent CTAs.
__device__ __forceinline__ int tc_row(int tile, int num_m) {
  return (tile % num_m + tile / num_m) % num_m;
}

template <int BN, int STAGES>
__global__ void __launch_bounds__(kGemmThreads, 1)
gemm_bf16_tc_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_w,
                    const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_b,
                    const int32_t* __restrict__ tile_unit_off, const int32_t* __restrict__ unit_blk,
                    float* __restrict__ y, int T, int D, int K, uint32_t* __restrict__ err) {
  using L = GemmSmem<BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBarrierOffset);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_m = (T + BM - 1) / BM;
  const int num_n = (D + BN - 1) / BN;
  const int num_tiles = num_m * num_n;
  const int num_kb = (K + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&acc_full[a], 1);
      ptx::mbar_init(&acc_empty[a], 4);       // one arrival per epilogue warp
    }
    ptx::fence_barrier_init();
    ptx::fence_proxy_async_smem();
    ptx::tma_prefetch_desc(&tmap_x);
    ptx::tma_prefetch_desc(&tmap_w);
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, 2 * BN);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        const int m_blk = tc_row(tile, num_m);
        const int m0 = m_blk * BM;
        const int n0 = (tile / num_m) * BN;
        const int n_extra = extra_kblocks(tile_unit_off, m_blk);
        const int u0 = n_extra ? tile_unit_off[m_blk] : 0;
        for (int kb = 0; kb < num_kb + n_extra; ++kb) {
          if (!ptx::mbar_wait(&empty[stage], phase ^ 1u, err)) { ok = false; break; }
          uint8_t* sa = smem + stage * L::kStageBytes;
          uint8_t* sb = sa + L::kABytes;
          ptx::mbar_arrive_expect_tx(&full[stage], L::kStageBytes);
          if (kb < num_kb) {
            ptx::tma_load_2d(sa, &tmap_x, &full[stage], kb * BK, m0);
            ptx::tma_load_2d(sb, &tmap_w, &full[stage], kb * BK, n0);
          } else {
            const int u = u0 + kb - num_kb;
            ptx::tma_load_2d(sa, &tmap_v, &full[stage], 0, u * BM);
            ptx::tma_load_2d(sb, &tmap_b, &full[stage], unit_blk[u] * kBlockCols, n0);
          }
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(BM, BN);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int local = 0;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x, ++local) {
        const int acc = local & 1;
        const uint32_t acc_phase = static_cast<uint32_t>(local >> 1) & 1u;
        if (!ptx::mbar_wait(&acc_empty[acc], acc_phase ^ 1u, err)) break;
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        const int n_kb = num_kb + extra_kblocks(tile_unit_off, tc_row(tile, num_m));
        for (int kb = 0; kb < n_kb; ++kb) {
          if (!ptx::mbar_wait(&full[stage], phase, err)) { ok = false; break; }
          ptx::tc_fence_after();
          const uint32_t a_addr = ptx::smem_u32(smem + stage * L::kStageBytes);
          const uint32_t b_addr = a_addr + L::kABytes;
          const uint64_t a_desc = ptx::sw128_kmajor_desc(a_addr);
          const uint64_t b_desc = ptx::sw128_kmajor_desc(b_addr);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            // advancing K by 16 elements = 32 bytes = 2 in the descriptor's address field
            ptx::umma_bf16(d_tmem, a_desc + 2u * k, b_desc + 2u * k, idesc, (kb > 0 || k > 0) ? 1u : 0u);
          }
          ptx::umma_commit(&empty[stage]);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        ptx::umma_commit(&acc_full[acc]);
      }
    }
  } else {
    // epilogue: warp w reads TMEM lanes 32*(w%4) .. +31
    const int quarter = warp & 3;
    const int row_in_tile = quarter * 32 + lane;
    int local = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++local) {
      const int m0 = tc_row(tile, num_m) * BM;
      const int n0 = (tile / num_m) * BN;
      const int acc = local & 1;
      const uint32_t acc_phase = static_cast<uint32_t>(local >> 1) & 1u;
      if (!ptx::mbar_wait(&acc_full[acc], acc_phase, err)) break;
      ptx::tc_fence_after();
      const int row = m0 + row_in_tile;
      float* yrow = y + static_cast<size_t>(row) * D;
#pragma unroll 1
      for (int c = 0; c < BN; c += 32) {
        uint32_t r[32];
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                               static_cast<uint32_t>(acc * BN + c);
        ptx::tmem_ld_32x32b_x32(taddr, r);
        ptx::tmem_ld_wait();
        const int col = n0 + c;
        if (row < T) {
          if (col + 32 <= D && (D & 3) == 0) {
            float4* dst = reinterpret_cast<float4*>(yrow + col);
#pragma unroll
            for (int v = 0; v < 8; ++v)
              dst[v] = make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                   __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
          } else {
#pragma unroll
            for (int v = 0; v < 32; ++v)
              if (col + v < D) yrow[col + v] = __uint_as_float(r[v]);
          }
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&acc_empty[acc]);
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, 2 * BN);
  }
}

// ---------------------------------------------------------------------------------------------
// Skinny variant for small batches (T <= 256, the decode case): the roles swap so that W is the
// A operand (128 output features per CTA) and all tokens form N (NT = T rounded up to 16), which
// reads every W element exactly once. K is split across the CTAs of a thread-block cluster; each
// CTA stages its fp32 partial tile P[t][o] in its own shared memory, and after a cluster barrier
// each CTA sums, for its share of the tokens, the partials of the CTAs that hold the same output
// block through distributed shared memory, always in K-split order (so the result is
// deterministic), and writes the output with coalesced 16-byte stores. The kernel runs on CTA
// pairs (gemm_bf16_skinny_pair_kernel below).
//
// The shrink of the LoRA side path rides along ("Multi-LoRA Serving Explained", batched
// serving: one large product shared by the batch plus each token's low-rank side path). The
// step's active slots (those named by at least one token, ascending) contribute extra
// 128-row blocks of A-operand rows: block b holds active slots b*(128/R) .. +128/R - 1, each
// slot's R rows of A_pool fetched by its own TMA box, so each active adapter is read once and x
// is shared with the base product. Their accumulators are v[t][a][q] = sum_i A_a[q][i] x[t][i]
// for every token t and active slot a (written to vfull); the expand kernel then picks each
// token's own slots.
struct SkinnyShrink {
  PoolView pool;             // expand operands: B rows of the slots prefetched into L2 meanwhile
  MetaView meta;
  int n_dchunk;              // column ranges of the expand that follows (0: no prefetch)
  const int32_t* act_slot;   // active slots, ascending
  const int32_t* n_act;      // device count of active slots
  float* vfull;              // [T][vfull_ld] fp32, active slot a at columns a*R .. a*R + R - 1
  int vfull_ld;
  int R;                     // rows per slot in the A pool (multiple of 8, divides 128)
  int n_ablk;                // A-row blocks in the grid (enough for every possible active slot)
};

// Tensor maps over the A pool with boxes of R, 2R, 4R, ... rows (up to 128): a run of 2^k active
// slots with consecutive ids is one box, since their rows are contiguous in the pool.
constexpr int kABoxMaps = 5;
struct SkinnyAMaps {
  CUtensorMap box[kABoxMaps];
};

constexpr int kPullLoads = 12;            // distributed-shared-memory loads in flight per thread
constexpr int kSkinnyABytes = BM * BK * 2;

// Split-K reduction of the skinny kernel: every CTA of the cluster holds its fp32 partial tile
// part[t][o] (t < NT, o < 128) in shared memory; this CTA sums, for tokens [t0, t1) and the first
// `rows` o, the partials of ranks 0 .. SPLIT-1 in that order (deterministic) and stores
// out[t * ld + o] for o < cols (out = the output rows of this block). Work item = 4 consecutive o
// of one token; each thread keeps the loads of several items in flight before summing.
template <int SPLIT>
__device__ __forceinline__ void skinny_pull(cooperative_groups::cluster_group& cluster, float* part, int t0, int t1,
                                            int rows, float* out, long ld, int cols, int rank0 = 0, int rstride = 1) {
  constexpr int kItems = kPullLoads / SPLIT > 1 ? kPullLoads / SPLIT : 1;
  const int n_items = (t1 - t0) * (BM / 4);
  const bool vec = (cols & 3) == 0 && (ld & 3) == 0 && (reinterpret_cast<uintptr_t>(out) & 15u) == 0;
  for (int w0 = threadIdx.x; w0 < n_items; w0 += kItems * kGemmThreads) {
    float4 pv[kItems][SPLIT];
#pragma unroll
    for (int h = 0; h < kItems; ++h) {
      const int w = w0 + h * kGemmThreads;
      const int t = t0 + w / (BM / 4), o4 = (w % (BM / 4)) * 4;
      if (w < n_items && o4 < rows) {
#pragma unroll
        for (int r = 0; r < SPLIT; ++r)
          pv[h][r] = *reinterpret_cast<const float4*>(cluster.map_shared_rank(part + t * BM + o4, rank0 + rstride * r));
      }
    }
#pragma unroll
    for (int h = 0; h < kItems; ++h) {
      const int w = w0 + h * kGemmThreads;
      const int t = t0 + w / (BM / 4), o4 = (w % (BM / 4)) * 4;
      if (w >= n_items || o4 >= rows) continue;
      float4 acc = pv[h][0];
#pragma unroll
      for (int r = 1; r < SPLIT; ++r) {
        acc.x += pv[h][r].x;
        acc.y += pv[h][r].y;
        acc.z += pv[h][r].z;
        acc.w += pv[h][r].w;
      }
      float* dst = out + static_cast<size_t>(t) * ld + o4;
      if (vec && o4 + 4 <= cols) {
        *reinterpret_cast<float4*>(dst) = acc;
      } else {
        if (o4 < cols) dst[0] = acc.x;
        if (o4 + 1 < cols) dst[1] = acc.y;
        if (o4 + 2 < cols) dst[2] = acc.z;
        if (o4 + 3 < cols) dst[3] = acc.w;
      }
    }
  }
}

// CTA-pair form of the skinny kernel. Two CTAs of a cluster form a pair (cta_group::2) for two
// consecutive 128-row output blocks: rank 2 k + h holds block 2 p + h's A rows and tokens
// h NT/2 .. h NT/2 + NT/2 - 1 of x for K share k, and the even CTA issues M = 256 x N = NT MMAs
// that read both CTAs' operands, accumulating each block in its own CTA's TMEM. Per 64-wide K
// block an SM then stages 16 KB of A rows and 16 KB of x instead of 16 + 32 KB, so six stages fit
// where four did, and x is read from L2 half as often. The K shares of a block (ranks h, h + 2,
// ...) reduce their partials with skinny_pull (above). A pair whose even block has no rows (an A
// block past the active slots, or a block past the grid) skips the main loop; an odd block
// without rows still stages its half of x and lets the pair compute rows that are then dropped.
constexpr int kSkinnyPairStages = 6;
constexpr int kSkinnyPairMaxSplit = 4;      // clusters of at most 8 CTAs

__host__ __device__ constexpr int skinny_pair_stage_bytes(int NT) { return kSkinnyABytes + (NT / 2) * BK * 2; }
__host__ __device__ constexpr int skinny_pair_smem_bytes(int NT) {
  return kSkinnyPairStages * skinny_pair_stage_bytes(NT) + 256 + 1024;
}

// Rows of A-operand data block `oblk` holds in the skinny kernel (0: none), and for an A block
// the number of active slots it covers.
__device__ __forceinline__ int skinny_block_rows(int oblk, int n_oblk, int n_wblk, const SkinnyShrink& sh, int n_act,
                                                 int* n_box) {
  *n_box = 0;
  if (oblk >= n_oblk) return 0;                         // a block past the grid (odd count)
  if (oblk < n_wblk) return BM;
  const int spb = BM / sh.R;
  const int a0 = (oblk - n_wblk) * spb;
  *n_box = max(0, min(spb, n_act - a0));
  return *n_box * sh.R;
}

__global__ void __launch_bounds__(kGemmThreads, 1)
gemm_bf16_skinny_pair_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_xh,
                             const __grid_constant__ SkinnyAMaps amaps, float* __restrict__ y, int T, int D, int K,
                             int NT, int splitk, int n_oblk, uint32_t tmem_cols, uint32_t* __restrict__ err,
                             SkinnyShrink sh) {
  namespace cg = cooperative_groups;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int stage_bytes = skinny_pair_stage_bytes(NT);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kSkinnyPairStages * stage_bytes);   // used in the even CTA
  uint64_t* empty = full + kSkinnyPairStages;                                              // in each CTA
  uint64_t* acc_full = empty + kSkinnyPairStages;                                          // in each CTA
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
  float* part = reinterpret_cast<float*>(smem);          // [NT][128] after the main loop

  cg::cluster_group cluster = cg::this_cluster();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = static_cast<int>(cluster.block_rank());
  const int half = rank & 1, ks = rank >> 1;
  const int n_wblk = (D + BM - 1) / BM;
  const int pair_o = blockIdx.x / (2 * splitk);
  const int oblk = 2 * pair_o + half;
  const bool a_blk = oblk < n_oblk && oblk >= n_wblk;   // a block of active-slot A rows
  const int spb = a_blk ? BM / sh.R : 0;
  const int a0 = a_blk ? (oblk - n_wblk) * spb : 0;
  const int o0 = oblk * BM;
  const int num_kb = (K + BK - 1) / BK;
  const int kb0 = ks * num_kb / splitk, kb1 = (ks + 1) * num_kb / splitk;
  const uint16_t pair_mask = static_cast<uint16_t>(3u << (rank & ~1));

  if (threadIdx.x == 0) {
    for (int s = 0; s < kSkinnyPairStages; ++s) {
      ptx::mbar_init(&full[s], 1);                      // the even CTA posts both halves' bytes
      ptx::mbar_init(&empty[s], 1);                     // one multicast commit per use
    }
    ptx::mbar_init(acc_full, 1);
    ptx::fence_barrier_init();
    ptx::fence_proxy_async_smem();
    ptx::tma_prefetch_desc(a_blk ? &amaps.box[0] : &tmap_w);
    ptx::tma_prefetch_desc(&tmap_xh);
  }
  if (warp == 2 && oblk < n_wblk)
    for (int kb = kb0 + lane; kb < kb1; kb += 32) ptx::tma_prefetch_l2_2d(&tmap_w, kb * BK, o0);
  if (warp == 1) {
    ptx::tmem_alloc_pair(tmem_slot, tmem_cols);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  ptx::cluster_sync_all();                              // barriers of the cluster initialised, TMEM allocated
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  ptx::grid_dependency_wait();                          // earlier kernels' writes are visible
  ptx::grid_dependents_launch();                        // the next kernel may start its set-up
  const int n_act = sh.n_ablk > 0 ? *sh.n_act : 0;
  int my_box = 0, peer_box = 0;
  const int my_rows = skinny_block_rows(oblk, n_oblk, n_wblk, sh, n_act, &my_box);
  const int peer_rows = skinny_block_rows(oblk ^ 1, n_oblk, n_wblk, sh, n_act, &peer_box);
  const int even_rows = half ? peer_rows : my_rows;
  const bool idle = even_rows == 0;                     // uniform across the cluster (the pair's even block)
  if (!idle && a_blk && my_box > 0 && warp == 2) {      // this block's adapter rows into L2
    for (int e = lane; e < my_box * (kb1 - kb0); e += 32) {
      const int i = e % my_box, kb = kb0 + e / my_box;
      ptx::tma_prefetch_l2_2d(&amaps.box[0], kb * BK, sh.act_slot[a0 + i] * sh.R);
    }
  }
  const int n_exp_items = sh.n_dchunk ? (sh.meta.J == 1 ? sh.meta.counts[2] : sh.meta.T) * sh.n_dchunk : 0;

  if (idle) {
    // nothing to multiply
  } else if (warp == 0) {
    if (lane == 0) {
      // this CTA's A rows: the active slots' R rows, one TMA box per run of 2^k slots with
      // consecutive ids (largest power of two first), or one W box of 128 rows; and its half of x
      int chunk_row[BM / 8], chunk_pos[BM / 8], chunk_k[BM / 8];
      int n_chunk = 0;
      if (a_blk) {
        for (int i = 0; i < my_box;) {
          const int s0 = sh.act_slot[a0 + i];
          int run = 1;
          while (i + run < my_box && sh.act_slot[a0 + i + run] == s0 + run) ++run;
          const int k = 31 - __clz(run);                // 2^k <= run
          chunk_row[n_chunk] = s0 * sh.R;
          chunk_pos[n_chunk] = i;
          chunk_k[n_chunk] = k;
          ++n_chunk;
          i += 1 << k;
        }
      }
      auto a_bytes = [&](int oblk_, int rows_, int box_) {
        return oblk_ >= n_oblk ? 0 : (oblk_ < n_wblk ? kSkinnyABytes : box_ * sh.R * BK * 2);
      };
      const uint32_t bytes = static_cast<uint32_t>(a_bytes(oblk, my_rows, my_box) + a_bytes(oblk ^ 1, peer_rows, peer_box) +
                                                   2 * (NT / 2) * BK * 2);
      const uint32_t bar0 = ptx::mapa_shared(ptx::smem_u32(&full[0]), static_cast<uint32_t>(rank & ~1));
      int stage = 0;
      uint32_t phase = 0;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!ptx::mbar_wait_short(&empty[stage], phase ^ 1u, err)) break;
        uint8_t* sa = smem + stage * stage_bytes;
        const uint32_t bar = bar0 + static_cast<uint32_t>(stage * sizeof(uint64_t));
        if (half == 0) ptx::mbar_arrive_expect_tx(&full[stage], bytes);
        if (a_blk) {
          for (int c = 0; c < n_chunk; ++c)
            ptx::tma_load_2d_pair(sa + chunk_pos[c] * sh.R * BK * 2, &amaps.box[chunk_k[c]], bar, kb * BK,
                                  chunk_row[c]);
        } else if (oblk < n_oblk) {
          ptx::tma_load_2d_pair(sa, &tmap_w, bar, kb * BK, o0);
        }
        ptx::tma_load_2d_pair(sa + kSkinnyABytes, &tmap_xh, bar, kb * BK, half * (NT / 2));
        if (++stage == kSkinnyPairStages) { stage = 0; phase ^= 1u; }
      }
      // tail: every commit addressed to this CTA's stage barriers has landed before it may exit
      for (int i = 0; i < kSkinnyPairStages; ++i) {
        if (!ptx::mbar_wait_short(&empty[stage], phase ^ 1u, err)) break;
        if (++stage == kSkinnyPairStages) { stage = 0; phase ^= 1u; }
      }
    }
  } else if (warp == 1) {
    if (half == 0 && lane == 0) {
      const uint32_t idesc = ptx::idesc_bf16_f32(2 * BM, NT);
      int stage = 0;
      uint32_t phase = 0;
      bool mma_ok = true;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!ptx::mbar_wait_short(&full[stage], phase, err)) { mma_ok = false; break; }
        ptx::tc_fence_after();
        const uint32_t a_addr = ptx::smem_u32(smem + stage * stage_bytes);
        const uint64_t a_desc = ptx::sw128_kmajor_desc(a_addr);
        const uint64_t b_desc = ptx::sw128_kmajor_desc(a_addr + kSkinnyABytes);
#pragma unroll
        for (int k = 0; k < BK / 16; ++k)
          ptx::umma_bf16_pair(tmem_base, a_desc + 2u * k, b_desc + 2u * k, idesc, (kb > kb0 || k > 0) ? 1u : 0u);
        ptx::umma_commit_pair(&empty[stage], pair_mask);
        if (++stage == kSkinnyPairStages) { stage = 0; phase ^= 1u; }
      }
      if (mma_ok) ptx::umma_commit_pair(acc_full, pair_mask);
    }
  } else {
    // While the main loop runs, bring into L2 the B rows the expand kernel will read (a share
    // of its items per block).
    for (int item = blockIdx.x; item < n_exp_items; item += gridDim.x)
      expand_vfull_prefetch(sh.pool, sh.meta, item, sh.n_dchunk, threadIdx.x - 64, kGemmThreads - 64);
    // TMEM lane = output row o of this CTA's block (warp w reads lanes 32*(w%4)..), columns = tokens
    const int quarter = warp & 3;
    const int o = quarter * 32 + lane;
    if (ptx::mbar_wait_short(acc_full, 0, err)) {
      ptx::tc_fence_after();
      const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
#pragma unroll 1
      for (int c = 0; c < NT; c += 64) {                // two loads in flight per wait
        uint32_t r0[32], r1[32];
        ptx::tmem_ld_32x32b_x32(lane_base + static_cast<uint32_t>(c), r0);
        if (c + 32 < NT) ptx::tmem_ld_32x32b_x32(lane_base + static_cast<uint32_t>(c + 32), r1);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) part[(c + i) * BM + o] = __uint_as_float(r0[i]);
        if (c + 32 < NT) {
#pragma unroll
          for (int i = 0; i < 32; ++i) part[(c + 32 + i) * BM + o] = __uint_as_float(r1[i]);
        }
      }
    }
  }
  ptx::tc_fence_before();
  ptx::cluster_sync_all();                              // every partial tile is in shared memory
  if (!idle && my_rows > 0) {
    // CTA (k, h) owns tokens [t0, t1) of block h: partials of ranks h, h + 2, ... summed in order
    const int per = (T + splitk - 1) / splitk;
    const int t0 = ks * per, t1 = min(T, t0 + per);
    const int rows = my_rows;
    float* out = a_blk ? sh.vfull + a0 * sh.R : y + o0;
    const long ld = a_blk ? sh.vfull_ld : D;
    const int cols = a_blk ? rows : min(BM, D - o0);
    switch (splitk) {
      case 1: skinny_pull<1>(cluster, part, t0, t1, rows, out, ld, cols, half, 2); break;
      case 2: skinny_pull<2>(cluster, part, t0, t1, rows, out, ld, cols, half, 2); break;
      case 3: skinny_pull<3>(cluster, part, t0, t1, rows, out, ld, cols, half, 2); break;
      default: skinny_pull<4>(cluster, part, t0, t1, rows, out, ld, cols, half, 2); break;
    }
  }
  ptx::tc_fence_before();
  ptx::cluster_sync_all();                              // no CTA leaves while others read its tile or TMEM
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, tmem_cols);
  }
}

// Token-split form of the skinny kernel (mlora_set_skinny_form(2)): K is not split, so there are
// no partial tiles to reduce. CTA (c, g) of a cluster of kTsC x G CTAs computes output block
// kTsC * cluster + c for token group g over the whole of K (M = 128 rows, N = the group's tokens)
// in its own TMEM and stores y (or v) from there. What CTAs share is fetched once per cluster by
// TMA multicast, with as few and as large copies as possible (each TMA instruction has a fixed
// cost): the block's 128 A-operand rows of K block kb (one W box, or the active slots' boxes) are
// issued by CTA kb mod G of row c for the whole row, and group g's x rows by CTA kb mod kTsC of
// column g for the whole column. A stage may be refilled only when every CTA that the refill
// writes into has finished reading it, so each CTA's MMA commit arrives on the stage's empty
// barrier in all CTAs of its row and its column (the CTAs whose loads write into it are exactly
// those). A row without rows (an A block past the active slots, or a block past the grid) still
// fetches its share of x and releases every stage.
// Measured on the decode shape (256 tokens, 4096 -> 4096 plus 90 active rank-16 slots): 38 us
// against 26 us for the split-K form. Multicast saves L2 reads but not SM ingress: an SM here
// receives 28 KB per K block for 128 x 96 x 64 products, a CTA of the split-K pair 32 KB for
// 128 x 256 x 64, and L2-to-SM bandwidth (about 100-115 GB/s per SM, measured in both) bounds both.
constexpr int kTsC = 2;                    // output blocks per cluster (they share x)
constexpr int kTsMaxG = 4;                 // token groups per cluster (they share the A rows)
constexpr int kTsMaxStages = 8;
constexpr int kTsSmemMax = 232448;         // opt-in shared memory per CTA (227 KB)
// The shared-memory ring holds few K blocks of A rows per row of the cluster (a third or less of
// a CTA's stage is its share of them), too few to keep enough HBM reads in flight; the producer
// therefore also asks L2 for its A-row boxes this many K blocks ahead of the block it loads.
constexpr int kTsPrefetchAhead = 24;

// Tokens per group: groups of ts_group_max(NT, G) tokens (a multiple of 16), the last one shorter.
__host__ __device__ constexpr int ts_group_max(int NT, int G) { return 16 * ((NT / 16 + G - 1) / G); }
__host__ __device__ constexpr int ts_stage_bytes(int n_gmax) { return kSkinnyABytes + n_gmax * BK * 2; }
__host__ __device__ constexpr int ts_stages(int n_gmax) {
  return (kTsSmemMax - 1280) / ts_stage_bytes(n_gmax) < kTsMaxStages ? (kTsSmemMax - 1280) / ts_stage_bytes(n_gmax)
                                                                     : kTsMaxStages;
}
__host__ __device__ constexpr int ts_smem_bytes(int n_gmax) {
  return ts_stages(n_gmax) * ts_stage_bytes(n_gmax) + 256 + 1024;
}

// A TMA load to the CTAs of cta_mask (a plain load when the mask is this CTA alone).
__device__ __forceinline__ void ts_load(void* dst, const void* tmap, uint64_t* bar, int32_t c0, int32_t c1,
                                        uint16_t cta_mask, uint16_t self_bit) {
  if (cta_mask == self_bit) ptx::tma_load_2d(dst, tmap, bar, c0, c1);
  else ptx::tma_load_2d_mc(dst, tmap, bar, c0, c1, cta_mask);
}

__global__ void __launch_bounds__(kGemmThreads, 1)
gemm_bf16_skinny_ts_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_x,
                           const __grid_constant__ SkinnyAMaps amaps, float* __restrict__ y, int T, int D, int K,
                           int NT, int G, int n_oblk, int stages, uint32_t tmem_cols, uint32_t* __restrict__ err,
                           SkinnyShrink sh) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int stage_bytes = ts_stage_bytes(ts_group_max(NT, G));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + stages * stage_bytes);
  uint64_t* empty = full + kTsMaxStages;
  uint64_t* acc_full = empty + kTsMaxStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = static_cast<int>(ptx::cluster_ctarank());
  const int g = rank % G, c = rank / G;
  const int cl = blockIdx.x / (kTsC * G);
  const int oblk = cl * kTsC + c;
  const int n_wblk = (D + BM - 1) / BM;
  const bool a_blk = oblk < n_oblk && oblk >= n_wblk;
  const int spb = a_blk ? BM / sh.R : 0;
  const int a0 = a_blk ? (oblk - n_wblk) * spb : 0;
  const int o0 = oblk * BM;
  const int n_gmax = ts_group_max(NT, G);
  const int t_g = g * n_gmax;
  const int n_g = min(n_gmax, NT - t_g);
  const int num_kb = (K + BK - 1) / BK;
  const uint16_t self_bit = static_cast<uint16_t>(1u << rank);
  const uint16_t row_mask = static_cast<uint16_t>(((1u << G) - 1u) << (c * G));
  uint16_t col_mask = 0;
  for (int cc = 0; cc < kTsC; ++cc) col_mask |= static_cast<uint16_t>(1u << (cc * G + g));
  const uint16_t peer_mask = row_mask | col_mask;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      ptx::mbar_init(&full[s], 1);                      // this CTA's expect_tx; bytes from row and column
      ptx::mbar_init(&empty[s], G + kTsC - 1);          // one commit from each CTA of the row and the column
    }
    ptx::mbar_init(acc_full, 1);
    ptx::fence_barrier_init();
    ptx::fence_proxy_async_smem();
    ptx::tma_prefetch_desc(a_blk ? &amaps.box[0] : &tmap_w);
    ptx::tma_prefetch_desc(&tmap_x);
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, tmem_cols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  ptx::cluster_sync_all();                              // barriers of the cluster initialised, TMEM allocated
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0 && lane == 0 && oblk < n_wblk) {       // W rows do not depend on earlier kernels
    for (int kb = g; kb < min(num_kb, stages); kb += G) ptx::tma_prefetch_l2_2d(&tmap_w, kb * BK, o0);
  }
  ptx::grid_dependency_wait();                          // earlier kernels' writes are visible
  ptx::grid_dependents_launch();                        // the next kernel may start its set-up
  const int n_act = sh.n_ablk > 0 ? *sh.n_act : 0;
  int my_box = 0;
  const int my_rows = skinny_block_rows(oblk, n_oblk, n_wblk, sh, n_act, &my_box);
  bool any_rows = false;                                // uniform across the cluster
  for (int cc = 0; cc < kTsC; ++cc) {
    int nb = 0;
    any_rows |= skinny_block_rows(cl * kTsC + cc, n_oblk, n_wblk, sh, n_act, &nb) > 0;
  }
  const int n_exp_items = sh.n_dchunk ? (sh.meta.J == 1 ? sh.meta.counts[2] : sh.meta.T) * sh.n_dchunk : 0;

  if (!any_rows) {
    // nothing to multiply in this cluster
  } else if (warp == 0) {
    if (lane == 0) {
      // the block's A rows: one W box of 32 rows each, or one box per run of 2^k active slots with
      // consecutive ids (largest power of two first); this CTA issues every G-th of them
      int chunk_row[BM / 8], chunk_pos[BM / 8], chunk_k[BM / 8];
      int n_chunk = 0;
      if (a_blk) {
        for (int i = 0; i < my_box;) {
          const int s0 = sh.act_slot[a0 + i];
          int run = 1;
          while (i + run < my_box && sh.act_slot[a0 + i + run] == s0 + run) ++run;
          const int k = 31 - __clz(run);                // 2^k <= run
          chunk_row[n_chunk] = s0 * sh.R;
          chunk_pos[n_chunk] = i;
          chunk_k[n_chunk] = k;
          ++n_chunk;
          i += 1 << k;
        }
      }
      const int a_bytes = oblk >= n_oblk ? 0 : (a_blk ? my_box * sh.R * BK * 2 : kSkinnyABytes);
      // every CTA of a column receives a whole box of n_gmax x rows (past NT: zero fill)
      const uint32_t bytes = static_cast<uint32_t>(a_bytes + n_gmax * BK * 2);
      auto prefetch_rows = [&](int kbp) {               // the block's A rows of K block kbp into L2
        if (a_blk) {
          for (int i = 0; i < n_chunk; ++i) ptx::tma_prefetch_l2_2d(&amaps.box[chunk_k[i]], kbp * BK, chunk_row[i]);
        } else if (oblk < n_oblk) {
          ptx::tma_prefetch_l2_2d(&tmap_w, kbp * BK, o0);
        }
      };
      int pf_next = stages + g;                         // next K block this CTA asks L2 for (step G)
      int stage = 0;
      uint32_t phase = 0;
      for (int kb = 0; kb < num_kb; ++kb) {
        if (!ptx::mbar_wait_short(&empty[stage], phase ^ 1u, err)) break;
        uint8_t* sa = smem + stage * stage_bytes;
        ptx::mbar_arrive_expect_tx(&full[stage], bytes);
        if (kb % G == g) {
          if (a_blk) {
            for (int i = 0; i < n_chunk; ++i)
              ts_load(sa + chunk_pos[i] * sh.R * BK * 2, &amaps.box[chunk_k[i]], &full[stage], kb * BK, chunk_row[i],
                      row_mask, self_bit);
          } else if (oblk < n_oblk) {
            ts_load(sa, &tmap_w, &full[stage], kb * BK, o0, row_mask, self_bit);
          }
        }
        if (kb % kTsC == c) ts_load(sa + kSkinnyABytes, &tmap_x, &full[stage], kb * BK, t_g, col_mask, self_bit);
        // at most one L2 request per K block, so that the copies the MMAs wait for go first
        if (pf_next < num_kb && pf_next < kb + kTsPrefetchAhead) {
          prefetch_rows(pf_next);
          pf_next += G;
        }
        if (++stage == stages) { stage = 0; phase ^= 1u; }
      }
      // tail: every commit addressed to this CTA's stage barriers has landed before it may exit
      for (int i = 0; i < stages; ++i) {
        if (!ptx::mbar_wait_short(&empty[stage], phase ^ 1u, err)) break;
        if (++stage == stages) { stage = 0; phase ^= 1u; }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const bool compute = my_rows > 0;
      const uint32_t idesc = ptx::idesc_bf16_f32(BM, n_g);
      int stage = 0;
      uint32_t phase = 0;
      bool mma_ok = true;
      for (int kb = 0; kb < num_kb; ++kb) {
        if (!ptx::mbar_wait_short(&full[stage], phase, err)) { mma_ok = false; break; }
        ptx::tc_fence_after();
        if (compute) {
          const uint32_t a_addr = ptx::smem_u32(smem + stage * stage_bytes);
          const uint64_t a_desc = ptx::sw128_kmajor_desc(a_addr);
          const uint64_t b_desc = ptx::sw128_kmajor_desc(a_addr + kSkinnyABytes);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            ptx::umma_bf16(tmem_base, a_desc + 2u * k, b_desc + 2u * k, idesc, (kb > 0 || k > 0) ? 1u : 0u);
        }
        ptx::umma_commit_mc(&empty[stage], peer_mask);
        if (++stage == stages) { stage = 0; phase ^= 1u; }
      }
      if (mma_ok) ptx::umma_commit(acc_full);
    }
  } else {
    // While the main loop runs, bring into L2 the B rows the expand kernel will read (a share
    // of its items per block).
    for (int item = blockIdx.x; item < n_exp_items; item += gridDim.x)
      expand_vfull_prefetch(sh.pool, sh.meta, item, sh.n_dchunk, threadIdx.x - 64, kGemmThreads - 64);
    // TMEM lane = output row o of the block (warp w reads lanes 32*(w%4)..), columns = the group's
    // tokens; each store instruction writes 32 consecutive outputs of one token
    if (my_rows > 0 && ptx::mbar_wait_short(acc_full, 0, err)) {
      ptx::tc_fence_after();
      const int quarter = warp & 3;
      const int o = quarter * 32 + lane;
      float* out = a_blk ? sh.vfull + a0 * sh.R : y + o0;
      const long ld = a_blk ? sh.vfull_ld : D;
      const int cols = a_blk ? my_rows : min(BM, D - o0);
      const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
      const int t_end = min(n_g, T - t_g);              // the group's real tokens
#pragma unroll 1
      for (int c0 = 0; c0 < n_g; c0 += 64) {           // two loads in flight per wait
        uint32_t r0[32], r1[32];
        ptx::tmem_ld_32x32b_x32(lane_base + static_cast<uint32_t>(c0), r0);
        if (c0 + 32 < n_g) ptx::tmem_ld_32x32b_x32(lane_base + static_cast<uint32_t>(c0 + 32), r1);
        ptx::tmem_ld_wait();
        if (o < cols) {
          float* dst = out + static_cast<size_t>(t_g) * ld + o;
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (c0 + i < t_end) dst[static_cast<size_t>(c0 + i) * ld] = __uint_as_float(r0[i]);
          if (c0 + 32 < n_g) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (c0 + 32 + i < t_end) dst[static_cast<size_t>(c0 + 32 + i) * ld] = __uint_as_float(r1[i]);
          }
        }
      }
    }
  }
  ptx::tc_fence_before();
  ptx::cluster_sync_all();                              // no CTA leaves while a peer may still address it
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, tmem_cols);
  }
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link-time libcuda).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// Row-major bf16 matrix [rows, cols] seen as a 2-D tensor, box = box_cols x box_rows, 128B swizzle.
bool make_tmap_bf16_impl(CUtensorMap* map, const void* base, long rows, int cols, int box_rows, int box_cols) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estride[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estride,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int BN, int STAGES>
cudaError_t launch_tc(const uint16_t* x, const uint16_t* W, float* y, int T, int K, int D, uint32_t* err,
                      int num_sms, const PoolView* pool, const MetaView* meta, cudaStream_t s) {
  using L = GemmSmem<BN, STAGES>;
  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(gemm_bf16_tc_kernel<BN, STAGES>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  CUtensorMap mx, mw, mv, mb;
  if (!make_tmap_bf16_impl(&mx, x, T, K, BM, BK) || !make_tmap_bf16_impl(&mw, W, D, K, BN, BK))
    return cudaErrorInvalidValue;
  const int32_t *tile_unit_off = nullptr, *unit_blk = nullptr;
  if (pool && meta) {                     // the fused side path: v tiles and the pool's B columns
    const long v_rows = static_cast<long>(meta->unit_cap) * BM;
    if (!make_tmap_bf16_impl(&mv, meta->vtile, v_rows, BK, BM, BK) ||
        !make_tmap_bf16_impl(&mb, pool->B, D, pool->C, BN, BK))
      return cudaErrorInvalidValue;
    tile_unit_off = meta->tile_unit_off;
    unit_blk = meta->unit_blk;
  } else {
    mv = mx;
    mb = mw;
  }
  const int tiles = ((T + BM - 1) / BM) * ((D + BN - 1) / BN);
  const int grid = tiles < num_sms ? tiles : num_sms;
  note_launch_begin(kKindGemm, s);
  gemm_bf16_tc_kernel<BN, STAGES><<<grid, kGemmThreads, L::kBytes, s>>>(mx, mw, mv, mb, tile_unit_off, unit_blk, y, T,
                                                                         D, K, err);
  cudaError_t e = cudaGetLastError();
  note_launch_end(kKindGemm, s);
  return e;
}


// Clusters of 2 x splitk CTAs of the CTA-pair small-batch kernel (one per SM: its shared memory)
// that can be resident at once on this device, cached per device and split. A cluster is placed
// within one GPC, so the count is not the SM count over the cluster size: GB300 reports 76, 36,
// 23 and 15 for splits 1-4, and a launch one cluster past that (24 clusters of 6, 16 of 8) took
// 34-35 us where the next smaller split took 23-25 us.
int skinny_pair_resident_clusters(int splitk) {
  static int cached_device = -1;
  static int cached[kSkinnyPairMaxSplit + 1] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (cached_device != dev) {
    int num_sms = 0;
    cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
    for (int k = 1; k <= kSkinnyPairMaxSplit; ++k) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(num_sms / (2 * k) * (2 * k), 1, 1);
      cfg.blockDim = dim3(kGemmThreads, 1, 1);
      cfg.dynamicSmemBytes = skinny_pair_smem_bytes(256);
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2 * k;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int clusters = 0;
      if (cudaOccupancyMaxActiveClusters(&clusters, gemm_bf16_skinny_pair_kernel, &cfg) != cudaSuccess) {
        cudaGetLastError();
        clusters = num_sms / (2 * k);                   // the count by SMs alone
      }
      cached[k] = clusters;
    }
    cached_device = dev;
  }
  return cached[splitk];
}

// The CTA-pair form: pairs of output blocks, K split over clusters of 2 x splitk CTAs.
cudaError_t launch_skinny_pair(const uint16_t* x, const uint16_t* W, float* y, int T, int K, int D, uint32_t* err,
                               int num_sms, const uint16_t* A_pool, int S, const SkinnyShrink& sh, cudaStream_t s) {
  const int NT = (T + 15) / 16 * 16;
  const int n_oblk = (D + BM - 1) / BM + sh.n_ablk;
  const int n_pairs = (n_oblk + 1) / 2;
  const int num_kb = (K + BK - 1) / BK;
  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(gemm_bf16_skinny_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         skinny_pair_smem_bytes(256));
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  // the widest K split whose clusters are all resident at once (a second wave of clusters costs
  // more than the shorter main loop saves)
  int splitk = num_sms / (2 * n_pairs);
  if (splitk > kSkinnyPairMaxSplit) splitk = kSkinnyPairMaxSplit;
  if (splitk > num_kb) splitk = num_kb;
  if (splitk < 1) splitk = 1;
  while (splitk > 1 && n_pairs > skinny_pair_resident_clusters(splitk)) --splitk;
  uint32_t tmem_cols = 32;
  while (tmem_cols < static_cast<uint32_t>(NT)) tmem_cols <<= 1;
  CUtensorMap mw, mxh;
  SkinnyAMaps ma;
  if (!make_tmap_bf16_impl(&mw, W, D, K, BM, BK) || !make_tmap_bf16_impl(&mxh, x, T, K, NT / 2, BK))
    return cudaErrorInvalidValue;
  for (int k = 0; k < kABoxMaps; ++k) {
    if (sh.n_ablk > 0 && (sh.R << k) <= BM) {
      if (!make_tmap_bf16_impl(&ma.box[k], A_pool, static_cast<long>(S) * sh.R, K, sh.R << k, BK))
        return cudaErrorInvalidValue;
    } else {
      ma.box[k] = mw;                                   // never used
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_pairs * 2 * splitk, 1, 1);
  cfg.blockDim = dim3(kGemmThreads, 1, 1);
  cfg.dynamicSmemBytes = skinny_pair_smem_bytes(NT);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2 * splitk;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  note_launch_begin(kKindGemm, s);
  cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_bf16_skinny_pair_kernel, mw, mxh, ma, y, T, D, K, NT, splitk, n_oblk,
                                     tmem_cols, err, sh);
  note_launch_end(kKindGemm, s);
  return e;
}

// Token groups of the token-split form for this shape (0: its grid does not fit one wave): the
// most groups (at most kTsMaxG, each of 16 tokens or more) whose grid fits one wave.
int skinny_ts_groups(int NT, int n_oblk, int num_sms) {
  const int n_cl = (n_oblk + kTsC - 1) / kTsC;
  int G = 0;
  for (int g = 1; g <= kTsMaxG && g <= NT / 16; ++g) {
    const int real = (NT + ts_group_max(NT, g) - 1) / ts_group_max(NT, g);   // groups that hold tokens
    if (real == g && n_cl * kTsC * g <= num_sms) G = g;
  }
  return G;
}

cudaError_t launch_skinny_ts(const uint16_t* x, const uint16_t* W, float* y, int T, int K, int D, uint32_t* err,
                             int G, const uint16_t* A_pool, int S, const SkinnyShrink& sh, cudaStream_t s) {
  const int NT = (T + 15) / 16 * 16;
  const int n_oblk = (D + BM - 1) / BM + sh.n_ablk;
  const int n_cl = (n_oblk + kTsC - 1) / kTsC;
  const int n_gmax = ts_group_max(NT, G);
  const int stages = ts_stages(n_gmax);
  uint32_t tmem_cols = 32;
  while (tmem_cols < static_cast<uint32_t>(n_gmax)) tmem_cols <<= 1;
  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(gemm_bf16_skinny_ts_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kTsSmemMax);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  CUtensorMap mw, mx;
  SkinnyAMaps ma;
  if (!make_tmap_bf16_impl(&mw, W, D, K, BM, BK) || !make_tmap_bf16_impl(&mx, x, T, K, n_gmax, BK))
    return cudaErrorInvalidValue;
  for (int k = 0; k < kABoxMaps; ++k) {
    if (sh.n_ablk > 0 && (sh.R << k) <= BM) {
      if (!make_tmap_bf16_impl(&ma.box[k], A_pool, static_cast<long>(S) * sh.R, K, sh.R << k, BK))
        return cudaErrorInvalidValue;
    } else {
      ma.box[k] = mw;                                   // never used
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_cl * kTsC * G, 1, 1);
  cfg.blockDim = dim3(kGemmThreads, 1, 1);
  cfg.dynamicSmemBytes = ts_smem_bytes(n_gmax);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kTsC * G;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  note_launch_begin(kKindGemm, s);
  cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_bf16_skinny_ts_kernel, mw, mx, ma, y, T, D, K, NT, G, n_oblk, stages,
                                     tmem_cols, err, sh);
  note_launch_end(kKindGemm, s);
  return e;
}

cudaError_t launch_skinny(const uint16_t* x, const uint16_t* W, float* y, int T, int K, int D, uint32_t* err,
                          int num_sms, const uint16_t* A_pool, int S, const SkinnyShrink& sh, cudaStream_t s) {
  const int NT = (T + 15) / 16 * 16;
  // The split-K form unless the token-split one is asked for: the token-split form delivers each
  // A row to all G CTAs of a row, and per-SM L2-to-SM bandwidth (about 100-115 GB/s measured in
  // both forms) then bounds it well below the split-K form on the decode and compose shapes.
  const int G = skinny_form() == 2 ? skinny_ts_groups(NT, (D + BM - 1) / BM + sh.n_ablk, num_sms) : 0;
  if (G > 0) return launch_skinny_ts(x, W, y, T, K, D, err, G, A_pool, S, sh, s);
  return launch_skinny_pair(x, W, y, T, K, D, err, num_sms, A_pool, S, sh, s);
}

}  // namespace

bool make_tmap_bf16(CUtensorMap* map, const void* base, long rows, int cols, int box_rows, int box_cols) {
  return make_tmap_bf16_impl(map, base, rows, cols, box_rows, box_cols);
}

bool make_tmap_f32_sw128(CUtensorMap* map, const void* base, long rows, int cols, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || (cols & 3) != 0 || (reinterpret_cast<uintptr_t>(base) & 15u) != 0) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 4};
  cuuint32_t box[2] = {32, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estride[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, estride,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

cudaError_t launch_base_gemm_lora(const uint16_t* x, const uint16_t* W, float* y, int T, int K, int D,
                                  uint32_t* err, int num_sms, const PoolView* pool, const MetaView* meta,
                                  cudaStream_t s) {
  if (T == 0 || D == 0) return cudaSuccess;
  if (T <= kSkinnyMaxT && !pool && (D + BM - 1) / BM <= num_sms) {   // its column blocks fill one wave
    SkinnyShrink none{};
    return launch_skinny(x, W, y, T, K, D, err, num_sms, nullptr, 0, none, s);
  }
  // Two or more 128-row tiles: the CTA-pair kernel whenever it is available, its N tile chosen by
  // estimated time. Even a single partial wave of 256-row pair tiles beats the one-CTA kernel's
  // narrower tiles on every shape measured (T = 512-2048). One 128-row tile, or
  // mlora_set_gemm_tile_n(-1): the one-CTA kernel with the largest N tile that still gives every
  // SM a tile; small problems take N = 64.
  const int m_tiles = (T + BM - 1) / BM;
  const int forced_n = gemm_tile_n();
  if (forced_n > 0) return launch_pair_gemm(x, W, y, T, K, D, err, pool, meta, forced_n, s);
  if (forced_n == 0 && m_tiles > 1 && pair_gemm_max_pairs() > 0)
    return launch_pair_gemm(x, W, y, T, K, D, err, pool, meta, 0, s);
  if (m_tiles * ((D + 255) / 256) >= num_sms)
    return launch_tc<256, 4>(x, W, y, T, K, D, err, num_sms, pool, meta, s);
  if (m_tiles * ((D + 127) / 128) >= num_sms)
    return launch_tc<128, 6>(x, W, y, T, K, D, err, num_sms, pool, meta, s);
  return launch_tc<64, 8>(x, W, y, T, K, D, err, num_sms, pool, meta, s);
}

bool base_gemm_uses_pair(int T) {
  const int forced_n = gemm_tile_n();
  if (forced_n > 0) return true;
  return forced_n == 0 && (T + BM - 1) / BM > 1 && pair_gemm_max_pairs() > 0;
}

cudaError_t launch_base_gemm(const uint16_t* x, const uint16_t* W, float* y, int T, int K, int D,
                             uint32_t* err, int num_sms, cudaStream_t s) {
  return launch_base_gemm_lora(x, W, y, T, K, D, err, num_sms, nullptr, nullptr, s);
}

}  // namespace mlora

namespace mlora {

bool skinny_shrink_fusable(int T, int J, int S, int R, int vfull_ld) {
  if (T < 1 || T > kSkinnyMaxT || T > kVfullMaxTokens) return false;
  if (R < 8 || R > BM || BM % R != 0) return false;
  const int max_act = std::min(S, T * J);
  return max_act * R <= vfull_ld;
}

cudaError_t launch_gemm_shrink_fused(const uint16_t* x, const uint16_t* W, float* y, const PoolView& pool,
                                     const MetaView& m, uint32_t* err, int num_sms, cudaStream_t s) {
  if (m.T == 0 || pool.D == 0) return cudaSuccess;
  const int max_act = std::min(pool.S, m.n);
  const int n_dchunk = (pool.D + kExpandVfullCols - 1) / kExpandVfullCols;
  SkinnyShrink sh{pool, m, n_dchunk, m.act_slot, m.counts + 4, m.vfull, m.vfull_ld, pool.R,
                  (max_act * pool.R + BM - 1) / BM};
  return launch_skinny(x, W, y, m.T, pool.K, pool.D, err, num_sms, pool.A, pool.S, sh, s);
}

}  // namespace mlora
