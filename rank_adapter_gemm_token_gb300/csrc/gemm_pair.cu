// Base product of the layer for batches of more than 256 tokens, on CTA pairs:
// y[T, D] (fp32) = x[T, K] * W[D, K]^T, bf16 operands, plus the fused side path of the
// tensor-core prefill (extra K blocks, below).
//
// "Multi-LoRA Serving Explained" (sevydevy.com), batched-serving section: every token of the
// mixed-tenant batch goes through the one shared base weight in a single large product; only
// the thin side path differs per token. "LoRA Serving" (vLLM learning book, ch. 09-04),
// section 3: the batch still runs x * W once as one GEMM.
//
// sm_103a design: a persistent kernel on clusters of two CTAs (ranks 0 and 1, one per SM) that
// own a 256 x BN tile of y together. Per 64-wide K block, rank r stages x rows m0 + 128 r ..
// +127 and W rows n0 + (BN/2) r .. + BN/2 - 1 (128-byte swizzle) in its own shared memory; one
// thread of rank 0 issues tcgen05.mma.cta_group::2 (M = 256, N = BN, K = 16), which reads both
// CTAs' operands and accumulates rows m0 + 128 r .. in the TMEM of rank r. With BN = 256 each SM
// stages 32 KB per K block instead of the 48 KB of a 128 x 256 tile on one SM for the same
// tensor-core work, so a deeper ring fits. BN (256, 224, 192 or 128) is chosen per shape so that
// the tiles fill the resident pairs in whole waves: a last wave that is mostly empty leaves SMs
// idle while the others finish.
//   warp 0      TMA producer in each CTA; its loads signal rank 0's stage barrier (the rank-0
//               producer posts the byte count of both halves);
//   warp 1      TMEM allocation in both CTAs (two accumulators: the one of a tile is drained
//               while the next accumulates); rank 0's lane 0 issues the MMAs and commits each
//               stage back to both producers;
//   warps 2..5  epilogue in each CTA: tcgen05.ld of its 128 rows (one per thread), stores to y,
//               then an arrival on rank 0's accumulator-free barrier.
// Extra K blocks (the expand of the LoRA side path, inside the accumulator): the pair tile covers
// M-tiles 2 mp and 2 mp + 1, whose units (64-column blocks of the slot space used by their
// tokens) may differ; the pair runs one block per entry of the union the metadata lists, in
// ascending block order. Rank r's A operand is the scaled v tile of its own M-tile's unit on that
// block, or zeros (an out-of-range TMA box) when its tile does not use the block; the B operand is
// the block's 64 columns of B for the pair's output rows, split between the ranks like W.
// Tile order: M fastest (the pairs working on one W column block run together, so W comes from
// HBM once), with the rows of each column rotated by the column index, so that a row with many
// extra blocks (decode tokens with many slots) is spread over all pairs instead of falling to the
// same pairs in every wave.
// Every wait is bounded (2 s); on a timeout a thread sets the error bit and leaves its loop.
// Both CTAs always reach the final cluster barrier, so a timeout never turns into a hang.
#include <cuda.h>

#include <algorithm>
#include <climits>

#include "internal.h"
#include "ptx.cuh"

namespace mlora {
namespace {

constexpr int kHalf = 128;                 // rows of y per CTA of the pair tile (M = 256 per pair)
constexpr int kPairM = 2 * kHalf;
constexpr int kPK = 64;                    // 64 bf16 = one 128-byte swizzle row
constexpr int kPairThreads = 192;
constexpr int kPairABytes = kHalf * kPK * 2;
constexpr int kEpiBoxBytes = 32 * 32 * 4;    // y staging box: 32 rows x 32 fp32 columns

// BN = columns of y per pair tile (W rows: BN / 2 per CTA); STAGES = ring depth that fits.
template <int BN, int STAGES>
struct PairCfg {
  static_assert(BN % 32 == 0 && BN >= 64 && BN <= 256, "N tile");
  static constexpr int kBRows = BN / 2;
  static constexpr int kBBytes = kBRows * kPK * 2;
  static constexpr int kStageBytes = kPairABytes + kBBytes;            // multiple of 1024
  static constexpr int kEpiOffset = STAGES * kStageBytes;              // y staging: 4 warps x 2 x 4 KB
  static constexpr int kEpiBytes = 4 * 2 * kEpiBoxBytes;
  static constexpr int kBarrierOffset = kEpiOffset + kEpiBytes;
  static constexpr int kBytes = kBarrierOffset + 256 + 1024;           // + barriers, + alignment slack
  static constexpr int kAccStride = BN <= 128 ? 128 : 256;            // TMEM columns per accumulator
  static constexpr uint32_t kTmemCols = 2 * kAccStride;
  static_assert(kStageBytes % 1024 == 0, "stage alignment");
  static_assert(kBytes <= 232448, "shared memory");
};

// M row of the pair tile with sequence number `tile` in the static order (no metadata): M fastest,
// rotated by the column index, which keeps every column's rows a permutation while a persistent
// pair's tiles walk through the rows.
__device__ __forceinline__ int pair_row(int tile, int num_mp) {
  return (tile % num_mp + tile / num_mp) % num_mp;
}

// Extra K blocks of pair tile mp (0 without the fused side path).
__device__ __forceinline__ int pair_extra(const int32_t* ptile_off, int mp) {
  return ptile_off ? ptile_off[mp + 1] - ptile_off[mp] : 0;
}

constexpr int kSchedDepth = 4;          // tile ids in flight from the scheduler to the other roles
constexpr uint32_t kSchedUsers = 10;    // readers of a tile id: rank 0's MMA thread and 4 epilogue
                                        // warps, rank 1's producer and 4 epilogue warps
constexpr uint32_t kEpiWarps = 8;       // epilogue warps of a pair: one count each per shrink sub-tile
constexpr int kABoxBytes = kBlockCols * kPK * 2;   // one 64-row box of the pool's A rows
constexpr long kHeavyFirstMaxW = 64L << 20;       // W bytes up to which heavy-first order is used
// K up to which the shrink runs as sub-tiles of the GEMM: a sub-tile takes a whole K loop on one
// pair, which for long K costs more than the separate split-K shrink kernel.
constexpr int kFuseMaxK = 8192;

// The side path of the step (null pointers and fused = 0 without metadata).
struct PairSide {
  const int32_t* ptile_off;    // [pair tiles + 1] entries of each pair tile
  const int32_t* pent_blk;     // column block of each entry
  const int32_t* pent_u0;      // unit of M-tile 2 mp on the entry's block (-1: none)
  const int32_t* pent_u1;      // unit of M-tile 2 mp + 1 on it
  const int32_t* grp_mp;       // shrink groups: up to kGroupUnits consecutive entries of one pair tile
  const int32_t* grp_ent;
  const int32_t* grp_cnt;
  const int32_t* n_groups;     // number of groups (device)
  const int32_t* ptile_order;  // pair tiles by entry count, most first
  uint32_t* sync;              // [0] ticket, [1] pairs done, [2 + mp] shrink sub-tiles written (x kEpiWarps)
  uint16_t* vtile;             // [units][128][64] bf16 scaled v
  const int32_t* pair_slot;    // [T * J] validated slot per pair
  const float* pair_scale;     // [T * J]
  const int32_t* col_slot;     // pool layout: owner of each column of the slot space
  const int32_t* slot_off;
  const int32_t* slot_rank;
  const float* slot_scale;
  int v_rows;                  // rows of vtile: a box from here on reads zeros
  int C;                       // columns of the slot space
  int J;
  int fused;                   // 1: shrink sub-tiles, dynamic order, dependency counters
  int heavy_first;             // 1: every tile of the pair tile with the most entries first (W fits in
                               //    L2); 0: column tiles in order, each column's pair tiles heaviest first
};

struct PairTile {
  int kind;     // 0: a tile of y, 1: a shrink sub-tile, 2: an empty shrink sub-tile (nothing to do)
  int mp;       // pair tile (M-tiles 2 mp and 2 mp + 1)
  int n_idx;    // column tile of y (kind 0)
  int e0, cnt;  // entries of the pair tile (kind 1)
};

// Tile t of the launch. With the fused side path, tickets 0 .. S - 1 are the shrink sub-tiles
// (each group of up to kGroupUnits entries split into kGroupUnits / per parts of `per` entries),
// then the tiles of y in one of two orders: pair tile by pair tile in the metadata's heavy-first
// order (the pairs that start first take the tiles with the most extra K blocks; W is streamed
// once per pair tile, so this is used when W fits in L2), or column tile by column tile with the
// pair tiles of each column heaviest first (W streamed once). Without the side path, the static
// order of pair_row.
__device__ __forceinline__ PairTile pair_tile(int t, int S, int per, int num_mp, int num_n, const PairSide& sp) {
  PairTile pt{};
  if (t < S) {
    const int parts = kGroupUnits / per;
    const int g = t / parts, part = t - g * parts;
    pt.mp = sp.grp_mp[g];
    pt.e0 = sp.grp_ent[g] + part * per;
    pt.cnt = min(per, sp.grp_cnt[g] - part * per);
    pt.kind = pt.cnt > 0 ? 1 : 2;
    return pt;
  }
  const int b = t - S;
  if (sp.fused && sp.heavy_first) {
    pt.mp = sp.ptile_order[b / num_n];
    pt.n_idx = b % num_n;
  } else if (sp.fused) {
    pt.mp = sp.ptile_order[b % num_mp];
    pt.n_idx = b / num_mp;
  } else {
    pt.mp = pair_row(b, num_mp);
    pt.n_idx = b / num_mp;
  }
  pt.kind = 0;
  return pt;
}

template <int BN, int STAGES>
__global__ void __launch_bounds__(kPairThreads, 1)
gemm_bf16_pair_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_w,
                      const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_b,
                      const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_y,
                      const PairSide sp, float* __restrict__ y, int y_tma, int T, int D, int K,
                      uint32_t* __restrict__ err) {
  using L = PairCfg<BN, STAGES>;
  constexpr int kPer = L::kBRows >= 2 * kBlockCols ? 4 : 2;   // entries per shrink sub-tile (N <= 2 kBRows)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBarrierOffset);   // used in rank 0
  uint64_t* empty = full + STAGES;                                           // in each CTA
  uint64_t* acc_full = empty + STAGES;                                       // in each CTA
  uint64_t* acc_empty = acc_full + 2;                                        // used in rank 0
  uint64_t* sched_full = acc_empty + 2;                                      // in each CTA
  uint64_t* sched_empty = sched_full + kSchedDepth;                          // used in rank 0
  int* sched_tile = reinterpret_cast<int*>(sched_empty + kSchedDepth);       // in each CTA
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sched_tile + kSchedDepth);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();          // 0 or 1 (clusters of two, along x)
  const int pair = blockIdx.x >> 1;
  const int n_pairs = gridDim.x >> 1;
  const int num_m = (T + kHalf - 1) / kHalf;             // 128-row M-tiles
  const int num_mp = (num_m + 1) / 2;                    // pair tiles along M
  const int num_n = (D + BN - 1) / BN;
  const int num_kb = (K + kPK - 1) / kPK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&full[s], 1);            // rank 0's producer posts both halves' bytes
      ptx::mbar_init(&empty[s], 1);           // one multicast commit per stage use
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&acc_full[a], 1);
      ptx::mbar_init(&acc_empty[a], 8);       // one arrival per epilogue warp of both CTAs
    }
    for (int k = 0; k < kSchedDepth; ++k) {
      ptx::mbar_init(&sched_full[k], 1);      // the scheduler's arrival after writing the id
      ptx::mbar_init(&sched_empty[k], kSchedUsers);
    }
    ptx::fence_barrier_init();
    ptx::fence_proxy_async_smem();
    ptx::tma_prefetch_desc(&tmap_x);
    ptx::tma_prefetch_desc(&tmap_w);
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(tmem_slot, L::kTmemCols);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  ptx::cluster_sync_all();                    // barriers of both CTAs initialised, TMEM allocated
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // programmatic dependent launch: the set-up above overlapped the previous kernel's tail; from
  // here on its results (x, the metadata) are read. The next kernel may start its own set-up.
  ptx::grid_dependency_wait();
  ptx::grid_dependents_launch();
  const int S = sp.fused ? *sp.n_groups * (kGroupUnits / kPer) : 0;
  const int total = S + num_mp * num_n;

  // Reads tile id number i of this pair (one thread of each reading role): waits for it, then
  // tells rank 0's scheduler that this reader is done with the slot. -1: no more tiles (or a
  // timeout). The wait polls with the plain barrier test (polling with cluster-scope acquires
  // slows the SM's TMA traffic); in rank 1, whose copy rank 0 wrote remotely, one more test of
  // the completed phase with acquire at cluster scope then orders the read of the id.
  auto read_tile = [&](int i) -> int {
    const int k = i % kSchedDepth;
    const uint32_t sph = static_cast<uint32_t>(i / kSchedDepth) & 1u;
    if (!ptx::mbar_wait_short(&sched_full[k], sph, err)) return -1;
    if (rank != 0) (void)ptx::mbar_try_wait_cluster(&sched_full[k], sph, 0);
    const int t = *reinterpret_cast<volatile int*>(&sched_tile[k]);
    if (rank == 0) ptx::mbar_arrive(&sched_empty[k]);
    else ptx::mbar_arrive_cluster(ptx::mapa_shared(ptx::smem_u32(&sched_empty[k]), 0));
    return t;
  };

  if (warp == 0) {
    if (lane == 0) {
      const int32_t* own_unit = rank == 0 ? sp.pent_u0 : sp.pent_u1;
      const int blk_out = (sp.C + kBlockCols - 1) / kBlockCols + 1;   // an A box past the end: zeros
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int i = 0; ok; ++i) {
        int t;
        if (rank == 0) {
          // the scheduler: the next tile id, to both CTAs of the pair
          const int k = i % kSchedDepth;
          const uint32_t sph = static_cast<uint32_t>(i / kSchedDepth) & 1u;
          if (!ptx::mbar_wait_short(&sched_empty[k], sph ^ 1u, err)) ok = false;
          if (!ok) {
            t = -1;
          } else if (sp.fused) {
            const int tk = static_cast<int>(atomicAdd(&sp.sync[0], 1u));
            t = tk < total ? tk : -1;
          } else {
            const long tk = pair + static_cast<long>(i) * n_pairs;
            t = tk < total ? static_cast<int>(tk) : -1;
          }
          sched_tile[k] = t;
          ptx::st_dsmem_u32(ptx::mapa_shared(ptx::smem_u32(&sched_tile[k]), 1), static_cast<uint32_t>(t));
          ptx::mbar_arrive_release_cluster(&sched_full[k]);
          ptx::mbar_arrive_cluster(ptx::mapa_shared(ptx::smem_u32(&sched_full[k]), 1));
        } else {
          t = read_tile(i);
        }
        if (t < 0) break;
        const PairTile pt = pair_tile(t, S, kPer, num_mp, num_n, sp);
        if (pt.kind == 2) continue;
        const int m_blk = 2 * pt.mp + static_cast<int>(rank);
        if (pt.kind == 1) {
          // shrink sub-tile: x rows of this CTA's M-tile against this CTA's half of the entries' A
          // rows (64-row boxes; entries past the sub-tile read zeros)
          const int boxes = pt.cnt <= 2 ? 1 : 2;
          const uint32_t sbytes = static_cast<uint32_t>(kPairABytes + boxes * kABoxBytes);
          for (int kb = 0; kb < num_kb; ++kb) {
            if (!ptx::mbar_wait_short(&empty[stage], phase ^ 1u, err)) { ok = false; break; }
            uint8_t* sa = smem + stage * L::kStageBytes;
            uint8_t* sb = sa + kPairABytes;
            const uint32_t bar = ptx::mapa_shared(ptx::smem_u32(&full[stage]), 0);
            if (rank == 0) ptx::mbar_arrive_expect_tx(&full[stage], 2 * sbytes);
            ptx::tma_load_2d_pair(sa, &tmap_x, bar, kb * kPK, m_blk * kHalf);
            for (int b = 0; b < boxes; ++b) {
              const int ent = static_cast<int>(rank) * boxes + b;
              const int blk = ent < pt.cnt ? sp.pent_blk[pt.e0 + ent] : blk_out;
              ptx::tma_load_2d_pair(sb + b * kABoxBytes, &tmap_a, bar, kb * kPK, blk * kBlockCols);
            }
            if (++stage == STAGES) { stage = 0; phase ^= 1u; }
          }
          continue;
        }
        const int n0 = pt.n_idx * BN + static_cast<int>(rank) * L::kBRows;
        const int n_extra = pair_extra(sp.ptile_off, pt.mp);
        // the tile's K blocks of x and W (kept free of other work: a branch in this loop slows it)
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!ptx::mbar_wait_short(&empty[stage], phase ^ 1u, err)) { ok = false; break; }
          uint8_t* sa = smem + stage * L::kStageBytes;
          uint8_t* sb = sa + kPairABytes;
          const uint32_t bar = ptx::mapa_shared(ptx::smem_u32(&full[stage]), 0);   // rank 0's barrier
          if (rank == 0) ptx::mbar_arrive_expect_tx(&full[stage], 2 * L::kStageBytes);
          ptx::tma_load_2d_pair(sa, &tmap_x, bar, kb * kPK, m_blk * kHalf);
          ptx::tma_load_2d_pair(sb, &tmap_w, bar, kb * kPK, n0);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok || n_extra == 0) continue;
        if (sp.fused) {
          // the v tiles of this pair tile come from its shrink sub-tiles of this launch
          const uint32_t target = kEpiWarps * static_cast<uint32_t>((n_extra + kPer - 1) / kPer);
          if (!ptx::wait_counter(&sp.sync[2 + pt.mp], target, err)) { ok = false; break; }
          ptx::fence_proxy_async_global();
        }
        // then one K block per entry of the pair tile: this M-tile's v tile (or zeros) and the
        // block's 64 columns of B
        const int e0 = sp.ptile_off[pt.mp];
        for (int e = e0; e < e0 + n_extra; ++e) {
          if (!ptx::mbar_wait_short(&empty[stage], phase ^ 1u, err)) { ok = false; break; }
          uint8_t* sa = smem + stage * L::kStageBytes;
          uint8_t* sb = sa + kPairABytes;
          const uint32_t bar = ptx::mapa_shared(ptx::smem_u32(&full[stage]), 0);
          if (rank == 0) ptx::mbar_arrive_expect_tx(&full[stage], 2 * L::kStageBytes);
          const int own = own_unit[e];
          const int vrow = own >= 0 ? own * kHalf : sp.v_rows;   // v_rows: past the end, zeros
          ptx::tma_load_2d_pair(sa, &tmap_v, bar, 0, vrow);
          ptx::tma_load_2d_pair(sb, &tmap_b, bar, sp.pent_blk[e] * kBlockCols, n0);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      // tail: every stage released, i.e. every commit addressed to this CTA's stage barriers has
      // landed before the CTA may exit
      for (int i = 0; i < STAGES && ok; ++i) {
        ok = ptx::mbar_wait_short(&empty[stage], phase ^ 1u, err);
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
    }
  } else if (warp == 1) {
    if (rank == 0 && lane == 0) {
      constexpr uint32_t idesc_y = ptx::idesc_bf16_f32(kPairM, BN);
      constexpr uint16_t kBoth = 0x3;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int local = 0;
      for (int i = 0; ok; ++i) {
        const int t = read_tile(i);
        if (t < 0) break;
        const PairTile pt = pair_tile(t, S, kPer, num_mp, num_n, sp);
        if (pt.kind == 2) continue;
        const int acc = local & 1;
        const uint32_t acc_phase = static_cast<uint32_t>(local >> 1) & 1u;
        if (!ptx::mbar_wait_short(&acc_empty[acc], acc_phase ^ 1u, err)) break;
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * L::kAccStride);
        const int n_kb = pt.kind == 1 ? num_kb : num_kb + pair_extra(sp.ptile_off, pt.mp);
        const uint32_t idesc = pt.kind == 1 ? ptx::idesc_bf16_f32(kPairM, pt.cnt <= 2 ? 128 : 256) : idesc_y;
        for (int kb = 0; kb < n_kb; ++kb) {
          if (!ptx::mbar_wait_short(&full[stage], phase, err)) { ok = false; break; }
          ptx::tc_fence_after();
          const uint32_t a_addr = ptx::smem_u32(smem + stage * L::kStageBytes);
          const uint64_t a_desc = ptx::sw128_kmajor_desc(a_addr);
          const uint64_t b_desc = ptx::sw128_kmajor_desc(a_addr + kPairABytes);
#pragma unroll
          for (int k = 0; k < kPK / 16; ++k)   // K advances 16 elements = 32 bytes = 2 descriptor units
            ptx::umma_bf16_pair(d_tmem, a_desc + 2u * k, b_desc + 2u * k, idesc, (kb > 0 || k > 0) ? 1u : 0u);
          ptx::umma_commit_pair(&empty[stage], kBoth);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        ptx::umma_commit_pair(&acc_full[acc], kBoth);
        ++local;
      }
    }
  } else {
    // epilogue: warp w reads TMEM lanes 32*(w%4) .. +31 = rows of this CTA's half of the tile.
    // Tiles of y: with y_tma, each 32 x 32 block goes through a swizzled staging box in shared
    // memory (two per warp, alternating) and out with a TMA store, which writes whole lines and
    // clips the ragged edges; otherwise every thread stores its own row. Shrink sub-tiles: each
    // thread masks its token's row to the columns of the token's own slots, scales it and writes
    // it as bf16 to the v tile of its M-tile's unit on each entry's block; then the warp counts
    // itself done for the pair tile.
    const int quarter = warp & 3;
    const int row_in_half = quarter * 32 + lane;
    uint8_t* stage_box = smem + L::kEpiOffset + quarter * 2 * kEpiBoxBytes;
    int box = 0;
    int local = 0;
    for (int i = 0;; ++i) {
      int t = 0;
      if (lane == 0) t = read_tile(i);
      t = __shfl_sync(0xffffffffu, t, 0);
      if (t < 0) break;
      const PairTile pt = pair_tile(t, S, kPer, num_mp, num_n, sp);
      if (pt.kind == 2) continue;
      const int acc = local & 1;
      const uint32_t acc_phase = static_cast<uint32_t>(local >> 1) & 1u;
      if (!ptx::mbar_wait_short(&acc_full[acc], acc_phase, err)) break;
      ptx::tc_fence_after();
      const uint32_t lane_tmem = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                 static_cast<uint32_t>(acc * L::kAccStride);
      const int m0 = (2 * pt.mp + static_cast<int>(rank)) * kHalf;
      if (pt.kind == 1) {
        const int tok = m0 + row_in_half;
        const bool row_ok = tok < T;
        // per column of the sub-tile's entries: the owning slot and its factor (0 past the rank or
        // in a gap), in this warp's staging area once its earlier stores have read it
        if (y_tma && lane == 0) ptx::bulk_wait_group_read<0>();
        __syncwarp();
        int* tab_own = reinterpret_cast<int*>(stage_box);
        float* tab_fac = reinterpret_cast<float*>(stage_box + 4 * kGroupUnits * kBlockCols);
        for (int c = lane; c < pt.cnt * kBlockCols; c += 32) {
          const int col = sp.pent_blk[pt.e0 + c / kBlockCols] * kBlockCols + c % kBlockCols;
          const int owner = col < sp.C ? sp.col_slot[col] : -1;
          float f = 0.f;
          if (owner >= 0 && col - sp.slot_off[owner] < sp.slot_rank[owner]) f = sp.slot_scale[owner];
          tab_own[c] = owner;
          tab_fac[c] = f;
        }
        __syncwarp();
        int sl[kMaxJ];
        float sc[kMaxJ];
#pragma unroll
        for (int j = 0; j < kMaxJ; ++j) {
          const bool in = row_ok && j < sp.J;
          sl[j] = in ? sp.pair_slot[static_cast<size_t>(tok) * sp.J + j] : -1;
          sc[j] = in ? sp.pair_scale[static_cast<size_t>(tok) * sp.J + j] : 0.f;
        }
        const int32_t* own_unit = rank == 0 ? sp.pent_u0 : sp.pent_u1;
        const bool one_slot = sp.J == 1;
        for (int e = 0; e < pt.cnt; ++e) {
          const int u = own_unit[pt.e0 + e];
          if (u < 0) continue;                                // this M-tile does not use the block
#pragma unroll 1
          for (int h = 0; h < 2; ++h) {
            const int c0 = e * kBlockCols + h * 32;
            uint32_t r[32];
            ptx::tmem_ld_32x32b_x32(lane_tmem + static_cast<uint32_t>(c0), r);
            ptx::tmem_ld_wait();
            if (!row_ok) continue;
            uint32_t w[16];
#pragma unroll
            for (int q = 0; q < 16; ++q) {
              float v2[2];
#pragma unroll
              for (int z = 0; z < 2; ++z) {
                const int c = c0 + 2 * q + z;
                const int owner = tab_own[c];
                float coef = 0.f;
                if (one_slot) {
                  coef = (owner >= 0 && sl[0] == owner) ? sc[0] : 0.f;
                } else {
#pragma unroll
                  for (int j = 0; j < kMaxJ; ++j)
                    if (owner >= 0 && sl[j] == owner) coef += sc[j];
                }
                v2[z] = coef * tab_fac[c] * __uint_as_float(r[2 * q + z]);
              }
              const __nv_bfloat162 b2 = __floats2bfloat162_rn(v2[0], v2[1]);
              w[q] = *reinterpret_cast<const uint32_t*>(&b2);
            }
            uint4* dst = reinterpret_cast<uint4*>(sp.vtile + (static_cast<size_t>(u) * kHalf + row_in_half) * kBlockCols + h * 32);
#pragma unroll
            for (int q = 0; q < 4; ++q) dst[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
          }
        }
        __threadfence();                                      // this warp's v rows, then its count
        __syncwarp();
        if (lane == 0) atomicAdd(&sp.sync[2 + pt.mp], 1u);
      } else {
        const int n0 = pt.n_idx * BN;
        const int row = m0 + row_in_half;
        float* yrow = y + static_cast<size_t>(row) * D;
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t r[32];
          ptx::tmem_ld_32x32b_x32(lane_tmem + static_cast<uint32_t>(c), r);
          ptx::tmem_ld_wait();
          const int col = n0 + c;
          if (y_tma) {
            // a box wholly past the edge is skipped outright, so that every staged box has exactly one
            // bulk group and "at most one group still reading" means the other box is free
            if (col >= D || m0 + quarter * 32 >= T) continue;
            uint8_t* b = stage_box + box * kEpiBoxBytes;
            if (lane == 0) ptx::bulk_wait_group_read<1>();   // the store that used this box has read it
            __syncwarp();
            float4* rowp = reinterpret_cast<float4*>(b + lane * 128);
#pragma unroll
            for (int v = 0; v < 8; ++v)             // 16-byte chunk v of the row sits at v ^ (row % 8)
              rowp[v ^ (lane & 7)] = make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                                 __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              ptx::tma_store_2d(&tmap_y, b, col, m0 + quarter * 32);
              ptx::bulk_commit_group();
            }
            box ^= 1;
          } else if (row < T) {
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
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(ptx::mapa_shared(ptx::smem_u32(&acc_empty[acc]), 0));
      ++local;
    }
    if (y_tma && lane == 0) ptx::bulk_wait_group_all();
  }

  ptx::tc_fence_before();
  ptx::cluster_sync_all();                    // both CTAs done with TMEM and each other's barriers
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, L::kTmemCols);
  }
  if (sp.fused && rank == 0 && threadIdx.x == 0) {
    // the last pair to finish resets the launch's counters for the next launch on this metadata
    __threadfence();
    const uint32_t done = atomicAdd(&sp.sync[1], 1u);
    if (done == static_cast<uint32_t>(n_pairs) - 1u) {
      sp.sync[0] = 0u;
      sp.sync[1] = 0u;
      for (int q = 0; q < num_mp; ++q) sp.sync[2 + q] = 0u;
      __threadfence();
    }
  }
}

// The N tiles the pair kernel is built for, each with the deepest ring that fits.
using Pair256 = PairCfg<256, 6>;

template <int BN, int STAGES>
cudaError_t configure_pair() {
  return cudaFuncSetAttribute(gemm_bf16_pair_kernel<BN, STAGES>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              PairCfg<BN, STAGES>::kBytes);
}

template <int BN, int STAGES>
cudaError_t launch_pair_bn(const uint16_t* x, const uint16_t* W, float* y, int T, int K, int D, uint32_t* err,
                           const PoolView* pool, const MetaView* meta, int max_pairs, bool fuse, cudaStream_t s) {
  using L = PairCfg<BN, STAGES>;
  CUtensorMap mx, mw, mv, mb, ma;
  if (!make_tmap_bf16(&mx, x, T, K, kHalf, kPK) || !make_tmap_bf16(&mw, W, D, K, L::kBRows, kPK))
    return cudaErrorInvalidValue;
  const int num_m = (T + kHalf - 1) / kHalf;
  PairSide sp{};
  if (pool && meta) {
    // the side path: its shrink as sub-tiles of this launch (the pool's A rows), its expand as
    // extra K blocks (the v tiles and the pool's B columns)
    sp.v_rows = meta->unit_cap * kHalf;
    if (!make_tmap_bf16(&mv, meta->vtile, sp.v_rows, kPK, kHalf, kPK) ||
        !make_tmap_bf16(&mb, pool->B, D, pool->C, L::kBRows, kPK) ||
        !make_tmap_bf16(&ma, pool->A, pool->C, pool->K, kBlockCols, kPK))
      return cudaErrorInvalidValue;
    sp.ptile_off = meta->ptile_off;
    sp.pent_blk = meta->pent_blk;
    sp.pent_u0 = meta->pent_u0;
    sp.pent_u1 = meta->pent_u1;
    sp.grp_mp = meta->grp_mp;
    sp.grp_ent = meta->grp_ent;
    sp.grp_cnt = meta->grp_cnt;
    sp.n_groups = meta->counts + 7;
    sp.ptile_order = meta->ptile_order;
    sp.sync = meta->sync;
    sp.vtile = meta->vtile;
    sp.pair_slot = meta->pair_slot;
    sp.pair_scale = meta->pair_scale;
    sp.col_slot = pool->col_slot;
    sp.slot_off = pool->slot_off;
    sp.slot_rank = pool->slot_rank;
    sp.slot_scale = pool->slot_scale;
    sp.C = pool->C;
    sp.J = meta->J;
    sp.fused = fuse ? 1 : 0;
    sp.heavy_first = static_cast<long>(D) * K * 2 <= kHeavyFirstMaxW ? 1 : 0;
  } else {
    mv = mx;
    mb = mw;
    ma = mx;
  }
  CUtensorMap my;
  const int y_tma = make_tmap_f32_sw128(&my, y, T, D, 32) ? 1 : 0;   // else plain row stores
  if (!y_tma) my = mx;
  // with the side path every resident pair is launched (the shrink sub-tiles are counted on the
  // device); otherwise no more pairs than tiles
  const int tiles = ((num_m + 1) / 2) * ((D + BN - 1) / BN);
  const int pairs = sp.fused ? max_pairs : (tiles < max_pairs ? tiles : max_pairs);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.blockDim = dim3(kPairThreads, 1, 1);
  cfg.dynamicSmemBytes = L::kBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  note_launch_begin(kKindGemm, s);
  cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_bf16_pair_kernel<BN, STAGES>, mx, mw, mv, mb, ma, my, sp, y, y_tma, T,
                                     D, K, err);
  note_launch_end(kKindGemm, s);
  return e;
}

// Estimated launch time for N tile bn, in units of one 256 x 256 pair tile: whole waves of the
// resident pairs (a partial last wave costs a full one) times the time of one tile. That time is
// mostly independent of the tile's width (x staging, pipeline fill, epilogue) and only partly
// proportional to it; the split is fitted to single-launch timings of the four widths at
// T = 512-2048, K = 4096-14336 on GB300.
double pair_time(int T, int D, int bn, int max_pairs) {
  const long mp = ((T + kHalf - 1) / kHalf + 1) / 2;
  const long tiles = mp * ((D + bn - 1) / bn);
  const long waves = (tiles + max_pairs - 1) / max_pairs;
  return static_cast<double>(waves) * (0.83 + 0.17 * bn / 256.0);
}

// The same with the dynamic schedule of the fused side path: the pairs that finish early take the
// remaining tiles, so a partial last wave costs its fraction (at least one tile per pair).
double pair_time_dynamic(int T, int D, int bn, int max_pairs) {
  const long mp = ((T + kHalf - 1) / kHalf + 1) / 2;
  const long tiles = mp * ((D + bn - 1) / bn);
  const double waves = std::max(1.0, static_cast<double>(tiles) / max_pairs);
  return waves * (0.83 + 0.17 * bn / 256.0);
}

}  // namespace

int pair_gemm_max_pairs() {
  static int cached_device = -1, cached = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  if (cached_device == dev) return cached;
  if (configure_pair<256, 6>() != cudaSuccess || configure_pair<224, 6>() != cudaSuccess ||
      configure_pair<192, 6>() != cudaSuccess || configure_pair<128, 8>() != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  int num_sms = 0;
  cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
  cfg.gridDim = dim3(num_sms / 2 * 2, 1, 1);
  cfg.blockDim = dim3(kPairThreads, 1, 1);
  cfg.dynamicSmemBytes = Pair256::kBytes;      // the largest of the variants: one CTA per SM for all
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, gemm_bf16_pair_kernel<256, 6>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    clusters = 0;
  }
  cached_device = dev;
  cached = clusters;
  return clusters;
}

int pair_gemm_pick_n(int T, int D, int max_pairs, bool dynamic) {
  static const int kChoices[] = {256, 224, 192, 128};
  int best = 256;
  double best_time = 0.0;
  for (int bn : kChoices) {
    // static schedule: the widest of equally fast choices; dynamic schedule: the narrowest (its
    // smaller tiles balance better around the tiles with many extra K blocks)
    const double t = dynamic ? pair_time_dynamic(T, D, bn, max_pairs) : pair_time(T, D, bn, max_pairs);
    if (bn == 256 || t < best_time - 1e-9 || (dynamic && t <= best_time + 1e-9)) {
      best_time = t;
      best = bn;
    }
  }
  return best;
}

bool pair_gemm_fuses_shrink(int K) { return K <= kFuseMaxK; }

cudaError_t launch_pair_gemm(const uint16_t* x, const uint16_t* W, float* y, int T, int K, int D, uint32_t* err,
                             const PoolView* pool, const MetaView* meta, int bn, cudaStream_t s) {
  const bool fuse = pool && meta && pair_gemm_fuses_shrink(K);
  const int max_pairs = pair_gemm_max_pairs();
  if (max_pairs < 1) return cudaErrorNotSupported;
  if (bn == 0) bn = pair_gemm_pick_n(T, D, max_pairs, fuse);
  switch (bn) {
    case 256: return launch_pair_bn<256, 6>(x, W, y, T, K, D, err, pool, meta, max_pairs, fuse, s);
    case 224: return launch_pair_bn<224, 6>(x, W, y, T, K, D, err, pool, meta, max_pairs, fuse, s);
    case 192: return launch_pair_bn<192, 6>(x, W, y, T, K, D, err, pool, meta, max_pairs, fuse, s);
    case 128: return launch_pair_bn<128, 8>(x, W, y, T, K, D, err, pool, meta, max_pairs, fuse, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mlora
