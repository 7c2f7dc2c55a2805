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

// M row of the pair tile with sequence number `tile`: M fastest, rotated by the column index, which
// keeps every column's rows a permutation while a persistent pair's tiles walk through the rows.
__device__ __forceinline__ int pair_row(int tile, int num_mp) {
  return (tile % num_mp + tile / num_mp) % num_mp;
}

// Extra K blocks of pair tile mp (0 without the fused side path).
__device__ __forceinline__ int pair_extra(const int32_t* ptile_off, int mp) {
  return ptile_off ? ptile_off[mp + 1] - ptile_off[mp] : 0;
}

template <int BN, int STAGES>
__global__ void __launch_bounds__(kPairThreads, 1)
gemm_bf16_pair_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_w,
                      const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_b,
                      const __grid_constant__ CUtensorMap tmap_y, const int32_t* __restrict__ ptile_off,
                      const int32_t* __restrict__ pent_blk, const int32_t* __restrict__ pent_u0,
                      const int32_t* __restrict__ pent_u1, int v_rows, float* __restrict__ y, int y_tma, int T, int D,
                      int K, uint32_t* __restrict__ err) {
  using L = PairCfg<BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBarrierOffset);   // used in rank 0
  uint64_t* empty = full + STAGES;                                           // in each CTA
  uint64_t* acc_full = empty + STAGES;                                       // in each CTA
  uint64_t* acc_empty = acc_full + 2;                                        // used in rank 0
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();          // 0 or 1 (clusters of two, along x)
  const int pair = blockIdx.x >> 1;
  const int n_pairs = gridDim.x >> 1;
  const int num_m = (T + kHalf - 1) / kHalf;             // 128-row M-tiles
  const int num_mp = (num_m + 1) / 2;                    // pair tiles along M
  const int num_n = (D + BN - 1) / BN;
  const int num_tiles = num_mp * num_n;
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

  if (warp == 0) {
    if (lane == 0) {
      const int32_t* own_unit = rank == 0 ? pent_u0 : pent_u1;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = pair; tile < num_tiles && ok; tile += n_pairs) {
        const int mp = pair_row(tile, num_mp);
        const int m_blk = 2 * mp + static_cast<int>(rank);
        const int n0 = (tile / num_mp) * BN + static_cast<int>(rank) * L::kBRows;
        const int n_extra = pair_extra(ptile_off, mp);
        const int e0 = n_extra ? ptile_off[mp] : 0;
        for (int kb = 0; kb < num_kb + n_extra; ++kb) {
          if (!ptx::mbar_wait_short(&empty[stage], phase ^ 1u, err)) { ok = false; break; }
          uint8_t* sa = smem + stage * L::kStageBytes;
          uint8_t* sb = sa + kPairABytes;
          const uint32_t bar = ptx::mapa_shared(ptx::smem_u32(&full[stage]), 0);   // rank 0's barrier
          if (rank == 0) ptx::mbar_arrive_expect_tx(&full[stage], 2 * L::kStageBytes);
          if (kb < num_kb) {
            ptx::tma_load_2d_pair(sa, &tmap_x, bar, kb * kPK, m_blk * kHalf);
            ptx::tma_load_2d_pair(sb, &tmap_w, bar, kb * kPK, n0);
          } else {
            const int e = e0 + kb - num_kb;
            const int own = own_unit[e];
            const int vrow = own >= 0 ? own * kHalf : v_rows;   // v_rows: past the end, zeros
            ptx::tma_load_2d_pair(sa, &tmap_v, bar, 0, vrow);
            ptx::tma_load_2d_pair(sb, &tmap_b, bar, pent_blk[e] * kBlockCols, n0);
          }
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
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(kPairM, BN);
      constexpr uint16_t kBoth = 0x3;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int local = 0;
      for (int tile = pair; tile < num_tiles && ok; tile += n_pairs, ++local) {
        const int acc = local & 1;
        const uint32_t acc_phase = static_cast<uint32_t>(local >> 1) & 1u;
        if (!ptx::mbar_wait_short(&acc_empty[acc], acc_phase ^ 1u, err)) break;
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * L::kAccStride);
        const int n_kb = num_kb + pair_extra(ptile_off, pair_row(tile, num_mp));
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
      }
    }
  } else {
    // epilogue: warp w reads TMEM lanes 32*(w%4) .. +31 = rows of this CTA's half of the tile.
    // With y_tma, each 32 x 32 block goes through a swizzled staging box in shared memory (two per
    // warp, alternating) and out with a TMA store, which writes whole lines and clips the ragged
    // edges; otherwise every thread stores its own row.
    const int quarter = warp & 3;
    const int row_in_half = quarter * 32 + lane;
    uint8_t* stage_box = smem + L::kEpiOffset + quarter * 2 * kEpiBoxBytes;
    int box = 0;
    int local = 0;
    for (int tile = pair; tile < num_tiles; tile += n_pairs, ++local) {
      const int m0 = (2 * pair_row(tile, num_mp) + static_cast<int>(rank)) * kHalf;
      const int n0 = (tile / num_mp) * BN;
      const int acc = local & 1;
      const uint32_t acc_phase = static_cast<uint32_t>(local >> 1) & 1u;
      if (!ptx::mbar_wait_short(&acc_full[acc], acc_phase, err)) break;
      ptx::tc_fence_after();
      const int row = m0 + row_in_half;
      float* yrow = y + static_cast<size_t>(row) * D;
#pragma unroll 1
      for (int c = 0; c < BN; c += 32) {
        uint32_t r[32];
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                               static_cast<uint32_t>(acc * L::kAccStride + c);
        ptx::tmem_ld_32x32b_x32(taddr, r);
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
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(ptx::mapa_shared(ptx::smem_u32(&acc_empty[acc]), 0));
    }
    if (y_tma && lane == 0) ptx::bulk_wait_group_all();
  }

  ptx::tc_fence_before();
  ptx::cluster_sync_all();                    // both CTAs done with TMEM and each other's barriers
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, L::kTmemCols);
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
                           const PoolView* pool, const MetaView* meta, int max_pairs, cudaStream_t s) {
  using L = PairCfg<BN, STAGES>;
  CUtensorMap mx, mw, mv, mb;
  if (!make_tmap_bf16(&mx, x, T, K, kHalf, kPK) || !make_tmap_bf16(&mw, W, D, K, L::kBRows, kPK))
    return cudaErrorInvalidValue;
  const int num_m = (T + kHalf - 1) / kHalf;
  const int32_t *ptile_off = nullptr, *pent_blk = nullptr, *pent_u0 = nullptr, *pent_u1 = nullptr;
  int v_rows = 0;
  if (pool && meta) {                     // the fused side path: v tiles and the pool's B columns
    v_rows = meta->unit_cap * kHalf;
    if (!make_tmap_bf16(&mv, meta->vtile, v_rows, kPK, kHalf, kPK) ||
        !make_tmap_bf16(&mb, pool->B, D, pool->C, L::kBRows, kPK))
      return cudaErrorInvalidValue;
    ptile_off = meta->ptile_off;
    pent_blk = meta->pent_blk;
    pent_u0 = meta->pent_u0;
    pent_u1 = meta->pent_u1;
  } else {
    mv = mx;
    mb = mw;
  }
  CUtensorMap my;
  const int y_tma = make_tmap_f32_sw128(&my, y, T, D, 32) ? 1 : 0;   // else plain row stores
  if (!y_tma) my = mx;
  const int tiles = ((num_m + 1) / 2) * ((D + BN - 1) / BN);
  const int pairs = tiles < max_pairs ? tiles : max_pairs;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.blockDim = dim3(kPairThreads, 1, 1);
  cfg.dynamicSmemBytes = L::kBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  note_launch_begin(kKindGemm, s);
  cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_bf16_pair_kernel<BN, STAGES>, mx, mw, mv, mb, my, ptile_off, pent_blk,
                                     pent_u0, pent_u1, v_rows, y, y_tma, T, D, K, err);
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

int pair_gemm_pick_n(int T, int D, int max_pairs) {
  static const int kChoices[] = {256, 224, 192, 128};
  int best = 256;
  double best_time = 0.0;
  for (int bn : kChoices) {                    // the widest of equally fast choices
    const double t = pair_time(T, D, bn, max_pairs);
    if (bn == 256 || t < best_time - 1e-9) {
      best_time = t;
      best = bn;
    }
  }
  return best;
}

cudaError_t launch_pair_gemm(const uint16_t* x, const uint16_t* W, float* y, int T, int K, int D, uint32_t* err,
                             const PoolView* pool, const MetaView* meta, int bn, cudaStream_t s) {
  const int max_pairs = pair_gemm_max_pairs();
  if (max_pairs < 1) return cudaErrorNotSupported;
  if (bn == 0) bn = pair_gemm_pick_n(T, D, max_pairs);
  switch (bn) {
    case 256: return launch_pair_bn<256, 6>(x, W, y, T, K, D, err, pool, meta, max_pairs, s);
    case 224: return launch_pair_bn<224, 6>(x, W, y, T, K, D, err, pool, meta, max_pairs, s);
    case 192: return launch_pair_bn<192, 6>(x, W, y, T, K, D, err, pool, meta, max_pairs, s);
    case 128: return launch_pair_bn<128, 8>(x, W, y, T, K, D, err, pool, meta, max_pairs, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mlora
