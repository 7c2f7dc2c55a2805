// Shrink of the LoRA side path on the tensor cores, for every batch that takes the tensor-core
// side path (the expand then runs inside the base GEMM).
//
// "Multi-LoRA Serving Explained" (sevydevy.com), batched-serving section: grouping a slot's
// tokens lets one small product per group read the adapter once (Punica's SGMV does this per
// segment); "[RFC] Per-request activation of multiple LoRA adapters" (vLLM issue 51940),
// Proposed Change: k slots per token, each with its own scale.
//
// The slots' rank rows form one column space (slot s owns columns off_s .. off_s + width_s - 1).
// The metadata lists, per 128-token M-tile, the 64-column blocks of that space that its active
// pairs' slots own ("units"), and per pair tile (M-tiles 2 mp and 2 mp + 1, the base GEMM's
// 256-row tiles) the union of both tiles' blocks ("entries"). For an entry (pair tile, block b):
//
//   V[t][c] = sum_i x[t][i] A[64 b + c][i]                       (256 tokens, fp32 in TMEM)
//   vtile[u][t][c] = bf16( coef(t, c) V[t][c] ),  u = the unit of t's M-tile on block b,
//   coef(t, c) = sum over t's slots j owning column 64 b + c of  s[t,j] * c(slot)   (0 otherwise)
//
// so a token keeps only the columns of its own slots, already scaled; the base GEMM adds
// vtile x B[:, 64 b .. 64 b + 63]^T as one more K block of that M-tile.
//
// Design: a cluster of 2 S CTAs per group of up to kGroupUnits entries of one pair tile
// (persistent: cluster c takes groups c, c + clusters, ...). CTAs 2p and 2p + 1 form a CTA pair
// (cta_group::2) for K share p of S: each stages its own M-tile's 128 x rows and half of the
// group's A blocks per 64-wide K block, and the even CTA issues tcgen05.mma.cta_group::2 (M = 256,
// N = 64 per entry rounded up to 128 or 256), so an A block used by both M-tiles is read once and
// each SM takes in at most 32 KB per K block. Warps 2..5 of each CTA move its fp32 partial
// accumulator to shared memory; after a cluster barrier, CTA (p, h) sums rows p * 128 / S .. of
// M-tile half h over the K shares in order through distributed shared memory (deterministic),
// masks, scales and writes the bf16 rows of its tile's units; a second barrier keeps the partials
// until every CTA is done. Waits are bounded (2 s); every CTA reaches both barriers of every group
// its cluster takes, and a timeout seen by rank 0 ends the cluster's loop for all of its CTAs.
#include "internal.h"
#include "ptx.cuh"

namespace mlora {
namespace {

constexpr int kTM = 128;                                  // tokens per M-tile (per CTA of a pair)
constexpr int kBK = 64;                                   // K elements per stage
constexpr int kMaxN = kGroupUnits * kBlockCols;           // MMA N of a full group (256)
constexpr int kStages = 6;
constexpr int kThreads = 192;
constexpr int kXBytes = kTM * kBK * 2;                    // 16 KB
constexpr int kABlockBytes = kBlockCols * kBK * 2;        // 8 KB: one 64-row A box
constexpr int kStageBytes = kXBytes + (kMaxN / 2 / kBlockCols) * kABlockBytes;   // 32 KB
constexpr int kRecvLd = kMaxN + 4;                        // fp32 row stride of the receive buffers
constexpr int kMaxPairs = 3;                              // K shares (CTA pairs) per cluster
constexpr int kSmemBytes = kStages * kStageBytes + 256 + 1024;
// rows the last of `pairs` K shares reduces (it takes the remainder), and the receive buffers
__host__ __device__ constexpr int share_rows(int pairs) { return kTM - (pairs - 1) * (kTM / pairs); }
static_assert(1 * share_rows(1) * kRecvLd * 4 <= kStages * kStageBytes && 2 * share_rows(2) * kRecvLd * 4 <= kStages * kStageBytes &&
                  3 * share_rows(3) * kRecvLd * 4 <= kStages * kStageBytes,
              "receive buffers fit in the ring");
static_assert(kStageBytes % 1024 == 0, "stage alignment");
static_assert(kSmemBytes <= 232448, "shared memory");

__global__ void __launch_bounds__(kThreads, 1)
lora_shrink_pair_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_a,
                        PoolView pool, MetaView m, int pairs, uint32_t* __restrict__ err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);   // used in the even CTA
  uint64_t* empty = full + kStages;                                             // in each CTA
  uint64_t* acc_full = empty + kStages;                                         // in each CTA
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
  uint32_t* stop_flag = tmem_slot + 1;                    // written by rank 0 into every CTA
  float* recv = reinterpret_cast<float*>(smem);           // [pairs][rows of my share][kRecvLd]: the
                                                          // K shares' partials of my rows, pushed in
  __shared__ int s_slot[kTM * kMaxJ];                     // this M-tile's pair slots and scales
  __shared__ float s_scale[kTM * kMaxJ];
  __shared__ float s_fac[kMaxN];                          // per column: slot factor, 0 outside a rank
  __shared__ int s_own[kMaxN / 4];                        // per four columns: the owning slot (-1: none)
  __shared__ int s_unit[kGroupUnits];                     // this M-tile's unit per entry (-1: none)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = static_cast<int>(ptx::cluster_ctarank());
  const int half = rank & 1, share = rank >> 1;
  const int csize = 2 * pairs;
  const int n_clusters = gridDim.x / csize;
  const int cluster_id = blockIdx.x / csize;
  const int num_kb = (pool.K + kBK - 1) / kBK;
  const int kb0 = share * num_kb / pairs, kb1 = (share + 1) * num_kb / pairs;
  const int J = m.J;
  const int rows_per = kTM / pairs;                       // rows reduced by each K share (the last: the rest)
  const int recv_rows = share_rows(pairs);                // rows per K share in a receive buffer
  const int n_tiles = (m.T + kTM - 1) / kTM;
  const int blk_out = (pool.C + kBlockCols - 1) / kBlockCols + 1;   // an A box past the end: zeros
  const uint16_t pair_mask = static_cast<uint16_t>(3u << (rank & ~1));

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&full[s], 1);                        // the even CTA posts both halves' bytes
      ptx::mbar_init(&empty[s], 1);                       // one multicast commit per use
    }
    ptx::mbar_init(acc_full, 1);
    *stop_flag = 0u;
    ptx::fence_barrier_init();
    ptx::fence_proxy_async_smem();
    ptx::tma_prefetch_desc(&tmap_x);
    ptx::tma_prefetch_desc(&tmap_a);
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(tmem_slot, kMaxN);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  ptx::cluster_sync_all();                                // barriers of the cluster initialised
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  ptx::grid_dependency_wait();                            // the previous kernel's results (x, metadata)
  ptx::grid_dependents_launch();                          // the next kernel may start its set-up
  const int n_groups = m.counts[7];

  int stage = 0;                                          // ring position (producer and MMA thread)
  uint32_t phase = 0;
  int iter = 0;
  bool have_acc = false;                                  // epilogue warps: this group's accumulator is complete
  for (int g = cluster_id; g < n_groups; g += n_clusters, ++iter) {
    const int mp = m.grp_mp[g], e0 = m.grp_ent[g], cnt = m.grp_cnt[g];
    const int npad = cnt <= 2 ? 2 : 4;                    // entries incl. zero boxes: N = 128 or 256
    const int boxes = npad / 2;                           // A boxes this CTA stages per K block
    const int n_cols = npad * kBlockCols;
    const int tile = 2 * mp + half;
    const uint32_t stage_bytes = static_cast<uint32_t>(kXBytes + boxes * kABlockBytes);
    if (warp == 0) {
      if (lane == 0) {
        const uint32_t bar0 = ptx::mapa_shared(ptx::smem_u32(&full[0]), static_cast<uint32_t>(rank & ~1));
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!ptx::mbar_wait_short(&empty[stage], phase ^ 1u, err)) break;
          uint8_t* sx = smem + stage * kStageBytes;
          const uint32_t bar = bar0 + static_cast<uint32_t>(stage * sizeof(uint64_t));
          if (half == 0) ptx::mbar_arrive_expect_tx(&full[stage], 2 * stage_bytes);
          ptx::tma_load_2d_pair(sx, &tmap_x, bar, kb * kBK, tile * kTM);     // past T: zeros
          for (int k = 0; k < boxes; ++k) {
            const int ent = half * boxes + k;
            const int blk = ent < cnt ? m.pent_blk[e0 + ent] : blk_out;
            ptx::tma_load_2d_pair(sx + kXBytes + k * kABlockBytes, &tmap_a, bar, kb * kBK, blk * kBlockCols);
          }
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
      }
    } else if (warp == 1) {
      if (half == 0 && lane == 0 && kb1 > kb0) {
        const uint32_t idesc = ptx::idesc_bf16_f32(2 * kTM, n_cols);
        bool ok = true;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!ptx::mbar_wait_short(&full[stage], phase, err)) { ok = false; break; }
          ptx::tc_fence_after();
          const uint32_t x_addr = ptx::smem_u32(smem + stage * kStageBytes);
          const uint64_t x_desc = ptx::sw128_kmajor_desc(x_addr);
          const uint64_t a_desc = ptx::sw128_kmajor_desc(x_addr + kXBytes);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            ptx::umma_bf16_pair(tmem_base, x_desc + 2u * kk, a_desc + 2u * kk, idesc, (kb > kb0 || kk > 0) ? 1u : 0u);
          ptx::umma_commit_pair(&empty[stage], pair_mask);
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
        if (ok) ptx::umma_commit_pair(acc_full, pair_mask);
      }
    } else {
      // while the main loop runs: this M-tile's pair slots and scales, its unit of every entry,
      // and per column of the group its owning slot and factor (the slot factor, or 0 past the
      // adapter's rank, in a gap, or in a padding entry)
      const int et = threadIdx.x - 64;
      for (int i = et; i < kTM * J; i += kThreads - 64) {
        const int p = tile * kTM * J + i;
        const bool in = tile < n_tiles && p < m.n;
        s_slot[i] = in ? m.pair_slot[p] : -1;
        s_scale[i] = in ? m.pair_scale[p] : 0.f;
      }
      if (et < kGroupUnits) s_unit[et] = et < cnt ? (half ? m.pent_u1 : m.pent_u0)[e0 + et] : -1;
      for (int c = et; c < n_cols; c += kThreads - 64) {
        const int k = c / kBlockCols;
        const int col = k < cnt ? m.pent_blk[e0 + k] * kBlockCols + c % kBlockCols : pool.C;
        const int owner = col < pool.C ? pool.col_slot[col] : -1;
        float f = 0.f;
        if (owner >= 0 && col - pool.slot_off[owner] < pool.slot_rank[owner]) f = pool.slot_scale[owner];
        s_fac[c] = f;
        if ((c & 3) == 0) s_own[c >> 2] = owner;           // one owner per aligned group of four columns
      }
      have_acc = kb1 > kb0 && ptx::mbar_wait_short(acc_full, static_cast<uint32_t>(iter) & 1u, err);
    }
    // every CTA of the cluster is done with its stage ring (its loads have landed and its pair's
    // MMAs have read them): from here the ring holds the receive buffers
    ptx::tc_fence_before();
    ptx::cluster_sync_all();
    ptx::tc_fence_after();
    if (warp >= 2) {
      // push: token row `row` of this CTA's partial accumulator (unscaled, one TMEM lane per thread)
      // goes to the CTA of the same half that reduces it, into its receive buffer for my K share
      const int quarter = warp & 3;
      const int row = quarter * 32 + lane;
      const int owner = min(row / rows_per, pairs - 1);
      const uint32_t dst = ptx::mapa_shared(ptx::smem_u32(recv), static_cast<uint32_t>(2 * owner + half)) +
                           static_cast<uint32_t>(((share * recv_rows) + (row - owner * rows_per)) * kRecvLd * 4);
      const bool have = have_acc;
      for (int c0 = 0; c0 < n_cols; c0 += 32) {
        uint32_t r[32];
        if (have) {
          ptx::tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(c0), r);
          ptx::tmem_ld_wait();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = 0u;             // no K blocks here (or a timed-out wait)
        }
#pragma unroll
        for (int i = 0; i < 8; ++i)
          ptx::st_dsmem_f4(dst + static_cast<uint32_t>((c0 + 4 * i) * 4),
                           make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                       __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3])));
      }
    }
    ptx::tc_fence_before();
    ptx::cluster_sync_all();                              // every partial row is in its owner's buffer
    ptx::tc_fence_after();

    // rows [r0, r1) of this M-tile: sum the K shares' partials in order (local shared memory),
    // mask, scale, store the entries whose block the tile uses. Item = 32 columns of one row: a
    // thread issues all of its item's loads before summing and writes 64 bytes of v at once.
    // Consecutive threads take consecutive rows of one chunk (with the 260-float row stride the
    // eight rows of a quarter-warp fall on distinct banks).
    const int r0 = share * rows_per, r1 = share == pairs - 1 ? kTM : r0 + rows_per;
    const int chunks = cnt * (kBlockCols / 32);           // real entries only
    const int n_rows = r1 - r0;
    const int n_items = tile < n_tiles ? n_rows * chunks : 0;
    for (int e = threadIdx.x; e < n_items; e += kThreads) {
      const int ch = e / n_rows, lr = e - ch * n_rows, c0 = ch * 32;
      const int row = r0 + lr;
      const int u = s_unit[c0 / kBlockCols];
      if (u < 0) continue;                                // this M-tile does not use the block
      float4 acc[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int src = 0; src < pairs; ++src) {
        const float4* rp = reinterpret_cast<const float4*>(recv + (src * recv_rows + lr) * kRecvLd + c0);
        float4 v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = rp[q];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          acc[q].x += v[q].x;
          acc[q].y += v[q].y;
          acc[q].z += v[q].z;
          acc[q].w += v[q].w;
        }
      }
      uint32_t w[16];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int c = c0 + 4 * q;
        const int owner = s_own[c >> 2];
        float coef = 0.f;
        for (int j = 0; j < J; ++j)
          if (owner >= 0 && s_slot[row * J + j] == owner) coef += s_scale[row * J + j];
        const __nv_bfloat162 lo = __floats2bfloat162_rn(coef * s_fac[c] * acc[q].x, coef * s_fac[c + 1] * acc[q].y);
        const __nv_bfloat162 hi = __floats2bfloat162_rn(coef * s_fac[c + 2] * acc[q].z, coef * s_fac[c + 3] * acc[q].w);
        w[2 * q] = *reinterpret_cast<const uint32_t*>(&lo);
        w[2 * q + 1] = *reinterpret_cast<const uint32_t*>(&hi);
      }
      uint4* dst = reinterpret_cast<uint4*>(m.vtile + (static_cast<size_t>(u) * kTM + row) * kBlockCols + c0 % kBlockCols);
#pragma unroll
      for (int q = 0; q < 4; ++q) dst[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
    }
    // rank 0 tells every CTA of the cluster (in its own shared memory, so that no CTA reads another
    // one's memory after the barrier, when that one may already have left) whether a wait timed out
    if (rank == 0 && threadIdx.x == 0) {
      const uint32_t stop = (*reinterpret_cast<volatile uint32_t*>(err) & ptx::kErrWaitTimeout) ? 1u : 0u;
      for (int r = 0; r < csize; ++r)
        ptx::st_dsmem_u32(ptx::mapa_shared(ptx::smem_u32(stop_flag), static_cast<uint32_t>(r)), stop);
    }
    ptx::tc_fence_before();
    ptx::cluster_sync_all();                              // no CTA reuses its partials while others read them
    ptx::tc_fence_after();
    if (*reinterpret_cast<volatile uint32_t*>(stop_flag)) break;   // a wait timed out: leave together
  }
  // both CTAs of each pair are done with TMEM (every epilogue waited for its group's last commit)
  ptx::tc_fence_before();
  ptx::cluster_sync_all();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, kMaxN);
  }
}

}  // namespace

cudaError_t launch_lora_shrink_tc(const uint16_t* x, const PoolView& pool, const MetaView& m, uint32_t* err,
                                  int num_sms, cudaStream_t s) {
  if (m.T == 0 || pool.C == 0) return cudaSuccess;
  static int configured_device = -1;
  static int max_clusters[kMaxPairs + 1] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  const int num_kb = (pool.K + kBK - 1) / kBK;
  // K shares: each CTA pair covers at least 16 K blocks (all of them below 32), up to 3 pairs per
  // cluster (clusters of 6 CTAs, 25 of which fit on 152 SMs at once)
  int pairs = num_kb / 16;
  if (pairs > kMaxPairs) pairs = kMaxPairs;
  if (pairs < 1) pairs = 1;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2 * pairs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(lora_shrink_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    for (int sp = 1; sp <= kMaxPairs; ++sp) max_clusters[sp] = 0;
    configured_device = dev;
  }
  if (max_clusters[pairs] == 0) {
    // clusters of this size that can be resident at once: the persistent grid
    cfg.gridDim = dim3(num_sms / (2 * pairs) * (2 * pairs), 1, 1);
    int c = 0;
    if (cudaOccupancyMaxActiveClusters(&c, lora_shrink_pair_kernel, &cfg) != cudaSuccess || c < 1) {
      cudaGetLastError();
      c = num_sms / (2 * pairs);
    }
    max_clusters[pairs] = c;
  }
  CUtensorMap mx, ma;
  if (!make_tmap_bf16(&mx, x, m.T, pool.K, kTM, kBK) || !make_tmap_bf16(&ma, pool.A, pool.C, pool.K, kBlockCols, kBK))
    return cudaErrorInvalidValue;
  cfg.gridDim = dim3(max_clusters[pairs] * 2 * pairs, 1, 1);
  cfg.stream = s;
  cfg.numAttrs = 2;                                       // with programmatic dependent launch
  note_launch_begin(kKindShrink, s);
  cudaError_t e = cudaLaunchKernelEx(&cfg, lora_shrink_pair_kernel, mx, ma, pool, m, pairs, err);
  note_launch_end(kKindShrink, s);
  return e;
}

}  // namespace mlora
