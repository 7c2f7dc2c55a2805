// Shrink of the LoRA side path on the tensor cores, for every batch that takes the tensor-core
// side path (the expand then runs inside the base GEMM).
//
// "Multi-LoRA Serving Explained" (sevydevy.com), batched-serving section: grouping a slot's
// tokens lets one small product per group read the adapter once (Punica's SGMV does this per
// segment); "[RFC] Per-request activation of multiple LoRA adapters" (vLLM issue 51940),
// Proposed Change: k slots per token, each with its own scale.
//
// The slots' rank rows form one column space (slot s owns columns off_s .. off_s + width_s - 1).
// The metadata lists, per 128-token M-tile of the batch, the 64-column blocks of that space that
// its active pairs' slots own ("units"). For a unit (tile, block b):
//
//   V[t][c]  = sum_i x[t][i] A[64 b + c][i]                      (tcgen05, fp32 in TMEM)
//   vtile[u][t][c] = bf16( coef(t, c) V[t][c] ),
//   coef(t, c) = sum over t's slots j owning column 64 b + c of  s[t,j] * c(slot)   (0 otherwise)
//
// so a token keeps only the columns of its own slots, already scaled; the base GEMM adds
// vtile x B[:, 64 b .. 64 b + 63]^T as one more K block of that M-tile.
//
// Design: persistent clusters of `splits` CTAs, cluster c taking shrink groups c, c + clusters,
// ...; a group is up to kGroupUnits consecutive units of one tile, multiplied together (MMA M =
// 128 tokens, N = 64 per unit, so the x tile is staged once for all of them). Each CTA of the
// cluster covers its share of the K blocks: warp 0 issues the TMA loads (x box, one 64-row A box
// per unit) into a ring of stages, warp 1 issues the MMAs from one thread, warps 2..5 move the
// fp32 partial accumulator to shared memory. After a cluster barrier CTA r sums rows r*128/splits
// .. of all partials in rank order through distributed shared memory (deterministic), masks,
// scales and writes the bf16 rows; a second barrier keeps the partials until every CTA is done.
// Waits are bounded (2 s); every CTA of a cluster reaches both barriers of every group it takes,
// and a timeout seen by rank 0 ends the cluster's loop for all of its CTAs at once.
#include "internal.h"
#include "ptx.cuh"

namespace mlora {
namespace {

constexpr int kTM = 128;                                  // tokens per M-tile
constexpr int kBK = 64;                                   // K elements per stage
constexpr int kMaxN = kGroupUnits * kBlockCols;           // MMA N of a full group
constexpr int kStages = 4;
constexpr int kThreads = 192;
constexpr int kXBytes = kTM * kBK * 2;
constexpr int kABlockBytes = kBlockCols * kBK * 2;
constexpr int kStageBytes = kXBytes + kGroupUnits * kABlockBytes;
constexpr int kPartLd = kMaxN + 4;                        // fp32 row stride of the partial tile
constexpr int kMaxSplits = 8;
constexpr int kSmemBytes = kStages * kStageBytes + 256 + 1024;
static_assert(kTM * kPartLd * 4 <= kStages * kStageBytes, "partial tile fits in the stage ring");
static_assert(kStageBytes % 1024 == 0, "stage alignment");
static_assert(kSmemBytes <= 232448, "shared memory");

__global__ void __launch_bounds__(kThreads, 1)
lora_shrink_tc_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_a,
                      PoolView pool, MetaView m, int splits, uint32_t* __restrict__ err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  uint64_t* empty = full + kStages;
  uint64_t* acc_full = empty + kStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
  uint32_t* stop_flag = tmem_slot + 1;                    // rank 0's copy ends the cluster's loop
  float* part = reinterpret_cast<float*>(smem);           // [128][kPartLd] between the two barriers
  __shared__ int s_slot[kTM * kMaxJ];                     // the tile's pair slots and scales
  __shared__ float s_scale[kTM * kMaxJ];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank_in = static_cast<int>(ptx::cluster_ctarank());
  const int n_clusters = gridDim.x / splits;
  const int cluster_id = blockIdx.x / splits;
  const int num_kb = (pool.K + kBK - 1) / kBK;
  const int kb0 = rank_in * num_kb / splits, kb1 = (rank_in + 1) * num_kb / splits;
  const int J = m.J;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    ptx::mbar_init(acc_full, 1);
    *stop_flag = 0u;
    ptx::fence_barrier_init();
    ptx::fence_proxy_async_smem();
    ptx::tma_prefetch_desc(&tmap_x);
    ptx::tma_prefetch_desc(&tmap_a);
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, kMaxN);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int n_groups = m.counts[7];

  int stage = 0;                                          // ring position (producer and MMA thread)
  uint32_t phase = 0;
  int iter = 0;
  for (int g = cluster_id; g < n_groups; g += n_clusters, ++iter) {
    const int u0 = m.grp_unit[g], cnt = m.grp_cnt[g];
    const int tile = m.unit_tile[u0];
    const int n_cols = cnt * kBlockCols;
    if (warp == 0) {
      if (lane == 0) {
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!ptx::mbar_wait(&empty[stage], phase ^ 1u, err)) break;
          uint8_t* sx = smem + stage * kStageBytes;
          ptx::mbar_arrive_expect_tx(&full[stage], static_cast<uint32_t>(kXBytes + cnt * kABlockBytes));
          ptx::tma_load_2d(sx, &tmap_x, &full[stage], kb * kBK, tile * kTM);
          for (int k = 0; k < cnt; ++k)
            ptx::tma_load_2d(sx + kXBytes + k * kABlockBytes, &tmap_a, &full[stage], kb * kBK,
                             m.unit_blk[u0 + k] * kBlockCols);
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
      }
    } else if (warp == 1) {
      if (lane == 0 && kb1 > kb0) {
        const uint32_t idesc = ptx::idesc_bf16_f32(kTM, n_cols);
        bool ok = true;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!ptx::mbar_wait(&full[stage], phase, err)) { ok = false; break; }
          ptx::tc_fence_after();
          const uint32_t x_addr = ptx::smem_u32(smem + stage * kStageBytes);
          const uint64_t x_desc = ptx::sw128_kmajor_desc(x_addr);
          const uint64_t a_desc = ptx::sw128_kmajor_desc(x_addr + kXBytes);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            ptx::umma_bf16(tmem_base, x_desc + 2u * kk, a_desc + 2u * kk, idesc, (kb > kb0 || kk > 0) ? 1u : 0u);
          ptx::umma_commit(&empty[stage]);
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
        if (ok) ptx::umma_commit(acc_full);
      }
    } else {
      // partial accumulator (unscaled) -> shared memory, one token row per thread
      const int quarter = warp & 3;
      const int row = quarter * 32 + lane;
      float* prow = part + row * kPartLd;
      const bool have = kb1 > kb0 && ptx::mbar_wait(acc_full, static_cast<uint32_t>(iter) & 1u, err);
      if (have) ptx::tc_fence_after();
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
          *reinterpret_cast<float4*>(prow + c0 + 4 * i) =
              make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]), __uint_as_float(r[4 * i + 2]),
                          __uint_as_float(r[4 * i + 3]));
      }
    }
    // the tile's pair slots and scales, for the masks below
    for (int i = threadIdx.x; i < kTM * J; i += kThreads) {
      const int p = tile * kTM * J + i;
      const bool in = p < m.n;
      s_slot[i] = in ? m.pair_slot[p] : -1;
      s_scale[i] = in ? m.pair_scale[p] : 0.f;
    }
    ptx::tc_fence_before();
    ptx::cluster_sync_all();                              // every partial tile is in shared memory
    ptx::tc_fence_after();

    // rows [r0, r1) of the tile: sum the partials of ranks 0, 1, ... in order, mask, scale, store
    const int rows_per = kTM / splits;
    const int r0 = rank_in * rows_per, r1 = rank_in == splits - 1 ? kTM : r0 + rows_per;
    const int c4n = n_cols / 4;
    for (int e = threadIdx.x; e < (r1 - r0) * c4n; e += kThreads) {
      const int row = r0 + e / c4n, c4 = (e % c4n) * 4;
      const uint32_t off = static_cast<uint32_t>((row * kPartLd + c4) * 4);
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int src = 0; src < splits; ++src) {
        const float4 v = ptx::ld_dsmem_f4(ptx::mapa_shared(ptx::smem_u32(part), static_cast<uint32_t>(src)) + off);
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
      }
      const int k = c4 / kBlockCols, cb = c4 % kBlockCols;
      const int col = m.unit_blk[u0 + k] * kBlockCols + cb;  // four columns of one 8-column granule
      const int owner = col < pool.C ? pool.col_slot[col] : -1;
      float coef = 0.f;
      int q = 0, rank = 0;
      if (owner >= 0) {
        for (int j = 0; j < J; ++j)
          if (s_slot[row * J + j] == owner) coef += s_scale[row * J + j] * pool.slot_scale[owner];
        q = col - pool.slot_off[owner];
        rank = pool.slot_rank[owner];
      }
      const float a0 = q < rank ? coef * acc.x : 0.f, a1 = q + 1 < rank ? coef * acc.y : 0.f;
      const float a2 = q + 2 < rank ? coef * acc.z : 0.f, a3 = q + 3 < rank ? coef * acc.w : 0.f;
      const __nv_bfloat162 lo = __floats2bfloat162_rn(a0, a1), hi = __floats2bfloat162_rn(a2, a3);
      uint16_t* dst = m.vtile + (static_cast<size_t>(u0 + k) * kTM + row) * kBlockCols + cb;
      *reinterpret_cast<uint2*>(dst) =
          make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
    }
    if (rank_in == 0 && threadIdx.x == 0) *stop_flag = (*reinterpret_cast<volatile uint32_t*>(err) & ptx::kErrWaitTimeout) ? 1u : 0u;
    ptx::tc_fence_before();
    ptx::cluster_sync_all();                              // no CTA reuses its partials while others read them
    ptx::tc_fence_after();
    if (ptx::ld_dsmem_u32(ptx::mapa_shared(ptx::smem_u32(stop_flag), 0))) break;   // a wait timed out: leave together
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, kMaxN);
  }
}

}  // namespace

cudaError_t launch_lora_shrink_tc(const uint16_t* x, const PoolView& pool, const MetaView& m, uint32_t* err,
                                  int num_sms, cudaStream_t s) {
  if (m.T == 0 || pool.C == 0) return cudaSuccess;
  static int configured_device = -1;
  static int max_clusters[kMaxSplits + 1] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  const int num_kb = (pool.K + kBK - 1) / kBK;
  // K splits: each CTA covers about 16 K blocks (at least one)
  int splits = num_kb / 16;
  if (splits > kMaxSplits) splits = kMaxSplits;
  if (splits < 1) splits = 1;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = splits;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(lora_shrink_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    for (int sp = 1; sp <= kMaxSplits; ++sp) max_clusters[sp] = 0;
    configured_device = dev;
  }
  if (max_clusters[splits] == 0) {
    // clusters of this size that can be resident at once: the persistent grid
    cfg.gridDim = dim3(num_sms / splits * splits, 1, 1);
    int c = 0;
    if (cudaOccupancyMaxActiveClusters(&c, lora_shrink_tc_kernel, &cfg) != cudaSuccess || c < 1) {
      cudaGetLastError();
      c = num_sms / splits;
    }
    max_clusters[splits] = c;
  }
  CUtensorMap mx, ma;
  if (!make_tmap_bf16(&mx, x, m.T, pool.K, kTM, kBK) || !make_tmap_bf16(&ma, pool.A, pool.C, pool.K, kBlockCols, kBK))
    return cudaErrorInvalidValue;
  cfg.gridDim = dim3(max_clusters[splits] * splits, 1, 1);
  cfg.stream = s;
  note_launch_begin(kKindShrink, s);
  cudaError_t e = cudaLaunchKernelEx(&cfg, lora_shrink_tc_kernel, mx, ma, pool, m, splits, err);
  note_launch_end(kKindShrink, s);
  return e;
}

}  // namespace mlora
