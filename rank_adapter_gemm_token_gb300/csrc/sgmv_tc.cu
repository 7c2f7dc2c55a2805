// Shrink of the LoRA side path on the tensor cores, for batches with long runs of one slot
// (prefill segments).
//
// "Multi-LoRA Serving Explained" (sevydevy.com), batched-serving section: grouping a slot's
// tokens lets one small product per group read the adapter once; Punica's SGMV does this per
// segment. Here the group is a 128-token M-tile of the base GEMM (tokens in x order) and one of
// the at most kTileSlots slots its pairs use (the metadata lists them per tile):
//
//   V[t][q] = sum_i x[t][i] A_slot[q][i]          (tcgen05, M = 128 tokens, N = 64, fp32 in TMEM)
//   vtile[tile][k][t][q] = bf16( coef(t, slot) * V[t][q] ),
//   coef(t, slot) = sum over t's slots j equal to slot of  s[t,j] * c(slot)   (0 for other tokens)
//
// The tiled base GEMM then adds vtile x B_slot^T as one extra 64-wide K block per (tile, slot),
// so the expand happens inside its accumulator (no read-modify-write of y). This path covers
// pools whose padded rank R is 64; a tile with more than kTileSlots slots (decode-like mixes) is
// left to the CUDA-core shrink/expand, which skip the pairs handled here.
//
// Design: a cluster of `splits` CTAs per (tile, slot), each over its share of the K blocks: warp
// 0 issues TMA loads of a 128 x 64 x tile and a 64 x 64 A tile per stage, warp 1 issues
// tcgen05.mma from one thread, warps 2..5 move the fp32 partial accumulator to shared memory.
// After a cluster barrier, CTA r sums rows r*128/splits .. of all partials in rank order (through
// distributed shared memory; deterministic), scales them and writes the bf16 rows. Waits are
// bounded (2 s) and every CTA of a cluster reaches both cluster barriers.
#include "internal.h"
#include "ptx.cuh"

namespace mlora {
namespace {

constexpr int kTM = 128;            // tokens per tile
constexpr int kBK = 64;
constexpr int kR = 64;              // rank width of the pools this path serves
constexpr int kStages = 6;
constexpr int kThreads = 192;
constexpr int kXBytes = kTM * kBK * 2;
constexpr int kABytes = kR * kBK * 2;
constexpr int kStageBytes = kXBytes + kABytes;
constexpr int kPartLd = kR + 4;     // fp32 row stride of the partial tile (16-byte stores spread over banks)
constexpr int kMaxSplits = 8;
constexpr int kSmemBytes = kStages * kStageBytes + 256 + 1024;
static_assert(kTM * kPartLd * 4 <= kStages * kStageBytes, "partial tile fits in the stage ring");

__global__ void __launch_bounds__(kThreads, 1)
sgmv_shrink_tc_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_a,
                      PoolView pool, MetaView m, int splits, uint32_t* __restrict__ err) {
  const int unit = blockIdx.x / splits;                  // (tile, slot entry) of this cluster
  const int tile = unit / kTileSlots, k = unit % kTileSlots;
  const int32_t* info = m.tile_info + tile * (kTileSlots + 1);
  const int cnt = info[0];
  if (cnt > kTileSlots || k >= cnt) return;               // overflow tile or unused entry: whole cluster
  const int slot = info[1 + k];
  const int rank_in = static_cast<int>(ptx::cluster_ctarank());

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  uint64_t* empty = full + kStages;
  uint64_t* acc_full = empty + kStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
  float* part = reinterpret_cast<float*>(smem);           // [128][kPartLd] after the main loop
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_kb = (pool.K + kBK - 1) / kBK;
  const int kb0 = rank_in * num_kb / splits, kb1 = (rank_in + 1) * num_kb / splits;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    ptx::mbar_init(acc_full, 1);
    ptx::fence_barrier_init();
    ptx::fence_proxy_async_smem();
    ptx::tma_prefetch_desc(&tmap_x);
    ptx::tma_prefetch_desc(&tmap_a);
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, kR);
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
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!ptx::mbar_wait(&empty[stage], phase ^ 1u, err)) break;
        uint8_t* sx = smem + stage * kStageBytes;
        ptx::mbar_arrive_expect_tx(&full[stage], kStageBytes);
        ptx::tma_load_2d(sx, &tmap_x, &full[stage], kb * kBK, tile * kTM);
        ptx::tma_load_2d(sx + kXBytes, &tmap_a, &full[stage], kb * kBK, slot * kR);
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && kb1 > kb0) {
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(kTM, kR);
      int stage = 0;
      uint32_t phase = 0;
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
    const bool have = kb1 > kb0 && ptx::mbar_wait(acc_full, 0, err);
    if (have) ptx::tc_fence_after();
#pragma unroll
    for (int c0 = 0; c0 < kR; c0 += 32) {
      uint32_t r[32];
      if (have) {
        ptx::tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(c0), r);
        ptx::tmem_ld_wait();
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) r[i] = 0u;               // no K blocks here (or a timed-out wait)
      }
#pragma unroll
      for (int i = 0; i < 8; ++i)
        *reinterpret_cast<float4*>(prow + c0 + 4 * i) =
            make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]), __uint_as_float(r[4 * i + 2]),
                        __uint_as_float(r[4 * i + 3]));
    }
  }
  ptx::tc_fence_before();
  ptx::cluster_sync_all();                                // every partial tile is in shared memory

  // rows [r0, r1) of the tile: sum the partials of ranks 0, 1, ... in order, scale, store bf16
  const int rows_per = kTM / splits;
  const int r0 = rank_in * rows_per, r1 = rank_in == splits - 1 ? kTM : r0 + rows_per;
  const float c_slot = pool.slot_scale[slot];
  const int rank = pool.slot_rank[slot];
  for (int e = threadIdx.x; e < (r1 - r0) * (kR / 4); e += kThreads) {
    const int row = r0 + e / (kR / 4), q4 = (e % (kR / 4)) * 4;
    const uint32_t off = static_cast<uint32_t>((row * kPartLd + q4) * 4);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int src = 0; src < splits; ++src) {
      const float4 v = ptx::ld_dsmem_f4(ptx::mapa_shared(ptx::smem_u32(part), static_cast<uint32_t>(src)) + off);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    const int t = tile * kTM + row;
    float coef = 0.f;
    if (t < m.T) {
      for (int j = 0; j < m.J; ++j) {
        const int p = t * m.J + j;
        if (m.pair_slot[p] == slot) coef += m.pair_scale[p] * c_slot;
      }
    }
    const float a0 = q4 < rank ? coef * acc.x : 0.f, a1 = q4 + 1 < rank ? coef * acc.y : 0.f;
    const float a2 = q4 + 2 < rank ? coef * acc.z : 0.f, a3 = q4 + 3 < rank ? coef * acc.w : 0.f;
    const __nv_bfloat162 lo = __floats2bfloat162_rn(a0, a1), hi = __floats2bfloat162_rn(a2, a3);
    uint16_t* dst = m.vtile + ((static_cast<size_t>(tile) * kTileSlots + k) * kTM + row) * kR + q4;
    *reinterpret_cast<uint2*>(dst) =
        make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
  }
  ptx::cluster_sync_all();                                // no CTA leaves while others read its tile
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, kR);
  }
}

}  // namespace

bool sgmv_tc_supported(int R) { return R == kR; }

cudaError_t launch_sgmv_shrink_tc(const uint16_t* x, const PoolView& pool, const MetaView& m, uint32_t* err,
                                  int num_sms, cudaStream_t s) {
  if (m.T == 0 || !sgmv_tc_supported(pool.R)) return cudaSuccess;
  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(sgmv_shrink_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  CUtensorMap mx, ma;
  if (!make_tmap_bf16(&mx, x, m.T, pool.K, kTM, kBK) ||
      !make_tmap_bf16(&ma, pool.A, static_cast<long>(pool.S) * pool.R, pool.K, kR, kBK))
    return cudaErrorInvalidValue;
  const int n_tiles = (m.T + kTM - 1) / kTM;
  // K splits: enough clusters of work for every SM when each tile uses about one slot
  const int num_kb = (pool.K + kBK - 1) / kBK;
  int splits = num_sms / n_tiles;
  if (splits > kMaxSplits) splits = kMaxSplits;
  if (splits > num_kb) splits = num_kb;
  if (splits < 1) splits = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_tiles * kTileSlots * splits, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = splits;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  note_launch_begin(kKindShrink, s);
  cudaError_t e = cudaLaunchKernelEx(&cfg, sgmv_shrink_tc_kernel, mx, ma, pool, m, splits, err);
  note_launch_end(kKindShrink, s);
  return e;
}

}  // namespace mlora
