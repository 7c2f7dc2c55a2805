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
// Design: one CTA per (tile, slot): warp 0 issues TMA loads of a 128 x 64 x tile and a 64 x 64
// A tile per stage, warp 1 issues tcgen05.mma from one thread, warps 2..5 read the accumulator
// (one token row per thread) and write the scaled bf16 row. Waits are bounded (2 s).
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
constexpr int kSmemBytes = kStages * kStageBytes + 256 + 1024;

__global__ void __launch_bounds__(kThreads, 1)
sgmv_shrink_tc_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_a,
                      PoolView pool, MetaView m, uint32_t* __restrict__ err) {
  const int tile = blockIdx.x / kTileSlots, k = blockIdx.x % kTileSlots;
  const int32_t* info = m.tile_info + tile * (kTileSlots + 1);
  const int cnt = info[0];
  if (cnt > kTileSlots || k >= cnt) return;               // overflow tile or unused list entry
  const int slot = info[1 + k];

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  uint64_t* empty = full + kStages;
  uint64_t* acc_full = empty + kStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = pool.K;
  const int num_kb = (K + kBK - 1) / kBK;

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
      for (int kb = 0; kb < num_kb; ++kb) {
        if (!ptx::mbar_wait(&empty[stage], phase ^ 1u, err)) break;
        uint8_t* sx = smem + stage * kStageBytes;
        ptx::mbar_arrive_expect_tx(&full[stage], kStageBytes);
        ptx::tma_load_2d(sx, &tmap_x, &full[stage], kb * kBK, tile * kTM);
        ptx::tma_load_2d(sx + kXBytes, &tmap_a, &full[stage], kb * kBK, slot * kR);
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(kTM, kR);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int kb = 0; kb < num_kb; ++kb) {
        if (!ptx::mbar_wait(&full[stage], phase, err)) { ok = false; break; }
        ptx::tc_fence_after();
        const uint32_t x_addr = ptx::smem_u32(smem + stage * kStageBytes);
        const uint64_t x_desc = ptx::sw128_kmajor_desc(x_addr);
        const uint64_t a_desc = ptx::sw128_kmajor_desc(x_addr + kXBytes);
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk)
          ptx::umma_bf16(tmem_base, x_desc + 2u * kk, a_desc + 2u * kk, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
        ptx::umma_commit(&empty[stage]);
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      }
      if (ok) ptx::umma_commit(acc_full);
    }
  } else {
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int t = tile * kTM + row;
    if (ptx::mbar_wait(acc_full, 0, err)) {
      ptx::tc_fence_after();
      float coef = 0.f;
      if (t < m.T) {
        const float c = pool.slot_scale[slot];
        for (int j = 0; j < m.J; ++j) {
          const int p = t * m.J + j;
          if (m.pair_slot[p] == slot) coef += m.pair_scale[p] * c;
        }
      }
      const int rank = pool.slot_rank[slot];
      uint16_t* dst = m.vtile + ((static_cast<size_t>(tile) * kTileSlots + k) * kTM + row) * kR;
#pragma unroll
      for (int c0 = 0; c0 < kR; c0 += 32) {
        uint32_t r[32];
        ptx::tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(c0), r);
        ptx::tmem_ld_wait();
        uint32_t packed[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int q = c0 + 2 * i;
          const float a = q < rank ? coef * __uint_as_float(r[2 * i]) : 0.f;
          const float b = q + 1 < rank ? coef * __uint_as_float(r[2 * i + 1]) : 0.f;
          const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
          packed[i] = *reinterpret_cast<const uint32_t*>(&h);
        }
        uint4* d4 = reinterpret_cast<uint4*>(dst + c0);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          d4[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
      }
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, kR);
  }
}

}  // namespace

bool sgmv_tc_supported(int R) { return R == kR; }

cudaError_t launch_sgmv_shrink_tc(const uint16_t* x, const PoolView& pool, const MetaView& m, uint32_t* err,
                                  cudaStream_t s) {
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
  note_launch_begin(kKindShrink, s);
  sgmv_shrink_tc_kernel<<<n_tiles * kTileSlots, kThreads, kSmemBytes, s>>>(mx, ma, pool, m, err);
  cudaError_t e = cudaGetLastError();
  note_launch_end(kKindShrink, s);
  return e;
}

}  // namespace mlora
