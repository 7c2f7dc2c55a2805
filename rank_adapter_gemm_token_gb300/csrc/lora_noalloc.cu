// The LoRA side path for callers that cannot allocate device memory.
//
// mlora_lora_apply_noalloc adds y += sum_j s c B_slot (A_slot x) using only memory the caller
// passes in plus one fixed workspace compiled into this library: a file-scope __device__ array
// that every GPU loading the library holds until the process exits. It is meant for callers
// such as a serving engine that hands all free device memory to its KV cache at start-up (a
// later cudaMalloc would fail), or code on a latency-critical path where the implicit device
// synchronisation of cudaMalloc/cudaFree is not acceptable. Nothing here calls cudaMalloc,
// cudaFree or any allocating routine.
//
// Two kernels: a gather shrink (one pair per block, whole K per adapter row, v written to the
// workspace) and a token-major expand that adds a token's slots in order j = 0..J-1.
#include <climits>
#include <cmath>
#include <cstdio>
#include <mutex>

#include "internal.h"
#include "mlora.h"
#include "ptx.cuh"

namespace mlora {
namespace {

// Workspace of the unscaled shrink output v, [T*J][R] fp32: 2^20 floats (4 MiB).
constexpr size_t kNoallocVFloats = size_t(1) << 20;
__device__ __align__(256) float g_noalloc_v[kNoallocVFloats];

constexpr int kNoallocThreads = 256;
constexpr int kNoallocCols = 512;          // output columns per expand block

// Device address of g_noalloc_v per device ordinal. In host code the symbol's name is only a
// host-side stand-in, so the address is looked up with that device current (on every call made
// outside stream capture) and kept here for calls made inside one.
float* g_noalloc_v_addr[64] = {};
std::mutex g_noalloc_mu;

__device__ __forceinline__ float nd_dot8(const uint4& a, const uint4& b) {
  float s = ptx::bf16_lo(a.x) * ptx::bf16_lo(b.x);
  s = fmaf(ptx::bf16_hi(a.x), ptx::bf16_hi(b.x), s);
  s = fmaf(ptx::bf16_lo(a.y), ptx::bf16_lo(b.y), s);
  s = fmaf(ptx::bf16_hi(a.y), ptx::bf16_hi(b.y), s);
  s = fmaf(ptx::bf16_lo(a.z), ptx::bf16_lo(b.z), s);
  s = fmaf(ptx::bf16_hi(a.z), ptx::bf16_hi(b.z), s);
  s = fmaf(ptx::bf16_lo(a.w), ptx::bf16_lo(b.w), s);
  s = fmaf(ptx::bf16_hi(a.w), ptx::bf16_hi(b.w), s);
  return s;
}

// A pair's slot if it names a slot in [0, S) whose rank is in [1, R], else -1 (adds nothing).
__device__ __forceinline__ int checked_slot(const int32_t* token_slots, const int32_t* slot_rank, int p, int S,
                                            int R) {
  const int s = token_slots[p];
  if (s < 0 || s >= S) return -1;
  const int r = slot_rank[s];
  return (r > 0 && r <= R) ? s : -1;
}

// One block per (token, slot) pair: warp w computes rows q = w, w + 8, ... of v = A_slot x_t over
// the whole K range (16-byte loads, warp-shuffle sum) and writes them to the workspace.
__global__ void __launch_bounds__(kNoallocThreads)
noalloc_shrink_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ token_slots,
                      const uint16_t* __restrict__ A_pool, const int32_t* __restrict__ slot_rank, int S, int R,
                      int K, int J, int n, float* __restrict__ v) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int p = blockIdx.x; p < n; p += gridDim.x) {
    const int s = checked_slot(token_slots, slot_rank, p, S, R);
    if (s < 0) continue;
    const int rank = slot_rank[s];
    const uint4* xv = reinterpret_cast<const uint4*>(x + static_cast<size_t>(p / J) * K);
    for (int q = warp; q < rank; q += kNoallocThreads / 32) {
      const uint4* av = reinterpret_cast<const uint4*>(A_pool + (static_cast<size_t>(s) * R + q) * K);
      float acc = 0.f;
      for (int u = lane; u < K / 8; u += 32) acc += nd_dot8(__ldg(av + u), __ldg(xv + u));
#pragma unroll
      for (int d = 16; d > 0; d >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, d);
      if (lane == 0) v[static_cast<size_t>(p) * R + q] = acc;
    }
  }
}

// One block per (token, 512 output columns): y[t][o] += sum_j s c sum_q B[o][q] v[q], j in order.
__global__ void __launch_bounds__(kNoallocThreads)
noalloc_expand_kernel(float* __restrict__ y, const int32_t* __restrict__ token_slots, const float* __restrict__ scales,
                      const uint16_t* __restrict__ B_pool, const float* __restrict__ slot_scale,
                      const int32_t* __restrict__ slot_rank, int S, int R, int D, int J, int T, int n_dchunk,
                      const float* __restrict__ v) {
  __shared__ __align__(16) float vs[kMaxJ][kMaxRank];
  __shared__ int ss[kMaxJ], rs[kMaxJ];
  const int items = T * n_dchunk;                       // checked to fit an int by the host
  for (int item = blockIdx.x; item < items; item += gridDim.x) {
    const int t = item / n_dchunk, dc = item - t * n_dchunk;
    __syncthreads();
    if (threadIdx.x < J) {
      const int p = t * J + threadIdx.x;
      const int s = checked_slot(token_slots, slot_rank, p, S, R);
      ss[threadIdx.x] = s;
      rs[threadIdx.x] = s >= 0 ? slot_rank[s] : 0;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < J * R; i += kNoallocThreads) {
      const int j = i / R, q = i - j * R;
      const int s = ss[j];
      float val = 0.f;
      if (s >= 0 && q < rs[j]) {
        const int p = t * J + j;
        const float coef = (scales ? scales[p] : 1.0f) * slot_scale[s];
        val = coef * v[static_cast<size_t>(p) * R + q];
      }
      vs[j][q] = val;
    }
    __syncthreads();
    const int oa = dc * kNoallocCols, ob = min(D, oa + kNoallocCols);
    for (int o = oa + threadIdx.x; o < ob; o += kNoallocThreads) {
      float acc = y[static_cast<size_t>(t) * D + o];
      for (int j = 0; j < J; ++j) {
        const int s = ss[j];
        if (s < 0) continue;
        const uint4* brow = reinterpret_cast<const uint4*>(B_pool + (static_cast<size_t>(s) * D + o) * R);
        float d = 0.f;
        for (int u = 0; u < (rs[j] + 7) / 8; ++u) {
          const uint4 bv = __ldg(brow + u);
          const float* w = &vs[j][8 * u];
          d = fmaf(ptx::bf16_lo(bv.x), w[0], d);
          d = fmaf(ptx::bf16_hi(bv.x), w[1], d);
          d = fmaf(ptx::bf16_lo(bv.y), w[2], d);
          d = fmaf(ptx::bf16_hi(bv.y), w[3], d);
          d = fmaf(ptx::bf16_lo(bv.z), w[4], d);
          d = fmaf(ptx::bf16_hi(bv.z), w[5], d);
          d = fmaf(ptx::bf16_lo(bv.w), w[6], d);
          d = fmaf(ptx::bf16_hi(bv.w), w[7], d);
        }
        acc += d;
      }
      y[static_cast<size_t>(t) * D + o] = acc;
    }
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace mlora

using namespace mlora;

extern "C" mlora_status mlora_lora_apply_noalloc(const mlora_bf16* x, float* y, const int32_t* token_slots,
                                                 const float* scales, int T, int J, const mlora_bf16* A_pool,
                                                 const mlora_bf16* B_pool, const float* slot_scale,
                                                 const int32_t* slot_rank, int n_slots, int r_pad, int K, int D,
                                                 void* stream) {
  if (T < 0 || J < 1 || J > MLORA_MAX_SLOTS_PER_TOKEN)
    return report_error(MLORA_ERR_INVALID_ARG, "T must be >= 0 and J in [1, 8]");
  if (n_slots < 1 || r_pad < 8 || r_pad > MLORA_MAX_RANK || r_pad % 8 != 0 || K < 8 || K % 8 != 0 || D < 1)
    return report_error(MLORA_ERR_INVALID_ARG,
                        "n_slots >= 1, r_pad a multiple of 8 in [8, 256], K a positive multiple of 8, D >= 1");
  if (T == 0) return MLORA_OK;
  if (!x || !y || !token_slots || !A_pool || !B_pool || !slot_scale || !slot_rank)
    return report_error(MLORA_ERR_INVALID_ARG, "a required pointer is NULL");
  if (!aligned16(x) || !aligned16(A_pool) || !aligned16(B_pool))
    return report_error(MLORA_ERR_INVALID_ARG, "x, A_pool and B_pool must be 16-byte aligned");
  const size_t need = static_cast<size_t>(T) * J * r_pad;
  if (need > kNoallocVFloats) {
    char msg[200];
    snprintf(msg, sizeof msg, "T*J*r_pad = %zu exceeds the built-in workspace of %zu floats", need,
             kNoallocVFloats);
    return report_error(MLORA_ERR_TOO_MANY_TOKENS, msg);
  }
  const size_t n_dchunk = (static_cast<size_t>(D) + kNoallocCols - 1) / kNoallocCols;
  if (static_cast<size_t>(T) * n_dchunk > static_cast<size_t>(INT_MAX))
    return report_error(MLORA_ERR_INVALID_ARG, "T * ceil(D / 512) must fit in an int");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return report_cuda_error(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return report_error(MLORA_ERR_INVALID_ARG, "device ordinal unsupported");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* v = nullptr;
  {
    // outside a capture the address is looked up again (it changes when the device's context is
    // re-created, e.g. after cudaDeviceReset); inside one the kept address is used
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) {
      cudaGetLastError();
      cap = cudaStreamCaptureStatusActive;
    }
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (cap == cudaStreamCaptureStatusNone || !g_noalloc_v_addr[dev]) {
      if (cap != cudaStreamCaptureStatusNone)
        return report_error(MLORA_ERR_INVALID_ARG,
                            "the first call on a device must come before any stream capture (workspace address)");
      void* addr = nullptr;
      e = cudaGetSymbolAddress(&addr, g_noalloc_v);
      if (e != cudaSuccess) return report_cuda_error(e, "cudaGetSymbolAddress(workspace)");
      g_noalloc_v_addr[dev] = static_cast<float*>(addr);
    }
    v = g_noalloc_v_addr[dev];
  }
  int num_sms = 0;
  e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return report_cuda_error(e, "SM count");
  const int n = T * J;
  int grid = n < num_sms * 8 ? n : num_sms * 8;
  note_launch_begin(kKindShrink, s);
  noalloc_shrink_kernel<<<grid, kNoallocThreads, 0, s>>>(x, token_slots, A_pool, slot_rank, n_slots, r_pad, K, J, n,
                                                         v);
  e = cudaGetLastError();
  note_launch_end(kKindShrink, s);
  if (e != cudaSuccess) return report_cuda_error(e, "shrink launch");
  const int items = T * static_cast<int>(n_dchunk);
  grid = items < num_sms * 8 ? items : num_sms * 8;
  note_launch_begin(kKindExpand, s);
  noalloc_expand_kernel<<<grid, kNoallocThreads, 0, s>>>(y, token_slots, scales, B_pool, slot_scale, slot_rank,
                                                         n_slots, r_pad, D, J, T, static_cast<int>(n_dchunk), v);
  e = cudaGetLastError();
  note_launch_end(kKindExpand, s);
  if (e != cudaSuccess) return report_cuda_error(e, "expand launch");
  return MLORA_OK;
}
