// Declarations shared by the library's translation units (host launchers and the
// device-side views of the pool and the per-step metadata). Not part of the C ABI.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace mlora {

constexpr int kMaxSlots = 2048;     // pool slots (GPU-resident adapters)
constexpr int kMaxRank = 256;       // r_max
constexpr int kMaxJ = 8;            // adapter slots per token
constexpr int kPairBlock = 16;      // pairs of one slot handled together by the shrink
constexpr int kMetaThreads = 1024;
constexpr int kMaxShrinkSplits = 16;   // K splits of the shrink (partial sums per split)
constexpr int kMaxTiles = 512;         // 128-token M-tiles of a step (65535 tokens)
constexpr int kTileSlots = 4;          // slots per M-tile handled on the tensor cores

// Device arrays of one adapter pool (one adapted linear).
struct PoolView {
  const uint16_t* A;        // [S, R, K] bf16, slot s row q at A + (s*R + q)*K
  const uint16_t* B;        // [S, D, R] bf16, slot s row o at B + (s*D + o)*R
  const float* slot_scale;  // [S] alpha/r or alpha/sqrt(r)
  const int32_t* slot_rank; // [S] true rank, 0 = empty slot
  int S, R, K, D;
};

// Device arrays of one step's metadata (see build_meta_kernel for the contents).
struct MetaView {
  int32_t* order;       // [n] pair indices p = t*J + j, stably sorted by slot (-1 first)
  int32_t* seg_slot;    // [n + 1] slot of each segment, ascending (-1 first if present)
  int32_t* seg_off;     // [n + 2] segment offsets into order, n_seg + 1 entries
  int32_t* pair_slot;   // [n] validated slot per pair (-1: sentinel or rejected)
  float* pair_scale;    // [n] per-pair scale (0 where pair_slot == -1)
  int32_t* blk_slot;    // [n] pair-blocks of at most kPairBlock pairs of one slot
  int32_t* blk_start;   // [n]   start of the block inside order
  int32_t* blk_count;   // [n]   pairs in the block
  int32_t* counts;      // [8] n_seg, n_active, n_blocks, first rejected pair (INT32_MAX if none),
                        //     n_act (distinct slots with an active pair), n_todo (entries of todo_blk)
  int32_t* pair_act;    // [n] index of the pair's slot among the active slots (-1: none)
  int32_t* act_slot;    // [n] active slots in ascending order
  uint32_t* err;        // device error word (ptx::kErr* bits)
  float* vpart;         // shrink output: [n_splits][n][R] fp32 partial sums of A x per K split
  float* vfull;         // small-batch shrink output: [T][act][R] fp32, row stride vfull_ld floats
  int vfull_ld;
  int32_t* tile_info;   // per 128-token M-tile: [count, slot_0 .. slot_{kTileSlots-1}] (ascending,
                        //   -1 unused); count > kTileSlots = too many slots (overflow tile)
  int32_t* pair_fused;  // [n] 1: the pair's side path runs on the tensor cores inside the GEMM
  int32_t* todo_blk;    // [n] ascending pair-block numbers holding a pair with pair_fused == 0
  uint16_t* vtile;      // tensor-core shrink output: [tiles][kTileSlots][128][64] bf16, s c v per token
  int n;                // pairs of the current step (T * J)
  int T, J;
};

// Small batches fold the shrink into the skinny GEMM (v of every token against every active
// slot, written to MetaView::vfull); the workspace covers these sizes.
constexpr int kVfullMaxTokens = 256;
constexpr int kVfullMaxAct = 512;

// Kernel kinds for the launch counter and the optional per-kernel event trace.
enum KernelKind : int { kKindMeta = 0, kKindGemm = 1, kKindShrink = 2, kKindExpand = 3, kKindSlot = 4, kNumKinds = 5 };

// Records the thread's last-error message and returns the status (mlora_runtime.cu).
int report_error(int status, const char* message);
int report_cuda_error(cudaError_t e, const char* what);

// Launch counter + tracing hooks (mlora_runtime.cu).
void note_launch_begin(int kind, cudaStream_t s);
void note_launch_end(int kind, cudaStream_t s);

// Row-major bf16 matrix [rows, cols] as a TMA tensor map with a box of box_rows x box_cols and
// the 128-byte swizzle (gemm_tc.cu). False if the encoder is unavailable or rejects it.
bool make_tmap_bf16(CUtensorMap* map, const void* base, long rows, int cols, int box_rows, int box_cols);
// Row-major fp32 matrix [rows, cols] with a box of box_rows x 32 columns (128 bytes, 128-byte
// swizzle), for tiled stores. False unless cols is a multiple of 4 and base 16-byte aligned.
bool make_tmap_f32_sw128(CUtensorMap* map, const void* base, long rows, int cols, int box_rows);

// Launchers. Each returns the cudaError_t of its launch.
cudaError_t launch_build_meta(const int32_t* token_slots, const float* scales, int T, int J, int S,
                              const int32_t* slot_rank, const MetaView& m, cudaStream_t s);

// y[T, D] (fp32) = x[T, K] (bf16, row-major) * W[D, K]^T (bf16, row-major), tcgen05 path.
cudaError_t launch_base_gemm(const uint16_t* x, const uint16_t* W, float* y, int T, int K, int D,
                             uint32_t* err, int num_sms, cudaStream_t s);

constexpr int kSkinnyMaxT = 256;   // batches up to this size use the split-K skinny GEMM

// Whether the skinny GEMM can compute the shrink alongside the base product for this step.
bool skinny_shrink_fusable(int T, int J, int S, int R, int vfull_ld);
// y = x W^T and vfull[t][a][q] = sum_i A_{act_slot[a]}[q][i] x[t][i] in one split-K tensor-core
// kernel (T <= kSkinnyMaxT).
cudaError_t launch_gemm_shrink_fused(const uint16_t* x, const uint16_t* W, float* y, const PoolView& pool,
                                     const MetaView& m, uint32_t* err, int num_sms, cudaStream_t s);
// y += sum_j s c B v with v from vfull; programmatic dependent launch after the fused GEMM.
cudaError_t launch_lora_expand_vfull(float* y, const PoolView& pool, const MetaView& m, int num_sms,
                                     cudaStream_t s);

// Overflow window of a large batch (T > kSkinnyMaxT): when the step has one or two 128-token tiles
// with more than kTileSlots slots (the metadata names them in counts[6], counts[7]; counts[6] is
// -1 otherwise), their pairs take the small-batch machinery: the skinny kernel in shrink-only
// mode over those 256 token rows (vfull row w = window row), then the vfull expand restricted to
// the pairs not handled on the tensor cores. Both kernels do nothing when there is no window.
bool window_shrink_supported(int T, int J, int S, int R, int vfull_ld, int vfull_rows);
cudaError_t launch_gemm_shrink_window(const uint16_t* x, const PoolView& pool, const MetaView& m, uint32_t* err,
                                      int num_sms, cudaStream_t s);
cudaError_t launch_lora_expand_window(float* y, const PoolView& pool, const MetaView& m, int num_sms,
                                      cudaStream_t s);

// Tensor-core prefill path (sgmv_tc.cu): pools with padded rank R == 64.
bool sgmv_tc_supported(int R);
// vtile = scaled (x A_slot^T) per (M-tile, slot) for tiles with at most kTileSlots slots.
cudaError_t launch_sgmv_shrink_tc(const uint16_t* x, const PoolView& pool, const MetaView& m, uint32_t* err,
                                  int num_sms, cudaStream_t s);
// Tiled base GEMM; with pool and meta it also adds vtile x B_slot^T as extra K blocks of the
// fused tiles.
cudaError_t launch_base_gemm_lora(const uint16_t* x, const uint16_t* W, float* y, int T, int K, int D,
                                  uint32_t* err, int num_sms, const PoolView* pool, const MetaView* meta,
                                  cudaStream_t s);
// One block waiting on an mbarrier nothing arrives on (wait_check.cu): exercises the bounded
// wait, which sets ptx::kErrWaitTimeout in *err after the limit and returns.
cudaError_t launch_wait_check(uint32_t* err, cudaStream_t s);

// CTA-pair (cta_group::2) tiled GEMM for large batches (gemm_pair.cu): 256 x 256 tiles of y on
// clusters of two CTAs, with the same fused side-path K blocks as the one-CTA tiled GEMM.
// pair_gemm_max_pairs() = clusters of two that can be resident at once (0: not available).
// pair_gemm_pick_n() = the N tile (256, 224, 192 or 128) that best fills whole waves; bn = 0 in
// launch_pair_gemm picks it. gemm_tile_n() is the process-wide choice set by
// mlora_set_gemm_tile_n (0 automatic, -1 never the pair kernel, else that N tile).
int pair_gemm_max_pairs();
int pair_gemm_pick_n(int T, int D, int max_pairs);
cudaError_t launch_pair_gemm(const uint16_t* x, const uint16_t* W, float* y, int T, int K, int D, uint32_t* err,
                             const PoolView* pool, const MetaView* meta, int bn, cudaStream_t s);
int gemm_tile_n();

// K elements per shrink split and the number of splits for a pool of width R.
void shrink_split(int K, int R, int* kc_len, int* n_ks);
// CUDA-core shrink / expand; with skip_fused they leave out the pairs the tensor-core path handles,
// and with window they also do nothing when the overflow-window kernels took the step's
// remaining pairs (counts[6] >= 0).
cudaError_t launch_lora_shrink(const uint16_t* x, const PoolView& pool, const MetaView& m, int num_sms,
                               cudaStream_t s, bool skip_fused = false, bool window = false);
cudaError_t launch_lora_expand(float* y, const PoolView& pool, const MetaView& m, int num_sms, cudaStream_t s,
                               bool skip_fused = false, bool window = false);

}  // namespace mlora
