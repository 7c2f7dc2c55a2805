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
constexpr int kBlockCols = 64;         // columns of the slot space per extra K block (one 128-byte row)
constexpr int kMaxTileUnits = 256;     // (M-tile, column block) units of one M-tile on the tensor cores
constexpr int kMaxUnits = 16384;       // units of one step on the tensor cores (v tiles of 16 KB each)
constexpr int kGroupUnits = 4;         // pair-tile entries shrunk together (MMA N = 64 per entry)

// Columns a slot of maximum rank r owns: 8, 16, 32 or 64, or a multiple of 64 above that, so that
// with each class starting on a multiple of min(width, 64) no slot straddles two 64-column blocks.
__host__ __device__ constexpr int slot_width(int r) {
  return r <= 8 ? 8 : r <= 16 ? 16 : r <= 32 ? 32 : r <= 64 ? 64 : (r + 63) / 64 * 64;
}

// Device arrays of one adapter pool (one adapted linear). The slots' rank rows form one column
// space of C columns: slot s owns columns off_s .. off_s + width_s - 1 (width = slot_width of its
// class's maximum rank); A holds row c of that space for every column c, B holds column c.
struct PoolView {
  const uint16_t* A;        // [C, K] bf16: slot s row q at A + (off_s + q) * K
  const uint16_t* B;        // [D, C] bf16: slot s row o at B + o * C + off_s
  const float* slot_scale;  // [S] alpha/r or alpha/sqrt(r)
  const int32_t* slot_rank; // [S] true rank, 0 = empty slot
  const int32_t* slot_off;  // [S] first column of the slot
  const int32_t* slot_width;// [S] columns of the slot
  const int32_t* col_slot;  // [C] slot owning each column (-1: a gap between classes)
  int S, R, C, K, D;        // R = the widest slot; with one rank class every slot is R wide (off_s = s R)
  int uniform;              // 1: one rank class
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
                        //     n_act (distinct slots with an active pair), n_todo (entries of todo_blk),
                        //     n_units, n_groups (tensor-core side path, below)
  int32_t* pair_act;    // [n] index of the pair's slot among the active slots (-1: none)
  int32_t* act_slot;    // [n] active slots in ascending order
  uint32_t* err;        // device error word (ptx::kErr* bits)
  float* vpart;         // shrink output: [n_splits][n][R] fp32 partial sums of A x per K split
  float* vfull;         // small-batch shrink output: [T][act][R] fp32, row stride vfull_ld floats
  int vfull_ld;
  // Tensor-core side path. A unit is an (M-tile of 128 tokens, 64-column block of the slot space)
  // with at least one active pair of the tile owning a column of the block; units are numbered
  // tile by tile, blocks ascending. An M-tile with more than kMaxTileUnits units, or whose units do
  // not fit in the unit capacity, overflows: its pairs take the CUDA-core kernels.
  int32_t* tile_unit_off; // [tiles + 1] units of tile i: [tile_unit_off[i], tile_unit_off[i + 1])
  int32_t* unit_blk;      // [U] column block of each unit
  int32_t* unit_tile;     // [U] M-tile of each unit
  int32_t* grp_mp;        // [U] shrink groups: pair tile of the group
  int32_t* grp_ent;       // [U]   first pair-tile entry (kGroupUnits consecutive entries of one pair tile)
  int32_t* grp_cnt;       // [U]   entries in the group
  int32_t* ptile_off;     // [pair tiles + 1] entries of pair tile mp (M-tiles 2mp, 2mp + 1), the union
                          //   of both tiles' units by block
  int32_t* pent_blk;      // [U] column block of each pair-tile entry (ascending within a pair tile)
  int32_t* pent_u0;       // [U] unit of M-tile 2mp with that block (-1: none)
  int32_t* pent_u1;       // [U] unit of M-tile 2mp + 1 with that block (-1: none)
  int32_t* ptile_order;   // [pair tiles] pair tiles by entry count, most first (ties ascending)
  uint32_t* sync;         // [2 + pair tiles] the pair GEMM's counters: [0] next tile ticket, [1] clusters
                          //   done, [2 + mp] shrink sub-tiles of pair tile mp written (one per epilogue
                          //   warp); zero between launches (the last cluster of a launch resets them)
  int32_t* pair_fused;    // [n] 1: the pair's side path runs on the tensor cores inside the GEMM
  int32_t* todo_blk;      // [n] ascending pair-block numbers holding a pair with pair_fused == 0
  uint16_t* vtile;        // [U][128][64] bf16: s c v of the unit's tokens on the block's columns
  int unit_cap;           // U
  int n;                  // pairs of the current step (T * J)
  int T, J;
};

// Small batches fold the shrink into the skinny GEMM (v of every token against every active
// slot, written to MetaView::vfull); the workspace covers these sizes.
constexpr int kVfullMaxTokens = 256;
constexpr int kVfullMaxAct = 512;

// Kernel kinds for the launch counter and the optional per-kernel event trace.
enum KernelKind : int {
  kKindMeta = 0, kKindGemm = 1, kKindShrink = 2, kKindExpand = 3, kKindSlot = 4, kKindEmbed = 5, kNumKinds = 6
};

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
// The step's metadata: sorted pairs, segments, pair-blocks, active slots and, for the tensor-core
// side path, the units of each M-tile over the pool's column blocks.
// mode kMetaSortOnly: the sort, segments, pair-blocks and active slots (every path needs them);
// kMetaUnitsOnly: the tensor-core side path's units, pair-tile entries and groups of the step
// whose sort ran earlier (token_slots and scales are not read); kMetaAll: both.
constexpr int kMetaAll = 0, kMetaSortOnly = 1, kMetaUnitsOnly = 2;
cudaError_t launch_build_meta(const int32_t* token_slots, const float* scales, int T, int J, const PoolView& pool,
                              const MetaView& m, cudaStream_t s, int mode = kMetaAll);

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

// Tensor-core shrink (shrink_tc.cu): vtile of every unit, i.e. for each (M-tile, column block)
// the tile's x rows times the block's A rows, masked to each token's own slots and scaled.
cudaError_t launch_lora_shrink_tc(const uint16_t* x, const PoolView& pool, const MetaView& m, uint32_t* err,
                                  int num_sms, cudaStream_t s);
// Tiled base GEMM; with pool and meta it also adds vtile x B^T as one extra K block per unit of
// each M-tile (the expand inside the accumulator).
cudaError_t launch_base_gemm_lora(const uint16_t* x, const uint16_t* W, float* y, int T, int K, int D,
                                  uint32_t* err, int num_sms, const PoolView* pool, const MetaView* meta,
                                  cudaStream_t s);
// One block waiting on an mbarrier nothing arrives on (wait_check.cu): exercises the bounded
// wait, which sets ptx::kErrWaitTimeout in *err after the limit and returns.
cudaError_t launch_wait_check(uint32_t* err, cudaStream_t s);

// CTA-pair (cta_group::2) tiled GEMM for large batches (gemm_pair.cu): 256 x 256 tiles of y on
// clusters of two CTAs, with the side path's K blocks of both M-tiles of a pair tile.
// pair_gemm_max_pairs() = clusters of two that can be resident at once (0: not available).
// pair_gemm_pick_n() = the N tile (256, 224, 192 or 128) that best fills whole waves; bn = 0 in
// launch_pair_gemm picks it. gemm_tile_n() is the process-wide choice set by
// mlora_set_gemm_tile_n (0 automatic, -1 never the pair kernel, else that N tile).
int pair_gemm_max_pairs();
// Form of the small-batch GEMM set by mlora_set_skinny_form (0 and 1 split-K, 2 token-split).
int skinny_form();
// Whether launch_base_gemm_lora takes the CTA-pair kernel for a batch of T tokens, and whether
// that kernel then also computes the shrink of the tensor-core side path (as tiles of its own
// schedule) for inputs of width K.
bool base_gemm_uses_pair(int T);
bool pair_gemm_fuses_shrink(int K);
int pair_gemm_pick_n(int T, int D, int max_pairs, bool dynamic);
cudaError_t launch_pair_gemm(const uint16_t* x, const uint16_t* W, float* y, int T, int K, int D, uint32_t* err,
                             const PoolView* pool, const MetaView* meta, int bn, cudaStream_t s);
int gemm_tile_n();

// K elements per shrink split and the number of splits for a pool of width R.
void shrink_split(int K, int R, int* kc_len, int* n_ks);
// CUDA-core shrink / expand; with skip_fused they leave out the pairs the tensor-core path handles.
cudaError_t launch_lora_shrink(const uint16_t* x, const PoolView& pool, const MetaView& m, int num_sms,
                               cudaStream_t s, bool skip_fused = false);
cudaError_t launch_lora_expand(float* y, const PoolView& pool, const MetaView& m, int num_sms, cudaStream_t s,
                               bool skip_fused = false);

// Embedding lookup with LoRA (embedding.cu) over an embedding pool (A stored token-major as
// A^T [V, C] in PoolView::A, V in PoolView::K): y[t] = E[ids[t]] + sum_j s c B A[:, ids[t]].
cudaError_t launch_embedding(const int32_t* ids, const uint16_t* E, float* y, const PoolView& pool, const MetaView& m,
                             int num_sms, cudaStream_t s);
// Writes columns off .. off + width - 1 of A^T [V, C] from an adapter's A [r, V] staged whole
// (zeros past the rank; r = 0 clears them).
cudaError_t launch_scatter_slot_at(uint16_t* At, int C, int off, int width, int V, const uint16_t* stage, int r,
                                   cudaStream_t s);

}  // namespace mlora
