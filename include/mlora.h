/*
 * mlora.h -- C ABI of a single-GPU (GB300, sm_103a) multi-LoRA batched linear layer.
 *
 * The layer (one adapted linear of a transformer) computes, for a mixed-tenant batch,
 *
 *     y[t, :] = x[t, :] W^T  +  sum_{j : slot[t,j] != -1}  s[t,j] * c(slot) * B_slot (A_slot x[t, :])
 *
 * with c = alpha / r, or alpha / sqrt(r) for rsLoRA adapters.
 * Sources:
 *   "Multi-LoRA Serving Explained" (sevydevy.com): LoRA basics (B is d x r, A is r x k,
 *     W x + (alpha/r) B(A x)); batched serving (one shared base product plus each token's
 *     side path, found through a GPU slot number, -1 = base model only); the stacked,
 *     zero-padded slot pool sized at the maximum rank; rejection of ranks above it.
 *   "[RFC] Per-request activation of multiple LoRA adapters" (vLLM issue 51940),
 *     Proposed Change: k adapters per request with per-adapter scales; a k-slot token map
 *     with unused slots holding the sentinel; a bound on adapters per request.
 *   "LoRA Serving" (vLLM learning book ch. 09-04), sections 4 and 6: slot activation copies
 *     an adapter's weights into a GPU slot; the per-step token -> slot mapping; shrink and
 *     expand.
 *   "[vLLM] LoRA" (secrett2633 blog), PEFTHelper: r, lora_alpha, use_rslora.
 *
 * Conventions
 *   - bf16 values are passed as their 16-bit patterns (mlora_bf16).
 *   - "device" pointers are CUDA global-memory pointers of the current device; "host"
 *     pointers are CPU memory (pinned memory gives asynchronous copies).
 *   - Streams are cudaStream_t values passed as void*; NULL means the legacy default stream.
 *   - Every call returns an mlora_status; MLORA_OK is 0. On failure mlora_last_error()
 *     gives a message for the calling thread. No call throws.
 *   - Errors of earlier asynchronous work surface as MLORA_ERR_CUDA on a later call.
 *   - Rows are contiguous (row-major); x rows hold K elements, W rows K, y rows D.
 *   - K must be a positive multiple of 8; x and W must be 16-byte aligned; y 16-byte aligned.
 */
#ifndef MLORA_H
#define MLORA_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MLORA_API __attribute__((visibility("default")))
#else
#define MLORA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef int mlora_status;
typedef uint16_t mlora_bf16;
typedef struct mlora_pool* mlora_pool_t;
typedef struct mlora_meta* mlora_meta_t;
typedef struct mlora_slot_cache* mlora_slot_cache_t;
typedef struct mlora_adapter_cache* mlora_adapter_cache_t;

enum {
  MLORA_OK = 0,
  MLORA_ERR_INVALID_ARG = 1,      /* null pointer, bad size, misaligned pointer             */
  MLORA_ERR_SLOT_RANGE = 2,       /* slot outside [0, n_slots)                              */
  MLORA_ERR_RANK_TOO_LARGE = 3,   /* adapter rank above the pool's r_max                    */
  MLORA_ERR_RANK_INVALID = 4,     /* rank < 1, or alpha not finite                           */
  MLORA_ERR_BAD_TOKEN_SLOT = 5,   /* a token named a slot outside [-1, n_slots) or an empty slot */
  MLORA_ERR_TOO_MANY_TOKENS = 6,  /* T or J above what the metadata object was created for  */
  MLORA_ERR_OOM = 7,              /* device or host allocation failed                       */
  MLORA_ERR_CUDA = 8,             /* a CUDA call failed (message has the CUDA error)         */
  MLORA_ERR_DEVICE_TIMEOUT = 9,   /* a kernel's bounded wait gave up (the GPU stays usable)  */
  MLORA_ERR_MISMATCH = 10,        /* pool and metadata or pool and operands do not fit     */
  MLORA_ERR_NO_FREE_SLOT = 11,    /* a step needs more adapters resident than slots allow  */
  MLORA_ERR_BAD_TOKEN_ID = 12     /* a token id outside [0, vocab) of an embedding table     */
};

/* Limits of this build. */
#define MLORA_MAX_SLOTS 2048
#define MLORA_MAX_RANK 256
#define MLORA_MAX_SLOTS_PER_TOKEN 8
#define MLORA_MAX_TOKENS 65535
#define MLORA_MAX_SLICES 8            /* output slices of one fused linear (mlora_load_adapter_sliced) */
#define MLORA_MAX_CLASSES 8           /* rank classes of one pool (mlora_pool_create_classes) */

/* ------------------------------------------------------------------ adapter pool ----- */

/* Creates the slot pool of one adapted linear (K inputs, D outputs), every slot sized for r_max
 * ("Multi-LoRA Serving Explained", max-lora-rank section: slots are zero blocks sized for the
 * maximum rank; a smaller adapter fills the top-left corner).
 * Layout: the slots' rank rows form one column space of C columns; slot s owns R columns
 * starting at off_s = s * R (C = n_slots * R), R = the slot width of r_max: 8, 16, 32 or 64 for
 * r_max up to 64, else r_max rounded up to a multiple of 64 (so no slot straddles a 64-column
 * block). A_pool [C, K] holds row
 * off_s + q of slot s's A (row q), B_pool [D, C] holds column off_s + q of slot s's B (column q),
 * both bf16 and zero beyond each adapter's rank; plus a per-slot factor c (fp32) and true rank.
 * A 64-column block of that space is what the tensor-core side path multiplies at once.
 * copy_stream: the stream adapter loads run on (NULL: the pool creates its own).
 * The pool allocates with cudaMalloc here and never on the hot path. */
MLORA_API mlora_status mlora_pool_create(int n_slots, int r_max, int K, int D, void* copy_stream, mlora_pool_t* out);

/* A pool whose slots come in rank classes ("Multi-LoRA Serving Explained", max-lora-rank
 * section: padding every slot to the largest rank wastes memory; "[vLLM] LoRA" (secrett2633
 * blog), S-LoRA section: adapters of different ranks served together from one memory pool).
 * Class c has class_slots[c] slots for adapters of rank at most class_rank[c]; slots are
 * numbered class by class (class 0 first) and slot i of class c owns w_c columns of the column
 * space, w_c = the slot width of class_rank[c] (as for mlora_pool_create), right after the
 * previous slot; each class starts on a multiple of min(w_c, 64) columns. So a rank-8 slot's B
 * row is 16 bytes and eight such slots share one 64-column block, and the pool holds
 * C * (K + D) * 2 bytes with C = the end of the last class (mlora_pool_layout).
 * n_classes in [1, MLORA_MAX_CLASSES], class_slots[c] >= 1 (at most MLORA_MAX_SLOTS in all),
 * class_rank[c] in [1, MLORA_MAX_RANK]; else MLORA_ERR_INVALID_ARG. Pools used with one metadata
 * object must have the same classes (MLORA_ERR_MISMATCH otherwise). mlora_pool_create(n, r, ...)
 * is this call with one class. */
MLORA_API mlora_status mlora_pool_create_classes(int n_classes, const int* class_slots, const int* class_rank, int K,
                                                 int D, void* copy_stream, mlora_pool_t* out);

/* The pool's column space: C, and per slot its first column and width (host arrays of n_slots
 * entries; any pointer may be NULL). */
MLORA_API mlora_status mlora_pool_layout(mlora_pool_t pool, int* C, int32_t* slot_off, int32_t* slot_width);

/* Waits for this pool's loads and uses to finish, then frees it. NULL is accepted. */
MLORA_API mlora_status mlora_pool_destroy(mlora_pool_t pool);

/* Copies one adapter into a slot ("LoRA Serving", section 4.1: activating an adapter copies its
 * weights into a free GPU slot; the caller chooses the slot and keeps the id -> slot map).
 *   A_host: [rank, K] bf16 row-major, B_host: [D, rank] bf16 row-major (host memory).
 *   rank <= the slot's maximum rank (r_max, or its class's rank; else MLORA_ERR_RANK_TOO_LARGE,
 *   message naming both ranks), alpha finite.
 *   rslora != 0 selects c = alpha / sqrt(rank), else c = alpha / rank.
 * Runs on the pool's copy stream after every mlora_linear already issued on this pool
 * (write-after-read ordering by event): the slot's A rows are zeroed and A is copied to rows
 * off_s .. off_s + rank - 1 of A_pool; B is copied whole into a staging buffer of the pool and a
 * kernel writes it to columns off_s .. off_s + R_s - 1 of B_pool (zeros past the rank). Returns
 * when the copies are queued; with pinned
 * host buffers they are asynchronous and the buffers must stay valid until
 * mlora_pool_sync() or the next mlora_linear on this pool has been ordered after them.
 * With pageable buffers the copy is complete on return. */
MLORA_API mlora_status mlora_load_adapter(mlora_pool_t pool, int slot, const mlora_bf16* A_host, const mlora_bf16* B_host,
                                int rank, float alpha, int rslora);

/* Per-slice adapter of a fused linear (qkv, gate_up): the D output columns are n_slices
 * consecutive slices of widths[i] columns (sum = D), and slice i has its own A_i [rank, K] and
 * B_i [widths[i], rank] (host bf16, row-major), all of one adapter config (rank, alpha, rslora):
 *   y[t, off_i .. off_i + widths[i]) += s c B_i (A_i x[t]),  c = alpha / rank (alpha / sqrt(rank)),
 * off_i = the sum of the earlier widths ("LoRA Serving" (vLLM learning book, ch. 09-04), section 7:
 * the merged QKV / merged column linear handles each sub-projection's adapter separately; "[vLLM]
 * LoRA" (secrett2633 blog), layer-implementation section: merged QKV / merged column variants). The slot stores it as one adapter of rank
 * n_slices * rank: A = [A_1; ...; A_n] and B block-diagonal (slice i's rows hold B_i in columns
 * i*rank .. and zeros elsewhere), with factor c; the layer kernels run unchanged and each output
 * slice gets exactly its own side path (the other blocks add exact zeros).
 * n_slices in [1, MLORA_MAX_SLICES], n_slices * rank <= r_max (else MLORA_ERR_RANK_TOO_LARGE),
 * widths > 0 and adding up to D (else MLORA_ERR_INVALID_ARG). Ordering, asynchrony and buffer
 * lifetime as for mlora_load_adapter. */
MLORA_API mlora_status mlora_load_adapter_sliced(mlora_pool_t pool, int slot, int n_slices, const int* widths,
                                                 const mlora_bf16* const* A_slices,
                                                 const mlora_bf16* const* B_slices, int rank, float alpha,
                                                 int rslora);


/* Zeroes a slot and marks it empty (tokens naming it are then rejected). */
MLORA_API mlora_status mlora_clear_slot(mlora_pool_t pool, int slot);

/* Blocks until every queued load of this pool has finished. */
MLORA_API mlora_status mlora_pool_sync(mlora_pool_t pool);

/* Device pointers and sizes of the pool (for inspection and tests; owned by the pool): r_pad is
 * the widest slot, A_pool is [C, K] and B_pool [D, C] (mlora_pool_layout gives C and the slots'
 * columns). */
MLORA_API mlora_status mlora_pool_info(mlora_pool_t pool, int* n_slots, int* r_pad, int* K, int* D, void** A_pool,
                             void** B_pool, void** slot_scale, void** slot_rank);

/* Bytes of device memory held by the A and B slots of mlora_pool_create's pool:
 * n_slots * R * (K + D) * 2 with R = the slot width of r_max ("Multi-LoRA Serving Explained",
 * memory maths: rank * (in + out) numbers per adapted layer, slots reserved at the maximum rank).
 * 0 for invalid sizes. */
MLORA_API size_t mlora_pool_bytes(int n_slots, int r_max, int K, int D);

/* ------------------------------------------------------------------ step metadata ---- */

/* Creates a metadata object for steps of at most max_tokens tokens and max_slots_per_token
 * (J) adapter slots per token ("[RFC] ...", item 5: max_loras_per_request), for pools whose
 * r_max is at most r_max. Holds the sorted pair order, the segment table, per-pair scales,
 * the CUDA-core shrink workspace (16 * max_tokens * J * R fp32, R the slot width of r_max) and
 * the tensor-core side path's unit lists with one 16 KB v tile per unit (units: pairs of an
 * M-tile of 128 tokens and a 64-column block of the slot space its tokens use; capacity
 * min(max_tokens * J * ceil(R / 64), tiles * 256, 16384)). */
MLORA_API mlora_status mlora_meta_create(int max_tokens, int max_slots_per_token, int r_max, mlora_meta_t* out);
MLORA_API mlora_status mlora_meta_destroy(mlora_meta_t meta);

/* Builds one step's metadata on the GPU ("Multi-LoRA Serving Explained", batched serving:
 * sort the batch's tokens by slot before shrink and expand; "[RFC] ...", item 2: k slots per
 * token, sentinel -1 in unused ones).
 *   token_slots: device int32 [T, J]; -1 = no adapter.
 *   scales:      device fp32 [T, J] per-(token, slot) scale s, or NULL for s = 1.
 *   pool:        validates slot ids against it (range and loaded); pools used with this
 *                metadata must have the same n_slots.
 * Pairs p = t*J + j are stably sorted by slot (-1 first); segments are runs of one slot in
 * ascending slot order. A pair naming a slot outside [-1, n_slots) or an empty slot is
 * treated as -1 and recorded; mlora_meta_status() reports it as MLORA_ERR_BAD_TOKEN_SLOT.
 * Asynchronous on `stream`; T = 0 is allowed. */
MLORA_API mlora_status mlora_build_meta(mlora_meta_t meta, const int32_t* token_slots, const float* scales, int T, int J,
                              mlora_pool_t pool, void* stream);

/* Synchronises with the last build/linear that used this metadata and reports device-side
 * errors (MLORA_ERR_BAD_TOKEN_SLOT with the first rejected pair in the message,
 * MLORA_ERR_DEVICE_TIMEOUT). Clears the error word. */
MLORA_API mlora_status mlora_meta_status(mlora_meta_t meta);

/* Copies the metadata to host (synchronising): order [T*J], seg_slot and seg_off
 * (n_seg and n_seg + 1 entries; arrays sized T*J + 2 suffice), counts. Any pointer may be NULL. */
MLORA_API mlora_status mlora_meta_read(mlora_meta_t meta, int32_t* order, int32_t* seg_slot, int32_t* seg_off, int* n_seg,
                             int* n_active);

/* ------------------------------------------------------------------ the layer ------- */

/* y = x W^T + sum_j s c B(A x) for the step described by `meta` ("LoRA Serving", section 7:
 * y = base_layer(x), then add_lora_linear(y, x, A_stacked, B_stacked, scaling)).
 *   x: device bf16 [T, K]; W: device bf16 [D, K] (nn.Linear layout); y: device fp32 [T, D],
 *   overwritten. T is the meta's last build. The base product runs on the tensor cores;
 *   when the step has no active pair the LoRA kernels do no work, and rows whose slots are
 *   all -1 equal the base product exactly. Orders itself after the pool's queued loads.
 * Two paths: small batches of a one-class pool (T <= 256, output column blocks within one wave
 * of the SMs, few active slots) run the base product and the shrink in one split-K kernel, then
 * the expand; every other step shrinks on the tensor cores per (M-tile, column block) and adds
 * the expand inside the base GEMM as extra K blocks (y written once).
 * Calls that share a meta or a pool must be ordered on one stream. */
MLORA_API mlora_status mlora_linear(mlora_pool_t pool, mlora_meta_t meta, const mlora_bf16* x, const mlora_bf16* W, float* y,
                          void* stream);

/* The same kernels one at a time (for per-kernel tests and timing):
 *   mlora_base_gemm:   y[T, D] = x[T, K] W[D, K]^T (fp32 out, tcgen05 tensor cores);
 *   mlora_lora_shrink: v = A_slot x per active pair into the meta's workspace;
 *   mlora_lora_expand: y += s c B_slot v per active pair (token-major, slot order j). */
MLORA_API mlora_status mlora_base_gemm(const mlora_bf16* x, const mlora_bf16* W, float* y, int T, int K, int D, void* stream);
MLORA_API mlora_status mlora_lora_shrink(mlora_pool_t pool, mlora_meta_t meta, const mlora_bf16* x, void* stream);
MLORA_API mlora_status mlora_lora_expand(mlora_pool_t pool, mlora_meta_t meta, float* y, void* stream);

/* Tile choice of the tiled base GEMM (batches of more than 256 tokens, and smaller batches
 * whose output is wider than one wave of 128-column blocks; process-wide; no counterpart on the
 * pages: a tuning control). The default, 0, picks per shape: the CTA-pair kernel (tcgen05
 * cta_group::2, 256 x N tiles with N in {256, 224, 192, 128} chosen by estimated time: whole
 * waves of the resident CTA pairs times a per-tile time) whenever the batch spans two or more
 * 128-row tiles, else the one-CTA kernel. -1 never uses the pair kernel; 256, 224, 192 or 128
 * always uses it with that N. Other values: MLORA_ERR_INVALID_ARG, nothing changed. Results
 * differ between choices only by fp32 summation order. Set it between steps, not while a
 * captured graph that launches the GEMM may be re-captured. */
MLORA_API mlora_status mlora_set_gemm_tile_n(int n);

/* Form of the small-batch GEMM (batches of up to 256 tokens; process-wide; no counterpart on the
 * pages: a tuning and test control). 0 (default) and 1: the split-K form (CTA pairs sharing the
 * token operand, K split across a cluster, partial tiles summed in K order). 2: the token-split
 * form whenever its grid fits one wave (each CTA multiplies a group of tokens by one 128-row
 * block over all of K; clusters share W rows and x rows by TMA multicast; no partial tiles),
 * else the split-K form. Other values: MLORA_ERR_INVALID_ARG, nothing changed. Both forms are
 * deterministic; their results differ only by fp32 summation order. Set it between steps. */
MLORA_API mlora_status mlora_set_skinny_form(int form);

/* Path choice of mlora_linear (process-wide; no counterpart on the pages: a tuning and test
 * control): 0 automatic (default), 1 the small-batch path whenever the step allows it, 2 always
 * the tensor-core side path. Other values: MLORA_ERR_INVALID_ARG. Results differ between paths
 * only by rounding (fp32 summation order; bf16 rounding of the scaled v on the tensor-core
 * path). Set it between steps. */
MLORA_API mlora_status mlora_set_path(int path);

/* Allocation-free LoRA side path (no counterpart on the pages: an addition for callers that
 * cannot allocate device memory, such as a serving engine that has handed all free device
 * memory to its KV cache at start-up, so a later cudaMalloc fails, or code on a
 * latency-critical path that cannot accept the implicit device synchronisation of
 * cudaMalloc/cudaFree). It needs no pool or metadata object:
 *   y[t, :] += sum_j s[t,j] * slot_scale[slot] * B_slot (A_slot x[t, :])  for slot = token_slots[t*J + j],
 * over caller-owned device buffers laid out slot by slot (A_pool [n_slots, r_pad, K],
 * B_pool [n_slots, D, r_pad] bf16, zero beyond each slot's rank -- not the column space of
 * mlora_pool_create's pools; slot_scale [n_slots] fp32; slot_rank [n_slots] int32, 0 = empty,
 * at most r_pad). scales may be NULL (s = 1). A token slot outside [0, n_slots), or naming a slot
 * whose rank is not in [1, r_pad], adds nothing. y must already hold the base product.
 * Its only workspace is a fixed array compiled into the library (4 MiB, held by every GPU
 * that loads it until the process exits), so T * J * r_pad must not exceed 1,048,576
 * (else MLORA_ERR_TOO_MANY_TOKENS, nothing launched). It calls no cudaMalloc, cudaFree or
 * other allocating routine. The workspace's device address is looked up (cudaGetSymbolAddress)
 * with the device current on every call made outside stream capture and kept per device; a
 * call inside a capture uses the kept address, so make the first call on each device (and the
 * first after a cudaDeviceReset) outside any capture. All calls share the workspace: calls that
 * overlap on the GPU (different streams, devices aside) race and must be ordered by the
 * caller. Nothing carries over between calls: every workspace value read was written earlier
 * in the same call. */
MLORA_API mlora_status mlora_lora_apply_noalloc(const mlora_bf16* x, float* y, const int32_t* token_slots,
                                                const float* scales, int T, int J, const mlora_bf16* A_pool,
                                                const mlora_bf16* B_pool, const float* slot_scale,
                                                const int32_t* slot_rank, int n_slots, int r_pad, int K, int D,
                                                void* stream);

/* ------------------------------------------------------------------ embedding lookup -- */

/* The slot pool of an embedding table with LoRA ("[vLLM] LoRA" (secrett2633 blog), layer
 * implementation section: the embedding is one of the LoRA layer variants; "LoRA Serving" (vLLM
 * learning book ch. 09-04), section 2). The lookup of token id i is the linear map of the one-hot
 * vector e_i with weight E^T, so an adapter with A [r, vocab] and B [dim, r] adds c B A[:, i].
 * Classes, slot numbering and the column space are those of mlora_pool_create_classes (one
 * class: class_slots = {n_slots}, class_rank = {r_max}); A is kept token-major, A_pool
 * [vocab, C] (row i holds column i of every slot's A), so a token's side path reads one
 * contiguous run of its rank; B_pool is [dim, C]. vocab >= 1; dim a positive even number
 * (else MLORA_ERR_INVALID_ARG). mlora_load_adapter, mlora_clear_slot, mlora_pool_sync,
 * mlora_pool_layout and mlora_pool_info (K = vocab, D = dim) work on it as on a linear pool;
 * A_host is the adapter's [rank, vocab] matrix, staged whole and written token-major by a
 * kernel on the copy stream. mlora_load_adapter_sliced and the linear-layer calls
 * (mlora_linear, mlora_lora_shrink, mlora_lora_expand) reject it with MLORA_ERR_INVALID_ARG. */
MLORA_API mlora_status mlora_embedding_pool_create(int n_classes, const int* class_slots, const int* class_rank,
                                                   int vocab, int dim, void* copy_stream, mlora_pool_t* out);

/* Embedding lookup with LoRA for the step described by `meta` (built by mlora_build_meta with
 * this pool or one of the same slots and classes):
 *     y[t, :] = E[ids[t], :] + sum_{j : slot[t,j] != -1} s[t,j] c(slot) B_slot A_slot[:, ids[t]]
 *   ids: device int32 [T] (T = the meta's last build); E: device bf16 [vocab, dim] row-major;
 *   y: device fp32 [T, dim], overwritten (rows whose slots are all -1 equal the table row
 *   exactly). E and y 16-byte aligned. A token id outside [0, vocab) gives a zero row and is
 *   reported by mlora_meta_status as MLORA_ERR_BAD_TOKEN_ID. One kernel on the CUDA cores (the
 *   lookup is bound by memory traffic); each output is a fixed sequence of fp32 operations.
 * Orders itself after the pool's queued loads; calls sharing a meta or a pool must be ordered
 * on one stream. */
MLORA_API mlora_status mlora_embedding(mlora_pool_t pool, mlora_meta_t meta, const int32_t* ids, const mlora_bf16* E,
                                       float* y, void* stream);

/* ------------------------------------------------------------------ slot residency ---- */

/* Which adapter id sits in which of n_slots GPU slots ("LoRA Serving", section 5: the LRU cache
 * model manager marks a hit as recent and on a miss evicts the oldest adapter that is not pinned;
 * "Multi-LoRA Serving Explained", serving section: a fixed number of GPU slots, least recently
 * used pushed out). Host logic only, no GPU work.
 * mlora_slot_cache_assign maps the ids of one step (n entries, e.g. one per token and slot;
 * -1 = no adapter -> slot -1) to slots: a resident id keeps its slot; each other id takes the
 * lowest free slot, else the slot used longest ago (lowest index on ties) that no id of this step
 * and no pinned id holds. Writes slots[n] and the (id, slot) pairs that must be loaded (first-seen
 * order) to load_ids / load_slots (capacity n each; either may be NULL) and their count to
 * *n_loads. MLORA_ERR_NO_FREE_SLOT when the step names more distinct ids than free or evictable
 * slots allow; nothing changes then. lookup gives an id's slot (-1 if not resident); pin keeps a
 * resident id from eviction (pinned != 0) or releases it; evict frees an id's slot. */
MLORA_API mlora_status mlora_slot_cache_create(int n_slots, mlora_slot_cache_t* out);
MLORA_API mlora_status mlora_slot_cache_destroy(mlora_slot_cache_t cache);
MLORA_API mlora_status mlora_slot_cache_assign(mlora_slot_cache_t cache, const int64_t* ids, int n, int32_t* slots,
                                               int64_t* load_ids, int32_t* load_slots, int* n_loads);
MLORA_API mlora_status mlora_slot_cache_lookup(mlora_slot_cache_t cache, int64_t id, int32_t* slot);
MLORA_API mlora_status mlora_slot_cache_pin(mlora_slot_cache_t cache, int64_t id, int pinned);
MLORA_API mlora_status mlora_slot_cache_evict(mlora_slot_cache_t cache, int64_t id);

/* The slot cache over the pools of one model (one pool per adapted linear, all with the same
 * n_slots): adapters registered by id with one host (A, B) pair per pool, in pool order
 * (A_host[i] [rank, K_i], B_host[i] [D_i, rank], bf16; the caller keeps them valid while
 * registered, pinned for asynchronous loads). mlora_adapter_cache_map assigns the step's ids as
 * mlora_slot_cache_assign does, queues mlora_load_adapter into every pool for each id that is
 * not resident (asynchronous on the pools' copy streams; each pool's next mlora_linear orders
 * itself after them) and writes the host token -> slot map token_slots[n] for mlora_build_meta.
 * An unregistered id: MLORA_ERR_INVALID_ARG, nothing changes. Registering an id again replaces
 * its buffers and drops its resident copy (the next step loads the new one); unregister also
 * unpins it. */
MLORA_API mlora_status mlora_adapter_cache_create(const mlora_pool_t* pools, int n_pools, mlora_adapter_cache_t* out);
MLORA_API mlora_status mlora_adapter_cache_destroy(mlora_adapter_cache_t cache);
MLORA_API mlora_status mlora_adapter_cache_register(mlora_adapter_cache_t cache, int64_t id,
                                                    const mlora_bf16* const* A_host, const mlora_bf16* const* B_host,
                                                    int rank, float alpha, int rslora);
MLORA_API mlora_status mlora_adapter_cache_unregister(mlora_adapter_cache_t cache, int64_t id);
MLORA_API mlora_status mlora_adapter_cache_pin(mlora_adapter_cache_t cache, int64_t id, int pinned);
MLORA_API mlora_status mlora_adapter_cache_map(mlora_adapter_cache_t cache, const int64_t* ids, int n,
                                               int32_t* token_slots, int* n_loaded);

/* ------------------------------------------------------------------ diagnostics ------ */

MLORA_API const char* mlora_status_string(mlora_status status);
MLORA_API const char* mlora_last_error(void);      /* thread-local; valid until the thread's next call */
MLORA_API int mlora_version(void);

/* Kernels this library has launched in this process (all kinds). */
MLORA_API uint64_t mlora_launch_count(void);

/* Check of the failure path every kernel's waits rely on (no counterpart on the pages). Runs on
 * `stream` one kernel whose mbarrier wait can never complete (nothing arrives on it); the wait
 * gives up after the library's limit (2 s), records the timeout in a device error word reserved
 * for this check and the kernel returns, leaving the context usable. Synchronises the stream.
 * Returns MLORA_ERR_DEVICE_TIMEOUT when the wait gave up as designed (the expected result),
 * MLORA_ERR_MISMATCH if no timeout was recorded, MLORA_ERR_CUDA on a CUDA error. Does not touch
 * the error word that mlora_meta_status reports. */
MLORA_API mlora_status mlora_check_wait_timeout(void* stream);

/* Per-kernel CUDA-event trace. While enabled, every kernel launch is bracketed by two events
 * on its own stream (at most `capacity` launches are kept). mlora_trace_read synchronises
 * and returns, for each kernel kind, the number of launches and their summed device time in
 * milliseconds; kinds: 0 meta, 1 base GEMM, 2 shrink, 3 expand, 4 slot bookkeeping, 5 embedding
 * lookup. */
MLORA_API mlora_status mlora_trace_enable(int capacity);
MLORA_API mlora_status mlora_trace_disable(void);
MLORA_API mlora_status mlora_trace_read(int n_kinds, int* launches, double* total_ms);
MLORA_API const char* mlora_kernel_kind_name(int kind);

#ifdef __cplusplus
}
#endif

#endif /* MLORA_H */
