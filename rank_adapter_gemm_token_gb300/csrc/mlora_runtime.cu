// Host runtime behind mlora.h: the adapter pool, the per-step metadata object, stream/event
// ordering between slot loads and layer calls, argument validation, status strings, the
// launch counter and the optional per-kernel event trace.
//
// Sources for the behaviour (see mlora.h for the per-call citations):
//   "Multi-LoRA Serving Explained" (sevydevy.com): stacked zero-padded slots at the maximum
//   rank; an adapter whose rank exceeds it is rejected with an error naming both ranks;
//   -1 = base model only.
//   "LoRA Serving" (vLLM learning book ch. 09-04), section 4.1: activating an adapter copies
//   its weights into a GPU slot; failure-injection list of section 13 (out-of-range slot,
//   incompatible rank, reload of a slot in use, cancelling a load).
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "mlora.h"
#include "internal.h"
#include "ptx.cuh"

using namespace mlora;

namespace {

thread_local std::string g_last_error;

mlora_status fail(mlora_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

mlora_status cuda_fail(cudaError_t e, const char* what) {
  return fail(MLORA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

#define MLORA_CUDA(call, what)                       \
  do {                                               \
    cudaError_t e__ = (call);                        \
    if (e__ != cudaSuccess) return cuda_fail(e__, what); \
  } while (0)

std::atomic<uint64_t> g_launches{0};
std::atomic<int> g_gemm_tile_n{0};          // mlora_set_gemm_tile_n
std::atomic<int> g_skinny_form{0};          // mlora_set_skinny_form
std::atomic<int> g_path{0};                 // mlora_set_path

// ---------------------------------------------------------------- trace
struct TraceRec {
  int kind;
  cudaEvent_t begin, end;
};
struct Trace {
  std::mutex mu;
  bool on = false;
  std::vector<TraceRec> recs;     // pre-created events
  size_t used = 0;
  size_t pending_begin = SIZE_MAX;
} g_trace;

// ---------------------------------------------------------------- per-device state
struct DeviceState {
  bool init = false;
  int num_sms = 0;
  uint32_t* err = nullptr;        // library-wide device error word (timeouts of bounded waits)
  uint32_t* check_err = nullptr;  // error word of mlora_check_wait_timeout only
};
DeviceState g_dev[64];
std::mutex g_dev_mu;

mlora_status device_state(DeviceState** out) {
  int dev = 0;
  MLORA_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(MLORA_ERR_INVALID_ARG, "device ordinal %d unsupported", dev);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceState& d = g_dev[dev];
  if (!d.init) {
    MLORA_CUDA(cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev), "SM count");
    MLORA_CUDA(cudaMalloc(&d.err, sizeof(uint32_t)), "cudaMalloc(error word)");
    MLORA_CUDA(cudaMemset(d.err, 0, sizeof(uint32_t)), "cudaMemset(error word)");
    MLORA_CUDA(cudaMalloc(&d.check_err, sizeof(uint32_t)), "cudaMalloc(check error word)");
    d.init = true;
  }
  *out = &d;
  return MLORA_OK;
}


bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// rank: rows of A in use (the kernels' bound); scale_rank: the r of the factor (the same for a
// plain adapter; the slice rank for a per-slice adapter of a fused linear).
__global__ void set_slot_kernel(float* slot_scale, int32_t* slot_rank, int slot, float alpha, int rank,
                                int scale_rank, int rslora) {
  // c = alpha / r, or alpha / sqrt(r) for rsLoRA ("[vLLM] LoRA", PEFTHelper), fp32, IEEE rounding.
  const float r = static_cast<float>(scale_rank);
  slot_scale[slot] = rank > 0 ? __fdiv_rn(alpha, rslora ? __fsqrt_rn(r) : r) : 0.0f;
  slot_rank[slot] = rank;
}

// Row ranges of the slices of a slot being loaded (a plain adapter is one slice of all D rows).
struct SliceRows {
  int n;
  int row0[MLORA_MAX_SLICES + 1];       // slice i covers rows row0[i] .. row0[i + 1] - 1
};

// Writes a slot's columns of B from the staged adapter: element (o, q), q < width, is slice i's
// B[o - row0[i]][q - i r] when o lies in slice i and q in its columns i r .. i r + r - 1, else 0.
// stage holds the slices one after another, each [rows_i, r] row-major. Thread = (row, 8 columns).
__global__ void scatter_slot_b_kernel(uint16_t* __restrict__ B, int C, int off, int width, int D,
                                      const uint16_t* __restrict__ stage, int r, SliceRows sl) {
  const int groups = width / 8;
  const long items = static_cast<long>(D) * groups;
  for (long it = blockIdx.x * static_cast<long>(blockDim.x) + threadIdx.x; it < items;
       it += static_cast<long>(gridDim.x) * blockDim.x) {
    const int o = static_cast<int>(it / groups), q0 = static_cast<int>(it % groups) * 8;
    int i = 0;
    while (i + 1 < sl.n && o >= sl.row0[i + 1]) ++i;
    uint16_t v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int q = q0 + k - i * r;
      v[k] = (i < sl.n && q >= 0 && q < r)
                 ? stage[static_cast<size_t>(sl.row0[i]) * r + static_cast<size_t>(o - sl.row0[i]) * r + q]
                 : static_cast<uint16_t>(0);
    }
    uint4 w;
    w.x = v[0] | (static_cast<uint32_t>(v[1]) << 16);
    w.y = v[2] | (static_cast<uint32_t>(v[3]) << 16);
    w.z = v[4] | (static_cast<uint32_t>(v[5]) << 16);
    w.w = v[6] | (static_cast<uint32_t>(v[7]) << 16);
    *reinterpret_cast<uint4*>(B + static_cast<size_t>(o) * C + off + q0) = w;
  }
}

}  // namespace

namespace mlora {

int report_error(int status, const char* message) { return fail(status, "%s", message); }
int report_cuda_error(cudaError_t e, const char* what) { return cuda_fail(e, what); }
int gemm_tile_n() { return g_gemm_tile_n.load(std::memory_order_relaxed); }
int skinny_form() { return g_skinny_form.load(std::memory_order_relaxed); }

void note_launch_begin(int kind, cudaStream_t s) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (!g_trace.on) return;
  std::lock_guard<std::mutex> lk(g_trace.mu);
  if (!g_trace.on || g_trace.used >= g_trace.recs.size()) return;
  TraceRec& r = g_trace.recs[g_trace.used];
  r.kind = kind;
  if (cudaEventRecord(r.begin, s) == cudaSuccess) g_trace.pending_begin = g_trace.used;
}

void note_launch_end(int kind, cudaStream_t s) {
  if (!g_trace.on) return;
  std::lock_guard<std::mutex> lk(g_trace.mu);
  if (g_trace.pending_begin != g_trace.used) return;
  TraceRec& r = g_trace.recs[g_trace.used];
  if (r.kind == kind && cudaEventRecord(r.end, s) == cudaSuccess) ++g_trace.used;
  g_trace.pending_begin = SIZE_MAX;
}

}  // namespace mlora

struct mlora_pool {
  int device = 0;
  int S = 0, r_max = 0, R = 0, K = 0, D = 0;
  int C = 0;                                   // columns of the slot space
  bool embed = false;                          // an embedding pool: A token-major, K = vocabulary
  uint16_t* A = nullptr;                       // [C, K] ([K, C] for an embedding pool)
  uint16_t* B = nullptr;                       // [D, C]
  float* slot_scale = nullptr;
  int32_t* slot_rank = nullptr;
  int32_t* slot_off = nullptr;                 // [S] first column of each slot
  int32_t* slot_width = nullptr;               // [S] columns of each slot
  int32_t* col_slot = nullptr;                 // [C] slot owning each column
  uint16_t* stage = nullptr;                   // [D * R] a loading adapter's B (or embedding A), before its scatter
  std::vector<int> class_slots, class_rank;    // the rank classes (one for mlora_pool_create)
  std::vector<int> h_rank, h_off, h_width, h_class;
  int max_span = 1;                            // most 64-column blocks one slot touches
  cudaStream_t copy_stream = nullptr;
  bool own_stream = false;
  cudaEvent_t load_done = nullptr, use_done = nullptr;
  bool has_load = false;
  uint64_t load_seq = 0;                       // number of loads/clears queued so far
  // Streams that have read this pool, with the load_seq each last waited for. A load orders
  // itself after all work already queued on them (write-after-read); a compute call waits for
  // the loads only when one was queued since its stream last waited. No event is recorded on
  // the compute path.
  std::vector<std::pair<cudaStream_t, uint64_t>> users;
  std::mutex mu;

  bool uniform() const { return class_slots.size() == 1; }
  PoolView view() const {
    return PoolView{A, B, slot_scale, slot_rank, slot_off, slot_width, col_slot, S, R, C, K, D, uniform() ? 1 : 0};
  }
};

struct mlora_meta {
  int device = 0;
  int max_tokens = 0, J_max = 0, r_max = 0, R_max = 0, n_max = 0;
  int32_t *order = nullptr, *seg_slot = nullptr, *seg_off = nullptr, *pair_slot = nullptr;
  float* pair_scale = nullptr;
  int32_t *blk_slot = nullptr, *blk_start = nullptr, *blk_count = nullptr, *counts = nullptr;
  int32_t *pair_act = nullptr, *act_slot = nullptr;
  uint32_t* err = nullptr;
  float* vpart = nullptr;
  float* vfull = nullptr;
  int vfull_ld = 0;
  int32_t *tile_unit_off = nullptr, *unit_blk = nullptr, *unit_tile = nullptr, *grp_mp = nullptr,
          *grp_ent = nullptr, *grp_cnt = nullptr, *ptile_off = nullptr, *pent_blk = nullptr, *pent_u0 = nullptr, *pent_u1 = nullptr,
          *pair_fused = nullptr, *todo_blk = nullptr, *ptile_order = nullptr;
  uint32_t* sync = nullptr;
  uint16_t* vtile = nullptr;
  int unit_cap = 0;
  int T = 0, J = 1, S = -1;
  std::vector<int> class_slots, class_rank;    // layout of the pool the last build used
  bool built = false;
  bool units_built = false;                    // the tensor-core path's units of the last build
  cudaEvent_t done = nullptr;
  cudaStream_t last_stream = nullptr;          // the stream of the last call that used the metadata

  MetaView view() const {
    MetaView v{};
    v.order = order;
    v.seg_slot = seg_slot;
    v.seg_off = seg_off;
    v.pair_slot = pair_slot;
    v.pair_scale = pair_scale;
    v.blk_slot = blk_slot;
    v.blk_start = blk_start;
    v.blk_count = blk_count;
    v.counts = counts;
    v.pair_act = pair_act;
    v.act_slot = act_slot;
    v.err = err;
    v.vpart = vpart;
    v.vfull = vfull;
    v.vfull_ld = vfull_ld;
    v.tile_unit_off = tile_unit_off;
    v.unit_blk = unit_blk;
    v.unit_tile = unit_tile;
    v.grp_mp = grp_mp;
    v.grp_ent = grp_ent;
    v.grp_cnt = grp_cnt;
    v.ptile_off = ptile_off;
    v.pent_blk = pent_blk;
    v.pent_u0 = pent_u0;
    v.pent_u1 = pent_u1;
    v.pair_fused = pair_fused;
    v.todo_blk = todo_blk;
    v.ptile_order = ptile_order;
    v.sync = sync;
    v.vtile = vtile;
    v.unit_cap = unit_cap;
    v.n = T * J;
    v.T = T;
    v.J = J;
    return v;
  }
};

extern "C" {

int mlora_version(void) { return 1; }

mlora_status mlora_check_wait_timeout(void* stream) {
  DeviceState* ds = nullptr;
  if (mlora_status st = device_state(&ds)) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t word = 0;
  MLORA_CUDA(cudaMemsetAsync(ds->check_err, 0, sizeof(uint32_t), s), "clear check error word");
  MLORA_CUDA(launch_wait_check(ds->check_err, s), "wait-check launch");
  MLORA_CUDA(cudaMemcpyAsync(&word, ds->check_err, sizeof(uint32_t), cudaMemcpyDeviceToHost, s), "read check word");
  MLORA_CUDA(cudaStreamSynchronize(s), "wait-check sync");
  if (word & ptx::kErrWaitTimeout) return fail(MLORA_ERR_DEVICE_TIMEOUT, "the check kernel's wait gave up, as designed");
  return fail(MLORA_ERR_MISMATCH, "the check kernel's wait did not report a timeout (error word %u)", word);
}

mlora_status mlora_set_gemm_tile_n(int n) {
  if (n != 0 && n != -1 && n != 256 && n != 224 && n != 192 && n != 128)
    return fail(MLORA_ERR_INVALID_ARG, "tile N must be 0 (automatic), -1 (one-CTA kernel), 256, 224, 192 or 128");
  g_gemm_tile_n.store(n);
  return MLORA_OK;
}

mlora_status mlora_set_skinny_form(int form) {
  if (form < 0 || form > 2) return fail(MLORA_ERR_INVALID_ARG, "form must be 0 (default, split-K), 1 (split-K) or 2 (token-split)");
  g_skinny_form.store(form);
  return MLORA_OK;
}

mlora_status mlora_set_path(int path) {
  if (path < 0 || path > 2) return fail(MLORA_ERR_INVALID_ARG, "path must be 0 (automatic), 1 or 2");
  g_path.store(path);
  return MLORA_OK;
}

uint64_t mlora_launch_count(void) { return g_launches.load(); }

const char* mlora_last_error(void) { return g_last_error.c_str(); }

const char* mlora_status_string(mlora_status s) {
  switch (s) {
    case MLORA_OK: return "ok";
    case MLORA_ERR_INVALID_ARG: return "invalid argument";
    case MLORA_ERR_SLOT_RANGE: return "slot out of range";
    case MLORA_ERR_RANK_TOO_LARGE: return "adapter rank larger than the pool's maximum rank";
    case MLORA_ERR_RANK_INVALID: return "invalid adapter rank or alpha";
    case MLORA_ERR_BAD_TOKEN_SLOT: return "a token named an invalid or empty slot";
    case MLORA_ERR_TOO_MANY_TOKENS: return "more tokens or slots per token than the metadata holds";
    case MLORA_ERR_OOM: return "out of memory";
    case MLORA_ERR_CUDA: return "CUDA error";
    case MLORA_ERR_DEVICE_TIMEOUT: return "a device-side wait timed out";
    case MLORA_ERR_MISMATCH: return "pool, metadata and operands do not fit together";
    case MLORA_ERR_NO_FREE_SLOT: return "more adapters needed at once than free or evictable slots";
    case MLORA_ERR_BAD_TOKEN_ID: return "a token id outside the embedding table";
    default: return "unknown status";
  }
}

const char* mlora_kernel_kind_name(int kind) {
  static const char* names[kNumKinds] = {"meta", "base_gemm", "shrink", "expand", "slot", "embedding"};
  return (kind >= 0 && kind < kNumKinds) ? names[kind] : "?";
}

size_t mlora_pool_bytes(int n_slots, int r_max, int K, int D) {
  if (n_slots < 1 || r_max < 1 || K < 1 || D < 1) return 0;
  return static_cast<size_t>(n_slots) * static_cast<size_t>(slot_width(r_max)) *
         (static_cast<size_t>(K) + static_cast<size_t>(D)) * 2u;
}

// ---------------------------------------------------------------- pool
// Slots are numbered class by class; slot i of class c owns the next width_c = slot_width(rank_c)
// columns of the slot space (each class starting on a multiple of min(width_c, 64), so no slot
// straddles two 64-column blocks), so a pool's layout is a function of its class list alone and
// pools created with the same classes lay out their slots identically.
static mlora_status pool_create(int n_classes, const int* class_slots, const int* class_rank, int K, int D,
                                void* copy_stream, mlora_pool_t* out, bool embed = false) {
  if (!out) return fail(MLORA_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (n_classes < 1 || n_classes > MLORA_MAX_CLASSES || !class_slots || !class_rank)
    return fail(MLORA_ERR_INVALID_ARG, "n_classes %d outside [1, %d] or a class array is NULL", n_classes,
                MLORA_MAX_CLASSES);
  long S = 0;
  int r_max = 0;
  for (int c = 0; c < n_classes; ++c) {
    if (class_slots[c] < 1) return fail(MLORA_ERR_INVALID_ARG, "class %d has %d slots", c, class_slots[c]);
    if (class_rank[c] < 1 || class_rank[c] > MLORA_MAX_RANK)
      return fail(MLORA_ERR_INVALID_ARG, "class %d: rank %d outside [1, %d]", c, class_rank[c], MLORA_MAX_RANK);
    S += class_slots[c];
    r_max = std::max(r_max, class_rank[c]);
  }
  if (S > MLORA_MAX_SLOTS) return fail(MLORA_ERR_INVALID_ARG, "%ld slots: more than %d", S, MLORA_MAX_SLOTS);
  if (embed) {
    if (K < 1) return fail(MLORA_ERR_INVALID_ARG, "vocabulary %d must be positive", K);
    if (D < 2 || D % 2 != 0) return fail(MLORA_ERR_INVALID_ARG, "embedding width %d must be a positive even number", D);
  } else {
    if (K < 8 || K % 8 != 0) return fail(MLORA_ERR_INVALID_ARG, "K %d must be a positive multiple of 8", K);
    if (D < 1) return fail(MLORA_ERR_INVALID_ARG, "D %d must be positive", D);
  }
  DeviceState* ds = nullptr;
  if (mlora_status st = device_state(&ds)) return st;
  mlora_pool* p = new (std::nothrow) mlora_pool();
  if (!p) return fail(MLORA_ERR_OOM, "host allocation failed");
  cudaGetDevice(&p->device);
  p->embed = embed;
  p->S = static_cast<int>(S);
  p->r_max = r_max;
  p->R = slot_width(r_max);
  p->K = K;
  p->D = D;
  p->class_slots.assign(class_slots, class_slots + n_classes);
  p->class_rank.assign(class_rank, class_rank + n_classes);
  p->h_rank.assign(p->S, 0);
  int col = 0;
  for (int c = 0; c < n_classes; ++c) {
    const int w = slot_width(class_rank[c]);
    const int align = std::min(w, kBlockCols);
    col = (col + align - 1) / align * align;
    for (int i = 0; i < class_slots[c]; ++i) {
      p->h_off.push_back(col);
      p->h_width.push_back(w);
      p->h_class.push_back(c);
      p->max_span = std::max(p->max_span, (col + w - 1) / kBlockCols - col / kBlockCols + 1);
      col += w;
    }
  }
  p->C = col;
  std::vector<int32_t> col_slot(p->C, -1);
  for (int sl = 0; sl < p->S; ++sl)
    for (int q = 0; q < p->h_width[sl]; ++q) col_slot[p->h_off[sl] + q] = sl;
  const size_t a_bytes = static_cast<size_t>(p->C) * K * 2;
  const size_t b_bytes = static_cast<size_t>(D) * p->C * 2;
  cudaError_t e = cudaSuccess;
  if ((e = cudaMalloc(&p->A, a_bytes)) != cudaSuccess || (e = cudaMalloc(&p->B, b_bytes)) != cudaSuccess ||
      (e = cudaMalloc(&p->slot_scale, p->S * sizeof(float))) != cudaSuccess ||
      (e = cudaMalloc(&p->slot_rank, p->S * sizeof(int32_t))) != cudaSuccess ||
      (e = cudaMalloc(&p->slot_off, p->S * sizeof(int32_t))) != cudaSuccess ||
      (e = cudaMalloc(&p->slot_width, p->S * sizeof(int32_t))) != cudaSuccess ||
      (e = cudaMalloc(&p->col_slot, p->C * sizeof(int32_t))) != cudaSuccess ||
      (e = cudaMalloc(&p->stage, static_cast<size_t>(embed ? std::max(D, K) : D) * p->R * 2)) != cudaSuccess) {
    cudaGetLastError();
    mlora_pool_destroy(p);
    return e == cudaErrorMemoryAllocation ? fail(MLORA_ERR_OOM, "cudaMalloc of %zu + %zu bytes failed", a_bytes, b_bytes)
                                          : cuda_fail(e, "cudaMalloc");
  }
  if ((e = cudaMemset(p->A, 0, a_bytes)) != cudaSuccess || (e = cudaMemset(p->B, 0, b_bytes)) != cudaSuccess ||
      (e = cudaMemset(p->slot_scale, 0, p->S * sizeof(float))) != cudaSuccess ||
      (e = cudaMemset(p->slot_rank, 0, p->S * sizeof(int32_t))) != cudaSuccess ||
      (e = cudaMemcpy(p->slot_off, p->h_off.data(), p->S * sizeof(int32_t), cudaMemcpyHostToDevice)) != cudaSuccess ||
      (e = cudaMemcpy(p->slot_width, p->h_width.data(), p->S * sizeof(int32_t), cudaMemcpyHostToDevice)) !=
          cudaSuccess ||
      (e = cudaMemcpy(p->col_slot, col_slot.data(), p->C * sizeof(int32_t), cudaMemcpyHostToDevice)) != cudaSuccess) {
    mlora_pool_destroy(p);
    return cuda_fail(e, "pool initialisation");
  }
  if (copy_stream) {
    p->copy_stream = static_cast<cudaStream_t>(copy_stream);
  } else {
    if ((e = cudaStreamCreateWithFlags(&p->copy_stream, cudaStreamNonBlocking)) != cudaSuccess) {
      mlora_pool_destroy(p);
      return cuda_fail(e, "cudaStreamCreate");
    }
    p->own_stream = true;
  }
  if ((e = cudaEventCreateWithFlags(&p->load_done, cudaEventDisableTiming)) != cudaSuccess ||
      (e = cudaEventCreateWithFlags(&p->use_done, cudaEventDisableTiming)) != cudaSuccess) {
    mlora_pool_destroy(p);
    return cuda_fail(e, "cudaEventCreate");
  }
  if ((e = cudaDeviceSynchronize()) != cudaSuccess) {
    mlora_pool_destroy(p);
    return cuda_fail(e, "pool initialisation");
  }
  *out = p;
  return MLORA_OK;
}

mlora_status mlora_pool_create(int n_slots, int r_max, int K, int D, void* copy_stream, mlora_pool_t* out) {
  if (out) *out = nullptr;
  if (n_slots < 1 || n_slots > MLORA_MAX_SLOTS)
    return fail(MLORA_ERR_INVALID_ARG, "n_slots %d outside [1, %d]", n_slots, MLORA_MAX_SLOTS);
  if (r_max < 1 || r_max > MLORA_MAX_RANK)
    return fail(MLORA_ERR_INVALID_ARG, "r_max %d outside [1, %d]", r_max, MLORA_MAX_RANK);
  return pool_create(1, &n_slots, &r_max, K, D, copy_stream, out);
}

mlora_status mlora_pool_create_classes(int n_classes, const int* class_slots, const int* class_rank, int K, int D,
                                       void* copy_stream, mlora_pool_t* out) {
  return pool_create(n_classes, class_slots, class_rank, K, D, copy_stream, out);
}

mlora_status mlora_embedding_pool_create(int n_classes, const int* class_slots, const int* class_rank, int vocab,
                                         int dim, void* copy_stream, mlora_pool_t* out) {
  return pool_create(n_classes, class_slots, class_rank, vocab, dim, copy_stream, out, true);
}

mlora_status mlora_pool_layout(mlora_pool_t p, int* C, int32_t* slot_off, int32_t* slot_width) {
  if (!p) return fail(MLORA_ERR_INVALID_ARG, "pool is NULL");
  if (C) *C = p->C;
  for (int sl = 0; sl < p->S; ++sl) {
    if (slot_off) slot_off[sl] = p->h_off[sl];
    if (slot_width) slot_width[sl] = p->h_width[sl];
  }
  return MLORA_OK;
}

mlora_status mlora_pool_destroy(mlora_pool_t p) {
  if (!p) return MLORA_OK;
  if (p->has_load) cudaEventSynchronize(p->load_done);
  for (auto& u : p->users) cudaStreamSynchronize(u.first);
  if (p->copy_stream) cudaStreamSynchronize(p->copy_stream);
  if (p->own_stream && p->copy_stream) cudaStreamDestroy(p->copy_stream);
  if (p->load_done) cudaEventDestroy(p->load_done);
  if (p->use_done) cudaEventDestroy(p->use_done);
  cudaFree(p->A);
  cudaFree(p->B);
  cudaFree(p->slot_scale);
  cudaFree(p->slot_rank);
  cudaFree(p->slot_off);
  cudaFree(p->slot_width);
  cudaFree(p->col_slot);
  cudaFree(p->stage);
  delete p;
  return MLORA_OK;
}

// Writes a slot on the pool's copy stream after every call already queued on the pool: zeroes
// its A rows (rows off .. off + width - 1) and copies n_slices adapters of rank r each; slice i's
// A [r, K] goes to rows off + i r ..; the slices' B [widths[i], r] are copied whole into the
// pool's staging buffer and a kernel writes the slot's B columns off .. off + width - 1 from it
// (slice i at rows o_i .. (o_i = sum of the earlier widths) and columns off + i r .., zeros
// elsewhere: block-diagonal; a plain adapter is one slice of width D). n_slices = 0 clears it.
static mlora_status write_slot_sliced(mlora_pool_t p, int slot, int n_slices, const int* widths,
                                      const mlora_bf16* const* A_host, const mlora_bf16* const* B_host, int r,
                                      float alpha, int rslora) {
  cudaStream_t cs = p->copy_stream;
  for (auto& u : p->users) {                   // after every call already queued on the pool
    MLORA_CUDA(cudaEventRecord(p->use_done, u.first), "record use event");
    MLORA_CUDA(cudaStreamWaitEvent(cs, p->use_done, 0), "wait for last use of the pool");
  }
  const size_t off = static_cast<size_t>(p->h_off[slot]);
  const size_t width = static_cast<size_t>(p->h_width[slot]);
  uint16_t* a_slot = p->A + off * p->K;
  if (!p->embed) MLORA_CUDA(cudaMemsetAsync(a_slot, 0, width * p->K * 2, cs), "zero slot A");
  SliceRows sl{};
  sl.n = n_slices;
  int row = 0;
  for (int i = 0; i < n_slices; ++i) {
    const int w = widths ? widths[i] : p->D;
    sl.row0[i] = row;
    if (!p->embed)
      MLORA_CUDA(cudaMemcpyAsync(a_slot + static_cast<size_t>(i) * r * p->K, A_host[i],
                                 static_cast<size_t>(r) * p->K * 2, cudaMemcpyHostToDevice, cs),
                 "copy A into slot");
    MLORA_CUDA(cudaMemcpyAsync(p->stage + static_cast<size_t>(row) * r, B_host[i], static_cast<size_t>(w) * r * 2,
                               cudaMemcpyHostToDevice, cs),
               "copy B to the staging buffer");
    row += w;
  }
  sl.row0[n_slices] = row;
  {
    const long items = static_cast<long>(p->D) * static_cast<long>(width / 8);
    const int grid = static_cast<int>(std::min<long>((items + 255) / 256, 4096));
    note_launch_begin(kKindSlot, cs);
    scatter_slot_b_kernel<<<grid, 256, 0, cs>>>(p->B, p->C, static_cast<int>(off), static_cast<int>(width), p->D,
                                                p->stage, r, sl);
    cudaError_t e = cudaGetLastError();
    note_launch_end(kKindSlot, cs);
    if (e != cudaSuccess) return cuda_fail(e, "scatter_slot_b_kernel");
  }
  if (p->embed) {
    // an embedding pool's A [r, V] is staged whole (after the B scatter, in stream order) and
    // written token-major into columns off .. off + width - 1 of A^T [V, C]
    const int ra = n_slices > 0 ? r : 0;
    if (ra > 0)
      MLORA_CUDA(cudaMemcpyAsync(p->stage, A_host[0], static_cast<size_t>(ra) * p->K * 2, cudaMemcpyHostToDevice, cs),
                 "copy A to the staging buffer");
    note_launch_begin(kKindSlot, cs);
    cudaError_t e = launch_scatter_slot_at(p->A, p->C, static_cast<int>(off), static_cast<int>(width), p->K, p->stage,
                                           ra, cs);
    note_launch_end(kKindSlot, cs);
    if (e != cudaSuccess) return cuda_fail(e, "scatter_slot_at_kernel");
  }
  const int rank = n_slices * r;
  note_launch_begin(kKindSlot, cs);
  set_slot_kernel<<<1, 1, 0, cs>>>(p->slot_scale, p->slot_rank, slot, alpha, rank, r, rslora);
  cudaError_t e = cudaGetLastError();
  note_launch_end(kKindSlot, cs);
  if (e != cudaSuccess) return cuda_fail(e, "set_slot_kernel");
  MLORA_CUDA(cudaEventRecord(p->load_done, cs), "record load event");
  p->has_load = true;
  ++p->load_seq;
  p->h_rank[slot] = rank;
  return MLORA_OK;
}

// The largest rank slot `slot` accepts (its class's rank).
static int slot_rank_limit(mlora_pool_t p, int slot) { return p->class_rank[p->h_class[slot]]; }

mlora_status mlora_load_adapter(mlora_pool_t p, int slot, const mlora_bf16* A_host, const mlora_bf16* B_host,
                                int rank, float alpha, int rslora) {
  if (!p) return fail(MLORA_ERR_INVALID_ARG, "pool is NULL");
  if (slot < 0 || slot >= p->S) return fail(MLORA_ERR_SLOT_RANGE, "slot %d outside [0, %d)", slot, p->S);
  if (rank < 1 || !std::isfinite(alpha))
    return fail(MLORA_ERR_RANK_INVALID, "rank %d must be >= 1 and alpha finite", rank);
  if (rank > slot_rank_limit(p, slot)) {
    if (p->uniform())
      return fail(MLORA_ERR_RANK_TOO_LARGE, "adapter rank %d is larger than the pool's max rank %d", rank, p->r_max);
    return fail(MLORA_ERR_RANK_TOO_LARGE, "adapter rank %d is larger than the max rank %d of slot %d's class", rank,
                slot_rank_limit(p, slot), slot);
  }
  if (!A_host || !B_host) return fail(MLORA_ERR_INVALID_ARG, "A_host or B_host is NULL");
  std::lock_guard<std::mutex> lk(p->mu);
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev != p->device) return fail(MLORA_ERR_MISMATCH, "pool lives on device %d, current is %d", p->device, dev);
  return write_slot_sliced(p, slot, 1, nullptr, &A_host, &B_host, rank, alpha, rslora);
}

mlora_status mlora_load_adapter_sliced(mlora_pool_t p, int slot, int n_slices, const int* widths,
                                       const mlora_bf16* const* A_slices, const mlora_bf16* const* B_slices, int rank,
                                       float alpha, int rslora) {
  if (!p) return fail(MLORA_ERR_INVALID_ARG, "pool is NULL");
  if (slot < 0 || slot >= p->S) return fail(MLORA_ERR_SLOT_RANGE, "slot %d outside [0, %d)", slot, p->S);
  if (n_slices < 1 || n_slices > MLORA_MAX_SLICES)
    return fail(MLORA_ERR_INVALID_ARG, "n_slices %d outside [1, %d]", n_slices, MLORA_MAX_SLICES);
  if (p->embed) return fail(MLORA_ERR_INVALID_ARG, "an embedding pool takes whole adapters (mlora_load_adapter)");
  if (!widths || !A_slices || !B_slices) return fail(MLORA_ERR_INVALID_ARG, "widths or slice arrays are NULL");
  long total = 0;
  for (int i = 0; i < n_slices; ++i) {
    if (widths[i] < 1) return fail(MLORA_ERR_INVALID_ARG, "slice %d has width %d", i, widths[i]);
    if (!A_slices[i] || !B_slices[i]) return fail(MLORA_ERR_INVALID_ARG, "slice %d: A or B is NULL", i);
    total += widths[i];
  }
  if (total != p->D) return fail(MLORA_ERR_INVALID_ARG, "slice widths add up to %ld, the pool's D is %d", total, p->D);
  if (rank < 1 || !std::isfinite(alpha))
    return fail(MLORA_ERR_RANK_INVALID, "rank %d must be >= 1 and alpha finite", rank);
  if (static_cast<long>(n_slices) * rank > slot_rank_limit(p, slot))
    return fail(MLORA_ERR_RANK_TOO_LARGE, "%d slices of rank %d need rank %d, larger than slot %d's max rank %d",
                n_slices, rank, n_slices * rank, slot, slot_rank_limit(p, slot));
  std::lock_guard<std::mutex> lk(p->mu);
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev != p->device) return fail(MLORA_ERR_MISMATCH, "pool lives on device %d, current is %d", p->device, dev);
  return write_slot_sliced(p, slot, n_slices, widths, A_slices, B_slices, rank, alpha, rslora);
}

mlora_status mlora_clear_slot(mlora_pool_t p, int slot) {
  if (!p) return fail(MLORA_ERR_INVALID_ARG, "pool is NULL");
  if (slot < 0 || slot >= p->S) return fail(MLORA_ERR_SLOT_RANGE, "slot %d outside [0, %d)", slot, p->S);
  std::lock_guard<std::mutex> lk(p->mu);
  return write_slot_sliced(p, slot, 0, nullptr, nullptr, nullptr, 0, 0.f, 0);
}

mlora_status mlora_pool_sync(mlora_pool_t p) {
  if (!p) return fail(MLORA_ERR_INVALID_ARG, "pool is NULL");
  if (p->has_load) MLORA_CUDA(cudaEventSynchronize(p->load_done), "pool sync");
  return MLORA_OK;
}

mlora_status mlora_pool_info(mlora_pool_t p, int* n_slots, int* r_pad, int* K, int* D, void** A_pool, void** B_pool,
                             void** slot_scale, void** slot_rank) {
  if (!p) return fail(MLORA_ERR_INVALID_ARG, "pool is NULL");
  if (n_slots) *n_slots = p->S;
  if (r_pad) *r_pad = p->R;
  if (K) *K = p->K;
  if (D) *D = p->D;
  if (A_pool) *A_pool = p->A;
  if (B_pool) *B_pool = p->B;
  if (slot_scale) *slot_scale = p->slot_scale;
  if (slot_rank) *slot_rank = p->slot_rank;
  return MLORA_OK;
}

// Orders stream s after the pool's queued loads (only if one was queued since s last waited)
// and remembers s as a user of the pool.
static mlora_status pool_use(mlora_pool_t p, cudaStream_t s) {
  std::lock_guard<std::mutex> lk(p->mu);
  for (auto& u : p->users) {
    if (u.first == s) {
      if (p->has_load && u.second != p->load_seq) {
        MLORA_CUDA(cudaStreamWaitEvent(s, p->load_done, 0), "wait for slot loads");
        u.second = p->load_seq;
      }
      return MLORA_OK;
    }
  }
  if (p->has_load) MLORA_CUDA(cudaStreamWaitEvent(s, p->load_done, 0), "wait for slot loads");
  p->users.emplace_back(s, p->load_seq);
  return MLORA_OK;
}

// ---------------------------------------------------------------- meta
mlora_status mlora_meta_create(int max_tokens, int J_max, int r_max, mlora_meta_t* out) {
  if (!out) return fail(MLORA_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (max_tokens < 1 || max_tokens > MLORA_MAX_TOKENS)
    return fail(MLORA_ERR_INVALID_ARG, "max_tokens %d outside [1, %d]", max_tokens, MLORA_MAX_TOKENS);
  if (J_max < 1 || J_max > MLORA_MAX_SLOTS_PER_TOKEN)
    return fail(MLORA_ERR_INVALID_ARG, "slots per token %d outside [1, %d]", J_max, MLORA_MAX_SLOTS_PER_TOKEN);
  if (r_max < 1 || r_max > MLORA_MAX_RANK)
    return fail(MLORA_ERR_INVALID_ARG, "r_max %d outside [1, %d]", r_max, MLORA_MAX_RANK);
  DeviceState* ds = nullptr;
  if (mlora_status st = device_state(&ds)) return st;
  mlora_meta* m = new (std::nothrow) mlora_meta();
  if (!m) return fail(MLORA_ERR_OOM, "host allocation failed");
  cudaGetDevice(&m->device);
  m->max_tokens = max_tokens;
  m->J_max = J_max;
  m->r_max = r_max;
  m->R_max = slot_width(r_max);
  m->n_max = max_tokens * J_max;
  const size_t n = static_cast<size_t>(m->n_max);
  cudaError_t e = cudaSuccess;
  auto alloc = [&](void** ptr, size_t bytes) {
    if (e == cudaSuccess) e = cudaMalloc(ptr, bytes);
  };
  alloc(reinterpret_cast<void**>(&m->order), n * 4);
  alloc(reinterpret_cast<void**>(&m->seg_slot), (n + 1) * 4);
  alloc(reinterpret_cast<void**>(&m->seg_off), (n + 2) * 4);
  alloc(reinterpret_cast<void**>(&m->pair_slot), n * 4);
  alloc(reinterpret_cast<void**>(&m->pair_scale), n * 4);
  alloc(reinterpret_cast<void**>(&m->blk_slot), n * 4);
  alloc(reinterpret_cast<void**>(&m->blk_start), n * 4);
  alloc(reinterpret_cast<void**>(&m->blk_count), n * 4);
  alloc(reinterpret_cast<void**>(&m->counts), 8 * 4);
  alloc(reinterpret_cast<void**>(&m->pair_act), n * 4);
  alloc(reinterpret_cast<void**>(&m->act_slot), (n + 1) * 4);
  alloc(reinterpret_cast<void**>(&m->err), 4);
  alloc(reinterpret_cast<void**>(&m->vpart), static_cast<size_t>(kMaxShrinkSplits) * n * m->R_max * 4);
  // tensor-core side path: units (M-tile, 64-column block), their shrink groups, the pair tiles'
  // entry lists and one bf16 v tile [128][64] per unit
  const size_t n_tiles = (static_cast<size_t>(max_tokens) + 127) / 128;
  const size_t span = static_cast<size_t>((m->R_max + kBlockCols - 1) / kBlockCols);   // blocks per slot
  m->unit_cap = static_cast<int>(std::min(std::min(n * span, n_tiles * kMaxTileUnits), static_cast<size_t>(kMaxUnits)));
  const size_t U = static_cast<size_t>(m->unit_cap);
  alloc(reinterpret_cast<void**>(&m->tile_unit_off), (n_tiles + 1) * 4);
  alloc(reinterpret_cast<void**>(&m->unit_blk), U * 4);
  alloc(reinterpret_cast<void**>(&m->unit_tile), U * 4);
  alloc(reinterpret_cast<void**>(&m->grp_mp), U * 4);
  alloc(reinterpret_cast<void**>(&m->grp_ent), U * 4);
  alloc(reinterpret_cast<void**>(&m->grp_cnt), U * 4);
  alloc(reinterpret_cast<void**>(&m->ptile_off), ((n_tiles + 1) / 2 + 1) * 4);
  alloc(reinterpret_cast<void**>(&m->pent_blk), U * 4);
  alloc(reinterpret_cast<void**>(&m->pent_u0), U * 4);
  alloc(reinterpret_cast<void**>(&m->pent_u1), U * 4);
  alloc(reinterpret_cast<void**>(&m->ptile_order), ((n_tiles + 1) / 2 + 1) * 4);
  alloc(reinterpret_cast<void**>(&m->sync), ((n_tiles + 1) / 2 + 2) * 4);
  alloc(reinterpret_cast<void**>(&m->pair_fused), n * 4);
  alloc(reinterpret_cast<void**>(&m->todo_blk), n * 4);
  alloc(reinterpret_cast<void**>(&m->vtile), U * 128 * kBlockCols * 2);
  // small-batch shrink output: v of every token (up to 256) against every active slot
  const int vt = std::min(max_tokens, kVfullMaxTokens);
  m->vfull_ld = std::min(m->n_max, kVfullMaxAct) * m->R_max;
  alloc(reinterpret_cast<void**>(&m->vfull), static_cast<size_t>(vt) * m->vfull_ld * 4);
  if (e == cudaSuccess) e = cudaMemset(m->err, 0, 4);
  if (e == cudaSuccess) e = cudaMemset(m->counts, 0, 32);
  if (e == cudaSuccess) e = cudaMemset(m->sync, 0, ((n_tiles + 1) / 2 + 2) * 4);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&m->done, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    cudaGetLastError();
    mlora_meta_destroy(m);
    return e == cudaErrorMemoryAllocation ? fail(MLORA_ERR_OOM, "metadata allocation failed")
                                          : cuda_fail(e, "metadata creation");
  }
  *out = m;
  return MLORA_OK;
}

mlora_status mlora_meta_destroy(mlora_meta_t m) {
  if (!m) return MLORA_OK;
  if (m->done) {
    cudaEventSynchronize(m->done);
    cudaEventDestroy(m->done);
  }
  cudaFree(m->order);
  cudaFree(m->seg_slot);
  cudaFree(m->seg_off);
  cudaFree(m->pair_slot);
  cudaFree(m->pair_scale);
  cudaFree(m->blk_slot);
  cudaFree(m->blk_start);
  cudaFree(m->blk_count);
  cudaFree(m->counts);
  cudaFree(m->err);
  cudaFree(m->vpart);
  cudaFree(m->vfull);
  cudaFree(m->pair_act);
  cudaFree(m->act_slot);
  cudaFree(m->tile_unit_off);
  cudaFree(m->unit_blk);
  cudaFree(m->unit_tile);
  cudaFree(m->grp_mp);
  cudaFree(m->grp_ent);
  cudaFree(m->grp_cnt);
  cudaFree(m->ptile_off);
  cudaFree(m->pent_blk);
  cudaFree(m->pent_u0);
  cudaFree(m->pent_u1);
  cudaFree(m->ptile_order);
  cudaFree(m->sync);
  cudaFree(m->pair_fused);
  cudaFree(m->todo_blk);
  cudaFree(m->vtile);
  delete m;
  return MLORA_OK;
}

mlora_status mlora_build_meta(mlora_meta_t m, const int32_t* token_slots, const float* scales, int T, int J,
                              mlora_pool_t pool, void* stream) {
  if (!m || !pool) return fail(MLORA_ERR_INVALID_ARG, "meta or pool is NULL");
  if (T < 0 || J < 1) return fail(MLORA_ERR_INVALID_ARG, "T %d must be >= 0 and J %d >= 1", T, J);
  if (T > m->max_tokens || J > m->J_max)
    return fail(MLORA_ERR_TOO_MANY_TOKENS, "T=%d, J=%d exceed the metadata's %d tokens x %d slots", T, J,
                m->max_tokens, m->J_max);
  if (T > 0 && !token_slots) return fail(MLORA_ERR_INVALID_ARG, "token_slots is NULL");
  if (pool->R > m->R_max)
    return fail(MLORA_ERR_MISMATCH, "pool rank width %d exceeds the metadata's %d", pool->R, m->R_max);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (mlora_status st = pool_use(pool, s)) return st;
  m->T = T;
  m->J = J;
  m->S = pool->S;
  m->class_slots = pool->class_slots;
  m->class_rank = pool->class_rank;
  MetaView v = m->view();
  // the sort only: the tensor-core side path's unit lists are built by the first linear that
  // takes that path (small-batch steps never need them)
  cudaError_t e = launch_build_meta(token_slots, scales, T, J, pool->view(), v, s, kMetaSortOnly);
  if (e != cudaSuccess) return cuda_fail(e, "build_meta launch");
  m->last_stream = s;
  m->built = true;
  m->units_built = false;
  return MLORA_OK;
}

// Waits for every call queued so far on the metadata's last stream.
static mlora_status meta_sync(mlora_meta_t m) {
  MLORA_CUDA(cudaEventRecord(m->done, m->last_stream), "record meta event");
  MLORA_CUDA(cudaEventSynchronize(m->done), "meta sync");
  return MLORA_OK;
}

mlora_status mlora_meta_status(mlora_meta_t m) {
  if (!m) return fail(MLORA_ERR_INVALID_ARG, "meta is NULL");
  if (mlora_status st = meta_sync(m)) return st;
  uint32_t err = 0, gerr = 0;
  int32_t counts[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  MLORA_CUDA(cudaMemcpy(&err, m->err, 4, cudaMemcpyDeviceToHost), "read meta error word");
  MLORA_CUDA(cudaMemcpy(counts, m->counts, 32, cudaMemcpyDeviceToHost), "read meta counts");
  DeviceState* ds = nullptr;
  if (mlora_status st = device_state(&ds)) return st;
  MLORA_CUDA(cudaMemcpy(&gerr, ds->err, 4, cudaMemcpyDeviceToHost), "read device error word");
  if (err) MLORA_CUDA(cudaMemset(m->err, 0, 4), "clear meta error word");
  if (gerr) MLORA_CUDA(cudaMemset(ds->err, 0, 4), "clear device error word");
  if ((err | gerr) & ptx::kErrWaitTimeout)
    return fail(MLORA_ERR_DEVICE_TIMEOUT, "a kernel's bounded wait timed out");
  if (err & ptx::kErrBadSlot) {
    const int p = counts[3];
    return fail(MLORA_ERR_BAD_TOKEN_SLOT, "pair %d (token %d, slot index %d) names an invalid or empty slot", p,
                m->J > 0 ? p / m->J : p, m->J > 0 ? p % m->J : 0);
  }
  if (err & ptx::kErrBadId) return fail(MLORA_ERR_BAD_TOKEN_ID, "a token id lies outside the embedding table");
  if ((err | gerr) & ptx::kErrShape) return fail(MLORA_ERR_INVALID_ARG, "a kernel saw unsupported sizes");
  return MLORA_OK;
}

mlora_status mlora_meta_read(mlora_meta_t m, int32_t* order, int32_t* seg_slot, int32_t* seg_off, int* n_seg,
                             int* n_active) {
  if (!m) return fail(MLORA_ERR_INVALID_ARG, "meta is NULL");
  if (!m->built) return fail(MLORA_ERR_INVALID_ARG, "metadata has not been built");
  if (mlora_status st = meta_sync(m)) return st;
  int32_t counts[8];
  MLORA_CUDA(cudaMemcpy(counts, m->counts, 32, cudaMemcpyDeviceToHost), "read counts");
  const size_t n = static_cast<size_t>(m->T) * m->J;
  if (order && n) MLORA_CUDA(cudaMemcpy(order, m->order, n * 4, cudaMemcpyDeviceToHost), "read order");
  if (seg_slot && counts[0])
    MLORA_CUDA(cudaMemcpy(seg_slot, m->seg_slot, static_cast<size_t>(counts[0]) * 4, cudaMemcpyDeviceToHost),
               "read seg_slot");
  if (seg_off)
    MLORA_CUDA(cudaMemcpy(seg_off, m->seg_off, static_cast<size_t>(counts[0] + 1) * 4, cudaMemcpyDeviceToHost),
               "read seg_off");
  if (n_seg) *n_seg = counts[0];
  if (n_active) *n_active = counts[1];
  return MLORA_OK;
}

// ---------------------------------------------------------------- the layer
static mlora_status check_operands(const void* x, const void* W, const void* y, int T, int K, int D) {
  if (T > 0 && (!x || !y)) return fail(MLORA_ERR_INVALID_ARG, "x or y is NULL");
  if (D > 0 && !W) return fail(MLORA_ERR_INVALID_ARG, "W is NULL");
  if (K < 8 || K % 8) return fail(MLORA_ERR_INVALID_ARG, "K %d must be a positive multiple of 8", K);
  if ((x && !aligned16(x)) || (W && !aligned16(W)) || (y && !aligned16(y)))
    return fail(MLORA_ERR_INVALID_ARG, "x, W and y must be 16-byte aligned");
  return MLORA_OK;
}

mlora_status mlora_base_gemm(const mlora_bf16* x, const mlora_bf16* W, float* y, int T, int K, int D,
                             void* stream) {
  if (T < 0 || D < 0) return fail(MLORA_ERR_INVALID_ARG, "T %d and D %d must be >= 0", T, D);
  if (mlora_status st = check_operands(x, W, y, T, K, D)) return st;
  DeviceState* ds = nullptr;
  if (mlora_status st = device_state(&ds)) return st;
  cudaError_t e = launch_base_gemm(x, W, y, T, K, D, ds->err, ds->num_sms, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "base GEMM launch");
  return MLORA_OK;
}

static mlora_status check_pair(mlora_pool_t p, mlora_meta_t m) {
  if (!p || !m) return fail(MLORA_ERR_INVALID_ARG, "pool or meta is NULL");
  if (!m->built) return fail(MLORA_ERR_INVALID_ARG, "metadata has not been built");
  if (m->S != p->S)
    return fail(MLORA_ERR_MISMATCH, "metadata was built for %d slots, pool has %d", m->S, p->S);
  if (m->class_slots != p->class_slots || m->class_rank != p->class_rank)
    return fail(MLORA_ERR_MISMATCH, "metadata was built on a pool with other rank classes");
  if (p->R > m->R_max) return fail(MLORA_ERR_MISMATCH, "pool rank width %d exceeds the metadata's %d", p->R, m->R_max);
  return MLORA_OK;
}

mlora_status mlora_lora_shrink(mlora_pool_t p, mlora_meta_t m, const mlora_bf16* x, void* stream) {
  if (p && p->embed) return fail(MLORA_ERR_INVALID_ARG, "an embedding pool: use mlora_embedding");
  if (mlora_status st = check_pair(p, m)) return st;
  if (m->T > 0 && (!x || !aligned16(x))) return fail(MLORA_ERR_INVALID_ARG, "x is NULL or misaligned");
  DeviceState* ds = nullptr;
  if (mlora_status st = device_state(&ds)) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (mlora_status st = pool_use(p, s)) return st;
  cudaError_t e = launch_lora_shrink(x, p->view(), m->view(), ds->num_sms, s);
  if (e != cudaSuccess) return cuda_fail(e, "shrink launch");
  m->last_stream = s;
  return MLORA_OK;
}

mlora_status mlora_lora_expand(mlora_pool_t p, mlora_meta_t m, float* y, void* stream) {
  if (p && p->embed) return fail(MLORA_ERR_INVALID_ARG, "an embedding pool: use mlora_embedding");
  if (mlora_status st = check_pair(p, m)) return st;
  if (m->T > 0 && (!y || !aligned16(y))) return fail(MLORA_ERR_INVALID_ARG, "y is NULL or misaligned");
  DeviceState* ds = nullptr;
  if (mlora_status st = device_state(&ds)) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (mlora_status st = pool_use(p, s)) return st;
  cudaError_t e = launch_lora_expand(y, p->view(), m->view(), ds->num_sms, s);
  if (e != cudaSuccess) return cuda_fail(e, "expand launch");
  m->last_stream = s;
  return MLORA_OK;
}

mlora_status mlora_linear(mlora_pool_t p, mlora_meta_t m, const mlora_bf16* x, const mlora_bf16* W, float* y,
                          void* stream) {
  if (p && p->embed) return fail(MLORA_ERR_INVALID_ARG, "an embedding pool: use mlora_embedding");
  if (mlora_status st = check_pair(p, m)) return st;
  if (mlora_status st = check_operands(x, W, y, m->T, p->K, p->D)) return st;
  DeviceState* ds = nullptr;
  if (mlora_status st = device_state(&ds)) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (mlora_status st = pool_use(p, s)) return st;
  const MetaView mv = m->view();
  const PoolView pv = p->view();
  cudaError_t e = cudaSuccess;
  if (m->T == 0) {
    m->last_stream = s;
    return MLORA_OK;
  }
  const int path = g_path.load(std::memory_order_relaxed);
  const bool small_ok = p->uniform() && skinny_shrink_fusable(m->T, m->J, p->S, p->R, m->vfull_ld) &&
                        (p->D + 127) / 128 <= ds->num_sms;
  // the small-batch kernel multiplies every token by every active slot's rows: worth it while
  // those rows add at most half of the output's 128-row blocks
  const long act_blocks = (static_cast<long>(std::min(p->S, m->T * m->J)) * p->R + 127) / 128;
  const bool small = small_ok && (path == 1 || (path == 0 && 2 * act_blocks <= (p->D + 127) / 128));
  if (small) {
    // small batch whose 128-column output blocks fit in one wave: one split-K tensor-core kernel
    // for the base product and the shrink of every active slot, then the expand as its
    // programmatic dependent
    if ((e = launch_gemm_shrink_fused(x, W, y, pv, mv, ds->err, ds->num_sms, s)) != cudaSuccess)
      return cuda_fail(e, "fused GEMM launch");
    if ((e = launch_lora_expand_vfull(y, pv, mv, ds->num_sms, s)) != cudaSuccess) return cuda_fail(e, "expand launch");
  } else {
    // tensor-core side path: the shrink of every unit (M-tile, column block), then the base GEMM
    // with the expand as extra K blocks; the CUDA-core kernels take the pairs of M-tiles that
    // overflow the unit lists, and are launched only when the sizes allow an overflow
    if (!m->units_built) {
      if ((e = launch_build_meta(nullptr, nullptr, m->T, m->J, pv, mv, s, kMetaUnitsOnly)) != cudaSuccess)
        return cuda_fail(e, "unit lists launch");
      m->units_built = true;
    }
    // (the CTA-pair GEMM computes the shrink itself, as tiles of its own schedule, for K <= 8192)
    const bool fused_shrink = base_gemm_uses_pair(m->T) && pair_gemm_fuses_shrink(p->K);
    if (!fused_shrink && (e = launch_lora_shrink_tc(x, pv, mv, ds->err, ds->num_sms, s)) != cudaSuccess)
      return cuda_fail(e, "tensor-core shrink launch");
    if ((e = launch_base_gemm_lora(x, W, y, m->T, p->K, p->D, ds->err, ds->num_sms, &pv, &mv, s)) != cudaSuccess)
      return cuda_fail(e, "base GEMM launch");
    const long n_blocks = (p->C + kBlockCols - 1) / kBlockCols;
    const long per_tile = std::min(128L * m->J * p->max_span, n_blocks);
    const long n_tiles = (m->T + 127) / 128;
    const bool overflow = per_tile > kMaxTileUnits ||
                          (n_tiles * per_tile > m->unit_cap && static_cast<long>(m->T) * m->J * p->max_span > m->unit_cap);
    if (overflow) {
      if ((e = launch_lora_shrink(x, pv, mv, ds->num_sms, s, true)) != cudaSuccess) return cuda_fail(e, "shrink launch");
      if ((e = launch_lora_expand(y, pv, mv, ds->num_sms, s, true)) != cudaSuccess) return cuda_fail(e, "expand launch");
    }
  }
  m->last_stream = s;
  return MLORA_OK;
}

mlora_status mlora_embedding(mlora_pool_t p, mlora_meta_t m, const int32_t* ids, const mlora_bf16* E, float* y,
                             void* stream) {
  if (p && !p->embed) return fail(MLORA_ERR_INVALID_ARG, "not an embedding pool (mlora_embedding_pool_create)");
  if (mlora_status st = check_pair(p, m)) return st;
  if (m->T > 0 && (!ids || !E || !y)) return fail(MLORA_ERR_INVALID_ARG, "ids, E or y is NULL");
  if ((E && !aligned16(E)) || (y && !aligned16(y))) return fail(MLORA_ERR_INVALID_ARG, "E and y must be 16-byte aligned");
  DeviceState* ds = nullptr;
  if (mlora_status st = device_state(&ds)) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (mlora_status st = pool_use(p, s)) return st;
  cudaError_t e = launch_embedding(ids, E, y, p->view(), m->view(), ds->num_sms, s);
  if (e != cudaSuccess) return cuda_fail(e, "embedding launch");
  m->last_stream = s;
  return MLORA_OK;
}

// ---------------------------------------------------------------- trace
mlora_status mlora_trace_enable(int capacity) {
  if (capacity < 1) return fail(MLORA_ERR_INVALID_ARG, "capacity must be positive");
  std::lock_guard<std::mutex> lk(g_trace.mu);
  while (g_trace.recs.size() < static_cast<size_t>(capacity)) {
    TraceRec r{0, nullptr, nullptr};
    MLORA_CUDA(cudaEventCreate(&r.begin), "trace event");
    MLORA_CUDA(cudaEventCreate(&r.end), "trace event");
    g_trace.recs.push_back(r);
  }
  g_trace.used = 0;
  g_trace.pending_begin = SIZE_MAX;
  g_trace.on = true;
  return MLORA_OK;
}

mlora_status mlora_trace_disable(void) {
  std::lock_guard<std::mutex> lk(g_trace.mu);
  g_trace.on = false;
  return MLORA_OK;
}

mlora_status mlora_trace_read(int n_kinds, int* launches, double* total_ms) {
  if (n_kinds < 0 || (n_kinds > 0 && (!launches || !total_ms))) return fail(MLORA_ERR_INVALID_ARG, "bad arrays");
  std::lock_guard<std::mutex> lk(g_trace.mu);
  for (int k = 0; k < n_kinds; ++k) {
    launches[k] = 0;
    total_ms[k] = 0.0;
  }
  for (size_t i = 0; i < g_trace.used; ++i) {
    const TraceRec& r = g_trace.recs[i];
    MLORA_CUDA(cudaEventSynchronize(r.end), "trace sync");
    float ms = 0.f;
    MLORA_CUDA(cudaEventElapsedTime(&ms, r.begin, r.end), "trace elapsed");
    if (r.kind < n_kinds) {
      launches[r.kind] += 1;
      total_ms[r.kind] += ms;
    }
  }
  g_trace.used = 0;
  return MLORA_OK;
}

}  // extern "C"
