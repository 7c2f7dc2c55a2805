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

int pad8(int r) { return (r + 7) / 8 * 8; }

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

}  // namespace

namespace mlora {

int report_error(int status, const char* message) { return fail(status, "%s", message); }
int report_cuda_error(cudaError_t e, const char* what) { return cuda_fail(e, what); }
int gemm_tile_n() { return g_gemm_tile_n.load(std::memory_order_relaxed); }

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
  uint16_t* A = nullptr;
  uint16_t* B = nullptr;
  float* slot_scale = nullptr;
  int32_t* slot_rank = nullptr;
  std::vector<int> h_rank;
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

  PoolView view() const { return PoolView{A, B, slot_scale, slot_rank, S, R, K, D}; }
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
  int32_t *tile_info = nullptr, *pair_fused = nullptr, *todo_blk = nullptr;
  uint16_t* vtile = nullptr;
  int T = 0, J = 1, S = -1;
  bool built = false;
  cudaEvent_t done = nullptr;
  cudaStream_t last_stream = nullptr;          // the stream of the last call that used the metadata

  MetaView view() const {
    return MetaView{order, seg_slot, seg_off, pair_slot, pair_scale, blk_slot, blk_start, blk_count, counts,
                    pair_act, act_slot, err, vpart, vfull, vfull_ld, tile_info, pair_fused, todo_blk, vtile,
                    T * J, T, J};
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
    default: return "unknown status";
  }
}

const char* mlora_kernel_kind_name(int kind) {
  static const char* names[kNumKinds] = {"meta", "base_gemm", "shrink", "expand", "slot"};
  return (kind >= 0 && kind < kNumKinds) ? names[kind] : "?";
}

size_t mlora_pool_bytes(int n_slots, int r_max, int K, int D) {
  if (n_slots < 1 || r_max < 1 || K < 1 || D < 1) return 0;
  return static_cast<size_t>(n_slots) * static_cast<size_t>(pad8(r_max)) *
         (static_cast<size_t>(K) + static_cast<size_t>(D)) * 2u;
}

// ---------------------------------------------------------------- pool
mlora_status mlora_pool_create(int n_slots, int r_max, int K, int D, void* copy_stream, mlora_pool_t* out) {
  if (!out) return fail(MLORA_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (n_slots < 1 || n_slots > MLORA_MAX_SLOTS)
    return fail(MLORA_ERR_INVALID_ARG, "n_slots %d outside [1, %d]", n_slots, MLORA_MAX_SLOTS);
  if (r_max < 1 || r_max > MLORA_MAX_RANK)
    return fail(MLORA_ERR_INVALID_ARG, "r_max %d outside [1, %d]", r_max, MLORA_MAX_RANK);
  if (K < 8 || K % 8 != 0) return fail(MLORA_ERR_INVALID_ARG, "K %d must be a positive multiple of 8", K);
  if (D < 1) return fail(MLORA_ERR_INVALID_ARG, "D %d must be positive", D);
  DeviceState* ds = nullptr;
  if (mlora_status st = device_state(&ds)) return st;
  mlora_pool* p = new (std::nothrow) mlora_pool();
  if (!p) return fail(MLORA_ERR_OOM, "host allocation failed");
  cudaGetDevice(&p->device);
  p->S = n_slots;
  p->r_max = r_max;
  p->R = pad8(r_max);
  p->K = K;
  p->D = D;
  p->h_rank.assign(n_slots, 0);
  const size_t a_bytes = static_cast<size_t>(n_slots) * p->R * K * 2;
  const size_t b_bytes = static_cast<size_t>(n_slots) * D * p->R * 2;
  cudaError_t e = cudaSuccess;
  if ((e = cudaMalloc(&p->A, a_bytes)) != cudaSuccess || (e = cudaMalloc(&p->B, b_bytes)) != cudaSuccess ||
      (e = cudaMalloc(&p->slot_scale, n_slots * sizeof(float))) != cudaSuccess ||
      (e = cudaMalloc(&p->slot_rank, n_slots * sizeof(int32_t))) != cudaSuccess) {
    cudaGetLastError();
    mlora_pool_destroy(p);
    return e == cudaErrorMemoryAllocation ? fail(MLORA_ERR_OOM, "cudaMalloc of %zu + %zu bytes failed", a_bytes, b_bytes)
                                          : cuda_fail(e, "cudaMalloc");
  }
  if ((e = cudaMemset(p->A, 0, a_bytes)) != cudaSuccess || (e = cudaMemset(p->B, 0, b_bytes)) != cudaSuccess ||
      (e = cudaMemset(p->slot_scale, 0, n_slots * sizeof(float))) != cudaSuccess ||
      (e = cudaMemset(p->slot_rank, 0, n_slots * sizeof(int32_t))) != cudaSuccess) {
    mlora_pool_destroy(p);
    return cuda_fail(e, "cudaMemset(pool)");
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
  delete p;
  return MLORA_OK;
}

// Writes a slot on the pool's copy stream after every call already queued on the pool: zeroes
// it, then copies n_slices adapters of rank r each; slice i's A [r, K] goes to rows i r .. and its
// B [widths[i], r] to rows off_i .. (off_i = sum of the earlier widths) and columns i r .. of the
// slot's B (block-diagonal; a plain adapter is one slice of width D). n_slices = 0 clears it.
static mlora_status write_slot_sliced(mlora_pool_t p, int slot, int n_slices, const int* widths,
                                      const mlora_bf16* const* A_host, const mlora_bf16* const* B_host, int r,
                                      float alpha, int rslora) {
  cudaStream_t cs = p->copy_stream;
  for (auto& u : p->users) {                   // after every call already queued on the pool
    MLORA_CUDA(cudaEventRecord(p->use_done, u.first), "record use event");
    MLORA_CUDA(cudaStreamWaitEvent(cs, p->use_done, 0), "wait for last use of the pool");
  }
  uint16_t* a_slot = p->A + static_cast<size_t>(slot) * p->R * p->K;
  uint16_t* b_slot = p->B + static_cast<size_t>(slot) * p->D * p->R;
  MLORA_CUDA(cudaMemsetAsync(a_slot, 0, static_cast<size_t>(p->R) * p->K * 2, cs), "zero slot A");
  MLORA_CUDA(cudaMemsetAsync(b_slot, 0, static_cast<size_t>(p->D) * p->R * 2, cs), "zero slot B");
  int off = 0;
  for (int i = 0; i < n_slices; ++i) {
    const int w = widths ? widths[i] : p->D;
    MLORA_CUDA(cudaMemcpyAsync(a_slot + static_cast<size_t>(i) * r * p->K, A_host[i], static_cast<size_t>(r) * p->K * 2,
                               cudaMemcpyHostToDevice, cs),
               "copy A into slot");
    MLORA_CUDA(cudaMemcpy2DAsync(b_slot + static_cast<size_t>(off) * p->R + static_cast<size_t>(i) * r,
                                 static_cast<size_t>(p->R) * 2, B_host[i], static_cast<size_t>(r) * 2,
                                 static_cast<size_t>(r) * 2, static_cast<size_t>(w), cudaMemcpyHostToDevice, cs),
               "copy B into slot");
    off += w;
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

mlora_status mlora_load_adapter(mlora_pool_t p, int slot, const mlora_bf16* A_host, const mlora_bf16* B_host,
                                int rank, float alpha, int rslora) {
  if (!p) return fail(MLORA_ERR_INVALID_ARG, "pool is NULL");
  if (slot < 0 || slot >= p->S) return fail(MLORA_ERR_SLOT_RANGE, "slot %d outside [0, %d)", slot, p->S);
  if (rank < 1 || !std::isfinite(alpha))
    return fail(MLORA_ERR_RANK_INVALID, "rank %d must be >= 1 and alpha finite", rank);
  if (rank > p->r_max)
    return fail(MLORA_ERR_RANK_TOO_LARGE, "adapter rank %d is larger than the pool's max rank %d", rank, p->r_max);
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
  if (static_cast<long>(n_slices) * rank > p->r_max)
    return fail(MLORA_ERR_RANK_TOO_LARGE, "%d slices of rank %d need rank %d, larger than the pool's max rank %d",
                n_slices, rank, n_slices * rank, p->r_max);
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
  m->R_max = pad8(r_max);
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
  // tensor-core prefill path: per-tile slot lists, fused-pair flags, scaled v tiles (bf16)
  const size_t n_tiles = (static_cast<size_t>(max_tokens) + 127) / 128;
  alloc(reinterpret_cast<void**>(&m->tile_info), n_tiles * (kTileSlots + 1) * 4);
  alloc(reinterpret_cast<void**>(&m->pair_fused), n * 4);
  alloc(reinterpret_cast<void**>(&m->todo_blk), n * 4);
  alloc(reinterpret_cast<void**>(&m->vtile), n_tiles * kTileSlots * 128 * 64 * 2);
  // small-batch shrink output: v of every token (up to 256) against every active slot
  const int vt = std::min(max_tokens, kVfullMaxTokens);
  m->vfull_ld = std::min(m->n_max, kVfullMaxAct) * m->R_max;
  alloc(reinterpret_cast<void**>(&m->vfull), static_cast<size_t>(vt) * m->vfull_ld * 4);
  if (e == cudaSuccess) e = cudaMemset(m->err, 0, 4);
  if (e == cudaSuccess) e = cudaMemset(m->counts, 0, 32);
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
  cudaFree(m->tile_info);
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
  MetaView v = m->view();
  cudaError_t e = launch_build_meta(token_slots, scales, T, J, pool->S, pool->slot_rank, v, s);
  if (e != cudaSuccess) return cuda_fail(e, "build_meta launch");
  m->last_stream = s;
  m->built = true;
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
  if (p->R > m->R_max) return fail(MLORA_ERR_MISMATCH, "pool rank width %d exceeds the metadata's %d", p->R, m->R_max);
  return MLORA_OK;
}

mlora_status mlora_lora_shrink(mlora_pool_t p, mlora_meta_t m, const mlora_bf16* x, void* stream) {
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
  if (mlora_status st = check_pair(p, m)) return st;
  if (mlora_status st = check_operands(x, W, y, m->T, p->K, p->D)) return st;
  DeviceState* ds = nullptr;
  if (mlora_status st = device_state(&ds)) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (mlora_status st = pool_use(p, s)) return st;
  const MetaView mv = m->view();
  const PoolView pv = p->view();
  cudaError_t e = cudaSuccess;
  if (skinny_shrink_fusable(m->T, m->J, p->S, p->R, m->vfull_ld) && (p->D + 127) / 128 <= ds->num_sms) {
    // small batch whose 128-column output blocks fit in one wave: one split-K tensor-core kernel
    // for the base product and the shrink of every active slot, then the expand as its
    // programmatic dependent (wider outputs, an LM head for instance, take the tiled GEMM and the
    // separate shrink and expand below)
    if ((e = launch_gemm_shrink_fused(x, W, y, pv, mv, ds->err, ds->num_sms, s)) != cudaSuccess)
      return cuda_fail(e, "fused GEMM launch");
    if ((e = launch_lora_expand_vfull(y, pv, mv, ds->num_sms, s)) != cudaSuccess) return cuda_fail(e, "expand launch");
  } else if (m->T > kSkinnyMaxT && sgmv_tc_supported(p->R)) {
    // larger batch, rank width 64: tiles whose tokens use few slots get the shrink on the tensor
    // cores and the expand as extra K blocks of the base GEMM; the rest take the CUDA-core path
    if ((e = launch_sgmv_shrink_tc(x, pv, mv, ds->err, ds->num_sms, s)) != cudaSuccess) return cuda_fail(e, "SGMV shrink launch");
    if ((e = launch_base_gemm_lora(x, W, y, m->T, p->K, p->D, ds->err, ds->num_sms, &pv, &mv, s)) != cudaSuccess)
      return cuda_fail(e, "base GEMM launch");
    // one or two overflow tiles (decode-like tokens of a mixed batch): the small-batch shrink and
    // expand over those tokens; more overflow tiles: the CUDA-core kernels (each kind does
    // nothing when the other one applies)
    const bool win = window_shrink_supported(m->T, m->J, p->S, p->R, m->vfull_ld,
                                             std::min(m->max_tokens, kVfullMaxTokens));
    if (win) {
      if ((e = launch_gemm_shrink_window(x, pv, mv, ds->err, ds->num_sms, s)) != cudaSuccess)
        return cuda_fail(e, "window shrink launch");
      if ((e = launch_lora_expand_window(y, pv, mv, ds->num_sms, s)) != cudaSuccess)
        return cuda_fail(e, "window expand launch");
    }
    if ((e = launch_lora_shrink(x, pv, mv, ds->num_sms, s, true, win)) != cudaSuccess)
      return cuda_fail(e, "shrink launch");
    if ((e = launch_lora_expand(y, pv, mv, ds->num_sms, s, true, win)) != cudaSuccess)
      return cuda_fail(e, "expand launch");
  } else {
    if ((e = launch_base_gemm(x, W, y, m->T, p->K, p->D, ds->err, ds->num_sms, s)) != cudaSuccess)
      return cuda_fail(e, "base GEMM launch");
    if ((e = launch_lora_shrink(x, pv, mv, ds->num_sms, s)) != cudaSuccess) return cuda_fail(e, "shrink launch");
    if ((e = launch_lora_expand(y, pv, mv, ds->num_sms, s)) != cudaSuccess) return cuda_fail(e, "expand launch");
  }
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
