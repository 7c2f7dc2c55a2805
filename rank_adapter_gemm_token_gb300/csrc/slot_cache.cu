// Slot residency: which adapter id sits in which GPU slot, with least-recently-used eviction, and
// an adapter cache that loads missing adapters into every pool of a model before a step.
//
// "LoRA Serving" (vLLM learning book, ch. 09-04), section 4.1: activating an adapter copies its
// weights into a free GPU slot; section 5: the LRU cache model manager marks a hit as recent and
// on a miss evicts the oldest adapter that is not pinned, then loads the new one. "Multi-LoRA
// Serving Explained" (sevydevy.com), serving section: adapters live on disk, in a CPU cache and in
// a fixed number of GPU slots, and each level pushes out the least recently used one when full.
// "LLM LoRA Adapter Cache in Production" (oh-bug.com), cache-architecture section: a GPU hot tier
// of bounded capacity above a CPU warm tier.
//
// Host code only (no kernel); the loads use mlora_load_adapter on each pool's copy stream, so they
// run asynchronously and the next mlora_linear on a pool orders itself after them.
#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <mutex>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "internal.h"
#include "mlora.h"

struct mlora_slot_cache {
  int S = 0;
  std::vector<int64_t> id_of;                 // [S] adapter id in the slot, -1 = free
  std::vector<uint64_t> last_use;             // [S] step counter of the last step that used it
  std::unordered_set<int64_t> pinned;         // ids never evicted while resident
  std::unordered_map<int64_t, int> slot_of;   // resident id -> slot
  uint64_t tick = 0;                          // steps assigned so far
  std::mutex mu;
};

struct mlora_adapter_cache {
  struct Entry {
    std::vector<const mlora_bf16*> A, B;      // one host buffer per pool (caller-owned)
    int rank = 0;
    float alpha = 0.f;
    int rslora = 0;
  };
  std::vector<mlora_pool_t> pools;
  mlora_slot_cache lru;
  std::unordered_map<int64_t, Entry> registry;
  uint64_t loads = 0;
  std::mutex mu;
};

namespace {

using mlora::report_error;

// The slot assignment of one step (mu held). Resident ids keep their slot; each other id takes
// the lowest free slot, else the slot whose last use is oldest (lowest index on ties) among the
// slots no id of this step uses and no pinned id holds. On any failure (more distinct ids than
// slots, or pinned slots leaving too few) nothing changes. Returns the loads to perform as
// (id, slot) in first-seen order.
mlora_status lru_assign(mlora_slot_cache& c, const int64_t* ids, int n, int32_t* slots,
                        std::vector<std::pair<int64_t, int>>* loads) {
  std::vector<int64_t> distinct;
  std::unordered_set<int64_t> seen;
  for (int i = 0; i < n; ++i) {
    if (ids[i] < -1) return report_error(MLORA_ERR_INVALID_ARG, "adapter ids must be >= 0 (or -1 for none)");
    if (ids[i] >= 0 && seen.insert(ids[i]).second) distinct.push_back(ids[i]);
  }
  if (static_cast<int>(distinct.size()) > c.S)
    return report_error(MLORA_ERR_NO_FREE_SLOT, "the step names more distinct adapters than there are slots");
  // work on copies; commit only when every id has a slot
  std::vector<int64_t> id_of = c.id_of;
  std::vector<uint64_t> last_use = c.last_use;
  std::unordered_map<int64_t, int> slot_of = c.slot_of;
  const uint64_t now = c.tick + 1;
  for (int64_t id : distinct) {
    auto it = slot_of.find(id);
    if (it != slot_of.end()) last_use[it->second] = now;          // resident: keep it this step
  }
  std::vector<std::pair<int64_t, int>> placed;
  for (int64_t id : distinct) {
    if (slot_of.count(id)) continue;
    int best = -1;
    for (int s = 0; s < c.S; ++s) {
      if (id_of[s] == -1) {
        best = s;
        break;
      }
      if (last_use[s] < now && !c.pinned.count(id_of[s]) && (best < 0 || last_use[s] < last_use[best])) best = s;
    }
    if (best < 0) return report_error(MLORA_ERR_NO_FREE_SLOT, "every slot holds a pinned or requested adapter");
    if (id_of[best] != -1) slot_of.erase(id_of[best]);            // evict the least recently used
    id_of[best] = id;
    last_use[best] = now;
    slot_of[id] = best;
    placed.emplace_back(id, best);
  }
  c.id_of.swap(id_of);
  c.last_use.swap(last_use);
  c.slot_of.swap(slot_of);
  c.tick = now;
  if (loads) *loads = std::move(placed);
  for (int i = 0; i < n; ++i) slots[i] = ids[i] < 0 ? -1 : c.slot_of[ids[i]];
  return MLORA_OK;
}

}  // namespace

using namespace mlora;

extern "C" {

mlora_status mlora_slot_cache_create(int n_slots, mlora_slot_cache_t* out) {
  if (!out) return report_error(MLORA_ERR_INVALID_ARG, "out is NULL");
  if (n_slots < 1 || n_slots > MLORA_MAX_SLOTS) return report_error(MLORA_ERR_INVALID_ARG, "n_slots outside [1, 2048]");
  mlora_slot_cache* c = new (std::nothrow) mlora_slot_cache();
  if (!c) return report_error(MLORA_ERR_OOM, "host allocation failed");
  c->S = n_slots;
  c->id_of.assign(n_slots, -1);
  c->last_use.assign(n_slots, 0);
  *out = c;
  return MLORA_OK;
}

mlora_status mlora_slot_cache_destroy(mlora_slot_cache_t c) {
  delete c;
  return MLORA_OK;
}

mlora_status mlora_slot_cache_assign(mlora_slot_cache_t c, const int64_t* ids, int n, int32_t* slots,
                                     int64_t* load_ids, int32_t* load_slots, int* n_loads) {
  if (!c || n < 0 || (n > 0 && (!ids || !slots))) return report_error(MLORA_ERR_INVALID_ARG, "bad arguments");
  std::lock_guard<std::mutex> lk(c->mu);
  std::vector<std::pair<int64_t, int>> loads;
  if (mlora_status st = lru_assign(*c, ids, n, slots, &loads)) return st;
  for (size_t i = 0; i < loads.size(); ++i) {
    if (load_ids) load_ids[i] = loads[i].first;
    if (load_slots) load_slots[i] = loads[i].second;
  }
  if (n_loads) *n_loads = static_cast<int>(loads.size());
  return MLORA_OK;
}

mlora_status mlora_slot_cache_lookup(mlora_slot_cache_t c, int64_t id, int32_t* slot) {
  if (!c || !slot) return report_error(MLORA_ERR_INVALID_ARG, "bad arguments");
  std::lock_guard<std::mutex> lk(c->mu);
  auto it = c->slot_of.find(id);
  *slot = it == c->slot_of.end() ? -1 : it->second;
  return MLORA_OK;
}

mlora_status mlora_slot_cache_pin(mlora_slot_cache_t c, int64_t id, int pinned) {
  if (!c || id < 0) return report_error(MLORA_ERR_INVALID_ARG, "bad arguments");
  std::lock_guard<std::mutex> lk(c->mu);
  if (pinned) c->pinned.insert(id);
  else c->pinned.erase(id);
  return MLORA_OK;
}

mlora_status mlora_slot_cache_evict(mlora_slot_cache_t c, int64_t id) {
  if (!c) return report_error(MLORA_ERR_INVALID_ARG, "cache is NULL");
  std::lock_guard<std::mutex> lk(c->mu);
  auto it = c->slot_of.find(id);
  if (it != c->slot_of.end()) {
    c->id_of[it->second] = -1;
    c->last_use[it->second] = 0;
    c->slot_of.erase(it);
  }
  return MLORA_OK;
}

mlora_status mlora_adapter_cache_create(const mlora_pool_t* pools, int n_pools, mlora_adapter_cache_t* out) {
  if (!out || !pools || n_pools < 1) return report_error(MLORA_ERR_INVALID_ARG, "pools or out is NULL");
  int S = 0;
  for (int i = 0; i < n_pools; ++i) {
    int s = 0;
    if (!pools[i] || mlora_pool_info(pools[i], &s, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr))
      return report_error(MLORA_ERR_INVALID_ARG, "a pool is NULL");
    if (i > 0 && s != S) return report_error(MLORA_ERR_MISMATCH, "the pools of one cache must have the same n_slots");
    S = s;
  }
  mlora_adapter_cache* c = new (std::nothrow) mlora_adapter_cache();
  if (!c) return report_error(MLORA_ERR_OOM, "host allocation failed");
  c->pools.assign(pools, pools + n_pools);
  c->lru.S = S;
  c->lru.id_of.assign(S, -1);
  c->lru.last_use.assign(S, 0);
  *out = c;
  return MLORA_OK;
}

mlora_status mlora_adapter_cache_destroy(mlora_adapter_cache_t c) {
  delete c;
  return MLORA_OK;
}

mlora_status mlora_adapter_cache_register(mlora_adapter_cache_t c, int64_t id, const mlora_bf16* const* A_host,
                                          const mlora_bf16* const* B_host, int rank, float alpha, int rslora) {
  if (!c || id < 0 || !A_host || !B_host) return report_error(MLORA_ERR_INVALID_ARG, "bad arguments");
  mlora_adapter_cache::Entry e;
  for (size_t i = 0; i < c->pools.size(); ++i) {
    if (!A_host[i] || !B_host[i]) return report_error(MLORA_ERR_INVALID_ARG, "an A or B buffer is NULL");
    e.A.push_back(A_host[i]);
    e.B.push_back(B_host[i]);
  }
  e.rank = rank;
  e.alpha = alpha;
  e.rslora = rslora;
  std::lock_guard<std::mutex> lk(c->mu);
  c->registry[id] = std::move(e);
  // a new version of a resident adapter: drop the stale copy so the next step loads this one
  std::lock_guard<std::mutex> lk2(c->lru.mu);
  auto it = c->lru.slot_of.find(id);
  if (it != c->lru.slot_of.end()) {
    c->lru.id_of[it->second] = -1;
    c->lru.last_use[it->second] = 0;
    c->lru.slot_of.erase(it);
  }
  return MLORA_OK;
}

mlora_status mlora_adapter_cache_unregister(mlora_adapter_cache_t c, int64_t id) {
  if (!c) return report_error(MLORA_ERR_INVALID_ARG, "cache is NULL");
  std::lock_guard<std::mutex> lk(c->mu);
  c->registry.erase(id);
  std::lock_guard<std::mutex> lk2(c->lru.mu);
  auto it = c->lru.slot_of.find(id);
  if (it != c->lru.slot_of.end()) {
    c->lru.id_of[it->second] = -1;
    c->lru.last_use[it->second] = 0;
    c->lru.slot_of.erase(it);
  }
  c->lru.pinned.erase(id);
  return MLORA_OK;
}

mlora_status mlora_adapter_cache_pin(mlora_adapter_cache_t c, int64_t id, int pinned) {
  if (!c) return report_error(MLORA_ERR_INVALID_ARG, "cache is NULL");
  return mlora_slot_cache_pin(&c->lru, id, pinned);
}

mlora_status mlora_adapter_cache_map(mlora_adapter_cache_t c, const int64_t* ids, int n, int32_t* token_slots,
                                     int* n_loaded) {
  if (!c || n < 0 || (n > 0 && (!ids || !token_slots))) return report_error(MLORA_ERR_INVALID_ARG, "bad arguments");
  std::lock_guard<std::mutex> lk(c->mu);
  for (int i = 0; i < n; ++i)
    if (ids[i] >= 0 && !c->registry.count(ids[i])) {
      char msg[160];
      snprintf(msg, sizeof msg, "entry %d names adapter id %lld, which is not registered", i,
               static_cast<long long>(ids[i]));
      return report_error(MLORA_ERR_INVALID_ARG, msg);
    }
  std::vector<std::pair<int64_t, int>> loads;
  {
    std::lock_guard<std::mutex> lk2(c->lru.mu);
    if (mlora_status st = lru_assign(c->lru, ids, n, token_slots, &loads)) return st;
  }
  for (size_t k = 0; k < loads.size(); ++k) {         // queue the copies on every pool's copy stream
    const mlora_adapter_cache::Entry& e = c->registry[loads[k].first];
    for (size_t p = 0; p < c->pools.size(); ++p) {
      const mlora_status st =
          mlora_load_adapter(c->pools[p], loads[k].second, e.A[p], e.B[p], e.rank, e.alpha, e.rslora);
      if (st != MLORA_OK) {
        std::lock_guard<std::mutex> lk2(c->lru.mu);   // slots not (fully) loaded: free them again
        for (size_t q = k; q < loads.size(); ++q) {
          c->lru.id_of[loads[q].second] = -1;
          c->lru.last_use[loads[q].second] = 0;
          c->lru.slot_of.erase(loads[q].first);
        }
        return st;
      }
    }
  }
  c->loads += loads.size();
  if (n_loaded) *n_loaded = static_cast<int>(loads.size());
  return MLORA_OK;
}

}  // extern "C"
