// Slot table: the device expert cache.
//
// "Strata 工作原理图解GPU内存SSD三级存储如何让125B模型塞进消费级显卡", sections "三级存储分工" and
// "专家缓存": the most used experts stay in VRAM and all experts sit pinned in host RAM. Experts
// are cached one at a time, not one layer at a time. Section "长文本": expert copies over PCIe
// overlap with computation.
//
// Host state: the owner (layer, expert) of each of n_slots device slots, an LRU list of
// slots (head = least recently used), and a host mirror of the device table slot_of[L][E].
// A miss takes the least recently used slot that the current call does not need. The
// record is copied from pinned host memory on the caller's copy stream. Every table entry
// that changed (the new owner, and the evicted owner in whatever layer it belonged to) is
// then written to the device table on the same stream, so a compute stream that waits on
// `ready` sees a table that matches the slot contents.
//
// Protocol: call slot_table_update for a layer only after the computation that read the
// slots of the previous update has completed (e.g. the host waited on an event recorded
// after it). An eviction may otherwise overwrite a slot that a kernel is still reading.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <vector>

#include "../../include/moe.h"

struct moe_slot_table {
  int32_t L = 0, E = 0, n_slots = 0;
  uint64_t slot_bytes = 0;
  char* d_pool = nullptr;
  int32_t* d_slot_of = nullptr;
  std::vector<const void*> h_records;
  moe_copy_fn copy_fn = nullptr;
  void* copy_user = nullptr;
  bool default_copier = true;
  int32_t* mirror = nullptr;  // host mirror of slot_of [L*E]; pinned with the default copier
  std::vector<int64_t> owner;  // [n_slots]: l*E + e, or -1 when empty
  std::vector<int32_t> prev, next;  // LRU list over slots
  int32_t head = -1, tail = -1;
  std::vector<uint32_t> mark;  // [E] epoch marks: expert is in the current call's active set
  uint32_t epoch = 0;
  moe_slot_stats stats{};
};

namespace {

thread_local char g_slot_err[256] = "";

int cuda_copy(void* dst, const void* src, size_t bytes, moe_stream_t stream, void*) {
  return (int)cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, reinterpret_cast<cudaStream_t>(stream));
}

void lru_unlink(moe_slot_table* t, int32_t s) {
  const int32_t p = t->prev[s], n = t->next[s];
  if (p >= 0) t->next[p] = n; else t->head = n;
  if (n >= 0) t->prev[n] = p; else t->tail = p;
  t->prev[s] = t->next[s] = -1;
}

void lru_push_tail(moe_slot_table* t, int32_t s) {
  t->prev[s] = t->tail;
  t->next[s] = -1;
  if (t->tail >= 0) t->next[t->tail] = s; else t->head = s;
  t->tail = s;
}

// Write the changed entries of the device table, one copy per run of adjacent keys.
int write_entries(moe_slot_table* t, std::vector<int64_t>& keys, moe_stream_t stream) {
  if (!t->d_slot_of || keys.empty()) return 0;
  std::sort(keys.begin(), keys.end());
  keys.erase(std::unique(keys.begin(), keys.end()), keys.end());
  size_t i = 0;
  while (i < keys.size()) {
    size_t j = i + 1;
    while (j < keys.size() && keys[j] == keys[j - 1] + 1) ++j;
    const int64_t k0 = keys[i];
    const size_t n = j - i;
    const int rc = t->copy_fn(t->d_slot_of + k0, t->mirror + k0, n * sizeof(int32_t), stream, t->copy_user);
    if (rc != 0) return rc;
    i = j;
  }
  return 0;
}

}  // namespace

extern "C" {

moe_status slot_table_create(moe_slot_table** out, int32_t L, int32_t E, int32_t n_slots, uint64_t slot_bytes,
                             void* d_pool, int32_t* d_slot_of, const void* const* h_records, moe_copy_fn copy_fn,
                             void* copy_user) {
  if (!out || L <= 0 || E <= 0 || n_slots <= 0 || slot_bytes == 0 || !h_records) return MOE_EINVAL;
  if ((int64_t)L * E > (int64_t)1 << 30) return MOE_EUNSUPPORTED;
  if (!copy_fn && (!d_pool || !d_slot_of)) return MOE_EINVAL;
  for (int64_t i = 0; i < (int64_t)L * E; ++i)
    if (!h_records[i]) return MOE_EINVAL;
  moe_slot_table* t = new moe_slot_table();
  t->L = L;
  t->E = E;
  t->n_slots = n_slots;
  t->slot_bytes = slot_bytes;
  t->d_pool = static_cast<char*>(d_pool);
  t->d_slot_of = d_slot_of;
  t->h_records.assign(h_records, h_records + (size_t)L * E);
  t->default_copier = copy_fn == nullptr;
  t->copy_fn = copy_fn ? copy_fn : cuda_copy;
  t->copy_user = copy_user;
  const size_t mbytes = sizeof(int32_t) * (size_t)L * E;
  if (t->default_copier) {
    if (cudaMallocHost(reinterpret_cast<void**>(&t->mirror), mbytes) != cudaSuccess) {
      delete t;
      return MOE_ECUDA;
    }
  } else {
    t->mirror = static_cast<int32_t*>(std::malloc(mbytes));
  }
  for (size_t i = 0; i < (size_t)L * E; ++i) t->mirror[i] = -1;
  t->owner.assign(n_slots, -1);
  t->prev.assign(n_slots, -1);
  t->next.assign(n_slots, -1);
  for (int32_t s = 0; s < n_slots; ++s) lru_push_tail(t, s);
  t->mark.assign(E, 0);
  if (d_slot_of) {
    if (t->default_copier) {
      if (cudaMemcpy(d_slot_of, t->mirror, mbytes, cudaMemcpyHostToDevice) != cudaSuccess) {
        cudaFreeHost(t->mirror);
        delete t;
        return MOE_ECUDA;
      }
    } else if (t->copy_fn(d_slot_of, t->mirror, mbytes, nullptr, t->copy_user) != 0) {
      std::free(t->mirror);
      delete t;
      return MOE_ECUDA;
    }
  }
  *out = t;
  return MOE_OK;
}

moe_status slot_table_update(moe_slot_table* t, int32_t layer, const int32_t* h_active, int32_t n_active,
                             moe_stream_t copy_stream, moe_event_t ready, int32_t* h_hits, int32_t* n_hits,
                             int32_t* h_misses, int32_t* n_misses, moe_slot_stats* stats_opt) {
  if (!t || layer < 0 || layer >= t->L || n_active < 0 || (n_active > 0 && !h_active)) return MOE_EINVAL;
  // validate ids, reject repeats (epoch marks)
  if (++t->epoch == 0) {
    std::fill(t->mark.begin(), t->mark.end(), 0);
    t->epoch = 1;
  }
  for (int32_t i = 0; i < n_active; ++i) {
    const int32_t e = h_active[i];
    if (e < 0 || e >= t->E || t->mark[e] == t->epoch) return MOE_EINVAL;
    t->mark[e] = t->epoch;
  }
  const int64_t base = (int64_t)layer * t->E;
  int32_t nh = 0, nm = 0;
  for (int32_t i = 0; i < n_active; ++i) (t->mirror[base + h_active[i]] >= 0 ? nh : nm)++;
  if (nm > t->n_slots - nh) {
    std::snprintf(g_slot_err, sizeof(g_slot_err), "%d misses, %d evictable slots", nm, t->n_slots - nh);
    return MOE_ENOSLOT;
  }
  // hits first: most recently used, so that no miss evicts them
  nh = nm = 0;
  for (int32_t i = 0; i < n_active; ++i) {
    const int32_t e = h_active[i];
    const int32_t s = t->mirror[base + e];
    if (s >= 0) {
      lru_unlink(t, s);
      lru_push_tail(t, s);
      if (h_hits) h_hits[nh] = e;
      ++nh;
    }
  }
  std::vector<int64_t> changed;
  moe_status rc = MOE_OK;
  for (int32_t i = 0; i < n_active; ++i) {
    const int32_t e = h_active[i];
    if (t->mirror[base + e] >= 0) continue;
    const int32_t s = t->head;  // least recently used; never one of this call's experts
    const int64_t old = t->owner[s];
    if (old >= 0) {
      t->mirror[old] = -1;
      changed.push_back(old);
      t->stats.evictions++;
    }
    t->owner[s] = -1;
    lru_unlink(t, s);
    lru_push_tail(t, s);
    const int cr = t->copy_fn(t->d_pool + (uint64_t)s * t->slot_bytes, t->h_records[base + e], t->slot_bytes,
                              copy_stream, t->copy_user);
    if (cr != 0) {
      std::snprintf(g_slot_err, sizeof(g_slot_err), "copy of expert %d failed (%d)", e, cr);
      rc = MOE_ECUDA;
      break;
    }
    t->owner[s] = base + e;
    t->mirror[base + e] = s;
    changed.push_back(base + e);
    t->stats.misses++;
    t->stats.bytes_h2d += t->slot_bytes;
    if (h_misses) h_misses[nm] = e;
    ++nm;
  }
  t->stats.hits += nh;
  if (write_entries(t, changed, copy_stream) != 0 && rc == MOE_OK) rc = MOE_ECUDA;
  if (ready && cudaEventRecord(reinterpret_cast<cudaEvent_t>(ready), reinterpret_cast<cudaStream_t>(copy_stream)) !=
                   cudaSuccess && rc == MOE_OK)
    rc = MOE_ECUDA;
  if (n_hits) *n_hits = nh;
  if (n_misses) *n_misses = nm;
  if (stats_opt) *stats_opt = t->stats;
  return rc;
}

moe_status slot_table_stats(const moe_slot_table* t, moe_slot_stats* out) {
  if (!t || !out) return MOE_EINVAL;
  *out = t->stats;
  return MOE_OK;
}

moe_status slot_table_snapshot(const moe_slot_table* t, int32_t* h_out) {
  if (!t || !h_out) return MOE_EINVAL;
  std::memcpy(h_out, t->mirror, sizeof(int32_t) * (size_t)t->L * t->E);
  return MOE_OK;
}

moe_status slot_table_destroy(moe_slot_table* t) {
  if (!t) return MOE_EINVAL;
  if (t->default_copier) cudaFreeHost(t->mirror);
  else std::free(t->mirror);
  delete t;
  return MOE_OK;
}

}  // extern "C"
