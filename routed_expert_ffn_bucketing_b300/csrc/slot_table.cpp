// Slot table: the device expert cache.
//
// "Strata 工作原理图解GPU内存SSD三级存储如何让125B模型塞进消费级显卡", sections "三级存储分工" and
// "专家缓存": the most used experts stay in VRAM and all experts sit pinned in host RAM. Experts
// are cached one at a time, not one layer at a time. Section "长文本": expert copies over PCIe
// overlap with computation.
//
// The same section says the cache starts from a shipped ranking of expert use and then learns
// which experts the current session uses most. Two replacement policies:
//   LRU  (default): a miss takes the least recently used slot that the current call does not
//        need;
//   FREQ: a miss takes the slot whose owner has the smallest use count decayed by half every
//        `half_life` update calls (ties: least recently used, then the lowest slot index).
// A profile of use weights can seed the counts and fill the empty slots (slot_table_warm).
//
// Host state: the owner (layer, expert) of each of n_slots device slots, an LRU list of
// slots (head = least recently used), a min-heap of slots by decayed count, the decayed
// count and last use of every (layer, expert), and a host mirror of the device table
// slot_of[L][E]. The record of a miss is copied from pinned host memory on the caller's copy
// stream. Every table entry that changed (the new owner, and the evicted owner in whatever
// layer it belonged to) is then written to the device table on the same stream, so a compute
// stream that waits on `ready` sees a table that matches the slot contents.
//
// Decay without touching every count: a use adds inc = g^c (g = 2^(1/half_life), c the
// number of update calls so far) to the expert's count, which orders counts exactly as
// decayed counts would. When inc passes 2^600 all counts and inc are multiplied by 2^-600
// (exact in binary floating point; counts that underflow were last used hundreds of
// half-lives ago).
//
// Protocol: call slot_table_update for a layer only after the computation that read the
// slots of the previous update has completed (e.g. the host waited on an event recorded
// after it). An eviction may otherwise overwrite a slot that a kernel is still reading.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <vector>

#include "moe_internal.h"

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
  // decayed use counts
  int32_t policy = MOE_SLOT_LRU;
  double g = 1.0, inc = 1.0;   // per-call growth of a use's weight, and the current weight
  int64_t calls = 0;
  std::vector<double> score;     // [L*E]
  std::vector<int64_t> last_use; // [L*E]: call number of the last use, -1 never
  std::vector<int32_t> heap, hpos;  // min-heap of slots by (count, last use, slot); hpos[slot]
  std::vector<uint8_t> pinned;      // [n_slots]: owner is in the current call (never a victim)
  std::vector<uint8_t> prefetched;  // [n_slots]: loaded by slot_table_prefetch, not yet hit
  uint64_t pf_loads = 0, pf_used = 0;
};

namespace {

// Records a formatted message as this thread's moe_last_error_string() and returns st.
moe_status slot_fail(moe_status st, const char* fmt, ...) {
  char buf[256];
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  return moe::report_error(st, buf);
}

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

// Heap order of slots: pinned slots last, empty slots first, then by decayed count, last use
// and slot index.
bool slot_less(const moe_slot_table* t, int32_t a, int32_t b) {
  if (t->pinned[a] != t->pinned[b]) return t->pinned[b];
  if (t->pinned[a]) return a < b;
  const int64_t oa = t->owner[a], ob = t->owner[b];
  if ((oa < 0) != (ob < 0)) return oa < 0;
  if (oa >= 0) {
    if (t->score[oa] != t->score[ob]) return t->score[oa] < t->score[ob];
    if (t->last_use[oa] != t->last_use[ob]) return t->last_use[oa] < t->last_use[ob];
  }
  return a < b;
}

void heap_swap(moe_slot_table* t, int32_t i, int32_t j) {
  std::swap(t->heap[i], t->heap[j]);
  t->hpos[t->heap[i]] = i;
  t->hpos[t->heap[j]] = j;
}

void heap_sift_down(moe_slot_table* t, int32_t i) {
  const int32_t n = (int32_t)t->heap.size();
  for (;;) {
    const int32_t l = 2 * i + 1, r = l + 1;
    int32_t m = i;
    if (l < n && slot_less(t, t->heap[l], t->heap[m])) m = l;
    if (r < n && slot_less(t, t->heap[r], t->heap[m])) m = r;
    if (m == i) break;
    heap_swap(t, i, m);
    i = m;
  }
}

// Restores the heap order after the key of slot s changed. Only valid when no other key has
// changed since the heap was last in order: each change is fixed before the next one.
void heap_fix(moe_slot_table* t, int32_t s) {
  int32_t i = t->hpos[s];
  while (i > 0) {
    const int32_t p = (i - 1) / 2;
    if (!slot_less(t, t->heap[i], t->heap[p])) break;
    heap_swap(t, i, p);
    i = p;
  }
  heap_sift_down(t, i);
}

// Rebuilds the heap bottom-up after many keys changed at once.
void heap_rebuild(moe_slot_table* t) {
  for (int32_t i = (int32_t)t->heap.size() / 2 - 1; i >= 0; --i) heap_sift_down(t, i);
}

// Starts a new update call: the weight of a use grows by g, with the rescale described above.
void advance_clock(moe_slot_table* t) {
  ++t->calls;
  t->inc *= t->g;
  if (t->inc > 0x1p600) {
    for (double& v : t->score) v *= 0x1p-600;
    t->inc *= 0x1p-600;
    heap_rebuild(t);  // counts that underflowed to equal values now tie
  }
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
  if (!out || L <= 0 || E <= 0 || n_slots <= 0 || slot_bytes == 0 || !h_records)
    return slot_fail(MOE_EINVAL, "slot_table_create: null pointer or L, E, n_slots, slot_bytes not > 0");
  if ((int64_t)L * E > (int64_t)1 << 30) return slot_fail(MOE_EUNSUPPORTED, "slot_table_create: L*E above 2^30");
  if (!copy_fn && (!d_pool || !d_slot_of))
    return slot_fail(MOE_EINVAL, "slot_table_create: the default copier needs d_pool and d_slot_of");
  for (int64_t i = 0; i < (int64_t)L * E; ++i)
    if (!h_records[i]) return slot_fail(MOE_EINVAL, "slot_table_create: h_records[%lld] is null", (long long)i);
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
      return slot_fail(MOE_ECUDA, "slot_table_create: cudaMallocHost of the table mirror failed");
    }
  } else {
    t->mirror = static_cast<int32_t*>(std::malloc(mbytes));
    if (!t->mirror) {
      delete t;
      return slot_fail(MOE_EINVAL, "slot_table_create: no host memory for the table mirror");
    }
  }
  for (size_t i = 0; i < (size_t)L * E; ++i) t->mirror[i] = -1;
  t->owner.assign(n_slots, -1);
  t->prev.assign(n_slots, -1);
  t->next.assign(n_slots, -1);
  for (int32_t s = 0; s < n_slots; ++s) lru_push_tail(t, s);
  t->mark.assign(E, 0);
  t->score.assign((size_t)L * E, 0.0);
  t->last_use.assign((size_t)L * E, -1);
  t->pinned.assign(n_slots, 0);
  t->prefetched.assign(n_slots, 0);
  t->heap.resize(n_slots);
  t->hpos.resize(n_slots);
  for (int32_t s = 0; s < n_slots; ++s) t->heap[s] = t->hpos[s] = s;
  if (d_slot_of) {
    if (t->default_copier) {
      if (cudaMemcpy(d_slot_of, t->mirror, mbytes, cudaMemcpyHostToDevice) != cudaSuccess) {
        cudaFreeHost(t->mirror);
        delete t;
        return slot_fail(MOE_ECUDA, "slot_table_create: clearing d_slot_of failed");
      }
    } else if (t->copy_fn(d_slot_of, t->mirror, mbytes, nullptr, t->copy_user) != 0) {
      std::free(t->mirror);
      delete t;
      return slot_fail(MOE_ECUDA, "slot_table_create: clearing d_slot_of failed");
    }
  }
  *out = t;
  return MOE_OK;
}

moe_status slot_table_update(moe_slot_table* t, int32_t layer, const int32_t* h_active, int32_t n_active,
                             moe_stream_t copy_stream, moe_event_t ready, int32_t* h_hits, int32_t* n_hits,
                             int32_t* h_misses, int32_t* n_misses, moe_slot_stats* stats_opt) {
  if (!t || n_active < 0 || (n_active > 0 && !h_active))
    return slot_fail(MOE_EINVAL, "slot_table_update: null table or active list, or n_active < 0");
  if (layer < 0 || layer >= t->L) return slot_fail(MOE_EINVAL, "slot_table_update: layer %d not in [0, %d)", layer, t->L);
  // validate ids, reject repeats (epoch marks)
  if (++t->epoch == 0) {
    std::fill(t->mark.begin(), t->mark.end(), 0);
    t->epoch = 1;
  }
  for (int32_t i = 0; i < n_active; ++i) {
    const int32_t e = h_active[i];
    if (e < 0 || e >= t->E || t->mark[e] == t->epoch)
      return slot_fail(MOE_EINVAL, "slot_table_update: expert id %d out of [0, %d) or repeated", e, t->E);
    t->mark[e] = t->epoch;
  }
  const int64_t base = (int64_t)layer * t->E;
  int32_t nh = 0, nm = 0;
  for (int32_t i = 0; i < n_active; ++i) (t->mirror[base + h_active[i]] >= 0 ? nh : nm)++;
  if (nm > t->n_slots - nh)
    return slot_fail(MOE_ENOSLOT, "slot_table_update: %d misses but %d slots not needed by this call", nm,
                     t->n_slots - nh);
  advance_clock(t);
  // every expert of the call counts one use; hits first become most recently used and
  // pinned, so that no miss evicts them (each slot's new key is fixed before the next change)
  std::vector<int32_t> pins;
  pins.reserve(n_active);
  nh = nm = 0;
  for (int32_t i = 0; i < n_active; ++i) {
    const int32_t e = h_active[i];
    t->score[base + e] += t->inc;
    t->last_use[base + e] = t->calls;
    const int32_t s = t->mirror[base + e];
    if (s >= 0) {
      if (t->prefetched[s]) {
        t->prefetched[s] = 0;
        ++t->pf_used;
      }
      lru_unlink(t, s);
      lru_push_tail(t, s);
      t->pinned[s] = 1;
      heap_fix(t, s);
      pins.push_back(s);
      if (h_hits) h_hits[nh] = e;
      ++nh;
    }
  }
  std::vector<int64_t> changed;
  moe_status rc = MOE_OK;
  for (int32_t i = 0; i < n_active; ++i) {
    const int32_t e = h_active[i];
    if (t->mirror[base + e] >= 0) continue;
    // LRU: the list's head; FREQ: the heap's root. Neither is one of this call's experts.
    const int32_t s = t->policy == MOE_SLOT_FREQ ? t->heap[0] : t->head;
    const int64_t old = t->owner[s];
    if (old >= 0) {
      t->mirror[old] = -1;
      changed.push_back(old);
      t->stats.evictions++;
    }
    t->prefetched[s] = 0;
    t->owner[s] = -1;
    lru_unlink(t, s);
    lru_push_tail(t, s);
    heap_fix(t, s);
    const int cr = t->copy_fn(t->d_pool + (uint64_t)s * t->slot_bytes, t->h_records[base + e], t->slot_bytes,
                              copy_stream, t->copy_user);
    if (cr != 0) {
      rc = slot_fail(MOE_ECUDA, "slot_table_update: copy of layer %d expert %d failed (%d)", layer, e, cr);
      break;
    }
    t->owner[s] = base + e;
    t->mirror[base + e] = s;
    t->pinned[s] = 1;
    heap_fix(t, s);
    pins.push_back(s);
    changed.push_back(base + e);
    t->stats.misses++;
    t->stats.bytes_h2d += t->slot_bytes;
    if (h_misses) h_misses[nm] = e;
    ++nm;
  }
  for (const int32_t s : pins) {
    t->pinned[s] = 0;
    heap_fix(t, s);
  }
  t->stats.hits += nh;
  if (write_entries(t, changed, copy_stream) != 0 && rc == MOE_OK)
    rc = slot_fail(MOE_ECUDA, "slot_table: writing the device table failed");
  if (ready && cudaEventRecord(reinterpret_cast<cudaEvent_t>(ready), reinterpret_cast<cudaStream_t>(copy_stream)) !=
                   cudaSuccess && rc == MOE_OK)
    rc = slot_fail(MOE_ECUDA, "slot_table: recording the ready event failed");
  if (n_hits) *n_hits = nh;
  if (n_misses) *n_misses = nm;
  if (stats_opt) *stats_opt = t->stats;
  return rc;
}

moe_status slot_table_prefetch(moe_slot_table* t, int32_t layer, const int32_t* h_ids, int32_t n_ids,
                               int32_t keep_layer, const int32_t* h_keep, int32_t n_keep, moe_stream_t copy_stream,
                               moe_event_t ready, int32_t* n_loaded) {
  if (!t || n_ids < 0 || n_keep < 0 || (n_ids > 0 && !h_ids) || (n_keep > 0 && !h_keep))
    return slot_fail(MOE_EINVAL, "slot_table_prefetch: null table or id list, or a negative count");
  if (layer < 0 || layer >= t->L || (n_keep > 0 && (keep_layer < 0 || keep_layer >= t->L)))
    return slot_fail(MOE_EINVAL, "slot_table_prefetch: layer %d or keep layer %d not in [0, %d)", layer, keep_layer,
                     t->L);
  for (int32_t i = 0; i < n_ids; ++i)
    if (h_ids[i] < 0 || h_ids[i] >= t->E)
      return slot_fail(MOE_EINVAL, "slot_table_prefetch: expert id %d out of [0, %d)", h_ids[i], t->E);
  for (int32_t i = 0; i < n_keep; ++i)
    if (h_keep[i] < 0 || h_keep[i] >= t->E)
      return slot_fail(MOE_EINVAL, "slot_table_prefetch: kept expert id %d out of [0, %d)", h_keep[i], t->E);
  // pin the kept experts' slots and the slots of this call's experts already resident
  std::vector<int32_t> pins;
  auto pin = [&](int64_t key) {
    const int32_t s = t->mirror[key];
    if (s >= 0 && !t->pinned[s]) {
      t->pinned[s] = 1;
      heap_fix(t, s);
      pins.push_back(s);
    }
  };
  for (int32_t i = 0; i < n_keep; ++i) pin((int64_t)keep_layer * t->E + h_keep[i]);
  const int64_t base = (int64_t)layer * t->E;
  for (int32_t i = 0; i < n_ids; ++i) pin(base + h_ids[i]);
  std::vector<int64_t> changed;
  moe_status rc = MOE_OK;
  int32_t loaded = 0;
  for (int32_t i = 0; i < n_ids; ++i) {
    const int64_t key = base + h_ids[i];
    if (t->mirror[key] >= 0) continue;  // resident, or loaded earlier in this call
    // the victim: LRU, the least recently used unpinned slot; FREQ, the heap's root
    int32_t s = -1;
    if (t->policy == MOE_SLOT_FREQ) {
      if (!t->pinned[t->heap[0]]) s = t->heap[0];
    } else {
      for (int32_t c = t->head; c >= 0; c = t->next[c])
        if (!t->pinned[c]) {
          s = c;
          break;
        }
    }
    if (s < 0) break;  // every slot is pinned: nothing more can be loaded
    const int64_t old = t->owner[s];
    if (old >= 0) {
      t->mirror[old] = -1;
      changed.push_back(old);
      t->stats.evictions++;
    }
    t->owner[s] = -1;
    lru_unlink(t, s);
    lru_push_tail(t, s);
    const int cr = t->copy_fn(t->d_pool + (uint64_t)s * t->slot_bytes, t->h_records[key], t->slot_bytes, copy_stream,
                              t->copy_user);
    if (cr != 0) {
      t->prefetched[s] = 0;
      heap_fix(t, s);
      rc = slot_fail(MOE_ECUDA, "slot_table_prefetch: copy of layer %d expert %d failed (%d)", layer, h_ids[i], cr);
      break;
    }
    t->owner[s] = key;
    t->mirror[key] = s;
    t->prefetched[s] = 1;
    t->pinned[s] = 1;
    heap_fix(t, s);
    pins.push_back(s);
    changed.push_back(key);
    t->stats.bytes_h2d += t->slot_bytes;
    ++t->pf_loads;
    ++loaded;
  }
  for (const int32_t s : pins) {
    t->pinned[s] = 0;
    heap_fix(t, s);
  }
  if (write_entries(t, changed, copy_stream) != 0 && rc == MOE_OK)
    rc = slot_fail(MOE_ECUDA, "slot_table: writing the device table failed");
  if (ready && cudaEventRecord(reinterpret_cast<cudaEvent_t>(ready), reinterpret_cast<cudaStream_t>(copy_stream)) !=
                   cudaSuccess && rc == MOE_OK)
    rc = slot_fail(MOE_ECUDA, "slot_table: recording the ready event failed");
  if (n_loaded) *n_loaded = loaded;
  return rc;
}

moe_status slot_table_prefetch_stats(const moe_slot_table* t, uint64_t* loads, uint64_t* used) {
  if (!t || !loads || !used) return slot_fail(MOE_EINVAL, "slot_table_prefetch_stats: NULL argument");
  *loads = t->pf_loads;
  *used = t->pf_used;
  return MOE_OK;
}

moe_status slot_table_set_policy(moe_slot_table* t, int32_t policy, double half_life) {
  if (!t || (policy != MOE_SLOT_LRU && policy != MOE_SLOT_FREQ) || !(half_life > 0.0) || !std::isfinite(half_life))
    return slot_fail(MOE_EINVAL, "slot_table_set_policy: null table, unknown policy %d or half-life not > 0", policy);
  t->policy = policy;
  t->g = std::pow(2.0, 1.0 / half_life);
  return MOE_OK;
}

moe_status slot_table_warm(moe_slot_table* t, const float* h_weight, moe_stream_t copy_stream, moe_event_t ready,
                           int32_t* n_loaded) {
  if (!t || !h_weight) return slot_fail(MOE_EINVAL, "slot_table_warm: null table or weights");
  const int64_t n_keys = (int64_t)t->L * t->E;
  for (int64_t i = 0; i < n_keys; ++i)
    if (!(h_weight[i] >= 0.0f) || !std::isfinite(h_weight[i]))
      return slot_fail(MOE_EINVAL, "slot_table_warm: weight %lld is negative or not finite", (long long)i);
  for (int64_t i = 0; i < n_keys; ++i) t->score[i] += (double)h_weight[i] * t->inc;
  heap_rebuild(t);
  // empty slots, lowest index first, take the best non-resident experts with a positive weight
  std::vector<int32_t> empty;
  for (int32_t s = 0; s < t->n_slots; ++s)
    if (t->owner[s] < 0) empty.push_back(s);
  std::vector<int64_t> cand;
  for (int64_t i = 0; i < n_keys; ++i)
    if (t->mirror[i] < 0 && h_weight[i] > 0.0f) cand.push_back(i);
  const size_t n = std::min(empty.size(), cand.size());
  std::partial_sort(cand.begin(), cand.begin() + n, cand.end(), [t](int64_t a, int64_t b) {
    return t->score[a] != t->score[b] ? t->score[a] > t->score[b] : a < b;
  });
  std::vector<int64_t> changed;
  moe_status rc = MOE_OK;
  int32_t loaded = 0;
  for (size_t j = 0; j < n; ++j) {
    const int32_t s = empty[j];
    const int64_t key = cand[j];
    const int cr = t->copy_fn(t->d_pool + (uint64_t)s * t->slot_bytes, t->h_records[key], t->slot_bytes, copy_stream,
                              t->copy_user);
    if (cr != 0) {
      rc = slot_fail(MOE_ECUDA, "slot_table_warm: copy of layer %lld expert %lld failed (%d)",
                     (long long)(key / t->E), (long long)(key % t->E), cr);
      break;
    }
    t->owner[s] = key;
    t->mirror[key] = s;
    heap_fix(t, s);
    changed.push_back(key);
    t->stats.bytes_h2d += t->slot_bytes;
    ++loaded;
  }
  // LRU order of the loaded slots: the lowest weight least recent, the highest weight most
  // recent, all after the slots still empty. Under LRU the first evictions then take the
  // experts the profile ranks lowest, not the best ones.
  for (int32_t j = loaded - 1; j >= 0; --j) {
    lru_unlink(t, empty[j]);
    lru_push_tail(t, empty[j]);
  }
  if (write_entries(t, changed, copy_stream) != 0 && rc == MOE_OK)
    rc = slot_fail(MOE_ECUDA, "slot_table: writing the device table failed");
  if (ready && cudaEventRecord(reinterpret_cast<cudaEvent_t>(ready), reinterpret_cast<cudaStream_t>(copy_stream)) !=
                   cudaSuccess && rc == MOE_OK)
    rc = slot_fail(MOE_ECUDA, "slot_table: recording the ready event failed");
  if (n_loaded) *n_loaded = loaded;
  return rc;
}

moe_status slot_table_lookup(const moe_slot_table* t, int32_t layer, const int32_t* h_ids, int32_t n,
                             int32_t* h_slot) {
  if (!t || n < 0 || (n > 0 && (!h_ids || !h_slot)))
    return slot_fail(MOE_EINVAL, "slot_table_lookup: null table or arrays, or n < 0");
  if (layer < 0 || layer >= t->L) return slot_fail(MOE_EINVAL, "slot_table_lookup: layer %d not in [0, %d)", layer, t->L);
  for (int32_t i = 0; i < n; ++i) {
    if (h_ids[i] < 0 || h_ids[i] >= t->E)
      return slot_fail(MOE_EINVAL, "slot_table_lookup: expert id %d out of [0, %d)", h_ids[i], t->E);
    h_slot[i] = t->mirror[(int64_t)layer * t->E + h_ids[i]];
  }
  return MOE_OK;
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
