// Native executor of the tiered L-layer stack: experts in pinned host memory, a device slot pool
// in front of them ("Strata 工作原理图解GPU内存SSD三级存储如何让125B模型塞进消费级显卡", sections
// "三级存储分工" and "专家缓存"). One moe_tiered_forward call runs every layer of one step:
//
//   per layer l: RMS norm of the residual stream; routing and bucketing (moe_route_permute);
//   the resident experts of the active list (moe_filter_resident) and, launched before the host
//   has read anything back, the expert FFN of those hit experts and the shared expert; the
//   active list back to the host, one event wait; the slot table's update (its miss copies on
//   the copy stream, `ready` recorded after them); after the compute stream has waited on
//   `ready`, the missed experts; the combine into the residual stream.
//
// With a bandwidth split (pcie_frac < 1, the pages' --pcie-frac: "Strata 性能基准与论文导读125B
// MoE在消费级硬件上的极限测量与瓶颈分析", section "如何测量"), the last floor((1 - pcie_frac) n)
// of a layer's n misses (active-list order) are not copied: the host computes them from their
// pinned records (moe_host_expert_ffn) while the copies run, and their output rows are copied
// into y_perm before the combine. Host-computed experts do not become resident.
//
// The steps and their order are those of the Python TieredStack (overlap mode), so both give
// the same results bit for bit; this one keeps the per-layer host work (one event wait, the
// slot update, the launches) in C++. The executor owns its buffers, allocated at creation.
// The hit FFN reads only slots of this layer's resident experts, which the update never evicts
// (its victims are never experts of the call), so it may run while the miss copies land.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <new>
#include <vector>

#include "moe_internal.h"

struct moe_tiered {
  moe_shape s, s_routed;
  int L = 0, fmt = MOE_FMT_INT8, cap = 0, P = 0;
  float eps = 1e-6f;
  std::vector<const float*> routers;
  std::vector<const void*> shared;
  std::vector<const void*> h_records;
  uint8_t* pool = nullptr;
  uint64_t slot_bytes = 0, n_slots = 0;
  int32_t* slot_of = nullptr;
  moe_slot_table* table = nullptr;
  // device buffers
  void* xn = nullptr;
  int32_t *topk_idx = nullptr, *counts = nullptr, *offsets = nullptr, *sorted_pair = nullptr, *inv_pos = nullptr,
          *active = nullptr, *d_hits = nullptr, *d_misses = nullptr;
  float *topk_w = nullptr, *y_perm = nullptr;
  void *ws = nullptr, *ws_miss = nullptr;
  size_t ws_bytes = 0, ws_miss_bytes = 0;
  // pinned host buffers
  int32_t *h_active = nullptr, *h_hits = nullptr, *h_misses = nullptr, *h_offsets = nullptr, *h_sorted = nullptr;
  uint16_t* h_xn = nullptr;
  float* h_y = nullptr;
  std::vector<int32_t> h_slot, h_upd, h_host;
  std::vector<const void*> h_host_recs;
  cudaStream_t copy_stream = nullptr;
  cudaEvent_t ready = nullptr, done = nullptr;
  double pcie_frac = 1.0;
  int host_threads = 0;
};

namespace {

moe_status cuda_err(cudaError_t e, const char* what) {
  char buf[256];
  snprintf(buf, sizeof(buf), "%s: %s", what, cudaGetErrorString(e));
  return moe::report_error(MOE_ECUDA, buf);
}

void release(moe_tiered* t) {
  if (!t) return;
  void* dev[] = {t->xn, t->topk_idx, t->counts, t->offsets, t->sorted_pair, t->inv_pos, t->active,
                 t->d_hits, t->d_misses, t->topk_w, t->y_perm, t->ws, t->ws_miss};
  for (void* p : dev)
    if (p) cudaFree(p);
  void* host[] = {t->h_active, t->h_hits, t->h_misses, t->h_offsets, t->h_sorted, t->h_xn, t->h_y};
  for (void* p : host)
    if (p) cudaFreeHost(p);
  if (t->ready) cudaEventDestroy(t->ready);
  if (t->done) cudaEventDestroy(t->done);
  if (t->copy_stream) cudaStreamDestroy(t->copy_stream);
  delete t;
}

template <typename P>
cudaError_t dev_zeros(P** p, size_t bytes) {
  void* v = nullptr;
  cudaError_t e = cudaMalloc(&v, bytes ? bytes : 16);
  if (e == cudaSuccess) e = cudaMemset(v, 0, bytes ? bytes : 16);
  *p = static_cast<P*>(v);
  return e;
}

template <typename P>
cudaError_t host_alloc(P** p, size_t bytes) {
  void* v = nullptr;
  const cudaError_t e = cudaHostAlloc(&v, bytes ? bytes : 16, cudaHostAllocDefault);
  if (e == cudaSuccess) std::memset(v, 0, bytes ? bytes : 16);
  *p = static_cast<P*>(v);
  return e;
}

}  // namespace

extern "C" {

moe_status moe_tiered_create(const moe_shape* shape, int32_t n_layers, const float* const* routers,
                             const void* const* shared, moe_slot_table* table, void* pool, uint64_t slot_bytes,
                             uint64_t n_slots, int32_t* slot_of, const void* const* h_records, int32_t format,
                             float eps, moe_tiered** out) {
  if (!shape || !routers || !table || !pool || !slot_of || !h_records || !out || n_layers <= 0)
    return moe::report_error(MOE_EINVAL, "moe_tiered_create: NULL argument or n_layers <= 0");
  *out = nullptr;
  const moe_shape& s = *shape;
  if (s.T <= 0 || s.d <= 0 || s.f <= 0 || s.E <= 0 || s.k <= 0 || s.k > s.E || s.n_shared < 0)
    return moe::report_error(MOE_EINVAL, "moe_tiered_create: bad shape");
  if (s.n_shared > 0 && !shared) return moe::report_error(MOE_EINVAL, "moe_tiered_create: shared is NULL");
  if (!(eps >= 0.0f) || !std::isfinite(eps)) return moe::report_error(MOE_EINVAL, "moe_tiered_create: bad eps");
  moe_expert_layout lay;
  moe_status st = moe_get_record_layout(s.d, s.f, format, &lay);
  if (st != MOE_OK) return st;
  if (slot_bytes < lay.record_bytes || slot_bytes % 256)
    return moe::report_error(MOE_EINVAL, "moe_tiered_create: slot_bytes below the record size or not a multiple of 256");
  moe_tiered* t = new (std::nothrow) moe_tiered();
  if (!t) return moe::report_error(MOE_EINVAL, "moe_tiered_create: out of host memory");
  t->s = s;
  t->s_routed = s;
  t->s_routed.n_shared = 0;
  t->L = n_layers;
  t->fmt = format;
  t->eps = eps;
  t->P = s.T * s.k;
  t->cap = std::min(s.E, t->P);
  t->routers.assign(routers, routers + n_layers);
  t->shared.assign(n_layers, nullptr);
  if (s.n_shared > 0) t->shared.assign(shared, shared + n_layers);
  t->h_records.assign(h_records, h_records + (size_t)n_layers * s.E);
  t->pool = static_cast<uint8_t*>(pool);
  t->slot_bytes = slot_bytes;
  t->n_slots = n_slots;
  t->slot_of = slot_of;
  t->table = table;
  size_t wsb = 0, wsm = 0;
  if ((st = moe_workspace_size(&t->s, &wsb)) != MOE_OK || (st = moe_workspace_size(&t->s_routed, &wsm)) != MOE_OK) {
    release(t);
    return st;
  }
  t->ws_bytes = wsb;
  t->ws_miss_bytes = wsm;
  const size_t T = s.T, d = s.d, P = t->P, rows = P + T * s.n_shared, cap1 = 1 + (size_t)t->cap;
  cudaError_t e = cudaSuccess;
  auto chk = [&](cudaError_t r) {
    if (e == cudaSuccess) e = r;
  };
  chk(dev_zeros(&t->xn, T * d * 2));
  chk(dev_zeros(&t->topk_idx, P * 4));
  chk(dev_zeros(&t->topk_w, P * 4));
  chk(dev_zeros(&t->counts, (size_t)s.E * 4));
  chk(dev_zeros(&t->offsets, ((size_t)s.E + 1) * 4));
  chk(dev_zeros(&t->sorted_pair, std::max<size_t>(P, 1) * 4));
  chk(dev_zeros(&t->inv_pos, std::max<size_t>(P, 1) * 4));
  chk(dev_zeros(&t->active, cap1 * 4));
  chk(dev_zeros(&t->d_hits, cap1 * 4));
  chk(dev_zeros(&t->d_misses, cap1 * 4));
  chk(dev_zeros(&t->y_perm, rows * d * 4));
  // workspaces zero-filled once: the decode expert FFN keeps counters there that each call leaves at zero
  chk(dev_zeros(&t->ws, std::max<size_t>(wsb, 256)));
  chk(dev_zeros(&t->ws_miss, std::max<size_t>(wsm, 256)));
  chk(host_alloc(&t->h_active, cap1 * 4));
  chk(host_alloc(&t->h_hits, cap1 * 4));
  chk(host_alloc(&t->h_misses, cap1 * 4));
  chk(host_alloc(&t->h_offsets, ((size_t)s.E + 1) * 4));
  chk(host_alloc(&t->h_sorted, std::max<size_t>(P, 1) * 4));
  chk(host_alloc(&t->h_xn, T * d * 2));
  chk(host_alloc(&t->h_y, std::max<size_t>(P, 1) * d * 4));
  chk(cudaStreamCreateWithFlags(&t->copy_stream, cudaStreamNonBlocking));
  chk(cudaEventCreateWithFlags(&t->ready, cudaEventDisableTiming));
  chk(cudaEventCreateWithFlags(&t->done, cudaEventDisableTiming));
  if (e == cudaSuccess) e = cudaEventRecord(t->ready, t->copy_stream);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    release(t);
    return cuda_err(e, "moe_tiered_create");
  }
  t->h_slot.resize(t->cap);
  t->h_upd.resize(t->cap);
  t->h_host.resize(t->cap);
  t->h_host_recs.resize(t->cap);
  *out = t;
  return MOE_OK;
}

moe_status moe_tiered_set_split(moe_tiered* t, double pcie_frac, int32_t host_threads) {
  if (!t) return moe::report_error(MOE_EINVAL, "moe_tiered_set_split: NULL executor");
  if (!(pcie_frac >= 0.0 && pcie_frac <= 1.0) || host_threads < 0)
    return moe::report_error(MOE_EINVAL, "moe_tiered_set_split: pcie_frac outside [0, 1] or host_threads < 0");
  t->pcie_frac = pcie_frac;
  t->host_threads = host_threads;
  return MOE_OK;
}

moe_status moe_tiered_forward(moe_tiered* t, void* resid, moe_stream_t stream_h, int32_t* h_layer_misses,
                              int32_t* h_layer_host) {
  if (!t || !resid) return moe::report_error(MOE_EINVAL, "moe_tiered_forward: NULL argument");
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_h);
  const moe_shape& s = t->s;
  const int E = s.E, cap1 = 1 + t->cap;
  const bool split = t->pcie_frac < 1.0;
  moe_status st;
  cudaError_t e;
#define MOE_T_CALL(x)               \
  do {                              \
    if ((st = (x)) != MOE_OK) return st; \
  } while (0)
#define MOE_T_CUDA(x, what)                            \
  do {                                                 \
    if ((e = (x)) != cudaSuccess) return cuda_err(e, what); \
  } while (0)
  for (int l = 0; l < t->L; ++l) {
    moe_expert_table tab{};
    tab.pool = t->pool;
    tab.slot_bytes = t->slot_bytes;
    tab.slot_of = t->slot_of + (size_t)l * E;
    tab.shared = s.n_shared > 0 ? t->shared[l] : nullptr;
    tab.n_slots = t->n_slots;
    tab.format = (uint32_t)t->fmt;
    MOE_T_CALL(moe_rms_norm(&s, resid, MOE_BF16, t->xn, MOE_BF16, t->eps, stream));
    MOE_T_CALL(moe_route_permute(&s, t->xn, MOE_BF16, t->routers[l], t->topk_idx, t->topk_w, nullptr, t->counts,
                                 t->offsets, t->sorted_pair, t->inv_pos, t->active, t->ws, t->ws_bytes, stream));
    // the experts resident now are the ones the slot update below counts as hits (the device
    // table is current: every earlier update's entries were waited for, or changed nothing)
    MOE_T_CALL(moe_filter_resident(t->active, tab.slot_of, E, t->d_hits, stream));
    MOE_T_CUDA(cudaMemcpyAsync(t->h_active, t->active, (size_t)cap1 * 4, cudaMemcpyDeviceToHost, stream), "active list");
    if (split) {  // what the host needs to compute experts itself
      MOE_T_CUDA(cudaMemcpyAsync(t->h_xn, t->xn, (size_t)s.T * s.d * 2, cudaMemcpyDeviceToHost, stream), "x copy");
      MOE_T_CUDA(cudaMemcpyAsync(t->h_offsets, t->offsets, ((size_t)E + 1) * 4, cudaMemcpyDeviceToHost, stream),
                 "offsets copy");
      MOE_T_CUDA(cudaMemcpyAsync(t->h_sorted, t->sorted_pair, (size_t)t->P * 4, cudaMemcpyDeviceToHost, stream),
                 "pairs copy");
    }
    // the host waits for the routing and for the previous layer's FFN (no slot it read may be
    // overwritten before); the hit experts' FFN, enqueued after the event, runs meanwhile
    MOE_T_CUDA(cudaEventRecord(t->done, stream), "event record");
    MOE_T_CALL(moe_expert_ffn(&s, MOE_MODE_AUTO, t->xn, MOE_BF16, &tab, t->offsets, t->sorted_pair, t->d_hits,
                              t->y_perm, MOE_F32, t->ws, t->ws_bytes, stream));
    MOE_T_CUDA(cudaEventSynchronize(t->done), "event wait");
    const int n = t->h_active[0];
    const int32_t* upd = t->h_active + 1;
    int n_upd = n, n_host = 0;
    if (split && n > 0) {
      MOE_T_CALL(slot_table_lookup(t->table, l, t->h_active + 1, n, t->h_slot.data()));
      int n_miss_all = 0;
      for (int i = 0; i < n; ++i) n_miss_all += t->h_slot[i] < 0;
      n_host = (int)(n_miss_all * (1.0 - t->pcie_frac));
      // the last n_host misses in active-list order stay on the host, in ascending expert order
      int skip = n_miss_all - n_host, hcount = 0;
      n_upd = 0;
      for (int i = 0; i < n; ++i) {
        const int ex = t->h_active[1 + i];
        if (t->h_slot[i] < 0) {
          if (skip > 0) {
            --skip;
          } else {
            t->h_host[hcount++] = ex;
            continue;
          }
        }
        t->h_upd[n_upd++] = ex;
      }
      std::sort(t->h_host.begin(), t->h_host.begin() + n_host);
      upd = t->h_upd.data();
    }
    if (h_layer_host) h_layer_host[l] = n_host;
    MOE_T_CALL(slot_table_update(t->table, l, upd, n_upd, t->copy_stream, t->ready, t->h_hits + 1, t->h_hits,
                                 t->h_misses + 1, t->h_misses, nullptr));
    const int n_miss = t->h_misses[0];
    if (h_layer_misses) h_layer_misses[l] = n_miss;
    if (n_miss) {
      MOE_T_CUDA(cudaStreamWaitEvent(stream, t->ready, 0), "wait for the miss copies");
      MOE_T_CUDA(cudaMemcpyAsync(t->d_misses, t->h_misses, (size_t)cap1 * 4, cudaMemcpyHostToDevice, stream),
                 "misses copy");
      moe_expert_table routed = tab;
      routed.shared = nullptr;
      // the missed experts only (a shape without the shared expert, already done)
      MOE_T_CALL(moe_expert_ffn(&t->s_routed, MOE_MODE_AUTO, t->xn, MOE_BF16, &routed, t->offsets, t->sorted_pair,
                                t->d_misses, t->y_perm, MOE_F32, t->ws_miss, t->ws_miss_bytes, stream));
    }
    if (n_host) {
      // the host computes the rest of the misses, then their rows go in
      for (int i = 0; i < n_host; ++i) t->h_host_recs[i] = t->h_records[(size_t)l * E + t->h_host[i]];
      MOE_T_CALL(moe_host_expert_ffn(&s, t->h_xn, MOE_BF16, t->h_host_recs.data(), t->h_host.data(), n_host,
                                     t->h_offsets, t->h_sorted, t->h_y, t->fmt, t->host_threads));
      for (int i = 0; i < n_host; ++i) {
        const int ex = t->h_host[i], r0 = t->h_offsets[ex], r1 = t->h_offsets[ex + 1];
        if (r1 > r0)
          MOE_T_CUDA(cudaMemcpyAsync(t->y_perm + (size_t)r0 * s.d, t->h_y + (size_t)r0 * s.d,
                                     (size_t)(r1 - r0) * s.d * 4, cudaMemcpyHostToDevice, stream),
                     "host rows copy");
      }
    }
    MOE_T_CALL(moe_combine(&s, t->y_perm, MOE_F32, t->inv_pos, t->topk_w, resid, resid, MOE_BF16, stream));
  }
#undef MOE_T_CALL
#undef MOE_T_CUDA
  return MOE_OK;
}

moe_status moe_tiered_status(moe_tiered* t, moe_stream_t stream, int32_t* h_status) {
  if (!t || !h_status) return moe::report_error(MOE_EINVAL, "moe_tiered_status: NULL argument");
  int32_t a = 0, b = 0;
  moe_status s1 = moe_read_status(t->ws, stream, &a);
  if (s1 == MOE_ECUDA) return s1;
  moe_status s2 = moe_read_status(t->ws_miss, stream, &b);
  if (s2 == MOE_ECUDA) return s2;
  *h_status = a | b;
  return *h_status ? MOE_EDEVICE : MOE_OK;
}

moe_status moe_tiered_destroy(moe_tiered* t) {
  if (!t) return MOE_OK;
  cudaStreamSynchronize(t->copy_stream);
  release(t);
  return MOE_OK;
}

}  // extern "C"
