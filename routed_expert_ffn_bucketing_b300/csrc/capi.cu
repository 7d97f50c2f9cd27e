// C-ABI entry points (include/moe.h): argument checks, workspace layout, kernel dispatch.
// Every check happens on the host before any launch; a failed check enqueues nothing.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <set>
#include <utility>

#include "moe_internal.h"

namespace moe {

static thread_local char g_err[512] = "";

static moe_status fail(moe_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return st;
}

moe_status report_error(moe_status st, const char* msg) { return fail(st, "%s", msg); }

static moe_status cuda_fail(cudaError_t e, const char* where) {
  return fail(MOE_ECUDA, "%s: %s", where, cudaGetErrorString(e));
}

static size_t align256(size_t n) { return (n + 255) & ~(size_t)255; }

constexpr uint64_t kDefaultWaitNs = 1000000000ull;  // 1 s
constexpr uint64_t kMaxWaitNs = 10000000000ull;     // 10 s
static std::atomic<uint64_t> g_wait_ns{kDefaultWaitNs};

uint64_t wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }

// Routed work items at most: experts with at least one pair.
static size_t P_items(const moe_shape& s) {
  const size_t P = (size_t)s.T * s.k;
  return P < (size_t)s.E ? P : (size_t)s.E;
}

int route_splits(int d) { return (d + kRouteRowsPerSplit - 1) / kRouteRowsPerSplit; }
int perm_chunks(int P) { return (P + kPermChunk - 1) / kPermChunk; }

WsLayout ws_layout(const moe_shape& s) {
  WsLayout L{};
  const size_t T = (size_t)s.T, P = (size_t)s.T * s.k;
  size_t o = 0;
  L.status = o;
  o += 256;
  L.route_partial = o;
  if (s.T <= kRouteGemvMaxT) o = align256(o + sizeof(float) * route_splits(s.d) * T * s.E);
  L.logits = o;
  if (s.T > kRouteGemvMaxT) o = align256(o + sizeof(float) * T * s.E);
  L.wparts = o;
  if (s.T > kRouteGemvMaxT) o = align256(o + sizeof(uint16_t) * 3 * (size_t)s.E * s.d);
  L.perm_cnt = o;
  const size_t C = P > (size_t)kPermChunk ? (size_t)perm_chunks((int)P) : 0;
  o = align256(o + sizeof(int32_t) * C * s.E);
  L.perm_keys = o;
  o = align256(o + sizeof(uint32_t) * C * kPermChunk);
  L.h = o;
  o = align256(o + sizeof(float) * (P + T * s.n_shared) * s.f);
  L.x16 = o;
  o = align256(o + sizeof(uint16_t) * T * s.d);
  L.xunscale = o;
  o = align256(o + sizeof(float) * T);
  // stream-K scratch of the decode kernels (T <= 8): tasks per kernel at most items * max(f/8, d/16)
  const size_t sk_tasks = s.T <= 8 ? (P_items(s) + s.n_shared) * (s.f / 8 > s.d / 16 ? s.f / 8 : s.d / 16) : 0;
  L.zero = o;
  L.item_done = o;  // then the exit counter and the abort flag of the persistent kernel
  o = align256(o + sizeof(int32_t) * (P_items(s) + s.n_shared + 2));
  L.hmax = o;
  o = align256(o + sizeof(uint32_t) * (P + T * s.n_shared));
  L.task_cnt = o;
  o = align256(o + sizeof(int32_t) * 2 * sk_tasks);
  L.zero_end = o;
  L.items = o;
  o = align256(o + sizeof(ItemRec) * ((P < (size_t)s.E ? P : (size_t)s.E) + s.n_shared));
  L.row_tok = o;
  o = align256(o + sizeof(int32_t) * (P + T * s.n_shared));
  L.h16 = o;
  o = align256(o + sizeof(uint16_t) * (P + T * s.n_shared) * s.f);
  L.hexp = o;
  o = align256(o + sizeof(int32_t) * (P + T * s.n_shared));
  L.item_cnt = o;
  o = align256(o + sizeof(int32_t) * ((P < (size_t)s.E ? P : (size_t)s.E) + s.n_shared + 2));
  L.xp16 = o;
  o = align256(o + sizeof(uint16_t) * (P + T * s.n_shared) * s.d);
  L.xexp = o;
  o = align256(o + sizeof(int32_t) * T);
  L.tiles = o;
  o = align256(o + sizeof(int32_t) * 2 * ((P + T * s.n_shared) / 128 + P_items(s) + s.n_shared + 2));
  L.part = o;
  o = align256(o + sizeof(float) * 2 * sk_tasks * 2 * 128);
  L.cx = o;
  o = align256(o + sizeof(float) * T * (s.d / 32));
  L.ch = o;
  o = align256(o + sizeof(float) * (P + T * s.n_shared) * (s.f / 32));
  L.total = o;
  return L;
}

cudaError_t ensure_dynamic_smem(const void* kernel, size_t bytes) {
  static std::mutex mu;
  static std::set<std::pair<const void*, int>> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (done.count({kernel, dev})) return cudaSuccess;
  int optin = 0;
  e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, kernel);
  if (e != cudaSuccess) return e;
  const size_t room = (size_t)optin - fa.sharedSizeBytes;  // static shared memory counts too
  if (bytes > room) return cudaErrorInvalidValue;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)room);
  if (e != cudaSuccess) return e;
  done.insert({kernel, dev});
  return cudaSuccess;
}

// CTAs of the persistent decode expert FFN: the SM count less min(T, 8). As a programmatic
// dependent of the routing kernels (moe_layer_forward) the grid starts while the routing tail's
// cluster of T CTAs still holds T SMs; a CTA planned for one of those SMs starts late and every
// cross-CTA wait then waits for it (measured at T = 4: 66.5 µs per layer pass with 144 CTAs,
// 77 µs with 148). The standalone launch uses the same count, so the stream-K split, and with it
// the fp32 summation order, is the same whichever call runs the kernel.
int persist_grid(const moe_shape& s, int sm_count) {
  const int t = s.T < 8 ? s.T : 8;
  return sm_count > 2 * t ? sm_count - t : sm_count;
}

int device_sm_count() {
  static std::mutex mu;
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n > 0 ? n : 148;
  }
  return cache[dev];
}

static bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

static moe_status check_shape(const moe_shape* s) {
  if (!s) return fail(MOE_EINVAL, "shape is NULL");
  if (s->T < 0 || s->d <= 0 || s->f <= 0 || s->E <= 0 || s->k <= 0 || s->n_shared < 0)
    return fail(MOE_EINVAL, "shape has a negative or zero field (T=%d d=%d f=%d E=%d k=%d n_shared=%d)", s->T,
                s->d, s->f, s->E, s->k, s->n_shared);
  if (s->d % 32 || s->f % 32) return fail(MOE_EINVAL, "d=%d and f=%d must be multiples of 32", s->d, s->f);
  if (s->k > s->E) return fail(MOE_EINVAL, "k=%d exceeds E=%d", s->k, s->E);
  if (s->k > 32) return fail(MOE_EUNSUPPORTED, "k=%d > 32", s->k);
  if (s->E > 1024) return fail(MOE_EUNSUPPORTED, "E=%d > 1024", s->E);
  if (s->T > 65535) return fail(MOE_EUNSUPPORTED, "T=%d > 65535", s->T);
  if (s->n_shared > 8) return fail(MOE_EUNSUPPORTED, "n_shared=%d > 8", s->n_shared);
  if ((int64_t)s->d * s->f > (int64_t)1 << 30) return fail(MOE_EUNSUPPORTED, "d*f too large");
  return MOE_OK;
}

static moe_status check_ws(const moe_shape* s, const void* ws, size_t ws_bytes) {
  if (!ws) return fail(MOE_EINVAL, "workspace is NULL");
  if (!aligned(ws, 256)) return fail(MOE_EINVAL, "workspace must be 256-byte aligned");
  const size_t need = ws_layout(*s).total;
  if (ws_bytes < need) return fail(MOE_EINVAL, "workspace has %zu bytes, needs %zu", ws_bytes, need);
  return MOE_OK;
}

static moe_status check_dtype(int dt, const char* what) {
  if (dt != MOE_BF16 && dt != MOE_F32) return fail(MOE_EINVAL, "%s dtype %d is not MOE_BF16 or MOE_F32", what, dt);
  return MOE_OK;
}

template <typename T>
static T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_last_error_string(void) { return g_err; }

moe_status moe_get_expert_layout(int32_t d, int32_t f, moe_expert_layout* out) {
  return moe_get_record_layout(d, f, MOE_FMT_INT8, out);
}

moe_status moe_get_record_layout(int32_t d, int32_t f, int32_t format, moe_expert_layout* out) {
  if (!out) return fail(MOE_EINVAL, "out is NULL");
  if (format != MOE_FMT_INT8 && format != MOE_FMT_Q2) return fail(MOE_EINVAL, "unknown record format %d", format);
  if (d <= 0 || f <= 0 || d % 32 || f % 32) return fail(MOE_EINVAL, "d=%d f=%d must be positive multiples of 32", d, f);
  if (format == MOE_FMT_Q2 && (d % 256 || f % 256))
    return fail(MOE_EINVAL, "the 2-bit format needs d=%d and f=%d to be multiples of 256", d, f);
  const uint64_t q = (uint64_t)d * f / (format == MOE_FMT_Q2 ? 4 : 1);
  const uint64_t sgu = (uint64_t)f * (d / 32) * 2, sd = (uint64_t)d * (f / 32) * 2;
  uint64_t o = 0;
  auto take = [&](uint64_t n) {
    const uint64_t r = o;
    o = (o + n + 255) & ~(uint64_t)255;
    return r;
  };
  out->gate_q = take(q);
  out->up_q = take(q);
  out->down_q = take(q);
  out->gate_s = take(sgu);
  out->up_s = take(sgu);
  out->down_s = take(sd);
  out->record_bytes = o;
  return MOE_OK;
}

moe_status moe_workspace_size(const moe_shape* shape, size_t* bytes) {
  moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  if (!bytes) return fail(MOE_EINVAL, "bytes is NULL");
  *bytes = ws_layout(*shape).total;
  return MOE_OK;
}

}  // extern "C"

namespace {

// moe_route, with two options a stack of layers uses: pdl_gemv launches the split-d router GEMV as
// a programmatic dependent of the kernel before it (the stack's RMS norm), and clear_status false
// leaves the status word as the earlier layers left it.
moe_status route_impl(const moe_shape* shape, const void* x, moe_dtype xdt, const float* w_router,
                      int32_t* topk_idx, float* topk_w, float* logits_opt, void* ws, size_t ws_bytes,
                      moe_stream_t stream, bool pdl_gemv, bool clear_status) {
  moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  if ((st = check_dtype(xdt, "x")) != MOE_OK) return st;
  if ((st = check_ws(shape, ws, ws_bytes)) != MOE_OK) return st;
  if (shape->T > 0) {
    if (!x || !w_router || !topk_idx || !topk_w) return fail(MOE_EINVAL, "moe_route: NULL argument");
    if (!aligned(x, 16) || !aligned(w_router, 16))
      return fail(MOE_EINVAL, "moe_route: x and w_router must be 16-byte aligned");
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const WsLayout L = ws_layout(*shape);
  int* status = at<int>(ws, L.status);
  cudaError_t e;
  if (shape->T == 0) {
    e = clear_status ? cudaMemsetAsync(status, 0, sizeof(int), s) : cudaSuccess;
    if (e != cudaSuccess) return cuda_fail(e, "moe_route: clearing the status word");
    return MOE_OK;
  }
  // the router kernel clears the status word, and the counters the decode expert FFN keeps in
  // this workspace, before anything reads them
  if (shape->T <= kRouteGemvMaxT) {
    float* partial = at<float>(ws, L.route_partial);
    e = launch_route_gemv(*shape, x, xdt, w_router, partial, status, at<uint8_t>(ws, L.zero), L.zero_end - L.zero,
                          s, pdl_gemv, clear_status);
    if (e == cudaSuccess)
      e = launch_topk_split(*shape, partial, route_splits(shape->d), topk_idx, topk_w, logits_opt, status, s);
  } else {
    float* logits = logits_opt ? logits_opt : at<float>(ws, L.logits);
    if (route_tc_supported(*shape, xdt))
      e = launch_route_tc(*shape, x, w_router, at<uint8_t>(ws, L.wparts), logits, status, s, clear_status);
    else
      e = launch_route_gemm(*shape, x, xdt, w_router, logits, status, s, clear_status);
    if (e == cudaSuccess) e = launch_topk(*shape, logits, topk_idx, topk_w, status, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "moe_route: launch");
  return MOE_OK;
}

}  // namespace

extern "C" {

moe_status moe_route(const moe_shape* shape, const void* x, moe_dtype xdt, const float* w_router,
                     int32_t* topk_idx, float* topk_w, float* logits_opt, void* ws, size_t ws_bytes,
                     moe_stream_t stream) {
  return route_impl(shape, x, xdt, w_router, topk_idx, topk_w, logits_opt, ws, ws_bytes, stream, false, true);
}

moe_status moe_permute(const moe_shape* shape, const int32_t* topk_idx, int32_t* counts, int32_t* offsets,
                       int32_t* sorted_pair, int32_t* inv_pos, int32_t* active, void* ws, size_t ws_bytes,
                       moe_stream_t stream) {
  moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  if ((st = check_ws(shape, ws, ws_bytes)) != MOE_OK) return st;
  if (!counts || !offsets || !active || (shape->T > 0 && (!topk_idx || !sorted_pair || !inv_pos)))
    return fail(MOE_EINVAL, "moe_permute: NULL argument");
  const WsLayout L = ws_layout(*shape);
  cudaError_t e = launch_permute(*shape, topk_idx, counts, offsets, sorted_pair, inv_pos, active,
                                 at<int32_t>(ws, L.perm_cnt), at<uint32_t>(ws, L.perm_keys), at<int>(ws, L.status),
                                 reinterpret_cast<cudaStream_t>(stream), false);
  if (e != cudaSuccess) return cuda_fail(e, "moe_permute: launch");
  return MOE_OK;
}

}  // extern "C"

namespace {

// moe_route_permute with route_impl's two stack options.
moe_status route_permute_impl(const moe_shape* shape, const void* x, moe_dtype xdt, const float* w_router,
                              int32_t* topk_idx, float* topk_w, float* logits_opt, int32_t* counts,
                              int32_t* offsets, int32_t* sorted_pair, int32_t* inv_pos, int32_t* active, void* ws,
                              size_t ws_bytes, moe_stream_t stream, bool pdl_gemv, bool clear_status) {
  moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  if ((st = check_dtype(xdt, "x")) != MOE_OK) return st;
  if ((st = check_ws(shape, ws, ws_bytes)) != MOE_OK) return st;
  if (shape->T == 0 || !route_tail_supported(*shape)) {
    st = route_impl(shape, x, xdt, w_router, topk_idx, topk_w, logits_opt, ws, ws_bytes, stream, pdl_gemv,
                    clear_status);
    if (st != MOE_OK) return st;
    return moe_permute(shape, topk_idx, counts, offsets, sorted_pair, inv_pos, active, ws, ws_bytes, stream);
  }
  if (!x || !w_router || !topk_idx || !topk_w || !counts || !offsets || !sorted_pair || !inv_pos || !active)
    return fail(MOE_EINVAL, "moe_route_permute: NULL argument");
  if (!aligned(x, 16) || !aligned(w_router, 16))
    return fail(MOE_EINVAL, "moe_route_permute: x and w_router must be 16-byte aligned");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const WsLayout L = ws_layout(*shape);
  int* status = at<int>(ws, L.status);
  float* partial = at<float>(ws, L.route_partial);
  cudaError_t e = launch_route_gemv(*shape, x, xdt, w_router, partial, status, at<uint8_t>(ws, L.zero),
                                    L.zero_end - L.zero, s, pdl_gemv, clear_status);
  if (e == cudaSuccess)
    e = launch_route_tail(*shape, partial, route_splits(shape->d), topk_idx, topk_w, logits_opt, counts, offsets,
                          sorted_pair, inv_pos, active, status, s);
  if (e != cudaSuccess) return cuda_fail(e, "moe_route_permute: launch");
  return MOE_OK;
}

}  // namespace

extern "C" {

moe_status moe_route_permute(const moe_shape* shape, const void* x, moe_dtype xdt, const float* w_router,
                             int32_t* topk_idx, float* topk_w, float* logits_opt, int32_t* counts, int32_t* offsets,
                             int32_t* sorted_pair, int32_t* inv_pos, int32_t* active, void* ws, size_t ws_bytes,
                             moe_stream_t stream) {
  return route_permute_impl(shape, x, xdt, w_router, topk_idx, topk_w, logits_opt, counts, offsets, sorted_pair,
                            inv_pos, active, ws, ws_bytes, stream, false, true);
}

}  // extern "C"

namespace {

// The combine that moe_expert_ffn_combine asks the expert FFN to fuse (already validated).
struct CombineReq {
  const int32_t* inv_pos;
  const float* topk_w;
  const void* residual;
  void* out;
  moe_dtype odt;
};

// moe_expert_ffn, and with `cmb` the combine launched after it on the same stream.
moe_status expert_ffn_impl(const moe_shape* shape, moe_mode mode, const void* x, moe_dtype xdt,
                           const moe_expert_table* experts, const int32_t* offsets, const int32_t* sorted_pair,
                           const int32_t* active, void* y_perm, moe_dtype ydt, void* ws, size_t ws_bytes,
                           moe_stream_t stream, const CombineReq* cmb, bool pdl_first = false) {
  moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  if ((st = check_dtype(xdt, "x")) != MOE_OK) return st;
  if ((st = check_dtype(ydt, "y_perm")) != MOE_OK) return st;
  if ((st = check_ws(shape, ws, ws_bytes)) != MOE_OK) return st;
  if (mode != MOE_MODE_AUTO && mode != MOE_MODE_DECODE && mode != MOE_MODE_PREFILL)
    return fail(MOE_EINVAL, "moe_expert_ffn: bad mode %d", (int)mode);
  if (shape->T == 0) return MOE_OK;
  if (!x || !experts || !offsets || !sorted_pair || !active || !y_perm)
    return fail(MOE_EINVAL, "moe_expert_ffn: NULL argument");
  if (!experts->pool || !experts->slot_of) return fail(MOE_EINVAL, "moe_expert_ffn: NULL pool or slot_of");
  if (experts->n_slots == 0 || experts->n_slots > ((uint64_t)1 << 31))
    return fail(MOE_EINVAL, "moe_expert_ffn: n_slots %llu must be in [1, 2^31]", (unsigned long long)experts->n_slots);
  if ((shape->n_shared > 0) != (experts->shared != nullptr))
    return fail(MOE_EINVAL, "moe_expert_ffn: shared must be non-NULL exactly when n_shared > 0");
  if (experts->format != MOE_FMT_INT8 && experts->format != MOE_FMT_Q2)
    return fail(MOE_EINVAL, "moe_expert_ffn: unknown record format %u", experts->format);
  moe_expert_layout lay;
  if ((st = moe_get_record_layout(shape->d, shape->f, (int32_t)experts->format, &lay)) != MOE_OK) return st;
  if (experts->slot_bytes < lay.record_bytes || experts->slot_bytes % 256)
    return fail(MOE_EINVAL, "moe_expert_ffn: slot_bytes %llu must be >= %llu and a multiple of 256",
                (unsigned long long)experts->slot_bytes, (unsigned long long)lay.record_bytes);
  if (!aligned(x, 16) || !aligned(y_perm, 16) || !aligned(experts->pool, 256) ||
      (experts->shared && !aligned(experts->shared, 256)))
    return fail(MOE_EINVAL, "moe_expert_ffn: misaligned x, y_perm, pool or shared");
  if (shape->T == 0) return MOE_OK;
  const WsLayout L = ws_layout(*shape);
  FfnArgs a{};
  a.x = x;
  a.xdt = xdt;
  a.pool = static_cast<const uint8_t*>(experts->pool);
  a.slot_bytes = experts->slot_bytes;
  a.slot_of = experts->slot_of;
  a.shared = static_cast<const uint8_t*>(experts->shared);
  a.n_slots = experts->n_slots;
  a.offsets = offsets;
  a.sorted_pair = sorted_pair;
  a.active = active;
  a.y = y_perm;
  a.ydt = ydt;
  a.h = at<float>(ws, L.h);
  a.status = at<int>(ws, L.status);
  a.wait_ns = wait_limit_ns();
  a.fmt = (int)experts->format;
  a.T = shape->T;
  a.d = shape->d;
  a.f = shape->f;
  a.E = shape->E;
  a.k = shape->k;
  a.n_shared = shape->n_shared;
  a.P = shape->T * shape->k;
  a.o_gate_q = lay.gate_q;
  a.o_up_q = lay.up_q;
  a.o_down_q = lay.down_q;
  a.o_gate_s = lay.gate_s;
  a.o_up_s = lay.up_s;
  a.o_down_s = lay.down_s;
  // PREFILL (and AUTO for T > 16 with bf16 x): tensor-core grouped GEMM. DECODE (and AUTO for few
  // tokens): streaming tensor-core kernels for bf16 x, fp32 SIMT kernels in the fp32 debug mode.
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (a.fmt == MOE_FMT_Q2 && !(xdt == MOE_BF16 && mode != MOE_MODE_PREFILL && persist_supported(a, device_sm_count())))
    return fail(MOE_EUNSUPPORTED,
                "moe_expert_ffn: 2-bit records run on the decode kernel only (bf16 x, T <= 8, d and f multiples of 256)");
  const bool want_prefill = mode == MOE_MODE_PREFILL || (mode == MOE_MODE_AUTO && shape->T > kDecodeMaxT && xdt == MOE_BF16);
  if (want_prefill && prefill_supported(a)) {
    const PrefillAux px{at<__half>(ws, L.xp16),    at<float>(ws, L.xunscale), at<int32_t>(ws, L.xexp),
                        at<uint32_t>(ws, L.hmax),   at<ItemRec>(ws, L.items),  at<int32_t>(ws, L.row_tok),
                        at<__half>(ws, L.h16),      at<int32_t>(ws, L.hexp),   at<int2>(ws, L.tiles),
                        at<int32_t>(ws, L.tiles) + 2 * ((size_t)(shape->T * shape->k + shape->T * shape->n_shared) / 128 +
                                                        P_items(*shape) + shape->n_shared + 1)};
    e = launch_ffn_prefill(a, px, device_sm_count(), cs);
  } else if (mode == MOE_MODE_PREFILL) {
    return fail(MOE_EUNSUPPORTED, "moe_expert_ffn: PREFILL needs bf16 x, d a multiple of 256 and f of 128");
  } else if (want_prefill) {
    // AUTO never drops many tokens onto the SIMT kernels; DECODE asks for them explicitly
    return fail(MOE_EUNSUPPORTED,
                "moe_expert_ffn: AUTO with T=%d > %d needs the tensor-core GEMM (d a multiple of 256, f of 128; "
                "here d=%d f=%d); pass MOE_MODE_DECODE to run the fp32 SIMT kernels",
                shape->T, kDecodeMaxT, shape->d, shape->f);
  } else if (xdt == MOE_BF16 && persist_supported(a, device_sm_count())) {
    const size_t items_max = (P_items(*shape)) + shape->n_shared;
    const size_t sk_tasks = items_max * (shape->f / 8 > shape->d / 16 ? shape->f / 8 : shape->d / 16);
    const PersistAux px{at<float>(ws, L.part),       at<int32_t>(ws, L.task_cnt), at<uint32_t>(ws, L.hmax),
                        at<int32_t>(ws, L.item_done), sk_tasks * 2 * 128,         sk_tasks,
                        at<int32_t>(ws, L.item_done) + items_max};
    e = launch_ffn_persist(a, px, persist_grid(*shape, device_sm_count()), cs, pdl_first);
  } else if (xdt == MOE_BF16 && stream_supported(a)) {
    const size_t items_max = (P_items(*shape)) + shape->n_shared;
    StreamAux aux{at<__half>(ws, L.x16),    at<float>(ws, L.xunscale), at<uint32_t>(ws, L.hmax),
                        at<ItemRec>(ws, L.items), at<int32_t>(ws, L.row_tok), at<__half>(ws, L.h16),
                        at<int32_t>(ws, L.hexp),  at<int32_t>(ws, L.item_cnt), at<float>(ws, L.cx),
                        at<float>(ws, L.ch),      at<int32_t>(ws, L.item_cnt) + items_max,
                        at<float>(ws, L.part),    at<int32_t>(ws, L.task_cnt),
                        0, 0};
    const size_t sk_tasks = shape->T <= 8 ? items_max * (shape->f / 8 > shape->d / 16 ? shape->f / 8 : shape->d / 16) : 0;
    aux.part_stride = sk_tasks * 2 * 128;
    aux.cnt_stride = sk_tasks;
    e = launch_ffn_stream(a, aux, device_sm_count(), cs);
  } else {
    e = launch_ffn_decode(a, cs);
  }
  if (e != cudaSuccess) return cuda_fail(e, "moe_expert_ffn: launch");
  if (cmb) {
    e = launch_combine(*shape, y_perm, ydt, cmb->inv_pos, cmb->topk_w, cmb->residual, cmb->out, cmb->odt, cs, true);
    if (e != cudaSuccess) return cuda_fail(e, "moe_expert_ffn_combine: combine launch");
  }
  return MOE_OK;
}

}  // namespace

extern "C" {

moe_status moe_expert_ffn(const moe_shape* shape, moe_mode mode, const void* x, moe_dtype xdt,
                          const moe_expert_table* experts, const int32_t* offsets, const int32_t* sorted_pair,
                          const int32_t* active, void* y_perm, moe_dtype ydt, void* ws, size_t ws_bytes,
                          moe_stream_t stream) {
  return expert_ffn_impl(shape, mode, x, xdt, experts, offsets, sorted_pair, active, y_perm, ydt, ws, ws_bytes,
                         stream, nullptr);
}

moe_status moe_expert_ffn_combine(const moe_shape* shape, moe_mode mode, const void* x, moe_dtype xdt,
                                  const moe_expert_table* experts, const int32_t* offsets,
                                  const int32_t* sorted_pair, const int32_t* active, void* y_perm, moe_dtype ydt,
                                  const int32_t* inv_pos, const float* topk_w, const void* residual_opt, void* out,
                                  moe_dtype odt, void* ws, size_t ws_bytes, moe_stream_t stream) {
  moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  if ((st = check_dtype(odt, "out")) != MOE_OK) return st;
  if (shape->T > 0) {
    if (!inv_pos || !topk_w || !out) return fail(MOE_EINVAL, "moe_expert_ffn_combine: NULL argument");
    if (!aligned(out, 16) || (residual_opt && !aligned(residual_opt, 16)))
      return fail(MOE_EINVAL, "moe_expert_ffn_combine: misaligned out or residual");
  }
  const CombineReq cmb{inv_pos, topk_w, residual_opt, out, odt};
  return expert_ffn_impl(shape, mode, x, xdt, experts, offsets, sorted_pair, active, y_perm, ydt, ws, ws_bytes,
                         stream, &cmb);
}

moe_status moe_layer_forward(const moe_shape* shape, const void* x, moe_dtype xdt, const float* w_router,
                             const moe_expert_table* experts, moe_mode mode, int32_t* topk_idx, float* topk_w,
                             float* logits_opt, int32_t* counts, int32_t* offsets, int32_t* sorted_pair,
                             int32_t* inv_pos, int32_t* active, void* y_perm, moe_dtype ydt, const void* residual_opt,
                             void* out, moe_dtype odt, void* ws, size_t ws_bytes, moe_stream_t stream) {
  moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  if ((st = check_dtype(odt, "out")) != MOE_OK) return st;
  if (shape->T > 0) {
    if (!out) return fail(MOE_EINVAL, "moe_layer_forward: NULL out");
    if (!aligned(out, 16) || (residual_opt && !aligned(residual_opt, 16)))
      return fail(MOE_EINVAL, "moe_layer_forward: misaligned out or residual");
  }
  st = moe_route_permute(shape, x, xdt, w_router, topk_idx, topk_w, logits_opt, counts, offsets, sorted_pair,
                         inv_pos, active, ws, ws_bytes, stream);
  if (st != MOE_OK) return st;
  // the kernel before the expert FFN on the stream is the bucketing kernel just enqueued
  const CombineReq cmb{inv_pos, topk_w, residual_opt, out, odt};
  return expert_ffn_impl(shape, mode, x, xdt, experts, offsets, sorted_pair, active, y_perm, ydt, ws, ws_bytes,
                         stream, &cmb, true);
}

moe_status moe_stack_forward(const moe_shape* shape, int32_t n_layers, const float* const* w_routers,
                             const moe_expert_table* experts, moe_mode mode, void* resid, moe_dtype rdt,
                             float eps, void* xn, int32_t* topk_idx, float* topk_w, int32_t* counts,
                             int32_t* offsets, int32_t* sorted_pair, int32_t* inv_pos, int32_t* active,
                             void* y_perm, moe_dtype ydt, void* ws, size_t ws_bytes, moe_stream_t stream) {
  moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  if ((st = check_dtype(rdt, "resid")) != MOE_OK) return st;
  if ((st = check_ws(shape, ws, ws_bytes)) != MOE_OK) return st;
  if (n_layers < 0) return fail(MOE_EINVAL, "moe_stack_forward: n_layers %d < 0", (int)n_layers);
  if (!(eps >= 0.0f) || !isfinite(eps)) return fail(MOE_EINVAL, "moe_stack_forward: eps must be finite and >= 0");
  if (n_layers > 0 && (!w_routers || !experts)) return fail(MOE_EINVAL, "moe_stack_forward: NULL layer arrays");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const WsLayout L = ws_layout(*shape);
  if (shape->T == 0 || n_layers == 0) {
    const cudaError_t e = cudaMemsetAsync(at<int>(ws, L.status), 0, sizeof(int), s);
    if (e != cudaSuccess) return cuda_fail(e, "moe_stack_forward: clearing the status word");
    return MOE_OK;
  }
  if (!resid || !xn) return fail(MOE_EINVAL, "moe_stack_forward: NULL resid or xn");
  if (!aligned(resid, 16) || !aligned(xn, 16)) return fail(MOE_EINVAL, "moe_stack_forward: misaligned resid or xn");
  if (xn == resid) return fail(MOE_EINVAL, "moe_stack_forward: xn must not alias resid");
  for (int32_t l = 0; l < n_layers; ++l) {
    // resid <- resid + MoE_l(rms_norm(resid)). From the second layer on every kernel is a
    // programmatic dependent of the one before it (each waits for its predecessor before it
    // reads or writes anything that kernel, or an earlier one, touches), and the status word is
    // kept, so after the call it holds the flags of every layer.
    cudaError_t e = launch_rms_norm(*shape, resid, rdt, xn, rdt, eps, s, l > 0);
    if (e != cudaSuccess)
      return fail(MOE_ECUDA, "moe_stack_forward: RMS norm launch (layer %d): %s", (int)l, cudaGetErrorString(e));
    st = route_permute_impl(shape, xn, rdt, w_routers[l], topk_idx, topk_w, nullptr, counts, offsets, sorted_pair,
                            inv_pos, active, ws, ws_bytes, stream, true, l == 0);
    if (st != MOE_OK) return st;
    const CombineReq cmb{inv_pos, topk_w, resid, resid, rdt};
    st = expert_ffn_impl(shape, mode, xn, rdt, &experts[l], offsets, sorted_pair, active, y_perm, ydt, ws, ws_bytes,
                         stream, &cmb, true);
    if (st != MOE_OK) return st;
  }
  return MOE_OK;
}

moe_status moe_combine(const moe_shape* shape, const void* y_perm, moe_dtype ydt, const int32_t* inv_pos,
                       const float* topk_w, const void* residual_opt, void* out, moe_dtype odt,
                       moe_stream_t stream) {
  moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  if ((st = check_dtype(ydt, "y_perm")) != MOE_OK) return st;
  if ((st = check_dtype(odt, "out")) != MOE_OK) return st;
  if (shape->T == 0) return MOE_OK;
  if (!y_perm || !inv_pos || !topk_w || !out) return fail(MOE_EINVAL, "moe_combine: NULL argument");
  if (!aligned(y_perm, 16) || !aligned(out, 16) || (residual_opt && !aligned(residual_opt, 16)))
    return fail(MOE_EINVAL, "moe_combine: misaligned y_perm, out or residual");
  cudaError_t e = launch_combine(*shape, y_perm, ydt, inv_pos, topk_w, residual_opt, out, odt,
                                 reinterpret_cast<cudaStream_t>(stream), false);
  if (e != cudaSuccess) return cuda_fail(e, "moe_combine: launch");
  return MOE_OK;
}

moe_status moe_rms_norm(const moe_shape* shape, const void* x, moe_dtype xdt, void* out, moe_dtype odt, float eps,
                        moe_stream_t stream) {
  moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  if ((st = check_dtype(xdt, "x")) != MOE_OK) return st;
  if ((st = check_dtype(odt, "out")) != MOE_OK) return st;
  if (!(eps >= 0.0f) || !isfinite(eps)) return fail(MOE_EINVAL, "moe_rms_norm: eps must be finite and >= 0");
  if (shape->T == 0) return MOE_OK;
  if (!x || !out) return fail(MOE_EINVAL, "moe_rms_norm: NULL argument");
  if (!aligned(x, 16) || !aligned(out, 16)) return fail(MOE_EINVAL, "moe_rms_norm: misaligned x or out");
  if (x == out && xdt != odt) return fail(MOE_EINVAL, "moe_rms_norm: in place needs xdt == odt");
  cudaError_t e = launch_rms_norm(*shape, x, xdt, out, odt, eps, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "moe_rms_norm: launch");
  return MOE_OK;
}

moe_status moe_filter_resident(const int32_t* active, const int32_t* slot_of, int32_t E, int32_t* out,
                               moe_stream_t stream) {
  if (!active || !slot_of || !out || E <= 0) return fail(MOE_EINVAL, "moe_filter_resident: NULL argument or E <= 0");
  if (out == active) return fail(MOE_EINVAL, "moe_filter_resident: out must not alias active");
  const cudaError_t e = launch_filter_resident(active, slot_of, E, out, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "moe_filter_resident: launch");
  return MOE_OK;
}

moe_status moe_set_wait_limit(uint64_t ns) {
  if (ns > kMaxWaitNs) return fail(MOE_EINVAL, "moe_set_wait_limit: %llu ns is above 10 s", (unsigned long long)ns);
  g_wait_ns.store(ns ? ns : kDefaultWaitNs, std::memory_order_relaxed);
  return MOE_OK;
}

moe_status moe_read_status(const void* ws, moe_stream_t stream, int32_t* h_status) {
  if (!ws || !h_status) return fail(MOE_EINVAL, "moe_read_status: NULL argument");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemcpy(h_status, ws, sizeof(int32_t), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "moe_read_status");
  return *h_status ? MOE_EDEVICE : MOE_OK;
}

}  // extern "C"
