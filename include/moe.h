/*
 * moe.h: C-ABI of the B300 (sm_103a) sparse MoE layer forward pass.
 *
 * One MoE layer's forward pass runs as four calls on one CUDA stream:
 *
 *   moe_route       router logits (fp32), top-k and renormalised gate weights
 *   moe_permute     bucketing: group the (token, slot) pairs by expert
 *   moe_expert_ffn  each selected expert's SwiGLU FFN over int8 (or 2-bit) block-32 weights,
 *                   looked up through the resident slot table, plus the always-on shared experts
 *   moe_combine     weighted sum of the expert outputs per token (unpermute)
 *
 * or fused: moe_route_permute (the first two), moe_expert_ffn_combine (the last two),
 * moe_layer_forward (all four in one call). Around them:
 *   moe_rms_norm    (stacks of layers) the normalised input of a pre-norm residual block
 *   moe_stack_forward  L resident layers in one call (norm and layer per layer, one chain)
 *   slot_table_*    host-side slot pool for experts that do not all fit on the device: a miss
 *                   is copied from pinned host memory on a side stream; early loading of a
 *                   later layer's experts; residency lookups
 *   moe_filter_resident  the resident experts of an active list, on the device
 *   moe_host_expert_ffn  the expert FFN on the host CPU (the bandwidth split of the miss path)
 *   moe_tiered_*    a native executor of a whole tiered L-layer step
 *   moe_permute_static  bucketing without a caller workspace
 *
 * Sources. The pages on the Strata engine describe the method:
 *   [run-5090] "单张RTX 5090跑125B大模型：Strata实测Qwen3.8 Flash Next", section "MoE专家按需调度":
 *        a light router picks the top-K experts per token and the other experts take no part;
 *        experts not selected can leave VRAM and are brought back when the router picks them.
 *   [tiers] "Strata 工作原理图解GPU内存SSD三级存储如何让125B模型塞进消费级显卡":
 *        section "三级存储分工": router and shared expert resident in VRAM, all experts pinned in RAM;
 *        section "专家缓存": a VRAM expert cache of the most used experts; misses live in RAM;
 *        section "长文本": the next layer's experts stream over PCIe while the current layer computes.
 *   [bench] "Strata 性能基准与论文导读125B MoE在消费级硬件上的极限测量与瓶颈分析", section "瓶颈分析 1️⃣":
 *        quantised expert matmuls on tensor cores without a separate dequantisation pass.
 * The pages leave the FFN form, weight format, gate and tie-break open. The readings taken
 * here are: SwiGLU without biases; int8 codes with one fp16 scale per 32 elements of the
 * reduction dimension; softmax over all E restricted to the top k and renormalised; ties to
 * the lowest expert index; and shared experts added with weight 1.
 *
 * Conventions for every call:
 *  - All pointers are DEVICE pointers unless the name starts with h_. The caller owns all
 *    memory, and the library allocates nothing on the calls of a pass (slot_table_create and
 *    moe_tiered_create allocate their own state once, at creation).
 *  - Arrays are dense and row-major. x, y_perm, out, w_router and the workspace must be
 *    16-byte aligned (the workspace 256-byte aligned). Expert records are 256-byte aligned.
 *  - Calls are asynchronous on `stream` and return at once. A negative moe_status is a
 *    host-side error found before any launch (nothing was enqueued) or a failed launch.
 *  - Errors found by kernels (a NaN logit, an expert index out of range, a routed expert
 *    with no resident slot) set bits of a device status word in the workspace. Nothing
 *    traps. moe_read_status() returns that word.
 *  - T == 0 is valid: moe_route clears the status word, moe_permute writes zero counts and
 *    an empty active list, and the other calls check their arguments and enqueue nothing.
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* the same type as cudaStream_t */
typedef struct CUevent_st* moe_event_t;   /* the same type as cudaEvent_t */

typedef enum {
  MOE_OK = 0,
  MOE_EINVAL = -1,        /* null pointer, bad shape, misalignment, k > E, d or f not a multiple of 32 */
  MOE_EUNSUPPORTED = -2,  /* valid but outside what the kernels handle (e.g. k > 32, E > 1024) */
  MOE_ECUDA = -3,         /* a CUDA launch or copy failed; moe_last_error_string() has the detail */
  MOE_ENOSLOT = -4,       /* slot_table_update: more misses than evictable slots */
  MOE_EDEVICE = -5        /* moe_read_status: the device status word is non-zero */
} moe_status;

/* device status word bits (moe_read_status) */
#define MOE_DEV_NAN_LOGIT    0x1  /* a router logit was NaN; it was ranked below every number */
#define MOE_DEV_BAD_EXPERT   0x2  /* a topk_idx entry was outside [0, E); outputs are undefined */
#define MOE_DEV_MISSING_SLOT 0x4  /* a routed expert had slot_of[e] < 0; its rows were left unwritten */
#define MOE_DEV_TIMEOUT      0x8  /* a kernel's bounded wait ran out; that kernel's outputs are incomplete */
#define MOE_DEV_BAD_SLOT     0x10 /* a routed expert had slot_of[e] >= n_slots; its rows were left unwritten */

typedef enum { MOE_BF16 = 0, MOE_F32 = 1 } moe_dtype;

/* Which expert-FFN kernels run (moe_expert_ffn). All give the same result within the bf16
 * tolerance; each is deterministic.
 *  DECODE   few tokens per expert: the int8 codes stream from HBM straight into f16
 *           tensor-core fragments (weights exact, x and h rounded once to f16 after a
 *           power-of-two rescale). T <= 8: one persistent cooperative kernel; 8 < T <= 16 (or
 *           shapes whose shared-memory staging does not fit): three kernels. xdt = MOE_F32
 *           (the fp32 debug mode), and DECODE asked for explicitly with T > 16, run the fp32
 *           SIMT kernels instead: exact-weight fp32 arithmetic, far slower than either
 *           tensor-core path.
 *  PREFILL  many tokens per expert: a tcgen05 grouped GEMM (int8 codes and token rows by TMA,
 *           the codes converted to f16 straight into tensor memory as the MMA's A operand, the
 *           token tile as its N, fp32 accumulators in tensor memory). Needs
 *           xdt = MOE_BF16, d a multiple of 256 and f of 128 (else MOE_EUNSUPPORTED).
 *  AUTO     xdt = MOE_F32: the fp32 SIMT kernels. xdt = MOE_BF16: DECODE for T <= 16 and
 *           PREFILL for T > 16; a shape that PREFILL does not take with T > 16 returns
 *           MOE_EUNSUPPORTED (nothing enqueued) rather than falling back to the SIMT kernels.
 *           Ask for DECODE explicitly to run those. */
typedef enum { MOE_MODE_AUTO = 0, MOE_MODE_DECODE = 1, MOE_MODE_PREFILL = 2 } moe_mode;

/* Problem shape. T tokens, model width d, expert hidden width f, E routed experts,
 * top-k, n_shared always-on experts. P = T * k routed (token, slot) pairs. */
typedef struct {
  int32_t T, d, f, E, k, n_shared;
} moe_shape;

/* Byte offsets of one expert record. Each section starts on a 256-byte boundary:
 *   gate_q [f][d] int8, up_q [f][d] int8, down_q [d][f] int8,
 *   gate_s [f][d/32] fp16, up_s [f][d/32] fp16, down_s [d][f/32] fp16.
 * Weight W[r][i] = q[r][i] * s[r][i/32]; blocks run along the reduction dimension.
 * Stored order of a code row of K codes: in each 64-code span (blocks 2p and 2p + 1) the
 * 16-byte chunk c holds codes 8c..8c+7 of block 2p and then codes 8c..8c+7 of block 2p + 1,
 * i.e. code i of the row sits at byte 64*(i/64) + 16*((i/8)%4) + 8*((i/32)%2) + i%8; a trailing
 * block without a partner (K not a multiple of 64) is stored in order. One 16-byte load then
 * gives a lane the same 8 codes of two blocks. Scales are stored in order. */
typedef struct {
  uint64_t gate_q, up_q, down_q, gate_s, up_s, down_s, record_bytes;
} moe_expert_layout;

/* Fills *out for (d, f). Host only, no CUDA call. MOE_EINVAL if d or f is not a positive
 * multiple of 32 or out is NULL. */
moe_status moe_get_expert_layout(int32_t d, int32_t f, moe_expert_layout* out);

/* Expert record formats (moe_expert_table.format).
 *  MOE_FMT_INT8  int8 codes and one fp16 scale per 32 weights (8.5 bits per weight), the layout
 *                of moe_get_expert_layout.
 *  MOE_FMT_Q2    the sub-4-bit format of the pages' ~2.4 bits-per-weight experts ("Strata 工作原理图解
 *                GPU内存SSD三级存储如何让125B模型塞进消费级显卡", sections "专家缓存" and "实测速度": 2-bit
 *                quantised experts, about 700 of them per GB): 2-bit codes c in 0..3 and one fp16
 *                scale s per 32 weights along the reduction dimension, W = s * (c - 1.5), 2.5 bits
 *                per weight. Sections as in MOE_FMT_INT8, the code sections a quarter of the size:
 *                gate_q [f][d/4], up_q [f][d/4], down_q [d][f/4] bytes. In a code row, each group of
 *                8 blocks (256 codes) is 64 bytes: 16-byte chunk q holds, for block b = 0..7, the
 *                little-endian 16-bit word of codes 8q..8q+7 of block b, code j (0..7) at bits
 *                2 * slot(j) with slot(0..7) = 0, 2, 1, 3, 4, 6, 5, 7. Needs d and f multiples of
 *                256, and the decode expert FFN (bf16 x, T <= 8); other kernels return
 *                MOE_EUNSUPPORTED for it. */
#define MOE_FMT_INT8 0
#define MOE_FMT_Q2 1

/* Fills *out for (d, f) in record format `format`. Host only. MOE_EINVAL for a bad format, d or f
 * not a positive multiple of 32 (of 256 for MOE_FMT_Q2), or out NULL. */
moe_status moe_get_record_layout(int32_t d, int32_t f, int32_t format, moe_expert_layout* out);

/* Where the experts of one layer live.
 *  pool       device: slot records, slot s at pool + s * slot_bytes, s < n_slots (records in
 *             `format`; a zero-filled table means MOE_FMT_INT8)
 *  slot_bytes stride of the pool: >= record_bytes and a multiple of 256
 *  slot_of    device int32 [E]: slot of routed expert e, or -1 when it is not resident
 *             (the row of one layer of the slot table; [tiers] "专家缓存")
 *  shared     device: n_shared records at shared + s * slot_bytes; NULL iff n_shared == 0
 *  n_slots    number of slots in the pool (> 0). A slot_of entry >= n_slots is an error
 *             (MOE_DEV_BAD_SLOT) and that expert's rows are not written.
 * The table is only read. It is the caller's (or slot_table_update's) job to keep it current. */
typedef struct {
  const void* pool;
  uint64_t slot_bytes;
  const int32_t* slot_of;
  const void* shared;
  uint64_t n_slots;
  uint32_t format; /* MOE_FMT_INT8 or MOE_FMT_Q2, for every record of the table */
} moe_expert_table;

/* Bytes of workspace that moe_route / moe_permute / moe_expert_ffn need for this shape
 * (any mode, either dtype). One workspace serves one layer's calls from moe_route to
 * moe_combine. Its first 256 bytes hold the device status word. Host only.
 * The decode expert FFN keeps counters in the workspace that must read zero when it starts.
 * moe_route clears them (and the status word) for its shape, and every moe_expert_ffn call
 * leaves them at zero, even one whose wait ran out. So fill a new workspace with zeros before
 * its first use (cudaMemset, torch.zeros), and again before using it with another shape, unless
 * moe_route with that shape comes first. */
moe_status moe_workspace_size(const moe_shape* shape, size_t* bytes);

/* Router and top-k ([run-5090] "MoE专家按需调度": the router picks the top-K experts per token).
 *  x          [T][d], bf16 (xdt = MOE_BF16) or fp32 (MOE_F32)
 *  w_router   fp32 [d][E]
 *  topk_idx   out int32 [T][k]: the k experts with the largest fp32 logits, descending
 *             logit, ties to the lowest index, -0.0 equal to +0.0, NaN below every number
 *  topk_w     out fp32 [T][k]: exp(l_j - l_0) / sum_j' exp(l_j' - l_0) over the selected
 *             logits (equal to softmax over all E, restricted and renormalised)
 *  logits_opt out fp32 [T][E] or NULL: logit[t][e] = sum_i x[t][i] * w_router[i][e], fp32
 *             accumulation in a fixed order (deterministic)
 *  ws         workspace of moe_workspace_size bytes. The status word is cleared here.
 * Limits: k <= 32 and E <= 1024 (else MOE_EUNSUPPORTED). */
moe_status moe_route(const moe_shape* shape, const void* x, moe_dtype xdt, const float* w_router,
                     int32_t* topk_idx, float* topk_w, float* logits_opt, void* ws, size_t ws_bytes,
                     moe_stream_t stream);

/* Bucketing and permutation of the P = T*k pairs by expert, so that each selected expert's
 * weights are streamed once for all of its tokens ([tiers] "专家缓存": the GPU computes the
 * experts the cache holds). Deterministic and free of atomics.
 *  topk_idx    int32 [T][k]; pair p = t*k + j routes token t to expert topk_idx[p]
 *  counts      out int32 [E]: pairs routed to each expert
 *  offsets     out int32 [E+1]: exclusive prefix sum of counts (offsets[E] = P)
 *  sorted_pair out int32 [P]: pair ids grouped by expert, ascending pair id inside a group
 *  inv_pos     out int32 [P]: position of pair p in sorted_pair
 *  active      out int32 [1 + min(E, P)]: active[0] = number of experts with a pair, then
 *              those experts in ascending order
 * An index outside [0, E) sets MOE_DEV_BAD_EXPERT (outputs then undefined, all writes in bounds). */
moe_status moe_permute(const moe_shape* shape, const int32_t* topk_idx, int32_t* counts,
                       int32_t* offsets, int32_t* sorted_pair, int32_t* inv_pos, int32_t* active,
                       void* ws, size_t ws_bytes, moe_stream_t stream);

/* moe_route followed by moe_permute, in one call: the same outputs, bit for bit, with the same
 * arguments (see both). For few tokens the top-k and the bucketing run as one kernel, a cluster
 * of T CTAs with one per token, which saves a launch and a round trip through global memory.
 * That takes T <= 8, T*k <= 256, E <= 512 with E a multiple of 4, and one token's router split
 * partial sums within 100 KB of shared memory; otherwise the two calls' kernels run one after
 * the other. */
moe_status moe_route_permute(const moe_shape* shape, const void* x, moe_dtype xdt, const float* w_router,
                             int32_t* topk_idx, float* topk_w, float* logits_opt, int32_t* counts,
                             int32_t* offsets, int32_t* sorted_pair, int32_t* inv_pos, int32_t* active,
                             void* ws, size_t ws_bytes, moe_stream_t stream);

/* Bucketing without a workspace, for callers that cannot allocate device memory where they
 * bucket: for example an engine that sizes all device memory once at start-up and lets no
 * library add to it, or a serving path where a cudaMalloc could stall the device. The pages
 * have no counterpart: this is the same computation as moe_permute, with the same outputs,
 * kernels and error bits, but its scratch is a fixed array inside this library. The array
 * is 512 KiB on every GPU that loads the library and is held until the process exits.
 *  status  out int32 (device): cleared by this call, then receives the MOE_DEV_* bits
 * Limits: T*k <= 65536 pairs and E <= 1024, else MOE_EUNSUPPORTED (nothing enqueued).
 * The first call on a device looks up the array's device address with that device current
 * (cudaGetSymbolAddress). Make that first call before any stream capture. It allocates nothing
 * (no cudaMalloc, no cudaFree). All calls in the process share the one array and every call
 * rewrites all of the scratch it reads, so nothing carries over from an earlier call. Two
 * calls whose work overlaps on the GPU (e.g. on two streams) race on the array and give
 * undefined results: order them on one stream or with events. */
moe_status moe_permute_static(const moe_shape* shape, const int32_t* topk_idx, int32_t* counts,
                              int32_t* offsets, int32_t* sorted_pair, int32_t* inv_pos,
                              int32_t* active, int32_t* status, moe_stream_t stream);

/* Expert FFN ([run-5090] "MoE专家按需调度": only the experts the router picked compute for a token;
 * [tiers] "专家缓存": each is computed from its copy in the VRAM expert cache, found through the
 * slot table; [tiers] "三级存储分工": the resident shared expert applies to every token): for
 * every expert in `active` (and every shared expert), for each of its rows
 * y = W_down (silu(W_gate x) * (W_up x)), silu(z) = z / (1 + e^-z), W = q * s per block of 32.
 * The expert's record is found through the slot table (experts->slot_of).
 *  x           [T][d] (xdt), the same activations given to moe_route
 *  offsets, sorted_pair, active: from moe_permute (active may also be any caller list in
 *              the same format, e.g. only the experts already resident)
 *  y_perm      out [P + T*n_shared][d] (ydt): row offsets[e] + i holds expert e's output for
 *              pair sorted_pair[offsets[e] + i]; row P + s*T + t holds shared expert s for token t
 *  ydt         MOE_F32 or MOE_BF16 (a bf16 y_perm halves the combine's reads)
 * mode: see moe_mode. A routed expert with slot_of[e] < 0 sets MOE_DEV_MISSING_SLOT and its
 * rows are not written. The call may run a memset and a cooperative launch on `stream`; a
 * bounded wait inside a kernel that runs out sets MOE_DEV_TIMEOUT (outputs incomplete). */
moe_status moe_expert_ffn(const moe_shape* shape, moe_mode mode, const void* x, moe_dtype xdt,
                          const moe_expert_table* experts, const int32_t* offsets,
                          const int32_t* sorted_pair, const int32_t* active, void* y_perm,
                          moe_dtype ydt, void* ws, size_t ws_bytes, moe_stream_t stream);

/* Expert FFN followed by the combine, in one call: moe_expert_ffn and then moe_combine with
 * these arguments, launched one after the other on `stream` (the same results, bit for bit).
 * Arguments as in moe_expert_ffn and moe_combine; out may alias residual_opt. */
moe_status moe_expert_ffn_combine(const moe_shape* shape, moe_mode mode, const void* x, moe_dtype xdt,
                                  const moe_expert_table* experts, const int32_t* offsets,
                                  const int32_t* sorted_pair, const int32_t* active, void* y_perm,
                                  moe_dtype ydt, const int32_t* inv_pos, const float* topk_w,
                                  const void* residual_opt, void* out, moe_dtype odt, void* ws,
                                  size_t ws_bytes, moe_stream_t stream);

/* The whole layer in one call: moe_route_permute, then moe_expert_ffn_combine with the same
 * arguments (the same results, bit for bit). Because the library enqueues every kernel of the
 * pass itself, the decode expert FFN starts as a programmatic dependent of the bucketing kernel
 * before it: it stages the activations while the bucketing runs and reads the bucketing's
 * outputs once that kernel has completed. (The separate calls never start a kernel early on
 * work the caller enqueued, which could be a copy or an event wait.) out may alias
 * residual_opt. */
moe_status moe_layer_forward(const moe_shape* shape, const void* x, moe_dtype xdt, const float* w_router,
                             const moe_expert_table* experts, moe_mode mode, int32_t* topk_idx, float* topk_w,
                             float* logits_opt, int32_t* counts, int32_t* offsets, int32_t* sorted_pair,
                             int32_t* inv_pos, int32_t* active, void* y_perm, moe_dtype ydt,
                             const void* residual_opt, void* out, moe_dtype odt, void* ws, size_t ws_bytes,
                             moe_stream_t stream);

/* Combine / unpermute ([run-5090]: the token's output is the gated mixture of its selected
 * experts; [tiers] "三级存储分工": the shared expert applies to every token):
 *   out[t] = sum_{j=0..k-1} topk_w[t][j] * y_perm[inv_pos[t*k+j]]
 *            + sum_s y_perm[P + s*T + t] + (residual_opt ? residual_opt[t] : 0)
 * summed in fp32 in exactly that order, then rounded once to odt (bf16: nearest-even).
 *  residual_opt [T][d] in odt's type, or NULL. out may alias residual_opt. */
moe_status moe_combine(const moe_shape* shape, const void* y_perm, moe_dtype ydt,
                       const int32_t* inv_pos, const float* topk_w, const void* residual_opt,
                       void* out, moe_dtype odt, moe_stream_t stream);

/* RMS normalisation of each token's row, the input of one layer of a stack. The pages run
 * the layers of a transformer but leave the residual block open; the reading taken here is
 * the pre-norm block x_{l+1} = x_l + MoE_l(n(x_l)), with n given by
 *   out[t][i] = x[t][i] / sqrt(mean_j x[t][j]^2 + eps)      (no learned gain)
 * The mean of squares is an fp32 sum in a fixed order (deterministic); out is rounded once
 * to odt. Only shape->T and shape->d are used.
 *  x    [T][d] in xdt's type; out [T][d] in odt's type; both 16-byte aligned. out may be x
 *       when xdt == odt.
 *  eps  finite and >= 0 (MOE_EINVAL otherwise). */
moe_status moe_rms_norm(const moe_shape* shape, const void* x, moe_dtype xdt, void* out,
                        moe_dtype odt, float eps, moe_stream_t stream);

/* A stack of n_layers resident MoE layers ([run-5090]: the router runs per layer of the
 * transformer; [tiers] "三级存储分工": every layer's router and shared expert stay in VRAM),
 * on the pre-norm residual reading of moe_rms_norm:
 *   for l = 0 .. n_layers-1:  resid <- resid + MoE_l(rms_norm(resid))
 * Each layer is moe_rms_norm(resid -> xn) followed by moe_layer_forward(xn, w_routers[l],
 * experts[l], residual = out = resid), with the same results bit for bit. The library
 * enqueues the whole chain itself, so from the second kernel on every kernel starts as a
 * programmatic dependent of the one before it (layer l+1's norm overlaps the end of layer l's
 * combine; the router overlaps the norm); each waits for its predecessor before touching
 * memory that an earlier kernel uses.
 *  n_layers    >= 0 (0, or T == 0: only the status word is cleared)
 *  w_routers   HOST array of n_layers device pointers, each fp32 [d][E], 16-byte aligned
 *  experts     HOST array of n_layers expert tables (see moe_expert_table)
 *  resid       in/out [T][d] in rdt's type (MOE_BF16 or MOE_F32); xn: [T][d] rdt scratch that
 *              holds the last layer's normalised input afterwards; neither may alias the other
 *  eps         the RMS norm's eps (finite, >= 0)
 *  topk_idx .. active, y_perm, ws: one set for all layers (as in moe_layer_forward); after the
 *              call they hold the last layer's routing, bucketing and expert outputs
 * The status word is cleared once, at the first layer, and gathers the flags of every layer.
 * A host-side error at layer l returns at once; the earlier layers' kernels stay enqueued. */
moe_status moe_stack_forward(const moe_shape* shape, int32_t n_layers, const float* const* w_routers,
                             const moe_expert_table* experts, moe_mode mode, void* resid, moe_dtype rdt,
                             float eps, void* xn, int32_t* topk_idx, float* topk_w, int32_t* counts,
                             int32_t* offsets, int32_t* sorted_pair, int32_t* inv_pos, int32_t* active,
                             void* y_perm, moe_dtype ydt, void* ws, size_t ws_bytes, moe_stream_t stream);

/* Limit of the bounded waits inside the expert-FFN kernels (a CTA waiting for work that other
 * CTAs or its own warps publish), in nanoseconds, for every moe_expert_ffn /
 * moe_expert_ffn_combine call made after this one in the process. 0 restores the default of
 * 1 s, which no legitimate wait comes near. A wait that runs out sets MOE_DEV_TIMEOUT and the
 * kernel abandons its remaining work; asynchronous copies and tensor-core operations already
 * issued are still waited for (with the default limit) before the kernel exits. A short limit
 * makes that failure path run on purpose, e.g. in a test, with no fault. MOE_EINVAL above
 * 10 s. No counterpart on the pages: this is error handling of the kernels. */
moe_status moe_set_wait_limit(uint64_t ns);

/* Waits for `stream`, then returns the device status word of workspace `ws` in *h_status.
 * MOE_OK if it is zero, MOE_EDEVICE if not, MOE_ECUDA if the copy failed. */
moe_status moe_read_status(const void* ws, moe_stream_t stream, int32_t* h_status);

/* Message of the last MOE_ECUDA / MOE_EINVAL returned on this host thread ("" if none). */
const char* moe_last_error_string(void);

/* ------------------------------------------------------------------------------------
 * Slot table: an expert cache for experts that do not all fit in device memory
 * ([tiers] "专家缓存" and "三级存储分工": the most used experts stay in VRAM, all experts
 * sit pinned in host RAM; [tiers] "长文本": expert copies overlap with computation).
 * The table keeps, on the host, the owner (layer, expert) of each of n_slots device slots,
 * their LRU order, and a decayed use count of every (layer, expert) ([tiers] "专家缓存": the
 * cache starts from a ranking of expert use and adapts to what the session uses most). The
 * device table d_slot_of [L][E] lives in caller memory. Row `layer` of it is what
 * moe_expert_ffn reads through moe_expert_table.slot_of.
 * ------------------------------------------------------------------------------------ */
typedef struct moe_slot_table moe_slot_table;

typedef struct {
  uint64_t hits, misses, evictions, bytes_h2d;
} moe_slot_stats;

/* Replacement policy (slot_table_set_policy). */
typedef enum {
  MOE_SLOT_LRU = 0,  /* evict the least recently used slot (the default) */
  MOE_SLOT_FREQ = 1  /* evict the slot whose owner has the smallest decayed use count */
} moe_slot_policy;

/* Copies `bytes` from host `h_src` to device `d_dst` on `stream`; returns 0 on success.
 * The default copier is cudaMemcpyAsync. A caller can pass its own (e.g. to add tracing,
 * or in tests to inject a failure). */
typedef int (*moe_copy_fn)(void* d_dst, const void* h_src, size_t bytes, moe_stream_t stream,
                           void* user);

/* Creates a table over n_slots slots of slot_bytes at d_pool (device), for L layers of E
 * experts whose records sit at h_records[l*E + e] (pinned host memory, slot_bytes each;
 * the same pointer may repeat). All slots start empty and d_slot_of is set to -1 (a
 * synchronous cudaMemset). copy_fn may be NULL (cudaMemcpyAsync). */
moe_status slot_table_create(moe_slot_table** out, int32_t L, int32_t E, int32_t n_slots,
                             uint64_t slot_bytes, void* d_pool, int32_t* d_slot_of,
                             const void* const* h_records, moe_copy_fn copy_fn, void* copy_user);

/* Makes every expert of h_active[0..n_active) (host array) resident for `layer`:
 *  - a resident expert is a hit; it moves to the most-recently-used end;
 *  - every expert of h_active counts one use (see slot_table_set_policy);
 *  - a miss takes, among the slots whose owner is not in h_active, an empty slot first, else
 *    the policy's victim: the least recently used slot (MOE_SLOT_LRU) or the slot whose
 *    owner has the smallest decayed use count, ties to the least recently used and then
 *    the lowest slot index (MOE_SLOT_FREQ). It is copied from h_records on copy_stream and
 *    marked most recent;
 *  - the changed entries of row `layer` of d_slot_of are then written on copy_stream, and
 *    `ready` (if not NULL) is recorded on copy_stream after all copies.
 * A compute stream that waits on `ready` sees the new row. Hits can run before `ready`.
 * Optional outputs: h_hits / h_misses (host int32 arrays of capacity n_active) receive
 * the hit and miss expert ids in h_active order, with their counts in *n_hits / *n_misses.
 * MOE_ENOSLOT if the misses outnumber the slots not owned by h_active (the table is left
 * unchanged), MOE_ECUDA if a copy fails (the failed expert is not marked resident),
 * MOE_EINVAL for a bad layer or expert id or a repeated id. */
moe_status slot_table_update(moe_slot_table* table, int32_t layer, const int32_t* h_active,
                             int32_t n_active, moe_stream_t copy_stream, moe_event_t ready,
                             int32_t* h_hits, int32_t* n_hits, int32_t* h_misses,
                             int32_t* n_misses, moe_slot_stats* stats_opt);

/* Early loading of the experts a later layer is expected to use, while the current layer
 * computes ("Strata 性能基准与论文导读125B MoE在消费级硬件上的极限测量与瓶颈分析", section "瓶颈分析
 * 1️⃣": next-layer experts streamed over PCIe behind the current layer's compute; "Strata 工作
 * 原理图解GPU内存SSD三级存储如何让125B模型塞进消费级显卡", section "长文本"). For every expert of
 * h_ids[0..n_ids) (host array, ids of `layer`) that is not resident: a victim slot is chosen as
 * in slot_table_update (an empty slot first, then the policy's victim) among the slots whose
 * owner is neither one of h_keep[0..n_keep) of keep_layer (the experts the current layer's
 * kernels read; keep_layer is ignored when n_keep == 0) nor one of h_ids; the record is copied
 * on copy_stream and the slot becomes the most recently used. When no slot can be taken the
 * call loads what it could and returns MOE_OK. Already resident experts are left as they are.
 * The loads are not uses (no use counts, hits or misses); bytes_h2d and evictions count them.
 * The changed entries of d_slot_of are written after the copies and `ready` (if not NULL) is
 * recorded after that: a compute stream must wait on it before it reads a prefetched slot.
 * *n_loaded (if not NULL) receives the number of experts copied. MOE_EINVAL for bad layers or
 * ids (nothing changed), MOE_ECUDA if a copy fails (the failed expert is not resident). The
 * protocol of slot_table_update holds: the kernels that read an evicted slot have completed. */
moe_status slot_table_prefetch(moe_slot_table* table, int32_t layer, const int32_t* h_ids, int32_t n_ids,
                               int32_t keep_layer, const int32_t* h_keep, int32_t n_keep, moe_stream_t copy_stream,
                               moe_event_t ready, int32_t* n_loaded);

/* Prefetched experts so far (*loads), and how many of them a later slot_table_update found
 * resident and counted as hits before they were evicted (*used). */
moe_status slot_table_prefetch_stats(const moe_slot_table* table, uint64_t* loads, uint64_t* used);

/* Sets the replacement policy (MOE_SLOT_LRU or MOE_SLOT_FREQ) and the half-life of the use
 * counts, in slot_table_update calls (> 0, finite): a use made h calls ago weighs 2^(-h /
 * half_life) of a use made now. Counts are kept under both policies (with no decay until a
 * half-life is set), so the policy can change at any time. MOE_EINVAL otherwise. */
moe_status slot_table_set_policy(moe_slot_table* table, int32_t policy, double half_life);

/* Warm start from a usage profile ([tiers] "专家缓存": a shipped ranking of expert use decides
 * which experts start in VRAM). h_weight: host float [L*E] of use weights (>= 0, finite;
 * one use = 1), added to the use counts. Then the empty slots, lowest index first, take the
 * non-resident experts of positive weight in decreasing order of use count (ties: lower
 * l*E + e first); their records are copied on copy_stream, the changed entries of d_slot_of
 * written after them, and `ready` (if not NULL) recorded. Nothing is evicted. The loaded
 * slots join the recency order after the slots still empty, in increasing order of use count
 * (the highest count most recent), so that under MOE_SLOT_LRU the first evictions take the
 * loaded experts the profile ranks lowest. *n_loaded (if
 * not NULL) receives the number of experts copied; bytes_h2d counts them, hits and misses do
 * not. MOE_EINVAL for a NULL table or weights or a negative or non-finite weight (nothing
 * changed); MOE_ECUDA if a copy fails (the experts copied before it stay resident). */
moe_status slot_table_warm(moe_slot_table* table, const float* h_weight, moe_stream_t copy_stream,
                           moe_event_t ready, int32_t* n_loaded);

/* Host computation of missed experts: the bandwidth split of the miss path ([tiers] "专家缓存": the
 * experts a layer misses are divided between PCIe copies into the VRAM cache and computation
 * where their weights are, in host RAM; the share copied is the pages' --pcie-frac setting,
 * "Strata 性能基准与论文导读125B MoE在消费级硬件上的极限测量与瓶颈分析", section "如何测量"). Host
 * only, synchronous, no CUDA call. For each expert h_experts[i] (routed ids, distinct), whose
 * record (in `format`) is at h_records[i] in host memory, the SwiGLU FFN of each of its tokens:
 * its rows h_offsets[e] .. h_offsets[e+1]-1 of y_perm, token sorted_pair[row] / k of h_x [T][d]
 * (xdt), written in fp32 to h_y [T*k][d] at those rows (other rows untouched). fp32 arithmetic on
 * the exactly expanded weights; n_threads OpenMP threads (0: all). h_offsets [E+1] and
 * h_sorted_pair [T*k] are host copies of moe_permute's outputs. MOE_EINVAL for NULL arguments,
 * a bad format, id or offsets. Off the default path: only a caller that asks for the split runs it. */
moe_status moe_host_expert_ffn(const moe_shape* shape, const void* h_x, moe_dtype xdt,
                               const void* const* h_records, const int32_t* h_experts, int32_t n_experts,
                               const int32_t* h_offsets, const int32_t* h_sorted_pair, float* h_y, int32_t format,
                               int32_t n_threads);

/* The resident experts of one layer's active list: out (device int32 [1 + n]) = [m, e...] with
 * the experts e of active ([n, e_0 .. e_{n-1}], device) whose slot_of[e] (device int32 [E],
 * one row of a slot table's device table) is >= 0, in active-list order. Launched on
 * `stream`: run before the slot table's update of that layer, it lists the experts the update
 * will count as hits, so their expert FFN can start before the host has read the active list.
 * MOE_EINVAL for a NULL pointer, E <= 0 or out aliasing active. */
moe_status moe_filter_resident(const int32_t* active, const int32_t* slot_of, int32_t E, int32_t* out,
                               moe_stream_t stream);

/* ------------------------------------------------------------------------------------
 * Native executor of a tiered L-layer stack (all layers of one step in one call): per layer
 * the RMS norm of the residual stream, routing and bucketing, the active list read back, the
 * slot table's update (miss copies on the executor's own copy stream), the expert FFN of the
 * hit experts and the shared expert while the copies run, the missed experts after them, and
 * the combine into the residual stream ("Strata 工作原理图解GPU内存SSD三级存储如何让125B模型塞进
 * 消费级显卡", sections "三级存储分工" and "专家缓存"). Optionally the bandwidth split of the
 * miss path: the last floor((1 - pcie_frac) n) of a layer's n misses are computed on the host
 * (moe_host_expert_ffn) instead of copied ("Strata 性能基准与论文导读125B MoE在消费级硬件上的极限
 * 测量与瓶颈分析", section "如何测量"). The executor allocates its buffers (device and pinned
 * host) at creation; a forward call allocates nothing.
 * ------------------------------------------------------------------------------------ */
typedef struct moe_tiered moe_tiered;

/* shape: one layer (T, d, f, E, k, n_shared); routers: n_layers device pointers, fp32 [d][E];
 * shared: n_layers device pointers to each layer's n_shared records (NULL when n_shared = 0);
 * table, pool, slot_bytes, n_slots, slot_of: the slot table and the device pool and table
 * [n_layers][E] it manages (the caller owns them and keeps them alive); h_records: the
 * n_layers * E pinned host records, (layer, expert) order; format: MOE_FMT_INT8 or MOE_FMT_Q2;
 * eps: the RMS norm's epsilon. MOE_EINVAL for a NULL pointer, a bad shape or slot size. */
moe_status moe_tiered_create(const moe_shape* shape, int32_t n_layers, const float* const* routers,
                             const void* const* shared, moe_slot_table* table, void* pool, uint64_t slot_bytes,
                             uint64_t n_slots, int32_t* slot_of, const void* const* h_records, int32_t format,
                             float eps, moe_tiered** out);

/* The bandwidth split: pcie_frac in [0, 1] (1: every miss is copied, the default) and the host
 * threads of the host expert FFN (0: the OpenMP default). MOE_EINVAL otherwise. */
moe_status moe_tiered_set_split(moe_tiered* t, double pcie_frac, int32_t host_threads);

/* One step: every layer on the residual stream resid (device bf16 [T][d], updated in place),
 * launched on `stream`. The host waits once per layer for that layer's routing (the active
 * list); the call returns with the last layer's work enqueued. h_layer_misses / h_layer_host
 * (optional, host int32 [n_layers]): each layer's copied misses and host-computed experts.
 * An error returns at once with the layers before it enqueued and none after; kernels'
 * errors are in the status words (moe_tiered_status). */
moe_status moe_tiered_forward(moe_tiered* t, void* resid, moe_stream_t stream, int32_t* h_layer_misses,
                              int32_t* h_layer_host);

/* Waits for `stream`; *h_status = the OR of the device status words of the executor's
 * workspaces. MOE_OK when zero, MOE_EDEVICE if not. */
moe_status moe_tiered_status(moe_tiered* t, moe_stream_t stream, int32_t* h_status);

/* Waits for the executor's copy stream and frees its buffers. NULL is accepted. */
moe_status moe_tiered_destroy(moe_tiered* t);

/* Residency of experts of one layer: h_slot[i] (host) = the slot of expert h_ids[i] of `layer`, or
 * -1 when it is not resident. No state changes. MOE_EINVAL for a bad layer or id. */
moe_status slot_table_lookup(const moe_slot_table* table, int32_t layer, const int32_t* h_ids, int32_t n,
                             int32_t* h_slot);

/* Cumulative counters since creation. */
moe_status slot_table_stats(const moe_slot_table* table, moe_slot_stats* out);

/* Host mirror of d_slot_of [L][E]: copies L*E int32 into h_out. */
moe_status slot_table_snapshot(const moe_slot_table* table, int32_t* h_out);

moe_status slot_table_destroy(moe_slot_table* table);

#ifdef __cplusplus
}
#endif
#endif /* MOE_B300_H */
