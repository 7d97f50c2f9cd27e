// Internal interface between the C-ABI layer (capi.cu) and the kernel files.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <cuda_fp16.h>

#include "../../include/moe.h"

namespace moe {

constexpr int MOE_DEV_NAN_LOGIT_BIT = MOE_DEV_NAN_LOGIT;
constexpr int MOE_DEV_BAD_EXPERT_BIT = MOE_DEV_BAD_EXPERT;
constexpr int MOE_DEV_MISSING_SLOT_BIT = MOE_DEV_MISSING_SLOT;
constexpr int MOE_DEV_TIMEOUT_BIT = MOE_DEV_TIMEOUT;
constexpr int MOE_DEV_BAD_SLOT_BIT = MOE_DEV_BAD_SLOT;

constexpr int kRouteGemvMaxT = 16;   // tokens up to which the router runs as a split-d GEMV
constexpr int kRouteRowsPerSplit = 128;
constexpr int kPermChunk = 1024;     // pairs per bucketing chunk (one CTA)
constexpr int kDecodeMaxT = 16;      // AUTO picks the decode kernels up to this many tokens
constexpr int kDecodeTokGroup = 4;   // decode kernels stream weights once per group of tokens

// Byte offsets of the workspace regions (all 256-byte aligned).
struct WsLayout {
  size_t status;         // int32 device status word
  size_t route_partial;  // fp32 [S][T][E]: split-d router partial sums (T <= kRouteGemvMaxT)
  size_t logits;         // fp32 [T][E]: router GEMM output (T > kRouteGemvMaxT)
  size_t wparts;         // bf16 [3][E][d]: the router weights split in three exact parts (T > kRouteGemvMaxT)
  size_t perm_cnt;       // int32 [C][E]: per-chunk counts, then per-chunk bases
  size_t perm_keys;      // uint32 [C * kPermChunk]: chunk-sorted (expert, pair) keys
  size_t h;              // [P + T*n_shared][f] fp32: SwiGLU activations between the FFN kernels
  size_t x16;            // f16 [T][d]: activations rescaled per token by a power of two (permuted)
  size_t xunscale;       // fp32 [T]: the power of two that undoes that rescale
  size_t zero;           // start of the block the decode launcher zeroes with one memset:
  size_t item_done;      //   int32 [min(E, P) + n_shared]: gate/up tasks finished per work item
  size_t hmax;           //   uint32 [P + T*n_shared]: bits of max |h| per h row
  size_t task_cnt;       //   int32 [2][tasks]: stream-K parts finished per task (T <= 8 only)
  size_t zero_end;       // end of that block
  size_t items;          // ItemRec [min(E, P) + n_shared]: work items of the expert FFN
  size_t row_tok;        // int32 [P + T*n_shared]: token of each y_perm / h row
  size_t h16;            // f16 [P + T*n_shared][f]: h rescaled per row by a power of two (permuted)
  size_t hexp;           // int32 [P + T*n_shared]: the exponent e of that rescale (h = h16 * 2^e)
  size_t item_cnt;       // int32 [min(E, P) + n_shared + 2]: finished gate/up tasks per work item,
                         // then the task counters of the two streaming kernels
  size_t xp16;           // f16 [P + T*n_shared][d]: prefill activations gathered by row, rescaled per token
  size_t xexp;           // int32 [T]: the exponent of each token's rescale (prefill)
  size_t tiles;          // int2 [P/128 + items + 2]: prefill token tiles (item, first row), then the count
  size_t part;           // fp32 [2][tasks][2][128]: stream-K partial sums (T <= 8 only)
  size_t cx;             // fp32 [T][d/32]: MMA accumulator inputs of the x16 blocks
  size_t ch;             // fp32 [P + T*n_shared][f/32]: MMA accumulator inputs of the h16 blocks
  size_t total;
};

WsLayout ws_layout(const moe_shape& s);

// Records `msg` as this host thread's moe_last_error_string() and returns st.
moe_status report_error(moe_status st, const char* msg);

// Raises a kernel's dynamic shared memory limit to at least `bytes` on the current device
// (once per kernel and device).
cudaError_t ensure_dynamic_smem(const void* kernel, size_t bytes);
int route_splits(int d);
int perm_chunks(int P);

// Arguments of the expert FFN kernels (device pointers, already validated).
struct FfnArgs {
  const void* x;
  int xdt;  // 0 bf16, 1 fp32
  const uint8_t* pool;
  uint64_t slot_bytes;
  const int32_t* slot_of;
  const uint8_t* shared;
  uint64_t n_slots;
  const int32_t* offsets;
  const int32_t* sorted_pair;
  const int32_t* active;
  void* y;
  int ydt;
  float* h;  // fp32 [P + T*n_shared][f]
  int* status;
  uint64_t wait_ns;  // limit of the kernels' bounded waits for other threads' work (moe_set_wait_limit)
  int fmt;           // expert record format: 0 int8 codes, 1 the 2-bit format (MOE_FMT_Q2)
  int T, d, f, E, k, n_shared, P;
  // record layout
  uint64_t o_gate_q, o_up_q, o_down_q, o_gate_s, o_up_s, o_down_s;
};

// One work item of the expert FFN as the streaming kernels see it: the expert's record (NULL
// when the expert has no resident slot), its first y_perm / h row and its number of rows.
struct ItemRec {
  const uint8_t* rec;
  int row0;
  int ntok;
  int slot;    // slot in the pool, or the index of the shared expert
  int shared;  // 1: a shared expert (its record is in the shared array)
  int pad[2];
};

// Workspace buffers of the streaming expert-FFN kernels.
struct StreamAux {
  __half* x16;
  float* xunscale;
  uint32_t* hmax;
  ItemRec* items;
  int32_t* row_tok;
  __half* h16;
  int32_t* hexp;
  int32_t* item_cnt;
  float* cx;  // [T][d/32]: -1152 * (sum of each block of x16), the MMA accumulator input
  float* ch;  // [P + T*n_shared][f/32]: the same for h16
  int32_t* sched;  // [2]: next task of the gate/up and of the down kernel
  float* part;         // [2][part_stride]: stream-K partial sums (128 floats per part, 2 parts per task)
  int32_t* task_cnt;   // [2][cnt_stride]: stream-K parts finished per task
  size_t part_stride, cnt_stride;
};


// Workspace buffers of the persistent decode expert FFN. item_done, hmax, task_cnt and exit
// hold zeros when the kernel starts (moe_route clears them, and each launch leaves them so).
struct PersistAux {
  float* part;         // [2][part_stride]
  int32_t* task_cnt;   // [2][cnt_stride]
  uint32_t* hmax;      // [P + T*n_shared]
  int32_t* item_done;  // [min(E, P) + n_shared]
  size_t part_stride, cnt_stride;
  int32_t* exit;       // [2]: CTAs finished, and 1 if one of them abandoned its work
};

// Workspace buffers of the prefill (tensor-core GEMM) expert FFN.
struct PrefillAux {
  __half* xp16;       // [P + T*n_shared][d]: activation rows in expert order, f16, rescaled per token,
                      // each 64-element K step in the records' stored code order
  float* xunscale;    // [T]: 2^e of each token's rescale
  int32_t* xexp;      // [T]: e
  uint32_t* hmax;     // [P + T*n_shared]: bits of max |h| per row
  ItemRec* items;
  int32_t* row_tok;
  __half* h16;        // [P + T*n_shared][f]: h rescaled per row, in the stored code order like xp16
  int32_t* hexp;      // [P + T*n_shared]
  int2* tiles;        // token tiles of up to 128 rows: (item, first row within the item)
  int32_t* n_tiles;   // [1]
};

// Launchers; each returns cudaSuccess or the launch error.
// The router GEMV also sets *status to 0 (unless clear_status is false: a stack keeps the word
// across its layers) and clears zero[0, zero_bytes) (16-byte aligned, a multiple of 16 bytes)
// before any other kernel of the layer reads them.
// pdl: launched as a programmatic dependent of the kernel before it (the kernel waits for it
// before reading x or clearing anything).
cudaError_t launch_route_gemv(const moe_shape& s, const void* x, int xdt, const float* w, float* partial,
                              int* status, void* zero, size_t zero_bytes, cudaStream_t st, bool pdl = false,
                              bool clear_status = true);
// Top-k from the router GEMV's split partial sums [splits][T][E]: one CTA per token.
cudaError_t launch_topk_split(const moe_shape& s, const float* partial, int splits, int32_t* idx, float* wts,
                              float* logits_out, int* status, cudaStream_t st);
// Decode routing tail: the top-k of the router GEMV's split partial sums and the bucketing of
// the pairs, in one CTA (route_tail_supported says whether the shape fits).
bool route_tail_supported(const moe_shape& s);
cudaError_t launch_route_tail(const moe_shape& s, const float* partial, int splits, int32_t* idx, float* wts,
                              float* logits_out, int32_t* counts, int32_t* offsets, int32_t* sorted_pair,
                              int32_t* inv_pos, int32_t* active, int* status, cudaStream_t st);
// Router logits for T > 16 on the tensor cores (bf16 x; d a multiple of 256): the fp32 weights
// split into three exact bf16 parts in `parts` (route_tc_parts_bytes), then a tcgen05 GEMM. Both
// this and the SIMT GEMM also clear *status when clear_status is true.
bool route_tc_supported(const moe_shape& s, int xdt);
size_t route_tc_parts_bytes(const moe_shape& s);
cudaError_t launch_route_tc(const moe_shape& s, const void* x, const float* w, void* parts, float* logits, int* status,
                            cudaStream_t st, bool clear_status = true);
cudaError_t launch_route_gemm(const moe_shape& s, const void* x, int xdt, const float* w, float* logits,
                              int* status, cudaStream_t st, bool clear_status = true);
// Top-k of logits already summed (after the router GEMM): one warp per token.
cudaError_t launch_topk(const moe_shape& s, const float* logits, int32_t* idx, float* wts, int* status,
                        cudaStream_t st);
cudaError_t launch_permute(const moe_shape& s, const int32_t* topk_idx, int32_t* counts, int32_t* offsets,
                           int32_t* sorted_pair, int32_t* inv_pos, int32_t* active, int32_t* cnt,
                           uint32_t* keys, int* status, cudaStream_t st, bool pdl = false);
// The resident experts (slot_of >= 0) of an active list, in order, as an active list.
cudaError_t launch_filter_resident(const int32_t* active, const int32_t* slot_of, int E, int32_t* out,
                                   cudaStream_t st);
cudaError_t launch_ffn_decode(const FfnArgs& a, cudaStream_t st);  // fp32 SIMT (any x dtype)
// Streaming tensor-core kernels (bf16 x); stream_supported() says whether the shape fits
cudaError_t launch_ffn_stream(const FfnArgs& a, const StreamAux& x, int sm_count, cudaStream_t st);
bool stream_supported(const FfnArgs& a);
// One persistent kernel for T <= 8 (bf16 x) on n_ctas SMs (at most the SM count);
// persist_supported() says whether the shape fits (its shared-memory copy of the activations
// included). pdl: launched as a programmatic dependent of the kernel the caller enqueued just
// before it (else a cooperative launch).
cudaError_t launch_ffn_persist(const FfnArgs& a, const PersistAux& x, int n_ctas, cudaStream_t st, bool pdl);
bool persist_supported(const FfnArgs& a, int sm_count);
// Tensor-core grouped GEMM for many tokens per expert (bf16 x); prefill_supported() says whether
// the shape fits (d a multiple of 256, f of 128).
cudaError_t launch_ffn_prefill(const FfnArgs& a, const PrefillAux& x, int sm_count, cudaStream_t st);
bool prefill_supported(const FfnArgs& a);
int device_sm_count();
// The limit, in nanoseconds, that the next expert-FFN launches give their bounded waits.
uint64_t wait_limit_ns();
cudaError_t launch_combine(const moe_shape& s, const void* y, int ydt, const int32_t* inv_pos,
                           const float* topk_w, const void* residual, void* out, int odt, cudaStream_t st,
                           bool pdl);
cudaError_t launch_rms_norm(const moe_shape& s, const void* x, int xdt, void* out, int odt, float eps,
                            cudaStream_t st, bool pdl = false);

}  // namespace moe
