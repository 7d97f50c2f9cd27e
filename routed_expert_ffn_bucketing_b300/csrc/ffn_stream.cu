// Expert FFN for few tokens per expert with bf16 activations: int8 weights streamed from HBM
// straight into registers, dot products on the tensor cores.
//
// Decode reads each selected expert's int8 rows once ("Strata 工作原理图解GPU内存SSD三级存储如何让
// 125B模型塞进消费级显卡", section "推测解码": one token plus up to three drafts per step, so T = 4),
// so its time is that of streaming those bytes from HBM. Three kernels:
//   prepare: activations to f16 (rescaled per token by a power of two) with their per-block
//            sums, the work-item table (each selected expert's record found through the slot
//            table), the token of every output row, cleared max |h| per row and counters;
//   gate/up: a task is (item, 8 rows of f): M rows 0..7 of the MMA are 8 rows of the gate
//            matrix and M rows 8..15 the same rows of the up matrix, so each lane holds g and
//            u of the same (row, token) and applies h = silu(g) * u in registers; h goes to
//            an fp32 buffer. The last task of an item to finish turns the item's h rows into
//            f16 (rescaled per row by a power of two from max |h|) with their per-block sums;
//   down:    a task is (item, 16 rows of d).
// A warp computes a whole task over all of K. Its lanes load the MMA fragments of the codes
// directly from global memory (8 bytes of one row per lane and block; in the paired code layout
// the loads of the two blocks of a pair together read each row's 64 bytes whole), eight blocks
// ahead of their use, so each SM keeps ~64 KB of loads in flight. This path serves T up to 16
// (two passes over a task for 8 < T <= 16) and shapes the persistent kernel cannot stage.
// Where they fit (decode sizes), each CTA first copies the activations the kernel reads (f16
// rows and their block sums) into shared memory, so the per-block activation fragment of the
// MMA is a shared-memory load instead of a cache access on the critical path. That copy ends
// in the kernels' only barrier; they have no wait.
//
// Conversion. One lop3 turns two int8 codes (bytes 0 and 2 of a word, or 1 and 3 after a
// shift) into the f16 pair 1152 + q, exactly (0x64 in the high byte, q + 128 in the low byte).
// The MMA's accumulator input is set to -1152 * (sum of the block's activations), so the MMA
// returns sum_k q_k x_k: every product (1152 + q) * x is exact in fp32 and the offset cancels
// to within ~1e-6 of the result. The pairs hold elements (0, 2) and (1, 3) of each group of
// four, so activations are stored in the same order (x0 x2 x1 x3 x4 x6 x5 x7 per group of 8).
// Each MMA stays inside one 32-element block; the block's fp16 scale multiplies its result.
// Activations are exact f16 copies after a per-token power-of-two rescale that puts max |x|
// in [2^14, 2^15) (bf16 has 8 significant bits); h is rounded once to f16 (11 bits) after its
// row's rescale. The row max is an atomic max of non-negative floats (order-free) and every
// sum has a fixed order: results are deterministic.
//
// Lane (g, c) = (lane / 4, lane % 4) of an m16n8k16 MMA holds M rows g and g + 8 and token
// columns 2c, 2c + 1 of the result; in MMA half hf (0, 1) of a block its k slots {2c, 2c+1,
// 2c+8, 2c+9} hold elements c*8 + hf*4 + {0, 2, 1, 3}, and the activation fragment of token g
// uses the same order, so the k permutation cancels in the sum.
#include "decode_mma.cuh"

namespace moe {

constexpr int kPassTok = 8;          // tokens per pass over a task (the 8 columns of an MMA)
// ------------------------------------------------------------------ prepare --------------

// CTA t: x16[t] = f16(x[t] * 2^-e_t) (permuted), xunscale[t] = 2^e_t, cx[t][b] the MMA input of
// block b. All CTAs: hmax[r] = 0 and row_tok[r] (token of output row r) for every row. CTA 0:
// the work-item table and its counters.
__global__ void __launch_bounds__(256) ffn_prepare_kernel(FfnArgs A, StreamAux X) {
  __shared__ float wmax[8];
  const int t = blockIdx.x;
  const int rows = A.P + A.T * A.n_shared;
  for (int r = t * blockDim.x + threadIdx.x; r < rows; r += gridDim.x * blockDim.x) {
    X.hmax[r] = 0u;
    X.row_tok[r] = r < A.P ? A.sorted_pair[r] / A.k : (r - A.P) % A.T;
  }
  if (t == 0) {
    const int n = n_items(A);
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      FfnItem it;
      ItemRec rec{};
      if (resolve_item(i, A, &it)) {
        rec.rec = it.rec;
        rec.row0 = it.row0;
        rec.ntok = it.ntok;
        rec.slot = it.slot;
        rec.shared = it.routed ? 0 : 1;
      }
      X.items[i] = rec;
      X.item_cnt[i] = 0;
    }
    if (threadIdx.x < 2) X.sched[threadIdx.x] = 0;
  }
  if (A.T <= kPassTok)  // stream-K cut-task counters of both kernels
    for (int i = t * blockDim.x + threadIdx.x; i < 2 * X.cnt_stride; i += gridDim.x * blockDim.x) X.task_cnt[i] = 0;
  const int d = A.d, nb = d / kQBlock;
  float m = 0.0f;
  for (int i = threadIdx.x; i < d; i += blockDim.x) m = fmaxf(m, fabsf(load_act(A.x, A.xdt, (size_t)t * d + i)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
  __syncthreads();
  m = 0.0f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) m = fmaxf(m, wmax[w]);
  const int e = f16_exp_for(m);
  const float down = pow2f(-e);
  if (threadIdx.x == 0) X.xunscale[t] = pow2f(e);
  for (int b = threadIdx.x; b < nb; b += blockDim.x) {
    float v[kQBlock];
#pragma unroll
    for (int i = 0; i < kQBlock; ++i) v[i] = load_act(A.x, A.xdt, (size_t)t * d + b * kQBlock + i) * down;
    X.cx[(size_t)t * nb + b] = store_block_f16(X.x16 + (size_t)t * d + b * kQBlock, v);
  }
}

// ------------------------------------------------------------------ streaming kernels ----

enum { kGateUp = 0, kDown = 1 };

constexpr int kWarps = 16;                // warps per CTA
constexpr int kThreads = 32 * kWarps;
constexpr int kDepth = 8;                 // weight blocks in flight per warp (kDepth x 512 bytes)

// Next task of this warp from the kernel's task counter (one atomic per task, lane 0).
__device__ __forceinline__ int grab_task(int* counter, int lane) {
  int t = 0;
  if (lane == 0) t = atomicAdd(counter, 1);
  return __shfl_sync(0xFFFFFFFFu, t, 0);
}

// Byte offset, from a lane's chunk (c * 16) of a code row, of that lane's 8 codes of block b:
// blocks come in pairs of 64 bytes, the second block's 8 codes right after the first's
// (K is a multiple of 128 on this path, so every block has a partner).
__device__ __forceinline__ int block_off(int b) { return (b >> 1) * 64 + (b & 1) * 8; }

// An activation-side vector: from shared memory when staged (S), else a read-only global load.
template <bool S, typename V>
__device__ __forceinline__ V ld_act(const V* p) {
  if (S) return *p;
  return __ldg(p);
}

// D f16 scales (D = 4 or 8) of one row, loaded with one vector load.
template <int D>
struct ScaleVec {
  uint32_t w[D / 2];
  __device__ __forceinline__ void load(const __half* p) {
    if (D == 8) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
      w[0] = v.x; w[1 % (D / 2)] = v.y; w[2 % (D / 2)] = v.z; w[3 % (D / 2)] = v.w;
    } else {
      const uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
      w[0] = v.x; w[1 % (D / 2)] = v.y;
    }
  }
  __device__ __forceinline__ float at(int j) const {
    const uint32_t v = w[j >> 1];
    return __half2float(__ushort_as_half((unsigned short)((j & 1) ? (v >> 16) : (v & 0xFFFFu))));
  }
};

// One warp computes the dot products of 16 M rows (lo: rows g, hi: rows g + 8 of the MMA) of
// one expert with up to 8 token columns, over blocks [b_lo, b_hi) of K (both multiples of D).
// wlo / whi point at byte c*8 of the rows' codes, slo / shi at their f16 scale rows, xrow at the
// lane's activation row (byte c*8 of it, permuted f16), cs0 / cs1 at the accumulator-input rows
// of columns 2c, 2c+1. Weights are loaded D blocks ahead of their use; scales and accumulator
// inputs are loaded with vector loads.
template <int D, bool S>
__device__ __forceinline__ void rows_dot(const uint8_t* wlo, const uint8_t* whi, const __half* slo,
                                         const __half* shi, const __half* xrow, bool has, const float* cs0,
                                         const float* cs1, int b_lo, int b_hi, float (&acc)[4]) {
  uint2 ql[D], qh[D];
#pragma unroll
  for (int j = 0; j < D; ++j) {
    ql[j] = ld_codes(wlo + block_off(b_lo + j));
    qh[j] = ld_codes(whi + block_off(b_lo + j));
  }
  for (int b0 = b_lo; b0 < b_hi; b0 += D) {
    ScaleVec<D> sl, sh;
    sl.load(slo + b0);
    sh.load(shi + b0);
    float4 c0, c1;  // accumulator inputs of blocks (j & ~3) .. + 3
#pragma unroll
    for (int j = 0; j < D; ++j) {
      const int b = b0 + j;
      if ((j & 3) == 0) {
        c0 = ld_act<S>(reinterpret_cast<const float4*>(cs0 + b));
        c1 = ld_act<S>(reinterpret_cast<const float4*>(cs1 + b));
      }
      const uint4 xv = has ? ld_act<S>(reinterpret_cast<const uint4*>(xrow + b * kQBlock)) : make_uint4(0, 0, 0, 0);
      const int jj = j & 3;
      const float ca = jj == 0 ? c0.x : jj == 1 ? c0.y : jj == 2 ? c0.z : c0.w;
      const float cb = jj == 0 ? c1.x : jj == 1 ? c1.y : jj == 2 ? c1.z : c1.w;
      float dd[4];
      block_mma(dd, ql[j], qh[j], xv, ca, cb);
      if (b + D < b_hi) {
        ql[j] = ld_codes(wlo + block_off(b + D));
        qh[j] = ld_codes(whi + block_off(b + D));
      }
      const float s_lo = sl.at(j), s_hi = sh.at(j);
      acc[0] = fmaf(s_lo, dd[0], acc[0]);
      acc[1] = fmaf(s_lo, dd[1], acc[1]);
      acc[2] = fmaf(s_hi, dd[2], acc[2]);
      acc[3] = fmaf(s_hi, dd[3], acc[3]);
    }
  }
}

// Where a task's operands are, for one pass of up to 8 tokens starting at token `base`.
struct TaskOps {
  ItemRec it;
  int item, row_lo, row_hi, base, ng;
  const uint8_t *wlo, *whi;
  const __half *slo, *shi, *xrow;
  const float *cs0, *cs1;
  bool has;
};

template <int KIND>
__device__ __forceinline__ bool task_rows(const FfnArgs& A, const StreamAux& X, int t, int tpi, int nb, int g,
                                          int c, TaskOps* o) {
  const int item = t / tpi, mt = t % tpi;
  o->it = X.items[item];
  o->item = item;
  if (o->it.rec == nullptr || o->it.ntok <= 0) return false;
  const uint8_t* rec = o->it.rec;
  const int d = A.d, f = A.f;
  if (KIND == kGateUp) {
    o->row_lo = o->row_hi = mt * 8 + g;  // gate row and up row of the same f index
    o->wlo = rec + A.o_gate_q + (size_t)o->row_lo * d + c * 16;
    o->whi = rec + A.o_up_q + (size_t)o->row_hi * d + c * 16;
    o->slo = reinterpret_cast<const __half*>(rec + A.o_gate_s) + (size_t)o->row_lo * nb;
    o->shi = reinterpret_cast<const __half*>(rec + A.o_up_s) + (size_t)o->row_hi * nb;
  } else {
    o->row_lo = mt * 16 + g;
    o->row_hi = o->row_lo + 8;
    o->wlo = rec + A.o_down_q + (size_t)o->row_lo * f + c * 16;
    o->whi = rec + A.o_down_q + (size_t)o->row_hi * f + c * 16;
    o->slo = reinterpret_cast<const __half*>(rec + A.o_down_s) + (size_t)o->row_lo * nb;
    o->shi = reinterpret_cast<const __half*>(rec + A.o_down_s) + (size_t)o->row_hi * nb;
  }
  return true;
}

// B operand (activation row of token column g) and C operand rows (columns 2c and 2c + 1) of
// the pass starting at token `base`. xb / cb: the activation rows and their block sums (x16 and
// cx for gate/up, h16 and ch for down), in global or shared memory.
template <int KIND>
__device__ __forceinline__ void task_pass(const FfnArgs& A, const StreamAux& X, int base, int nb, int g, int c,
                                          TaskOps* o, const __half* xb, const float* cb) {
  const ItemRec& it = o->it;
  o->base = base;
  o->ng = min(kPassTok, it.ntok - base);
  o->has = g < o->ng;
  const int rg_ = it.row0 + base + (o->has ? g : 0);
  const int r0 = it.row0 + base + (2 * c < o->ng ? 2 * c : 0);
  const int r1 = it.row0 + base + (2 * c + 1 < o->ng ? 2 * c + 1 : 0);
  if (KIND == kGateUp) {
    o->xrow = xb + (size_t)X.row_tok[rg_] * A.d + c * 8;
    o->cs0 = cb + (size_t)X.row_tok[r0] * nb;
    o->cs1 = cb + (size_t)X.row_tok[r1] * nb;
  } else {
    o->xrow = xb + (size_t)rg_ * A.f + c * 8;
    o->cs0 = cb + (size_t)r0 * nb;
    o->cs1 = cb + (size_t)r1 * nb;
  }
}

// Epilogue of one pass: lane (g, c) holds rows row_lo (q = 0, 1) / row_hi (q = 2, 3) for tokens
// 2c, 2c + 1 of the pass.
template <int KIND>
__device__ __forceinline__ void task_epilogue(const FfnArgs& A, const StreamAux& X, const TaskOps& o, int g, int c,
                                              const float (&acc)[4]) {
  const ItemRec& it = o.it;
  const int ng = o.ng, base = o.base;
  if (KIND == kGateUp) {
    float m[2] = {0.f, 0.f};
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int tcol = 2 * c + q;
      if (tcol < ng) {
        const int r = it.row0 + base + tcol;
        const float xs = X.xunscale[X.row_tok[r]];
        const float hv = silu(acc[q] * xs) * (acc[2 + q] * xs);
        A.h[(size_t)r * A.f + o.row_lo] = hv;
        m[q] = fabsf(hv);
      }
    }
#pragma unroll
    for (int s = 4; s < 32; s <<= 1) {
      m[0] = fmaxf(m[0], __shfl_xor_sync(0xFFFFFFFFu, m[0], s));
      m[1] = fmaxf(m[1], __shfl_xor_sync(0xFFFFFFFFu, m[1], s));
    }
    if (g == 0) {
      const int r = it.row0 + base + 2 * c;
      if (2 * c < ng) atomicMax(X.hmax + r, __float_as_uint(m[0]));
      if (2 * c + 1 < ng) atomicMax(X.hmax + r + 1, __float_as_uint(m[1]));
    }
  } else {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int tcol = 2 * c + q;
      if (tcol < ng) {
        const int r = it.row0 + base + tcol;
        const float up = pow2f(X.hexp[r]);
        const float v_lo = acc[q] * up, v_hi = acc[2 + q] * up;
        const size_t off = (size_t)r * A.d;
        if (A.ydt == 1) {
          static_cast<float*>(A.y)[off + o.row_lo] = v_lo;
          static_cast<float*>(A.y)[off + o.row_hi] = v_hi;
        } else {
          static_cast<__nv_bfloat16*>(A.y)[off + o.row_lo] = __float2bfloat16_rn(v_lo);
          static_cast<__nv_bfloat16*>(A.y)[off + o.row_hi] = __float2bfloat16_rn(v_hi);
        }
      }
    }
  }
}

// After a gate/up task's epilogue: the last task of its item to finish turns the item's h rows
// into f16 for the down kernel. The warp fences its h and hmax writes before counting the task,
// so the counter reaches tpi only after all of the item's writes are visible.
__device__ __forceinline__ void gateup_task_done(const FfnArgs& A, const StreamAux& X, const TaskOps& o, int tpi,
                                                 int lane) {
  __threadfence();
  int last = 0;
  if (lane == 0) last = atomicAdd(X.item_cnt + o.item, 1) == tpi - 1;
  if (!__shfl_sync(0xFFFFFFFFu, last, 0)) return;
  __threadfence();
  const int f = A.f, nbf = f / kQBlock;
  const ItemRec& it = o.it;
  for (int i = lane; i < it.ntok * nbf; i += 32) {
    const int r = it.row0 + i / nbf, b = i % nbf;
    const int e = f16_exp_for(__uint_as_float(__ldcg(X.hmax + r)));
    const float down = pow2f(-e);
    float v[kQBlock];
    const float4* src = reinterpret_cast<const float4*>(A.h + (size_t)r * f + b * kQBlock);
#pragma unroll
    for (int q = 0; q < kQBlock / 4; ++q) {
      const float4 w4 = __ldcg(src + q);
      v[4 * q] = w4.x * down;
      v[4 * q + 1] = w4.y * down;
      v[4 * q + 2] = w4.z * down;
      v[4 * q + 3] = w4.w * down;
    }
    X.ch[(size_t)r * nbf + b] = store_block_f16(X.h16 + (size_t)r * f + b * kQBlock, v);
    if (b == 0) X.hexp[r] = e;
  }
}

// The streaming kernel. A task is (item, 16 M rows): for gate/up, 8 rows of f taken from both
// the gate and the up matrix (M rows 0..7 and 8..15); for down, 16 rows of d.
//
// When every item has at most 8 tokens (T <= 8: one pass per task), the work is split
// stream-K: the (task, group of D blocks) sequence is cut into one contiguous range per warp,
// equal to within one group, so all warps stream the same number of bytes. A task cut between
// two warps (never more: a range is at least one task long) is finished by the second of them
// to arrive: it adds the partial sums as part 0 + part 1 (a fixed order) and runs the epilogue.
// Otherwise warps take whole tasks, pass by pass, from an atomic counter.
template <int KIND, int D, bool S>
__global__ void __launch_bounds__(kThreads) ffn_stream_kernel(FfnArgs A, StreamAux X) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int K = KIND == kGateUp ? A.d : A.f;
  const int nb = K / kQBlock;
  const int tpi = KIND == kGateUp ? A.f / 8 : A.d / 16;  // tasks per item
  const int n_tasks = n_items(A) * tpi;
  // activation rows: the T tokens' x for gate/up, every output row's h for down
  const __half* xb = KIND == kGateUp ? X.x16 : X.h16;
  const float* cb = KIND == kGateUp ? X.cx : X.ch;
  if (S) {
    extern __shared__ __align__(16) uint8_t act_smem[];
    const int rows = KIND == kGateUp ? A.T : A.P + A.T * A.n_shared;
    __half* sx = reinterpret_cast<__half*>(act_smem);
    float* sc = reinterpret_cast<float*>(act_smem + (size_t)rows * K * sizeof(__half));
    const int nx = rows * K / 8, nc = rows * nb / 4;  // uint4 / float4 counts
    for (int i = threadIdx.x; i < nx; i += blockDim.x)
      reinterpret_cast<uint4*>(sx)[i] = __ldcg(reinterpret_cast<const uint4*>(xb) + i);
    for (int i = threadIdx.x; i < nc; i += blockDim.x)
      reinterpret_cast<float4*>(sc)[i] = __ldcg(reinterpret_cast<const float4*>(cb) + i);
    __syncthreads();
    xb = sx;
    cb = sc;
  }
  if (A.T <= kPassTok) {
    const int gpt = nb / D;  // groups of D blocks per task
    const long long total = (long long)n_tasks * gpt;
    const int nw = min(gridDim.x * kWarps, n_tasks);  // each range at least one task long
    const int wid = blockIdx.x * kWarps + warp;
    if (wid >= nw) return;
    float* part = X.part + (size_t)KIND * X.part_stride;
    int* cnt = X.task_cnt + (size_t)KIND * X.cnt_stride;
    const long long G1 = (long long)(wid + 1) * total / nw;
    for (long long G = (long long)wid * total / nw; G < G1;) {
      const int t = (int)(G / gpt), gs = (int)(G % gpt);
      const int ge = (int)min((long long)gpt, gs + (G1 - G));
      G += ge - gs;
      TaskOps o;
      if (!task_rows<KIND>(A, X, t, tpi, nb, g, c, &o)) continue;
      task_pass<KIND>(A, X, 0, nb, g, c, &o, xb, cb);
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      rows_dot<D, S>(o.wlo, o.whi, o.slo, o.shi, o.xrow, o.has, o.cs0, o.cs1, gs * D, ge * D, acc);
      if (gs != 0 || ge != gpt) {
        // a cut task: publish this part, and the second part to arrive finishes the task
        const int my = gs == 0 ? 0 : 1;
        float4* slot = reinterpret_cast<float4*>(part + ((size_t)t * 2 + my) * 128);
        slot[lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        __threadfence();
        int second = 0;
        if (lane == 0) second = atomicAdd(cnt + t, 1) == 1;
        if (!__shfl_sync(0xFFFFFFFFu, second, 0)) continue;
        __threadfence();
        const float4 p0 = __ldcg(reinterpret_cast<const float4*>(part + (size_t)t * 2 * 128) + lane);
        const float4 p1 = __ldcg(reinterpret_cast<const float4*>(part + ((size_t)t * 2 + 1) * 128) + lane);
        acc[0] = p0.x + p1.x;
        acc[1] = p0.y + p1.y;
        acc[2] = p0.z + p1.z;
        acc[3] = p0.w + p1.w;
      }
      task_epilogue<KIND>(A, X, o, g, c, acc);
      if (KIND == kGateUp) gateup_task_done(A, X, o, tpi, lane);
    }
    return;
  }
  int* counter = X.sched + KIND;
  for (int t = grab_task(counter, lane); t < n_tasks; t = grab_task(counter, lane)) {
    TaskOps o;
    if (!task_rows<KIND>(A, X, t, tpi, nb, g, c, &o)) continue;
    for (int base = 0; base < o.it.ntok; base += kPassTok) {
      task_pass<KIND>(A, X, base, nb, g, c, &o, xb, cb);
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      rows_dot<D, S>(o.wlo, o.whi, o.slo, o.shi, o.xrow, o.has, o.cs0, o.cs1, 0, nb, acc);
      task_epilogue<KIND>(A, X, o, g, c, acc);
    }
    if (KIND == kGateUp) gateup_task_done(A, X, o, tpi, lane);
  }
}

bool stream_supported(const FfnArgs& a) { return a.d % 128 == 0 && a.f % 128 == 0; }

constexpr size_t kStageMax = 160 * 1024;  // largest activation copy kept in shared memory

template <int KIND, int D>
static cudaError_t launch_stream_d(const FfnArgs& a, const StreamAux& x, int grid, size_t smem, cudaStream_t st) {
  if (smem <= kStageMax) {
    const cudaError_t e = ensure_dynamic_smem((const void*)ffn_stream_kernel<KIND, D, true>, smem);
    if (e != cudaSuccess) return e;
    ffn_stream_kernel<KIND, D, true><<<grid, kThreads, smem, st>>>(a, x);
  } else {
    ffn_stream_kernel<KIND, D, false><<<grid, kThreads, 0, st>>>(a, x);
  }
  return cudaGetLastError();
}

template <int KIND>
static cudaError_t launch_stream(const FfnArgs& a, const StreamAux& x, int grid, int K, size_t smem,
                                 cudaStream_t st) {
  return (K / kQBlock) % 8 == 0 ? launch_stream_d<KIND, 8>(a, x, grid, smem, st)
                                : launch_stream_d<KIND, 4>(a, x, grid, smem, st);
}

cudaError_t launch_ffn_stream(const FfnArgs& a, const StreamAux& x, int sm_count, cudaStream_t st) {
  const int items_max = (a.P < a.E ? a.P : a.E) + a.n_shared;
  if (items_max == 0) return cudaSuccess;
  ffn_prepare_kernel<<<a.T, 256, 0, st>>>(a, x);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int gu_tasks = items_max * (a.f / 8), dn_tasks = items_max * (a.d / 16);
  auto grid = [&](int tasks) {
    const int warps = tasks < sm_count * kWarps ? tasks : sm_count * kWarps;
    return (warps + kWarps - 1) / kWarps;
  };
  // D = 8 blocks in flight where the block count allows it (K a multiple of 256), else 4;
  // activations staged in shared memory where they fit
  const size_t rows = (size_t)a.P + (size_t)a.T * a.n_shared;
  const size_t sm_gu = (size_t)a.T * a.d * sizeof(__half) + (size_t)a.T * (a.d / kQBlock) * sizeof(float);
  const size_t sm_dn = rows * a.f * sizeof(__half) + rows * (a.f / kQBlock) * sizeof(float);
  if ((e = launch_stream<kGateUp>(a, x, grid(gu_tasks), a.d, sm_gu, st)) != cudaSuccess) return e;
  return launch_stream<kDown>(a, x, grid(dn_tasks), a.f, sm_dn, st);
}

}  // namespace moe
