// Router logits and top-k gate of the MoE layer.
//
// The router picks the top-K experts of each token; the other experts take no part
// ("单张RTX 5090跑125B大模型：Strata实测Qwen3.8 Flash Next", section "MoE专家按需调度"). It is
// resident in VRAM ("Strata 工作原理图解GPU内存SSD三级存储如何让125B模型塞进消费级显卡", section
// "三级存储分工"). Logits are fp32 with a fixed summation order, so results are deterministic.
//
//  * T <= 16 (decode, spec-verify): the router is a GEMV that streams w_router [d][E] once.
//    The d rows are split into chunks of 128 so that the whole matrix is in flight at
//    once (one CTA per 128 rows x 128 experts). Each chunk writes a partial sum; the top-k
//    kernel (one CTA per token) copies the token's partial sums to shared memory at once and
//    adds them in a fixed order.
//  * T > 16 (prefill): a tiled fp32 GEMM, 128 x 128 outputs per CTA. Each output sums its
//    32-long k-blocks separately before adding them up, which keeps the fp32 error of a
//    2048-long dot product near that of a tree sum.
//  * top-k: one warp per token selects. Each lane holds E/32 logits as order-preserving
//    integer keys, and k rounds of warp max (redux.sync) pick the experts. A tie goes to the
//    lowest index.
#include <cooperative_groups.h>

#include "bucket.cuh"
#include "sm100_ptx.cuh"

namespace moe {

namespace cg = cooperative_groups;

// ------------------------------------------------------------------ top-k helpers ---------

// Order-preserving key of an fp32 logit: larger float, larger key. -0.0 maps like +0.0 and
// NaN maps to 0, below every number (-inf has key 0x007FFFFF).
__device__ __forceinline__ uint32_t logit_key(float v, bool* nan) {
  uint32_t u = __float_as_uint(v);
  if (u == 0x80000000u) u = 0u;
  if (v != v) {
    *nan = true;
    return 0u;
  }
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_logit(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key ^ 0x80000000u) : ~key);
}

// Descending bitonic sort of N (a power of two) values held in registers.
template <int N>
__device__ __forceinline__ void sort_desc_regs(uint64_t (&v)[N]) {
#pragma unroll
  for (int size = 2; size <= N; size <<= 1)
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1)
#pragma unroll
      for (int i = 0; i < N; ++i) {
        const int j = i ^ stride;
        if (j > i) {
          const bool desc = (i & size) == 0;  // direction of this pair in the bitonic merge
          const uint64_t a = v[i], b = v[j];
          const bool swap = desc ? (a < b) : (a > b);
          v[i] = swap ? b : a;
          v[j] = swap ? a : b;
        }
      }
}

// Writes token t's selection, lane j holding its j-th expert and key (j < k), with the
// renormalised gate weights: exp(l_j - l_0) over their sum (a fixed butterfly order).
__device__ __forceinline__ void topk_write(int my_e, uint32_t my_key, int k, int t, int32_t* idx, float* wts,
                                           int* idx_smem) {
  const int lane = threadIdx.x & 31;
  const float val = key_logit(my_key);
  const float m = __shfl_sync(0xFFFFFFFFu, val, 0);
  const float ex = lane < k ? expf(val - m) : 0.0f;
  float sum = ex;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
  if (lane < k) {
    idx[(size_t)t * k + lane] = my_e;
    wts[(size_t)t * k + lane] = ex / sum;
    if (idx_smem) idx_smem[t * k + lane] = my_e;
  }
}

// Selection of the k largest keys among the E logits held as PER keys per lane (logit e in
// lane e % 32, slot e / 32), then the renormalised gate weights; one warp, one token. Each
// candidate is the 64-bit value (key, ~e): a larger value is a larger logit, or an equal one
// with a lower expert index. Each lane sorts its candidates once; a round then takes the
// largest head over the lanes (two warp max reductions, on the key and then on ~e among the
// lanes holding that key) and the winning lane pops its head. Experts >= E are 0 and never win
// while a real candidate (NaN included, key 0 but ~e > 0) is left.
template <int PER>
__device__ __forceinline__ void select_topk_warp(uint32_t (&key)[PER], int E, int k, int t, int32_t* idx,
                                                 float* wts, int* idx_smem = nullptr) {
  const int lane = threadIdx.x & 31;
  uint64_t v[PER];
#pragma unroll
  for (int p = 0; p < PER; ++p) {
    const int e = lane + 32 * p;
    v[p] = e < E ? ((uint64_t)key[p] << 32) | (uint64_t)(~(uint32_t)e) : 0ull;
  }
  sort_desc_regs<PER>(v);
  int my_e = 0;
  uint32_t my_key = 0u;
  for (int j = 0; j < k; ++j) {
    const uint32_t hk = (uint32_t)(v[0] >> 32);
    const uint32_t mk = __reduce_max_sync(0xFFFFFFFFu, hk);
    const uint32_t lo = hk == mk ? (uint32_t)v[0] : 0u;
    const uint32_t ml = __reduce_max_sync(0xFFFFFFFFu, lo);
    if (hk == mk && (uint32_t)v[0] == ml) {  // the unique winner pops its head
#pragma unroll
      for (int p = 0; p + 1 < PER; ++p) v[p] = v[p + 1];
      v[PER - 1] = 0ull;
    }
    if (lane == j) {
      my_e = (int)(~ml);
      my_key = mk;
    }
  }
  topk_write(my_e, my_key, k, t, idx, wts, idx_smem);
}

// The same selection by every warp of a block at once, for one token whose logits are in
// shared memory (lg[0, E), E <= 32 * warps, k <= 32): warp w takes the k largest of experts
// 32w..32w+31 in k rounds of two warp max reductions (one candidate per lane) and lists them
// best first in cand[w * k ..]; then warp 0 merges the lists, lane l following list l, each
// round popping the largest head. Every round of both levels takes the largest remaining
// (key, ~e), so the experts come out in the order select_topk_warp gives, and topk_write
// makes the weights: the outputs are identical. Returns with warp 0 done (no block barrier
// after the write).
__device__ __forceinline__ void select_topk_block(const float* lg, int E, int k, int t, int32_t* idx, float* wts,
                                                  int* idx_smem, uint64_t* cand, bool* nan) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nw = (E + 31) / 32;
  if (warp < nw) {
    const int e = warp * 32 + lane;
    uint64_t v = e < E ? ((uint64_t)logit_key(lg[e], nan) << 32) | (uint64_t)(~(uint32_t)e) : 0ull;
    for (int j = 0; j < k; ++j) {
      const uint32_t hk = (uint32_t)(v >> 32);
      const uint32_t mk = __reduce_max_sync(0xFFFFFFFFu, hk);
      const uint32_t lo = hk == mk ? (uint32_t)v : 0u;
      const uint32_t ml = __reduce_max_sync(0xFFFFFFFFu, lo);
      if (hk == mk && (uint32_t)v == ml) v = 0ull;  // the unique winner leaves
      if (lane == 0) cand[warp * k + j] = ((uint64_t)mk << 32) | ml;
    }
  }
  __syncthreads();
  if (warp != 0) return;
  int ptr = 0;
  uint64_t head = lane < nw ? cand[lane * k] : 0ull;
  int my_e = 0;
  uint32_t my_key = 0u;
  for (int j = 0; j < k; ++j) {
    const uint32_t hk = (uint32_t)(head >> 32);
    const uint32_t mk = __reduce_max_sync(0xFFFFFFFFu, hk);
    const uint32_t lo = hk == mk ? (uint32_t)head : 0u;
    const uint32_t ml = __reduce_max_sync(0xFFFFFFFFu, lo);
    if (hk == mk && (uint32_t)head == ml) {  // the winning list moves to its next candidate
      ++ptr;
      head = ptr < k ? cand[lane * k + ptr] : 0ull;
    }
    if (lane == j) {
      my_e = (int)(~ml);
      my_key = mk;
    }
  }
  topk_write(my_e, my_key, k, t, idx, wts, idx_smem);
}

// ------------------------------------------------------------------ split-d GEMV ----------


// Adds the S split partial sums held at slab[sp * stride] in four interleaved chains, then the
// chains (a fixed order).
__device__ __forceinline__ float sum_splits(const float* slab, int S, int stride) {
  float c0 = 0.f, c1 = 0.f, c2 = 0.f, c3 = 0.f;
  int sp = 0;
  for (; sp + 4 <= S; sp += 4) {
    c0 += slab[(sp + 0) * stride];
    c1 += slab[(sp + 1) * stride];
    c2 += slab[(sp + 2) * stride];
    c3 += slab[(sp + 3) * stride];
  }
  for (; sp < S; ++sp) c0 += slab[sp * stride];
  return (c0 + c1) + (c2 + c3);
}

__device__ __forceinline__ void cp_async_f4(float* dst, const float* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_f1(float* dst, const float* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
               : "memory");
}

template <int TT, int VEC>
__global__ void __launch_bounds__(256) router_gemv_kernel(const void* __restrict__ x, int xdt,
                                                          const float* __restrict__ w,
                                                          float* __restrict__ partial, int T, int d,
                                                          int E, int* status, int clear_status, uint4* zero,
                                                          int zero_n16) {
  constexpr int R = kRouteRowsPerSplit;  // rows of d per CTA
  pdl_trigger();  // the top-k kernel may launch now; it waits for this grid before reading
  // launched as a programmatic dependent (a stack's RMS norm before it), this grid may start
  // early: it waits for that kernel, and with it for every earlier kernel of the stream, before
  // it reads x or clears anything (at once when launched normally)
  pdl_wait();
  // ordered after every earlier kernel of the stream: clear the layer's status word (unless a
  // stack keeps it across layers) and the expert FFN's counters here, so no memset precedes the pass
  {
    const int cta = blockIdx.y * gridDim.x + blockIdx.x, n_cta = gridDim.x * gridDim.y;
    if (clear_status && cta == 0 && threadIdx.x == 0) *status = 0;
    for (int i = cta * blockDim.x + threadIdx.x; i < zero_n16; i += n_cta * blockDim.x) zero[i] = make_uint4(0, 0, 0, 0);
  }
  constexpr int COLS = 32 * VEC;         // experts per CTA
  extern __shared__ float sm[];
  float* xs = sm;            // [TT][R]
  float* red = sm + TT * R;  // [8][TT][COLS]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i0 = blockIdx.y * R;
  const int rows = min(R, d - i0);
  for (int j = threadIdx.x; j < TT * R; j += blockDim.x) {
    const int t = j / R, i = j % R;
    xs[j] = (t < T && i < rows) ? load_act(x, xdt, (size_t)t * d + i0 + i) : 0.0f;
  }
  __syncthreads();

  const int c0 = blockIdx.x * COLS + lane * VEC;
  float acc[TT][VEC];
#pragma unroll
  for (int t = 0; t < TT; ++t)
#pragma unroll
    for (int v = 0; v < VEC; ++v) acc[t][v] = 0.0f;

  float wv[R / 8][VEC];
#pragma unroll
  for (int rr = 0; rr < R / 8; ++rr) {  // all loads first: R/8 independent rows in flight
    const int i = warp + rr * 8;
    const float* row = w + (size_t)(i0 + i) * E;
    if constexpr (VEC == 4) {
      if (i < rows && c0 + 3 < E) {
        const float4 v4 = __ldg(reinterpret_cast<const float4*>(row + c0));
        wv[rr][0] = v4.x; wv[rr][1] = v4.y; wv[rr][2] = v4.z; wv[rr][3] = v4.w;
        continue;
      }
    }
#pragma unroll
    for (int v = 0; v < VEC; ++v) wv[rr][v] = (i < rows && c0 + v < E) ? __ldg(row + c0 + v) : 0.0f;
  }
#pragma unroll
  for (int rr = 0; rr < R / 8; ++rr) {
    const int i = warp + rr * 8;
#pragma unroll
    for (int t = 0; t < TT; ++t) {
      const float xv = xs[t * R + i];
#pragma unroll
      for (int v = 0; v < VEC; ++v) acc[t][v] = fmaf(xv, wv[rr][v], acc[t][v]);
    }
  }
#pragma unroll
  for (int t = 0; t < TT; ++t)
#pragma unroll
    for (int v = 0; v < VEC; ++v) red[(warp * TT + t) * COLS + lane * VEC + v] = acc[t][v];
  __syncthreads();
  for (int j = threadIdx.x; j < TT * COLS; j += blockDim.x) {
    const int t = j / COLS, c = j % COLS;
    float s = 0.0f;
#pragma unroll
    for (int w8 = 0; w8 < 8; ++w8) s += red[(w8 * TT + t) * COLS + c];
    const int e = blockIdx.x * COLS + c;
    if (t < T && e < E) partial[((size_t)blockIdx.y * T + t) * E + e] = s;
  }

}

template <int TT, int VEC>
static cudaError_t gemv_launch(const moe_shape& s, const void* x, int xdt, const float* w, float* partial,
                               int* status, int clear, void* zero, size_t zero_bytes, cudaStream_t st, bool pdl) {
  constexpr int COLS = 32 * VEC;
  const size_t smem = sizeof(float) * (TT * kRouteRowsPerSplit + 8 * TT * COLS);
  auto kern = router_gemv_kernel<TT, VEC>;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  dim3 grid((s.E + COLS - 1) / COLS, route_splits(s.d));
  return launch_maybe_pdl(pdl, kern, grid, dim3(256), smem, st, x, xdt, w, partial, s.T, s.d, s.E, status, clear,
                          static_cast<uint4*>(zero), (int)(zero_bytes / 16));
}

template <int VEC>
static cudaError_t gemv_dispatch_t(const moe_shape& s, const void* x, int xdt, const float* w, float* p, int* status,
                                   int c, void* z, size_t zb, cudaStream_t st, bool pdl) {
  if (s.T <= 1) return gemv_launch<1, VEC>(s, x, xdt, w, p, status, c, z, zb, st, pdl);
  if (s.T <= 2) return gemv_launch<2, VEC>(s, x, xdt, w, p, status, c, z, zb, st, pdl);
  if (s.T <= 4) return gemv_launch<4, VEC>(s, x, xdt, w, p, status, c, z, zb, st, pdl);
  if (s.T <= 8) return gemv_launch<8, VEC>(s, x, xdt, w, p, status, c, z, zb, st, pdl);
  return gemv_launch<16, VEC>(s, x, xdt, w, p, status, c, z, zb, st, pdl);
}

cudaError_t launch_route_gemv(const moe_shape& s, const void* x, int xdt, const float* w, float* partial,
                              int* status, void* zero, size_t zero_bytes, cudaStream_t st, bool pdl,
                              bool clear_status) {
  const int c = clear_status ? 1 : 0;
  if (s.E % 4 == 0) return gemv_dispatch_t<4>(s, x, xdt, w, partial, status, c, zero, zero_bytes, st, pdl);
  return gemv_dispatch_t<1>(s, x, xdt, w, partial, status, c, zero, zero_bytes, st, pdl);
}

// ------------------------------------------------------------------ tiled GEMM -------------

// out[T][E] = x[T][d] . w[d][E]; CTA tile 128 x 128, k-tile 8, 256 threads with 8 x 8 outputs.
// Every 32 k the block sum is added to the running total (two-level accumulation).
__global__ void __launch_bounds__(256) router_gemm_kernel(const void* __restrict__ x, int xdt,
                                                          const float* __restrict__ w,
                                                          float* __restrict__ out, int T, int d, int E,
                                                          int* status, int clear_status) {
  // ordered after every earlier kernel of the stream, and before the top-k that flags NaNs
  if (clear_status && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *status = 0;
  __shared__ __align__(16) float As[2][8][128];  // [k][token]
  __shared__ __align__(16) float Bs[2][8][128];  // [k][expert]
  const int tid = threadIdx.x;
  const int m0 = blockIdx.y * 128, n0 = blockIdx.x * 128;
  const int ty = tid >> 4, tx = tid & 15;
  // global->shared mapping: A: token row tid/2, k 4*(tid%2)..+4; B: k row tid/32, experts 4*(tid%32)..+4
  const int a_row = tid >> 1, a_k = (tid & 1) * 4;
  const int b_k = tid >> 5, b_col = (tid & 31) * 4;

  float acc[8][8], blk[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = blk[i][j] = 0.0f;

  float ra[4], rb[4];
  auto load_tile = [&](int kt) {
    const int tok = m0 + a_row;
#pragma unroll
    for (int q = 0; q < 4; ++q)
      ra[q] = tok < T ? load_act(x, xdt, (size_t)tok * d + kt * 8 + a_k + q) : 0.0f;
    const int krow = kt * 8 + b_k;
    const float* wr = w + (size_t)krow * E + n0 + b_col;
    if (n0 + b_col + 3 < E && (E % 4) == 0) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(wr));
      rb[0] = v.x; rb[1] = v.y; rb[2] = v.z; rb[3] = v.w;
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q) rb[q] = (n0 + b_col + q < E) ? __ldg(wr + q) : 0.0f;
    }
  };
  auto store_tile = [&](int buf) {
#pragma unroll
    for (int q = 0; q < 4; ++q) As[buf][a_k + q][a_row] = ra[q];
    *reinterpret_cast<float4*>(&Bs[buf][b_k][b_col]) = make_float4(rb[0], rb[1], rb[2], rb[3]);
  };

  const int nk = d / 8;
  load_tile(0);
  store_tile(0);
  __syncthreads();
  for (int kt = 0; kt < nk; ++kt) {
    const int buf = kt & 1;
    if (kt + 1 < nk) load_tile(kt + 1);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      float a[8], b[8];
      const float4 a0 = *reinterpret_cast<const float4*>(&As[buf][kk][ty * 8]);
      const float4 a1 = *reinterpret_cast<const float4*>(&As[buf][kk][ty * 8 + 4]);
      const float4 b0 = *reinterpret_cast<const float4*>(&Bs[buf][kk][tx * 8]);
      const float4 b1 = *reinterpret_cast<const float4*>(&Bs[buf][kk][tx * 8 + 4]);
      a[0] = a0.x; a[1] = a0.y; a[2] = a0.z; a[3] = a0.w; a[4] = a1.x; a[5] = a1.y; a[6] = a1.z; a[7] = a1.w;
      b[0] = b0.x; b[1] = b0.y; b[2] = b0.z; b[3] = b0.w; b[4] = b1.x; b[5] = b1.y; b[6] = b1.z; b[7] = b1.w;
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) blk[i][j] = fmaf(a[i], b[j], blk[i][j]);
    }
    if ((kt & 3) == 3 || kt + 1 == nk) {  // close a 32-long k-block
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          acc[i][j] += blk[i][j];
          blk[i][j] = 0.0f;
        }
    }
    if (kt + 1 < nk) store_tile(buf ^ 1);
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int tok = m0 + ty * 8 + i;
    if (tok >= T) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = n0 + tx * 8 + j;
      if (e < E) out[(size_t)tok * E + e] = acc[i][j];
    }
  }
}

cudaError_t launch_route_gemm(const moe_shape& s, const void* x, int xdt, const float* w, float* logits,
                              int* status, cudaStream_t st, bool clear_status) {
  dim3 grid((s.E + 127) / 128, (s.T + 127) / 128);
  router_gemm_kernel<<<grid, 256, 0, st>>>(x, xdt, w, logits, s.T, s.d, s.E, status, clear_status ? 1 : 0);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ top-k ------------------

// Logits already summed (router GEMM): one warp per token.
template <int PER>
__global__ void __launch_bounds__(128) topk_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                   int32_t* __restrict__ idx, float* __restrict__ wts,
                                                   int* status) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 4 + (threadIdx.x >> 5);
  if (t >= T) return;
  uint32_t key[PER];
  bool nan = false;
#pragma unroll
  for (int p = 0; p < PER; ++p) {
    const int e = lane + 32 * p;
    key[p] = e < E ? logit_key(logits[(size_t)t * E + e], &nan) : 0u;
  }
  select_topk_warp<PER>(key, E, k, t, idx, wts);
  if (__any_sync(0xFFFFFFFFu, nan) && lane == 0) flag_status(status, MOE_DEV_NAN_LOGIT_BIT);
}

// Split-d partial sums (router GEMV): one CTA per token. The token's S x E partials are copied
// to shared memory with every copy in flight at once (cp.async), added in a fixed order (four
// interleaved chains over the splits, then the chains), and warp 0 selects.
template <int PER>
__global__ void __launch_bounds__(512) topk_split_kernel(const float* __restrict__ partial, int S, int T, int E,
                                                         int k, int32_t* __restrict__ idx, float* __restrict__ wts,
                                                         float* __restrict__ logits_out, int* status) {
  extern __shared__ float slab[];  // [S][E], then the logits [E]
  __shared__ int nan_any;
  const int t = blockIdx.x;
  float* lg = slab + (size_t)S * E;
  if (threadIdx.x == 0) nan_any = 0;
  pdl_trigger();
  pdl_wait();  // the router GEMV's partial sums
  if (E % 4 == 0) {
    for (int i = threadIdx.x; i < S * (E / 4); i += blockDim.x) {
      const int c4 = i % (E / 4), sp = i / (E / 4);
      cp_async_f4(slab + (size_t)sp * E + c4 * 4, partial + ((size_t)sp * T + t) * E + c4 * 4);
    }
  } else {
    for (int i = threadIdx.x; i < S * E; i += blockDim.x) {
      const int c = i % E, sp = i / E;
      cp_async_f1(slab + (size_t)sp * E + c, partial + ((size_t)sp * T + t) * E + c);
    }
  }
  asm volatile("cp.async.commit_group;\ncp.async.wait_all;" ::: "memory");
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const float v = sum_splits(slab + e, S, E);
    lg[e] = v;
    if (logits_out) logits_out[(size_t)t * E + e] = v;
    if (v != v) nan_any = 1;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    uint32_t key[PER];
    bool nan = false;
#pragma unroll
    for (int p = 0; p < PER; ++p) {
      const int e = lane + 32 * p;
      key[p] = e < E ? logit_key(lg[e], &nan) : 0u;
    }
    select_topk_warp<PER>(key, E, k, t, idx, wts);
    if (lane == 0 && nan_any) flag_status(status, MOE_DEV_NAN_LOGIT_BIT);
  }
}

// Decode routing tail as one cluster of T CTAs (T <= 8), CTA t for token t: bulk copies bring
// the token's S split partial sums of the router GEMV, they are added in the fixed order of
// topk_split_kernel, the block selects the token's top k (select_topk_block: every warp at
// once) and warp 0 writes the experts of its pairs into CTA 0's shared memory (distributed
// shared memory); after the cluster barrier CTA 0 buckets the T*k pairs with
// bucket_count_block. The outputs are those of topk_split_kernel followed by
// bucket_count_kernel, bit for bit, from one launch instead of two.
__global__ void __launch_bounds__(512) route_tail_kernel(const float* __restrict__ partial, int S, int T, int E,
                                                          int k, int32_t* __restrict__ idx, float* __restrict__ wts,
                                                          float* __restrict__ logits_out, int32_t* counts,
                                                          int32_t* offsets, int32_t* sorted_pair, int32_t* inv_pos,
                                                          int32_t* active, int* status) {
  extern __shared__ __align__(16) float tail_sm[];  // [S][E] this token's partial sums, then [E] logits
  __shared__ uint64_t bar;
  __shared__ int ex[256];
  __shared__ int cs[512];
  __shared__ int warp_sums[33];
  __shared__ uint64_t cand[512];
  __shared__ int nan_any;
  cg::cluster_group cluster = cg::this_cluster();
  const int tid = threadIdx.x, t = blockIdx.x;
  float* lg = tail_sm + (size_t)S * E;
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    nan_any = 0;
  }
  __syncthreads();
  pdl_wait();  // the router GEMV's partial sums
  // The expert FFN may launch now and stage its activations meanwhile. It reads them before its
  // own wait, so it may start only once every kernel before this one has completed: after this
  // wait, not before it (the router GEMV has completed, and it completed only after its own wait
  // for the kernel before it, e.g. the RMS norm that wrote those activations).
  pdl_trigger();
  if (tid == 0) {
    mbar_arrive_expect_tx(&bar, (uint32_t)(S * E * 4));
    for (int sp = 0; sp < S; ++sp)
      bulk_g2s(tail_sm + (size_t)sp * E, partial + ((size_t)sp * T + t) * E, (uint32_t)(E * 4), &bar);
  }
  // a copy that never lands cannot be waited out; it is flagged and the tail goes on (its
  // outputs are then not to be trusted, as MOE_DEV_TIMEOUT says)
  if (!mbar_wait(&bar, 0) && tid == 0) flag_status(status, MOE_DEV_TIMEOUT_BIT);
  for (int e = tid; e < E; e += blockDim.x) {
    const float v = sum_splits(tail_sm + e, S, E);
    lg[e] = v;
    if (logits_out) logits_out[(size_t)t * E + e] = v;
    if (v != v) nan_any = 1;
  }
  __syncthreads();
  {
    bool nan = false;
    select_topk_block(lg, E, k, t, idx, wts, cluster.map_shared_rank(ex, 0), cand, &nan);
  }
  if (tid == 0 && nan_any) flag_status(status, MOE_DEV_NAN_LOGIT_BIT);
  cluster.sync();  // every token's experts are in CTA 0's ex[]
  if (cluster.block_rank() == 0)
    bucket_count_block(ex, T * k, E, cs, warp_sums, counts, offsets, sorted_pair, inv_pos, active);
}

#define MOE_TOPK_DISPATCH(LAUNCH)    \
  do {                               \
    const int per = (s.E + 31) / 32; \
    if (per <= 1) LAUNCH(1);         \
    else if (per <= 2) LAUNCH(2);    \
    else if (per <= 4) LAUNCH(4);    \
    else if (per <= 8) LAUNCH(8);    \
    else if (per <= 16) LAUNCH(16);  \
    else LAUNCH(32);                 \
  } while (0)

cudaError_t launch_topk(const moe_shape& s, const float* logits, int32_t* idx, float* wts, int* status,
                        cudaStream_t st) {
  const dim3 grid((s.T + 3) / 4);
#define L_ONE(P) topk_kernel<P><<<grid, 128, 0, st>>>(logits, s.T, s.E, s.k, idx, wts, status)
  MOE_TOPK_DISPATCH(L_ONE);
#undef L_ONE
  return cudaGetLastError();
}

cudaError_t launch_topk_split(const moe_shape& s, const float* partial, int splits, int32_t* idx, float* wts,
                              float* logits_out, int* status, cudaStream_t st) {
  const size_t smem = sizeof(float) * (size_t)(splits + 1) * s.E;
  const int threads = s.E >= 512 ? 512 : (s.E + 31) / 32 * 32;
#define L_SPLIT(P)                                                                                     \
  do {                                                                                                 \
    const cudaError_t e = ensure_dynamic_smem((const void*)topk_split_kernel<P>, smem);               \
    if (e != cudaSuccess) return e;                                                                    \
    const cudaError_t e2 = launch_pdl(topk_split_kernel<P>, dim3(s.T), dim3(threads), smem, st, partial, splits, s.T, \
                                      s.E, s.k, idx, wts, logits_out, status);                                     \
    if (e2 != cudaSuccess) return e2;                                                                                 \
  } while (0)
  MOE_TOPK_DISPATCH(L_SPLIT);
#undef L_SPLIT
  return cudaGetLastError();
}

bool route_tail_supported(const moe_shape& s) {
  const size_t smem = sizeof(float) * (size_t)(route_splits(s.d) + 1) * s.E;
  return s.T >= 1 && s.T <= 8 && s.T * s.k <= 256 && s.E <= 512 && s.E % 4 == 0 && smem <= 100 * 1024;
}

cudaError_t launch_route_tail(const moe_shape& s, const float* partial, int splits, int32_t* idx, float* wts,
                              float* logits_out, int32_t* counts, int32_t* offsets, int32_t* sorted_pair,
                              int32_t* inv_pos, int32_t* active, int* status, cudaStream_t st) {
  const size_t smem = sizeof(float) * (size_t)(splits + 1) * s.E;
  int n = s.T * s.k > s.E ? s.T * s.k : s.E;
  n = (n + 31) / 32 * 32;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(s.T);
  cfg.blockDim = dim3(n);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = s.T;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = ensure_dynamic_smem((const void*)route_tail_kernel, smem);
  if (e != cudaSuccess) return e;
  e = cudaLaunchKernelEx(&cfg, route_tail_kernel, partial, splits, s.T, s.E, s.k, idx, wts, logits_out, counts, offsets,
                         sorted_pair, inv_pos, active, status);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace moe
