// Expert FFN for few tokens per expert (decode and speculative verification).
//
// For T = 4 tokens and top-10 (one token plus three drafts per step, "Strata 工作原理图解GPU内存SSD
// 三级存储如何让125B模型塞进消费级显卡", section "推测解码") almost every selected expert sees one token.
// The work is then a GEMV per expert, and its time is that of streaming the selected experts'
// int8 rows and fp16 scales from HBM. Each byte is read once: the bucketing step gave
// every expert all of its tokens, so one pass over the weights serves all of them.
//
// Two kernels, each with a 2-D grid of (row block, work item). A work item is a routed
// expert from the active list or a shared expert:
//  * gate/up: for each row r of the expert's gate and up matrices [f][d], both dot products
//    with the token activations (staged as fp32 in shared memory), then
//    h = silu(g) * u -> fp32 h [P + T*n_shared][f] in the workspace;
//  * down: for each row n of the down matrix [d][f], the dot product with h -> y_perm.
// Weights are dequantised exactly (int8 * fp16 is exact in fp32) and all arithmetic is fp32.
// Rows are read with 128-bit loads that skip L1, and each lane keeps several rows' chunks
// in flight. A row's 32-element block shares one scale, and the partial sum of each
// 16-element chunk is scaled once.
#include "moe_common.cuh"

namespace moe {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kGateUpRowsPerCta = 16;  // 2 rows per warp
constexpr int kDownRowsPerCta = 32;

// Shared-memory layout of staged vectors: a length-n vector is n/16 chunks of four float4;
// float4 j of chunk c of vector t sits at index (t * 4 + j) * (n / 16) + c. Lanes that read
// consecutive chunks then read consecutive float4s (no bank conflicts). Vectors are staged in
// the stored order of the code rows (code_pos), so chunk c of a vector meets chunk c of a row.
__device__ __forceinline__ int il_index(int t, int j, int c, int nch) { return (t * 4 + j) * nch + c; }

// Stage activations of tokens [g0, g0 + ng) of item `it` into xs (fp32, interleaved layout).
__device__ __forceinline__ void stage_x(const FfnArgs& A, const FfnItem& it, int g0, int ng, float4* xs) {
  const int nch = A.d / 16;
  for (int t = 0; t < ng; ++t) {
    const int tok = item_token(A, it, g0 + t);
    if (A.xdt == 0) {
      const uint16_t* src = static_cast<const uint16_t*>(A.x) + (size_t)tok * A.d;
      for (int i = threadIdx.x * 8; i < A.d; i += kThreads * 8) {  // d % 32 == 0: 16-byte loads
        const uint4 v = *reinterpret_cast<const uint4*>(src + i);
        const int pk = code_pos(i, A.d);  // the 8 elements stay together
        const int c = pk >> 4, j = (pk & 15) >> 2;
        xs[il_index(t, j, c, nch)] = make_float4(bf16_bits_to_f32(v.x & 0xFFFFu), bf16_bits_to_f32(v.x >> 16),
                                                 bf16_bits_to_f32(v.y & 0xFFFFu), bf16_bits_to_f32(v.y >> 16));
        xs[il_index(t, j + 1, c, nch)] = make_float4(bf16_bits_to_f32(v.z & 0xFFFFu), bf16_bits_to_f32(v.z >> 16),
                                                     bf16_bits_to_f32(v.w & 0xFFFFu), bf16_bits_to_f32(v.w >> 16));
      }
    } else {
      const float* src = static_cast<const float*>(A.x) + (size_t)tok * A.d;
      for (int i = threadIdx.x * 4; i < A.d; i += kThreads * 4) {
        const int pk = code_pos(i & ~7, A.d) + (i & 7);
        xs[il_index(t, (pk & 15) >> 2, pk >> 4, nch)] = *reinterpret_cast<const float4*>(src + i);
      }
    }
  }
}

// Stage h rows [row, row + ng) (fp32 [.][f] in global memory) into hs (interleaved layout).
__device__ __forceinline__ void stage_h(const float* h, int f, int ng, float4* hs) {
  const int nch = f / 16;
  for (int i = threadIdx.x * 4; i < ng * f; i += kThreads * 4) {
    const int t = i / f, e = i % f;
    const int pk = code_pos(e & ~7, f) + (e & 7);
    hs[il_index(t, (pk & 15) >> 2, pk >> 4, nch)] = *reinterpret_cast<const float4*>(h + i);
  }
}

// The scales of the two 8-code halves of stored chunk c of a row with K codes (scales: the
// row's block scales): a paired chunk holds 8 codes of blocks 2p and 2p + 1, a chunk of a
// trailing unpaired block 16 codes of that block.
__device__ __forceinline__ void chunk_scales(const __half* scales, int c, int K, float* s0, float* s1) {
  if (c < (K >> 6) * 4) {
    *s0 = __half2float(scales[(c >> 2) * 2]);
    *s1 = __half2float(scales[(c >> 2) * 2 + 1]);
  } else {
    *s0 = *s1 = __half2float(scales[c >> 1]);
  }
}

// acc[t] += s0 * dot(q[0..8), ...) + s1 * dot(q[8..16), ...) with chunk c of staged vector t,
// for t < ng <= NT. One 32-bit word (four codes) at a time, so that few values are live at
// once. `ng` is the same for the whole CTA, so the token guards do not diverge.
template <int NT>
__device__ __forceinline__ void dot16(const uint4& w, float s0, float s1, const float4* vs, int c, int nch, int ng,
                                      float* acc) {
  float s[NT];
  const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float q[4];
    i8x4_to_f32(words[j], q);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      if (t < ng) {
        const float4 v = vs[il_index(t, j, c, nch)];
        float p = (j == 0 || j == 2) ? q[0] * v.x : fmaf(q[0], v.x, s[t]);
        p = fmaf(q[1], v.y, p);
        p = fmaf(q[2], v.z, p);
        s[t] = fmaf(q[3], v.w, p);
      }
    }
    if (j == 1 || j == 3) {
#pragma unroll
      for (int t = 0; t < NT; ++t)
        if (t < ng) acc[t] = fmaf(j == 1 ? s0 : s1, s[t], acc[t]);
    }
  }
}

template <int NT>
__device__ __forceinline__ float warp_sum_get(float (&v)[NT], int t) {
  float r = 0.0f;
#pragma unroll
  for (int i = 0; i < NT; ++i) r = (i == t) ? v[i] : r;
  return r;
}

// ---------------------------------------------------------------- gate/up + SwiGLU ---------

template <int NT>
__device__ __forceinline__ void gateup_group(const FfnArgs& A, const FfnItem& it, int g0, int ng,
                                             const float4* xs) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = A.d, nch = d / 16;  // 16-byte chunks per row
  const int nb = d / kQBlock;
  const uint8_t* gq = it.rec + A.o_gate_q;
  const uint8_t* uq = it.rec + A.o_up_q;
  const __half* gs = reinterpret_cast<const __half*>(it.rec + A.o_gate_s);
  const __half* us = reinterpret_cast<const __half*>(it.rec + A.o_up_s);
  const int rbase = blockIdx.x * kGateUpRowsPerCta + warp * 2;
  for (int rr = 0; rr < 2; ++rr) {
    const int r = rbase + rr;
    if (r >= A.f) break;
    float ag[NT], au[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) ag[t] = au[t] = 0.0f;
    const uint8_t* growp = gq + (size_t)r * d;
    const uint8_t* urowp = uq + (size_t)r * d;
    for (int c0 = 0; c0 < nch; c0 += 32 * 4) {  // up to 4 chunks per lane in flight per matrix
      uint4 wg[4], wu[4];
      float sg0[4], sg1[4], su0[4], su1[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c < nch) {
          wg[u] = ld_stream16(growp + c * 16);
          wu[u] = ld_stream16(urowp + c * 16);
          chunk_scales(gs + (size_t)r * nb, c, d, &sg0[u], &sg1[u]);
          chunk_scales(us + (size_t)r * nb, c, d, &su0[u], &su1[u]);
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c < nch) {
          dot16<NT>(wg[u], sg0[u], sg1[u], xs, c, nch, ng, ag);
          dot16<NT>(wu[u], su0[u], su1[u], xs, c, nch, ng, au);
        }
      }
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        ag[t] += __shfl_xor_sync(0xFFFFFFFFu, ag[t], o);
        au[t] += __shfl_xor_sync(0xFFFFFFFFu, au[t], o);
      }
    }
    if (lane < ng) {
      const float g = warp_sum_get<NT>(ag, lane), u = warp_sum_get<NT>(au, lane);
      A.h[(size_t)(it.row0 + g0 + lane) * A.f + r] = silu(g) * u;
    }
  }
}

__global__ void __launch_bounds__(kThreads, 2) ffn_gateup_decode_kernel(FfnArgs A) {
  extern __shared__ __align__(16) float4 xs[];  // [min(T, 8)][d] fp32, interleaved
  FfnItem it;
  if (!resolve_item(blockIdx.y, A, &it)) return;
  for (int g0 = 0; g0 < it.ntok; g0 += kDecodeTokGroup) {
    const int ng = min(kDecodeTokGroup, it.ntok - g0);
    __syncthreads();
    stage_x(A, it, g0, ng, xs);
    __syncthreads();
    gateup_group<kDecodeTokGroup>(A, it, g0, ng, xs);
  }
}

// ---------------------------------------------------------------- down ---------------------

// LPR lanes per row; each lane walks the row's 16-byte chunks with stride LPR.
template <int NT, int LPR>
__device__ __forceinline__ void down_group(const FfnArgs& A, const FfnItem& it, int g0, int ng,
                                           const float4* hs) {
  constexpr int RPW = 32 / LPR;  // rows per warp at once
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = lane / LPR, sl = lane % LPR;
  const int f = A.f, nch = f / 16, nb = f / kQBlock;
  const uint8_t* dq = it.rec + A.o_down_q;
  const __half* ds = reinterpret_cast<const __half*>(it.rec + A.o_down_s);
  const int rows_per_warp = kDownRowsPerCta / kWarps;
  for (int r0 = 0; r0 < rows_per_warp; r0 += RPW) {
    const int n = blockIdx.x * kDownRowsPerCta + warp * rows_per_warp + r0 + sub;
    const bool valid = (r0 + sub) < rows_per_warp && n < A.d;
    float acc[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[t] = 0.0f;
    if (valid) {
      const uint8_t* rowp = dq + (size_t)n * f;
      for (int c0 = 0; c0 < nch; c0 += LPR * 4) {
        uint4 w[4];
        float sc0[4], sc1[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int c = c0 + u * LPR + sl;
          if (c < nch) {
            w[u] = ld_stream16(rowp + c * 16);
            chunk_scales(ds + (size_t)n * nb, c, f, &sc0[u], &sc1[u]);
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int c = c0 + u * LPR + sl;
          if (c < nch) dot16<NT>(w[u], sc0[u], sc1[u], hs, c, nch, ng, acc);
        }
      }
    }
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int o = LPR / 2; o > 0; o >>= 1) acc[t] += __shfl_xor_sync(0xFFFFFFFFu, acc[t], o);
    if (valid && sl < ng) {
      const float v = warp_sum_get<NT>(acc, sl);
      const size_t off = (size_t)(it.row0 + g0 + sl) * A.d + n;
      if (A.ydt == 1) static_cast<float*>(A.y)[off] = v;
      else static_cast<__nv_bfloat16*>(A.y)[off] = __float2bfloat16_rn(v);
    }
  }
}

template <int LPR>
__global__ void __launch_bounds__(kThreads, 2) ffn_down_decode_kernel(FfnArgs A) {
  extern __shared__ __align__(16) float4 hs[];  // [min(T, 8)][f] fp32, interleaved
  FfnItem it;
  if (!resolve_item(blockIdx.y, A, &it)) return;
  for (int g0 = 0; g0 < it.ntok; g0 += kDecodeTokGroup) {
    const int ng = min(kDecodeTokGroup, it.ntok - g0);
    __syncthreads();
    stage_h(A.h + (size_t)(it.row0 + g0) * A.f, A.f, ng, hs);
    __syncthreads();
    down_group<kDecodeTokGroup, LPR>(A, it, g0, ng, hs);
  }
}

// Tokens staged at once: an expert has at most T tokens.
static int group_cap(const FfnArgs& a) { return a.T < kDecodeTokGroup ? a.T : kDecodeTokGroup; }

template <int LPR>
static cudaError_t launch_down(const FfnArgs& a, int items, cudaStream_t st) {
  const size_t smem = sizeof(float) * group_cap(a) * a.f;
  auto kern = ffn_down_decode_kernel<LPR>;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  dim3 grid((a.d + kDownRowsPerCta - 1) / kDownRowsPerCta, items);
  kern<<<grid, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_ffn_decode(const FfnArgs& a, cudaStream_t st) {
  const int items = (a.P < a.E ? a.P : a.E) + a.n_shared;
  if (items == 0) return cudaSuccess;
  {
    const size_t smem = sizeof(float) * group_cap(a) * a.d;
    cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(ffn_gateup_decode_kernel), smem);
    if (e != cudaSuccess) return e;
    dim3 grid((a.f + kGateUpRowsPerCta - 1) / kGateUpRowsPerCta, items);
    ffn_gateup_decode_kernel<<<grid, kThreads, smem, st>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  // lanes per down row: the largest power of two (<= 32) dividing the f/16 chunks of a row
  const int nch = a.f / 16;
  if (nch % 32 == 0) return launch_down<32>(a, items, st);
  if (nch % 16 == 0) return launch_down<16>(a, items, st);
  if (nch % 8 == 0) return launch_down<8>(a, items, st);
  if (nch % 4 == 0) return launch_down<4>(a, items, st);
  return launch_down<2>(a, items, st);
}

}  // namespace moe
