// Combine / unpermute: each token's output is the gated mixture of its selected experts
// ("单张RTX 5090跑125B大模型：Strata实测Qwen3.8 Flash Next", section "MoE专家按需调度"), plus the
// shared expert applied to every token ("Strata 工作原理图解GPU内存SSD三级存储如何让125B模型塞进消费级显卡",
// section "三级存储分工"):
//   out[t] = sum_j w[t][j] * y_perm[inv_pos[t*k + j]] + sum_s y_perm[P + s*T + t] (+ residual[t])
// The sum is fp32 in exactly that order (deterministic) and is rounded once to the output type.
// One thread produces 4 consecutive columns of one token. The token's k rows and weights are
// read once per CTA into shared memory; each thread then requests all of its k rows before it
// adds any of them, so the loads are in flight together instead of one after another.
#include "moe_common.cuh"

namespace moe {

__device__ __forceinline__ float4 load4(const void* p, int dt, size_t off) {
  if (dt == 1) return *reinterpret_cast<const float4*>(static_cast<const float*>(p) + off);
  const uint2 v = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(p) + off);
  return make_float4(bf16_bits_to_f32(v.x & 0xFFFFu), bf16_bits_to_f32(v.x >> 16),
                     bf16_bits_to_f32(v.y & 0xFFFFu), bf16_bits_to_f32(v.y >> 16));
}

__device__ __forceinline__ void fma4(float w, const float4& v, float4& a) {
  a.x = fmaf(w, v.x, a.x); a.y = fmaf(w, v.y, a.y); a.z = fmaf(w, v.z, a.z); a.w = fmaf(w, v.w, a.w);
}

__global__ void __launch_bounds__(256) combine_kernel(const void* __restrict__ y, int ydt,
                                                      const int32_t* __restrict__ inv_pos,
                                                      const float* __restrict__ topk_w,
                                                      const void* residual, void* out, int odt, int T, int d,
                                                      int k, int n_shared) {
  __shared__ int s_row[32];
  __shared__ float s_w[32];
  const int t = blockIdx.y;
  const int c = (blockIdx.x * blockDim.x + threadIdx.x) * 4;
  pdl_wait();  // y_perm from the expert FFN
  if (threadIdx.x < k) {
    s_row[threadIdx.x] = inv_pos[(size_t)t * k + threadIdx.x];
    s_w[threadIdx.x] = topk_w[(size_t)t * k + threadIdx.x];
  }
  __syncthreads();
  if (c >= d) return;
  const size_t P = (size_t)T * k;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j0 = 0; j0 < k; j0 += 8) {  // k <= 32: up to 8 rows requested before they are added
    float4 v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (j0 + q < k) v[q] = load4(y, ydt, (size_t)s_row[j0 + q] * d + c);
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (j0 + q < k) fma4(s_w[j0 + q], v[q], acc);
  }
  for (int s = 0; s < n_shared; ++s) {
    const float4 v = load4(y, ydt, (P + (size_t)s * T + t) * d + c);
    acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
  }
  if (residual) {
    const float4 v = load4(residual, odt, (size_t)t * d + c);
    acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
  }
  const size_t o = (size_t)t * d + c;
  if (odt == 1) {
    *reinterpret_cast<float4*>(static_cast<float*>(out) + o) = acc;
  } else {
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 v;
    v.x = *reinterpret_cast<uint32_t*>(&lo);
    v.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + o) = v;
  }
}

cudaError_t launch_combine(const moe_shape& s, const void* y, int ydt, const int32_t* inv_pos,
                           const float* topk_w, const void* residual, void* out, int odt, cudaStream_t st,
                           bool pdl) {
  const int threads = 256;
  dim3 grid((s.d / 4 + threads - 1) / threads, s.T);
  return launch_maybe_pdl(pdl, combine_kernel, grid, dim3(threads), 0, st, y, ydt, inv_pos, topk_w, residual, out, odt,
                          s.T, s.d,
                    s.k, s.n_shared);
}

// RMS normalisation of each token's row, the input of a pre-norm residual block:
//   out[t] = x[t] / sqrt(mean_i x[t][i]^2 + eps)   (no learned gain)
// One CTA per token. Each thread sums the squares of its columns (4 at a time, in column
// order), the warps reduce by a fixed butterfly and warp 0 adds the 8 warp sums in order, so
// the result is deterministic. x and out may be the same buffer.
__global__ void __launch_bounds__(256) rms_norm_kernel(const void* x, int xdt, void* out, int odt, int d,
                                                       float eps) {
  __shared__ float wsum[8];
  __shared__ float inv_s;
  const int t = blockIdx.x;
  pdl_trigger();  // the router may launch; it waits for this grid before reading out
  pdl_wait();     // x from the kernel before (a layer's combine in a stack)
  const size_t row = (size_t)t * d;
  float ss = 0.0f;
  for (int c = threadIdx.x * 4; c < d; c += blockDim.x * 4) {
    const float4 v = load4(x, xdt, row + c);
    ss = fmaf(v.x, v.x, ss);
    ss = fmaf(v.y, v.y, ss);
    ss = fmaf(v.z, v.z, ss);
    ss = fmaf(v.w, v.w, ss);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
  if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    float tot = 0.0f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += wsum[w];
    inv_s = 1.0f / sqrtf(tot / (float)d + eps);
  }
  __syncthreads();
  const float inv = inv_s;
  for (int c = threadIdx.x * 4; c < d; c += blockDim.x * 4) {
    float4 v = load4(x, xdt, row + c);
    v.x *= inv; v.y *= inv; v.z *= inv; v.w *= inv;
    if (odt == 1) {
      *reinterpret_cast<float4*>(static_cast<float*>(out) + row + c) = v;
    } else {
      __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
      uint2 u;
      u.x = *reinterpret_cast<uint32_t*>(&lo);
      u.y = *reinterpret_cast<uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + row + c) = u;
    }
  }
}

cudaError_t launch_rms_norm(const moe_shape& s, const void* x, int xdt, void* out, int odt, float eps,
                            cudaStream_t st, bool pdl) {
  return launch_maybe_pdl(pdl, rms_norm_kernel, dim3(s.T), dim3(256), 0, st, x, xdt, out, odt, s.d, eps);
}

}  // namespace moe
