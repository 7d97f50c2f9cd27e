// Router logits on the tcgen05 tensor cores, for many tokens (prefill), at fp32 accuracy.
//
// The router picks the top-K experts of each token ("单张RTX 5090跑125B大模型：Strata实测Qwen3.8
// Flash Next", section "MoE专家按需调度"); for a prefill chunk of thousands of tokens its logits
// logit[t][e] = sum_i x[t][i] * w[i][e] are a dense GEMM (2 T d E flops), the one dense
// contraction of the layer that is not an expert.
//
// Exactness of the operands. x is bf16, so it enters a bf16 MMA exactly. Each fp32 router weight
// is split into three bf16 parts, w = hi + mid + lo, each part the bf16 rounding of what the parts
// before it leave: 24 significant bits in 3 x 8, so the sum is exact (for |w| above the bf16
// normal range's lower end times 2^16). Every product x * part is then exact in fp32, and the
// logit is the sum of 3 d exact products: the one rounding is the fp32 accumulation of the MMAs.
//
// Depth of that accumulation. K (= d) is cut into four quarters; each quarter accumulates into
// its own TMEM accumulator (the three parts of every K step into the same one), and the four are
// added in a fixed order at the end, (q0 + q1) + (q2 + q3). At d = 2048 a quarter is 512 K
// elements, 96 chained MMA accumulations of 16-element chunks, so the addition depth stays near
// that of the SIMT kernel's blocked sum. The result is deterministic.
//
// Kernels: router_split_kernel writes the parts transposed, [3][E][d] bf16 (each expert's column
// contiguous in K, the operand layout the MMA reads), and clears the layer's status word. Then
// router_tc_kernel: one CTA per 128 tokens x 128 experts; warp 0 lane 0 issues the TMA copies of
// one stage (the x tile and the three part tiles, 64 elements of K, 128-byte swizzle; 3 stages),
// warp 1 lane 0 issues 12 tcgen05.mma (M128 N128 K16) per stage, warps 2..5 read the four
// accumulators (tcgen05.ld) and write fp32 logits. Every wait is bounded; one that runs out sets
// MOE_DEV_TIMEOUT, and the copies and MMAs already issued are waited for before TMEM is freed.
#include <cuda.h>

#include "moe_common.cuh"
#include "sm100_ptx.cuh"
#include "tmap.h"

namespace moe {

namespace {

constexpr int kRM = 128;                              // tokens per tile (UMMA M)
constexpr int kRN = 128;                              // experts per tile (UMMA N)
constexpr int kRK = 64;                               // K elements per stage (128 bytes of bf16)
constexpr int kRStages = 3;
constexpr int kRTileA = kRM * 128;                    // 16 KB
constexpr int kRTileB = kRN * 128;                    // 16 KB per part
constexpr int kRStageBytes = kRTileA + 3 * kRTileB;   // 64 KB
constexpr int kRThreads = 192;                        // warp 0: TMA, 1: MMA, 2..5: epilogue
constexpr size_t kRHeadBytes = 1024;
constexpr size_t kRSmem = kRHeadBytes + 1024 + (size_t)kRStages * kRStageBytes;

struct RHead {
  uint64_t full[kRStages];
  uint64_t empty[kRStages];
  uint64_t acc;
  uint64_t drain;
  uint32_t tmem;
  int abort;
};
static_assert(sizeof(RHead) <= kRHeadBytes, "head too large");

__device__ __forceinline__ uint64_t r_sw128_desc(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// kind::f16 instruction descriptor: fp32 accumulator, bf16 A and B (both K-major), N and M.
constexpr uint32_t bf16_idesc(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ bool r_aborted(const RHead& H) { return *(volatile const int*)&H.abort != 0; }

__device__ __forceinline__ void r_set_abort(RHead& H, int* status) {
  if (!r_aborted(H)) {
    H.abort = 1;
    flag_status(status, MOE_DEV_TIMEOUT_BIT);
  }
}

// parts[p][e][i] (bf16) for w[i][e] (fp32): 32 x 32 tiles through shared memory. Also clears the
// status word (unless a stack keeps it across layers): this kernel is the first of the layer on
// the stream.
__global__ void __launch_bounds__(256) router_split_kernel(const float* __restrict__ w, __nv_bfloat16* parts,
                                                           int d, int E, int* status, int clear_status) {
  __shared__ float tile[32][33];
  if (clear_status && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *status = 0;
  const int e0 = blockIdx.x * 32, i0 = blockIdx.y * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 8 rows per pass
  for (int r = ty; r < 32; r += 8) {
    const int i = i0 + r, e = e0 + tx;
    tile[r][tx] = (i < d && e < E) ? w[(size_t)i * E + e] : 0.0f;
  }
  __syncthreads();
  for (int r = ty; r < 32; r += 8) {
    const int e = e0 + r, i = i0 + tx;
    if (e >= E || i >= d) continue;
    const float v = tile[tx][r];
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    const float r1 = v - __bfloat162float(hi);  // exact
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const __nv_bfloat16 lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));  // exact difference, exact part
    const size_t o = (size_t)e * d + i, pe = (size_t)E * d;
    parts[o] = hi;
    parts[pe + o] = mid;
    parts[2 * pe + o] = lo;
  }
}

__global__ void __launch_bounds__(kRThreads, 1) router_tc_kernel(const __grid_constant__ CUtensorMap tm_x,
                                                                 const __grid_constant__ CUtensorMap tm_w,
                                                                 float* __restrict__ logits, int T, int d, int E,
                                                                 int* status, uint64_t wait_ns) {
  extern __shared__ __align__(1024) uint8_t dyn[];
  RHead& H = *reinterpret_cast<RHead*>(dyn);
  uint8_t* ring = dyn + kRHeadBytes;
  {
    const uint32_t a = smem_u32(ring);
    ring += ((a + 1023u) & ~1023u) - a;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * kRM, n0 = blockIdx.y * kRN;
  const int KC = d / kRK, KQ = KC / 4;  // K steps, and K steps per quarter

  if (threadIdx.x == 0) {
    for (int s = 0; s < kRStages; ++s) {
      mbar_init(&H.full[s], 1);
      mbar_init(&H.empty[s], 1);
    }
    mbar_init(&H.acc, 1);
    mbar_init(&H.drain, 1);
    H.abort = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_x);
    prefetch_tmap(&tm_w);
  }
  if (warp == 1) {
    tmem_alloc(&H.tmem, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = H.tmem;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      int issued = 0;
      for (int kc = 0; kc < KC; ++kc) {
        const int s = kc % kRStages;
        const uint32_t ph = (uint32_t)(kc / kRStages) & 1u;
        if (!mbar_wait(&H.empty[s], ph ^ 1u, wait_ns) || r_aborted(H)) {
          r_set_abort(H, status);
          break;
        }
        uint8_t* st = ring + (size_t)s * kRStageBytes;
        mbar_arrive_expect_tx(&H.full[s], kRStageBytes);
        tma_load_2d(st, &tm_x, kc * kRK, m0, &H.full[s]);
        for (int p = 0; p < 3; ++p) tma_load_2d(st + kRTileA + p * kRTileB, &tm_w, kc * kRK, p * E + n0, &H.full[s]);
        ++issued;
      }
      if (r_aborted(H))  // no copy may still be landing in shared memory when the CTA exits
        for (int j = issued > kRStages ? issued - kRStages : 0; j < issued; ++j)
          mbar_wait(&H.full[j % kRStages], (uint32_t)(j / kRStages) & 1u);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = bf16_idesc(kRM, kRN);
      for (int kc = 0; kc < KC; ++kc) {
        const int s = kc % kRStages;
        const uint32_t ph = (uint32_t)(kc / kRStages) & 1u;
        if (!mbar_wait(&H.full[s], ph, wait_ns) || r_aborted(H)) {
          r_set_abort(H, status);
          break;
        }
        tc_fence_after();
        const uint32_t a = smem_u32(ring + (size_t)s * kRStageBytes);
        const int q = kc / KQ;
        const uint32_t d_tmem = tmem + (uint32_t)(q * kRN);
#pragma unroll
        for (int k = 0; k < kRK / 16; ++k)
#pragma unroll
          for (int p = 0; p < 3; ++p)
            umma_f16(d_tmem, r_sw128_desc(a + k * 32), r_sw128_desc(a + kRTileA + p * kRTileB + k * 32), idesc,
                     (kc % KQ) != 0 || k != 0 || p != 0);
        umma_commit(&H.empty[s]);
      }
      umma_commit(&H.acc);
      // every MMA this thread issued has completed before TMEM and the ring are freed
      umma_commit(&H.drain);
      mbar_wait(&H.drain, 0);
    }
  } else {
    // ---------------- epilogue ----------------
    const int qd = warp & 3;  // TMEM lane quarter this warp may read
    const bool ok = mbar_wait(&H.acc, 0, wait_ns) && !r_aborted(H);
    if (__all_sync(0xFFFFFFFFu, ok)) {
      tc_fence_after();
      const int m = m0 + qd * 32 + lane;
      const uint32_t t_row = tmem + ((uint32_t)(qd * 32) << 16);
      for (int c = 0; c < kRN; c += 16) {
        uint32_t v0[16], v1[16], v2[16], v3[16];
        tmem_ld16(t_row + c, v0);
        tmem_ld16(t_row + kRN + c, v1);
        tmem_ld16(t_row + 2 * kRN + c, v2);
        tmem_ld16(t_row + 3 * kRN + c, v3);
        // one wait for the four loads; the other three only tie their registers to it, so that
        // no use of them is scheduled above the wait
        tmem_ld_wait16(v0);
        tmem_ld_wait16(v1);
        tmem_ld_wait16(v2);
        tmem_ld_wait16(v3);
        if (m < T) {
          float v[16];
#pragma unroll
          for (int j = 0; j < 16; ++j)
            v[j] = (__uint_as_float(v0[j]) + __uint_as_float(v1[j])) + (__uint_as_float(v2[j]) + __uint_as_float(v3[j]));
          float* dst = logits + (size_t)m * E + n0 + c;
          if ((E & 3) == 0 && n0 + c + 16 <= E) {
#pragma unroll
            for (int j = 0; j < 16; j += 4) *reinterpret_cast<float4*>(dst + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (n0 + c + j < E) dst[j] = v[j];
          }
        }
      }
    } else if (lane == 0) {
      r_set_abort(H, status);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

bool route_tc_supported(const moe_shape& s, int xdt) {
  return xdt == 0 && s.T > kRouteGemvMaxT && s.d % (4 * kRK) == 0 && tmap_available();
}

size_t route_tc_parts_bytes(const moe_shape& s) { return sizeof(__nv_bfloat16) * 3 * (size_t)s.E * s.d; }

cudaError_t launch_route_tc(const moe_shape& s, const void* x, const float* w, void* parts, float* logits, int* status,
                            cudaStream_t st, bool clear_status) {
  CUtensorMap tm_x, tm_w;
  if (!tmap_encode_2d(&tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, (uint64_t)s.d, (uint64_t)s.T, (uint64_t)s.d * 2,
                      kRK, kRM, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !tmap_encode_2d(&tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, parts, (uint64_t)s.d, (uint64_t)3 * s.E,
                      (uint64_t)s.d * 2, kRK, kRN, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  router_split_kernel<<<dim3((s.E + 31) / 32, (s.d + 31) / 32), 256, 0, st>>>(
      w, static_cast<__nv_bfloat16*>(parts), s.d, s.E, status, clear_status ? 1 : 0);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if ((e = ensure_dynamic_smem(reinterpret_cast<const void*>(router_tc_kernel), kRSmem)) != cudaSuccess) return e;
  router_tc_kernel<<<dim3((s.T + kRM - 1) / kRM, (s.E + kRN - 1) / kRN), kRThreads, kRSmem, st>>>(
      tm_x, tm_w, logits, s.T, s.d, s.E, status, wait_limit_ns());
  return cudaGetLastError();
}

}  // namespace moe
