// Expert FFN for many tokens per expert (prefill): a grouped GEMM on the tcgen05 tensor cores.
//
// Prefill runs long prompts through the layer in chunks of up to 8192 tokens ("Strata 工作原理图解
// GPU内存SSD三级存储如何让125B模型塞进消费级显卡", section "长文本"), and its expert matmuls run on
// the tensor cores without a separate dequantisation pass ("Strata 性能基准与论文导读125B MoE在
// 消费级硬件上的极限测量与瓶颈分析", section "瓶颈分析 1️⃣"). Kernels:
//   prepare: per-token power-of-two scale of x, the work-item table, the token of every row,
//            cleared max |h| per row, and the list of 128-row M tiles of every item;
//   gather:  xp16[r] = f16(x[token of r] * 2^-e): the rows of every expert contiguous;
//   gemm<GU>: for each (M tile, 128 columns of f): D[128][256] = A[128][d] . B[256][d]^T with
//            B rows 0..127 the gate rows and 128..255 the same up rows, then h = silu(g) * u
//            (fp32) and an atomic max |h| per row;
//   convert: h16[r] = f16(h[r] * 2^-e_r) with e_r from max |h| of the row;
//   gemm<DN>: for each (M tile, 256 rows of d): D[128][256] = h16[128][f] . Wd[256][f]^T.
//
// The GEMM is persistent (one CTA per SM, a static stride over the work list) and warp
// specialised:
//   warp 0, lane 0: TMA. Per 64-element K step (one pair of 32-element blocks) it loads the A
//            tile (128 rows x 128 bytes of f16, 128-byte swizzle) and the int8 codes of the 256 B
//            rows (256 x 64 bytes, each row's pair of blocks in the stored order: 16-byte chunk c
//            holds codes 8c..8c+7 of both blocks).
//   warps 1..8: converters. Each thread turns 4 x 16 codes into f16 (q * s, one rounding; the
//            fp16 scale s of the code's 32-element block) and writes them into the B tile in the
//            128-byte-swizzled K-major layout the tensor core reads, then fences them into the
//            async proxy. The int8 codes stay exact until this single rounding.
//   warp 9, lane 0: issues 4 tcgen05.mma (M = 128, N = 256, K = 16) per K step into one of two
//            TMEM accumulators (2 x 256 columns) and commits each stage back to the producers.
//   warps 12..15: epilogue. TMEM lanes 32 q .. 32 q + 31 (q = warp % 4) hold rows of the tile;
//            tcgen05.ld 16 columns at a time while the next tile accumulates in the other buffer.
// Activations enter as f16 exactly (bf16 has 8 significant bits; each row is rescaled by a power
// of two that puts its max |x| in [2^14, 2^15)), and h is rescaled per row the same way.
//
// Every wait is bounded. A wait that runs out sets MOE_DEV_TIMEOUT and the CTA stops its work;
// every role still reaches the final barrier, so the TMEM columns are always freed.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "moe_common.cuh"
#include "sm100_ptx.cuh"

namespace moe {

constexpr int kPM = 128;                     // rows per M tile (UMMA M)
constexpr int kPN = 256;                     // UMMA N
constexpr int kPK = 64;                      // K elements per stage (128 bytes of f16)
constexpr int kPAStage = kPM * 128;          // 16 KB
constexpr int kPBStage = kPN * 128;          // 32 KB
constexpr int kPIStage = kPN * kPK;          // 16 KB of int8 codes
constexpr int kPStages = 3;                  // A / B ring depth
constexpr int kPIStages = 4;                 // int8 ring depth
constexpr int kPConv = 8;                    // converter warps
constexpr int kPThreads = 32 * 16;           // 0: TMA, 1..8: convert, 9: MMA, 12..15: epilogue
constexpr int kPMmaWarp = 9;
constexpr int kPEpiWarp0 = 12;

enum { kPGateUp = 0, kPDown = 1 };

struct PHead {
  uint64_t a_full[kPStages];
  uint64_t b_full[kPStages];
  uint64_t ab_empty[kPStages];
  uint64_t i_full[kPIStages];
  uint64_t i_empty[kPIStages];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint32_t tmem;
  int abort;
};
constexpr size_t kPHeadBytes = 1024;
static_assert(sizeof(PHead) <= kPHeadBytes, "head too large");
constexpr size_t kPSmem = kPHeadBytes + 1024 + (size_t)kPStages * (kPAStage + kPBStage) + (size_t)kPIStages * kPIStage;

__device__ __forceinline__ float p_pow2f(int e) { return __uint_as_float((uint32_t)(127 + e) << 23); }

__device__ __forceinline__ int p_f16_exp_for(float m) {
  if (!(m > 0.0f)) return 0;
  const int e = (int)((__float_as_uint(m) >> 23) & 0xFF) - 127 - 14;
  return e < -100 ? -100 : (e > 100 ? 100 : e);
}

__device__ __forceinline__ bool p_aborted(const PHead& H) { return *(volatile const int*)&H.abort != 0; }

__device__ __forceinline__ void p_set_abort(PHead& H, int* status) {
  if (!p_aborted(H)) {
    H.abort = 1;
    flag_status(status, MOE_DEV_TIMEOUT_BIT);
  }
}

// Shared-memory descriptor of a K-major operand tile with 128-byte rows in the 128-byte
// swizzle: 8-row atoms of 1024 bytes stacked along M/N (stride 1024), descriptor version 1.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// kind::f16 instruction descriptor: fp32 accumulator, f16 A and B, both K-major, N and M.
__host__ __device__ constexpr uint32_t f16_idesc(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// A lane's 16 stored codes (8 of each block of a pair) -> 16 f16 values q * s: codes 0..7 with
// the first block's scale into lo, codes 8..15 with the second block's into hi.
__device__ __forceinline__ void codes_to_f16(const uint4& q, __half2 s_lo, __half2 s_hi, uint4* lo, uint4* hi) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  uint32_t o[8];
  const __half2 off = __half2half2(__ushort_as_half(0x6480));  // 1152
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t u = w[i] ^ 0x80808080u;
    const uint32_t p01 = __byte_perm(u, 0x64646464u, 0x5140), p23 = __byte_perm(u, 0x64646464u, 0x5342);
    const __half2 s2 = i < 2 ? s_lo : s_hi;
    const __half2 h01 = __hmul2(__hsub2(*reinterpret_cast<const __half2*>(&p01), off), s2);
    const __half2 h23 = __hmul2(__hsub2(*reinterpret_cast<const __half2*>(&p23), off), s2);
    o[2 * i] = *reinterpret_cast<const uint32_t*>(&h01);
    o[2 * i + 1] = *reinterpret_cast<const uint32_t*>(&h23);
  }
  *lo = make_uint4(o[0], o[1], o[2], o[3]);
  *hi = make_uint4(o[4], o[5], o[6], o[7]);
}

// ------------------------------------------------------------------ prepare / gather ------

// CTA t: exponent and unscale of token t. All CTAs: hmax[r] = 0 and row_tok[r]. CTA 0: items
// and the M-tile list (tiles in item order, then by row).
__global__ void __launch_bounds__(256) prefill_prepare_kernel(FfnArgs A, PrefillAux X) {
  __shared__ float wmax[8];
  __shared__ int scan[257];
  const int t = blockIdx.x;
  const int rows = A.P + A.T * A.n_shared;
  for (int r = t * blockDim.x + threadIdx.x; r < rows; r += gridDim.x * blockDim.x) {
    X.hmax[r] = 0u;
    X.row_tok[r] = r < A.P ? A.sorted_pair[r] / A.k : (r - A.P) % A.T;
  }
  if (t == 0) {
    const int n = A.active[0] + A.n_shared;
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
    }
    __syncthreads();
    // thread j owns items [j * per, (j + 1) * per): count its tiles, scan, write them
    const int per = (n + blockDim.x - 1) / blockDim.x;
    const int i0 = threadIdx.x * per, i1 = min(n, i0 + per);
    int cnt = 0;
    for (int i = i0; i < i1; ++i) {
      const ItemRec rec = X.items[i];
      if (rec.rec) cnt += (rec.ntok + kPM - 1) / kPM;
    }
    scan[threadIdx.x + 1] = cnt;
    if (threadIdx.x == 0) scan[0] = 0;
    __syncthreads();
    if (threadIdx.x == 0)
      for (int j = 1; j <= (int)blockDim.x; ++j) scan[j] += scan[j - 1];
    __syncthreads();
    int o = scan[threadIdx.x];
    for (int i = i0; i < i1; ++i) {
      const ItemRec rec = X.items[i];
      if (!rec.rec) continue;
      for (int m0 = 0; m0 < rec.ntok; m0 += kPM) X.tiles[o++] = make_int2(i, m0);
    }
    if (threadIdx.x == 0) X.n_tiles[0] = scan[blockDim.x];
  }
  const int d = A.d;
  float m = 0.0f;
  for (int i = threadIdx.x; i < d; i += blockDim.x) m = fmaxf(m, fabsf(load_act(A.x, A.xdt, (size_t)t * d + i)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
  __syncthreads();
  m = 0.0f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) m = fmaxf(m, wmax[w]);
  if (threadIdx.x == 0) {
    const int e = p_f16_exp_for(m);
    X.xexp[t] = e;
    X.xunscale[t] = p_pow2f(e);
  }
}

// xp16[r][:] = f16(x[token of r][:] * 2^-e): 8 elements per thread.
__global__ void __launch_bounds__(256) prefill_gather_kernel(FfnArgs A, PrefillAux X) {
  const int rows = A.P + A.T * A.n_shared, d = A.d, per_row = d / 8;
  const size_t n = (size_t)rows * per_row;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const int r = (int)(i / per_row), c = (int)(i % per_row) * 8;
    const int tok = X.row_tok[r];
    const float down = p_pow2f(-X.xexp[tok]);
    float v[8];
    if (A.xdt == 0) {
      const uint4 b = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(A.x) + (size_t)tok * d + c);
      const uint32_t w[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[2 * j] = bf16_bits_to_f32(w[j] & 0xFFFFu);
        v[2 * j + 1] = bf16_bits_to_f32(w[j] >> 16);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = static_cast<const float*>(A.x)[(size_t)tok * d + c + j];
    }
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __half2 h = __floats2half2_rn(v[2 * j] * down, v[2 * j + 1] * down);
      o[j] = *reinterpret_cast<const uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(X.xp16 + (size_t)r * d + c) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// h16[r] = f16(h[r] * 2^-e_r), hexp[r] = e_r, with e_r from max |h| of row r: 8 per thread.
__global__ void __launch_bounds__(256) prefill_convert_h_kernel(FfnArgs A, PrefillAux X) {
  const int rows = A.P + A.T * A.n_shared, f = A.f, per_row = f / 8;
  const size_t n = (size_t)rows * per_row;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const int r = (int)(i / per_row), c = (int)(i % per_row) * 8;
    const int e = p_f16_exp_for(__uint_as_float(X.hmax[r]));
    const float down = p_pow2f(-e);
    const float4 a = *reinterpret_cast<const float4*>(A.h + (size_t)r * f + c);
    const float4 b = *reinterpret_cast<const float4*>(A.h + (size_t)r * f + c + 4);
    const __half2 h0 = __floats2half2_rn(a.x * down, a.y * down), h1 = __floats2half2_rn(a.z * down, a.w * down);
    const __half2 h2 = __floats2half2_rn(b.x * down, b.y * down), h3 = __floats2half2_rn(b.z * down, b.w * down);
    *reinterpret_cast<uint4*>(X.h16 + (size_t)r * f + c) =
        make_uint4(*reinterpret_cast<const uint32_t*>(&h0), *reinterpret_cast<const uint32_t*>(&h1),
                   *reinterpret_cast<const uint32_t*>(&h2), *reinterpret_cast<const uint32_t*>(&h3));
    if (c == 0) X.hexp[r] = e;
  }
}

// ------------------------------------------------------------------ the GEMM --------------

struct PWork {
  int item, rowA, nrows, n0, slot, shared;
  const uint8_t* rec;
};

template <int KIND>
__device__ __forceinline__ bool work_at(const FfnArgs& A, const PrefillAux& X, int w, int nch, PWork* out) {
  const int2 tl = X.tiles[w / nch];
  const ItemRec it = X.items[tl.x];
  if (!it.rec) return false;
  out->item = tl.x;
  out->rowA = it.row0 + tl.y;
  out->nrows = min(kPM, it.ntok - tl.y);
  out->n0 = (w % nch) * (KIND == kPGateUp ? 128 : kPN);
  out->slot = it.slot;
  out->shared = it.shared;
  out->rec = it.rec;
  return true;
}

template <int KIND>
__global__ void __launch_bounds__(kPThreads, 1) prefill_gemm_kernel(FfnArgs A, PrefillAux X,
                                                                   const __grid_constant__ CUtensorMap tm_a,
                                                                   const __grid_constant__ CUtensorMap tm_q_pool,
                                                                   const __grid_constant__ CUtensorMap tm_q_shared) {
  extern __shared__ __align__(1024) uint8_t dyn[];
  PHead& H = *reinterpret_cast<PHead*>(dyn);
  uint8_t* base = dyn + kPHeadBytes;
  {
    const uint32_t a = smem_u32(base);
    base += ((a + 1023u) & ~1023u) - a;
  }
  uint8_t* ringA = base;
  uint8_t* ringB = ringA + kPStages * kPAStage;
  uint8_t* ringI = ringB + kPStages * kPBStage;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = KIND == kPGateUp ? A.d : A.f;
  const int KC = K / kPK;
  const int nch = KIND == kPGateUp ? A.f / 128 : A.d / kPN;
  const int n_work = X.n_tiles[0] * nch;
  const int nb = K / kQBlock;  // scale blocks per B row

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPStages; ++s) {
      mbar_init(&H.a_full[s], 1);
      mbar_init(&H.b_full[s], kPConv);
      mbar_init(&H.ab_empty[s], 1);
    }
    for (int s = 0; s < kPIStages; ++s) {
      mbar_init(&H.i_full[s], 1);
      mbar_init(&H.i_empty[s], kPConv);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&H.acc_full[b], 1);
      mbar_init(&H.acc_empty[b], 4);
    }
    H.abort = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_a);
    prefetch_tmap(&tm_q_pool);
    prefetch_tmap(&tm_q_shared);
  }
  if (warp == kPMmaWarp) {
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
      int sa = 0, si = 0, issued = 0;
      uint32_t pa = 0, pi = 0;
      for (int w = blockIdx.x; w < n_work && !p_aborted(H); w += gridDim.x) {
        PWork wk;
        if (!work_at<KIND>(A, X, w, nch, &wk)) continue;
        const CUtensorMap* tq = wk.shared ? &tm_q_shared : &tm_q_pool;
        for (int kc = 0; kc < KC; ++kc) {
          if (!mbar_wait(&H.ab_empty[sa], pa ^ 1u) || !mbar_wait(&H.i_empty[si], pi ^ 1u)) {
            p_set_abort(H, A.status);
            break;
          }
          mbar_arrive_expect_tx(&H.a_full[sa], kPAStage);
          tma_load_2d(ringA + (size_t)sa * kPAStage, &tm_a, kc * kPK, wk.rowA, &H.a_full[sa]);
          mbar_arrive_expect_tx(&H.i_full[si], kPIStage);
          if (KIND == kPGateUp)
            tma_load_4d(ringI + (size_t)si * kPIStage, tq, kc * kPK, wk.n0, 0, wk.slot, &H.i_full[si]);
          else
            tma_load_3d(ringI + (size_t)si * kPIStage, tq, kc * kPK, wk.n0, wk.slot, &H.i_full[si]);
          ++issued;
          if (++sa == kPStages) { sa = 0; pa ^= 1u; }
          if (++si == kPIStages) { si = 0; pi ^= 1u; }
        }
      }
      if (p_aborted(H)) {  // no copy may still be landing in shared memory when the CTA exits
        for (int j = issued > kPStages ? issued - kPStages : 0; j < issued; ++j)
          mbar_wait(&H.a_full[j % kPStages], (j / kPStages) & 1);
        for (int j = issued > kPIStages ? issued - kPIStages : 0; j < issued; ++j)
          mbar_wait(&H.i_full[j % kPIStages], (j / kPIStages) & 1);
      }
    }
  } else if (warp >= 1 && warp <= kPConv) {
    // ---------------- converters ----------------
    const int ct = threadIdx.x - 32;  // 0..255
    const int rb = ct >> 2, c = ct & 3;
    int sb = 0, si = 0;
    uint32_t pb = 0, pi = 0;
    for (int w = blockIdx.x; w < n_work; w += gridDim.x) {
      PWork wk;
      if (!work_at<KIND>(A, X, w, nch, &wk)) continue;
      // scale rows of this thread's four B rows rb + 64 i
      const __half* srow[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = rb + 64 * i;
        if (KIND == kPGateUp)
          srow[i] = reinterpret_cast<const __half*>(wk.rec + (r < 128 ? A.o_gate_s : A.o_up_s)) +
                    (size_t)(wk.n0 + (r & 127)) * nb;
        else
          srow[i] = reinterpret_cast<const __half*>(wk.rec + A.o_down_s) + (size_t)(wk.n0 + r) * nb;
      }
      bool ok = true;
      for (int kc = 0; kc < KC; ++kc) {
        // this K step is one pair of blocks: 2 kc and 2 kc + 1
        __half s0[4], s1[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          s0[i] = srow[i][kc * 2];
          s1[i] = srow[i][kc * 2 + 1];
        }
        const bool w1 = mbar_wait(&H.i_full[si], pi), w2 = mbar_wait(&H.ab_empty[sb], pb ^ 1u);
        if (!__all_sync(0xFFFFFFFFu, w1 && w2 && !p_aborted(H))) {
          if (lane == 0) p_set_abort(H, A.status);
          ok = false;
          break;
        }
        const uint8_t* src = ringI + (size_t)si * kPIStage;
        uint8_t* dst = ringB + (size_t)sb * kPBStage;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = rb + 64 * i;
          // stored chunk c: codes 8c..8c+7 of both blocks -> K-major chunks c and 4 + c
          const uint4 q = *reinterpret_cast<const uint4*>(src + r * kPK + c * 16);
          uint4 lo, hi;
          codes_to_f16(q, __half2half2(s0[i]), __half2half2(s1[i]), &lo, &hi);
          // odd rows write their high chunk first, so that the 8 lanes of a store phase (two
          // rows) hit 8 distinct 16-byte bank groups
          const bool odd = (r & 1) != 0;
          const int ch_lo = c ^ (r & 7), ch_hi = (4 + c) ^ (r & 7);
          *reinterpret_cast<uint4*>(dst + r * 128 + ((odd ? ch_hi : ch_lo) << 4)) = odd ? hi : lo;
          *reinterpret_cast<uint4*>(dst + r * 128 + ((odd ? ch_lo : ch_hi) << 4)) = odd ? lo : hi;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&H.i_empty[si]);
          mbar_arrive(&H.b_full[sb]);
        }
        if (++sb == kPStages) { sb = 0; pb ^= 1u; }
        if (++si == kPIStages) { si = 0; pi ^= 1u; }
      }
      if (!ok) break;
    }
  } else if (warp == kPMmaWarp) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = f16_idesc(kPM, kPN);
      int s = 0, lt = 0;
      uint32_t p = 0;
      for (int w = blockIdx.x; w < n_work; w += gridDim.x) {
        PWork wk;
        if (!work_at<KIND>(A, X, w, nch, &wk)) continue;
        const int buf = lt & 1;
        if (!mbar_wait(&H.acc_empty[buf], ((lt >> 1) & 1) ^ 1u)) {
          p_set_abort(H, A.status);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)(buf * kPN);
        bool ok = true;
        for (int kc = 0; kc < KC; ++kc) {
          if (!mbar_wait(&H.a_full[s], p) || !mbar_wait(&H.b_full[s], p) || p_aborted(H)) {
            p_set_abort(H, A.status);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(ringA + (size_t)s * kPAStage), b_addr = smem_u32(ringB + (size_t)s * kPBStage);
#pragma unroll
          for (int k = 0; k < kPK / 16; ++k)
            umma_f16(d_tmem, sw128_desc(a_addr + k * 32), sw128_desc(b_addr + k * 32), idesc, (kc | k) != 0);
          umma_commit(&H.ab_empty[s]);
          if (++s == kPStages) { s = 0; p ^= 1u; }
        }
        if (!ok) break;
        umma_commit(&H.acc_full[buf]);
        ++lt;
      }
    }
  } else if (warp >= kPEpiWarp0) {
    // ---------------- epilogue ----------------
    const int q = warp & 3;  // TMEM lane quarter
    const int m = q * 32 + lane;
    int lt = 0;
    for (int w = blockIdx.x; w < n_work; w += gridDim.x) {
      PWork wk;
      if (!work_at<KIND>(A, X, w, nch, &wk)) continue;
      const int buf = lt & 1;
      const bool ok = mbar_wait(&H.acc_full[buf], (lt >> 1) & 1) && !p_aborted(H);
      if (!__all_sync(0xFFFFFFFFu, ok)) {
        if (lane == 0) p_set_abort(H, A.status);
        break;
      }
      tc_fence_after();
      const uint32_t t_row = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * kPN);
      const bool valid = m < wk.nrows;
      const int r = wk.rowA + m;
      if (KIND == kPGateUp) {
        const float xs = valid ? X.xunscale[X.row_tok[r]] : 0.0f;
        float mx = 0.0f;
        for (int ch = 0; ch < 128; ch += 16) {
          uint32_t gv[16], uv[16];
          tmem_ld16(t_row + ch, gv);
          tmem_ld16(t_row + 128 + ch, uv);
          tmem_ld_wait();
          float hv[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            hv[j] = silu(__uint_as_float(gv[j]) * xs) * (__uint_as_float(uv[j]) * xs);
            mx = fmaxf(mx, fabsf(hv[j]));
          }
          if (valid) {
            float4* dst = reinterpret_cast<float4*>(A.h + (size_t)r * A.f + wk.n0 + ch);
#pragma unroll
            for (int j = 0; j < 4; ++j) dst[j] = make_float4(hv[4 * j], hv[4 * j + 1], hv[4 * j + 2], hv[4 * j + 3]);
          }
        }
        if (valid) atomicMax(X.hmax + r, __float_as_uint(mx));
      } else {
        const float up = valid ? p_pow2f(X.hexp[r]) : 0.0f;
        for (int ch = 0; ch < kPN; ch += 16) {
          uint32_t v[16];
          tmem_ld16(t_row + ch, v);
          tmem_ld_wait();
          if (valid) {
            const size_t off = (size_t)r * A.d + wk.n0 + ch;
            if (A.ydt == 1) {
              float4* dst = reinterpret_cast<float4*>(static_cast<float*>(A.y) + off);
#pragma unroll
              for (int j = 0; j < 4; ++j)
                dst[j] = make_float4(__uint_as_float(v[4 * j]) * up, __uint_as_float(v[4 * j + 1]) * up,
                                     __uint_as_float(v[4 * j + 2]) * up, __uint_as_float(v[4 * j + 3]) * up);
            } else {
              uint32_t o[8];
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const __nv_bfloat162 b2 =
                    __floats2bfloat162_rn(__uint_as_float(v[2 * j]) * up, __uint_as_float(v[2 * j + 1]) * up);
                o[j] = *reinterpret_cast<const uint32_t*>(&b2);
              }
              uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(A.y) + off);
              dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
              dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&H.acc_empty[buf]);
      ++lt;
    }
  }
  // Every role ends here. The MMA thread's last commit has been waited for by the epilogue, or
  // the work was abandoned; wait (bounded) for the tensor core to finish before freeing TMEM.
  tc_fence_before();
  __syncthreads();
  if (warp == kPMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------ host side ------------

namespace {

PFN_cuTensorMapEncodeTiled_v12000 p_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool p_encode(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base, const cuuint64_t* dims,
              const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle sw) {
  const cuuint32_t es[5] = {1, 1, 1, 1, 1};
  return p_encode_fn()(m, dt, rank, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A operand: rows x K f16, boxes of 64 x 128 in the 128-byte swizzle.
bool encode_a(CUtensorMap* m, const void* base, int K, int rows) {
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  const cuuint32_t box[2] = {kPK, kPM};
  return p_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// Codes of the gate/up matrices of n records: (K byte, row, gate|up, slot), boxes 64 x 128 x 2.
bool encode_q_gu(CUtensorMap* m, const uint8_t* recs, uint64_t n, const FfnArgs& a, uint64_t slot_bytes) {
  const cuuint64_t dims[4] = {(cuuint64_t)a.d, (cuuint64_t)a.f, 2, n};
  const cuuint64_t strides[3] = {(cuuint64_t)a.d, (cuuint64_t)(a.o_up_q - a.o_gate_q), slot_bytes};
  const cuuint32_t box[4] = {kPK, 128, 2, 1};
  return p_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, recs + a.o_gate_q, dims, strides, box,
                  CU_TENSOR_MAP_SWIZZLE_NONE);
}

// Codes of the down matrix of n records: (K byte, row, slot), boxes 64 x 256.
bool encode_q_dn(CUtensorMap* m, const uint8_t* recs, uint64_t n, const FfnArgs& a, uint64_t slot_bytes) {
  const cuuint64_t dims[3] = {(cuuint64_t)a.f, (cuuint64_t)a.d, n};
  const cuuint64_t strides[2] = {(cuuint64_t)a.f, slot_bytes};
  const cuuint32_t box[3] = {kPK, kPN, 1};
  return p_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, recs + a.o_down_q, dims, strides, box,
                  CU_TENSOR_MAP_SWIZZLE_NONE);
}

}  // namespace

bool prefill_supported(const FfnArgs& a) {
  return a.xdt == 0 && a.d % kPN == 0 && a.f % 128 == 0 && p_encode_fn() != nullptr;
}

cudaError_t launch_ffn_prefill(const FfnArgs& a, const PrefillAux& x, const void* pool, const void* shared,
                               uint64_t n_slots, uint64_t slot_bytes, int sm_count, cudaStream_t st) {
  const int rows = a.P + a.T * a.n_shared;
  if (rows == 0) return cudaSuccess;
  CUtensorMap tm_x, tm_h, qgu_pool, qgu_sh, qdn_pool, qdn_sh;
  const uint8_t* pl = static_cast<const uint8_t*>(pool);
  const uint8_t* sh = a.n_shared > 0 ? static_cast<const uint8_t*>(shared) : pl;
  const uint64_t nsh = a.n_shared > 0 ? (uint64_t)a.n_shared : 1;
  if (!encode_a(&tm_x, x.xp16, a.d, rows) || !encode_a(&tm_h, x.h16, a.f, rows) ||
      !encode_q_gu(&qgu_pool, pl, n_slots, a, slot_bytes) || !encode_q_gu(&qgu_sh, sh, nsh, a, slot_bytes) ||
      !encode_q_dn(&qdn_pool, pl, n_slots, a, slot_bytes) || !encode_q_dn(&qdn_sh, sh, nsh, a, slot_bytes))
    return cudaErrorInvalidValue;
  prefill_prepare_kernel<<<a.T, 256, 0, st>>>(a, x);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int grid_rows = sm_count * 8;
  prefill_gather_kernel<<<grid_rows, 256, 0, st>>>(a, x);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  auto gu = prefill_gemm_kernel<kPGateUp>;
  auto dn = prefill_gemm_kernel<kPDown>;
  if ((e = ensure_dynamic_smem(reinterpret_cast<const void*>(gu), kPSmem)) != cudaSuccess) return e;
  if ((e = ensure_dynamic_smem(reinterpret_cast<const void*>(dn), kPSmem)) != cudaSuccess) return e;
  gu<<<sm_count, kPThreads, kPSmem, st>>>(a, x, tm_x, qgu_pool, qgu_sh);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  prefill_convert_h_kernel<<<grid_rows, 256, 0, st>>>(a, x);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  dn<<<sm_count, kPThreads, kPSmem, st>>>(a, x, tm_h, qdn_pool, qdn_sh);
  return cudaGetLastError();
}

}  // namespace moe
