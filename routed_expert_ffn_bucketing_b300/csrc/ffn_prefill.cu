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
// specialised, with three shared-memory rings, each with its own full and empty barriers: A (4
// stages of 16 KB, filled by TMA), the int8 codes of B (4 stages of 16 KB, filled by TMA) and the
// converted f16 B tile (3 stages of 32 KB). The codes come by TMA rather than by per-thread loads
// into registers: such loads land through L1, and with ~160 KB of shared memory taken the L1
// left over bounds how many of them are in flight (measured: 48 KB of unused shared memory more
// made the FFN 1.34x slower), while TMA copies bypass it and the ring sets the prefetch depth.
//   warp 0, lane 0: TMA of the A tile of each 64-element K step (one pair of 32-element
//            blocks): 128 rows x 128 bytes of f16 in the 128-byte swizzle; freed by the MMA.
//   warp 10, lane 0: TMA of the codes of each K step: 256 B rows x 64 bytes; freed by the
//            converters once they hold them in registers.
//   warps 1..8: converters. Each thread owns 4 B rows and one 16-byte chunk of each row's 64
//            stored codes per K step (chunk c holds codes 8c..8c+7 of both blocks of the pair),
//            with the blocks' fp16 scales loaded from the expert record two pairs of K steps
//            ahead. It turns them into f16 (q * s, one rounding) and writes them into the B tile
//            in the 128-byte-swizzled K-major layout the tensor core reads, then fences them
//            into the async proxy. The int8 codes stay exact until this single rounding.
//   warp 9, lane 0: issues 4 tcgen05.mma (M = 128, N = 256, K = 16) per K step into one of two
//            TMEM accumulators (2 x 256 columns) and commits each stage back to the A and B rings.
//   warps 12..15: epilogue. TMEM lanes 32 q .. 32 q + 31 (q = warp % 4) hold rows of the tile;
//            tcgen05.ld 16 columns at a time while the next tile accumulates in the other buffer.
// Activations enter as f16 exactly (bf16 has 8 significant bits; each row is rescaled by a power
// of two that puts its max |x| in [2^14, 2^15)), and h is rescaled per row the same way.
//
// Every wait is bounded. A wait that runs out sets MOE_DEV_TIMEOUT and the CTA stops its work;
// every role still reaches the final barrier, so the TMEM columns are always freed. Before
// that, the A producer waits for its TMA copies still in flight and the MMA thread for its
// last tcgen05.mma (a final commit to the drain barrier), with the default limit.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "moe_common.cuh"
#include "sm100_ptx.cuh"
#include "tmap.h"

namespace moe {

constexpr int kPM = 128;                     // rows per M tile (UMMA M)
constexpr int kPN = 256;                     // UMMA N
constexpr int kPK = 64;                      // K elements per stage (128 bytes of f16)
constexpr int kPAStage = kPM * 128;          // 16 KB
constexpr int kPBStage = kPN * 128;          // 32 KB
constexpr int kPQStage = kPN * kPK;          // 16 KB: int8 codes of one K step of the 256 B rows
constexpr int kPAStages = 4;                 // A ring (TMA; freed by the MMA)
constexpr int kPBStages = 3;                 // f16 B ring (converters; freed by the MMA)
constexpr int kPQStages = 4;                 // int8 code ring (TMA; freed by the converters)
constexpr int kPConv = 8;                    // converter warps
constexpr int kPThreads = 32 * 16;           // 0: A TMA, 1..8: convert, 9: MMA, 10: code TMA, 12..15: epilogue
constexpr int kPMmaWarp = 9;
constexpr int kPQWarp = 10;
constexpr int kPEpiWarp0 = 12;
constexpr int kPPairsAhead = 2;              // pairs of K steps of scales a converter holds in registers

enum { kPGateUp = 0, kPDown = 1 };

struct PHead {
  uint64_t a_full[kPAStages];
  uint64_t a_empty[kPAStages];
  uint64_t b_full[kPBStages];
  uint64_t b_empty[kPBStages];
  uint64_t q_full[kPQStages];
  uint64_t q_empty[kPQStages];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t drain;  // the MMA thread's last commit: every MMA it issued has completed
  uint32_t tmem;
  int abort;
};
constexpr size_t kPHeadBytes = 1024;
static_assert(sizeof(PHead) <= kPHeadBytes, "head too large");
constexpr size_t kPSmem = kPHeadBytes + 1024 + (size_t)kPAStages * kPAStage + (size_t)kPBStages * kPBStage +
                          (size_t)kPQStages * kPQStage;
static_assert(kPSmem <= 232448, "shared memory of the GEMM above the per-block limit");

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

// Loads issued where they stand: the converters' prefetch only hides memory latency if the
// compiler does not sink these loads down to the first use of their registers.
__device__ __forceinline__ uint2 p_ld_scales(const void* p) {
  uint2 r;
  asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}

// The four fp16 scales (two K steps, two blocks each) of one converter thread's four B rows for
// one pair of K steps, one 8-byte word per row.
struct PScales {
  uint2 s[4];
};

// A cursor over the CTA's sequence of (work item, pair of K steps), in the order the MMA consumes
// them; it loads one thread's PScales straight from the expert record (global memory).
template <int KIND>
struct PCursor {
  const __half* srow[4];
  int w, kc;

  __device__ __forceinline__ void seek(const FfnArgs& A, const PrefillAux& X, int w0, int nch, int n_work, int rb,
                                       int K) {
    const int nb = K / kQBlock;
    for (w = w0; w < n_work; w += gridDim.x) {
      PWork wk;
      if (!work_at<KIND>(A, X, w, nch, &wk)) continue;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = rb + 64 * i;
        const int n = KIND == kPGateUp ? wk.n0 + (r & 127) : wk.n0 + r;
        const uint64_t os = KIND == kPGateUp ? (r < 128 ? A.o_gate_s : A.o_up_s) : A.o_down_s;
        srow[i] = reinterpret_cast<const __half*>(wk.rec + os) + (size_t)n * nb;
      }
      kc = 0;
      return;
    }
  }

  // Loads the scales of the pair at the cursor and moves one pair forward; false past the CTA's
  // last work.
  __device__ __forceinline__ bool next(const FfnArgs& A, const PrefillAux& X, int nch, int n_work, int rb, int K,
                                       PScales& p) {
    if (w >= n_work) return false;
#pragma unroll
    for (int i = 0; i < 4; ++i) p.s[i] = p_ld_scales(srow[i] + kc * 2);
    kc += 2;
    if (kc * kPK >= K) seek(A, X, w + gridDim.x, nch, n_work, rb, K);
    return true;
  }
};

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
  uint8_t* ringB = ringA + kPAStages * kPAStage;
  uint8_t* ringQ = ringB + kPBStages * kPBStage;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = KIND == kPGateUp ? A.d : A.f;
  const int KC = K / kPK;
  const int nch = KIND == kPGateUp ? A.f / 128 : A.d / kPN;
  const int n_work = X.n_tiles[0] * nch;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPAStages; ++s) {
      mbar_init(&H.a_full[s], 1);
      mbar_init(&H.a_empty[s], 1);
    }
    for (int s = 0; s < kPBStages; ++s) {
      mbar_init(&H.b_full[s], kPConv);
      mbar_init(&H.b_empty[s], 1);
    }
    for (int s = 0; s < kPQStages; ++s) {
      mbar_init(&H.q_full[s], 1);
      mbar_init(&H.q_empty[s], kPConv);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&H.acc_full[b], 1);
      mbar_init(&H.acc_empty[b], 4);
    }
    mbar_init(&H.drain, 1);
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
    // ---------------- TMA producer of the A tiles ----------------
    if (lane == 0) {
      int s = 0, issued = 0;
      uint32_t ph = 0;
      for (int w = blockIdx.x; w < n_work && !p_aborted(H); w += gridDim.x) {
        PWork wk;
        if (!work_at<KIND>(A, X, w, nch, &wk)) continue;
        for (int kc = 0; kc < KC; ++kc) {
          if (!mbar_wait(&H.a_empty[s], ph ^ 1u, A.wait_ns)) {
            p_set_abort(H, A.status);
            break;
          }
          mbar_arrive_expect_tx(&H.a_full[s], kPAStage);
          tma_load_2d(ringA + (size_t)s * kPAStage, &tm_a, kc * kPK, wk.rowA, &H.a_full[s]);
          ++issued;
          if (++s == kPAStages) { s = 0; ph ^= 1u; }
        }
      }
      if (p_aborted(H))  // no copy may still be landing in shared memory when the CTA exits
        for (int j = issued > kPAStages ? issued - kPAStages : 0; j < issued; ++j)
          mbar_wait(&H.a_full[j % kPAStages], (j / kPAStages) & 1);  // default limit

    }
  } else if (warp >= 1 && warp <= kPConv) {
    // ---------------- converters ----------------
    // Thread ct owns B rows rb + 64 i (i < 4) and 16-byte chunk c of each row's 64 stored codes
    // per K step (chunk c holds codes 8c..8c+7 of both blocks of the pair). The codes arrive by
    // TMA in the int8 ring; the blocks' fp16 scales come straight from the expert record,
    // kPPairsAhead pairs of K steps ahead, into registers.
    const int ct = threadIdx.x - 32;  // 0..255
    const int rb = ct >> 2, c = ct & 3;
    int sb = 0, sq = 0;
    uint32_t pb = 0, pq = 0;
    PCursor<KIND> cur;
    cur.seek(A, X, blockIdx.x, nch, n_work, rb, K);
    PScales ps[kPPairsAhead];
    bool have[kPPairsAhead];
#pragma unroll
    for (int j = 0; j < kPPairsAhead; ++j) have[j] = cur.next(A, X, nch, n_work, rb, K, ps[j]);
    bool ok = true;
    while (ok && have[0]) {
#pragma unroll
      for (int j = 0; j < kPPairsAhead; ++j) {
        if (!have[j]) break;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const bool w1 = mbar_wait(&H.q_full[sq], pq, A.wait_ns);
          const bool w2 = w1 && mbar_wait(&H.b_empty[sb], pb ^ 1u, A.wait_ns);
          if (!__all_sync(0xFFFFFFFFu, w2 && !p_aborted(H))) {
            if (lane == 0) p_set_abort(H, A.status);
            ok = false;
            break;
          }
          const uint8_t* src = ringQ + (size_t)sq * kPQStage;
          uint4 lo[4], hi[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int r = rb + 64 * i;
            // this K step is one pair of blocks; their scales are the low and high half of one
            // 32-bit word of the pair of K steps' scales
            const uint32_t sw = h ? ps[j].s[i].y : ps[j].s[i].x;
            const __half2 s01 = *reinterpret_cast<const __half2*>(&sw);
            const uint4 q = *reinterpret_cast<const uint4*>(src + r * kPK + c * 16);
            codes_to_f16(q, __low2half2(s01), __high2half2(s01), &lo[i], &hi[i]);
          }
          // every lane has its codes in registers: the code stage goes back to the TMA
          __syncwarp();
          if (lane == 0) mbar_arrive(&H.q_empty[sq]);
          uint8_t* dst = ringB + (size_t)sb * kPBStage;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int r = rb + 64 * i;
            // stored chunk c -> K-major chunks c and 4 + c; odd rows write their high chunk
            // first, so that the 8 lanes of a store phase (two rows) hit 8 distinct 16-byte
            // bank groups
            const bool odd = (r & 1) != 0;
            const int ch_lo = c ^ (r & 7), ch_hi = (4 + c) ^ (r & 7);
            *reinterpret_cast<uint4*>(dst + r * 128 + ((odd ? ch_hi : ch_lo) << 4)) = odd ? hi[i] : lo[i];
            *reinterpret_cast<uint4*>(dst + r * 128 + ((odd ? ch_lo : ch_hi) << 4)) = odd ? lo[i] : hi[i];
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&H.b_full[sb]);
          if (++sb == kPBStages) { sb = 0; pb ^= 1u; }
          if (++sq == kPQStages) { sq = 0; pq ^= 1u; }
        }
        if (!ok) break;
        have[j] = cur.next(A, X, nch, n_work, rb, K, ps[j]);
      }
    }
  } else if (warp == kPQWarp) {
    // ---------------- TMA producer of the int8 code tiles ----------------
    // One K step of the work item's 256 B rows: gate rows n0..n0+127 then the same up rows (one
    // 4-D box), or down rows n0..n0+255 (one 3-D box); 64 bytes per row, rows back to back.
    if (lane == 0) {
      int s = 0, issued = 0;
      uint32_t ph = 0;
      for (int w = blockIdx.x; w < n_work && !p_aborted(H); w += gridDim.x) {
        PWork wk;
        if (!work_at<KIND>(A, X, w, nch, &wk)) continue;
        const CUtensorMap* tq = wk.shared ? &tm_q_shared : &tm_q_pool;
        for (int kc = 0; kc < KC; ++kc) {
          if (!mbar_wait(&H.q_empty[s], ph ^ 1u, A.wait_ns)) {
            p_set_abort(H, A.status);
            break;
          }
          mbar_arrive_expect_tx(&H.q_full[s], kPQStage);
          if (KIND == kPGateUp)
            tma_load_4d(ringQ + (size_t)s * kPQStage, tq, kc * kPK, wk.n0, 0, wk.slot, &H.q_full[s]);
          else
            tma_load_3d(ringQ + (size_t)s * kPQStage, tq, kc * kPK, wk.n0, wk.slot, &H.q_full[s]);
          ++issued;
          if (++s == kPQStages) { s = 0; ph ^= 1u; }
        }
      }
      if (p_aborted(H))  // no copy may still be landing in shared memory when the CTA exits
        for (int j = issued > kPQStages ? issued - kPQStages : 0; j < issued; ++j)
          mbar_wait(&H.q_full[j % kPQStages], (j / kPQStages) & 1);  // default limit
    }
  } else if (warp == kPMmaWarp) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = f16_idesc(kPM, kPN);
      int sa = 0, sb = 0, lt = 0;
      uint32_t pa = 0, pb = 0;
      for (int w = blockIdx.x; w < n_work; w += gridDim.x) {
        PWork wk;
        if (!work_at<KIND>(A, X, w, nch, &wk)) continue;
        const int buf = lt & 1;
        if (!mbar_wait(&H.acc_empty[buf], ((lt >> 1) & 1) ^ 1u, A.wait_ns)) {
          p_set_abort(H, A.status);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)(buf * kPN);
        bool ok = true;
        for (int kc = 0; kc < KC; ++kc) {
          if (!mbar_wait(&H.a_full[sa], pa, A.wait_ns) || !mbar_wait(&H.b_full[sb], pb, A.wait_ns) ||
              p_aborted(H)) {
            p_set_abort(H, A.status);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(ringA + (size_t)sa * kPAStage);
          const uint32_t b_addr = smem_u32(ringB + (size_t)sb * kPBStage);
#pragma unroll
          for (int k = 0; k < kPK / 16; ++k)
            umma_f16(d_tmem, sw128_desc(a_addr + k * 32), sw128_desc(b_addr + k * 32), idesc, (kc | k) != 0);
          umma_commit(&H.a_empty[sa]);
          umma_commit(&H.b_empty[sb]);
          if (++sa == kPAStages) { sa = 0; pa ^= 1u; }
          if (++sb == kPBStages) { sb = 0; pb ^= 1u; }
        }
        if (!ok) break;
        umma_commit(&H.acc_full[buf]);
        ++lt;
      }
      // Drain: one more commit arrives once every MMA this thread issued has completed,
      // including those left queued when a wait above ran out. TMEM and the rings are freed
      // only after it (waited for with the default limit, not the caller's shorter one).
      umma_commit(&H.drain);
      mbar_wait(&H.drain, 0);
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
      const bool ok = mbar_wait(&H.acc_full[buf], (lt >> 1) & 1, A.wait_ns) && !p_aborted(H);
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
            hv[j] = silu_fast(__uint_as_float(gv[j]) * xs) * (__uint_as_float(uv[j]) * xs);
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
  // Every role ends here. The MMA thread has waited for its drain commit, so no MMA is still
  // reading the rings or writing TMEM, and the A producer has waited for its copies in flight.
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

// A operand: rows x K f16, boxes of 64 x 128 in the 128-byte swizzle.
bool encode_a(CUtensorMap* m, const void* base, int K, int rows) {
  return tmap_encode_2d(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, base, (uint64_t)K, (uint64_t)rows, (uint64_t)K * 2, kPK,
                        kPM, CU_TENSOR_MAP_SWIZZLE_128B);
}

// Codes of the gate/up matrices of n records: (K byte, row, gate|up, record), boxes 64 x 128 x 2.
bool encode_q_gu(CUtensorMap* m, const uint8_t* recs, uint64_t n, const FfnArgs& a) {
  const cuuint64_t dims[4] = {(cuuint64_t)a.d, (cuuint64_t)a.f, 2, n};
  const cuuint64_t strides[3] = {(cuuint64_t)a.d, (cuuint64_t)(a.o_up_q - a.o_gate_q), a.slot_bytes};
  const cuuint32_t box[4] = {kPK, 128, 2, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return p_encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<uint8_t*>(recs + a.o_gate_q), dims, strides,
                       box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Codes of the down matrix of n records: (K byte, row, record), boxes 64 x 256.
bool encode_q_dn(CUtensorMap* m, const uint8_t* recs, uint64_t n, const FfnArgs& a) {
  const cuuint64_t dims[3] = {(cuuint64_t)a.f, (cuuint64_t)a.d, n};
  const cuuint64_t strides[2] = {(cuuint64_t)a.f, a.slot_bytes};
  const cuuint32_t box[3] = {kPK, kPN, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return p_encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(recs + a.o_down_q), dims, strides,
                       box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool tmap_available() { return p_encode_fn() != nullptr; }

bool tmap_encode_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t rows,
                    uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle sw) {
  if (!p_encode_fn()) return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t es[2] = {1, 1};
  return p_encode_fn()(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool prefill_supported(const FfnArgs& a) {
  return a.xdt == 0 && a.d % kPN == 0 && a.f % 128 == 0 && tmap_available();
}

cudaError_t launch_ffn_prefill(const FfnArgs& a, const PrefillAux& x, int sm_count, cudaStream_t st) {
  const int rows = a.P + a.T * a.n_shared;
  if (rows == 0) return cudaSuccess;
  // the shared experts' records follow one another at the pool's record stride
  CUtensorMap tm_x, tm_h, qgu_pool, qgu_sh, qdn_pool, qdn_sh;
  const uint8_t* sh = a.n_shared > 0 ? a.shared : a.pool;
  const uint64_t nsh = a.n_shared > 0 ? (uint64_t)a.n_shared : 1;
  if (!encode_a(&tm_x, x.xp16, a.d, rows) || !encode_a(&tm_h, x.h16, a.f, rows) ||
      !encode_q_gu(&qgu_pool, a.pool, a.n_slots, a) || !encode_q_gu(&qgu_sh, sh, nsh, a) ||
      !encode_q_dn(&qdn_pool, a.pool, a.n_slots, a) || !encode_q_dn(&qdn_sh, sh, nsh, a))
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
