// Expert FFN for many tokens per expert (prefill): a grouped GEMM on the tcgen05 tensor cores.
//
// Prefill runs long prompts through the layer in chunks of up to 8192 tokens ("Strata 工作原理图解
// GPU内存SSD三级存储如何让125B模型塞进消费级显卡", section "长文本"), and its expert matmuls run on
// the tensor cores without a separate dequantisation pass ("Strata 性能基准与论文导读125B MoE在
// 消费级硬件上的极限测量与瓶颈分析", section "瓶颈分析 1️⃣"). Kernels:
//   prepare: per-token power-of-two scale of x, the work-item table, the token of every row,
//            cleared max |h| per row, and the list of token tiles (up to 128 rows) of every item;
//   gather:  xp16[r] = f16(x[token of r] * 2^-e): the rows of every expert contiguous;
//   gemm<GU>: for each (token tile, 64 columns of f): D[128][N] = W[128][d] . X[N][d]^T with W
//            rows 2i and 2i + 1 the gate and the up row of column i, N the tile's rows rounded up
//            to 16, then h = silu(g) * u (fp32) and a max |h| per row;
//   convert: h16[r] = f16(h[r] * 2^-e_r) with e_r from max |h| of the row;
//   gemm<DN>: for each (token tile, 128 rows of d): D[128][N] = Wd[128][f] . h16[N][f]^T.
//
// The weights are the MMA's A operand and sit in tensor memory; the token rows are B, in shared
// memory. Converted weights thus never pass through shared memory: per K step of 64 it carries
// the token tile (TMA write, one MMA read) and the int8 codes (TMA write, one converter read),
// 48 KB for a 128-row tile, where a layout with the weights as a shared-memory operand also
// writes and reads their f16 copy. And N follows the tile's rows, so an expert with a few
// tokens costs a few columns of MMA work, not a 128-row tile.
//
// K order. An expert record stores each 64-element K step of a row as four 16-byte chunks,
// chunk c holding elements 8c..8c+7 of the step's first 32-element block and then the same of
// its second block (the layout the decode kernels load as MMA fragments). The GEMMs keep that
// order: A column pair p of a K step holds stored bytes 2p and 2p + 1, and xp16 and h16 store
// each K step of their rows in the same permuted order (a dot product does not depend on the
// order of its terms; every K step of A and B uses the same one).
//
// The GEMM is persistent (one CTA per SM, a static stride over the work list) and warp
// specialised. A stage holds two K steps (K = 128). Rings, stage s of each carrying the same K
// range: the token tile X (4 stages of up to 32 KB in shared memory, TMA, boxes of 32 rows), the
// int8 codes (4 stages of 16 KB in shared memory, TMA, 128-byte swizzle) and the converted f16
// weights (4 stages of 64 tensor-memory columns). Two fp32 accumulators of 128 columns in
// tensor memory let the epilogue of one tile overlap the next tile's MMAs. A tcgen05.mma costs
// its issuing thread about 50 cycles and an mbarrier test about 90 even when the phase has
// completed, so a stage carries 8 MMAs per pair of barrier tests and one commit (with K = 64
// stages that thread's overhead rather than the tensor core set the pace: measured 730 cycles
// per K step with every operand ready thousands of cycles early).
//   warp 0, lane 0: TMA of the token tile of each stage (N rows x 2 x 128 bytes, 128-byte swizzle).
//   warp 10, lane 0: TMA of the 128 weight rows' codes of each stage (128 bytes per row).
//   warps 1..8: converters. Thread (warp w, lane l) owns weight row 32 (w % 4) + l (the
//            tensor-memory lane its warp may access) and one K step of each stage (warps 1..4
//            the first, 5..8 the second): it reads the row's 64 stored codes, with the pair's
//            two fp16 scales loaded from the expert record a few stages ahead, turns them into
//            f16 (q * s, one rounding; the codes stay exact until then) and writes 32 columns
//            of its lane with tcgen05.st.
//   warp 9: the MMA issuer (one elected lane issues): 8 tcgen05.mma (M = 128, N, K = 16; A from
//            tensor memory) per stage, the commit that frees the stage's X and A slots, and the
//            one that hands a finished accumulator to the epilogue.
//   warps 12..15: epilogue. Tensor-memory lanes 32 q .. 32 q + 31 (q = warp % 4) are weight
//            rows; tcgen05.ld 16 token columns at a time, the next load in flight while the
//            current columns are processed.
// Activations enter as f16 exactly (bf16 has 8 significant bits; each row is rescaled by a power
// of two that puts its max |x| in [2^14, 2^15)), and h is rescaled per row the same way.
//
// Every wait is bounded. A wait that runs out sets MOE_DEV_TIMEOUT and the CTA stops its work;
// every role still reaches the final barrier, so the tensor-memory columns are always freed.
// Before that, the TMA producers wait for their copies still in flight and the MMA thread for
// its last tcgen05.mma (a final commit to the drain barrier), with the default limit.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "moe_common.cuh"
#include "sm100_ptx.cuh"
#include "tmap.h"

namespace moe {

constexpr int kPM = 128;                     // token rows per tile (the largest UMMA N used)
constexpr int kPW = 128;                     // weight rows per tile (UMMA M)
constexpr int kPK = 64;                      // K elements per K step (one pair of blocks; 128 bytes of f16)
constexpr int kPKS = 2 * kPK;                // K elements per stage: two K steps
constexpr int kPBox = 32;                    // token rows per TMA box of the X tile
constexpr int kPXHalf = kPM * 128;           // 16 KB: the X rows of one K step
constexpr int kPXStage = 2 * kPXHalf;        // 32 KB
constexpr int kPQStage = kPW * kPKS;         // 16 KB: int8 codes of one stage of the 128 weight rows
constexpr int kPXStages = 4;                 // X ring (TMA; freed by the MMA together with the A stage)
constexpr int kPQStages = 4;                 // int8 code ring (TMA; freed by the converters)
constexpr int kPAStages = 4;                 // f16 weight ring in tensor memory (converters; freed by the MMA)
constexpr int kPAcc = 128;                   // tensor-memory columns per accumulator
constexpr uint32_t kPACol0 = 2 * kPAcc;      // first column of the weight ring (64 columns per stage)
constexpr int kPConv = 8;                    // converter warps
constexpr int kPThreads = 32 * 16;           // 0: X TMA, 1..8: convert, 9: MMA, 10: code TMA, 12..15: epilogue
constexpr int kPMmaWarp = 9;
constexpr int kPQWarp = 10;
constexpr int kPEpiWarp0 = 12;
constexpr int kPPairsAhead = 3;              // stages of scales a converter holds in registers

enum { kPGateUp = 0, kPDown = 1 };

// Stage s of the X, A and code rings carries the same K range: x_full (the TMA) and a_full (the
// converters) fill the X and A stages, and one MMA commit to xa_empty frees both.
struct PHead {
  uint64_t x_full[kPXStages];
  uint64_t a_full[kPAStages];
  uint64_t xa_empty[kPAStages];
  uint64_t q_full[kPQStages];
  uint64_t q_empty[kPQStages];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t drain;  // the MMA warp's last commit: every MMA it issued has completed
  uint32_t tmem;
  int abort;
  int epi_ok[2];
};
constexpr size_t kPHeadBytes = 1024;
static_assert(sizeof(PHead) <= kPHeadBytes, "head too large");
// epilogue scratch: a per-column scale and the four lane quarters' column maxima, two buffers
constexpr size_t kPEpiBytes = sizeof(float) * 2 * (kPM + 4 * kPM);
constexpr size_t kPSmem = kPHeadBytes + 1024 + (size_t)kPXStages * kPXStage + (size_t)kPQStages * kPQStage + kPEpiBytes;
static_assert(kPSmem <= 232448, "shared memory of the GEMM above the per-block limit");
static_assert(kPACol0 + kPAStages * 64 <= 512, "tensor-memory columns");
static_assert(kPAStages == kPQStages && kPAStages == kPXStages, "one stage index for the X, A and code rings");

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
// swizzle: 8-row atoms of 1024 bytes stacked along N (stride 1024), descriptor version 1.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// kind::f16 instruction descriptor: fp32 accumulator, f16 A and B, both K-major, N and M.
__host__ __device__ constexpr uint32_t f16_idesc(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Position of logical element k (0..63) of a K step in the stored order: chunk (k % 32) / 8,
// then the block k / 32, then k % 8.
__host__ __device__ __forceinline__ int stored_pos(int k) { return ((k & 31) >> 3) * 16 + (k >> 5) * 8 + (k & 7); }

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
// and the token-tile list (tiles of up to 128 rows, in item order, then by row).
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

// xp16[r][:] = f16(x[token of r][:] * 2^-e): 8 elements per thread, each K step of 64 in the
// stored order (8 consecutive elements stay together).
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
    const int cs = (c & ~63) + stored_pos(c & 63);
    *reinterpret_cast<uint4*>(X.xp16 + (size_t)r * d + cs) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// h16[r] = f16(h[r] * 2^-e_r), hexp[r] = e_r, with e_r from max |h| of row r: 8 per thread, in
// the stored order like xp16.
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
    const int cs = (c & ~63) + stored_pos(c & 63);
    *reinterpret_cast<uint4*>(X.h16 + (size_t)r * f + cs) =
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

// Work w: token tile w / nch, weight chunk w % nch (64 columns of f for gate/up, 128 rows of d
// for down).
template <int KIND>
__device__ __forceinline__ bool work_at(const FfnArgs& A, const PrefillAux& X, int w, int nch, PWork* out) {
  const int2 tl = X.tiles[w / nch];
  const ItemRec it = X.items[tl.x];
  if (!it.rec) return false;
  out->item = tl.x;
  out->rowA = it.row0 + tl.y;
  out->nrows = min(kPM, it.ntok - tl.y);
  out->n0 = (w % nch) * (KIND == kPGateUp ? kPW / 2 : kPW);
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

// A cursor over the CTA's sequence of (work item, pair of K steps), in the order the MMA consumes
// them; it loads the fp16 scales of one weight row for a pair of K steps (blocks 4p .. 4p + 3, one
// 8-byte word) straight from the expert record.
template <int KIND>
struct PCursor {
  const uint32_t* srow;  // the row's scales as 32-bit words: word kc = the two blocks of K step kc
  int w, kc;

  __device__ __forceinline__ void seek(const FfnArgs& A, const PrefillAux& X, int w0, int nch, int n_work, int L,
                                       int K) {
    const int nb = K / kQBlock;
    for (w = w0; w < n_work; w += gridDim.x) {
      PWork wk;
      if (!work_at<KIND>(A, X, w, nch, &wk)) continue;
      uint64_t os;
      int row;
      if (KIND == kPGateUp) {
        os = (L & 1) ? A.o_up_s : A.o_gate_s;
        row = wk.n0 + (L >> 1);
      } else {
        os = A.o_down_s;
        row = wk.n0 + L;
      }
      srow = reinterpret_cast<const uint32_t*>(wk.rec + os + (size_t)row * nb * 2);
      kc = 0;
      return;
    }
  }

  // Loads the scales of the pair at the cursor and moves one pair forward; false past the CTA's
  // last work.
  __device__ __forceinline__ bool next(const FfnArgs& A, const PrefillAux& X, int nch, int n_work, int L, int K,
                                       uint2& p) {
    if (w >= n_work) return false;
    p = p_ld_scales(srow + kc);
    kc += 2;
    if (kc * kPK >= K) seek(A, X, w + gridDim.x, nch, n_work, L, K);
    return true;
  }
};

template <int KIND>
__global__ void __launch_bounds__(kPThreads, 1) prefill_gemm_kernel(FfnArgs A, PrefillAux X,
                                                                   const __grid_constant__ CUtensorMap tm_x,
                                                                   const __grid_constant__ CUtensorMap tm_q_pool,
                                                                   const __grid_constant__ CUtensorMap tm_q_shared) {
  extern __shared__ __align__(1024) uint8_t dyn[];
  PHead& H = *reinterpret_cast<PHead*>(dyn);
  uint8_t* base = dyn + kPHeadBytes;
  {
    const uint32_t a = smem_u32(base);
    base += ((a + 1023u) & ~1023u) - a;
  }
  uint8_t* ringX = base;
  uint8_t* ringQ = ringX + kPXStages * kPXStage;
  float* col_s = reinterpret_cast<float*>(ringQ + kPQStages * kPQStage);  // [2][kPM]
  float* hm_s = col_s + 2 * kPM;                                          // [2][4][kPM]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = KIND == kPGateUp ? A.d : A.f;
  const int KC = K / kPKS;  // stages per work item
  const int nch = KIND == kPGateUp ? A.f / (kPW / 2) : A.d / kPW;
  const int n_work = X.n_tiles[0] * nch;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPXStages; ++s) {
      mbar_init(&H.x_full[s], 1);
      mbar_init(&H.xa_empty[s], 1);
    }
    for (int s = 0; s < kPQStages; ++s) {
      mbar_init(&H.q_full[s], 1);
      mbar_init(&H.q_empty[s], kPConv);
    }
    for (int s = 0; s < kPAStages; ++s) mbar_init(&H.a_full[s], kPConv);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&H.acc_full[b], 1);
      mbar_init(&H.acc_empty[b], 4);
    }
    mbar_init(&H.drain, 1);
    H.abort = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_x);
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
    // ---------------- TMA producer of the token tiles ----------------
    if (lane == 0) {
      int s = 0, issued = 0;
      uint32_t ph = 0;
      for (int w = blockIdx.x; w < n_work && !p_aborted(H); w += gridDim.x) {
        PWork wk;
        if (!work_at<KIND>(A, X, w, nch, &wk)) continue;
        const int nbox = (wk.nrows + kPBox - 1) / kPBox;
        for (int kc = 0; kc < KC; ++kc) {
          if (!mbar_wait(&H.xa_empty[s], ph ^ 1u, A.wait_ns)) {
            p_set_abort(H, A.status);
            break;
          }
          mbar_arrive_expect_tx(&H.x_full[s], (uint32_t)(2 * nbox) * kPBox * 128);
          for (int hk = 0; hk < 2; ++hk)
            for (int j = 0; j < nbox; ++j)
              tma_load_2d(ringX + (size_t)s * kPXStage + hk * kPXHalf + j * kPBox * 128, &tm_x, kc * kPKS + hk * kPK,
                          wk.rowA + j * kPBox, &H.x_full[s]);
          ++issued;
          if (++s == kPXStages) { s = 0; ph ^= 1u; }
        }
      }
      if (p_aborted(H))  // no copy may still be landing in shared memory when the CTA exits
        for (int j = issued > kPXStages ? issued - kPXStages : 0; j < issued; ++j)
          mbar_wait(&H.x_full[j % kPXStages], (j / kPXStages) & 1);  // default limit
    }
  } else if (warp >= 1 && warp <= kPConv) {
    // ---------------- converters ----------------
    // Thread (warp, lane) owns weight row L = 32 (warp % 4) + lane, which is tensor-memory lane
    // L of the A stages, and K step hf = (warp - 1) / 4 of each stage (warps 1..4 the first,
    // 5..8 the second). The codes arrive by TMA in the 128-byte swizzle (chunk c of row R at
    // chunk c ^ (R % 8)); the blocks' fp16 scales come straight from the expert record,
    // kPPairsAhead stages ahead, into registers.
    const int q = warp & 3, L = q * 32 + lane, hf = (warp - 1) >> 2;
    const uint32_t t_lane = tmem + ((uint32_t)(q * 32) << 16) + kPACol0 + (uint32_t)(32 * hf);
    int s = 0;
    uint32_t ph = 0;
    PCursor<KIND> cur;
    cur.seek(A, X, blockIdx.x, nch, n_work, L, K);
    uint2 ps[kPPairsAhead];
    bool have[kPPairsAhead];
#pragma unroll
    for (int j = 0; j < kPPairsAhead; ++j) have[j] = cur.next(A, X, nch, n_work, L, K, ps[j]);
    bool ok = true;
    while (ok && have[0]) {
#pragma unroll
      for (int j = 0; j < kPPairsAhead; ++j) {
        if (!have[j]) break;
        const bool w1 = mbar_wait(&H.q_full[s], ph, A.wait_ns);
        const bool w2 = w1 && mbar_wait(&H.xa_empty[s], ph ^ 1u, A.wait_ns);
        if (!__all_sync(0xFFFFFFFFu, w2 && !p_aborted(H))) {
          if (lane == 0) p_set_abort(H, A.status);
          ok = false;
          break;
        }
        tc_fence_after();  // the MMAs that read this A stage have completed
        const uint8_t* src = ringQ + (size_t)s * kPQStage + L * kPKS;
        uint4 qc[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) qc[c] = *reinterpret_cast<const uint4*>(src + (((4 * hf + c) ^ (L & 7)) << 4));
        // every lane has its codes in registers: the code stage goes back to the TMA
        __syncwarp();
        if (lane == 0) mbar_arrive(&H.q_empty[s]);
        // this K step is one pair of blocks; their scales are the low and high half of one
        // 32-bit word of the stage's scales
        const uint32_t swd = hf ? ps[j].y : ps[j].x;
        const __half2 s01 = *reinterpret_cast<const __half2*>(&swd);
        uint32_t r[32];
#pragma unroll
        for (int c = 0; c < 4; ++c)
          codes_to_f16(qc[c], __low2half2(s01), __high2half2(s01), reinterpret_cast<uint4*>(r + 8 * c),
                       reinterpret_cast<uint4*>(r + 8 * c + 4));
        tmem_st16(t_lane + (uint32_t)(64 * s), r);
        tmem_st16(t_lane + (uint32_t)(64 * s + 16), r + 16);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&H.a_full[s]);
        if (++s == kPAStages) { s = 0; ph ^= 1u; }
        have[j] = cur.next(A, X, nch, n_work, L, K, ps[j]);
      }
    }
  } else if (warp == kPQWarp) {
    // ---------------- TMA producer of the int8 code tiles ----------------
    // One K step of the work item's 128 weight rows, 64 bytes per row: gate and up row of
    // columns n0..n0+63 interleaved (one 4-D box), or down rows n0..n0+127 (one 3-D box).
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
            tma_load_4d(ringQ + (size_t)s * kPQStage, tq, kc * kPKS, 0, wk.n0, wk.slot, &H.q_full[s]);
          else
            tma_load_3d(ringQ + (size_t)s * kPQStage, tq, kc * kPKS, wk.n0, wk.slot, &H.q_full[s]);
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
    // The whole warp runs the loop, so that its control values and descriptors stay warp
    // uniform (uniform registers, no per-instruction moves into them); lane 0 issues every MMA
    // and every commit (a commit tracks the MMAs of the thread that issues it).
    // The tensor core queues few MMAs ahead of the one it executes, so the thread's own work
    // between stages (an mbarrier test costs about 90 cycles even when the phase has completed)
    // would leave it idle: the next stage's barriers are tested without blocking between the
    // two halves of this stage's MMAs. The work entries come by two dependent loads (tile list,
    // then item table), issued a tile ahead: at the start of tile w the item of tile w + G (whose
    // list entry came during the previous tile) and the list entry of tile w + 2G, G the grid
    // size. The tile list holds only items with a record, so no work is skipped.
    int s = 0, lt = 0;
    uint32_t ph = 0;
    bool ready = false;  // stage s known to be filled
    const uint64_t x_desc0 = sw128_desc(smem_u32(ringX));
    constexpr uint64_t kH = kPXHalf >> 4;
    const int G = gridDim.x;
    int w = blockIdx.x;
    PWork wk{};
    bool have = w < n_work && work_at<KIND>(A, X, w, nch, &wk);
    int2 tl_n = w + G < n_work ? X.tiles[(w + G) / nch] : make_int2(0, 0);
    while (have) {
      const int w1 = w + G, w2 = w + 2 * G;
      const ItemRec it_n = w1 < n_work ? X.items[tl_n.x] : ItemRec{};
      const int2 tl_nn = w2 < n_work ? X.tiles[w2 / nch] : make_int2(0, 0);
      const int buf = lt & 1;
      // every decision warp uniform: elect.sync below needs all 32 lanes
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&H.acc_empty[buf], ((lt >> 1) & 1) ^ 1u, A.wait_ns))) {
        p_set_abort(H, A.status);
        break;
      }
      tc_fence_after();
      const uint32_t idesc = f16_idesc(kPW, (wk.nrows + 15) & ~15);
      const uint32_t d_tmem = tmem + (uint32_t)(buf * kPAcc);
      bool ok = true;
      for (int kc = 0; kc < KC; ++kc) {
        if (!ready) {
          const bool got = mbar_wait(&H.x_full[s], ph, A.wait_ns) && mbar_wait(&H.a_full[s], ph, A.wait_ns);
          if (!__all_sync(0xFFFFFFFFu, got)) {
            p_set_abort(H, A.status);
            ok = false;
            break;
          }
        }
        tc_fence_after();
        const int s1 = s + 1 == kPAStages ? 0 : s + 1;
        const uint32_t ph1 = s1 == 0 ? ph ^ 1u : ph;
        // K = 16 per MMA: 8 A columns, 32 bytes of the X rows (2 in the descriptor's address
        // field); the stage's second K step 32 columns and 16 KB (1024) further on
        const uint32_t a_tmem = tmem + kPACol0 + (uint32_t)(64 * s);
        const uint64_t xd = x_desc0 + (uint64_t)(s * (kPXStage >> 4));
        if (lane == 0) {
          umma_f16_ts(d_tmem, a_tmem, xd, idesc, kc != 0);
          umma_f16_ts(d_tmem, a_tmem + 8, xd + 2, idesc, 1);
          umma_f16_ts(d_tmem, a_tmem + 16, xd + 4, idesc, 1);
          umma_f16_ts(d_tmem, a_tmem + 24, xd + 6, idesc, 1);
        }
        __syncwarp();
        const bool nr = mbar_test(&H.x_full[s1], ph1) && mbar_test(&H.a_full[s1], ph1);
        if (lane == 0) {
          umma_f16_ts(d_tmem, a_tmem + 32, xd + kH, idesc, 1);
          umma_f16_ts(d_tmem, a_tmem + 40, xd + kH + 2, idesc, 1);
          umma_f16_ts(d_tmem, a_tmem + 48, xd + kH + 4, idesc, 1);
          umma_f16_ts(d_tmem, a_tmem + 56, xd + kH + 6, idesc, 1);
          umma_commit(&H.xa_empty[s]);
        }
        ready = __all_sync(0xFFFFFFFFu, nr);
        s = s1;
        ph = ph1;
      }
      if (!ok) break;
      if (lane == 0) umma_commit(&H.acc_full[buf]);
      __syncwarp();
      ++lt;
      have = w1 < n_work;
      if (have) {
        wk.item = tl_n.x;
        wk.rowA = it_n.row0 + tl_n.y;
        wk.nrows = min(kPM, it_n.ntok - tl_n.y);
        wk.n0 = (w1 % nch) * (KIND == kPGateUp ? kPW / 2 : kPW);
        wk.slot = it_n.slot;
        wk.shared = it_n.shared;
        wk.rec = it_n.rec;
      }
      w = w1;
      tl_n = tl_nn;
    }
    // Drain: one more commit arrives once every MMA this warp issued has completed, including
    // those left queued when a wait above ran out. Tensor memory and the rings are freed only
    // after it (waited for with the default limit, not the caller's shorter one).
    if (lane == 0) umma_commit(&H.drain);
    __syncwarp();
    mbar_wait(&H.drain, 0);
  } else if (warp >= kPEpiWarp0) {
    // ---------------- epilogue ----------------
    // Lane L = 32 q + lane of an accumulator is weight row L, its columns the tile's tokens. The
    // four warps take every decision together: warp 12 waits for the accumulator and passes the
    // outcome on through shared memory at a named barrier.
    const int q = warp & 3;
    const int L = q * 32 + lane;
    int lt = 0;
    for (int w = blockIdx.x; w < n_work; w += gridDim.x) {
      PWork wk;
      if (!work_at<KIND>(A, X, w, nch, &wk)) continue;
      const int buf = lt & 1;
      float* cs = col_s + buf * kPM;
      {
        // the per-column factor: x's unscale (gate/up), or h's 2^e (down)
        const int m = L;
        float v = 0.0f;
        if (m < wk.nrows) {
          const int r = wk.rowA + m;
          v = KIND == kPGateUp ? X.xunscale[X.row_tok[r]] : p_pow2f(X.hexp[r]);
        }
        cs[m] = v;
      }
      if (warp == kPEpiWarp0) {
        const bool ok = mbar_wait(&H.acc_full[buf], (lt >> 1) & 1, A.wait_ns) && !p_aborted(H);
        if (lane == 0) {
          if (!ok) p_set_abort(H, A.status);
          H.epi_ok[buf] = ok ? 1 : 0;
        }
      }
      named_sync(1, 128);
      if (!H.epi_ok[buf]) break;
      tc_fence_after();
      const uint32_t t_row = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * kPAcc);
      const int n_cols = (wk.nrows + 15) & ~15;
      // 16 token columns of this lane's weight row, from v
      auto process16 = [&](const uint32_t* v, int ch) {
        if (KIND == kPGateUp) {
          // lanes 2i and 2i + 1 hold the gate and the up row of column f = n0 + 16 q + i; the
          // even lane computes h for the chunk's first 8 tokens, the odd lane for the last 8
          const int fcol = wk.n0 + q * 16 + (lane >> 1);
          const int odd = lane & 1;
          float* hm = hm_s + (buf * 4 + q) * kPM;
          float mx[8];
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            const uint32_t give = odd ? v[jj] : v[8 + jj];  // the column the partner computes
            const uint32_t keep = odd ? v[8 + jj] : v[jj];
            const uint32_t got = __shfl_xor_sync(0xFFFFFFFFu, give, 1);
            const float g = __uint_as_float(odd ? got : keep), u = __uint_as_float(odd ? keep : got);
            const int col = ch + odd * 8 + jj;
            const float xs = cs[col];
            const float hv = silu_fast(g * xs) * (u * xs);
            float a = 0.0f;
            if (col < wk.nrows) {
              A.h[(size_t)(wk.rowA + col) * A.f + fcol] = hv;
              a = fabsf(hv);
            }
            mx[jj] = a;
          }
          // max over the 16 lanes of the same parity (the 16 columns of f of this quarter)
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
#pragma unroll
            for (int o = 2; o < 32; o <<= 1) mx[jj] = fmaxf(mx[jj], __shfl_xor_sync(0xFFFFFFFFu, mx[jj], o));
          }
          if (lane < 2) {
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) hm[ch + odd * 8 + jj] = mx[jj];
          }
        } else {
          const int drow = wk.n0 + L;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int col = ch + j;
            if (col < wk.nrows) {
              const float y = __uint_as_float(v[j]) * cs[col];
              const size_t off = (size_t)(wk.rowA + col) * A.d + drow;
              if (A.ydt == 1)
                static_cast<float*>(A.y)[off] = y;
              else
                static_cast<__nv_bfloat16*>(A.y)[off] = __float2bfloat16_rn(y);
            }
          }
        }
      };
      // 16 columns per tcgen05.ld, two register sets: the next load is in flight while the
      // current columns are processed. (Loads of 32 columns, two sets of 32 registers, made
      // the FFN 1.11x slower: 115 registers per thread against 80.)
      uint32_t va[16], vb[16];
      tmem_ld16(t_row, va);
      tmem_ld_wait16(va);
      for (int ch = 0; ch < n_cols; ch += 32) {
        const bool more1 = ch + 16 < n_cols, more2 = ch + 32 < n_cols;
        if (more1) tmem_ld16(t_row + ch + 16, vb);
        process16(va, ch);
        if (more1) {
          tmem_ld_wait16(vb);
          if (more2) tmem_ld16(t_row + ch + 32, va);
          process16(vb, ch + 16);
          if (more2) tmem_ld_wait16(va);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&H.acc_empty[buf]);
      if (KIND == kPGateUp) {
        // max |h| of each token row over this chunk's 64 columns of f: the four quarters' maxima
        named_sync(1, 128);
        if (L < wk.nrows) {
          const float* hb = hm_s + buf * 4 * kPM;
          const float m4 = fmaxf(fmaxf(hb[L], hb[kPM + L]), fmaxf(hb[2 * kPM + L], hb[3 * kPM + L]));
          atomicMax(X.hmax + wk.rowA + L, __float_as_uint(m4));
        }
      }
      ++lt;
    }
  }
  // Every role ends here. The MMA thread has waited for its drain commit, so no MMA is still
  // reading the rings or writing tensor memory, and the TMA producers have waited for their
  // copies in flight.
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

// Token rows (xp16 or h16): rows x K f16, boxes of 64 x 32 in the 128-byte swizzle.
bool encode_x(CUtensorMap* m, const void* base, int K, int rows) {
  return tmap_encode_2d(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, base, (uint64_t)K, (uint64_t)rows, (uint64_t)K * 2, kPK,
                        kPBox, CU_TENSOR_MAP_SWIZZLE_128B);
}

// Codes of the gate/up matrices of n records: (K byte, gate|up, row, record), boxes 128 x 2 x 64,
// so that box row 2i + g is the gate (g = 0) or up (g = 1) row of column i; 128-byte swizzle.
bool encode_q_gu(CUtensorMap* m, const uint8_t* recs, uint64_t n, const FfnArgs& a) {
  const cuuint64_t dims[4] = {(cuuint64_t)a.d, 2, (cuuint64_t)a.f, n};
  const cuuint64_t strides[3] = {(cuuint64_t)(a.o_up_q - a.o_gate_q), (cuuint64_t)a.d, a.slot_bytes};
  const cuuint32_t box[4] = {kPKS, 2, kPW / 2, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return p_encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<uint8_t*>(recs + a.o_gate_q), dims, strides,
                       box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Codes of the down matrix of n records: (K byte, row, record), boxes 128 x 128; 128-byte swizzle.
bool encode_q_dn(CUtensorMap* m, const uint8_t* recs, uint64_t n, const FfnArgs& a) {
  const cuuint64_t dims[3] = {(cuuint64_t)a.f, (cuuint64_t)a.d, n};
  const cuuint64_t strides[2] = {(cuuint64_t)a.f, a.slot_bytes};
  const cuuint32_t box[3] = {kPKS, kPW, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return p_encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(recs + a.o_down_q), dims, strides,
                       box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
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
  return a.xdt == 0 && a.d % 256 == 0 && a.f % 128 == 0 && tmap_available();
}

cudaError_t launch_ffn_prefill(const FfnArgs& a, const PrefillAux& x, int sm_count, cudaStream_t st) {
  const int rows = a.P + a.T * a.n_shared;
  if (rows == 0) return cudaSuccess;
  // the shared experts' records follow one another at the pool's record stride
  CUtensorMap tm_x, tm_h, qgu_pool, qgu_sh, qdn_pool, qdn_sh;
  const uint8_t* sh = a.n_shared > 0 ? a.shared : a.pool;
  const uint64_t nsh = a.n_shared > 0 ? (uint64_t)a.n_shared : 1;
  if (!encode_x(&tm_x, x.xp16, a.d, rows) || !encode_x(&tm_h, x.h16, a.f, rows) ||
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
