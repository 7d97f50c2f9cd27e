// Expert FFN for few tokens per expert with bf16 activations: weights streamed by TMA tensor
// copies into a shared-memory ring, dot products on the tensor cores.
//
// Decode reads each selected expert's int8 rows once ("Strata 工作原理图解GPU内存SSD三级存储如何让
// 125B模型塞进消费级显卡", section "推测解码": one token plus up to three drafts per step, so T = 4),
// so its time is that of streaming those bytes from HBM. Three kernels:
//   prepare: activations to f16 (rescaled per token by a power of two), the work-item table
//            (each selected expert's slot found through the slot table), the token of every
//            output row, cleared max |h| per row and per-item unit counters;
//   gate/up: a work unit is (item, 32 rows of f). Stage kc of a unit holds K bytes
//            [128 kc, 128 kc + 128) of those 32 gate rows and the same 32 up rows: one 8 KB
//            TMA box of a 4-D view (K byte, row, gate|up, slot) of the expert pool. An MMA
//            tile takes 8 gate rows as M rows 0..7 and the same 8 up rows as M rows 8..15,
//            so each lane holds g and u of the same (row, token) and applies h = silu(g) * u
//            in registers; h goes to an fp32 buffer. The last unit of an item to finish turns
//            the item's h rows into f16 (rescaled per row by a power of two from max |h|);
//   down:    a work unit is (item, 64 rows of d); stage kc holds K bytes [128 kc, +128) of
//            those rows (one 8 KB box of a 3-D view (K byte, row, slot)).
// Both streaming kernels are persistent (one CTA per SM); each CTA takes a contiguous range of
// units. One producer thread keeps up to 24 stages (192 KB) in flight. Eight consumer warps
// split every stage: warp (mt, kh) owns M tile mt (16 rows) and K half kh (two 32-element
// blocks of the stage). The two K halves of an M tile are added once per pass, through
// shared memory, in a fixed order.
//
// Shared-memory layout. The boxes use the 128-byte swizzle: byte k of box line L sits at
// L * 128 + ((k / 16) ^ (L % 8)) * 16 + k % 16. Lane group g of an MMA reads line rho(g)
// (mod 8) with rho = (0, 2, 4, 6, 1, 3, 5, 7), so the four rows read by each half-warp sit in
// four different 32-byte bank groups: the weight reads are free of bank conflicts.
//
// Why MMA for a GEMV: one SM must take in ~22 weight bytes per clock at ~6.5 TB/s. A warp
// MMA consumes 256 weights per instruction with its operands in registers.
//
// Exactness. Weight codes become f16 pairs exactly (a byte permute into 1024 + (q + 128),
// then one packed subtraction). Each MMA stays inside one 32-element block, so the block's
// fp16 scale multiplies the fp32 MMA result. Activations are exact f16 copies after a
// per-token power-of-two rescale that puts max |x| in [2^14, 2^15) (bf16 has 8 significant
// bits). h is rounded once to f16 (11 bits) after its row's power-of-two rescale. The row
// max is an atomic max of non-negative floats (order-free) and every sum has a fixed order:
// results are deterministic.
//
// Lane (g, c) = (lane / 4, lane % 4) of an m16n8k16 MMA holds M rows g and g + 8 and token
// columns 2c, 2c + 1 of the result. In MMA half hf (0, 1) of a 32-element block, its k
// slots {2c, 2c+1, 2c+8, 2c+9} hold elements c*8 + hf*4 + {0..3}; the activation fragment of
// token g uses the same order, so the k permutation cancels in the sum.
//
// Every wait is bounded. A wait that runs out sets MOE_DEV_TIMEOUT in the status word; the
// CTA then stops its work, lets its copies in flight land and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "moe_common.cuh"
#include "sm100_ptx.cuh"

namespace moe {

constexpr int kSlice = 128;        // K bytes per stage: one 128-byte swizzle span
constexpr int kGuUnitRows = 64;     // gate rows (and up rows) per gate/up unit
constexpr int kDnUnitRows = 128;    // down rows per down unit
constexpr int kStageBytes = 16384;  // 2 * 64 * 128 = 128 * 128
constexpr int kConsumers = 16;      // 8 M tiles x 2 K halves
constexpr int kThreads = 32 * (1 + kConsumers);
constexpr int kStages = 13;         // 208 KB of boxes in flight per SM
constexpr int kPassTok = 16;       // tokens per pass over a unit (two MMA column groups)
constexpr size_t kSmemBudget = 227 * 1024;

// ------------------------------------------------------------------ small helpers --------

__device__ __forceinline__ void mma_f16_16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two int8 codes of a word whose bytes were offset by 128 (bytes selected by SEL) -> exact f16 pair.
template <uint32_t SEL>
__device__ __forceinline__ uint32_t i8x2_to_f16x2(uint32_t biased) {
  const uint32_t h = __byte_perm(biased, 0x64646464u, SEL);  // halves 1024 + (q + 128)
  const __half2 v = __hsub2(*reinterpret_cast<const __half2*>(&h), __half2half2(__ushort_as_half(0x6480)));
  return *reinterpret_cast<const uint32_t*>(&v);
}

// d (zeroed here) = block product of M rows g, g+8 (8 codes each: w_lo, w_hi) with this
// lane's 8 activations of token g (xv: 4 f16 pairs), as two MMAs.
__device__ __forceinline__ void block_mma(float* d, uint2 w_lo, uint2 w_hi, const uint4& xv) {
  d[0] = d[1] = d[2] = d[3] = 0.0f;
  const uint32_t r0 = w_lo.x ^ 0x80808080u, r1 = w_lo.y ^ 0x80808080u;
  const uint32_t s0 = w_hi.x ^ 0x80808080u, s1 = w_hi.y ^ 0x80808080u;
  mma_f16_16816(d, i8x2_to_f16x2<0x5140>(r0), i8x2_to_f16x2<0x5140>(s0), i8x2_to_f16x2<0x5342>(r0),
                i8x2_to_f16x2<0x5342>(s0), xv.x, xv.y);
  mma_f16_16816(d, i8x2_to_f16x2<0x5140>(r1), i8x2_to_f16x2<0x5140>(s1), i8x2_to_f16x2<0x5342>(r1),
                i8x2_to_f16x2<0x5342>(s1), xv.z, xv.w);
}

__device__ __forceinline__ float pow2f(int e) { return __uint_as_float((uint32_t)(127 + e) << 23); }

// e with m * 2^-e in [2^14, 2^15) for a normal m > 0 (clamped to [-100, 100]); 0 for m == 0.
// Scaling a row by 2^-e puts its largest magnitude near the top of the f16 range, so values
// down to 2^-28 of that maximum stay normal f16 numbers.
__device__ __forceinline__ int f16_exp_for(float m) {
  if (!(m > 0.0f)) return 0;
  const int e = (int)((__float_as_uint(m) >> 23) & 0xFF) - 127 - 14;
  return e < -100 ? -100 : (e > 100 ? 100 : e);
}

__device__ __forceinline__ uint32_t f16x2_bits(float a, float b) {
  const __half2 v = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ float half_lo(uint32_t v) { return __half2float(__ushort_as_half((unsigned short)(v & 0xFFFFu))); }
__device__ __forceinline__ float half_hi(uint32_t v) { return __half2float(__ushort_as_half((unsigned short)(v >> 16))); }

// Contiguous range [t0, t1) of this CTA's units out of n, split over gridDim.x CTAs.
__device__ __forceinline__ void cta_range(int n, int* t0, int* t1) {
  *t0 = (int)((long long)blockIdx.x * n / gridDim.x);
  *t1 = (int)((long long)(blockIdx.x + 1) * n / gridDim.x);
}

__device__ __forceinline__ int n_items(const FfnArgs& A) { return A.active[0] + A.n_shared; }

__device__ __forceinline__ int rho(int g) { return ((g & 3) << 1) | (g >> 2); }

// Byte offset of byte k (0..127) of line L in a box written with the 128-byte swizzle.
__device__ __forceinline__ uint32_t sw128(int line, int k) {
  return (uint32_t)line * 128u + ((uint32_t)(((k >> 4) ^ line) & 7) << 4) + (uint32_t)(k & 15);
}

// ------------------------------------------------------------------ prepare --------------

// CTA t: x16[t] = f16(x[t] * 2^-e_t), xunscale[t] = 2^e_t. All CTAs: hmax[r] = 0 and
// row_tok[r] (token of output row r) for every row. CTA 0: the work-item table and its counters.
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
  const int e = f16_exp_for(m);
  const float down = pow2f(-e);
  if (threadIdx.x == 0) X.xunscale[t] = pow2f(e);
  for (int i = threadIdx.x * 2; i < d; i += blockDim.x * 2) {
    const float a = load_act(A.x, A.xdt, (size_t)t * d + i), b = load_act(A.x, A.xdt, (size_t)t * d + i + 1);
    *reinterpret_cast<uint32_t*>(X.x16 + (size_t)t * d + i) = f16x2_bits(a * down, b * down);
  }
}

// ------------------------------------------------------------------ pipeline --------------

struct Head {
  uint64_t full[kStages];    // stage s holds its box (TMA completion)
  uint64_t empty[kStages];   // every consumer warp is done with stage s
  uint64_t red_full[8];      // M tile mt: K half 1 wrote its partial sums
  uint64_t red_empty[8];     // M tile mt: K half 0 read them
  uint64_t unit_done;        // every consumer warp finished its part of a unit
  uint64_t unit_decided;     // the unit's "last of its item" decision is in last[]
  int abort;
  int last[2];               // per unit parity: 1 if the unit was the last of its item
  float red[8][32][8];       // K half 1's partial sums of each M tile, per lane, (2 groups x 4)
};
constexpr size_t kHeadBytes = (sizeof(Head) + 1023) & ~(size_t)1023;
constexpr size_t kSmemBytes = kHeadBytes + 1024 + (size_t)kStages * kStageBytes;  // 1024: ring alignment slack
static_assert(kSmemBytes <= kSmemBudget, "ring does not fit in shared memory");

__device__ __forceinline__ bool aborted(const Head& H) { return *(volatile const int*)&H.abort != 0; }

__device__ __forceinline__ void set_abort(Head& H, int* status) {
  if (!aborted(H)) {
    H.abort = 1;
    flag_status(status, MOE_DEV_TIMEOUT_BIT);
  }
}

// Ring base: the first 1024-byte boundary (of the shared-memory window) after the head.
__device__ __forceinline__ uint8_t* ring_base(uint8_t* dyn) {
  const uint32_t a = smem_u32(dyn + kHeadBytes);
  return dyn + kHeadBytes + (((a + 1023u) & ~1023u) - a);
}

// Position in the ring: stage index and the parity of its current use.
struct RingPos {
  int s = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void next() {
    if (++s == kStages) {
      s = 0;
      phase ^= 1u;
    }
  }
};

enum { kGateUp = 0, kDown = 1 };

template <int KIND>
struct Geo {
  static constexpr int unit_rows = KIND == kGateUp ? kGuUnitRows : kDnUnitRows;
};

// Accumulates one stage into acc for NG token groups (8 tokens each): this warp's two
// 32-element blocks of M rows line_lo / line_hi of the box, with their scales slo / shi.
template <int NG>
__device__ __forceinline__ void stage_mma(const uint8_t* st, int off_lo0, int off_hi0, int off_lo1, int off_hi1,
                                          uint32_t slo, uint32_t shi, const uint4 (&bv)[2][2], float (&acc)[2][4]) {
#pragma unroll
  for (int jj = 0; jj < 2; ++jj) {
    const uint2 wl = *reinterpret_cast<const uint2*>(st + (jj ? off_lo1 : off_lo0));
    const uint2 wh = *reinterpret_cast<const uint2*>(st + (jj ? off_hi1 : off_hi0));
    const float s_lo = jj ? half_hi(slo) : half_lo(slo);
    const float s_hi = jj ? half_hi(shi) : half_lo(shi);
#pragma unroll
    for (int gi = 0; gi < NG; ++gi) {
      float dd[4];
      block_mma(dd, wl, wh, bv[gi][jj]);
      acc[gi][0] = fmaf(s_lo, dd[0], acc[gi][0]);
      acc[gi][1] = fmaf(s_lo, dd[1], acc[gi][1]);
      acc[gi][2] = fmaf(s_hi, dd[2], acc[gi][2]);
      acc[gi][3] = fmaf(s_hi, dd[3], acc[gi][3]);
    }
  }
}

// The streaming kernel. KIND = kGateUp: K = d over the gate/up matrices; kDown: K = f over down.
template <int KIND>
__global__ void __launch_bounds__(kThreads, 1) ffn_tma_kernel(FfnArgs A, StreamAux X,
                                                             const __grid_constant__ CUtensorMap tm_pool,
                                                             const __grid_constant__ CUtensorMap tm_shared) {
  extern __shared__ __align__(1024) uint8_t dyn[];
  Head& H = *reinterpret_cast<Head*>(dyn);
  uint8_t* ring = ring_base(dyn);
  const int d = A.d, f = A.f;
  const int K = KIND == kGateUp ? d : f;
  const int KC = K / kSlice;
  const int nb = K / kQBlock;  // scale blocks per row of the streamed matrix
  const int upi = (KIND == kGateUp ? f : d) / Geo<KIND>::unit_rows;
  const int n_units = n_items(A) * upi;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&H.full[s], 1);
      mbar_init(&H.empty[s], kConsumers);
    }
    for (int m = 0; m < 8; ++m) {
      mbar_init(&H.red_full[m], 1);
      mbar_init(&H.red_empty[m], 1);
    }
    mbar_init(&H.unit_done, kConsumers);
    mbar_init(&H.unit_decided, 1);
    H.abort = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_pool);
    prefetch_tmap(&tm_shared);
  }
  __syncthreads();
  int u0, u1;
  cta_range(n_units, &u0, &u1);

  if (warp == 0) {
    // ---------------- producer: one thread issues every stage's TMA box ----------------
    if (lane != 0) return;
    RingPos rp;
    int issued = 0, cur = -1;
    ItemRec it{};
    for (int u = u0; u < u1 && !aborted(H); ++u) {
      const int item = u / upi, rb = u % upi;
      if (item != cur) {
        it = X.items[item];
        cur = item;
      }
      if (it.rec == nullptr || it.ntok <= 0) continue;
      // the unit's scale rows: ask L2 for them now, the consumers load them per stage
      if (KIND == kGateUp) {
        const uint32_t sb = (uint32_t)(kGuUnitRows * nb * 2);
        prefetch_l2(it.rec + A.o_gate_s + (size_t)rb * sb, sb);
        prefetch_l2(it.rec + A.o_up_s + (size_t)rb * sb, sb);
      } else {
        const uint32_t sb = (uint32_t)(kDnUnitRows * nb * 2);
        prefetch_l2(it.rec + A.o_down_s + (size_t)rb * sb, sb);
      }
      const CUtensorMap* tm = it.shared ? &tm_shared : &tm_pool;
      const int passes = (it.ntok + kPassTok - 1) / kPassTok;
      for (int p = 0; p < passes; ++p) {
        for (int kc = 0; kc < KC; ++kc, rp.next(), ++issued) {
          if (!mbar_wait(&H.empty[rp.s], rp.phase ^ 1u) || aborted(H)) {
            set_abort(H, A.status);
            goto drain;
          }
          mbar_arrive_expect_tx(&H.full[rp.s], kStageBytes);
          uint8_t* st = ring + (size_t)rp.s * kStageBytes;
          if (KIND == kGateUp) tma_load_4d(st, tm, kc * kSlice, rb * kGuUnitRows, 0, it.slot, &H.full[rp.s]);
          else tma_load_3d(st, tm, kc * kSlice, rb * kDnUnitRows, it.slot, &H.full[rp.s]);
        }
      }
    }
  drain:
    for (int s = 0; s < kStages && s < issued; ++s) {  // wait for every copy still in flight
      const int last = s + kStages * ((issued - 1 - s) / kStages);
      mbar_wait(&H.full[s], (last / kStages) & 1);
    }
    return;
  }

  // ---------------- consumers ----------------
  const int cw = warp - 1, mt = cw & 7, kh = cw >> 3;
  const int g = lane >> 2, c = lane & 3, rg = rho(g);
  const int ct = threadIdx.x - 32;  // 0 .. 32 * kConsumers - 1
  // box lines of this lane's M rows g (lo) and g + 8 (hi), and the byte offsets in a stage of
  // its 8 codes in each of this warp's two blocks
  const int line_lo = KIND == kGateUp ? mt * 8 + rg : mt * 16 + rg;
  const int line_hi = KIND == kGateUp ? kGuUnitRows + mt * 8 + rg : mt * 16 + 8 + rg;
  const int k0 = (kh * 2) * kQBlock + c * 8, k1 = k0 + kQBlock;
  const int off_lo0 = (int)sw128(line_lo, k0), off_lo1 = (int)sw128(line_lo, k1);
  const int off_hi0 = (int)sw128(line_hi, k0), off_hi1 = (int)sw128(line_hi, k1);
  // Bounded wait by every lane; a timeout aborts the CTA's work.
  auto warp_wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    const bool ok = mbar_wait(bar, parity);
    if (__all_sync(0xFFFFFFFFu, ok)) return true;
    if (lane == 0) set_abort(H, A.status);
    return false;
  };
  RingPos rp;
  int cur = -1, npass = 0, nunit = 0;
  ItemRec it{};
  for (int u = u0; u < u1; ++u) {
    const int item = u / upi, rb = u % upi;
    if (item != cur) {
      it = X.items[item];
      cur = item;
    }
    if (it.rec == nullptr || it.ntok <= 0) continue;
    // matrix rows of M rows g (lo) and g + 8 (hi), and their scale rows
    int row_lo, row_hi;
    const uint8_t *sc_lo, *sc_hi;
    if (KIND == kGateUp) {
      row_lo = row_hi = rb * kGuUnitRows + mt * 8 + rg;  // gate row and up row of the same f index
      sc_lo = it.rec + A.o_gate_s + (size_t)row_lo * nb * 2;
      sc_hi = it.rec + A.o_up_s + (size_t)row_hi * nb * 2;
    } else {
      row_lo = rb * kDnUnitRows + mt * 16 + rg;
      row_hi = row_lo + 8;
      sc_lo = it.rec + A.o_down_s + (size_t)row_lo * nb * 2;
      sc_hi = it.rec + A.o_down_s + (size_t)row_hi * nb * 2;
    }
    const int passes = (it.ntok + kPassTok - 1) / kPassTok;
    for (int p = 0; p < passes; ++p) {
      const int base = p * kPassTok;
      const int ng0 = min(8, it.ntok - base), ng1 = min(8, it.ntok - base - 8);  // ng1 <= 0: one group
      // activation rows of this lane's token column g in groups 0 and 1
      const __half* bsrc[2];
      bool has[2];
#pragma unroll
      for (int gi = 0; gi < 2; ++gi) {
        const int idx = base + gi * 8 + g;
        has[gi] = g < (gi ? ng1 : ng0);
        const int r = it.row0 + (has[gi] ? idx : base);
        bsrc[gi] = KIND == kGateUp ? X.x16 + (size_t)X.row_tok[r] * d + c * 8 : X.h16 + (size_t)r * f + c * 8;
      }
      float acc[2][4];
#pragma unroll
      for (int gi = 0; gi < 2; ++gi)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[gi][q] = 0.0f;

      for (int kc = 0; kc < KC; ++kc, rp.next()) {
        const int b0 = kc * 4 + kh * 2;  // first of this warp's two blocks
        // loads that do not depend on the stage: scales (2 blocks) and activations
        const uint32_t slo = __ldg(reinterpret_cast<const unsigned int*>(sc_lo + b0 * 2));
        const uint32_t shi = __ldg(reinterpret_cast<const unsigned int*>(sc_hi + b0 * 2));
        uint4 bv[2][2];
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
          bv[0][jj] = has[0] ? __ldg(reinterpret_cast<const uint4*>(bsrc[0] + (b0 + jj) * kQBlock))
                             : make_uint4(0, 0, 0, 0);
          bv[1][jj] = has[1] ? __ldg(reinterpret_cast<const uint4*>(bsrc[1] + (b0 + jj) * kQBlock))
                             : make_uint4(0, 0, 0, 0);
        }
        if (!warp_wait(&H.full[rp.s], rp.phase)) return;
        const uint8_t* st = ring + (size_t)rp.s * kStageBytes;
        if (ng1 > 0) stage_mma<2>(st, off_lo0, off_hi0, off_lo1, off_hi1, slo, shi, bv, acc);
        else stage_mma<1>(st, off_lo0, off_hi0, off_lo1, off_hi1, slo, shi, bv, acc);
        __syncwarp();
        if (lane == 0) mbar_arrive(&H.empty[rp.s]);
      }

      // K half 1 hands its partial sums to K half 0 (fixed order: half 0 + half 1)
      const uint32_t par = npass & 1;
      ++npass;
      if (kh == 1) {
        if (!warp_wait(&H.red_empty[mt], par ^ 1)) return;
#pragma unroll
        for (int gi = 0; gi < 2; ++gi)
#pragma unroll
          for (int q = 0; q < 4; ++q) H.red[mt][lane][gi * 4 + q] = acc[gi][q];
        __syncwarp();
        if (lane == 0) mbar_arrive(&H.red_full[mt]);
        continue;
      }
      if (!warp_wait(&H.red_full[mt], par)) return;
#pragma unroll
      for (int gi = 0; gi < 2; ++gi)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[gi][q] += H.red[mt][lane][gi * 4 + q];
      __syncwarp();
      if (lane == 0) mbar_arrive(&H.red_empty[mt]);

      // epilogue: lane (g, c) holds rows row_lo (q = 0, 1) / row_hi (q = 2, 3), tokens 2c, 2c+1
#pragma unroll
      for (int gi = 0; gi < 2; ++gi) {
        const int ng = gi ? ng1 : ng0;
        if (ng <= 0) break;
        if (KIND == kGateUp) {
          float m[2] = {0.f, 0.f};
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int tcol = 2 * c + q;
            if (tcol < ng) {
              const int r = it.row0 + base + gi * 8 + tcol;
              const float xs = X.xunscale[X.row_tok[r]];
              const float hv = silu(acc[gi][q] * xs) * (acc[gi][2 + q] * xs);
              A.h[(size_t)r * f + row_lo] = hv;
              m[q] = fabsf(hv);
            }
          }
#pragma unroll
          for (int o = 4; o < 32; o <<= 1) {
            m[0] = fmaxf(m[0], __shfl_xor_sync(0xFFFFFFFFu, m[0], o));
            m[1] = fmaxf(m[1], __shfl_xor_sync(0xFFFFFFFFu, m[1], o));
          }
          if (g == 0) {
            const int r = it.row0 + base + gi * 8 + 2 * c;
            if (2 * c < ng) atomicMax(X.hmax + r, __float_as_uint(m[0]));
            if (2 * c + 1 < ng) atomicMax(X.hmax + r + 1, __float_as_uint(m[1]));
          }
        } else {
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int tcol = 2 * c + q;
            if (tcol < ng) {
              const int r = it.row0 + base + gi * 8 + tcol;
              const float up = pow2f(X.hexp[r]);
              const float v_lo = acc[gi][q] * up, v_hi = acc[gi][2 + q] * up;
              const size_t off = (size_t)r * d;
              if (A.ydt == 1) {
                static_cast<float*>(A.y)[off + row_lo] = v_lo;
                static_cast<float*>(A.y)[off + row_hi] = v_hi;
              } else {
                static_cast<__nv_bfloat16*>(A.y)[off + row_lo] = __float2bfloat16_rn(v_lo);
                static_cast<__nv_bfloat16*>(A.y)[off + row_hi] = __float2bfloat16_rn(v_hi);
              }
            }
          }
        }
      }
    }

    if (KIND == kGateUp) {
      // The last unit of this item to finish turns the item's h rows into f16 for the down
      // kernel. Every warp fences its h and hmax writes before the unit is counted, so the
      // counter reaches upi only after all of the item's writes are visible.
      const uint32_t par = nunit & 1;
      ++nunit;
      __threadfence();
      __syncwarp();
      if (lane == 0) mbar_arrive(&H.unit_done);
      if (ct == 0) {
        const bool ok = mbar_wait(&H.unit_done, par);
        if (!ok) set_abort(H, A.status);
        H.last[par] = ok && atomicAdd(X.item_cnt + item, 1) == upi - 1;
        mbar_arrive(&H.unit_decided);
      }
      if (!warp_wait(&H.unit_decided, par)) return;
      if (*(volatile int*)&H.last[par]) {
        __threadfence();
        const int half = f / 2;
        for (int i = ct; i < it.ntok * half; i += 32 * kConsumers) {
          const int r = it.row0 + i / half, col = (i % half) * 2;
          const int e = f16_exp_for(__uint_as_float(__ldcg(X.hmax + r)));
          const float down = pow2f(-e);
          const float2 v = __ldcg(reinterpret_cast<const float2*>(A.h + (size_t)r * f + col));
          *reinterpret_cast<uint32_t*>(X.h16 + (size_t)r * f + col) = f16x2_bits(v.x * down, v.y * down);
          if (col == 0) X.hexp[r] = e;
        }
      }
    }
  }
}

// ------------------------------------------------------------------ host side ------------

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

struct MapSet {
  CUtensorMap gu_pool, gu_shared, dn_pool, dn_shared;
};

struct MapKey {
  const void* pool;
  const void* shared;
  uint64_t n_slots, slot_bytes;
  int d, f, n_shared;
  bool operator==(const MapKey& o) const {
    return pool == o.pool && shared == o.shared && n_slots == o.n_slots && slot_bytes == o.slot_bytes &&
           d == o.d && f == o.f && n_shared == o.n_shared;
  }
};

// 4-D view (K byte, row, gate|up, slot) of the gate/up codes of `n` records at `base`.
bool encode_gu(CUtensorMap* m, const uint8_t* base, uint64_t n, const FfnArgs& a, uint64_t slot_bytes) {
  const cuuint64_t dims[4] = {(cuuint64_t)a.d, (cuuint64_t)a.f, 2, n};
  const cuuint64_t strides[3] = {(cuuint64_t)a.d, (cuuint64_t)(a.o_up_q - a.o_gate_q), slot_bytes};
  const cuuint32_t box[4] = {kSlice, kGuUnitRows, 2, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, (void*)(base + a.o_gate_q), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D view (K byte, row, slot) of the down codes of `n` records at `base`.
bool encode_dn(CUtensorMap* m, const uint8_t* base, uint64_t n, const FfnArgs& a, uint64_t slot_bytes) {
  const cuuint64_t dims[3] = {(cuuint64_t)a.f, (cuuint64_t)a.d, n};
  const cuuint64_t strides[2] = {(cuuint64_t)a.f, slot_bytes};
  const cuuint32_t box[3] = {kSlice, kDnUnitRows, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, (void*)(base + a.o_down_q), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The four tensor maps of a pool view, encoded once per distinct view (a few are cached).
bool get_maps(const FfnArgs& a, const PoolView& pv, MapSet* out) {
  static std::mutex mu;
  static MapKey keys[8];
  static MapSet sets[8];
  static int n_cached = 0, next = 0;
  const MapKey key{pv.pool, pv.shared, pv.n_slots, pv.slot_bytes, a.d, a.f, a.n_shared};
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n_cached; ++i)
    if (keys[i] == key) {
      *out = sets[i];
      return true;
    }
  if (!encode_fn()) return false;
  MapSet m;
  const uint8_t* pool = static_cast<const uint8_t*>(pv.pool);
  const uint8_t* sh = a.n_shared > 0 ? static_cast<const uint8_t*>(pv.shared) : pool;
  const uint64_t nsh = a.n_shared > 0 ? (uint64_t)a.n_shared : 1;
  if (!encode_gu(&m.gu_pool, pool, pv.n_slots, a, pv.slot_bytes) ||
      !encode_gu(&m.gu_shared, sh, nsh, a, pv.slot_bytes) ||
      !encode_dn(&m.dn_pool, pool, pv.n_slots, a, pv.slot_bytes) ||
      !encode_dn(&m.dn_shared, sh, nsh, a, pv.slot_bytes))
    return false;
  keys[next] = key;
  sets[next] = m;
  next = (next + 1) % 8;
  if (n_cached < 8) ++n_cached;
  *out = m;
  return true;
}

}  // namespace

bool stream_supported(const FfnArgs& a) {
  return a.d % kDnUnitRows == 0 && a.f % kGuUnitRows == 0 && a.d % kSlice == 0 && a.f % kSlice == 0 &&
         encode_fn() != nullptr;
}

cudaError_t launch_ffn_stream(const FfnArgs& a, const StreamAux& x, const PoolView& pv, int sm_count,
                              cudaStream_t st) {
  const int items_max = (a.P < a.E ? a.P : a.E) + a.n_shared;
  if (items_max == 0) return cudaSuccess;
  MapSet maps;
  if (!get_maps(a, pv, &maps)) return cudaErrorInvalidValue;
  ffn_prepare_kernel<<<a.T, 256, 0, st>>>(a, x);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const size_t smem = kSmemBytes;
  {
    auto kern = ffn_tma_kernel<kGateUp>;
    if ((e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), smem)) != cudaSuccess) return e;
    const int units = items_max * (a.f / kGuUnitRows);
    kern<<<units < sm_count ? units : sm_count, kThreads, smem, st>>>(a, x, maps.gu_pool, maps.gu_shared);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  auto kern = ffn_tma_kernel<kDown>;
  if ((e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), smem)) != cudaSuccess) return e;
  const int units = items_max * (a.d / kDnUnitRows);
  kern<<<units < sm_count ? units : sm_count, kThreads, smem, st>>>(a, x, maps.dn_pool, maps.dn_shared);
  return cudaGetLastError();
}

}  // namespace moe
