// Expert FFN for few tokens per expert with bf16 activations: weights streamed by TMA bulk
// copies into a shared-memory ring, dot products on the tensor cores.
//
// Decode reads each selected expert's int8 rows once ("Strata 工作原理图解GPU内存SSD三级存储如何让
// 125B模型塞进消费级显卡", section "推测解码": one token plus up to three drafts per step, so T = 4),
// so its time is that of streaming those bytes from HBM. Two persistent kernels, one CTA per
// SM, stream them:
//   gate/up: tiles of 16 rows of the gate and up matrices (and their scales), one tile per
//            (work item, 16 rows of f); h = silu(g) * u goes to an fp32 buffer.
//   down:    tiles of 64 rows of the down matrix, one tile per (work item, 64 rows of d).
// Each CTA takes a contiguous range of tiles, so consecutive tiles mostly belong to the same
// expert and reuse its activations from L1 / shared memory. A producer lane keeps up to NS
// tiles in flight with cp.async.bulk: one copy per weight row, into rows padded by 32 bytes
// so that the fragment reads are free of bank conflicts. The copies complete on an mbarrier
// per stage. Sixteen consumer warps split each tile between them, multiply with warp-level
// m16n8k16 MMAs (f16 operands, fp32 accumulation), and add their partial sums in shared
// memory in a fixed order.
//
// Why MMA for a GEMV: one SM must take in ~23 weight bytes per clock at ~6 TB/s. A SIMT loop
// that turns every code into an fp32 and multiplies in fp32 spends about one instruction per
// byte and is issue-bound well below that. A warp-level MMA consumes 256 weights per
// instruction, and its operands stay in registers.
//
// Exactness. Weight codes become f16 pairs exactly (a byte permute into 1024 + (q + 128),
// then one packed subtraction). Each MMA stays inside one 32-element block, so the block's
// fp16 scale multiplies the fp32 MMA result. Activations are f16 copies, exact after a
// per-token power-of-two rescale that puts max |x| in [2^14, 2^15) (bf16 has 8 significant bits).
// h is rescaled per row by a power of two from max |h| of that row and rounded once to f16
// (11 bits). That max is an atomic max of non-negative floats, so it does not depend on order.
//
// Lane (g, c) = (lane / 4, lane % 4) of an MMA holds rows g and g + 8. In MMA half h (0, 1)
// of block b, its k slots {2c, 2c+1, 2c+8, 2c+9} hold elements b*32 + c*8 + h*4 + {0..3}.
// The activation fragment uses the same order, so the k permutation cancels in the sum.
//
// Every wait is bounded. A wait that runs out sets MOE_DEV_TIMEOUT in the status word; the
// CTA then stops its work, lets its copies in flight land and returns.
#include "moe_common.cuh"
#include "sm100_ptx.cuh"

namespace moe {

constexpr int kConsumerWarps = 16;
constexpr int kStreamThreads = 32 * (1 + kConsumerWarps);
constexpr int kRowPad = 32;                 // bytes of padding per staged weight row
constexpr int kGateUpTileRows = 16;
constexpr int kDownTileRows = 64;           // kDownSub subtiles of 16 rows
constexpr int kDownSub = kDownTileRows / 16;
constexpr int kDownKSplit = kConsumerWarps / kDownSub;
constexpr int kHPad = 32;                   // f16 padding per staged h row
constexpr int kMaxStages = 8;
constexpr size_t kSmemBudget = 227 * 1024;  // dynamic shared memory per CTA

// ------------------------------------------------------------------ PTX helpers ----------

// Barrier of the consumer warps only (the producer warp does not take part).
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(32 * kConsumerWarps) : "memory");
}

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

// d (zeroed here) = block product of rows g, g+8 (8 codes each: wg, wg8) with this lane's 8
// activations (xv: 4 f16 pairs), as two MMAs.
__device__ __forceinline__ void block_mma(float* d, uint2 wg, uint2 wg8, const uint4& xv) {
  d[0] = d[1] = d[2] = d[3] = 0.0f;
  const uint32_t r0 = wg.x ^ 0x80808080u, r1 = wg.y ^ 0x80808080u;
  const uint32_t s0 = wg8.x ^ 0x80808080u, s1 = wg8.y ^ 0x80808080u;
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

// Contiguous range [t0, t1) of this CTA's tiles out of n, split over gridDim.x CTAs.
__device__ __forceinline__ void cta_tiles(int n, int* t0, int* t1) {
  *t0 = (int)((long long)blockIdx.x * n / gridDim.x);
  *t1 = (int)((long long)(blockIdx.x + 1) * n / gridDim.x);
}

// ------------------------------------------------------------------ work list ------------

struct Tile {
  const uint8_t* rec;
  int item, row0, ntok, routed, rt;  // rt: row tile index inside the item
};

__device__ __forceinline__ int n_items(const FfnArgs& A) { return A.active[0] + A.n_shared; }

__device__ __forceinline__ bool tile_at(const FfnArgs& A, int t, int tiles_per_item, Tile* out) {
  FfnItem it;
  out->item = t / tiles_per_item;
  if (!resolve_item(out->item, A, &it)) return false;
  out->rec = it.rec;
  out->row0 = it.row0;
  out->ntok = it.ntok;
  out->routed = it.routed;
  out->rt = t % tiles_per_item;
  return true;
}

// ------------------------------------------------------------------ activation staging ---

// x16[t][d] = f16(x[t] * 2^-e_t), xunscale[t] = 2^e_t; also clears hmax for every h row.
__global__ void __launch_bounds__(256) stage_x_f16_kernel(const void* x, int xdt, int T, int d, __half* x16,
                                                          float* xunscale, uint32_t* hmax, int h_rows) {
  __shared__ float wmax[8];
  const int t = blockIdx.x;
  for (int r = t * blockDim.x + threadIdx.x; r < h_rows; r += gridDim.x * blockDim.x) hmax[r] = 0u;
  float m = 0.0f;
  for (int i = threadIdx.x; i < d; i += blockDim.x) m = fmaxf(m, fabsf(load_act(x, xdt, (size_t)t * d + i)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
  __syncthreads();
  m = 0.0f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) m = fmaxf(m, wmax[w]);
  const int e = f16_exp_for(m);
  const float down = pow2f(-e);
  if (threadIdx.x == 0) xunscale[t] = pow2f(e);
  for (int i = threadIdx.x * 2; i < d; i += blockDim.x * 2) {
    const float a = load_act(x, xdt, (size_t)t * d + i), b = load_act(x, xdt, (size_t)t * d + i + 1);
    *reinterpret_cast<__half2*>(x16 + (size_t)t * d + i) = __floats2half2_rn(a * down, b * down);
  }
}

// ------------------------------------------------------------------ shared skeleton ------

struct StreamSmem {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  int abort;
  float red[2][kConsumerWarps][32][8];  // consumer partial sums, double-buffered
};

__device__ __forceinline__ void init_barriers(StreamSmem& S, int NS) {
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 1);
    }
    S.abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
}

// Producer (one lane): for each tile of this CTA, wait for a free stage and issue its copies
// with issue(tile, stage, full barrier). A tile whose item does not resolve completes its
// phase with no bytes. At the end, waits for every copy still in flight.
template <typename IssueFn>
__device__ __forceinline__ void producer_loop(const FfnArgs& A, StreamSmem& S, uint8_t* ring, size_t stage_bytes,
                                              int NS, int n_tiles, int tiles_per_item, IssueFn issue) {
  int j = 0, t0, t1;
  int last_use[kMaxStages];
  for (int s = 0; s < kMaxStages; ++s) last_use[s] = -1;
  cta_tiles(n_tiles, &t0, &t1);
  for (int t = t0; t < t1; ++t, ++j) {
    const int s = j % NS;
    if (!mbar_wait(&S.empty[s], ((j / NS) & 1) ^ 1) || *(volatile int*)&S.abort) {
      if (!*(volatile int*)&S.abort) {
        S.abort = 1;
        flag_status(A.status, MOE_DEV_TIMEOUT_BIT);
      }
      break;
    }
    Tile tl;
    if (tile_at(A, t, tiles_per_item, &tl)) issue(tl, ring + (size_t)s * stage_bytes, &S.full[s]);
    else mbar_arrive(&S.full[s]);
    last_use[s] = j / NS;
  }
  for (int s = 0; s < NS; ++s)
    if (last_use[s] >= 0) mbar_wait(&S.full[s], last_use[s] & 1);
}

// Consumer side of one tile's full barrier: bounded wait, then a consumer-wide decision on
// whether to go on (all consumer warps take the same branch).
__device__ __forceinline__ bool consumer_acquire(const FfnArgs& A, StreamSmem& S, int s, int j, int NS) {
  const bool ok = mbar_wait(&S.full[s], (j / NS) & 1);
  if (!ok && (threadIdx.x & 31) == 0) {
    S.abort = 1;
    flag_status(A.status, MOE_DEV_TIMEOUT_BIT);
  }
  consumer_sync();
  return !*(volatile int*)&S.abort;
}

// ------------------------------------------------------------------ gate/up + SwiGLU -----

__global__ void __launch_bounds__(kStreamThreads, 1) ffn_gateup_stream_kernel(FfnArgs A, const __half* x16,
                                                                             const float* xunscale, uint32_t* hmax,
                                                                             int NS) {
  extern __shared__ __align__(128) uint8_t dyn[];
  StreamSmem& S = *reinterpret_cast<StreamSmem*>(dyn);
  uint8_t* ring = dyn + ((sizeof(StreamSmem) + 127) & ~(size_t)127);
  const int d = A.d, nb = d / kQBlock, ldr = d + kRowPad;
  const int tiles_per_item = A.f / kGateUpTileRows;
  const int n_tiles = n_items(A) * tiles_per_item;
  // stage: gate rows [16][ldr] i8 | up rows [16][ldr] i8 | gate scales [16][nb] f16 | up scales
  const size_t o_up = (size_t)kGateUpTileRows * ldr, o_gs = 2 * o_up;
  const size_t o_us = o_gs + (size_t)kGateUpTileRows * nb * 2;
  const size_t stage_bytes = (o_us + (size_t)kGateUpTileRows * nb * 2 + 127) & ~(size_t)127;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  init_barriers(S, NS);

  if (warp == 0) {
    if (lane == 0) {
      producer_loop(A, S, ring, stage_bytes, NS, n_tiles, tiles_per_item,
                    [&](const Tile& tl, uint8_t* st, uint64_t* bar) {
                      const uint32_t srow = (uint32_t)(kGateUpTileRows * nb * 2);
                      mbar_arrive_expect_tx(bar, (uint32_t)(2 * kGateUpTileRows * d) + 2 * srow);
                      const int r0 = tl.rt * kGateUpTileRows;
                      const uint8_t* gq = tl.rec + A.o_gate_q + (size_t)r0 * d;
                      const uint8_t* uq = tl.rec + A.o_up_q + (size_t)r0 * d;
                      for (int r = 0; r < kGateUpTileRows; ++r) {
                        bulk_g2s(st + (size_t)r * ldr, gq + (size_t)r * d, d, bar);
                        bulk_g2s(st + o_up + (size_t)r * ldr, uq + (size_t)r * d, d, bar);
                      }
                      bulk_g2s(st + o_gs, tl.rec + A.o_gate_s + (size_t)r0 * nb * 2, srow, bar);
                      bulk_g2s(st + o_us, tl.rec + A.o_up_s + (size_t)r0 * nb * 2, srow, bar);
                    });
    }
    return;
  }

  // consumers: warp cw takes blocks [kb0, kb1) of every tile
  const int cw = warp - 1, ct = threadIdx.x - 32;
  const int g = lane >> 2, c = lane & 3;
  const int kb0 = cw * nb / kConsumerWarps, kb1 = (cw + 1) * nb / kConsumerWarps;
  int j = 0, t0, t1, rb = 0;
  cta_tiles(n_tiles, &t0, &t1);
  for (int t = t0; t < t1; ++t, ++j) {
    const int s = j % NS;
    if (!consumer_acquire(A, S, s, j, NS)) break;
    Tile tl;
    if (tile_at(A, t, tiles_per_item, &tl)) {
      const uint8_t* st = ring + (size_t)s * stage_bytes;
      const __half* gs = reinterpret_cast<const __half*>(st + o_gs);
      const __half* us = reinterpret_cast<const __half*>(st + o_us);
      for (int g0 = 0; g0 < tl.ntok; g0 += 8) {
        const int ng = min(8, tl.ntok - g0);
        const bool has_x = g < ng;
        const int tok = has_x ? (tl.routed ? A.sorted_pair[tl.row0 + g0 + g] / A.k : g0 + g) : 0;
        const __half* xrow = x16 + (size_t)tok * d + c * 8;
        float ag[4] = {0.f, 0.f, 0.f, 0.f}, au[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 2
        for (int b = kb0; b < kb1; ++b) {
          const uint4 xv = has_x ? __ldg(reinterpret_cast<const uint4*>(xrow + b * kQBlock)) : make_uint4(0, 0, 0, 0);
          const size_t wo = (size_t)g * ldr + b * kQBlock + c * 8;
          const uint2 wg = *reinterpret_cast<const uint2*>(st + wo);
          const uint2 wg8 = *reinterpret_cast<const uint2*>(st + wo + 8 * ldr);
          const uint2 wu = *reinterpret_cast<const uint2*>(st + o_up + wo);
          const uint2 wu8 = *reinterpret_cast<const uint2*>(st + o_up + wo + 8 * ldr);
          const float sg = __half2float(gs[g * nb + b]), sg8 = __half2float(gs[(g + 8) * nb + b]);
          const float su = __half2float(us[g * nb + b]), su8 = __half2float(us[(g + 8) * nb + b]);
          float dg[4], du[4];
          block_mma(dg, wg, wg8, xv);
          block_mma(du, wu, wu8, xv);
          ag[0] = fmaf(sg, dg[0], ag[0]); ag[1] = fmaf(sg, dg[1], ag[1]);
          ag[2] = fmaf(sg8, dg[2], ag[2]); ag[3] = fmaf(sg8, dg[3], ag[3]);
          au[0] = fmaf(su, du[0], au[0]); au[1] = fmaf(su, du[1], au[1]);
          au[2] = fmaf(su8, du[2], au[2]); au[3] = fmaf(su8, du[3], au[3]);
        }
        // The two reduction buffers alternate. A warp writes buffer X again only after the
        // next barrier, which the readers of X reach only after they have read it.
        float(*red)[32][8] = S.red[rb];
        rb ^= 1;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          red[cw][lane][q] = ag[q];
          red[cw][lane][4 + q] = au[q];
        }
        consumer_sync();
        if (ct < 128) {
          const int src = ct >> 2, q = ct & 3;  // source lane, accumulator slot
          float gv = 0.f, uv = 0.f;
#pragma unroll
          for (int w = 0; w < kConsumerWarps; ++w) {
            gv += red[w][src][q];
            uv += red[w][src][4 + q];
          }
          const int tcol = 2 * (src & 3) + (q & 1);
          const int row = tl.rt * kGateUpTileRows + (src >> 2) + (q >> 1) * 8;
          if (tcol < ng) {
            const int ttok = tl.routed ? A.sorted_pair[tl.row0 + g0 + tcol] / A.k : g0 + tcol;
            const float us_ = xunscale[ttok];
            const float hv = silu(gv * us_) * (uv * us_);
            const int hr = tl.row0 + g0 + tcol;
            A.h[(size_t)hr * A.f + row] = hv;
            atomicMax(hmax + hr, __float_as_uint(fabsf(hv)));
          }
        }
      }
    }
    if (ct == 0) mbar_arrive(&S.empty[s]);  // every consumer read the stage before the last barrier
  }
}

// ------------------------------------------------------------------ down ------------------

__global__ void __launch_bounds__(kStreamThreads, 1) ffn_down_stream_kernel(FfnArgs A, const uint32_t* hmax,
                                                                           int NS) {
  extern __shared__ __align__(128) uint8_t dyn[];
  StreamSmem& S = *reinterpret_cast<StreamSmem*>(dyn);
  const int f = A.f, nb = f / kQBlock, ldr = f + kRowPad, ldh = f + kHPad;
  __half* h16 = reinterpret_cast<__half*>(dyn + ((sizeof(StreamSmem) + 127) & ~(size_t)127));  // [8][ldh]
  float* hunscale = reinterpret_cast<float*>(h16 + 8 * ldh);                                      // [8]
  uint8_t* ring = reinterpret_cast<uint8_t*>(hunscale) + 128;
  const int tiles_per_item = A.d / kDownTileRows;
  const int n_tiles = n_items(A) * tiles_per_item;
  const size_t o_s = (size_t)kDownTileRows * ldr;
  const size_t stage_bytes = (o_s + (size_t)kDownTileRows * nb * 2 + 127) & ~(size_t)127;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  init_barriers(S, NS);

  if (warp == 0) {
    if (lane == 0) {
      producer_loop(A, S, ring, stage_bytes, NS, n_tiles, tiles_per_item,
                    [&](const Tile& tl, uint8_t* st, uint64_t* bar) {
                      const uint32_t sbytes = (uint32_t)(kDownTileRows * nb * 2);
                      mbar_arrive_expect_tx(bar, (uint32_t)(kDownTileRows * f) + sbytes);
                      const int n0 = tl.rt * kDownTileRows;
                      const uint8_t* dq = tl.rec + A.o_down_q + (size_t)n0 * f;
                      for (int r = 0; r < kDownTileRows; ++r) bulk_g2s(st + (size_t)r * ldr, dq + (size_t)r * f, f, bar);
                      bulk_g2s(st + o_s, tl.rec + A.o_down_s + (size_t)n0 * nb * 2, sbytes, bar);
                    });
    }
    return;
  }

  // consumers: kDownSub row subtiles of 16 x kDownKSplit parts of the blocks
  const int cw = warp - 1, ct = threadIdx.x - 32;
  const int sub = cw / kDownKSplit, kq = cw % kDownKSplit;
  const int g = lane >> 2, c = lane & 3;
  const int kb0 = kq * nb / kDownKSplit, kb1 = (kq + 1) * nb / kDownKSplit;
  const int rl = sub * 16 + g;  // local rows rl and rl + 8 of this lane
  int j = 0, t0, t1, rb = 0;
  int staged_row0 = -1;  // first h row staged in h16 (the same value in every consumer thread)
  cta_tiles(n_tiles, &t0, &t1);
  for (int t = t0; t < t1; ++t, ++j) {
    const int s = j % NS;
    if (!consumer_acquire(A, S, s, j, NS)) break;
    Tile tl;
    if (tile_at(A, t, tiles_per_item, &tl)) {
      const uint8_t* st = ring + (size_t)s * stage_bytes;
      const __half* sc = reinterpret_cast<const __half*>(st + o_s);
      for (int g0 = 0; g0 < tl.ntok; g0 += 8) {
        const int ng = min(8, tl.ntok - g0);
        if (staged_row0 != tl.row0 + g0) {  // stage these h rows as f16, rescaled per row
          consumer_sync();  // the previous group's readers of h16 / hunscale are done
          staged_row0 = tl.row0 + g0;
          for (int i = ct; i < ng * (f / 2); i += 32 * kConsumerWarps) {
            const int r = i / (f / 2), e = (i % (f / 2)) * 2;
            const int hr = staged_row0 + r;
            const int ex = f16_exp_for(__uint_as_float(hmax[hr]));
            const float down = pow2f(-ex);
            const float2 v = *reinterpret_cast<const float2*>(A.h + (size_t)hr * f + e);
            *reinterpret_cast<__half2*>(h16 + r * ldh + e) = __floats2half2_rn(v.x * down, v.y * down);
            if (e == 0) hunscale[r] = pow2f(ex);
          }
          consumer_sync();
        }
        const bool has_h = g < ng;
        const __half* hrow = h16 + g * ldh + c * 8;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 2
        for (int b = kb0; b < kb1; ++b) {
          const uint4 hv = has_h ? *reinterpret_cast<const uint4*>(hrow + b * kQBlock) : make_uint4(0, 0, 0, 0);
          const size_t wo = (size_t)rl * ldr + b * kQBlock + c * 8;
          const uint2 w = *reinterpret_cast<const uint2*>(st + wo);
          const uint2 w8 = *reinterpret_cast<const uint2*>(st + wo + 8 * ldr);
          const float s0 = __half2float(sc[rl * nb + b]), s8 = __half2float(sc[(rl + 8) * nb + b]);
          float dd[4];
          block_mma(dd, w, w8, hv);
          acc[0] = fmaf(s0, dd[0], acc[0]); acc[1] = fmaf(s0, dd[1], acc[1]);
          acc[2] = fmaf(s8, dd[2], acc[2]); acc[3] = fmaf(s8, dd[3], acc[3]);
        }
        float(*red)[32][8] = S.red[rb];
        rb ^= 1;
#pragma unroll
        for (int q = 0; q < 4; ++q) red[cw][lane][q] = acc[q];
        consumer_sync();
        {
          const int sb = ct >> 7, src = (ct >> 2) & 31, q = ct & 3;
          float v = 0.f;
#pragma unroll
          for (int w = 0; w < kDownKSplit; ++w) v += red[sb * kDownKSplit + w][src][q];
          const int tcol = 2 * (src & 3) + (q & 1);
          const int col = tl.rt * kDownTileRows + sb * 16 + (src >> 2) + (q >> 1) * 8;
          if (tcol < ng) {
            v *= hunscale[tcol];
            const size_t off = (size_t)(tl.row0 + g0 + tcol) * A.d + col;
            if (A.ydt == 1) static_cast<float*>(A.y)[off] = v;
            else static_cast<__nv_bfloat16*>(A.y)[off] = __float2bfloat16_rn(v);
          }
        }
      }
    }
    if (ct == 0) mbar_arrive(&S.empty[s]);
  }
}

// ------------------------------------------------------------------ launch ---------------

static size_t head_bytes() { return (sizeof(StreamSmem) + 127) & ~(size_t)127; }
static size_t down_extra_bytes(int f) { return ((size_t)8 * (f + kHPad) * 2 + 127) / 128 * 128 + 128; }

static int stages_for(size_t stage_bytes, size_t fixed) {
  const size_t room = kSmemBudget > fixed ? kSmemBudget - fixed : 0;
  const int ns = (int)(room / stage_bytes);
  return ns > kMaxStages ? kMaxStages : ns;
}

static size_t stage_bytes_gateup(int d) {
  const size_t ldr = d + kRowPad, nb = d / kQBlock;
  return (2 * kGateUpTileRows * ldr + 2 * kGateUpTileRows * nb * 2 + 127) & ~(size_t)127;
}

static size_t stage_bytes_down(int f) {
  const size_t ldr = f + kRowPad, nb = f / kQBlock;
  return (kDownTileRows * ldr + kDownTileRows * nb * 2 + 127) & ~(size_t)127;
}

bool stream_supported(const FfnArgs& a) {
  return a.d % kDownTileRows == 0 && stages_for(stage_bytes_gateup(a.d), head_bytes()) >= 2 &&
         stages_for(stage_bytes_down(a.f), head_bytes() + down_extra_bytes(a.f)) >= 2;
}

cudaError_t launch_ffn_decode_tc(const FfnArgs& a, __half* x16, float* xunscale, uint32_t* hmax, int sm_count,
                                 cudaStream_t st) {
  const int items_max = (a.P < a.E ? a.P : a.E) + a.n_shared;
  if (items_max == 0) return cudaSuccess;
  const int h_rows = a.P + a.T * a.n_shared;
  stage_x_f16_kernel<<<a.T, 256, 0, st>>>(a.x, a.xdt, a.T, a.d, x16, xunscale, hmax, h_rows);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  {
    const size_t sb = stage_bytes_gateup(a.d);
    const int ns = stages_for(sb, head_bytes());
    const size_t smem = head_bytes() + ns * sb;
    if ((e = ensure_dynamic_smem(reinterpret_cast<const void*>(ffn_gateup_stream_kernel), smem)) != cudaSuccess)
      return e;
    const int tiles = items_max * (a.f / kGateUpTileRows);
    const int grid = tiles < sm_count ? tiles : sm_count;
    ffn_gateup_stream_kernel<<<grid, kStreamThreads, smem, st>>>(a, x16, xunscale, hmax, ns);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  const size_t sb = stage_bytes_down(a.f);
  const size_t fixed = head_bytes() + down_extra_bytes(a.f);
  const int ns = stages_for(sb, fixed);
  const size_t smem = fixed + ns * sb;
  if ((e = ensure_dynamic_smem(reinterpret_cast<const void*>(ffn_down_stream_kernel), smem)) != cudaSuccess) return e;
  const int tiles = items_max * (a.d / kDownTileRows);
  const int grid = tiles < sm_count ? tiles : sm_count;
  ffn_down_stream_kernel<<<grid, kStreamThreads, smem, st>>>(a, hmax, ns);
  return cudaGetLastError();
}

}  // namespace moe
