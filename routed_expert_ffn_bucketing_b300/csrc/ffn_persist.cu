// Decode expert FFN (few tokens per expert, bf16 activations) as one persistent kernel: the
// gate/up projections with SwiGLU and the down projection of every selected expert, streamed
// from HBM once ("Strata 工作原理图解GPU内存SSD三级存储如何让125B模型塞进消费级显卡", section
// "推测解码": a decode step verifies one token plus up to three drafts, T = 4).
//
// One CTA of 16 warps per SM, launched cooperatively (all CTAs resident). Phases:
//   0. each CTA builds the work-item table (each selected expert's record through the slot
//      table, then the shared experts) and the token of every output row in shared memory,
//      issues its warps' first weight loads, and converts x to f16 in shared memory: block b
//      of every token is scaled by the power of two 2^-e_b that puts the block's largest
//      magnitude (over the T tokens) near the top of the f16 range;
//   1. gate/up: a task is (item, 8 rows of f); M rows 0..7 of the MMA are gate rows and 8..15
//      the same up rows, so each lane holds g and u of one (row, token) and writes
//      h = silu(g) * u (fp32) and the row's max |h| (an order-free atomic max); the task then
//      counts itself done for its item in shared memory. When all its warps are through, the
//      CTA fences once and adds its counts to the per-item counters in global memory (a fence
//      per task would wait for the warp's next weight loads already in flight);
//   2. each warp issues the first weight loads of its down work. The CTA waits (bounded) until
//      every gate/up task of the items its down work covers is done, and converts those
//      items' h rows to f16 in shared memory (power-of-two rescale from each row's max);
//   3. down: a task is (item, 16 rows of d); y_perm rows are written in fp32 or bf16.
// Within a phase the (task, group of D blocks) sequence is cut into one contiguous range per
// warp, equal to within one group (stream-K). A warp streams its range without a break: the
// weights of the next group (one 16-byte load per lane, row and pair of blocks), and its
// scales, are requested while the current group is multiplied, across task boundaries. A task cut between two warps is finished by the second
// to arrive, which adds the two partial sums in a fixed order (part 0 + part 1). A warp's down
// range covers about the same items as its gate/up range, so the waits of phase 2 are mostly on
// work of the same or neighbouring CTAs.
//
// The counters (per-item tasks done, stream-K parts, row maxima) hold zeros at launch: moe_route
// clears them, and every launch leaves them cleared (the finisher of a cut task resets its
// counter; the last CTA out resets the rest), so no memset stands between the bucketing kernel
// and this one: in moe_layer_forward the kernel launches as a programmatic dependent of the
// bucketing kernel and stages x before its dependency wait. Every wait is bounded: one that runs
// out sets MOE_DEV_TIMEOUT and the CTA stops before its down work.
#include "decode_mma.cuh"
#include "sm100_ptx.cuh"

namespace moe {

namespace {

constexpr int kPW = 16;  // warps per CTA
constexpr int kPThreads = 32 * kPW;
enum { kGU = 0, kDN = 1 };

__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
// Waits until at most N of this thread's committed cp.async groups are still pending.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__host__ __device__ inline uint32_t align16(uint32_t v) { return (v + 15u) & ~15u; }

// Row strides of the staged activations, chosen against shared-memory bank conflicts: an f16
// row of K elements is padded to 64 bytes past a multiple of 128 (the 8 lanes of a 16-byte
// access phase read rows g, g + 1 at offsets c*16: 64 bytes apart), a row of K/32 fp32 block
// sums to 16 bytes past a multiple of 128 (rows 2c and 2c + 1 for c = 0..3 fall in 4 distinct
// 16-byte bank groups).
__host__ __device__ inline uint32_t act_stride(int K) { return (((uint32_t)K * 2u + 127u) & ~127u) + 64u; }
__host__ __device__ inline uint32_t sum_stride(int K) { return (((uint32_t)(K / 32) * 4u + 127u) & ~127u) + 16u; }

// Most h rows one CTA stages for its down work. A CTA stages the rows [r_lo, r_hi) from its
// first down item's first row to its last item's last row. The active list may be any subset of
// the routed experts (e.g. only those a slot table has just loaded), whose rows lie anywhere in
// [0, P) with other experts' rows between them, so the span is bounded only by all the rows.
__host__ __device__ inline int p_rows_cap(int T, int d, int items_max, int rows, int n_warps) {
  (void)T;
  (void)d;
  (void)items_max;
  (void)n_warps;
  return rows;
}

// Shared-memory layout of one CTA (byte offsets), the same on host and device.
struct PLayout {
  uint32_t items, done, rowtok, hexp, xe, bmax, sring, act, total;
};

template <int DG, int DD, int FMT>
__host__ __device__ inline PLayout p_layout(int T, int d, int f, int items_max, int rows, int rows_cap) {
  PLayout L;
  uint32_t o = 0;
  L.items = o;
  o = align16(o + (uint32_t)items_max * (uint32_t)sizeof(ItemRec));
  L.done = o;  // int32 [items]: gate/up tasks this CTA finished per item
  o = align16(o + 4u * items_max);
  L.rowtok = o;
  o = align16(o + 4u * rows);
  L.hexp = o;
  o = align16(o + 4u * rows);
  L.xe = o;  // fp32 [d/32]: 2^e_b, the unscale of x block b
  o = align16(o + 4u * (d / kQBlock));
  L.bmax = o;  // uint32 [d/32]: bits of max |x| over block b of every token
  o = align16(o + 4u * (d / kQBlock));
  L.sring = o;  // per warp: 2 slots (int8) or 4 (2-bit format) x 16 rows x D f16 scales
  const int dmax = DG > DD ? DG : DD;
  o = align16(o + (uint32_t)kPW * (FMT == 1 ? 4u : 2u) * 16u * dmax * 2u);
  L.act = o;  // x rows for gate/up, then this CTA's h rows for down
  const uint32_t xb = (uint32_t)T * (act_stride(d) + sum_stride(d));
  const uint32_t hb = (uint32_t)rows_cap * (act_stride(f) + sum_stride(f));
  o = align16(o + (xb > hb ? xb : hb));
  L.total = o;
  return L;
}

struct PAux {
  float* part;         // [2][part_stride]: stream-K partial sums, 128 floats per part, 2 parts per task
  int32_t* task_cnt;   // [2][cnt_stride]: stream-K parts finished per task (0 at launch)
  uint32_t* hmax;      // [rows]: bits of max |h| per h row (0 at launch)
  int32_t* item_done;  // [items]: gate/up tasks finished per item (0 at launch)
  size_t part_stride, cnt_stride;
  int rows_cap;
  int32_t* exit;       // [2]: CTAs finished; abandoned work (0 at launch)
};

// What one lane needs for one task: the addresses it loads codes and scales from, and where its
// activation fragment and accumulator inputs are in shared memory.
struct PTask {
  const uint8_t* wlo;   // codes of M row g at chunk c (byte c*16; add 64 per pair of blocks); row g + 8 is
                        // hi_delta(A) further
  const uint8_t* ssrc;  // lanes 0..15: f16 scales of M row (lane) (add 2 per block); else unused
  uint32_t xrow;        // shared-memory offset of the activation row of token column g, element c*8
  uint32_t cs0, cs1;    // shared-memory offsets of the accumulator-input rows of columns 2c, 2c + 1
  int item, row0, ntok, mt;
  bool valid, has;
};

// Distance from the codes of M row g to those of M row g + 8: the up matrix's row (gate/up) or
// the down row 8 further (down).
template <int KIND, int FMT>
__device__ __forceinline__ long long hi_delta(const FfnArgs& A) {
  return KIND == 0 ? (long long)A.o_up_q - (long long)A.o_gate_q : 8LL * A.f / (FMT == 1 ? 4 : 1);
}

// sx, sc: shared-memory offsets of the staged activation rows and of their accumulator inputs
// (for down: of row 0, which may lie before the staged span; only staged rows are addressed).
template <int KIND, int FMT>
__device__ __forceinline__ PTask make_task(const FfnArgs& A, const ItemRec* items, const int* rowtok, uint32_t sx,
                                           uint32_t sc, int t, int lane) {
  const int g = lane >> 2, c = lane & 3;
  const int tpi = KIND == kGU ? A.f / 8 : A.d / 16;
  PTask p;
  p.item = t / tpi;
  p.mt = t % tpi;
  const ItemRec it = items[p.item];
  p.valid = it.rec != nullptr && it.ntok > 0;
  p.row0 = it.row0;
  p.ntok = it.ntok < 8 ? it.ntok : 8;
  p.has = g < p.ntok;
  const uint8_t* rec = p.valid ? it.rec : A.pool;  // a valid address even for a skipped task
  const int r0 = 2 * c < p.ntok ? 2 * c : 0, r1 = 2 * c + 1 < p.ntok ? 2 * c + 1 : 0;
  if (KIND == kGU) {
    const int d = A.d, nb = d / kQBlock;
    p.wlo = rec + A.o_gate_q + (size_t)(p.mt * 8 + g) * (d / (FMT == 1 ? 4 : 1)) + c * 16;
    const int srow = p.mt * 8 + (lane & 7);
    p.ssrc = rec + (lane < 8 ? A.o_gate_s : A.o_up_s) + (size_t)srow * nb * 2;
    const int tg = p.valid ? rowtok[p.row0 + (p.has ? g : 0)] : 0;
    p.xrow = sx + (uint32_t)tg * act_stride(d) + c * 16u;
    p.cs0 = sc + (uint32_t)(p.valid ? rowtok[p.row0 + r0] : 0) * sum_stride(d);
    p.cs1 = sc + (uint32_t)(p.valid ? rowtok[p.row0 + r1] : 0) * sum_stride(d);
  } else {
    const int f = A.f, nb = f / kQBlock;
    p.wlo = rec + A.o_down_q + (size_t)(p.mt * 16 + g) * (f / (FMT == 1 ? 4 : 1)) + c * 16;
    p.ssrc = rec + A.o_down_s + (size_t)(p.mt * 16 + (lane & 15)) * nb * 2;
    p.xrow = sx + (uint32_t)(p.row0 + (p.has ? g : 0)) * act_stride(f) + c * 16u;
    p.cs0 = sc + (uint32_t)(p.row0 + r0) * sum_stride(f);
    p.cs1 = sc + (uint32_t)(p.row0 + r1) * sum_stride(f);
  }
  return p;
}

// The codes of the group being multiplied, in registers: int8, one 8-byte fragment per block and
// row; 2-bit format (groups of 8 blocks), one 16-byte chunk per row.
template <int D, int FMT>
struct Ring {
  uint2 lo[D], hi[D];
};
constexpr int kQ2Ahead = 4;  // groups of 2-bit codes a warp has requested ahead of the one it multiplies
template <>
struct Ring<8, 1> {
  uint4 lo[kQ2Ahead], hi[kQ2Ahead];  // group G0 + m kQ2Ahead + q of a range at position q
};

// Requests group gs of task p: D blocks of both rows into the ring, and the 16 rows' D scales
// into scale slot `slot` of this warp (lanes 0..15, one cp.async each).
template <int D, int FMT>
__device__ __forceinline__ void issue_group(const PTask& p, long long dhi, int gs, Ring<D, FMT>& ring,
                                            uint32_t sring_w, int slot, int lane) {
  if (!p.valid) return;
  if constexpr (FMT == 0) {
#pragma unroll
    for (int j = 0; j < D; j += 2) {  // one 16-byte load: this lane's codes of blocks j and j + 1
      const uint4 a = ld_codes16(p.wlo + (size_t)(gs * D + j) * kQBlock);
      const uint4 b = ld_codes16(p.wlo + dhi + (size_t)(gs * D + j) * kQBlock);
      ring.lo[j] = make_uint2(a.x, a.y);
      ring.lo[j + 1] = make_uint2(a.z, a.w);
      ring.hi[j] = make_uint2(b.x, b.y);
      ring.hi[j + 1] = make_uint2(b.z, b.w);
    }
  }
  if (lane < 16) {
    const uint32_t dst = sring_w + (uint32_t)(slot * 16 + lane) * (D * 2);
    if (D == 8) cp_async16(dst, p.ssrc + gs * D * 2);
    else cp_async8(dst, p.ssrc + gs * D * 2);
  }
}

// Writes the 32 values v of block b (row order) as f16 in the permuted order to the staged row
// at `row` (shared memory) and returns -offset * (sum of the f16 values), the block's MMA
// accumulator input (offset 1152 for int8 codes, 1025.5 for the 2-bit format). The block is written as four 16-byte chunks, chunk (q + b/2) % 4 at step
// q, so that 8 threads storing blocks b..b+7 of a row hit 8 distinct 16-byte bank groups.
__device__ __forceinline__ float stage_block_f16(uint8_t* row, int b, const float* v, float offset) {
  uint32_t w[16];
  float s = 0.0f;
#pragma unroll
  for (int i = 0; i < kQBlock; i += 4) {
    // within each group of 4 the order is (0, 2, 1, 3)
    const __half h0 = __float2half_rn(v[i]), h1 = __float2half_rn(v[i + 1]);
    const __half h2 = __float2half_rn(v[i + 2]), h3 = __float2half_rn(v[i + 3]);
    s += __half2float(h0);
    s += __half2float(h1);
    s += __half2float(h2);
    s += __half2float(h3);
    w[i / 2] = (uint32_t)__half_as_ushort(h0) | ((uint32_t)__half_as_ushort(h2) << 16);
    w[i / 2 + 1] = (uint32_t)__half_as_ushort(h1) | ((uint32_t)__half_as_ushort(h3) << 16);
  }
  uint4* dst = reinterpret_cast<uint4*>(row + (size_t)b * kQBlock * 2);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int k = (q + (b >> 1)) & 3;
    uint4 u;
    u.x = k == 0 ? w[0] : k == 1 ? w[4] : k == 2 ? w[8] : w[12];
    u.y = k == 0 ? w[1] : k == 1 ? w[5] : k == 2 ? w[9] : w[13];
    u.z = k == 0 ? w[2] : k == 1 ? w[6] : k == 2 ? w[10] : w[14];
    u.w = k == 0 ? w[3] : k == 1 ? w[7] : k == 2 ? w[11] : w[15];
    dst[k] = u;
  }
  return -offset * s;
}

// 32 bf16 values (64 bytes at p, 16-byte aligned) to fp32.
__device__ __forceinline__ void load_bf16_block(const uint16_t* p, float* v) {
  const uint4* src = reinterpret_cast<const uint4*>(p);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 u = __ldcg(src + q);  // through L2: an earlier kernel may have rewritten x
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int z = 0; z < 4; ++z) {
      v[q * 8 + 2 * z] = bf16_bits_to_f32(w[z] & 0xFFFFu);
      v[q * 8 + 2 * z + 1] = bf16_bits_to_f32(w[z] >> 16);
    }
  }
}

// Phase epilogues. Lane (g, c) holds M rows g (acc 0, 1) and g + 8 (acc 2, 3) for token
// columns 2c, 2c + 1 of the task's item.
template <int KIND>
__device__ __forceinline__ void p_epilogue(const FfnArgs& A, const PAux& X, const PTask& p, const int* hexp, int lane,
                                           const float (&acc)[4], int* s_done) {
  const int g = lane >> 2, c = lane & 3;
  if (KIND == kGU) {
    float m[2] = {0.f, 0.f};
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int tc = 2 * c + q;
      if (tc < p.ntok) {
        const int r = p.row0 + tc;
        const float hv = silu(acc[q]) * acc[2 + q];
        A.h[(size_t)r * A.f + p.mt * 8 + g] = hv;
        m[q] = fabsf(hv);
      }
    }
#pragma unroll
    for (int s = 4; s < 32; s <<= 1) {
      m[0] = fmaxf(m[0], __shfl_xor_sync(0xFFFFFFFFu, m[0], s));
      m[1] = fmaxf(m[1], __shfl_xor_sync(0xFFFFFFFFu, m[1], s));
    }
    if (g == 0) {
      if (2 * c < p.ntok) atomicMax(X.hmax + p.row0 + 2 * c, __float_as_uint(m[0]));
      if (2 * c + 1 < p.ntok) atomicMax(X.hmax + p.row0 + 2 * c + 1, __float_as_uint(m[1]));
    }
    // the task is done: counted for its item in this CTA (published after the phase)
    if (lane == 0) atomicAdd(s_done + p.item, 1);
  } else {
    const int row_lo = p.mt * 16 + g, row_hi = row_lo + 8;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int tc = 2 * c + q;
      if (tc < p.ntok) {
        const int r = p.row0 + tc;
        const float up = pow2f(hexp[r]);
        const size_t off = (size_t)r * A.d;
        if (A.ydt == 1) {
          static_cast<float*>(A.y)[off + row_lo] = acc[q] * up;
          static_cast<float*>(A.y)[off + row_hi] = acc[2 + q] * up;
        } else {
          static_cast<__nv_bfloat16*>(A.y)[off + row_lo] = __float2bfloat16_rn(acc[q] * up);
          static_cast<__nv_bfloat16*>(A.y)[off + row_hi] = __float2bfloat16_rn(acc[2 + q] * up);
        }
      }
    }
  }
}

// This warp's range [G0, G1) of the phase's (task, group) sequence, or an empty range.
__device__ __forceinline__ void warp_range(int n_tasks, int gpt, int wid, int n_warps, long long* G0, long long* G1) {
  const int nw = n_warps < n_tasks ? n_warps : n_tasks;  // each range at least one task long
  if (wid >= nw) {
    *G0 = *G1 = 0;
    return;
  }
  const long long total = (long long)n_tasks * gpt;
  *G0 = (long long)wid * total / nw;
  *G1 = (long long)(wid + 1) * total / nw;
}

// Streams groups [G0, G1) of one phase. On entry the ring and scale slot `slot` hold group G0
// (issue_group was called for it and its cp.async committed). On return `slot` is the slot the
// next phase's first group goes to. xe: for gate/up, the shared-memory offset of the x block
// unscales (each block's MMA result is multiplied by its own power of two).
template <int KIND, int D, int FMT>
__device__ __forceinline__ void p_stream(const FfnArgs& A, const PAux& X, const uint8_t* psm, const ItemRec* items,
                                         const int* rowtok, uint32_t sx, uint32_t sc, uint32_t xe, const int* hexp,
                                         uint32_t sring_w, const uint16_t* sring_p, long long G0, long long G1,
                                         int gpt, Ring<D, FMT>& ring, int& slot, int lane, int* s_done) {
  static_assert(FMT == 0, "the 2-bit format streams through p_stream_q2");
  if (G0 >= G1) return;
  const int g = lane >> 2;
  const long long dhi = hi_delta<KIND, FMT>(A);
  float* part = X.part + (size_t)KIND * X.part_stride;
  int* cnt = X.task_cnt + (size_t)KIND * X.cnt_stride;
  int t = (int)(G0 / gpt);
  PTask cur = make_task<KIND, FMT>(A, items, rowtok, sx, sc, t, lane);
  PTask nxt = cur;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (long long G = G0; G < G1; ++G) {
    const int gs = (int)(G - (long long)t * gpt);
    const long long Gn = G + 1;
    const bool more = Gn < G1;
    const int tn = more ? (int)(Gn / gpt) : t;
    if (more && tn != t) nxt = make_task<KIND, FMT>(A, items, rowtok, sx, sc, tn, lane);
    const int gsn = (int)(Gn - (long long)tn * gpt);
    const PTask& src = tn != t ? nxt : cur;
    __syncwarp();
    if (more && src.valid && lane < 16) {
      const uint32_t dst = sring_w + (uint32_t)((slot ^ 1) * 16 + lane) * (D * 2);
      if (D == 8) cp_async16(dst, src.ssrc + gsn * D * 2);
      else cp_async8(dst, src.ssrc + gsn * D * 2);
    }
    cp_async_commit();
    cp_async_wait1();
    __syncwarp();
    if (cur.valid) {
      // this group's scales of rows g (lo) and g + 8 (hi)
      uint32_t slo[D / 2], shi[D / 2];
      const uint16_t* sp = sring_p + (size_t)(slot * 16) * D;
      if (D == 8) {
        const uint4 a = *reinterpret_cast<const uint4*>(sp + g * D);
        const uint4 b = *reinterpret_cast<const uint4*>(sp + (8 + g) * D);
        slo[0] = a.x; slo[1 % (D / 2)] = a.y; slo[2 % (D / 2)] = a.z; slo[3 % (D / 2)] = a.w;
        shi[0] = b.x; shi[1 % (D / 2)] = b.y; shi[2 % (D / 2)] = b.z; shi[3 % (D / 2)] = b.w;
      } else {
        const uint2 a = *reinterpret_cast<const uint2*>(sp + g * D);
        const uint2 b = *reinterpret_cast<const uint2*>(sp + (8 + g) * D);
        slo[0] = a.x; slo[1 % (D / 2)] = a.y;
        shi[0] = b.x; shi[1 % (D / 2)] = b.y;
      }
      float4 c0, c1, xu;
#pragma unroll
      for (int j = 0; j < D; ++j) {
        const int b = gs * D + j;
        if ((j & 3) == 0) {
          c0 = *reinterpret_cast<const float4*>(psm + cur.cs0 + b * 4);
          c1 = *reinterpret_cast<const float4*>(psm + cur.cs1 + b * 4);
          if (KIND == kGU) xu = *reinterpret_cast<const float4*>(psm + xe + b * 4);
        }
        const uint4 xv =
            cur.has ? *reinterpret_cast<const uint4*>(psm + cur.xrow + b * kQBlock * 2) : make_uint4(0, 0, 0, 0);
        const int jj = j & 3;
        const float ca = jj == 0 ? c0.x : jj == 1 ? c0.y : jj == 2 ? c0.z : c0.w;
        const float cb = jj == 0 ? c1.x : jj == 1 ? c1.y : jj == 2 ? c1.z : c1.w;
        float dd[4];
        block_mma(dd, ring.lo[j], ring.hi[j], xv, ca, cb);
        {
          if (more && src.valid && (j & 1)) {  // blocks j - 1 and j are consumed: refill both
            const uint4 a = ld_codes16(src.wlo + (size_t)(gsn * D + j - 1) * kQBlock);
            const uint4 b = ld_codes16(src.wlo + dhi + (size_t)(gsn * D + j - 1) * kQBlock);
            ring.lo[j - 1] = make_uint2(a.x, a.y);
            ring.lo[j] = make_uint2(a.z, a.w);
            ring.hi[j - 1] = make_uint2(b.x, b.y);
            ring.hi[j] = make_uint2(b.z, b.w);
          }
        }
        const uint32_t wl = slo[j >> 1], wh = shi[j >> 1];
        float s_lo = __half2float(__ushort_as_half((unsigned short)((j & 1) ? (wl >> 16) : (wl & 0xFFFFu))));
        float s_hi = __half2float(__ushort_as_half((unsigned short)((j & 1) ? (wh >> 16) : (wh & 0xFFFFu))));
        if (KIND == kGU) {
          const float u = jj == 0 ? xu.x : jj == 1 ? xu.y : jj == 2 ? xu.z : xu.w;
          s_lo *= u;
          s_hi *= u;
        }
        acc[0] = fmaf(s_lo, dd[0], acc[0]);
        acc[1] = fmaf(s_lo, dd[1], acc[1]);
        acc[2] = fmaf(s_hi, dd[2], acc[2]);
        acc[3] = fmaf(s_hi, dd[3], acc[3]);
      }
    } else if (more && src.valid) {
      {
#pragma unroll
        for (int j = 0; j < D; j += 2) {
          const uint4 a = ld_codes16(src.wlo + (size_t)(gsn * D + j) * kQBlock);
          const uint4 b = ld_codes16(src.wlo + dhi + (size_t)(gsn * D + j) * kQBlock);
          ring.lo[j] = make_uint2(a.x, a.y);
          ring.lo[j + 1] = make_uint2(a.z, a.w);
          ring.hi[j] = make_uint2(b.x, b.y);
          ring.hi[j + 1] = make_uint2(b.z, b.w);
        }
      }
    }
    slot ^= 1;
    if (gs == gpt - 1 || !more) {
      // the task ends in this range: finish it, or publish this part of a cut task
      if (cur.valid) {
        const long long t0 = (long long)t * gpt;
        const bool first = G0 <= t0, last = G1 >= t0 + gpt;
        bool finish = true;
        if (!(first && last)) {
          const int my = first ? 0 : 1;
          float4* slot_p = reinterpret_cast<float4*>(part + ((size_t)t * 2 + my) * 128);
          slot_p[lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
          __threadfence();
          __syncwarp();
          int second = 0;
          if (lane == 0) {
            second = atomicAdd(cnt + t, 1) == 1;
            if (second) cnt[t] = 0;  // both parts are in: the counter is free for the next launch
          }
          finish = __shfl_sync(0xFFFFFFFFu, second, 0) != 0;
          if (finish) {
            __threadfence();
            const float4 p0 = __ldcg(reinterpret_cast<const float4*>(part + (size_t)t * 2 * 128) + lane);
            const float4 p1 = __ldcg(reinterpret_cast<const float4*>(part + ((size_t)t * 2 + 1) * 128) + lane);
            acc[0] = p0.x + p1.x;
            acc[1] = p0.y + p1.y;
            acc[2] = p0.z + p1.z;
            acc[3] = p0.w + p1.w;
          }
        }
        if (finish) p_epilogue<KIND>(A, X, cur, hexp, lane, acc, s_done);
      }
      acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
    }
    if (more && tn != t) {
      cur = nxt;
      t = tn;
    }
  }
}

// ------------------------------------------------------------------ 2-bit format ---------
// A group of the 2-bit format is 8 blocks: 64 bytes of codes per M row (one 16-byte chunk per
// lane) and 16 bytes of fp16 scales per row. Bytes per group are a quarter of int8's, so with
// one group in flight per warp the streaming would be bound by latency, not bandwidth: a warp
// keeps kQ2Ahead groups requested ahead, the codes in a register queue (Ring<8, 1>) and the
// scales in a cp.async ring of kQ2Ahead slots (one commit per group).

// Requests group gs of task p: its codes into (lo, hi), its scales into scale slot `slot`;
// commits one cp.async group in any case.
__device__ __forceinline__ void q2_request(const PTask& p, long long dhi, int gs, uint4& lo, uint4& hi,
                                           uint32_t sring_w, int slot, int lane) {
  if (p.valid) {
    lo = ld_codes16(p.wlo + (size_t)gs * 64);
    hi = ld_codes16(p.wlo + dhi + (size_t)gs * 64);
    if (lane < 16) cp_async16(sring_w + (uint32_t)(slot * 16 + lane) * 16u, p.ssrc + gs * 16);
  }
  cp_async_commit();
}

// Requests the first kQ2Ahead groups of the range [G0, G1) into queue positions 0..kQ2Ahead-1.
template <int KIND>
__device__ __forceinline__ void q2_prime(const FfnArgs& A, const ItemRec* items, const int* rowtok, uint32_t sx,
                                         uint32_t sc, long long G0, long long G1, int gpt, Ring<8, 1>& ring,
                                         uint32_t sring_w, int lane) {
  const long long dhi = hi_delta<KIND, 1>(A);
  int t = -1;
  PTask p{};
#pragma unroll
  for (int i = 0; i < kQ2Ahead; ++i) {
    const long long G = G0 + i;
    if (G < G1) {
      if ((int)(G / gpt) != t) {
        t = (int)(G / gpt);
        p = make_task<KIND, 1>(A, items, rowtok, sx, sc, t, lane);
      }
      q2_request(p, dhi, (int)(G - (long long)t * gpt), ring.lo[i], ring.hi[i], sring_w, (int)(G % kQ2Ahead), lane);
    } else {
      cp_async_commit();
    }
  }
}

// Streams groups [G0, G1) of one phase of the 2-bit format (primed by q2_prime). As p_stream,
// with the group requested kQ2Ahead ahead instead of one.
template <int KIND>
__device__ __forceinline__ void p_stream_q2(const FfnArgs& A, const PAux& X, const uint8_t* psm,
                                            const ItemRec* items, const int* rowtok, uint32_t sx, uint32_t sc,
                                            uint32_t xe, const int* hexp, uint32_t sring_w, const uint16_t* sring_p,
                                            long long G0, long long G1, int gpt, Ring<8, 1>& ring, int lane,
                                            int* s_done) {
  if (G0 >= G1) return;
  const int g = lane >> 2;
  const long long dhi = hi_delta<KIND, 1>(A);
  float* part = X.part + (size_t)KIND * X.part_stride;
  int* cnt = X.task_cnt + (size_t)KIND * X.cnt_stride;
  int t = (int)(G0 / gpt);
  PTask cur = make_task<KIND, 1>(A, items, rowtok, sx, sc, t, lane);
  int tl = -1;  // task of the group requested ahead
  PTask la = cur;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  // kQ2Ahead groups per outer step: group G0 + m kQ2Ahead + q sits at queue position q (as
  // q2_prime placed the first ones), so every position is a fixed register set; the group
  // requested kQ2Ahead ahead refills the position just consumed
  for (long long Gb = G0; Gb < G1; Gb += kQ2Ahead) {
#pragma unroll
    for (int q = 0; q < kQ2Ahead; ++q) {
      const long long G = Gb + q;
      if (G >= G1) break;
      const int gs = (int)(G - (long long)t * gpt);
      cp_async_wait<kQ2Ahead - 1>();  // this group's scales have landed
      __syncwarp();
      if (cur.valid) {
        const uint16_t* sp = sring_p + (size_t)((int)(G % kQ2Ahead) * 16) * 8;
        const uint4 sa = *reinterpret_cast<const uint4*>(sp + g * 8);
        const uint4 sb = *reinterpret_cast<const uint4*>(sp + (8 + g) * 8);
        const uint32_t slo[4] = {sa.x, sa.y, sa.z, sa.w}, shi[4] = {sb.x, sb.y, sb.z, sb.w};
        const uint32_t qlo[4] = {ring.lo[q].x, ring.lo[q].y, ring.lo[q].z, ring.lo[q].w};
        const uint32_t qhi[4] = {ring.hi[q].x, ring.hi[q].y, ring.hi[q].z, ring.hi[q].w};
        float4 c0, c1, xu;
        float2 f_lo, f_hi;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int b = gs * 8 + j;
          if ((j & 3) == 0) {
            c0 = *reinterpret_cast<const float4*>(psm + cur.cs0 + b * 4);
            c1 = *reinterpret_cast<const float4*>(psm + cur.cs1 + b * 4);
            if (KIND == kGU) xu = *reinterpret_cast<const float4*>(psm + xe + b * 4);
          }
          if ((j & 1) == 0) {  // the scales of blocks j and j + 1, rows g and g + 8
            f_lo = __half22float2(*reinterpret_cast<const __half2*>(&slo[j >> 1]));
            f_hi = __half22float2(*reinterpret_cast<const __half2*>(&shi[j >> 1]));
          }
          const uint4 xv =
              cur.has ? *reinterpret_cast<const uint4*>(psm + cur.xrow + b * kQBlock * 2) : make_uint4(0, 0, 0, 0);
          const int jj = j & 3;
          const float ca = jj == 0 ? c0.x : jj == 1 ? c0.y : jj == 2 ? c0.z : c0.w;
          const float cb = jj == 0 ? c1.x : jj == 1 ? c1.y : jj == 2 ? c1.z : c1.w;
          float dd[4];
          const uint32_t wl = qlo[j >> 1], wh = qhi[j >> 1];
          block_mma_q2(dd, (j & 1) ? (wl >> 16) : (wl & 0xFFFFu), (j & 1) ? (wh >> 16) : (wh & 0xFFFFu), xv, ca, cb);
          float s_lo = (j & 1) ? f_lo.y : f_lo.x;
          float s_hi = (j & 1) ? f_hi.y : f_hi.x;
          if (KIND == kGU) {
            const float u = jj == 0 ? xu.x : jj == 1 ? xu.y : jj == 2 ? xu.z : xu.w;
            s_lo *= u;
            s_hi *= u;
          }
          acc[0] = fmaf(s_lo, dd[0], acc[0]);
          acc[1] = fmaf(s_lo, dd[1], acc[1]);
          acc[2] = fmaf(s_hi, dd[2], acc[2]);
          acc[3] = fmaf(s_hi, dd[3], acc[3]);
        }
      }
      // group G + kQ2Ahead goes to position q, its scales into the slot this group's scales
      // occupied (every lane has read them)
      __syncwarp();
      const long long Gl = G + kQ2Ahead;
      if (Gl < G1) {
        const int tn = (int)(Gl / gpt);
        if (tn != tl) {
          tl = tn;
          la = tl == t ? cur : make_task<KIND, 1>(A, items, rowtok, sx, sc, tl, lane);
        }
        q2_request(la, dhi, (int)(Gl - (long long)tl * gpt), ring.lo[q], ring.hi[q], sring_w, (int)(Gl % kQ2Ahead),
                   lane);
      } else {
        cp_async_commit();
      }
      if (gs == gpt - 1 || G + 1 == G1) {
        // the task ends in this range: finish it, or publish this part of a cut task
        if (cur.valid) {
          const long long t0 = (long long)t * gpt;
          const bool first = G0 <= t0, last = G1 >= t0 + gpt;
          bool finish = true;
          if (!(first && last)) {
            const int my = first ? 0 : 1;
            float4* slot_p = reinterpret_cast<float4*>(part + ((size_t)t * 2 + my) * 128);
            slot_p[lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
            __threadfence();
            __syncwarp();
            int second = 0;
            if (lane == 0) {
              second = atomicAdd(cnt + t, 1) == 1;
              if (second) cnt[t] = 0;  // both parts are in: the counter is free for the next launch
            }
            finish = __shfl_sync(0xFFFFFFFFu, second, 0) != 0;
            if (finish) {
              __threadfence();
              const float4 p0 = __ldcg(reinterpret_cast<const float4*>(part + (size_t)t * 2 * 128) + lane);
              const float4 p1 = __ldcg(reinterpret_cast<const float4*>(part + ((size_t)t * 2 + 1) * 128) + lane);
              acc[0] = p0.x + p1.x;
              acc[1] = p0.y + p1.y;
              acc[2] = p0.z + p1.z;
              acc[3] = p0.w + p1.w;
            }
          }
          if (finish) p_epilogue<KIND>(A, X, cur, hexp, lane, acc, s_done);
        }
        acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
        if (G + 1 < G1) {
          t = (int)((G + 1) / gpt);
          cur = tl == t ? la : make_task<KIND, 1>(A, items, rowtok, sx, sc, t, lane);
        }
      }
    }
  }
}

// End of every CTA: the last CTA to finish puts the counters back to zero for the next launch
// (per-item tasks done, row maxima, the exit counter itself; all stream-K counters too if a
// CTA abandoned its work, which leaves some of them unpaired). A stream-K counter is otherwise
// reset by the warp that finishes its task.
__device__ __forceinline__ void p_exit(const FfnArgs& A, const PAux& X, int rows, int items_max, int tid) {
  __shared__ int s_last;
  __syncthreads();  // every thread of this CTA is done with the counters
  if (tid == 0) {
    __threadfence();
    s_last = atomicAdd(X.exit, 1) == (int)gridDim.x - 1;
    if (s_last) __threadfence();
  }
  __syncthreads();
  if (!s_last) return;
  for (int i = tid; i < items_max; i += kPThreads) X.item_done[i] = 0;
  for (int r = tid; r < rows; r += kPThreads) X.hmax[r] = 0u;
  if (__ldcg(X.exit + 1))
    for (size_t i = tid; i < 2 * X.cnt_stride; i += kPThreads) X.task_cnt[i] = 0;
  __syncthreads();
  if (tid == 0) {
    X.exit[0] = 0;
    X.exit[1] = 0;
  }
}

template <int DG, int DD, int FMT>
__global__ void __launch_bounds__(kPThreads, 1) ffn_persist_kernel(FfnArgs A, PAux X) {
  constexpr float kOff = FMT == 1 ? kOffsetQ2 : kOffset;  // MMA offset of a code (1024 + c or 1152 + q)
  extern __shared__ __align__(16) uint8_t psm[];
  __shared__ int s_ok;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_trigger();  // the combine may launch; it waits for this grid before reading y_perm
  const int T = A.T, d = A.d, f = A.f;
  const int rows = A.P + T * A.n_shared;
  const int items_max = (A.P < A.E ? A.P : A.E) + A.n_shared;
  const PLayout Lo = p_layout<DG, DD, FMT>(T, d, f, items_max, rows, X.rows_cap);
  ItemRec* items = reinterpret_cast<ItemRec*>(psm + Lo.items);
  int* s_done = reinterpret_cast<int*>(psm + Lo.done);
  int* rowtok = reinterpret_cast<int*>(psm + Lo.rowtok);
  int* hexp = reinterpret_cast<int*>(psm + Lo.hexp);
  float* xe = reinterpret_cast<float*>(psm + Lo.xe);
  uint32_t* bmax = reinterpret_cast<uint32_t*>(psm + Lo.bmax);
  const int dmax = DG > DD ? DG : DD;
  const int n_sslot = FMT == 1 ? 4 : 2;  // scale slots per warp
  const uint32_t sring_w = smem_u32(psm + Lo.sring) + (uint32_t)warp * n_sslot * 16u * dmax * 2u;
  const uint16_t* sring_p = reinterpret_cast<const uint16_t*>(psm + Lo.sring) + (size_t)warp * n_sslot * 16 * dmax;
  const int nbd = d / kQBlock, nbf = f / kQBlock;

  // ---- phase 0 --------------------------------------------------------------------------
  // Before the kernel's inputs from the bucketing kernel are complete (programmatic dependent
  // launch: this grid may start while that kernel runs): x to f16 in shared memory, with one
  // power of two per block over all tokens. x was written by a kernel that has completed: the
  // kernel before this one lets it launch only after its own wait, which returns once every
  // kernel before that one has completed. (CTAs start at different blocks, so they do not all
  // read the same lines.)
  const int rot = (int)((blockIdx.x * 7u) % (uint32_t)nbd);
  const bool xmine = tid < T * nbd;
  const int xb = (tid / T + rot) % nbd, xt = tid % T;
  const uint32_t o_sx = Lo.act, o_scx = Lo.act + (uint32_t)T * act_stride(d);
  {
    float xv[kQBlock];
    if (xmine) load_bf16_block(static_cast<const uint16_t*>(A.x) + (size_t)xt * d + xb * kQBlock, xv);
    for (int b = tid; b < nbd; b += kPThreads) bmax[b] = 0u;
    __syncthreads();
    if (xmine) {
      float m = 0.0f;
#pragma unroll
      for (int q = 0; q < kQBlock; ++q) m = fmaxf(m, fabsf(xv[q]));
      atomicMax(bmax + xb, __float_as_uint(m));
    }
    __syncthreads();
    if (xmine) {
      const int e = f16_exp_for(__uint_as_float(bmax[xb]));
      const float down = pow2f(-e);
#pragma unroll
      for (int q = 0; q < kQBlock; ++q) xv[q] *= down;
      *reinterpret_cast<float*>(psm + o_scx + (size_t)xt * sum_stride(d) + xb * 4) =
          stage_block_f16(psm + o_sx + (size_t)xt * act_stride(d), xb, xv, kOff);
      if (xt == 0) xe[xb] = pow2f(e);
    }
  }
  pdl_wait();  // the active list, offsets and sorted pairs of this layer (and the slot table)

  // work items (row span kept even for an expert with no slot), row tokens
  const int n_active = A.active[0];
  const int n_items = n_active + A.n_shared;
  for (int i = tid; i < items_max; i += kPThreads) {
    ItemRec rec{};
    if (i < n_active) {
      const int e = A.active[1 + i];
      const int s = A.slot_of[e];
      rec.row0 = A.offsets[e];
      rec.ntok = A.offsets[e + 1] - rec.row0;
      rec.slot = s;
      if (s < 0) flag_status(A.status, MOE_DEV_MISSING_SLOT_BIT);
      else if ((uint64_t)s >= A.n_slots) flag_status(A.status, MOE_DEV_BAD_SLOT_BIT);
      else rec.rec = A.pool + (uint64_t)s * A.slot_bytes;
    } else if (i < n_items) {
      const int sh = i - n_active;
      rec.rec = A.shared + (uint64_t)sh * A.slot_bytes;
      rec.row0 = A.P + sh * T;
      rec.ntok = T;
      rec.slot = sh;
      rec.shared = 1;
    }
    items[i] = rec;
    s_done[i] = 0;
  }
  for (int r = tid; r < rows; r += kPThreads) rowtok[r] = r < A.P ? A.sorted_pair[r] / A.k : (r - A.P) % T;
  __syncthreads();  // items, row tokens and the staged x are visible to every warp

  const int n_warps = gridDim.x * kPW, wid = blockIdx.x * kPW + warp;
  long long G0, G1;
  const int gpt_gu = nbd / DG;
  warp_range(n_items * (f / 8), gpt_gu, wid, n_warps, &G0, &G1);
  Ring<DG, FMT> rg;
  int slot = 0;
  if constexpr (FMT == 1) {
    q2_prime<kGU>(A, items, rowtok, o_sx, o_scx, G0, G1, gpt_gu, rg, sring_w, lane);
  } else {
    if (G0 < G1) {
      const PTask p = make_task<kGU, FMT>(A, items, rowtok, o_sx, o_scx, (int)(G0 / gpt_gu), lane);
      issue_group<DG, FMT>(p, hi_delta<kGU, FMT>(A), (int)(G0 % gpt_gu), rg, sring_w, slot, lane);
    }
    cp_async_commit();
  }

  // ---- phase 1: gate/up ----------------------------------------------------------------
  if constexpr (FMT == 1)
    p_stream_q2<kGU>(A, X, psm, items, rowtok, o_sx, o_scx, Lo.xe, hexp, sring_w, sring_p, G0, G1, gpt_gu, rg, lane,
                     s_done);
  else
    p_stream<kGU, DG, FMT>(A, X, psm, items, rowtok, o_sx, o_scx, Lo.xe, hexp, sring_w, sring_p, G0, G1, gpt_gu, rg,
                           slot, lane, s_done);

  // ---- phase 2: publish this CTA's gate/up work; first down loads; wait for this CTA's
  // items; their h rows to f16 -------------------------------------------------------------
  // (every thread fences its own h writes and row maxima; no weight load is in flight now)
  __threadfence();
  __syncthreads();
  for (int i = tid; i < items_max; i += kPThreads)
    if (s_done[i] > 0) atomicAdd(X.item_done + i, s_done[i]);
  const int gpt_dn = nbf / DD;
  const int n_dn = n_items * (d / 16);
  warp_range(n_dn, gpt_dn, wid, n_warps, &G0, &G1);
  // the items this CTA's down work covers, and their rows [r_lo, r_hi)
  long long C0, C1, tmp;
  const int w_first = blockIdx.x * kPW;
  const int nw_dn = n_warps < n_dn ? n_warps : n_dn;
  const int w_last = w_first + kPW - 1 < nw_dn - 1 ? w_first + kPW - 1 : nw_dn - 1;
  warp_range(n_dn, gpt_dn, w_first, n_warps, &C0, &tmp);
  warp_range(n_dn, gpt_dn, w_last, n_warps, &tmp, &C1);
  const bool cta_dn = w_first < nw_dn && C0 < C1;
  const int tpi_dn = d / 16;
  const int i_lo = cta_dn ? (int)(C0 / gpt_dn) / tpi_dn : 0;
  const int i_hi = cta_dn ? (int)((C1 - 1) / gpt_dn) / tpi_dn : -1;
  const int r_lo = cta_dn ? items[i_lo].row0 : 0;
  const int r_hi = cta_dn ? items[i_hi].row0 + items[i_hi].ntok : 0;
  const uint32_t o_sh = Lo.act - (uint32_t)r_lo * act_stride(f);
  const uint32_t o_sch = Lo.act + (uint32_t)X.rows_cap * act_stride(f) - (uint32_t)r_lo * sum_stride(f);
  Ring<DD, FMT> rd;
  __syncwarp();
  if constexpr (FMT == 1) {
    q2_prime<kDN>(A, items, rowtok, o_sh, o_sch, G0, G1, gpt_dn, rd, sring_w, lane);
  } else {
    if (G0 < G1) {
      const PTask p = make_task<kDN, FMT>(A, items, rowtok, o_sh, o_sch, (int)(G0 / gpt_dn), lane);
      issue_group<DD, FMT>(p, hi_delta<kDN, FMT>(A), (int)(G0 % gpt_dn), rd, sring_w, slot, lane);
    }
    cp_async_commit();
  }
  if (tid == 0) {
    int ok = r_hi - r_lo <= X.rows_cap;
    const uint64_t t0 = globaltimer_ns();
    const int need = f / 8;  // gate/up tasks per item
    for (int i = i_lo; ok && i <= i_hi; ++i) {
      if (items[i].rec == nullptr || items[i].ntok <= 0) continue;  // never computed
      for (uint32_t k = 0;; ++k) {
        int v;
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(X.item_done + i) : "memory");
        if (v >= need) break;
        if ((k & 15u) == 15u && globaltimer_ns() - t0 > A.wait_ns) {
          ok = 0;
          break;
        }
      }
    }
    s_ok = ok;
  }
  __syncthreads();  // also: every warp of this CTA is past gate/up, so the x rows may be overwritten
  if (!s_ok) {
    if (tid == 0) {
      flag_status(A.status, MOE_DEV_TIMEOUT_BIT);
      atomicExch(X.exit + 1, 1);  // stream-K counters of this CTA's down tasks stay unpaired
    }
    cp_async_wait_all();
    p_exit(A, X, rows, items_max, tid);
    return;
  }
  for (int r = r_lo + tid; r < r_hi; r += kPThreads) hexp[r] = f16_exp_for(__uint_as_float(__ldcg(X.hmax + r)));
  __syncthreads();
  for (int i = tid; i < (r_hi - r_lo) * nbf; i += kPThreads) {
    const int r = r_lo + i / nbf, b = i % nbf;
    const float down = pow2f(-hexp[r]);
    const float4* src = reinterpret_cast<const float4*>(A.h + (size_t)r * f + b * kQBlock);
    float v[kQBlock];
#pragma unroll
    for (int q = 0; q < kQBlock / 4; ++q) {
      const float4 w4 = __ldcg(src + q);
      v[4 * q] = w4.x * down;
      v[4 * q + 1] = w4.y * down;
      v[4 * q + 2] = w4.z * down;
      v[4 * q + 3] = w4.w * down;
    }
    // staged row r sits at (o_sh + r * stride) mod 2^32, i.e. (r - r_lo) strides into the region
    *reinterpret_cast<float*>(psm + (uint32_t)(o_sch + (uint32_t)r * sum_stride(f)) + b * 4) =
        stage_block_f16(psm + (uint32_t)(o_sh + (uint32_t)r * act_stride(f)), b, v, kOff);
  }
  __syncthreads();

  // ---- phase 3: down -------------------------------------------------------------------
  if constexpr (FMT == 1)
    p_stream_q2<kDN>(A, X, psm, items, rowtok, o_sh, o_sch, 0u, hexp, sring_w, sring_p, G0, G1, gpt_dn, rd, lane,
                     s_done);
  else
    p_stream<kDN, DD, FMT>(A, X, psm, items, rowtok, o_sh, o_sch, 0u, hexp, sring_w, sring_p, G0, G1, gpt_dn, rd,
                           slot, lane, s_done);
  cp_async_wait_all();
  p_exit(A, X, rows, items_max, tid);
}

int persist_rows_cap(const FfnArgs& a, int sm_count) {
  const int rows = a.P + a.T * a.n_shared;
  const int items_max = (a.P < a.E ? a.P : a.E) + a.n_shared;
  return p_rows_cap(a.T, a.d, items_max, rows, sm_count * kPW);
}

template <int DG, int DD, int FMT>
cudaError_t launch_persist_d(const FfnArgs& a, const PersistAux& x, int n_ctas, cudaStream_t st, bool pdl) {
  const int rows = a.P + a.T * a.n_shared;
  const int items_max = (a.P < a.E ? a.P : a.E) + a.n_shared;
  const int rows_cap = persist_rows_cap(a, n_ctas);
  const PLayout L = p_layout<DG, DD, FMT>(a.T, a.d, a.f, items_max, rows, rows_cap);
  const void* fn = (const void*)ffn_persist_kernel<DG, DD, FMT>;
  cudaError_t e = ensure_dynamic_smem(fn, L.total);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ffn_persist_kernel<DG, DD, FMT>, kPThreads, L.total);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  PAux px{x.part, x.task_cnt, x.hmax, x.item_done, x.part_stride, x.cnt_stride, rows_cap, x.exit};
  // One CTA per SM, n_ctas <= the SM count (the occupancy check above: a CTA takes every
  // register of its SM). With pdl,
  // a programmatic dependent of the bucketing kernel the caller enqueued just before: the CTAs
  // stage x while the bucketing runs and wait for its outputs (griddepcontrol.wait); every CTA's
  // waits for other CTAs are bounded. Otherwise a cooperative launch, which guarantees that all
  // CTAs are resident at once.
  if (pdl) return launch_pdl(ffn_persist_kernel<DG, DD, FMT>, dim3(n_ctas), dim3(kPThreads), L.total, st, a, px);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_ctas);
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = L.total;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, ffn_persist_kernel<DG, DD, FMT>, a, px);
}

}  // namespace

size_t persist_smem_bytes(const FfnArgs& a, int sm_count) {
  const int rows = a.P + a.T * a.n_shared;
  const int items_max = (a.P < a.E ? a.P : a.E) + a.n_shared;
  const int cap = persist_rows_cap(a, sm_count);
  return a.fmt == 1 ? p_layout<8, 8, 1>(a.T, a.d, a.f, items_max, rows, cap).total
                    : p_layout<8, 8, 0>(a.T, a.d, a.f, items_max, rows, cap).total;
}

bool persist_supported(const FfnArgs& a, int sm_count) {
  return a.xdt == 0 && a.T >= 1 && a.T <= 8 && a.d % 128 == 0 && a.f % 128 == 0 &&
         (a.fmt == 0 || (a.d % 256 == 0 && a.f % 256 == 0)) &&
         a.T * (a.d / kQBlock) <= kPThreads && persist_smem_bytes(a, sm_count) <= 200 * 1024;
}

cudaError_t launch_ffn_persist(const FfnArgs& a, const PersistAux& x, int n_ctas, cudaStream_t st, bool pdl) {
  if (a.fmt == 1) return launch_persist_d<8, 8, 1>(a, x, n_ctas, st, pdl);  // d and f multiples of 256
  const bool g8 = (a.d / kQBlock) % 8 == 0, d8 = (a.f / kQBlock) % 8 == 0;
  if (g8 && d8) return launch_persist_d<8, 8, 0>(a, x, n_ctas, st, pdl);
  if (g8) return launch_persist_d<8, 4, 0>(a, x, n_ctas, st, pdl);
  if (d8) return launch_persist_d<4, 8, 0>(a, x, n_ctas, st, pdl);
  return launch_persist_d<4, 4, 0>(a, x, n_ctas, st, pdl);
}

}  // namespace moe
