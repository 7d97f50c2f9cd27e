// Device helpers of the decode expert-FFN kernels: int8 codes to f16 MMA fragments, the
// warp-level f16 MMA of one 32-element block, and the power-of-two rescale of activations.
//
// Codes are stored in pairs of blocks (code_pos): a lane's 16-byte chunk c of a 64-code span
// holds codes 8c..8c+7 of both blocks, so each lane of an m16n8k16 MMA pair finds its 8 codes of
// a block at one 8-byte half of its chunk.
//
// Conversion. One lop3 turns two int8 codes (bytes 0 and 2 of a word, or 1 and 3 after a
// shift) into the f16 pair 1152 + q, exactly (0x64 in the high byte, q + 128 in the low byte).
// The MMA's accumulator input is set to -1152 * (sum of the block's activations), so the MMA
// returns sum_k q_k x_k: every product (1152 + q) * x is exact in fp32 and the offset cancels
// to within ~1e-6 of the result. The pairs hold elements (0, 2) and (1, 3) of each group of
// four, so activations are stored in the same order (x0 x2 x1 x3 x4 x6 x5 x7 per group of 8).
//
// Lane (g, c) = (lane / 4, lane % 4) of an m16n8k16 MMA holds M rows g and g + 8 and token
// columns 2c, 2c + 1 of the result; in MMA half hf (0, 1) of a block its k slots {2c, 2c+1,
// 2c+8, 2c+9} hold elements c*8 + hf*4 + {0, 2, 1, 3}, and the activation fragment of token g
// uses the same order, so the k permutation cancels in the sum.
#pragma once
#include "moe_common.cuh"

namespace moe {

constexpr float kOffset = 1152.0f;   // f16 code of a weight = 1152 + q

// ------------------------------------------------------------------ small helpers --------

__device__ __forceinline__ void mma_f16_16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// f16 pair (1152 + q(byte 0), 1152 + q(byte 2)) of a word of int8 codes: the low bytes xor 0x80
// under the mask, 0x64 in the high bytes (lop3 function b ? a ^ c : c).
__device__ __forceinline__ uint32_t codes02(uint32_t w) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(r) : "r"(w), "r"(0x00FF00FFu), "r"(0x64806480u));
  return r;
}

// d = C + block product of M rows g, g+8 (8 codes each: w_lo, w_hi) with this lane's 8
// activations of token g (xv: pairs (0,2), (1,3), (4,6), (5,7)), as two MMAs. C is -1152 times
// the block sums of the activations of columns 2c, 2c+1 (c0, c1).
__device__ __forceinline__ void block_mma(float* d, uint2 w_lo, uint2 w_hi, const uint4& xv, float c0, float c1) {
  // first MMA: accumulator input (c0, c1, c0, c1) read straight from c0 / c1; second: chained
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%11,%10,%11};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(codes02(w_lo.x)), "r"(codes02(w_hi.x)), "r"(codes02(w_lo.x >> 8)), "r"(codes02(w_hi.x >> 8)), "r"(xv.x),
        "r"(xv.y), "f"(c0), "f"(c1));
  mma_f16_16816(d, codes02(w_lo.y), codes02(w_hi.y), codes02(w_lo.y >> 8), codes02(w_hi.y >> 8), xv.z, xv.w);
}

// The 2-bit format (w = s (c - 1.5)). A lane's 8 codes of one row of a block are one 16-bit word
// u, code j at bits 2 * slot(j) with slot order (0, 2, 1, 3, 4, 6, 5, 7), so that the codes of
// each MMA register pair sit at bits 4r and 4r + 2 of u, r = 0..3. With t = u | (u << 14) the two
// codes of pair r are at bits 4r and 4r + 16 of t (the bits where the two copies of u overlap,
// 14 and 15, are never read), and one lop3 of t >> 4r turns them into the f16 pair
// (1024 + c_a, 1024 + c_b) exactly (0x64 in the high byte). The
// accumulator input is -1025.5 times the block sum of the activations, so the MMA returns
// sum_k (c_k - 1.5) x_k.
constexpr float kOffsetQ2 = 1025.5f;

__device__ __forceinline__ uint32_t q2pair(uint32_t t) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(t), "r"(0x00030003u), "r"(0x64006400u));  // (a & b) | c
  return r;
}

// d = C + block product of M rows g, g+8 (16-bit code words u_lo, u_hi of the 2-bit format) with
// this lane's 8 activations of token g, as two MMAs; C as in block_mma, with the offset 1025.5.
__device__ __forceinline__ void block_mma_q2(float* d, uint32_t u_lo, uint32_t u_hi, const uint4& xv, float c0,
                                             float c1) {
  const uint32_t tl = u_lo | (u_lo << 14), th = u_hi | (u_hi << 14);
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%11,%10,%11};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(q2pair(tl)), "r"(q2pair(th)), "r"(q2pair(tl >> 4)), "r"(q2pair(th >> 4)), "r"(xv.x), "r"(xv.y),
        "f"(c0), "f"(c1));
  mma_f16_16816(d, q2pair(tl >> 8), q2pair(th >> 8), q2pair(tl >> 12), q2pair(th >> 12), xv.z, xv.w);
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


__device__ __forceinline__ int n_items(const FfnArgs& A) { return A.active[0] + A.n_shared; }

// Element i of a row is stored at perm_pos(i): within each group of 4, order (0, 2, 1, 3).
__device__ __forceinline__ int perm_pos(int i) { return (i & ~3) | ((i & 1) << 1) | ((i >> 1) & 1); }

// Writes the 32 values v (one block, row order) to dst in the permuted order as f16 and
// returns -1152 * (sum of the f16 values), the MMA accumulator input of that block.
__device__ __forceinline__ float store_block_f16(__half* dst, const float* v) {
  float s = 0.0f;
#pragma unroll
  for (int i = 0; i < kQBlock; ++i) {
    const __half q = __float2half_rn(v[i]);
    dst[perm_pos(i)] = q;
    s += __half2float(q);
  }
  return -kOffset * s;
}

// 8 int8 codes of one row at p (8-byte aligned), streamed once: no L1 allocation.
__device__ __forceinline__ uint2 ld_codes(const uint8_t* p) {
  uint2 r;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}

// 16 int8 codes at p (16-byte aligned), streamed once: no L1 allocation.
__device__ __forceinline__ uint4 ld_codes16(const uint8_t* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

}  // namespace moe
