// Device implementation of the seeded expert-record generator of synth/__init__.py.
//
// Input preparation only: it fills expert records with the same bytes as the numpy
// generator (SplitMix64 counter stream -> Irwin-Hall(4) normal -> block-32 int8 + fp16
// quantiser), so that large workloads (hundreds of experts per layer, tens of layers) can
// be made in place on the device. Every floating-point step is a single IEEE operation
// with round-to-nearest (no contraction), as in the numpy version. None of the MoE
// layer's arithmetic is here.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ull;

__host__ __device__ inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__host__ __device__ inline uint64_t stream_key(uint64_t seed, uint64_t tag, uint64_t a, uint64_t b) {
  return mix64(mix64(seed) + ((tag << 48) ^ (a << 24) ^ b));
}

struct Section {
  uint64_t q_off, s_off;  // byte offsets in the record
  int rows, cols;         // stored array [rows][cols], blocks of 32 along cols
  int tag;
};

struct FillArgs {
  uint64_t seed;
  int layer, expert0, n_experts;
  int fmt;  // 0: int8 codes; 1: 2-bit codes of w = s (c - 1.5), 4 per byte
  float sigma;
  uint8_t* dst;
  uint64_t stride;
  Section sec[3];
  uint64_t blocks_per_expert, blocks_sec[3];
};

__global__ void fill_records_kernel(FillArgs a) {
  const uint64_t warp = (blockIdx.x * (uint64_t)blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= a.blocks_per_expert * (uint64_t)a.n_experts) return;
  const int ex = (int)(warp / a.blocks_per_expert);
  uint64_t b = warp % a.blocks_per_expert;
  int si = 0;
  while (b >= a.blocks_sec[si]) {
    b -= a.blocks_sec[si];
    ++si;
  }
  const Section s = a.sec[si];
  const int bpr = s.cols / 32;
  const uint64_t row = b / bpr, bc = b % bpr;
  const uint64_t i = row * s.cols + bc * 32 + lane;
  const int expert = a.expert0 + ex;
  const uint64_t key = stream_key(a.seed, s.tag, a.layer, expert);
  const uint64_t r = mix64(key + (i + 1) * kGolden);
  const int sum = (int)(r & 0xFFFF) + (int)((r >> 16) & 0xFFFF) + (int)((r >> 32) & 0xFFFF) + (int)(r >> 48);
  const float zscale = __uint_as_float(0x37DDB3D7u);  // fp32(sqrt 3) * 2^-16
  const float z = __fmul_rn(__int2float_rn(sum - 131070), zscale);
  const float w = __fmul_rn(z, a.sigma);
  const unsigned amax_bits = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(fabsf(w)));
  const float amax = __uint_as_float(amax_bits);
  uint8_t* rec = a.dst + (uint64_t)ex * a.stride;
  if (a.fmt == 1) {
    // 2-bit format: s = fp16(amax / 1.5), c = clamp(rint(w / s + 1.5), 0, 3); stored as in
    // synth.pack_codes_q2: per group of 8 blocks (64 bytes), 16-byte chunk q holds for each block
    // b one 16-bit word of codes 8q..8q+7, code j at bits 2 * slot(j), slot = (0 2 1 3 4 6 5 7)
    const __half s16 = __float2half_rn(__fdiv_rn(amax, 1.5f));
    const float sf = __half2float(s16);
    float cf = 0.0f;
    if (sf != 0.0f) cf = fminf(fmaxf(rintf(__fadd_rn(__fdiv_rn(w, sf), 1.5f)), 0.0f), 3.0f);
    const int j = lane & 7, q = lane >> 3;
    const int slot = (j & 4) | ((j & 1) << 1) | ((j >> 1) & 1);
    unsigned word = ((unsigned)(int)cf) << (2 * slot);
    word |= __shfl_xor_sync(0xFFFFFFFFu, word, 1);
    word |= __shfl_xor_sync(0xFFFFFFFFu, word, 2);
    word |= __shfl_xor_sync(0xFFFFFFFFu, word, 4);
    if (j == 0) {
      const uint64_t group = bc / 8, blk = bc % 8;
      uint8_t* rowp = rec + s.q_off + row * (uint64_t)(s.cols / 4);
      *reinterpret_cast<uint16_t*>(rowp + group * 64 + q * 16 + blk * 2) = (uint16_t)word;
    }
    if (lane == 0) reinterpret_cast<__half*>(rec + s.s_off)[row * bpr + bc] = s16;
    return;
  }
  const __half s16 = __float2half_rn(__fdiv_rn(amax, 127.0f));
  const float sf = __half2float(s16);
  float qf = 0.0f;
  if (sf != 0.0f) qf = fminf(fmaxf(rintf(__fdiv_rn(w, sf)), -127.0f), 127.0f);
  // stored order of a code row: in each 64-code span, chunk c (16 bytes) holds codes 8c..8c+7
  // of the first block and then of the second; a trailing unpaired block stays as it is
  const int k = (int)(bc * 32 + lane), K = s.cols;
  const int pos = k >= (K & ~63) ? k : ((k & ~63) | (((k >> 3) & 3) << 4) | (((k >> 5) & 1) << 3) | (k & 7));
  reinterpret_cast<int8_t*>(rec + s.q_off)[row * (uint64_t)s.cols + pos] = (int8_t)(int)qf;
  if (lane == 0) reinterpret_cast<__half*>(rec + s.s_off)[row * bpr + bc] = s16;
}

uint64_t align256(uint64_t n) { return (n + 255) & ~(uint64_t)255; }

}  // namespace

extern "C" {

// Fills records of experts expert0 .. expert0+n_experts-1 of `layer` at dst + j * stride
// (device memory), in the record layout gate_q, up_q, down_q, gate_s, up_s, down_s with
// 256-byte aligned sections; fmt 0: int8 codes, fmt 1: the 2-bit format (d and f multiples of
// 256). Returns 0 or a cudaError_t code.
int synth_fill_expert_records_fmt(uint64_t seed, int layer, int expert0, int n_experts, int d, int f, float sigma,
                                  void* dst, uint64_t stride, int fmt, void* stream) {
  if (d % 32 || f % 32 || n_experts < 0 || !dst || (fmt != 0 && fmt != 1)) return (int)cudaErrorInvalidValue;
  if (fmt == 1 && (d % 256 || f % 256)) return (int)cudaErrorInvalidValue;
  if (n_experts == 0) return 0;
  const uint64_t qn = (uint64_t)f * d, q = fmt == 1 ? qn / 4 : qn;
  const uint64_t sgu = (uint64_t)f * (d / 32) * 2, sd = (uint64_t)d * (f / 32) * 2;
  const uint64_t o_gq = 0, o_uq = align256(q), o_dq = o_uq + align256(q), o_gs = o_dq + align256(q);
  const uint64_t o_us = o_gs + align256(sgu), o_ds = o_us + align256(sgu);
  FillArgs a;
  a.seed = seed;
  a.layer = layer;
  a.expert0 = expert0;
  a.n_experts = n_experts;
  a.fmt = fmt;
  a.sigma = sigma;
  a.dst = static_cast<uint8_t*>(dst);
  a.stride = stride;
  a.sec[0] = Section{o_gq, o_gs, f, d, 1};
  a.sec[1] = Section{o_uq, o_us, f, d, 2};
  a.sec[2] = Section{o_dq, o_ds, d, f, 3};
  a.blocks_sec[0] = a.blocks_sec[1] = a.blocks_sec[2] = qn / 32;
  a.blocks_per_expert = 3 * (qn / 32);
  const uint64_t threads = a.blocks_per_expert * (uint64_t)n_experts * 32;
  const unsigned grid = (unsigned)((threads + 255) / 256);
  fill_records_kernel<<<grid, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(a);
  return (int)cudaGetLastError();
}

int synth_fill_expert_records(uint64_t seed, int layer, int expert0, int n_experts, int d, int f, float sigma,
                              void* dst, uint64_t stride, void* stream) {
  return synth_fill_expert_records_fmt(seed, layer, expert0, n_experts, d, f, sigma, dst, stride, 0, stream);
}

}  // extern "C"
