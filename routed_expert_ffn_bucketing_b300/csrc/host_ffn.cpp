// Expert FFN of missed experts on the host CPU: the bandwidth split of the miss path.
//
// The pages' engine divides the experts a layer misses between the two ways of bringing them to
// the token: some are copied over PCIe into the VRAM cache, the others are computed where their
// weights already are, in host RAM, so that PCIe and the host's memory bandwidth work at once
// ("Strata 工作原理图解GPU内存SSD三级存储如何让125B模型塞进消费级显卡", section "专家缓存"; the
// share that goes over PCIe is the --pcie-frac setting of "Strata 性能基准与论文导读125B MoE在消费级
// 硬件上的极限测量与瓶颈分析", section "如何测量"). This file is the host half: for each expert given,
// the SwiGLU FFN of its tokens computed from its pinned record, y = W_d (silu(W_g x) * (W_u x)),
// with W = q * s per block of 32 (int8 codes) or W = s * (c - 1.5) (2-bit codes), in fp32.
//
// The records are read in their stored order (see moe_get_record_layout). For int8 codes the
// activations are placed in that order once, and each row is a sum of 8-code pieces, each scaled
// by its block's scale (AVX2 when the CPU has it). A 2-bit row is expanded to fp32 first (exact:
// a level times an fp16 scale). OpenMP threads share the rows: first every gate/up row of every
// expert, then every down row.
#include <immintrin.h>
#include <omp.h>

#include <cmath>
#include <cstdio>
#include <cstring>
#include <vector>

#include "moe_internal.h"

namespace {

// IEEE binary16 to binary32, exactly (normal, subnormal, zero, inf and NaN).
inline float half_to_float(uint16_t h) {
  const uint32_t sign = (uint32_t)(h & 0x8000u) << 16;
  const uint32_t exp = (h >> 10) & 0x1Fu, man = h & 0x3FFu;
  uint32_t bits;
  if (exp == 0) {
    if (man == 0) {
      bits = sign;
    } else {  // subnormal: man * 2^-24
      const float v = (float)man * 5.9604644775390625e-08f;
      std::memcpy(&bits, &v, 4);
      bits |= sign;
    }
  } else if (exp == 31) {
    bits = sign | 0x7F800000u | (man << 13);
  } else {
    bits = sign | ((exp + 112u) << 23) | (man << 13);
  }
  float f;
  std::memcpy(&f, &bits, 4);
  return f;
}

inline float bf16_to_float(uint16_t b) {
  const uint32_t bits = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &bits, 4);
  return f;
}

// Row of K weights from the 2-bit format: per group of 8 blocks (256 codes, 64 bytes), chunk qc
// (16 bytes) holds for block b one little-endian 16-bit word with codes 8qc..8qc+7 of block b,
// code j at bits 2 * slot(j), slot order 0, 2, 1, 3, 4, 6, 5, 7. W = s * (c - 1.5).
void expand_row_q2(const uint8_t* q, const uint16_t* s, int K, float* w) {
  static const int kSlot[8] = {0, 2, 1, 3, 4, 6, 5, 7};
  for (int g = 0; g < K / 256; ++g)
    for (int qc = 0; qc < 4; ++qc)
      for (int b = 0; b < 8; ++b) {
        const uint8_t* p = q + g * 64 + qc * 16 + b * 2;
        const uint32_t word = (uint32_t)p[0] | ((uint32_t)p[1] << 8);
        const int blk = g * 8 + b;
        const float sc = half_to_float(s[blk]);
        for (int j = 0; j < 8; ++j) {
          const int c = (word >> (2 * kSlot[j])) & 3;
          w[blk * 32 + 8 * qc + j] = sc * ((float)c - 1.5f);
        }
      }
}

__attribute__((target_clones("avx2", "default"))) float dot(const float* a, const float* b, int n) {
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  int i = 0;
  for (; i + 8 <= n; i += 8)
    for (int l = 0; l < 8; ++l) acc[l] += a[i + l] * b[i + l];
  float s = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
  for (; i < n; ++i) s += a[i] * b[i];
  return s;
}

// Stored position of element i of an int8 code row of K codes (the paired-block order).
inline int i8_pos(int i, int K) {
  const int K64 = K / 64 * 64;
  if (i >= K64) return i;
  return (i & ~63) | (((i >> 3) & 3) << 4) | (((i >> 5) & 1) << 3) | (i & 7);
}

// out[t] = sum_i W[i] * xp[t][i] for one int8 row (K stored codes q, K/32 fp16 scales s) and ntok
// activation rows xp already in the stored order (row stride ldx). In a 64-code span the 8-code
// pieces alternate between the span's two blocks, so each piece is scaled by its block's scale and
// accumulated 8 lanes wide; a trailing unpaired block is stored in order.
void row_dots_i8_scalar(const int8_t* q, const float* sc, const float* xp, int K, int ntok, int ldx, float* out) {
  const int K64 = K / 64 * 64;
  for (int t = 0; t < ntok; ++t) {
    const float* x = xp + (size_t)t * ldx;
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int p = 0; p < K; p += 8) {
      const float v = sc[p < K64 ? (p >> 6) * 2 + ((p >> 3) & 1) : (p >> 5)];
      for (int j = 0; j < 8; ++j) acc[j] += ((float)q[p + j] * v) * x[p + j];
    }
    out[t] = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
  }
}

__attribute__((target("avx2,fma"))) void row_dots_i8_avx2(const int8_t* q, const float* sc, const float* xp, int K,
                                                          int ntok, int ldx, float* out) {
  const int K64 = K / 64 * 64;
  for (int t = 0; t < ntok; ++t) {
    const float* x = xp + (size_t)t * ldx;
    __m256 acc0 = _mm256_setzero_ps(), acc1 = _mm256_setzero_ps();
    for (int p = 0; p < K64; p += 64) {
      const __m256 v0 = _mm256_set1_ps(sc[p >> 5]), v1 = _mm256_set1_ps(sc[(p >> 5) + 1]);
      for (int c = 0; c < 64; c += 16) {
        const __m128i raw = _mm_loadu_si128(reinterpret_cast<const __m128i*>(q + p + c));
        const __m256 w0 = _mm256_cvtepi32_ps(_mm256_cvtepi8_epi32(raw));
        const __m256 w1 = _mm256_cvtepi32_ps(_mm256_cvtepi8_epi32(_mm_srli_si128(raw, 8)));
        acc0 = _mm256_fmadd_ps(_mm256_mul_ps(w0, v0), _mm256_loadu_ps(x + p + c), acc0);
        acc1 = _mm256_fmadd_ps(_mm256_mul_ps(w1, v1), _mm256_loadu_ps(x + p + c + 8), acc1);
      }
    }
    for (int p = K64; p < K; p += 8) {
      const __m256 v = _mm256_set1_ps(sc[p >> 5]);
      const __m256 w = _mm256_cvtepi32_ps(_mm256_cvtepi8_epi32(_mm_loadl_epi64(reinterpret_cast<const __m128i*>(q + p))));
      acc0 = _mm256_fmadd_ps(_mm256_mul_ps(w, v), _mm256_loadu_ps(x + p), acc0);
    }
    alignas(32) float l[8];
    _mm256_store_ps(l, _mm256_add_ps(acc0, acc1));
    out[t] = ((l[0] + l[1]) + (l[2] + l[3])) + ((l[4] + l[5]) + (l[6] + l[7]));
  }
}

void row_dots_i8(const int8_t* q, const uint16_t* s, const float* xp, int K, int ntok, int ldx, float* out,
                 float* sc) {
  for (int b = 0; b < K / 32; ++b) sc[b] = half_to_float(s[b]);
  static const bool avx2 = __builtin_cpu_supports("avx2") && __builtin_cpu_supports("fma");
  if (avx2) row_dots_i8_avx2(q, sc, xp, K, ntok, ldx, out);
  else row_dots_i8_scalar(q, sc, xp, K, ntok, ldx, out);
}

struct Job {
  const uint8_t* rec;
  int r0, ntok;
};

}  // namespace

extern "C" {

moe_status moe_host_expert_ffn(const moe_shape* shape, const void* h_x, moe_dtype xdt,
                               const void* const* h_records, const int32_t* h_experts, int32_t n_experts,
                               const int32_t* h_offsets, const int32_t* h_sorted_pair, float* h_y, int32_t format,
                               int32_t n_threads) {
  if (!shape || n_experts < 0 || (n_experts > 0 && (!h_x || !h_records || !h_experts || !h_offsets ||
                                                    !h_sorted_pair || !h_y)))
    return moe::report_error(MOE_EINVAL, "moe_host_expert_ffn: NULL argument or negative count");
  if (xdt != MOE_BF16 && xdt != MOE_F32) return moe::report_error(MOE_EINVAL, "moe_host_expert_ffn: bad x dtype");
  moe_expert_layout lay;
  const moe_status st = moe_get_record_layout(shape->d, shape->f, format, &lay);
  if (st != MOE_OK) return st;
  if (shape->T <= 0 || n_experts == 0) return MOE_OK;
  const int d = shape->d, f = shape->f, k = shape->k, E = shape->E, P = shape->T * shape->k;
  std::vector<Job> jobs;
  for (int32_t i = 0; i < n_experts; ++i) {
    const int e = h_experts[i];
    if (e < 0 || e >= E || !h_records[i]) return moe::report_error(MOE_EINVAL, "moe_host_expert_ffn: bad expert or record");
    const int r0 = h_offsets[e], r1 = h_offsets[e + 1];
    if (r0 < 0 || r1 < r0 || r1 > P) return moe::report_error(MOE_EINVAL, "moe_host_expert_ffn: bad offsets");
    if (r1 > r0) jobs.push_back(Job{static_cast<const uint8_t*>(h_records[i]), r0, r1 - r0});
  }
  // each expert's tokens as fp32 rows, and its gate/up outputs h [f][ntok]
  std::vector<size_t> xoff(jobs.size() + 1, 0), hoff(jobs.size() + 1, 0);
  for (size_t j = 0; j < jobs.size(); ++j) {
    xoff[j + 1] = xoff[j] + (size_t)jobs[j].ntok * d;
    hoff[j + 1] = hoff[j] + (size_t)jobs[j].ntok * f;
  }
  std::vector<float> xs(xoff.back()), h(hoff.back());
  const bool q2 = format == MOE_FMT_Q2;
  // int8 rows are multiplied in their stored order: the activations are placed in that order once
  for (size_t j = 0; j < jobs.size(); ++j)
    for (int t = 0; t < jobs[j].ntok; ++t) {
      const int tok = h_sorted_pair[jobs[j].r0 + t] / k;
      float* dst = xs.data() + xoff[j] + (size_t)t * d;
      for (int i = 0; i < d; ++i)
        dst[q2 ? i : i8_pos(i, d)] = xdt == MOE_BF16
                                         ? bf16_to_float(static_cast<const uint16_t*>(h_x)[(size_t)tok * d + i])
                                         : static_cast<const float*>(h_x)[(size_t)tok * d + i];
    }
  const int cb = q2 ? 4 : 1;  // codes per byte
  const int nt = n_threads > 0 ? n_threads : omp_get_max_threads();
  const long long n_gu = (long long)jobs.size() * f, n_dn = (long long)jobs.size() * d;
#pragma omp parallel num_threads(nt)
  {
    std::vector<float> wg(d), wu(d), wd(f), gv(64), uv(64), sc((d > f ? d : f) / 32);
#pragma omp for schedule(static)
    for (long long it = 0; it < n_gu; ++it) {
      const Job& jb = jobs[it / f];
      const int r = (int)(it % f);
      const uint8_t* gq = jb.rec + lay.gate_q + (size_t)r * d / cb;
      const uint8_t* uq = jb.rec + lay.up_q + (size_t)r * d / cb;
      const uint16_t* gs = reinterpret_cast<const uint16_t*>(jb.rec + lay.gate_s) + (size_t)r * (d / 32);
      const uint16_t* us = reinterpret_cast<const uint16_t*>(jb.rec + lay.up_s) + (size_t)r * (d / 32);
      const size_t j = (size_t)(it / f);
      if (q2) {
        expand_row_q2(gq, gs, d, wg.data());
        expand_row_q2(uq, us, d, wu.data());
        for (int t = 0; t < jb.ntok; ++t) {
          const float* xr = xs.data() + xoff[j] + (size_t)t * d;
          const float g = dot(wg.data(), xr, d), u = dot(wu.data(), xr, d);
          h[hoff[j] + (size_t)t * f + r] = g / (1.0f + std::exp(-g)) * u;
        }
      } else {
        for (int t0 = 0; t0 < jb.ntok; t0 += 64) {
          const int nt_ = jb.ntok - t0 < 64 ? jb.ntok - t0 : 64;
          const float* xr = xs.data() + xoff[j] + (size_t)t0 * d;
          row_dots_i8(reinterpret_cast<const int8_t*>(gq), gs, xr, d, nt_, d, gv.data(), sc.data());
          row_dots_i8(reinterpret_cast<const int8_t*>(uq), us, xr, d, nt_, d, uv.data(), sc.data());
          for (int t = 0; t < nt_; ++t)
            h[hoff[j] + (size_t)(t0 + t) * f + r] = gv[t] / (1.0f + std::exp(-gv[t])) * uv[t];
        }
      }
    }
    // (the implicit barrier of the loop above: every h is written); int8: h into the stored order
    // of the down rows' codes, one expert-token row per iteration
#pragma omp for schedule(static)
    for (long long it = 0; it < (long long)jobs.size(); ++it) {
      if (q2) continue;
      for (int t = 0; t < jobs[it].ntok; ++t) {
        float* hr = h.data() + hoff[it] + (size_t)t * f;
        for (int i = 0; i < f; ++i) wd[i8_pos(i, f)] = hr[i];
        std::memcpy(hr, wd.data(), sizeof(float) * f);
      }
    }
#pragma omp for schedule(static)
    for (long long it = 0; it < n_dn; ++it) {
      const Job& jb = jobs[it / d];
      const int c = (int)(it % d);
      const uint8_t* dq = jb.rec + lay.down_q + (size_t)c * f / cb;
      const uint16_t* ds = reinterpret_cast<const uint16_t*>(jb.rec + lay.down_s) + (size_t)c * (f / 32);
      const size_t j = (size_t)(it / d);
      if (q2) {
        expand_row_q2(dq, ds, f, wd.data());
        for (int t = 0; t < jb.ntok; ++t)
          h_y[(size_t)(jb.r0 + t) * d + c] = dot(wd.data(), h.data() + hoff[j] + (size_t)t * f, f);
      } else {
        for (int t0 = 0; t0 < jb.ntok; t0 += 64) {
          const int nt_ = jb.ntok - t0 < 64 ? jb.ntok - t0 : 64;
          row_dots_i8(reinterpret_cast<const int8_t*>(dq), ds, h.data() + hoff[j] + (size_t)t0 * f, f, nt_, f,
                      gv.data(), sc.data());
          for (int t = 0; t < nt_; ++t) h_y[(size_t)(jb.r0 + t0 + t) * d + c] = gv[t];
        }
      }
    }
  }
  return MOE_OK;
}

}  // extern "C"
