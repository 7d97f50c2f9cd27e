// Device helpers shared by the sm_103a kernels of the MoE layer.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_internal.h"

namespace moe {

constexpr int kQBlock = 32;  // elements per int8 quantisation block

// Position of code k in a row of K int8 codes. Within each 64-code span (two blocks) the codes
// are stored as four 16-byte chunks, chunk c holding codes 8c..8c+7 of the first block and then
// 8c..8c+7 of the second: a lane that loads one 16-byte chunk gets the same 8 codes of both
// blocks, the fragment the decode kernels multiply. A trailing block without a partner (K not a
// multiple of 64) is stored as is.
__host__ __device__ __forceinline__ int code_pos(int k, int K) {
  if (k >= (K & ~63)) return k;
  return (k & ~63) | (((k >> 3) & 3) << 4) | (((k >> 5) & 1) << 3) | (k & 7);
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

// 128-bit streaming load of read-only data that is used once: no L1 allocation.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

// Four int8 codes of one 32-bit word to fp32, exactly. Each byte is offset by 128 (xor of
// the sign bit), placed in the low mantissa byte of 2^23 (0x4B0000uu = 2^23 + u), and the
// offset 2^23 + 128 is subtracted; all steps are exact.
__device__ __forceinline__ void i8x4_to_f32(uint32_t w, float* o) {
  const uint32_t u = w ^ 0x80808080u;
  o[0] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7540)) - 8388736.0f;
  o[1] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7541)) - 8388736.0f;
  o[2] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7542)) - 8388736.0f;
  o[3] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7543)) - 8388736.0f;
}

__device__ __forceinline__ void i8x16_to_f32(const uint4& w, float* o) {
  i8x4_to_f32(w.x, o);
  i8x4_to_f32(w.y, o + 4);
  i8x4_to_f32(w.z, o + 8);
  i8x4_to_f32(w.w, o + 12);
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }
// The same with the fast exponential and division intrinsics (relative error about 1e-6, far
// below the f16 rounding of h that follows): the prefill epilogue evaluates it for every element
// of h, and the accurate forms made that epilogue the GEMM's bottleneck.
__device__ __forceinline__ float silu_fast(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// Programmatic dependent launch. A kernel launched with launch_pdl may start while the kernel
// before it on the stream is still running; pdl_wait() returns once that kernel has completed
// and its memory writes are visible (at once when there is no such kernel), so it comes before
// the first read of the predecessor's outputs. pdl_trigger() lets the next such kernel launch.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// A kernel is launched as a programmatic dependent only when the library enqueued the kernel
// before it on the stream in the same call: with anything else between them (a memset, a copy,
// an event wait) the early start could read inputs that are not there yet. launch_maybe_pdl
// launches normally when `pdl` is false.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

template <typename... KArgs, typename... Args>
cudaError_t launch_maybe_pdl(bool pdl, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                             Args... args) {
  if (pdl) return launch_pdl(kernel, grid, block, smem, st, args...);
  kernel<<<grid, block, smem, st>>>(static_cast<KArgs>(args)...);
  return cudaGetLastError();
}

__device__ __forceinline__ void flag_status(int* status, int bit) {
  // error reporting only (rare path); bits from several threads must all survive
  atomicOr(status, bit);
}

// Load element i of activations stored as bf16 or fp32.
__device__ __forceinline__ float load_act(const void* x, int xdt, size_t i) {
  return xdt == 0 ? bf16_bits_to_f32(static_cast<const uint16_t*>(x)[i]) : static_cast<const float*>(x)[i];
}

// One work item of the expert FFN: a routed expert from the active list, or a shared expert.
struct FfnItem {
  const uint8_t* rec;  // expert record
  int row0;            // first y_perm / h row of this expert
  int ntok;            // rows (tokens) of this expert
  int routed;          // 1: tokens come from sorted_pair; 0: shared expert, tokens 0..T-1
  int slot;            // pool slot (routed) or shared-expert index
};

__device__ __forceinline__ bool resolve_item(int a, const FfnArgs& A, FfnItem* it) {
  const int n_active = A.active[0];
  if (a < n_active) {
    const int e = A.active[1 + a];
    const int s = A.slot_of[e];
    if (s < 0) {
      flag_status(A.status, MOE_DEV_MISSING_SLOT_BIT);
      return false;
    }
    if ((uint64_t)s >= A.n_slots) {
      flag_status(A.status, MOE_DEV_BAD_SLOT_BIT);
      return false;
    }
    it->rec = A.pool + (uint64_t)s * A.slot_bytes;
    it->slot = s;
    it->row0 = A.offsets[e];
    it->ntok = A.offsets[e + 1] - A.offsets[e];
    it->routed = 1;
    return it->ntok > 0;
  }
  const int sh = a - n_active;
  if (sh < A.n_shared) {
    it->rec = A.shared + (uint64_t)sh * A.slot_bytes;
    it->slot = sh;
    it->row0 = A.P + sh * A.T;
    it->ntok = A.T;
    it->routed = 0;
    return A.T > 0;
  }
  return false;
}

__device__ __forceinline__ int item_token(const FfnArgs& A, const FfnItem& it, int i) {
  return it.routed ? A.sorted_pair[it.row0 + i] / A.k : i;
}

}  // namespace moe
