// moe_permute_static: the bucketing step without a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they bucket tokens. One
// example is a host engine that plans all device memory ahead of time and does not let a
// library grow it. Another is a serving path where a cudaMalloc could stall the device or
// fragment a pool that was sized once at start-up. For them this entry point keeps the
// bucketing scratch (per-chunk expert counts and chunk-sorted keys) in one fixed device
// array of this library, sized for at most kStaticMaxPairs (token, slot) pairs.
// It runs the same kernels as moe_permute.
//
// The array lives in every GPU that loads the library until the process exits (512 KiB).
// Host code cannot use its name as a device address. The first call on each device looks
// the address up with cudaGetSymbolAddress while that device is current, and later calls
// reuse it.
#include <cstdio>
#include <mutex>

#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kStaticMaxPairs = 65536;
constexpr int kStaticMaxChunks = kStaticMaxPairs / kPermChunk;  // 64
constexpr int kStaticMaxExperts = 1024;
constexpr size_t kStaticCntWords = (size_t)kStaticMaxChunks * kStaticMaxExperts;
constexpr size_t kStaticKeyWords = (size_t)kStaticMaxChunks * kPermChunk;

// [kStaticMaxChunks][kStaticMaxExperts] int32 counts, then [kStaticMaxChunks * 1024] keys.
static __device__ __align__(256) uint32_t g_permute_scratch[kStaticCntWords + kStaticKeyWords];

// Device address of g_permute_scratch on the current device (looked up once per device).
cudaError_t scratch_address(uint32_t** out) {
  static std::mutex mu;
  static uint32_t* addr[64] = {nullptr};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_permute_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = static_cast<uint32_t*>(p);
  }
  *out = addr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

moe_status moe_permute_static(const moe_shape* shape, const int32_t* topk_idx, int32_t* counts, int32_t* offsets,
                              int32_t* sorted_pair, int32_t* inv_pos, int32_t* active, int32_t* status,
                              moe_stream_t stream) {
  size_t unused = 0;
  moe_status st = moe_workspace_size(shape, &unused);  // the common shape checks
  if (st != MOE_OK) return st;
  const long long P = (long long)shape->T * shape->k;
  if (P > kStaticMaxPairs || shape->E > kStaticMaxExperts) {
    char msg[200];
    std::snprintf(msg, sizeof(msg),
                  "moe_permute_static: %lld pairs and %d experts exceed its fixed scratch (at most %d pairs, %d "
                  "experts); use moe_permute with a workspace",
                  P, shape->E, kStaticMaxPairs, kStaticMaxExperts);
    return report_error(MOE_EUNSUPPORTED, msg);
  }
  if (!counts || !offsets || !active || !status || (shape->T > 0 && (!topk_idx || !sorted_pair || !inv_pos)))
    return report_error(MOE_EINVAL, "moe_permute_static: NULL argument");
  uint32_t* scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(status, 0, sizeof(int32_t), s);
  if (e == cudaSuccess)
    e = launch_permute(*shape, topk_idx, counts, offsets, sorted_pair, inv_pos, active,
                       reinterpret_cast<int32_t*>(scratch), scratch + kStaticCntWords, status, s);
  if (e != cudaSuccess) {
    char msg[200];
    std::snprintf(msg, sizeof(msg), "moe_permute_static: %s", cudaGetErrorString(e));
    return report_error(MOE_ECUDA, msg);
  }
  return MOE_OK;
}

}  // extern "C"
