// Block-level pieces of the bucketing (stable grouping of the pairs p = t*k + j by expert),
// shared by the bucketing kernels and the decode routing tail that selects and buckets in one
// CTA.
#pragma once
#include "moe_common.cuh"

namespace moe {

// Block-wide exclusive scan of one int per thread (a multiple of 32 threads, at most 1024);
// returns the total in *total.
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < (int)(blockDim.x >> 5) ? warp_sums[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xFFFFFFFFu, wi, o);
      if (lane >= o) wi += n;
    }
    warp_sums[lane] = wi - w;  // exclusive over warps
    if (lane == 31) warp_sums[32] = wi;
  }
  __syncthreads();
  const int r = warp_sums[warp] + incl - v;
  *total = warp_sums[32];
  __syncthreads();
  return r;
}

// The counting bucketing of P <= 256 pairs in one CTA of n >= max(P, E) threads (a multiple of
// 32). ex (shared memory) holds the expert of pair i for i < P, written before the call; cs
// (shared, >= E ints) and warp_sums (33 ints) are scratch. Each pair's rank is the number of
// earlier pairs of its expert, and the last pair of each expert writes that expert's count
// (one writer per expert, no atomics); one scan gives the offsets and one the active list.
__device__ __forceinline__ void bucket_count_block(const int* ex, int P, int E, int* cs, int* warp_sums,
                                                   int32_t* counts, int32_t* offsets, int32_t* sorted_pair,
                                                   int32_t* inv_pos, int32_t* active) {
  const int i = threadIdx.x;
  if (i < E) cs[i] = 0;
  __syncthreads();
  const int e = i < P ? ex[i] : 0;
  int rank = 0;
  if (i < P) {
    bool last = true;
    for (int q = 0; q < P; ++q) {
      const bool same = ex[q] == e;
      rank += (q < i && same) ? 1 : 0;
      last = last && !(q > i && same);
    }
    if (last) cs[e] = rank + 1;
  }
  __syncthreads();
  const int v = i < E ? cs[i] : 0;
  int total = 0, n_act = 0;
  const int off = block_exclusive_scan(v, warp_sums, &total);
  const int ar = block_exclusive_scan(v > 0 ? 1 : 0, warp_sums, &n_act);
  if (i < E) {
    counts[i] = v;
    offsets[i] = off;
    if (v > 0) active[1 + ar] = i;
    cs[i] = off;
  }
  if (i == 0) {
    offsets[E] = total;
    active[0] = n_act;
  }
  __syncthreads();
  if (i < P) {
    const int pos = cs[e] + rank;
    sorted_pair[pos] = i;
    inv_pos[i] = pos;
  }
}

}  // namespace moe
