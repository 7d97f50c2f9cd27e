// Bucketing and permutation of (token, slot) pairs by expert.
//
// After the router, each token's k pairs are grouped by expert, so that an expert's weights
// are read once for all of its tokens. On the pages this is what lets the GPU compute the
// experts its cache holds ("Strata 工作原理图解GPU内存SSD三级存储如何让125B模型塞进消费级显卡",
// section "专家缓存"). The result is a stable counting sort of the flat pair ids p = t*k + j by
// expert.
//
// The design is deterministic and uses no atomics. Pairs are cut into chunks of 1024, one CTA
// per chunk. Each chunk sorts its keys (expert << 10 | local index) with a shared-memory
// bitonic network. The keys are unique, so the sort is stable by construction. Run
// lengths give the chunk's per-expert counts, a column scan over chunks gives every
// (chunk, expert) its base, and the scatter writes sorted_pair / inv_pos. When all pairs fit in
// one chunk (decode), one CTA does all of it in a single launch; up to 256 pairs it counts
// instead of sorting: each pair's rank is the number of earlier pairs of its expert, and the
// last pair of each expert writes that expert's count (one writer per expert, no atomics).
#include "bucket.cuh"

namespace moe {

constexpr int CH = kPermChunk;  // 1024

// Ascending bitonic sort of n = blockDim.x keys (a power of two), one key per thread.
__device__ __forceinline__ void bitonic_sort_block(uint32_t* keys) {
  const int i = threadIdx.x, n = blockDim.x;
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const int j = i ^ stride;
      if (j > i) {
        const uint32_t a = keys[i], b = keys[j];
        const bool up = (i & size) == 0;
        if ((a > b) == up) {
          keys[i] = b;
          keys[j] = a;
        }
      }
      __syncthreads();
    }
  }
}

// first position in keys[0..n) whose key is >= v (keys ascending)
__device__ __forceinline__ int lower_bound_u32(const uint32_t* keys, int n, uint32_t v) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (keys[mid] < v) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

__device__ __forceinline__ uint32_t load_pair_key(const int32_t* topk_idx, int p, int local, int P, int E,
                                                  int* status) {
  if (p >= P) return 0xFFFFFFFFu;
  int e = topk_idx[p];
  if (e < 0 || e >= E) {
    flag_status(status, MOE_DEV_BAD_EXPERT_BIT);
    e = e < 0 ? 0 : E - 1;  // keep every later write in bounds
  }
  return ((uint32_t)e << 10) | (uint32_t)local;
}

// All P <= 1024 pairs in one CTA of n >= P threads (a power of two, at least 32): sort,
// offsets, active list, scatter.
__global__ void __launch_bounds__(CH) bucket_single_kernel(const int32_t* __restrict__ topk_idx, int P, int E,
                                                           int32_t* __restrict__ counts,
                                                           int32_t* __restrict__ offsets,
                                                           int32_t* __restrict__ sorted_pair,
                                                           int32_t* __restrict__ inv_pos,
                                                           int32_t* __restrict__ active, int* status) {
  __shared__ uint32_t keys[CH];
  __shared__ int warp_sums[33];
  const int i = threadIdx.x;
  keys[i] = load_pair_key(topk_idx, i, i, P, E, status);
  __syncthreads();
  bitonic_sort_block(keys);
  const uint32_t key = keys[i];
  const int e = (int)(key >> 10);
  if (i < P) {
    const int p = (int)(key & 1023u);
    sorted_pair[i] = p;
    inv_pos[p] = i;
  }
  const int start = (i < P) && (i == 0 || (keys[i - 1] >> 10) != (uint32_t)e);
  int n_active = 0;
  const int rank = block_exclusive_scan(start, warp_sums, &n_active);
  if (start) active[1 + rank] = e;
  if (i == 0) active[0] = n_active;
  for (int ee = i; ee <= E; ee += blockDim.x) {
    const int lb = lower_bound_u32(keys, P, (uint32_t)ee << 10);
    offsets[ee] = lb;
    if (ee < E) counts[ee] = lower_bound_u32(keys, P, (uint32_t)(ee + 1) << 10) - lb;
  }
}

// At most 256 pairs in one CTA of n >= max(P, E) threads (a multiple of 32): the experts of
// the pairs are read into shared memory, then bucket_count_block.
__global__ void __launch_bounds__(1024) bucket_count_kernel(const int32_t* __restrict__ topk_idx, int P, int E,
                                                          int32_t* __restrict__ counts,
                                                          int32_t* __restrict__ offsets,
                                                          int32_t* __restrict__ sorted_pair,
                                                          int32_t* __restrict__ inv_pos,
                                                          int32_t* __restrict__ active, int* status) {
  __shared__ int ex[256];
  __shared__ int cs[1024];
  __shared__ int warp_sums[33];
  const int i = threadIdx.x;
  pdl_wait();  // topk_idx from the router
  // the expert FFN may launch now and stage its activations meanwhile: after the wait, so that
  // every kernel before this one has completed when it reads them
  pdl_trigger();
  if (i < P) {
    int e = topk_idx[i];
    if (e < 0 || e >= E) {
      flag_status(status, MOE_DEV_BAD_EXPERT_BIT);
      e = e < 0 ? 0 : E - 1;  // keep every later write in bounds
    }
    ex[i] = e;
  }
  bucket_count_block(ex, P, E, cs, warp_sums, counts, offsets, sorted_pair, inv_pos, active);
}

// Multi-chunk, step 1: sort each chunk; write its keys and its per-expert counts cnt[c][e].
__global__ void __launch_bounds__(CH) bucket_chunk_kernel(const int32_t* __restrict__ topk_idx, int P, int E,
                                                          uint32_t* __restrict__ chunk_keys,
                                                          int32_t* __restrict__ cnt, int* status) {
  __shared__ uint32_t keys[CH];
  const int c = blockIdx.x, i = threadIdx.x;
  const int base = c * CH;
  const int n = min(CH, P - base);
  keys[i] = load_pair_key(topk_idx, base + i, i, P, E, status);
  int32_t* row = cnt + (size_t)c * E;
  for (int ee = i; ee < E; ee += CH) row[ee] = 0;
  __syncthreads();
  bitonic_sort_block(keys);
  const uint32_t key = keys[i];
  chunk_keys[base + i] = key;  // the workspace holds C * 1024 keys
  if (i < n) {
    const uint32_t e = key >> 10;
    if (i == 0 || (keys[i - 1] >> 10) != e) row[e] = lower_bound_u32(keys, n, (e + 1) << 10) - i;
  }
}

// Multi-chunk, step 2 (one CTA): column scan of cnt over chunks, scan of totals over experts,
// active list; cnt[c][e] becomes the first output position of chunk c's pairs of expert e.
__global__ void __launch_bounds__(CH) bucket_scan_kernel(int C, int E, int32_t* __restrict__ cnt,
                                                         int32_t* __restrict__ counts,
                                                         int32_t* __restrict__ offsets,
                                                         int32_t* __restrict__ active) {
  __shared__ int warp_sums[33];
  for (int e = threadIdx.x; e < E; e += CH) {
    int run = 0;
    for (int c = 0; c < C; ++c) {
      const int v = cnt[(size_t)c * E + e];
      cnt[(size_t)c * E + e] = run;
      run += v;
    }
    counts[e] = run;
  }
  __syncthreads();
  int carry = 0, carry_active = 0;
  for (int e0 = 0; e0 < E; e0 += CH) {
    const int e = e0 + threadIdx.x;
    const int v = e < E ? counts[e] : 0;
    int tot = 0, tot_a = 0;
    const int ex = block_exclusive_scan(v, warp_sums, &tot);
    const int ar = block_exclusive_scan(v > 0 ? 1 : 0, warp_sums, &tot_a);
    if (e < E) {
      offsets[e] = carry + ex;
      for (int c = 0; c < C; ++c) cnt[(size_t)c * E + e] += carry + ex;
      if (v > 0) active[1 + carry_active + ar] = e;
    }
    carry += tot;
    carry_active += tot_a;
  }
  if (threadIdx.x == 0) {
    offsets[E] = carry;
    active[0] = carry_active;
  }
}

// Multi-chunk, step 3: scatter each chunk's sorted pairs to their final positions.
__global__ void __launch_bounds__(CH) bucket_scatter_kernel(int P, const uint32_t* __restrict__ chunk_keys,
                                                            const int32_t* __restrict__ cnt, int E,
                                                            int32_t* __restrict__ sorted_pair,
                                                            int32_t* __restrict__ inv_pos) {
  __shared__ uint32_t keys[CH];
  const int c = blockIdx.x, i = threadIdx.x;
  const int base = c * CH;
  const int n = min(CH, P - base);
  keys[i] = chunk_keys[base + i];
  __syncthreads();
  if (i < n) {
    const uint32_t key = keys[i];
    const uint32_t e = key >> 10;
    const int rank = i - lower_bound_u32(keys, n, e << 10);
    const int dest = cnt[(size_t)c * E + e] + rank;
    const int p = base + (int)(key & 1023u);
    sorted_pair[dest] = p;
    inv_pos[p] = dest;
  }
}

// The resident experts of an active list ([n, e_0, ..., e_{n-1}]), in the same order, as a list
// of the same form: the experts whose slot_of entry is >= 0. One warp, ballots in chunks of 32.
__global__ void __launch_bounds__(32) filter_resident_kernel(const int32_t* __restrict__ active,
                                                             const int32_t* __restrict__ slot_of, int E,
                                                             int32_t* __restrict__ out) {
  const int lane = threadIdx.x;
  const int n = active[0];
  int m = 0;
  for (int i0 = 0; i0 < n; i0 += 32) {
    const int i = i0 + lane;
    int e = -1;
    bool res = false;
    if (i < n) {
      e = active[1 + i];
      res = e >= 0 && e < E && slot_of[e] >= 0;
    }
    const uint32_t b = __ballot_sync(0xFFFFFFFFu, res);
    if (res) out[1 + m + __popc(b & ((1u << lane) - 1u))] = e;
    m += __popc(b);
  }
  if (lane == 0) out[0] = m;
}

cudaError_t launch_filter_resident(const int32_t* active, const int32_t* slot_of, int E, int32_t* out,
                                   cudaStream_t st) {
  filter_resident_kernel<<<1, 32, 0, st>>>(active, slot_of, E, out);
  return cudaGetLastError();
}

cudaError_t launch_permute(const moe_shape& s, const int32_t* topk_idx, int32_t* counts, int32_t* offsets,
                           int32_t* sorted_pair, int32_t* inv_pos, int32_t* active, int32_t* cnt,
                           uint32_t* keys, int* status, cudaStream_t st, bool pdl) {
  const int P = s.T * s.k;
  if (P <= 256) {
    const int need = P > s.E ? P : s.E;
    const int n = (need + 31) / 32 * 32;
    return launch_maybe_pdl(pdl, bucket_count_kernel, dim3(1), dim3(n), 0, st, topk_idx, P, s.E, counts, offsets,
                            sorted_pair,
                      inv_pos, active, status);
  }
  if (P <= CH) {
    int n = 32;
    while (n < P) n <<= 1;
    bucket_single_kernel<<<1, n, 0, st>>>(topk_idx, P, s.E, counts, offsets, sorted_pair, inv_pos, active,
                                           status);
    return cudaGetLastError();
  }
  const int C = perm_chunks(P);
  bucket_chunk_kernel<<<C, CH, 0, st>>>(topk_idx, P, s.E, keys, cnt, status);
  bucket_scan_kernel<<<1, CH, 0, st>>>(C, s.E, cnt, counts, offsets, active);
  bucket_scatter_kernel<<<C, CH, 0, st>>>(P, keys, cnt, s.E, sorted_pair, inv_pos);
  return cudaGetLastError();
}

}  // namespace moe
