// Top-k selection (csa2_topk): "Main sparse selection: 512 entries"
// (perchy.ai, card "Full. Reindex. Reuse."); the candidate pool of 2,048 blocks
// of 8 ("a 16,384-entry candidate pool that layer 20 chose by blocks of 8",
// DeepSeek-V4.1-Flash study, lightning-indexer note).
//
// Every item gets a unique 64-bit key  (order_key(score) << 32) | ~index :
// larger key = higher score, then lower index.  Selecting the k largest keys
// therefore gives the top-k with lower-index tie-break, and a radix select over
// these keys needs no separate tie pass.
//
// Rows of up to kDirectCap items are selected by one CTA from shared memory.
// Longer rows (1M-entry Full-layer rows, 131,072-block pool rows) first go
// through a multi-CTA filter: a 4,096-bin histogram of the top 12 key bits finds
// the bin that holds the k-th key, and only items in that bin or above are kept
// as candidates (usually a few thousand).  A row whose candidates overflow the
// buffer falls back to an exact radix select straight over the score row.
#include "common.cuh"

namespace csa2 {

constexpr int kDirectCap = 16384;   // items held in shared memory by one CTA
constexpr int kCandCap = 16384;     // candidate buffer per query (filter path)
constexpr int kHistBins = 4096;     // top 12 bits of the 32-bit score key
constexpr int kMaxK = 2048;
constexpr int kTopkThreads = 1024;

struct TopkSrc {
  const float *scores;
  int64_t stride;
  const int32_t *n_valid;
  const int32_t *pool;    // [n_q][2048] block ids, or null
  int block;              // 1 or 8
  int64_t n_max;          // entries per row (Full) or 16384 (pool)
  int64_t n_items;        // items per row
};

// Key of item i of query q; false if the item is not valid.
__device__ __forceinline__ bool item_key(const TopkSrc &S, int q, int64_t i, int nv, uint64_t &key, int *status) {
  const float *row = S.scores + (int64_t)q * S.stride;
  if (S.pool != nullptr) {
    const int blk = __ldg(S.pool + (int64_t)q * kPoolBlocks + (i >> 3));
    if (blk < 0) return false;
    const int64_t j = (int64_t)blk * kBlock + (i & 7);
    if (j >= nv) {
      if ((int64_t)blk * kBlock >= S.n_max) record_error(status, CSA2_ERR_BOUNDS);
      return false;
    }
    key = ((uint64_t)order_key(__ldg(row + i)) << 32) | (uint32_t)(~(uint32_t)j);
    return true;
  }
  if (S.block == 1) {
    if (i >= nv) return false;
    key = ((uint64_t)order_key(__ldg(row + i)) << 32) | (uint32_t)(~(uint32_t)i);
    return true;
  }
  const int64_t j0 = i * kBlock;
  if (j0 >= nv) return false;
  uint32_t m = 0;
  const int64_t j1 = min((int64_t)nv, j0 + kBlock);
  for (int64_t j = j0; j < j1; j++) m = max(m, order_key(__ldg(row + j)));
  key = ((uint64_t)m << 32) | (uint32_t)(~(uint32_t)i);
  return true;
}

__device__ __forceinline__ int query_nv(const TopkSrc &S, int q, int *status) {
  int nv = __ldg(S.n_valid + q);
  const int64_t lim = S.n_max;
  if (nv < 0 || (int64_t)nv > lim) {
    record_error(status, CSA2_ERR_BOUNDS);
    nv = nv < 0 ? 0 : (int)min((int64_t)nv, lim);
  }
  return nv;
}

// ---- block-wide pieces (blockDim.x == kTopkThreads) ----
struct SelectShared {
  uint32_t hist[256];
  int digit;
  int above;
  int count;
};

// Warp 0 finds digit d with (#keys above d) < rem <= (#keys above d) + hist[d].
__device__ __forceinline__ void find_digit(SelectShared &sh, int rem) {
  const int lane = threadIdx.x & 31;
  if (threadIdx.x < 32) {
    uint32_t part = 0;
#pragma unroll
    for (int b = 0; b < 8; b++) part += sh.hist[8 * lane + b];
    // exclusive suffix sum over lanes (lanes above hold larger digits)
    uint32_t incl = part;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      uint32_t v = __shfl_down_sync(0xFFFFFFFFu, incl, o);
      if (lane + o < 32) incl += v;
    }
    const uint32_t above = incl - part;
    if (above < (uint32_t)rem && (uint32_t)rem <= incl) {
      uint32_t run = above;
      for (int b = 7; b >= 0; b--) {
        const uint32_t h = sh.hist[8 * lane + b];
        if (run + h >= (uint32_t)rem) { sh.digit = 8 * lane + b; sh.above = (int)run; break; }
        run += h;
      }
    }
  }
}

// Exact threshold T: exactly k of the n keys are >= T (requires n >= k, unique keys).
template <class Get>
__device__ uint64_t radix_threshold(Get get, int64_t n, int k, SelectShared &sh) {
  uint64_t prefix = 0, mask = 0;
  int rem = k;
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += blockDim.x) sh.hist[i] = 0;
    __syncthreads();
    for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
      uint64_t key;
      if (get(i, key) && (key & mask) == prefix) atomicAdd(&sh.hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    find_digit(sh, rem);
    __syncthreads();
    const int d = sh.digit;
    prefix |= (uint64_t)d << shift;
    mask |= (uint64_t)0xFF << shift;
    rem -= sh.above;
    const bool done = (int)sh.hist[d] == rem;
    __syncthreads();
    if (done) break;
  }
  return prefix;
}

// Ascending bitonic sort of n_pow2 ints in shared memory.
__device__ void bitonic_sort(int32_t *a, int n_pow2) {
  for (int size = 2; size <= n_pow2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < n_pow2; i += blockDim.x) {
        const int j = i ^ stride;
        if (j > i) {
          const bool up = (i & size) == 0;
          const int32_t x = a[i], y = a[j];
          if ((x > y) == up) { a[i] = y; a[j] = x; }
        }
      }
      __syncthreads();
    }
  }
}

// Select from `get` (n items), write the sorted indices of the top k to out.
template <class Get>
__device__ void select_and_write(Get get, int64_t n, int n_valid_items, int k, int32_t *out, SelectShared &sh,
                                 int32_t *sel) {
  const int take = min(k, n_valid_items);
  uint64_t T = 0;
  if (take < n_valid_items) T = radix_threshold(get, n, take, sh);
  if (threadIdx.x == 0) sh.count = 0;
  __syncthreads();
  if (take > 0) {
    for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
      uint64_t key;
      if (get(i, key) && key >= T) {
        const int p = atomicAdd(&sh.count, 1);
        if (p < kMaxK) sel[p] = (int32_t)(~(uint32_t)(key & 0xFFFFFFFFu));
      }
    }
  }
  __syncthreads();
  int np2 = 1;
  while (np2 < take) np2 <<= 1;
  for (int i = take + threadIdx.x; i < np2; i += blockDim.x) sel[i] = INT32_MAX;
  __syncthreads();
  bitonic_sort(sel, np2);
  for (int i = threadIdx.x; i < k; i += blockDim.x) out[i] = i < take ? sel[i] : -1;
}

// ---------------------------------------------------------------- direct path
__global__ void __launch_bounds__(kTopkThreads) topk_direct_kernel(TopkSrc S, int k, int32_t *__restrict__ out,
                                                                    int *status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  uint64_t *keys = reinterpret_cast<uint64_t *>(smem_raw);                       // [kDirectCap]
  int32_t *sel = reinterpret_cast<int32_t *>(keys + kDirectCap);                 // [kMaxK]
  __shared__ SelectShared sh;
  __shared__ int n_keys;
  const int q = blockIdx.x;
  const int nv = query_nv(S, q, status);
  if (threadIdx.x == 0) n_keys = 0;
  __syncthreads();
  for (int64_t b0 = 0; b0 < S.n_items; b0 += blockDim.x) {   // uniform trip count: ballots see full warps
    const int64_t i = b0 + threadIdx.x;
    uint64_t key = 0;
    const bool v = i < S.n_items && item_key(S, q, i, nv, key, status);
    const unsigned ballot = __ballot_sync(0xFFFFFFFFu, v);
    int base = 0;
    if ((threadIdx.x & 31) == 0 && ballot) base = atomicAdd(&n_keys, __popc(ballot));
    base = __shfl_sync(0xFFFFFFFFu, base, 0);
    if (v) keys[base + __popc(ballot & ((1u << (threadIdx.x & 31)) - 1u))] = key;
  }
  __syncthreads();
  const int n = n_keys;
  auto get = [&](int64_t i, uint64_t &key) { key = keys[i]; return true; };
  select_and_write(get, n, n, k, out + (int64_t)q * k, sh, sel);
}

// ---------------------------------------------------------------- filter path
__global__ void __launch_bounds__(kTopkThreads) topk_hist_kernel(TopkSrc S, int slices, uint32_t *__restrict__ ghist,
                                                                  int *status) {
  __shared__ uint32_t h[kHistBins];
  const int q = blockIdx.y;
  const int nv = query_nv(S, q, status);
  for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) h[i] = 0;
  __syncthreads();
  const int64_t per = (S.n_items + slices - 1) / slices;
  const int64_t i0 = (int64_t)blockIdx.x * per, i1 = min(S.n_items, i0 + per);
  for (int64_t i = i0 + threadIdx.x; i < i1; i += blockDim.x) {
    uint64_t key;
    if (item_key(S, q, i, nv, key, status)) atomicAdd(&h[(uint32_t)(key >> 52)], 1u);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < kHistBins; i += blockDim.x)
    if (h[i]) atomicAdd(ghist + (int64_t)q * kHistBins + i, h[i]);
}

// Lowest bin b* such that the bins >= b* hold at least k items (0 if fewer).
__device__ int find_bin(const uint32_t *__restrict__ hist, int k, int *sh_scan) {
  // each thread owns 4 consecutive bins; block-wide suffix sums
  const int t = threadIdx.x;
  uint32_t c[4];
  uint32_t part = 0;
#pragma unroll
  for (int b = 0; b < 4; b++) { c[b] = __ldg(hist + 4 * t + b); part += c[b]; }
  sh_scan[t] = (int)part;
  __syncthreads();
  for (int o = 1; o < kTopkThreads; o <<= 1) {   // inclusive suffix scan (Hillis-Steele)
    const int v = (t + o < kTopkThreads) ? sh_scan[t + o] : 0;
    __syncthreads();
    sh_scan[t] += v;
    __syncthreads();
  }
  __shared__ int bin;
  if (t == 0) bin = 0;
  __syncthreads();
  const int incl = sh_scan[t];
  const int above = incl - (int)part;
  if (above < k && k <= incl) {
    int run = above;
    for (int b = 3; b >= 0; b--) {
      run += (int)c[b];
      if (run >= k) { bin = 4 * t + b; break; }
    }
  }
  __syncthreads();
  return bin;
}

__global__ void __launch_bounds__(kTopkThreads) topk_filter_kernel(TopkSrc S, int slices, int k,
                                                                    const uint32_t *__restrict__ ghist,
                                                                    uint32_t *__restrict__ gcount,
                                                                    uint64_t *__restrict__ cand, int *status) {
  __shared__ int scan[kTopkThreads];
  const int q = blockIdx.y;
  const int nv = query_nv(S, q, status);
  const int bstar = find_bin(ghist + (int64_t)q * kHistBins, k, scan);
  const int64_t per = (S.n_items + slices - 1) / slices;
  const int64_t i0 = (int64_t)blockIdx.x * per, i1 = min(S.n_items, i0 + per);
  const int lane = threadIdx.x & 31;
  for (int64_t base = i0; base < i1; base += blockDim.x) {
    const int64_t i = base + threadIdx.x;
    uint64_t key = 0;
    const bool v = i < i1 && item_key(S, q, i, nv, key, status) && (int)(key >> 52) >= bstar;
    const unsigned ballot = __ballot_sync(0xFFFFFFFFu, v);
    uint32_t pos = 0;
    if (lane == 0 && ballot) pos = atomicAdd(gcount + q, (uint32_t)__popc(ballot));
    pos = __shfl_sync(0xFFFFFFFFu, pos, 0) + __popc(ballot & ((1u << lane) - 1u));
    if (v && pos < (uint32_t)kCandCap) cand[(int64_t)q * kCandCap + pos] = key;
  }
}

__global__ void __launch_bounds__(kTopkThreads) topk_final_kernel(TopkSrc S, int k, const uint32_t *__restrict__ gcount,
                                                                   const uint64_t *__restrict__ cand,
                                                                   const uint32_t *__restrict__ ghist,
                                                                   int32_t *__restrict__ out, int *status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  uint64_t *keys = reinterpret_cast<uint64_t *>(smem_raw);
  int32_t *sel = reinterpret_cast<int32_t *>(keys + kCandCap);
  __shared__ SelectShared sh;
  const int q = blockIdx.x;
  const uint32_t cnt = gcount[q];
  // number of valid items = histogram total
  __shared__ int total;
  if (threadIdx.x == 0) total = 0;
  __syncthreads();
  int part = 0;
  for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) part += (int)ghist[(int64_t)q * kHistBins + i];
  atomicAdd(&total, part);
  __syncthreads();
  const int n_valid_items = total;
  if (cnt <= (uint32_t)kCandCap) {
    for (uint32_t i = threadIdx.x; i < cnt; i += blockDim.x) keys[i] = cand[(int64_t)q * kCandCap + i];
    __syncthreads();
    auto get = [&](int64_t i, uint64_t &key) { key = keys[i]; return true; };
    // candidates hold every item at or above the k-th key's bin, so the top-k of
    // the candidates is the top-k of the row
    select_and_write(get, (int64_t)cnt, min((int)cnt, n_valid_items), k, out + (int64_t)q * k, sh, sel);
  } else {
    const int nv = query_nv(S, q, status);
    auto get = [&](int64_t i, uint64_t &key) { return item_key(S, q, i, nv, key, status); };
    select_and_write(get, S.n_items, n_valid_items, k, out + (int64_t)q * k, sh, sel);
  }
}

// ---------------------------------------------------------------- host side
size_t topk_workspace_bytes(int n_q, int64_t n_items) {
  if (n_items <= kDirectCap) return 0;
  size_t b = (size_t)n_q * kHistBins * 4 + (size_t)n_q * 4;
  b = (b + 255) & ~(size_t)255;
  return b + (size_t)n_q * kCandCap * 8;
}

cudaError_t launch_topk(const float *scores, int64_t stride, int n_q, const int32_t *n_valid, int64_t n_max, int k,
                        int block, const int32_t *pool, int32_t *out, void *ws, int *status, cudaStream_t st) {
  TopkSrc S;
  S.scores = scores;
  S.stride = stride;
  S.n_valid = n_valid;
  S.pool = pool;
  S.block = block;
  S.n_max = n_max;
  S.n_items = pool ? (int64_t)kPoolSlots : (block == 1 ? n_max : (n_max + kBlock - 1) / kBlock);
  const size_t dsm = (size_t)kDirectCap * 8 + (size_t)kMaxK * 4;
  int dev = 0;
  cudaGetDevice(&dev);
  static bool attr_done[64] = {};
  if (dev >= 0 && dev < 64 && !attr_done[dev]) {
    cudaFuncSetAttribute(topk_direct_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dsm);
    cudaFuncSetAttribute(topk_final_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dsm);
    attr_done[dev] = true;
  }
  if (S.n_items <= kDirectCap) {
    topk_direct_kernel<<<n_q, kTopkThreads, dsm, st>>>(S, k, out, status);
    return cudaGetLastError();
  }
  uint32_t *ghist = static_cast<uint32_t *>(ws);
  uint32_t *gcount = ghist + (size_t)n_q * kHistBins;
  size_t off = ((size_t)n_q * kHistBins * 4 + (size_t)n_q * 4 + 255) & ~(size_t)255;
  uint64_t *cand = reinterpret_cast<uint64_t *>(static_cast<char *>(ws) + off);
  cudaError_t e = cudaMemsetAsync(ghist, 0, (size_t)n_q * kHistBins * 4 + (size_t)n_q * 4, st);
  if (e != cudaSuccess) return e;
  int slices = (int)max((int64_t)1, min((S.n_items + 4095) / 4096, (int64_t)((2 * 152 + n_q - 1) / n_q)));
  dim3 grid(slices, n_q);
  topk_hist_kernel<<<grid, kTopkThreads, 0, st>>>(S, slices, ghist, status);
  topk_filter_kernel<<<grid, kTopkThreads, 0, st>>>(S, slices, k, ghist, gcount, cand, status);
  topk_final_kernel<<<n_q, kTopkThreads, dsm, st>>>(S, k, gcount, cand, ghist, out, status);
  return cudaGetLastError();
}

}  // namespace csa2
