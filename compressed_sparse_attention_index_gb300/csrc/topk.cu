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
// Longer rows (1M-entry Full-layer rows, 131,072-block pool rows) take two
// launches: a bandwidth pass writes the maximum key of every group of 128 items;
// then one CTA per row finds T, the k-th largest group maximum (a lower bound of
// the k-th best key), rescans only the groups whose maximum reaches T, and runs
// the exact selection on those candidates (usually about 2k items).  A row whose
// candidates overflow the buffer falls back to an exact radix select straight
// over the score row.
#include "common.cuh"

namespace csa2 {

constexpr int kDirectCap = 16384;   // items held in shared memory by one CTA
constexpr int kMaxGroup = 128;      // largest group of items per group maximum (long rows)
constexpr int kMaxGroups = 8192;    // groups a long row may have
constexpr int kCandCap = 8192;      // candidates kept in shared memory (long rows)
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
  uint32_t *whist;   // [32 warps][256] private histograms (dynamic shared memory)
  int digit;
  int above;
  int count;
};

// sh.hist[d] = number of items i < n with digit_of(i, d) true.  Each warp counts
// into its own histogram (no cross-warp contention on the few busy bins of a
// skewed distribution), then the 32 histograms are summed.
template <class F>
__device__ void block_hist(SelectShared &sh, int64_t n, F digit_of) {
  uint32_t *wh = sh.whist + (threadIdx.x >> 5) * 256;
  for (int i = threadIdx.x; i < 32 * 256; i += blockDim.x) sh.whist[i] = 0;
  __syncthreads();
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
    uint32_t d;
    if (digit_of(i, d)) atomicAdd(&wh[d], 1u);
  }
  __syncthreads();
  for (int b = threadIdx.x; b < 256; b += blockDim.x) {
    uint32_t c = 0;
#pragma unroll 8
    for (int w = 0; w < 32; w++) c += sh.whist[w * 256 + b];
    sh.hist[b] = c;
  }
  __syncthreads();
}

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
    block_hist(sh, n, [&](int64_t i, uint32_t &d) {
      uint64_t key;
      if (!get(i, key) || (key & mask) != prefix) return false;
      d = (uint32_t)((key >> shift) & 255u);
      return true;
    });
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

// Descending bitonic sort of n_pow2 64-bit keys in shared memory.
__device__ void bitonic_sort_desc_u64(uint64_t *a, int n_pow2) {
  for (int size = 2; size <= n_pow2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < n_pow2; i += blockDim.x) {
        const int j = i ^ stride;
        if (j > i) {
          const bool desc = (i & size) == 0;
          const uint64_t x = a[i], y = a[j];
          if ((x < y) == desc) { a[i] = y; a[j] = x; }
        }
      }
      __syncthreads();
    }
  }
}

// Exact top-k of n unique keys already in shared memory (capacity >= the next
// power of two of n), by sorting them: cheaper than radix passes for small n.
// The keys array is reordered.
__device__ void select_small(uint64_t *keys, int n, int k, int32_t *out, int32_t *sel) {
  int np2 = 1;
  while (np2 < n) np2 <<= 1;
  for (int i = n + threadIdx.x; i < np2; i += blockDim.x) keys[i] = 0;   // below every valid key
  __syncthreads();
  bitonic_sort_desc_u64(keys, np2);
  const int take = min(k, n);
  int sp2 = 1;
  while (sp2 < take) sp2 <<= 1;
  for (int i = threadIdx.x; i < sp2; i += blockDim.x)
    sel[i] = i < take ? (int32_t)(~(uint32_t)(keys[i] & 0xFFFFFFFFu)) : INT32_MAX;
  __syncthreads();
  bitonic_sort(sel, sp2);
  for (int i = threadIdx.x; i < k; i += blockDim.x) out[i] = i < take ? sel[i] : -1;
}

constexpr int kSortMax = 4096;     // sets up to this size are selected by sorting
constexpr int kRankMax = 1536;     // sets up to this size are selected by ranking

// Exact top-k of n unique keys in shared memory by counting: a key is selected
// iff fewer than k keys are larger; its output slot is the number of selected
// keys with a smaller index.  O(n^2) comparisons, two barriers.
__device__ void select_rank(const uint64_t *keys, int n, int k, int32_t *out, int32_t *sel) {
  const int take = min(k, n);
  __shared__ int n_sel;
  if (threadIdx.x == 0) n_sel = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const uint64_t ki = keys[i];
    int above = 0;
    for (int j = 0; j < n; j++) above += keys[j] > ki;
    if (above < take) sel[atomicAdd(&n_sel, 1)] = (int32_t)(~(uint32_t)(ki & 0xFFFFFFFFu));
  }
  __syncthreads();
  for (int i = threadIdx.x; i < take; i += blockDim.x) {
    const int32_t xi = sel[i];
    int before = 0;
    for (int j = 0; j < take; j++) before += sel[j] < xi;
    out[before] = xi;
  }
  for (int i = take + threadIdx.x; i < k; i += blockDim.x) out[i] = -1;
}

// ---------------------------------------------------------------- direct path
__global__ void __launch_bounds__(kTopkThreads) topk_direct_kernel(TopkSrc S, int k, int32_t *__restrict__ out,
                                                                    int *status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  uint64_t *keys = reinterpret_cast<uint64_t *>(smem_raw);                       // [kDirectCap]
  int32_t *sel = reinterpret_cast<int32_t *>(keys + kDirectCap);                 // [kMaxK]
  __shared__ SelectShared sh;
  sh.whist = reinterpret_cast<uint32_t *>(sel + kMaxK);                          // [32][256]
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
  if (n <= kRankMax) {
    select_rank(keys, n, k, out + (int64_t)q * k, sel);
  } else if (n <= kSortMax) {
    select_small(keys, n, k, out + (int64_t)q * k, sel);
  } else {
    auto get = [&](int64_t i, uint64_t &key) { key = keys[i]; return true; };
    select_and_write(get, n, n, k, out + (int64_t)q * k, sh, sel);
  }
}

// ---------------------------------------------------------------- long rows
// Group maxima: the max key over each group of G consecutive items (0 if the
// group holds no valid item), G a power of two in [8, 128].  A warp covers
// 32 * ipl items (ipl = max(1, G/32) per lane) and reduces within groups.
__global__ void __launch_bounds__(256) topk_groupmax_kernel(TopkSrc S, int G, int n_groups,
                                                             uint32_t *__restrict__ gmax, int *status) {
  const int q = blockIdx.y;
  const int nv = query_nv(S, q, status);
  const int lane = threadIdx.x & 31;
  const int warps = blockDim.x >> 5;
  const int ipl = G >= 32 ? G / 32 : 1;          // items per lane
  const int lpg = G >= 32 ? 32 : G;              // lanes per group
  const int64_t span = 32 * ipl;                 // items per warp step
  const int64_t n_steps = ((int64_t)n_groups * G + span - 1) / span;
  for (int64_t w = (int64_t)blockIdx.x * warps + (threadIdx.x >> 5); w < n_steps; w += (int64_t)gridDim.x * warps) {
    uint32_t m = 0;
    const int64_t i0 = w * span + (int64_t)lane * ipl;
    const float *rowp = S.scores + (int64_t)q * S.stride;
    if (ipl == 4 && S.block == 1 && S.pool == nullptr && i0 + 4 <= nv &&
        ((reinterpret_cast<uintptr_t>(rowp + i0) & 15u) == 0)) {
      const float4 v = __ldg(reinterpret_cast<const float4 *>(rowp + i0));
      m = max(max(order_key(v.x), order_key(v.y)), max(order_key(v.z), order_key(v.w)));
    } else {
      for (int u = 0; u < ipl; u++) {
        uint64_t key;
        if (i0 + u < S.n_items && item_key(S, q, i0 + u, nv, key, status)) m = max(m, (uint32_t)(key >> 32));
      }
    }
    for (int o = lpg >> 1; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    const int64_t g = i0 >> (__ffs(G) - 1);
    if ((lane & (lpg - 1)) == 0 && g < n_groups) gmax[(int64_t)q * n_groups + g] = m;
  }
}

// k-th largest of n 32-bit values (counted with multiplicity; requires at
// least k valid values): 8-bit radix passes narrowing a prefix, down to bit
// min_shift (the lower bits of the result are zero).
template <class Get>
__device__ uint32_t radix_kth_u32(Get get, int n, int k, SelectShared &sh, int min_shift = 0) {
  uint32_t prefix = 0, mask = 0;
  int rem = k;
  for (int shift = 24; shift >= min_shift; shift -= 8) {
    block_hist(sh, n, [&](int64_t i, uint32_t &d) {
      uint32_t v;
      if (!get((int)i, v) || (v & mask) != prefix) return false;
      d = (v >> shift) & 255u;
      return true;
    });
    find_digit(sh, rem);
    __syncthreads();
    prefix |= (uint32_t)sh.digit << shift;
    mask |= 0xFFu << shift;
    rem -= sh.above;
    __syncthreads();
  }
  return prefix;
}

// One CTA per query.  T = the k-th largest group maximum: at least k groups
// reach T, so at least k items do, so the k-th best item key is >= T and every
// item of the top-k lies in a group whose maximum is >= T.  Those groups are
// listed, their items scanned by all threads at once for keys >= T (a superset
// of the top-k, usually ~2k items), and the exact selection runs on that set.
__global__ void __launch_bounds__(kTopkThreads) topk_group_select_kernel(TopkSrc S, int G, int n_groups, int k,
                                                                          const uint32_t *__restrict__ gmax,
                                                                          int32_t *__restrict__ out, int *status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  uint64_t *cand = reinterpret_cast<uint64_t *>(smem_raw);               // [kCandCap]
  uint32_t *gm = reinterpret_cast<uint32_t *>(cand + kCandCap);          // [kMaxGroups] group maxima
  int32_t *glist = reinterpret_cast<int32_t *>(gm + kMaxGroups);         // [kMaxGroups] groups to scan
  int32_t *sel = glist + kMaxGroups;                                     // [kMaxK]
  __shared__ SelectShared sh;
  sh.whist = reinterpret_cast<uint32_t *>(sel + kMaxK);                  // [32][256]
  __shared__ int n_cand, n_valid_groups, n_list;
  const int q = blockIdx.x;
  const int nv = query_nv(S, q, status);
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) { n_cand = 0; n_valid_groups = 0; n_list = 0; }
  __syncthreads();
  int live_groups = 0;
  for (int b0 = 0; b0 < n_groups; b0 += 8 * blockDim.x) {     // eight loads in flight per thread
    uint32_t m[8];
#pragma unroll
    for (int u = 0; u < 8; u++) {
      const int g = b0 + u * blockDim.x + threadIdx.x;
      m[u] = g < n_groups ? __ldg(gmax + (int64_t)q * n_groups + g) : 0u;
    }
#pragma unroll
    for (int u = 0; u < 8; u++) {
      const int g = b0 + u * blockDim.x + threadIdx.x;
      if (g < n_groups) gm[g] = m[u];
      live_groups += m[u] != 0;
    }
  }
  atomicAdd(&n_valid_groups, live_groups);
  __syncthreads();
  uint32_t T = 1;                                    // nonzero keys: every valid item
  if (n_valid_groups > k) {
    auto get = [&](int i, uint32_t &v) { v = gm[i]; return v != 0; };
    // the k-th largest group maximum to 16-bit resolution: its upper 16 bits
    // (lower bits zero) are still a lower bound of the k-th best key
    T = radix_kth_u32(get, n_groups, k, sh, 16);
  }
  // list the groups whose maximum reaches T
  for (int b0 = 0; b0 < n_groups; b0 += blockDim.x) {
    const int g = b0 + threadIdx.x;
    const bool v = g < n_groups && gm[g] >= T;
    const unsigned b = __ballot_sync(0xFFFFFFFFu, v);
    int base = 0;
    if (lane == 0 && b) base = atomicAdd(&n_list, __popc(b));
    base = __shfl_sync(0xFFFFFFFFu, base, 0) + __popc(b & ((1u << lane) - 1u));
    if (v) glist[base] = g;
  }
  __syncthreads();
  // scan their items: every thread keeps kScanU item loads in flight
  constexpr int kScanU = 8;
  const int lg = __ffs(G) - 1;                      // G is a power of two
  const int total = n_list << lg;
  const bool plain = S.pool == nullptr && S.block == 1;
  const float *row = S.scores + (int64_t)q * S.stride;
  const bool row16 = (reinterpret_cast<uintptr_t>(row) & 15u) == 0;
  if (plain) {
    // four consecutive items per thread and load (G is a multiple of 4)
    constexpr int kV = 4;
    for (int b0 = 0; b0 < total; b0 += 4 * kV * blockDim.x) {
      float4 sc[kV];
      int64_t base[kV];
#pragma unroll
      for (int u = 0; u < kV; u++) {
        const int f = b0 + 4 * (u * blockDim.x + threadIdx.x);
        base[u] = -1;
        sc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (f < total) {
          base[u] = ((int64_t)glist[f >> lg] << lg) + (f & (G - 1));
          if (row16 && base[u] + 4 <= nv) {
            sc[u] = __ldg(reinterpret_cast<const float4 *>(row + base[u]));
          } else {                                   // ragged end or unaligned row: element loads
            const int64_t b = base[u];
            if (b < nv) sc[u].x = __ldg(row + b);
            if (b + 1 < nv) sc[u].y = __ldg(row + b + 1);
            if (b + 2 < nv) sc[u].z = __ldg(row + b + 2);
            if (b + 3 < nv) sc[u].w = __ldg(row + b + 3);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kV; u++) {
        const float vals[4] = {sc[u].x, sc[u].y, sc[u].z, sc[u].w};
#pragma unroll
        for (int e = 0; e < 4; e++) {
          const int64_t i = base[u] + e;
          uint32_t kk = 0;
          const bool ok = base[u] >= 0 && i < nv && (kk = order_key(vals[e])) >= T;
          if (!__any_sync(0xFFFFFFFFu, ok)) continue;   // most rounds have no candidate
          const unsigned b = __ballot_sync(0xFFFFFFFFu, ok);
          int pos0 = 0;
          if (lane == 0 && b) pos0 = atomicAdd(&n_cand, __popc(b));
          pos0 = __shfl_sync(0xFFFFFFFFu, pos0, 0) + __popc(b & ((1u << lane) - 1u));
          if (ok && pos0 < kCandCap) cand[pos0] = ((uint64_t)kk << 32) | (uint32_t)(~(uint32_t)i);
        }
      }
    }
  } else
  for (int b0 = 0; b0 < total; b0 += kScanU * blockDim.x) {
    uint64_t key[kScanU];
    bool v[kScanU];
#pragma unroll
    for (int u = 0; u < kScanU; u++) {
      const int f = b0 + u * blockDim.x + threadIdx.x;
      key[u] = 0;
      v[u] = false;
      if (f < total) {
        const int64_t i = ((int64_t)glist[f >> lg] << lg) + (f & (G - 1));
        if (plain) {
          v[u] = i < nv;
          if (v[u]) key[u] = ((uint64_t)order_key(__ldg(row + i)) << 32) | (uint32_t)(~(uint32_t)i);
        } else {
          v[u] = i < S.n_items && item_key(S, q, i, nv, key[u], status);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kScanU; u++) {
      const bool ok = v[u] && (uint32_t)(key[u] >> 32) >= T;
      if (!__any_sync(0xFFFFFFFFu, ok)) continue;
      const unsigned b = __ballot_sync(0xFFFFFFFFu, ok);
      int base = 0;
      if (lane == 0 && b) base = atomicAdd(&n_cand, __popc(b));
      base = __shfl_sync(0xFFFFFFFFu, base, 0) + __popc(b & ((1u << lane) - 1u));
      if (ok && base < kCandCap) cand[base] = key[u];
    }
  }
  __syncthreads();
  const int nc = n_cand;
  if (nc <= kRankMax) {
    select_rank(cand, nc, k, out + (int64_t)q * k, sel);
  } else if (nc <= kSortMax) {
    select_small(cand, nc, k, out + (int64_t)q * k, sel);
  } else if (nc <= kCandCap) {
    auto get = [&](int64_t i, uint64_t &key) { key = cand[i]; return true; };
    select_and_write(get, nc, nc, k, out + (int64_t)q * k, sh, sel);
  } else {
    // too many ties at T for the buffer: exact selection straight over the row
    __shared__ int nvi;
    if (threadIdx.x == 0) nvi = 0;
    __syncthreads();
    int c = 0;
    for (int64_t i = threadIdx.x; i < S.n_items; i += blockDim.x) {
      uint64_t key;
      c += item_key(S, q, i, nv, key, status) ? 1 : 0;
    }
    atomicAdd(&nvi, c);
    __syncthreads();
    auto get = [&](int64_t i, uint64_t &key) { return item_key(S, q, i, nv, key, status); };
    select_and_write(get, S.n_items, nvi, k, out + (int64_t)q * k, sh, sel);
  }
}

// ---------------------------------------------------------------- host side
static int64_t topk_items(int64_t n_max, int block, bool pool) {
  return pool ? (int64_t)kPoolSlots : (block == 1 ? n_max : (n_max + kBlock - 1) / kBlock);
}

// Group size for long rows: the smallest power of two >= 8 that keeps the
// groups within kMaxGroups, doubled while at least 4k groups remain.
static int topk_group(int64_t n_items, int k) {
  int G = 8;
  while (G <= kMaxGroup && ((n_items + G - 1) / G > kMaxGroups || n_items / (2 * G) >= 4 * (int64_t)k) &&
         !(G == kMaxGroup && (n_items + G - 1) / G <= kMaxGroups))
    G <<= 1;
  return G;
}

size_t topk_workspace_bytes(int n_q, int64_t n_items, int k) {
  if (n_items <= kDirectCap) return 0;
  const int G = topk_group(n_items, k);
  return (size_t)n_q * ((n_items + G - 1) / G) * 4;
}

bool topk_items_supported(int64_t n_items, int k) {
  if (n_items <= kDirectCap) return true;
  const int G = topk_group(n_items, k);
  return G <= kMaxGroup && (n_items + G - 1) / G <= kMaxGroups;
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
  S.n_items = topk_items(n_max, block, pool != nullptr);
  const size_t dsm_direct = (size_t)kDirectCap * 8 + (size_t)kMaxK * 4 + 32 * 256 * 4;
  const size_t dsm_group = (size_t)kCandCap * 8 + (size_t)kMaxGroups * 8 + (size_t)kMaxK * 4 + 32 * 256 * 4;
  int dev = 0;
  cudaGetDevice(&dev);
  static bool attr_done[64] = {};
  if (dev >= 0 && dev < 64 && !attr_done[dev]) {
    cudaFuncSetAttribute(topk_direct_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dsm_direct);
    cudaFuncSetAttribute(topk_group_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dsm_group);
    attr_done[dev] = true;
  }
  if (S.n_items <= kDirectCap) {
    topk_direct_kernel<<<n_q, kTopkThreads, dsm_direct, st>>>(S, k, out, status);
    return cudaGetLastError();
  }
  const int G = topk_group(S.n_items, k);
  const int n_groups = (int)((S.n_items + G - 1) / G);
  uint32_t *gmax = static_cast<uint32_t *>(ws);
  const int64_t warp_steps = ((int64_t)n_groups * G + 32 * (G >= 32 ? G / 32 : 1) - 1) / (32 * (G >= 32 ? G / 32 : 1));
  const int64_t gx = (warp_steps + 7) / 8;            // one warp step per warp: every load in flight at once
  topk_groupmax_kernel<<<dim3((unsigned)gx, n_q), 256, 0, st>>>(S, G, n_groups, gmax, status);
  topk_group_select_kernel<<<n_q, kTopkThreads, dsm_group, st>>>(S, G, n_groups, k, gmax, out, status);
  return cudaGetLastError();
}

}  // namespace csa2
