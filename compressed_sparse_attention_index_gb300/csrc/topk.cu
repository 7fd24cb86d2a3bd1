// Top-k selection (csa2_topk): the 512 entries each query attends to
// (perchy.ai/models/deepseek, card "Full. Reindex. Reuse."), and the candidate
// pool of 2,048 blocks of 8 entries that Reindex layers score (An
// infra-oriented diagram of the DeepSeek-V4.1-Flash architecture,
// lightning-indexer note).
//
// Every item gets a unique 64-bit key  (order_key(score) << 32) | ~index :
// larger key = higher score, then lower index.  Selecting the k largest keys
// therefore gives the top-k with lower-index tie-break, and a radix select over
// these keys needs no separate tie pass.
//
// Rows of up to kDirectCap items are selected by one CTA from shared memory.
// Longer rows (1M-entry Full-layer rows, 131,072-block pool rows) take two
// passes: the maximum key of every supergroup of items (512 items for k = 512
// over 1M entries; written by a bandwidth pass, or by the indexer's epilogue
// inside csa2_decode); then a thread-block cluster of P CTAs per row finds a
// threshold T from the supergroup maxima alone (radix-256 steps below the
// leading bits all maxima share), streams only the supergroups whose maximum
// reaches T (about k), and CTA 0 runs the exact selection on the candidates
// gathered from the cluster (about k items).  A row whose lists overflow
// shared memory falls back to an exact radix select straight over the row.
#include <algorithm>

#include "common.cuh"
#include "launch.cuh"
#include "tc_ptx.cuh"

namespace csa2 {

constexpr int kDirectCap = 16384;   // items held in shared memory by one CTA
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
  // optional (plain rows): latent cache records [n_seq][n_max][288] that the
  // attention reads next; the collecting CTAs prefetch their candidates' ones
  // into L2
  const uint8_t *kv_pf;
  const int32_t *q_seq;
  int n_seq;
  // optional (pool rows): the maximum order key of each 8-entry block's
  // valid entries, 0 for none, [n_q][bstride] (written by the pool-mode
  // indexer inside csa2_decode_reindex)
  const uint32_t *bmax;
  int64_t bstride;
};

// Key of item i of query q; false if the item is not valid.
// The key of item i from its score and (pool mode) its block id, already
// loaded (pool mode or S.block == 1).
__device__ __forceinline__ bool item_key_of(const TopkSrc &S, int64_t i, int nv, float score, int blk, uint64_t &key,
                                            int *status) {
  if (S.pool != nullptr) {
    if (blk < 0) return false;
    const int64_t j = (int64_t)blk * kBlock + (i & 7);
    if (j >= nv) {
      if ((int64_t)blk * kBlock >= S.n_max) record_error(status, CSA2_ERR_BOUNDS);
      return false;
    }
    key = ((uint64_t)order_key(score) << 32) | (uint32_t)(~(uint32_t)j);
    return true;
  }
  if (i >= nv) return false;
  key = ((uint64_t)order_key(score) << 32) | (uint32_t)(~(uint32_t)i);
  return true;
}

__device__ __forceinline__ bool item_key(const TopkSrc &S, int q, int64_t i, int nv, uint64_t &key, int *status) {
  const float *row = S.scores + (int64_t)q * S.stride;
  if (S.pool != nullptr || S.block == 1)
    return item_key_of(S, i, nv, __ldg(row + i), S.pool != nullptr ? __ldg(S.pool + (int64_t)q * kPoolBlocks + (i >> 3)) : 0,
                       key, status);
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

// ---- block-wide pieces (blockDim.x a multiple of 32, <= kTopkThreads) ----
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
  const int nw = blockDim.x >> 5;
  for (int i = threadIdx.x; i < nw * 256; i += blockDim.x) sh.whist[i] = 0;
  __syncthreads();
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
    uint32_t d;
    if (digit_of(i, d)) atomicAdd(&wh[d], 1u);
  }
  __syncthreads();
  for (int b = threadIdx.x; b < 256; b += blockDim.x) {
    uint32_t c = 0;
#pragma unroll 8
    for (int w = 0; w < nw; w++) c += sh.whist[w * 256 + b];
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

// Block-wide exclusive scans over nb counters in shared memory (nb a multiple
// of blockDim.x, blockDim.x a multiple of 32): suffix (counts of the bins
// above) and prefix (counts of the bins below).
template <bool kSuffix>
__device__ void block_offsets(uint32_t *h, int nb) {
  __shared__ uint32_t wsum[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int per = nb / blockDim.x;
  const int b0 = threadIdx.x * per;
  uint32_t part = 0;
  for (int j = 0; j < per; j++) part += h[b0 + j];
  uint32_t incl = part;                              // inclusive scan toward this thread
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = kSuffix ? __shfl_down_sync(0xFFFFFFFFu, incl, o) : __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (kSuffix ? lane + o < 32 : lane >= o) incl += v;
  }
  if (lane == 0) wsum[warp] = 0;
  __syncthreads();
  if (kSuffix ? lane == 0 : lane == 31) wsum[warp] = incl;
  __syncthreads();
  const bool other = lane < nw && (kSuffix ? lane > warp : lane < warp);
  uint32_t run = incl - part + __reduce_add_sync(0xFFFFFFFFu, other ? wsum[lane] : 0u);
  if (kSuffix) {
    for (int j = per - 1; j >= 0; j--) { const uint32_t v = h[b0 + j]; h[b0 + j] = run; run += v; }
  } else {
    for (int j = 0; j < per; j++) { const uint32_t v = h[b0 + j]; h[b0 + j] = run; run += v; }
  }
  __syncthreads();
}

// Warp-wide sum of one int per lane (shuffles; every lane gets it).
__device__ __forceinline__ int warp_sum(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// Block-wide exclusive prefix sum of one int per thread, in thread order;
// *total receives the sum.  Two barriers.
__device__ int block_excl_scan(int c, int *total) {
  __shared__ int wsum[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int incl = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += v;
  }
  __syncthreads();                                   // an earlier call's readers are done with wsum
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  const int w = lane < nw ? wsum[lane] : 0;
  *total = __reduce_add_sync(0xFFFFFFFFu, w);
  return __reduce_add_sync(0xFFFFFFFFu, lane < warp ? w : 0) + incl - c;
}

// Block-wide: a lower bound of the rem-th largest (with multiplicity) of the
// values v[0..n) in shared memory, 0 meaning "no value" (1 <= rem <= the
// number of nonzero values), exact in its bits from 31 down to `low`, with
// the bits below `low` cleared, so at least rem values reach it.  The bits
// every nonzero value shares (those above the highest bit where the maximum
// and the smallest nonzero value differ) are taken from the maximum; the rest go
// eight bits per step: a 256-bin histogram of the next digit among the values
// that match the prefix so far (shared-memory atomics; a warp whose values all
// share the digit adds them with one), then warp 0 finds the digit by a suffix
// scan while the other threads clear the next step's histogram (two
// alternate).  With max_steps set, the search stops after that many steps and
// returns the prefix found (a coarser, still valid, lower bound).  hist: 512
// counters.  Not inlined: every call site shares one copy of the code.
__device__ __noinline__ uint32_t block_kth256(const uint32_t *v, int n, int rem, int low, uint32_t *hist,
                                             int max_steps = 32) {
  __shared__ uint32_t prefix_sh, ext_sh[2][32];
  __shared__ int rem_sh;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  uint32_t mx = 0u, mn = ~0u;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const uint32_t x = v[i];
    mx = max(mx, x);
    if (x != 0u) mn = min(mn, x);
  }
  mx = __reduce_max_sync(0xFFFFFFFFu, mx);
  mn = __reduce_min_sync(0xFFFFFFFFu, mn);
  if (lane == 0) { ext_sh[0][warp] = mx; ext_sh[1][warp] = mn; }
  for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0u;
  if (threadIdx.x == 0) rem_sh = rem;
  __syncthreads();
  mx = __reduce_max_sync(0xFFFFFFFFu, lane < nw ? ext_sh[0][lane] : 0u);
  mn = __reduce_min_sync(0xFFFFFFFFu, lane < nw ? ext_sh[1][lane] : ~0u);
  const uint32_t lowmask = low >= 32 ? ~0u : (1u << low) - 1u;
  const int hb = (mx ^ mn) == 0u ? -1 : 31 - __clz(mx ^ mn);   // highest differing bit
  uint32_t pmask = hb >= 31 ? 0u : ~((2u << hb) - 1u);
  uint32_t prefix = mx & pmask;
  if (hb < low) {                                              // the bits from `low` up are common
    __syncthreads();                                           // ext_sh is read; the next call may rewrite it
    return mx & ~lowmask;
  }
  int shift = max(hb - 7, low);
  for (int step = 0, buf = 0;; step++, buf ^= 1) {
    uint32_t *h = hist + buf * 256;
    for (int b0 = 0; b0 < n; b0 += blockDim.x) {      // uniform trip count: whole warps
      const int i = b0 + threadIdx.x;
      const uint32_t x = i < n ? v[i] : 0u;
      const bool ok = i < n && (x & pmask) == prefix;
      const unsigned act = __ballot_sync(0xFFFFFFFFu, ok);
      if (ok) {
        const uint32_t d = (x >> shift) & 255u;
        const int first = __ffs(act) - 1;
        const uint32_t d0 = __shfl_sync(act, d, first);
        if (__all_sync(act, d == d0)) {
          if (lane == first) atomicAdd(&h[d], (uint32_t)__popc(act));
        } else {
          atomicAdd(&h[d], 1u);
        }
      }
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      // lane l owns digits 8l .. 8l+7; suffix sums over the lanes above
      uint32_t c[8], part = 0u;
#pragma unroll
      for (int j = 0; j < 8; j++) { c[j] = h[8 * lane + j]; part += c[j]; }
      uint32_t incl = part;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_down_sync(0xFFFFFFFFu, incl, o);
        if (lane + o < 32) incl += t;
      }
      const int r = rem_sh;
      uint32_t above = incl - part;                  // values in the digits of the lanes above
      if (above < (uint32_t)r && (uint32_t)r <= incl) {
#pragma unroll
        for (int j = 7; j >= 0; j--) {
          if (above + c[j] >= (uint32_t)r) {
            prefix_sh = prefix | ((uint32_t)(8 * lane + j) << shift);
            rem_sh = r - (int)above;
            break;
          }
          above += c[j];
        }
      }
    } else {
      for (int i = threadIdx.x - 32; i < 256; i += blockDim.x - 32) hist[(buf ^ 1) * 256 + i] = 0u;
    }
    __syncthreads();
    prefix = prefix_sh;
    pmask |= 255u << shift;
    if (shift == low || step + 1 == max_steps) break;
    shift = max(shift - 8, low);
  }
  __syncthreads();                                   // prefix_sh is read; the next call may rewrite it
  return prefix & ~((1u << shift) - 1u);
}

// Block-wide min / max of one value per thread; every thread gets the result.
// The two slot rows alternate, so back-to-back calls need one barrier each.
struct BlockReduce {
  uint32_t (*slots)[32];
  int parity;
  template <bool kMax>
  __device__ uint32_t run(uint32_t v) {
    const int lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    v = kMax ? __reduce_max_sync(0xFFFFFFFFu, v) : __reduce_min_sync(0xFFFFFFFFu, v);
    if (lane == 0) slots[parity][threadIdx.x >> 5] = v;
    __syncthreads();
    const uint32_t w = lane < nw ? slots[parity][lane] : (kMax ? 0u : ~0u);
    parity ^= 1;
    return kMax ? __reduce_max_sync(0xFFFFFFFFu, w) : __reduce_min_sync(0xFFFFFFFFu, w);
  }
};

// Block-wide exclusive suffix sum of one value per thread (threads with a
// larger index come first); *total receives the sum.  Two barriers.
__device__ uint32_t block_excl_suffix(uint32_t c, uint32_t *total) {
  __shared__ uint32_t wsum[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  uint32_t incl = c;                                 // inclusive suffix within the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_down_sync(0xFFFFFFFFu, incl, o);
    if (lane + o < 32) incl += v;
  }
  __syncthreads();                                   // an earlier call's readers are done with wsum
  if (lane == 0) wsum[warp] = incl;
  __syncthreads();
  const uint32_t w = lane < nw ? wsum[lane] : 0u;
  *total = __reduce_add_sync(0xFFFFFFFFu, w);
  return __reduce_add_sync(0xFFFFFFFFu, lane > warp ? w : 0u) + incl - c;
}

constexpr int kWideBins = 4096;                      // 12-bit digits

// Common-prefix split of the nonzero values v[0..n): the bits above the
// highest bit where the largest and the smallest nonzero value differ are
// shared by every nonzero value; the 12-bit digit just below them orders the
// values.  Block-wide; every thread gets the same result.  Clears hist
// (kWideBins counters) on the way (the first barrier orders it).
struct WideDigit {
  uint32_t prefix, pmask;
  int sh;        // digit = (x >> sh) & 4095; -1: all nonzero values are equal (or none)
  uint32_t mx;
};
template <class Get>
__device__ WideDigit wide_digit(Get get, int n, uint32_t *hist) {
  __shared__ uint32_t ext_sh[2][32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  uint32_t mx = 0u, mn = ~0u;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const uint32_t x = get(i);
    mx = max(mx, x);
    if (x != 0u) mn = min(mn, x);
  }
  mx = __reduce_max_sync(0xFFFFFFFFu, mx);
  mn = __reduce_min_sync(0xFFFFFFFFu, mn);
  __syncthreads();                                   // an earlier call's readers are done with ext_sh
  if (lane == 0) { ext_sh[0][warp] = mx; ext_sh[1][warp] = mn; }
  for (int i = threadIdx.x; i < kWideBins; i += blockDim.x) hist[i] = 0u;
  __syncthreads();
  WideDigit d;
  d.mx = __reduce_max_sync(0xFFFFFFFFu, lane < nw ? ext_sh[0][lane] : 0u);
  mn = __reduce_min_sync(0xFFFFFFFFu, lane < nw ? ext_sh[1][lane] : ~0u);
  const uint32_t diff = mn == ~0u ? 0u : (d.mx ^ mn);
  const int hb = diff == 0u ? -1 : 31 - __clz(diff);
  d.sh = hb < 0 ? -1 : max(hb - 11, 0);
  d.pmask = hb < 0 ? ~0u : (hb >= 31 ? 0u : ~((2u << hb) - 1u));
  d.prefix = d.mx & d.pmask;
  return d;
}

// After the digits' histogram: the digit D that holds the rem-th largest
// value (values in digits above D: *above < rem <= *above + hist[D]).  Four
// bins per thread (blockDim.x * 4 == kWideBins).  Three barriers.
__device__ int wide_find(const uint32_t *hist, int rem, uint32_t *above_out) {
  __shared__ int d_sh;
  __shared__ uint32_t a_sh;
  const int b0 = threadIdx.x * 4;
  const uint32_t c0 = hist[b0], c1 = hist[b0 + 1], c2 = hist[b0 + 2], c3 = hist[b0 + 3];
  uint32_t total;
  uint32_t above = block_excl_suffix(c0 + c1 + c2 + c3, &total);
  const uint32_t c[4] = {c0, c1, c2, c3};
#pragma unroll
  for (int j = 3; j >= 0; j--) {
    if (above < (uint32_t)rem && (uint32_t)rem <= above + c[j]) { d_sh = b0 + j; a_sh = above; }
    above += c[j];
  }
  __syncthreads();
  *above_out = a_sh;
  return d_sh;
}

// Block-wide: a lower bound L of the rem-th largest (with multiplicity) of the
// values v[0..n) in shared memory, 0 meaning "no value" (1 <= rem <= the
// number of nonzero values), such that at least rem values are >= L: exact in
// the bits every nonzero value shares and in the 12 bits below them, and in
// 12 more when more than 64 values share the digit found, lower bits cleared.
// Each step is one 4,096-bin histogram and a block-wide scan (blockDim.x ==
// 1024).  hist: kWideBins counters.
__device__ __forceinline__ uint32_t block_kth_bound12(const uint32_t *v, int n, int rem, uint32_t *hist) {
  const WideDigit wd = wide_digit([&](int i) { return v[i]; }, n, hist);
  if (wd.sh < 0) {
    __syncthreads();
    return wd.mx;
  }
  uint32_t prefix = wd.prefix, pmask = wd.pmask;
  int sh = wd.sh;
  for (int step = 0;; step++) {
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      const uint32_t x = v[i];
      if (x != 0u && (x & pmask) == prefix) atomicAdd(&hist[(x >> sh) & (kWideBins - 1)], 1u);
    }
    __syncthreads();
    uint32_t above;
    const int D = wide_find(hist, rem, &above);
    // digits above D hold `above` < rem of the values matching the prefix,
    // digit D the rest: at least rem values are >= prefix | D << sh
    prefix |= (uint32_t)D << sh;
    pmask |= (uint32_t)(kWideBins - 1) << sh;
    rem -= (int)above;
    const uint32_t cnt = hist[D];
    if (step == 1 || sh == 0 || cnt <= 64u) break;     // uniform
    __syncthreads();                                    // hist[D] is read everywhere
    for (int i = threadIdx.x; i < kWideBins; i += blockDim.x) hist[i] = 0u;
    sh = max(sh - 12, 0);
    __syncthreads();
  }
  __syncthreads();                                      // hist is read; the caller may reuse it
  return prefix & ~((1u << sh) - 1u);
}

// Exact top-k of n unique nonzero 64-bit keys held in shared memory in
// ascending index order, k < n <= blockDim.x (one key per thread): the digit
// of the k-th largest key is found by one 4,096-bin histogram of the 12 bits
// below the common prefix of the score halves, the keys in that digit (at
// most kBinCap) are ranked among themselves, and the selected keys are
// written out by one order-keeping compaction: out[0..k) ascending indices,
// and *kth (shared) = the smallest selected key, also stored to *pub (global,
// optional) as soon as it is known.
// Returns false, having written nothing, when that digit holds more than
// kBinCap keys (many equal scores); the caller then runs select_block.
// hist: kWideBins counters; bin_keys: kBinCap keys of scratch.
constexpr int kBinCap = 256;
__device__ __forceinline__ bool select_small(const uint64_t *keys, int n, int k, int32_t *out, uint32_t *hist,
                                          uint64_t *bin_keys, uint64_t *kth, uint64_t *pub) {
  __shared__ int n_bin;
  const int t = threadIdx.x;
  const uint64_t x = t < n ? keys[t] : 0ull;
  const uint32_t hi = (uint32_t)(x >> 32);
  if (t == 0) n_bin = 0;
  const WideDigit wd = wide_digit([&](int i) { return (uint32_t)(keys[i] >> 32); }, n, hist);
  const int sh = wd.sh < 0 ? 0 : wd.sh;
  const int d = wd.sh < 0 ? 0 : (int)((hi >> sh) & (kWideBins - 1));
  if (t < n) atomicAdd(&hist[d], 1u);
  __syncthreads();
  uint32_t above;
  const int D = wide_find(hist, k, &above);
  const int in_d = (int)hist[D], take_d = k - (int)above;   // keys of digit D, and how many of them are kept
  if (in_d > kBinCap) {                                      // uniform: every thread read the same counts
    __syncthreads();                                         // hist is read; the caller may reuse it
    return false;
  }
  if (t < n && d == D) bin_keys[atomicAdd(&n_bin, 1)] = x;
  __syncthreads();
  int selected = 0;
  if (t < n) {
    if (d > D) {
      selected = 1;
    } else if (d == D) {
      int r = 0;                                             // keys of digit D larger than this one
      for (int j = 0; j < in_d; j++) r += bin_keys[j] > x ? 1 : 0;
      selected = r < take_d;
      if (r == take_d - 1) {                                 // exactly one key (1 <= take_d <= in_d)
        *kth = x;
        if (pub != nullptr) ptx::st_relaxed_u64(pub, x);
      }
    }
  }
  int total;
  const int pos = block_excl_scan(selected, &total);
  if (selected) out[pos] = (int32_t)(~(uint32_t)(x & 0xFFFFFFFFu));
  __syncthreads();
  return true;
}

// Exact top-k of n unique nonzero keys in shared memory (n <= kCandCap), for
// candidate sets a little larger than k.  The k-th largest key is found on
// the score halves (sk[i] = keys[i] >> 32) by a radix-256 search, then, among
// the keys tied on that score, on the index halves.  The block then compacts
// the selected indices and places them in ascending order by bucketing them
// by index (buckets of power-of-two width; a few indices per bucket).  keys
// and sk are reused as scratch.  sel: >= k ints; bins: >= 4096 counters.
// out[0..k): ascending indices, -1 padding.  by_index: keys[] is already in ascending index order; the selected keys are
// then written out by one order-keeping compaction.  kth (shared, optional):
// receives K, the smallest key that is selected or 1 when all are; pub
// (global, optional) too, at once.
__device__ void select_block(uint64_t *keys, uint32_t *sk, int n, int k, int32_t *out, int32_t *sel,
                                          uint32_t *bins, bool by_index = false, uint64_t *kth = nullptr,
                                          uint64_t *pub = nullptr) {
  __shared__ int cnt_sh[2];
  __shared__ int n_sel;
  __shared__ uint32_t red_slots[2][32];
  BlockReduce br{red_slots, 0};
  const int take = min(k, n);
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) { n_sel = 0; cnt_sh[0] = 0; cnt_sh[1] = 0; }
  uint64_t K = 1;                                    // keys >= K are selected
  if (take < n) {
    const uint32_t t32 = block_kth256(sk, n, take, 0, bins);
    int c_gt = 0, c_eq = 0;
    for (int i = threadIdx.x; i < n; i += blockDim.x) { c_gt += sk[i] > t32; c_eq += sk[i] == t32; }
    c_gt = warp_sum(c_gt);
    c_eq = warp_sum(c_eq);
    if (lane == 0) { atomicAdd(&cnt_sh[0], c_gt); atomicAdd(&cnt_sh[1], c_eq); }
    __syncthreads();
    const int need = take - cnt_sh[0];
    uint32_t tlo = 0u;
    if (need < cnt_sh[1]) {
      // several keys tie on the score: the `need` largest index halves among them
      for (int i = threadIdx.x; i < n; i += blockDim.x) sk[i] = sk[i] == t32 ? (uint32_t)keys[i] : 0u;
      __syncthreads();
      tlo = block_kth256(sk, n, need, 0, bins);
    }
    K = ((uint64_t)t32 << 32) | tlo;
  }
  if (kth != nullptr && threadIdx.x == 0) {
    *kth = K;
    if (pub != nullptr) ptx::st_relaxed_u64(pub, K);
  }
  __syncthreads();
  if (by_index) {
    // thread t keeps keys [t * per, t * per + per) in order
    const int per = (n + blockDim.x - 1) / blockDim.x, i0 = threadIdx.x * per;
    int c = 0;
    for (int j = 0; j < per; j++) c += (i0 + j < n && keys[i0 + j] >= K) ? 1 : 0;
    int total;
    int pos = block_excl_scan(c, &total);
    for (int j = 0; j < per; j++) {
      const int i = i0 + j;
      if (i < n && keys[i] >= K) {
        const int32_t idx = (int32_t)(~(uint32_t)(keys[i] & 0xFFFFFFFFu));
        out[pos++] = idx;
      }
    }
    for (int i = take + threadIdx.x; i < k; i += blockDim.x) out[i] = -1;
    __syncthreads();
    return;
  }
  // ---- compact the selected indices
  for (int b0 = 0; b0 < n; b0 += blockDim.x) {
    const int i = b0 + threadIdx.x;
    const uint64_t x = i < n ? keys[i] : 0ull;
    const bool ok = x != 0ull && x >= K;
    const unsigned bal = __ballot_sync(0xFFFFFFFFu, ok);
    if (!bal) continue;
    int base = 0;
    if (lane == 0) base = atomicAdd(&n_sel, __popc(bal));
    base = __shfl_sync(0xFFFFFFFFu, base, 0) + __popc(bal & ((1u << lane) - 1u));
    if (ok) sel[base] = (int32_t)(~(uint32_t)(x & 0xFFFFFFFFu));
  }
  __syncthreads();
  // ---- ascending index order: 2,048 index buckets (counts, cursors); the
  // key buffer (the keys are in registers now) receives them bucket by bucket
  uint32_t *h2 = bins, *c2 = bins + 2048;
  for (int i = threadIdx.x; i < 4096; i += blockDim.x) bins[i] = 0;
  int mx = 0;
  for (int i = threadIdx.x; i < take; i += blockDim.x) mx = max(mx, sel[i]);
  const int max_idx = (int)br.run<true>((uint32_t)mx);  // its barrier also orders the clearing above
  const int sh2 = max(0, 32 - __clz(max_idx) - 11);    // (max index >> sh2) < 2048
  for (int i = threadIdx.x; i < take; i += blockDim.x) atomicAdd(&h2[sel[i] >> sh2], 1u);
  __syncthreads();
  block_offsets<false>(h2, 2048);                      // h2[b] <- indices in the buckets below b
  int32_t *by = reinterpret_cast<int32_t *>(keys);
  for (int i = threadIdx.x; i < take; i += blockDim.x) {
    const int b = sel[i] >> sh2;
    by[h2[b] + atomicAdd(&c2[b], 1u)] = sel[i];
  }
  __syncthreads();
  for (int p = threadIdx.x; p < take; p += blockDim.x) {
    const int32_t v = by[p];
    const int b = v >> sh2;
    const int start = (int)h2[b], cnt = (int)c2[b];
    int r = 0;
    for (int j = start; j < start + cnt; j++) r += by[j] < v;   // buckets hold very few indices
    out[start + r] = v;
  }
  for (int i = take + threadIdx.x; i < k; i += blockDim.x) out[i] = -1;
  __syncthreads();
}

// ---------------------------------------------------------------- direct path
// Shared memory of the direct path for rows of up to `cap` items (a multiple
// of 4, <= kDirectCap): keys [cap] | sel [kMaxK] | 32 warp histograms [32][256]
// | score halves sk [max(min(cap, kCandCap), 4096)] (rows of n <= cap keys, or
// their group maxima, or the candidates above their threshold): short rows
// (a prefill's) take less of it.
__host__ __device__ constexpr int direct_sk_cap(int cap) { return (cap < kCandCap ? cap : kCandCap) > 4096 ? (cap < kCandCap ? cap : kCandCap) : 4096; }
// the warp histograms' region in words (also the exact selection's 4,096
// bucket counters, and the candidates of the group-maxima path as 64-bit keys)
__host__ __device__ constexpr int direct_whist_words(int threads) {
  return (threads / 32) * 256 > 4096 ? (threads / 32) * 256 : 4096;
}
__host__ __device__ constexpr size_t direct_smem_bytes(int cap, int threads) {
  return (size_t)cap * 8 + (size_t)kMaxK * 4 + (size_t)direct_whist_words(threads) * 4 + (size_t)direct_sk_cap(cap) * 4;
}
// rows of up to this many items take a CTA of 256 threads (three per SM),
// longer ones 1,024
constexpr int kDirectSmallItems = 4096;

__global__ void __launch_bounds__(kTopkThreads) topk_direct_kernel(TopkSrc S, int k, int32_t *__restrict__ out,
                                                                    int *status, int cap) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  uint64_t *keys = reinterpret_cast<uint64_t *>(smem_raw);                       // [cap]
  int32_t *sel = reinterpret_cast<int32_t *>(keys + cap);                        // [kMaxK]
  __shared__ SelectShared sh;
  sh.whist = reinterpret_cast<uint32_t *>(sel + kMaxK);                          // [32][256]
  __shared__ int n_keys;
  griddep_wait();
  griddep_launch();
  const int q = blockIdx.x;
  const int nv = query_nv(S, q, status);
  if (threadIdx.x == 0) n_keys = 0;
  __syncthreads();
  // the row's keys, compacted into shared memory (uniform trip counts:
  // ballots see full warps)
  auto put = [&](bool v, uint64_t key) {
    const unsigned ballot = __ballot_sync(0xFFFFFFFFu, v);
    int base = 0;
    if ((threadIdx.x & 31) == 0 && ballot) base = atomicAdd(&n_keys, __popc(ballot));
    base = __shfl_sync(0xFFFFFFFFu, base, 0);
    if (v) keys[base + __popc(ballot & ((1u << (threadIdx.x & 31)) - 1u))] = key;
  };
  if (S.pool != nullptr && S.bmax != nullptr) {
    // Pool rows with the indexer's block maxima: a lower bound T of the k-th
    // largest block maximum is one of the k-th largest item too (at least k
    // blocks reach it, each with an item at its maximum), so only the blocks
    // reaching T are read, item by item, and the exact selection runs on
    // their items that reach T.  T is taken two radix steps deep (16 bits
    // below the bits all maxima share), which is enough to leave few more
    // candidates than k.  Where the blocks hold more items than the
    // selection's buffer, the whole row is read as below.
    uint32_t *bm = sh.whist + direct_whist_words(blockDim.x);                   // [kPoolBlocks]
    int32_t *cb = reinterpret_cast<int32_t *>(keys + cap) ;                      // (sel) [kPoolBlocks]
    __shared__ int n_cb;
    __shared__ uint32_t T_bm;
    const uint32_t *src = S.bmax + (int64_t)q * S.bstride;
    for (int i = threadIdx.x; i < kPoolBlocks; i += blockDim.x) bm[i] = __ldg(src + i);
    if (threadIdx.x == 0) n_cb = 0;
    __syncthreads();
    const uint32_t t = block_kth256(bm, kPoolBlocks, k < kPoolBlocks ? k : kPoolBlocks, 0, sh.whist, 2);
    if (threadIdx.x == 0) T_bm = t;
    __syncthreads();
    const uint32_t T = T_bm;
    for (int b0 = 0; b0 < kPoolBlocks; b0 += blockDim.x) {
      const int b = b0 + threadIdx.x;
      const bool c = b < kPoolBlocks && bm[b] != 0u && bm[b] >= T;
      const unsigned bal = __ballot_sync(0xFFFFFFFFu, c);
      int base = 0;
      if ((threadIdx.x & 31) == 0 && bal) base = atomicAdd(&n_cb, __popc(bal));
      base = __shfl_sync(0xFFFFFFFFu, base, 0);
      if (c) cb[base + __popc(bal & ((1u << (threadIdx.x & 31)) - 1u))] = b;
    }
    __syncthreads();
    const int ncb = n_cb, total = ncb * kBlock;
    if (total <= direct_sk_cap(cap) && total <= 8 * (int)blockDim.x) {
      // the candidate blocks' items: all loads out before the first ballot
      constexpr int kBatch = 8;
      const float *row = S.scores + (int64_t)q * S.stride;
      float sv[kBatch];
      int bv[kBatch], iv[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; u++) {
        const int idx = u * blockDim.x + threadIdx.x;
        const int b = idx < total ? cb[idx >> 3] : 0;
        iv[u] = b * kBlock + (idx & 7);
        sv[u] = idx < total ? __ldg(row + iv[u]) : 0.f;
        bv[u] = idx < total ? __ldg(S.pool + (int64_t)q * kPoolBlocks + b) : -1;
      }
      __syncthreads();                                   // cb (in sel) is read: the selection may reuse it
#pragma unroll
      for (int u = 0; u < kBatch; u++) {
        if (u * (int)blockDim.x >= total) break;
        const int idx = u * blockDim.x + threadIdx.x;
        uint64_t key = 0;
        const bool v = idx < total && item_key_of(S, iv[u], nv, sv[u], bv[u], key, status);
        put(v && (uint32_t)(key >> 32) >= T, key);
      }
      __syncthreads();
      const int n = n_keys;
      uint32_t *sk = bm;                                 // (the block maxima are no longer read)
      for (int i = threadIdx.x; i < ((n + 3) & ~3); i += blockDim.x) sk[i] = i < n ? (uint32_t)(keys[i] >> 32) : 0u;
      __syncthreads();
      select_block(keys, sk, n, k, out + (int64_t)q * k, sel, sh.whist);
      return;
    }
    if (threadIdx.x == 0) n_keys = 0;
    __syncthreads();
  }
  if (S.pool != nullptr) {
    // pool mode (rows of 16,384 items): scores and block ids kBatch rounds
    // at a time, all loads out before the first ballot: one round trip per
    // batch instead of per round (measured: no gain for a prefill's shorter
    // rows, whose items past the visible length are not read at all)
    constexpr int kBatch = 8;
    const float *row = S.scores + (int64_t)q * S.stride;
    for (int64_t b0 = 0; b0 < S.n_items; b0 += (int64_t)kBatch * blockDim.x) {
      float sv[kBatch];
      int bv[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; u++) {
        const int64_t i = b0 + (int64_t)u * blockDim.x + threadIdx.x;
        sv[u] = i < S.n_items ? __ldg(row + i) : 0.f;
        bv[u] = i < S.n_items && S.pool != nullptr ? __ldg(S.pool + (int64_t)q * kPoolBlocks + (i >> 3)) : 0;
      }
#pragma unroll
      for (int u = 0; u < kBatch; u++) {
        if (b0 + (int64_t)u * blockDim.x >= S.n_items) break;
        const int64_t i = b0 + (int64_t)u * blockDim.x + threadIdx.x;
        uint64_t key = 0;
        put(i < S.n_items && item_key_of(S, i, nv, sv[u], bv[u], key, status), key);
      }
    }
  } else {
    for (int64_t b0 = 0; b0 < S.n_items; b0 += blockDim.x) {
      const int64_t i = b0 + threadIdx.x;
      uint64_t key = 0;
      put(i < S.n_items && item_key(S, q, i, nv, key, status), key);
    }
  }
  __syncthreads();
  const int n = n_keys;
  int32_t *oq = out + (int64_t)q * k;
  uint32_t *sk = sh.whist + direct_whist_words(blockDim.x);                     // [direct_sk_cap(cap)]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  // Larger sets: a threshold from the maxima of groups of gsz keys (the
  // largest power of two <= 32 leaving >= 4k groups): at least k groups reach
  // the k-th largest maximum T, so the top-k keys all have scores >= T; those
  // candidates go to select_block.  Sets too small for groups of two (fewer
  // than 8k keys) go to select_block whole, as do sets of <= 2,048.
  int gsz = 32;
  while (gsz > 1 && n / gsz < 4 * k) gsz >>= 1;
  if (n <= 2048 || (gsz < 2 && n <= direct_sk_cap(cap))) {
    for (int i = threadIdx.x; i < ((n + 3) & ~3); i += blockDim.x) sk[i] = i < n ? (uint32_t)(keys[i] >> 32) : 0u;
    __syncthreads();
    select_block(keys, sk, n, k, oq, sel, sh.whist);
    return;
  }
  bool done = false;
  if (gsz >= 2) {
    __shared__ uint32_t T_sh;
    __shared__ int n_c;
    const int ng = (n + gsz - 1) / gsz;
    // group maxima of the score halves: gsz lanes per group
    for (int b0 = warp * 32; b0 < ng * gsz; b0 += nw * 32) {
      const int i = b0 + lane;
      uint32_t v = i < n ? (uint32_t)(keys[i] >> 32) : 0u;
      for (int o = 1; o < gsz; o <<= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
      if ((lane & (gsz - 1)) == 0 && i / gsz < ng) sk[i / gsz] = v;
    }
    for (int i = ng + threadIdx.x; i < ((ng + 3) & ~3); i += blockDim.x) sk[i] = 0u;
    if (threadIdx.x == 0) { T_sh = 1u; n_c = 0; }
    __syncthreads();
    if (ng > k) {
      const uint32_t t = block_kth256(sk, ng, k, 16, reinterpret_cast<uint32_t *>(sel));
      if (threadIdx.x == 0) T_sh = t;
    }
    __syncthreads();
    const uint32_t T = T_sh;
    uint64_t *cand = reinterpret_cast<uint64_t *>(sh.whist);                     // [kDirCand]
    const int kDirCand = direct_whist_words(blockDim.x) / 2;
    for (int b0 = 0; b0 < n; b0 += blockDim.x) {
      const int i = b0 + threadIdx.x;
      const uint64_t x = i < n ? keys[i] : 0ull;
      const bool ok = i < n && (uint32_t)(x >> 32) >= T;
      const unsigned bal = __ballot_sync(0xFFFFFFFFu, ok);
      if (!bal) continue;
      int base = 0;
      if (lane == 0) base = atomicAdd(&n_c, __popc(bal));
      base = __shfl_sync(0xFFFFFFFFu, base, 0) + __popc(bal & ((1u << lane) - 1u));
      if (ok && base < kDirCand) cand[base] = x;
    }
    __syncthreads();
    const int nc = n_c;
    if (nc <= kDirCand) {
      for (int i = threadIdx.x; i < ((nc + 3) & ~3); i += blockDim.x) sk[i] = i < nc ? (uint32_t)(cand[i] >> 32) : 0u;
      __syncthreads();
      select_block(cand, sk, nc, k, oq, sel, reinterpret_cast<uint32_t *>(keys));  // keys is free: bucket counters
      done = true;
    }
  }
  if (!done) {
    auto get = [&](int64_t i, uint64_t &key) { key = keys[i]; return true; };
    select_and_write(get, n, n, k, oq, sh, sel);
  }
}

// ---------------------------------------------------------------- long rows
// Two streaming passes over the row.  Pass 1 writes the maximum key of every
// supergroup of SGI consecutive items (SGI a power of two, so that a row has
// about 4k supergroups).  Pass 2 (P CTAs per row) takes T = the k-th largest
// supergroup maximum with its low 16 bits cleared: at least k supergroups
// reach T, so at least k items do, so the k-th best item key is >= T and every
// top-k item has a key >= T.  The P CTAs of a row form one thread-block
// cluster.  Each streams its share of the row and gathers the items with key
// >= T (a small superset of the top-k) in its own shared memory; after a
// cluster barrier, CTA 0 reads every CTA's candidates through distributed
// shared memory and runs the exact selection on them, or on the whole row if
// they overflow its buffer.  A second cluster barrier keeps the other CTAs
// (and their shared memory) alive until CTA 0 has read them.
//
// Workspace, per row q: smax[q][sstride] (the supergroup maxima, 0 = no valid
// item); slots past a row's valid length are never read.
constexpr int kCollectThreads = 1024;
constexpr int kSuperCap = 16384;    // supergroups per row (held in shared memory by pass 2)


// Items per supergroup: the largest power of two in [8, 512] that leaves at
// least 4k supergroups, doubled further while a row has more than kSuperCap.
__host__ __device__ inline int64_t long_row_sgi(int64_t n_items, int k) {
  int64_t sgi = 512;
  while (sgi > 8 && n_items / sgi < 4 * (int64_t)k) sgi >>= 1;
  while ((n_items + sgi - 1) / sgi > kSuperCap) sgi <<= 1;
  return sgi;
}

__host__ __device__ inline LongRowWs long_row_ws(void *ws, int n_q, int64_t n_items, int k) {
  LongRowWs w;
  const int64_t sgi = long_row_sgi(n_items, k);
  w.sstride = ((n_items + sgi - 1) / sgi + 3) / 4 * 4;
  w.smax = static_cast<uint32_t *>(ws);
  return w;
}

__host__ __device__ inline size_t long_row_ws_bytes(int n_q, int64_t n_items, int k) {
  const LongRowWs w = long_row_ws(nullptr, n_q, n_items, k);
  return (size_t)n_q * (size_t)w.sstride * 4;
}

// Pass 1.  A warp step covers 32 x IPL items: plain rows one float4 (IPL = 4)
// per lane, block rows one item per lane.  A warp takes four steps at a time
// (four loads in flight per lane) and a pass of max(sgi, 4 steps) items, so
// no two warps share a supergroup.  Supergroups smaller than a step reduce
// over sgi / IPL lanes; larger ones over the whole warp and over steps.
template <bool kPlain>
__global__ void __launch_bounds__(256) topk_smax_kernel(TopkSrc S, int64_t sgi, LongRowWs W, int *status) {
  constexpr int IPL = kPlain ? 4 : 1;
  constexpr int64_t kStep = 32 * IPL;
  griddep_wait();
  griddep_launch();
  const int q = blockIdx.y;
  const int nv = query_nv(S, q, status);
  const int lane = threadIdx.x & 31;
  const int64_t wid = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t n_warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int lsg = __ffsll(sgi) - 1;
  uint32_t *sq = W.smax + (int64_t)q * W.sstride;
  const float *row = S.scores + (int64_t)q * S.stride;
  const bool row16 = (reinterpret_cast<uintptr_t>(row) & 15u) == 0;
  const int64_t span = sgi > 4 * kStep ? sgi : 4 * kStep;
  const int64_t n_pass = (S.n_items + span - 1) / span;
  for (int64_t w = wid; w < n_pass; w += n_warps) {
    uint32_t acc = 0;
    for (int64_t c0 = w * span; c0 < (w + 1) * span; c0 += 4 * kStep) {
      uint32_t m[4];
#pragma unroll
      for (int u = 0; u < 4; u++) {
        const int64_t i0 = c0 + u * kStep + lane * IPL;
        m[u] = 0;
        if (kPlain) {
          if (i0 < nv) {
            if (row16 && i0 + 4 <= nv) {
              const float4 v = __ldg(reinterpret_cast<const float4 *>(row + i0));
              m[u] = order_key(fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)));   // order_key is monotonic
            } else {                                 // ragged end or unaligned row
              for (int j = 0; j < 4; j++)
                if (i0 + j < nv) m[u] = max(m[u], order_key(__ldg(row + i0 + j)));
            }
          }
        } else {
          uint64_t key;
          if (i0 < S.n_items && item_key(S, q, i0, nv, key, status)) m[u] = (uint32_t)(key >> 32);
        }
      }
      if (sgi < kStep) {
#pragma unroll
        for (int u = 0; u < 4; u++) {
          uint32_t x = m[u];
          for (int o = 1; o < sgi / IPL; o <<= 1) x = max(x, __shfl_xor_sync(0xFFFFFFFFu, x, o));
          const int64_t i0 = c0 + u * kStep + lane * IPL;
          if ((lane & (sgi / IPL - 1)) == 0 && i0 < S.n_items) sq[i0 >> lsg] = x;
        }
      } else {
        uint32_t xs[4];
#pragma unroll
        for (int u = 0; u < 4; u++) xs[u] = __reduce_max_sync(0xFFFFFFFFu, m[u]);
        if (sgi <= 2 * kStep) {                      // one or two steps per supergroup
#pragma unroll
          for (int u = 0; u < 4; u++) {
            if (sgi == 2 * kStep && (u & 1)) continue;
            const uint32_t x = sgi == 2 * kStep ? max(xs[u], xs[u | 1]) : xs[u];
            const int64_t i0 = c0 + u * kStep;
            if (lane == 0 && i0 < S.n_items) sq[i0 >> lsg] = x;
          }
        } else {
          acc = max(acc, max(max(xs[0], xs[1]), max(xs[2], xs[3])));
        }
      }
    }
    if (sgi > 2 * kStep && lane == 0 && w * span < S.n_items) sq[(w * span) >> lsg] = acc;
  }
}

// Distributed shared memory of the cluster: the address of this CTA's
// shared-memory location p in the CTA of cluster rank r, and loads from it.
__device__ __forceinline__ uint32_t dsmem_addr(const void *p, uint32_t r) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(a)
               : "r"((uint32_t)__cvta_generic_to_shared(p)), "r"(r));
  return a;
}
__device__ __forceinline__ uint32_t dsmem_ld32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ void dsmem_st32(uint32_t a, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}
__device__ __forceinline__ void dsmem_st64(uint32_t a, uint64_t v) {
  asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(a), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t dsmem_ld64(uint32_t a) {
  uint64_t v;
  asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(a) : "memory");
  return v;
}
// Every thread of every CTA of the cluster; orders shared-memory writes before
// the barrier with reads after it, across the cluster.
__device__ __forceinline__ void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
constexpr int kMaxCluster = 16;
static_assert(kMaxCluster <= kHandCtas && kHandSeg >= 256, "handoff segments");

// Puts the n <= 256 unique keys lc[0..n) in ascending index order (rank = the
// number of larger index halves, the index halves being ~index): tpe lanes of
// a warp count for one key, each over every tpe-th key.  Block-wide
// (blockDim.x == 1024); ends with lc written, not with a barrier.
constexpr int kSortCap = 256;
__device__ __forceinline__ void sort_by_index(uint64_t *lc, int n) {
  const int tpe = n <= 32 ? 32 : n <= 64 ? 16 : n <= 128 ? 8 : 4;
  const int e = (int)threadIdx.x / tpe, sub = (int)threadIdx.x & (tpe - 1);
  uint64_t mine = 0;
  int r = 0;
  if (e < n) {
    mine = lc[e];
    const uint32_t lo = (uint32_t)mine;
    for (int j = sub; j < n; j += tpe) r += (uint32_t)lc[j] > lo ? 1 : 0;
  }
  for (int o = tpe >> 1; o > 0; o >>= 1) r += __shfl_xor_sync(0xFFFFFFFFu, r, o);
  __syncthreads();
  if (e < n && sub == 0) lc[r] = mine;
}

// Pass 2: grid (P, n_q), clusters of P CTAs along x (P <= kMaxCluster): the
// cluster rank of a CTA is blockIdx.x.  No thread returns before the second
// cluster barrier.
// GROUPS: plain rows with the indexer's unit partial maxima (parts == 4) and
// 32-entry group maxima (csa2_decode's plan for 1M rows); compiled on its own,
// without the code of the other paths, since it runs once per step with cold
// instruction caches.
template <bool GROUPS>
__global__ void __launch_bounds__(kCollectThreads) topk_collect_kernel(TopkSrc S, int64_t sgi, int parts, int k,
                                                                       LongRowWs W, int32_t *__restrict__ out,
                                                                       int *status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  uint64_t *keys = reinterpret_cast<uint64_t *>(smem_raw);               // [kCandCap] (CTA 0)
  int32_t *sel = reinterpret_cast<int32_t *>(keys + kCandCap);           // [kMaxK]
  uint32_t *sv = reinterpret_cast<uint32_t *>(sel + kMaxK);              // [kSuperCap] supergroup maxima
  __shared__ SelectShared sh;
  sh.whist = sv + kSuperCap;                                             // [32][256]
  __shared__ uint32_t T_sh;
  __shared__ int n_vs, n_lc, lc_sorted, n_g;
  __shared__ int c_off[kMaxCluster + 1], c_bad, c_sorted;
  __shared__ int c_cnt[kMaxCluster], c_srt[kMaxCluster];   // (CTA 0) pushed by every CTA of the cluster
  __shared__ uint64_t kth_sh;                                // (CTA 0) the smallest selected key
  griddep_wait();
  griddep_launch();
  const int q = blockIdx.y, P = gridDim.x, part = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const bool plain = GROUPS || (S.pool == nullptr && S.block == 1);
  // Plain rows with the maxima of their 32-entry groups as well (written by
  // the indexer's epilogue, parts == 4): CTA p of the cluster takes the groups
  // [g_lo, g_hi) of the row and streams only those reaching T, about one per
  // listed supergroup, instead of listing supergroups and streaming all of
  // their entries.  Its groups' maxima are loaded up front, with the
  // supergroup maxima, before the row's length is known (slots past it hold
  // stale values and are masked once it is).
  constexpr bool by_groups = GROUPS;
  const int gps = (int)(sgi >> 5);                                       // groups per supergroup
  const int64_t g_all = (W.sstride / 4) * gps;                           // group slots of a row
  const int64_t g_lo = part * g_all / P, g_hi = (part + 1) * g_all / P;
  constexpr int kGPre = 4;
  uint32_t gpre[kGPre];
  const uint32_t *gq = W.gmax + (int64_t)q * W.gstride;
  if (by_groups) {
#pragma unroll
    for (int j = 0; j < kGPre; j++) {
      const int64_t gid = g_lo + threadIdx.x + (int64_t)j * blockDim.x;
      gpre[j] = gid < g_hi ? __ldcg(gq + gid) : 0u;
    }
  }
  // the supergroup maxima: 16-B loads over every slot of the row
  const uint4 *src = reinterpret_cast<const uint4 *>(W.smax + (int64_t)q * W.sstride);
  const int n_vec = (int)(W.sstride / 4);
  uint4 vpre[2];
#pragma unroll
  for (int j = 0; j < 2; j++) {
    const int i = threadIdx.x + j * blockDim.x;
    vpre[j] = i < n_vec ? __ldcg(src + i) : make_uint4(0u, 0u, 0u, 0u);
  }
  const int nv = query_nv(S, q, status);
  const int pf_seq = S.kv_pf != nullptr ? __ldg(S.q_seq + q) : -1;   // used at the end
  const int64_t valid_items = plain ? nv : (S.pool != nullptr ? S.n_items : ((int64_t)nv + kBlock - 1) / kBlock);
  const int ns = (int)((valid_items + sgi - 1) / sgi);                   // supergroups that may hold a valid item
  if (threadIdx.x == 0) { n_vs = 0; T_sh = 1u; n_lc = 0; n_g = 0; }    // T = 1: every valid item
  __syncthreads();
  // parts == 4: each supergroup's maximum is stored as four partial maxima.
  {
    int vs = 0;
    for (int i = threadIdx.x; i < n_vec; i += blockDim.x) {
      const int j = (i - threadIdx.x) / blockDim.x;
      const uint4 v = j < 2 ? vpre[j] : __ldcg(src + i);
      if (parts == 4) {
        if (i < ns) {
          const uint32_t x = max(max(v.x, v.y), max(v.z, v.w));
          sv[i] = x;
          vs += x != 0u;
        }
      } else {
        const uint32_t e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int jj = 0; jj < 4; jj++) {
          if (4 * i + jj < ns) {
            sv[4 * i + jj] = e[jj];
            vs += e[jj] != 0u;
          }
        }
      }
    }
    vs = __reduce_add_sync(0xFFFFFFFFu, vs);
    if (lane == 0 && vs) atomicAdd(&n_vs, vs);
  }
  __syncthreads();
  // ---- T: a lower bound of the k-th largest supergroup maximum, exact in
  // the 12 (or 24) bits below the leading bits all maxima share
  if (n_vs > k) {
    const uint32_t t = block_kth_bound12(sv, ns, k, sh.whist);
    if (threadIdx.x == 0) T_sh = t;
  }
  __syncthreads();
  const uint32_t T = T_sh;
  uint64_t *lc = reinterpret_cast<uint64_t *>(sv);    // this CTA's keys >= T (over sv, once T is known)
  constexpr int kLocalCap = kSuperCap / 2;
  {
    const float *row = S.scores + (int64_t)q * S.stride;
    const bool row16 = (reinterpret_cast<uintptr_t>(row) & 15u) == 0;
    int32_t *slist = reinterpret_cast<int32_t *>(keys);
    int nsl = 0;
    if (!by_groups) {
      // ---- list the supergroups that reach T in index order; this CTA takes a
      // contiguous, equal share of that list (ranks [r_lo, r_hi)), so that the
      // CTAs' candidates follow one another in index order and every CTA streams
      // the same number of supergroups however they bunch together
      const int run = (ns + blockDim.x - 1) / blockDim.x, g0 = threadIdx.x * run;   // this thread's supergroups
      int c = 0;
      for (int j = 0; j < run; j++) {
        const int i = g0 + j;
        c += (i < ns && sv[i] >= T && sv[i] != 0u) ? 1 : 0;
      }
      int n_listed;
      int rank = block_excl_scan(c, &n_listed);
      const int r_lo = (int)((int64_t)part * n_listed / P), r_hi = (int)((int64_t)(part + 1) * n_listed / P);
      for (int j = 0; j < run && rank < r_hi; j++) {
        const int i = g0 + j;
        if (i < ns && sv[i] >= T && sv[i] != 0u) {
          if (rank >= r_lo) slist[rank - r_lo] = i;
          rank++;
        }
      }
      __syncthreads();
      nsl = r_hi - r_lo;
    }
    const int64_t total = (int64_t)nsl * sgi;                 // items of the listed supergroups
    if (by_groups) {
      // ---- this CTA's groups that reach T (their maxima were loaded up front)
      constexpr int kGCap = 32 * 256;
      int32_t *glist = reinterpret_cast<int32_t *>(sh.whist);   // [kGCap]: free since T was found
      const int64_t g_valid = (int64_t)ns * gps;                 // groups of the supergroups holding valid entries
      for (int64_t b0 = g_lo, j = 0; b0 < g_hi; b0 += blockDim.x, j++) {   // uniform trip count
        const int64_t gid = b0 + threadIdx.x;
        const uint32_t m0 = gpre[0];                             // this pass's prefetched maximum
#pragma unroll
        for (int t = 0; t + 1 < kGPre; t++) gpre[t] = gpre[t + 1];
        gpre[kGPre - 1] = 0u;
        bool ok = false;
        if (gid < g_hi && gid < g_valid) {
          const uint32_t m = j < kGPre ? m0 : __ldcg(gq + gid);
          ok = m >= T && m != 0u;
        }
        const unsigned bal = __ballot_sync(0xFFFFFFFFu, ok);
        if (bal == 0u) continue;
        int base = 0;
        if (lane == 0) base = atomicAdd(&n_g, __popc(bal));
        base = __shfl_sync(0xFFFFFFFFu, base, 0) + __popc(bal & ((1u << lane) - 1u));
        if (ok && base < kGCap) glist[base] = (int32_t)gid;
      }
      __syncthreads();
      // too many groups for the list: report an overflowing candidate list,
      // so that the row is selected exactly from its scores instead
      const int ng = n_g <= kGCap ? n_g : 0;
      if (n_g > kGCap && threadIdx.x == 0) n_lc = kLocalCap + 1;
      for (int b0 = 0; b0 < ng * 8; b0 += blockDim.x) {        // 8 threads per group, a float4 each
        const int j = b0 + threadIdx.x;
        float4 v = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        int64_t e0 = -1;
        if (j < ng * 8) {
          e0 = (int64_t)glist[j >> 3] * 32 + (j & 7) * 4;
          if (row16 && e0 + 4 <= nv) {
            v = __ldcg(reinterpret_cast<const float4 *>(row + e0));
          } else {
            if (e0 < nv) v.x = __ldcg(row + e0);
            if (e0 + 1 < nv) v.y = __ldcg(row + e0 + 1);
            if (e0 + 2 < nv) v.z = __ldcg(row + e0 + 2);
            if (e0 + 3 < nv) v.w = __ldcg(row + e0 + 3);
          }
        }
#pragma unroll
        for (int e = 0; e < 4; e++) {
          const float x = e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
          const bool ok = e0 >= 0 && e0 + e < nv && order_key(x) >= T;
          const unsigned bal = __ballot_sync(0xFFFFFFFFu, ok);
          if (bal == 0u) continue;
          int base = 0;
          if (lane == 0) base = atomicAdd(&n_lc, __popc(bal));
          base = __shfl_sync(0xFFFFFFFFu, base, 0) + __popc(bal & ((1u << lane) - 1u));
          if (ok && base < kLocalCap) lc[base] = ((uint64_t)order_key(x) << 32) | (uint32_t)(~(uint32_t)(e0 + e));
        }
      }
    }
    // Plain rows with T above the key of +0: key(x) >= T exactly when the raw
    // bits of x, read as a signed integer, are >= those of T's float (NaN,
    // -0 and the -inf of missing items included).
    const bool fast = plain && T > 0x80000000u;
    const int tb = (int)(T & 0x7FFFFFFFu);
    constexpr int kU = 6;
    const int64_t step = plain ? 4 : 1;
    const int lsg = __ffsll(sgi) - 1;
    for (int64_t b0 = 0; !by_groups && b0 < total; b0 += kU * step * blockDim.x) {
      float4 sc[kU];
      uint64_t gk[kU];
      int64_t base_i[kU];
#pragma unroll
      for (int u = 0; u < kU; u++) {
        const int64_t f = b0 + (u * (int64_t)blockDim.x + threadIdx.x) * step;   // flat position
        sc[u] = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        gk[u] = 0;
        base_i[u] = -1;
        if (f < total) {
          const int64_t i0 = ((int64_t)slist[f >> lsg] << lsg) + (f & (sgi - 1));
          base_i[u] = i0;
          if (plain) {
            if (row16 && i0 + 4 <= nv) {
              sc[u] = __ldcg(reinterpret_cast<const float4 *>(row + i0));
            } else {
              if (i0 < nv) sc[u].x = __ldcg(row + i0);
              if (i0 + 1 < nv) sc[u].y = __ldcg(row + i0 + 1);
              if (i0 + 2 < nv) sc[u].z = __ldcg(row + i0 + 2);
              if (i0 + 3 < nv) sc[u].w = __ldcg(row + i0 + 3);
            }
          } else {
            uint64_t key;
            if (i0 < S.n_items && item_key(S, q, i0, nv, key, status)) gk[u] = key;
          }
        }
      }
      if (fast) {
        // one integer compare per item; then one reservation per warp, each
        // thread writing its own candidates in a run
        int c = 0;
#pragma unroll
        for (int u = 0; u < kU; u++)
          c += (__float_as_int(sc[u].x) >= tb) + (__float_as_int(sc[u].y) >= tb) + (__float_as_int(sc[u].z) >= tb) +
               (__float_as_int(sc[u].w) >= tb);
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
          if (lane >= o) incl += y;
        }
        const int wtot = __shfl_sync(0xFFFFFFFFu, incl, 31);
        if (wtot == 0) continue;                       // most warps of most rounds
        int base = 0;
        if (lane == 31) base = atomicAdd(&n_lc, wtot);
        base = __shfl_sync(0xFFFFFFFFu, base, 31) + incl - c;
        if (c > 0) {
#pragma unroll
          for (int u = 0; u < kU; u++) {
#pragma unroll
            for (int e = 0; e < 4; e++) {
              const float x = e == 0 ? sc[u].x : e == 1 ? sc[u].y : e == 2 ? sc[u].z : sc[u].w;
              if (__float_as_int(x) >= tb) {
                if (base < kLocalCap)
                  lc[base] = ((uint64_t)order_key(x) << 32) | (uint32_t)(~(uint32_t)(base_i[u] + e));
                base++;
              }
            }
          }
        }
        continue;
      }
      // the round's keys >= T: ballots first, then one reservation per warp
      constexpr int kE = 4;                            // items per load (plain rows; block rows use e = 0)
      unsigned bal[kU * kE];
      int cnt = 0;
#pragma unroll
      for (int u = 0; u < kU; u++) {
#pragma unroll
        for (int e = 0; e < kE; e++) {
          bool ok = false;
          if (plain) {
            const float x = e == 0 ? sc[u].x : e == 1 ? sc[u].y : e == 2 ? sc[u].z : sc[u].w;
            ok = base_i[u] >= 0 && base_i[u] + e < nv && order_key(x) >= T;
          } else if (e == 0) {
            ok = gk[u] != 0 && (uint32_t)(gk[u] >> 32) >= T;
          }
          bal[u * kE + e] = __ballot_sync(0xFFFFFFFFu, ok);
          cnt += __popc(bal[u * kE + e]);
        }
      }
      if (cnt == 0) continue;                          // most rounds of most warps
      int base = 0;
      if (lane == 0) base = atomicAdd(&n_lc, cnt);
      base = __shfl_sync(0xFFFFFFFFu, base, 0);
      const unsigned below = (1u << lane) - 1u;
#pragma unroll
      for (int u = 0; u < kU; u++) {
#pragma unroll
        for (int e = 0; e < kE; e++) {
          const unsigned b = bal[u * kE + e];
          if (b & (1u << lane)) {
            const int pos = base + __popc(b & below);
            uint64_t key;
            if (plain) {
              const float x = e == 0 ? sc[u].x : e == 1 ? sc[u].y : e == 2 ? sc[u].z : sc[u].w;
              key = ((uint64_t)order_key(x) << 32) | (uint32_t)(~(uint32_t)(base_i[u] + e));
            } else {
              key = gk[u];
            }
            if (pos < kLocalCap) lc[pos] = key;
          }
          base += __popc(b);
        }
      }
    }
  }
  // ---- a short list is put in index order: the lists of the CTAs, taken
  // in cluster order, then run in index order
  __syncthreads();                                     // lc and n_lc are final
  // L2 prefetch of the latent records of this CTA's candidates (a superset of
  // the selected entries, which the attention gathers next), as soon as they
  // are known: spread over the cluster
  if (plain && pf_seq >= 0 && pf_seq < S.n_seq) {
    const uint8_t *pf = S.kv_pf + (int64_t)pf_seq * S.n_max * kKvBytes;
    const int nl = min(n_lc, kLocalCap);
    for (int i = threadIdx.x; i < 4 * nl; i += blockDim.x) {   // a record spans at most four 128-B lines
      const uint32_t idx = ~(uint32_t)lc[i >> 2];
      if ((int64_t)idx >= S.n_max) continue;
      const uint8_t *rec = pf + (int64_t)idx * kKvBytes;
      asm volatile("prefetch.global.L2 [%0];" ::"l"(rec + ((i & 3) == 3 ? kKvBytes - 1 : (i & 3) * 128)));
    }
  }
  {
    const int nl = n_lc;
    if (nl <= kSortCap) sort_by_index(lc, nl);
    if (threadIdx.x == 0) lc_sorted = nl <= kSortCap ? 1 : 0;
  }
  // ---- every CTA pushes its list into CTA 0's shared memory: slot `part`
  // of keys (slot_cap keys each), with its length and sorted flag; after the
  // cluster barrier CTA 0 holds the cluster's candidates and nobody reads
  // another CTA's shared memory, so the others may leave
  const int slot_cap = kCandCap / P;
  __syncthreads();                                     // the sorted lc is written
  if (W.hand.flag != nullptr) {
    // hand this CTA's candidates to the attention grid (already running): in
    // index order or not at all; they are counted in after the cluster
    // barrier, by when these stores have long landed
    const int nl = n_lc;
    const bool give = nl <= kSortCap && nl <= kHandSeg;
    if (give)
      for (int i = threadIdx.x; i < nl; i += blockDim.x)
        W.hand.cand[((int64_t)q * kHandCtas + part) * kHandSeg + i] = lc[i];
    if (threadIdx.x == 0) W.hand.flag[q * kHandWords + 8 + part] = give ? (uint32_t)nl : kHandFallback;
  }
  {
    const int nl = n_lc;
    const int np = min(nl, min(kLocalCap, slot_cap));
    for (int i = threadIdx.x; i < np; i += blockDim.x) dsmem_st64(dsmem_addr(keys + part * slot_cap + i, 0u), lc[i]);
    if (threadIdx.x == 0) {
      dsmem_st32(dsmem_addr(&c_cnt[part], 0u), (uint32_t)nl);
      dsmem_st32(dsmem_addr(&c_srt[part], 0u), (uint32_t)lc_sorted);
    }
  }
  cluster_barrier();                                   // the pushed lists are in CTA 0
  if (W.hand.flag != nullptr && threadIdx.x == blockDim.x - 1)
    ptx::red_release_add_u32(W.hand.flag + q * kHandWords, 1u);   // this CTA's candidates are out
  if (part == 0) {
    if (warp == 0) {
      const int c = lane < P ? c_cnt[lane] : 0;
      const int srt = lane < P ? c_srt[lane] : 1;
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
      }
      if (lane <= kMaxCluster) c_off[lane] = incl - c;   // c_off[P] = the total
      const bool over = __any_sync(0xFFFFFFFFu, c > kLocalCap || c > slot_cap);
      const bool all_sorted = __all_sync(0xFFFFFFFFu, srt != 0);
      if (lane == 0) {
        c_bad = over ? 1 : 0;
        c_sorted = all_sorted ? 1 : 0;
      }
    }
    __syncthreads();
    if (!c_bad) {
      // close the gaps between the slots: read every key, then write it
      constexpr int kPer = kCandCap / kCollectThreads;
      const int nc = c_off[P];
      uint64_t tmp[kPer];
#pragma unroll
      for (int j = 0; j < kPer; j++) {
        const int i = threadIdx.x + j * kCollectThreads;
        if (i < nc) {
          int r = 0;
          while (i >= c_off[r + 1]) r++;
          tmp[j] = keys[r * slot_cap + (i - c_off[r])];
        }
      }
      __syncthreads();
#pragma unroll
      for (int j = 0; j < kPer; j++) {
        const int i = threadIdx.x + j * kCollectThreads;
        if (i < nc) keys[i] = tmp[j];
      }
    }
  }
  if (part != 0) return;
  int32_t *oq = out + (int64_t)q * k;
  if (threadIdx.x == 0) kth_sh = 1ull;                 // (overwritten by the exact selection)
  uint64_t *kth_pub = W.hand.flag != nullptr ? reinterpret_cast<uint64_t *>(W.hand.flag + q * kHandWords + 2) : nullptr;
  if (!c_bad) {
    const int nc = c_off[P];
    __syncthreads();                                   // lc (over sv) is read above
    for (int i = threadIdx.x; i < ((nc + 3) & ~3); i += blockDim.x)
      sv[i] = i < nc ? (uint32_t)(keys[i] >> 32) : 0u;   // score halves, zero-padded
    __syncthreads();
    // pool items run in slot order, not index order: only plain and block rows keep order
    const bool by_index = c_sorted != 0 && S.pool == nullptr;
    if (!(by_index && nc > k && nc <= (int)blockDim.x &&
          select_small(keys, nc, k, oq, sh.whist, reinterpret_cast<uint64_t *>(sel), &kth_sh, kth_pub)))
      select_block(keys, sv, nc, k, oq, sel, sh.whist, by_index, &kth_sh, kth_pub);
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
    select_and_write(get, S.n_items, nvi, k, oq, sh, sel);
  }
  if (W.hand.flag != nullptr) {
    // the selection (oq) is final
    __syncthreads();
    if (threadIdx.x == 0) {
      ptx::st_relaxed_u64(kth_pub, kth_sh);              // (again, where no exact pass ran)
      ptx::st_release_u32(W.hand.flag + q * kHandWords + 1, 1u);
    }
  }
}

// ---------------------------------------------------------------- host side
static int64_t topk_items(int64_t n_max, int block, bool pool) {
  return pool ? (int64_t)kPoolSlots : (block == 1 ? n_max : (n_max + kBlock - 1) / kBlock);
}

size_t topk_workspace_bytes(int n_q, int64_t n_items, int k) {
  if (n_items <= kDirectCap) return 0;
  return long_row_ws_bytes(n_q, n_items, k);
}

bool topk_items_supported(int64_t n_items, int k) {
  (void)k;
  return n_items < ((int64_t)1 << 31) - 64;          // int32 item indices
}

static size_t collect_smem_bytes() {
  return (size_t)kCandCap * 8 + (size_t)kMaxK * 4 + (size_t)kSuperCap * 4 + 32 * 256 * 4;
}

// Collecting CTAs per row (the cluster size P): one CTA per SM over all rows
// (the shared memory allows one), at most one per 4,096 items, at most 16,
// and no larger than lets all n_q clusters be resident at once (a second wave
// of clusters would double the kernel's time).  Sets the kernel's attributes
// on first use on a device.
static unsigned collect_ctas(int dev, int n_q, int64_t n_items, int reserve = 0) {
  static std::atomic<int> fit[kMaxDevices][kMaxCluster + 1];   // resident clusters of each size + 1 (0: unknown)
  static std::atomic<int> attr_done[kMaxDevices];
  if (dev < 0 || dev >= kMaxDevices) return 1;
  const size_t dsm = collect_smem_bytes();
  once_per_device(attr_done, dev, [&] {
    cudaFuncSetAttribute(topk_collect_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dsm);
    cudaFuncSetAttribute(topk_collect_kernel<false>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    cudaFuncSetAttribute(topk_collect_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dsm);
    cudaFuncSetAttribute(topk_collect_kernel<true>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    cudaGetLastError();                                // a refused attribute leaves no error behind
    return cudaSuccess;
  });
  const int m = device_sm_count(dev);
  int p = (int)std::min<int64_t>(std::min<int64_t>(m / std::max(n_q, 1), n_items / 4096), kMaxCluster);
  if (reserve > 0 && (m - reserve) / std::max(n_q, 1) >= 4) p = std::min(p, (m - reserve) / std::max(n_q, 1));
  for (; p > 1; p--) {
    int f = fit[dev][p].load(std::memory_order_relaxed);
    if (f == 0) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(p, 1);
      cfg.blockDim = dim3(kCollectThreads);
      cfg.dynamicSmemBytes = dsm;
      cudaLaunchAttribute at;
      at.id = cudaLaunchAttributeClusterDimension;
      at.val.clusterDim.x = p;
      at.val.clusterDim.y = 1;
      at.val.clusterDim.z = 1;
      cfg.attrs = &at;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, topk_collect_kernel<false>, &cfg) != cudaSuccess) n = 0;
      cudaGetLastError();
      f = n + 1;
      fit[dev][p].store(f, std::memory_order_relaxed);
    }
    if (f - 1 >= n_q) break;
  }
  return (unsigned)std::max(p, 1);
}

cudaError_t launch_topk(const float *scores, int64_t stride, int n_q, const int32_t *n_valid, int64_t n_max, int k,
                        int block, const int32_t *pool, int32_t *out, void *ws, int *status, cudaStream_t st,
                        const uint32_t *bmax, int64_t bstride) {
  TopkSrc S;
  S.bmax = pool != nullptr ? bmax : nullptr;
  S.bstride = bstride;
  S.scores = scores;
  S.stride = stride;
  S.n_valid = n_valid;
  S.pool = pool;
  S.block = block;
  S.n_max = n_max;
  S.n_items = topk_items(n_max, block, pool != nullptr);
  S.kv_pf = nullptr;
  S.q_seq = nullptr;
  S.n_seq = 0;
  const size_t dsm_direct = direct_smem_bytes(kDirectCap, kTopkThreads);
  const size_t dsm_collect = collect_smem_bytes();
  const int dev = current_device();
  static std::atomic<int> attr_done[kMaxDevices];
  const cudaError_t ea = once_per_device(attr_done, dev, [&] {
    return cudaFuncSetAttribute(topk_direct_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dsm_direct);
  });
  if (ea != cudaSuccess) return ea;
  if (S.n_items <= kDirectCap) {
    const int cap = (int)((S.n_items + 3) / 4 * 4);
    const int threads = S.n_items <= kDirectSmallItems ? 256 : kTopkThreads;
    return launch_pdl(topk_direct_kernel, dim3(n_q), dim3(threads), direct_smem_bytes(cap, threads), st, 1u, S, k,
                      out, status, cap);
  }
  const int64_t sgi = long_row_sgi(S.n_items, k);
  const LongRowWs W = long_row_ws(ws, n_q, S.n_items, k);
  const bool plain = pool == nullptr && block == 1;
  const int64_t span = std::max<int64_t>(sgi, plain ? 4 * 128 : 4 * 32);
  const int64_t n_pass = (S.n_items + span - 1) / span;
  const int64_t gx = std::min<int64_t>((n_pass + 7) / 8, 65535);       // one warp pass per warp
  cudaError_t e = plain ? launch_pdl(topk_smax_kernel<true>, dim3((unsigned)gx, n_q), dim3(256), 0, st, 1u, S, sgi,
                                     W, status)
                        : launch_pdl(topk_smax_kernel<false>, dim3((unsigned)gx, n_q), dim3(256), 0, st, 1u, S, sgi,
                                     W, status);
  if (e != cudaSuccess) return e;
  const unsigned P = collect_ctas(dev, n_q, S.n_items);
  return launch_pdl(topk_collect_kernel<false>, dim3(P, n_q), dim3(kCollectThreads), dsm_collect, st, P, S, sgi, 1, k, W,
                    out, status);
}

// ---------------------------------------------------------------- fused decode
// When the indexer's epilogue writes the supergroup maxima (csa2_decode), the
// selection runs only the collection pass.  mode 3: supergroups are the
// indexer's 512-entry work units, each stored as four partial maxima, plus the
// maxima of their 32-entry groups (only the groups that reach the threshold
// are streamed); mode 2: supergroups of 32 entries; 0: the maxima pass runs
// (other supergroup sizes); -1: rows short enough for one CTA (no scratch).
FusedTopk topk_fused_plan(void *ws, int n_q, int64_t n_max, int k) {
  FusedTopk F;
  F.mode = 0;
  F.sgi = 0;
  F.parts = 1;
  F.W = LongRowWs{};
  F.kv = nullptr;
  F.q_seq = nullptr;
  F.n_seq = 0;
  F.reserve = 0;
  if (n_max <= kDirectCap) { F.mode = -1; return F; }
  const int64_t sgi = long_row_sgi(n_max, k);
  if (sgi != 512 && sgi != 32) return F;
  F.mode = sgi == 512 ? 3 : 2;
  F.sgi = sgi;
  F.parts = sgi == 512 ? 4 : 1;
  LongRowWs &W = F.W;
  W.sstride = sgi == 512 ? (n_max + 511) / 512 * 4 : ((n_max + 31) / 32 + 3) / 4 * 4;
  W.smax = static_cast<uint32_t *>(ws);
  if (F.mode == 3) {
    // then the maxima of the 32-entry groups, [n_q][n_max / 32], 256-B aligned
    W.gstride = (n_max + 511) / 512 * 16;
    const size_t off = ((size_t)n_q * (size_t)W.sstride * 4 + 255) / 256 * 256;
    W.gmax = ws == nullptr ? nullptr : reinterpret_cast<uint32_t *>(static_cast<unsigned char *>(ws) + off);
  }
  return F;
}

int topk_fused_ctas(const FusedTopk &F, int n_q, int64_t n_max) {
  if (F.mode <= 0) return -1;
  return (int)collect_ctas(current_device(), n_q, n_max, F.reserve) * n_q;
}

size_t topk_fused_bytes(int n_q, int64_t n_max, int k) {
  const FusedTopk F = topk_fused_plan(nullptr, n_q, n_max, k);
  if (F.mode == -1) return 0;
  if (F.mode == 0) return topk_workspace_bytes(n_q, n_max, k);
  size_t b = (size_t)n_q * (size_t)F.W.sstride * 4;
  if (F.mode == 3) b = (b + 255) / 256 * 256 + (size_t)n_q * (size_t)F.W.gstride * 4;
  return b;
}

cudaError_t launch_topk_fused(const float *scores, int64_t stride, int n_q, const int32_t *n_valid, int64_t n_max,
                              int k, const FusedTopk &F, int32_t *out, void *ws, int *status, cudaStream_t st) {
  if (F.mode <= 0) return launch_topk(scores, stride, n_q, n_valid, n_max, k, 1, nullptr, out, ws, status, st);
  TopkSrc S;
  S.bmax = nullptr;
  S.bstride = 0;
  S.scores = scores;
  S.stride = stride;
  S.n_valid = n_valid;
  S.pool = nullptr;
  S.block = 1;
  S.n_max = n_max;
  S.n_items = n_max;
  S.kv_pf = F.kv;
  S.q_seq = F.q_seq;
  S.n_seq = F.n_seq;
  const size_t dsm_collect = collect_smem_bytes();
  const unsigned P = collect_ctas(current_device(), n_q, n_max, F.reserve);
  if (F.parts == 4 && F.W.gmax != nullptr)
    return launch_pdl(topk_collect_kernel<true>, dim3(P, n_q), dim3(kCollectThreads), dsm_collect, st, P, S, F.sgi,
                      F.parts, k, F.W, out, status);
  return launch_pdl(topk_collect_kernel<false>, dim3(P, n_q), dim3(kCollectThreads), dsm_collect, st, P, S, F.sgi,
                    F.parts, k, F.W, out, status);
}

}  // namespace csa2
