// Host-side launchers shared by the C ABI (api.cu, topk_noalloc.cu) and the
// kernel files that define them.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

namespace csa2 {

// Host-side caches, one entry per device ordinal below kMaxDevices.  Host
// threads may make their first calls at the same time, so every entry is an
// atomic read and written with relaxed ordering: racing fillers store the same
// value, and a reader sees either nothing yet (and fills it itself) or that value.
constexpr int kMaxDevices = 64;

// Runs init() (which returns a cudaError_t) on the first call for device dev
// and remembers success; two threads racing on the first call may both run it,
// which must be harmless (kernel attributes set twice to the same value).
template <class F>
cudaError_t once_per_device(std::atomic<int> (&done)[kMaxDevices], int dev, F init) {
  if (dev < 0 || dev >= kMaxDevices) return init();
  if (done[dev].load(std::memory_order_relaxed)) return cudaSuccess;
  const cudaError_t e = init();
  if (e == cudaSuccess) done[dev].store(1, std::memory_order_relaxed);
  return e;
}

// Number of SMs of device dev (cached), or `fallback` if it cannot be read.
inline int device_sm_count(int dev, int fallback = 148) {
  static std::atomic<int> counts[kMaxDevices];
  if (dev < 0 || dev >= kMaxDevices) return fallback;
  int c = counts[dev].load(std::memory_order_relaxed);
  if (c == 0) {
    if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || c <= 0) {
      cudaGetLastError();
      return fallback;
    }
    counts[dev].store(c, std::memory_order_relaxed);
  }
  return c;
}

inline int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  return dev;
}

// Candidate handoff inside csa2_decode.  Every CTA of a query's selection
// cluster publishes its candidates (its entries reaching the threshold, in
// ascending index order; together a superset of the selected entries) as soon
// as it has them; CTA 0 publishes the smallest selected key the moment its
// exact selection finds it.  The attention gathers and scores the candidates
// meanwhile and masks those below that key.  Per query, flag holds kHandWords
// words: [0] selection CTAs that have published (release); [1] nonzero once
// the selection (sel) is final (release); [2..3] the smallest selected key
// (never 0; it is the only datum read after it, so a plain store);
// [8 + p] CTA p's candidate count, or kHandFallback where its list cannot be
// handed over (the attention then reads the final selection).  Words 0-3 are
// zeroed by the indexer of the same call.  cand holds
// [n_q][kHandCtas][kHandSeg] keys, CTA p's in segment p.
constexpr int kHandCap = 640;       // candidates the attention takes (5 chunks of 128)
constexpr int kHandCtas = 16;       // selection CTAs per query, at most
constexpr int kHandSeg = 256;       // candidates per CTA, at most
constexpr int kHandWords = 32;
constexpr uint32_t kHandFallback = 0xFFFFFFFFu;
struct Handoff {
  uint32_t *flag;
  uint64_t *cand;
  int parts;                        // selection CTAs per query
};

// Scratch of a long-row top-k: smax[q][sstride], the supergroup maxima (or
// partial maxima) of row q.
struct LongRowWs {
  uint32_t *smax;
  int64_t sstride;
  // optional (plain rows): the maxima of every 32 consecutive entries,
  // gmax[q][gstride] (entry j in group j / 32), or null; (pool rows, the
  // indexer's smax_mode 1) the maxima of the pool's 8-entry blocks
  uint32_t *gmax = nullptr;
  int64_t gstride = 0;
  // optional (csa2_decode): the candidate handoff to the attention, or null
  Handoff hand = {nullptr, nullptr, 0};
  // optional (csa2_decode): the indexer's claim counter for its last rounds of
  // units, and this call's tag (never 0; see index_score_tc_kernel)
  unsigned long long *steal = nullptr;
  uint32_t call_id = 0;
};

// Launch `kern` with programmatic stream serialisation (the kernel calls
// griddep_wait before it reads what an earlier grid wrote) and, when
// cluster_x > 1, thread-block clusters of cluster_x CTAs along x.
template <class... Params, class... Args>
cudaError_t launch_pdl(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       unsigned cluster_x, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[2];
  unsigned na = 0;
  at[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[na].val.programmaticStreamSerializationAllowed = 1;
  na++;
  if (cluster_x > 1) {
    at[na].id = cudaLaunchAttributeClusterDimension;
    at[na].val.clusterDim.x = cluster_x;
    at[na].val.clusterDim.y = 1;
    at[na].val.clusterDim.z = 1;
    na++;
  }
  cfg.attrs = at;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Top-k plan of the fused decode: mode -1 one CTA per row (no scratch); 0 the
// standalone passes; 2 / 3 the indexer's epilogue writes the maxima (32-entry
// groups / 512-entry units as four partials and their 32-entry groups) and
// only the collection runs.
struct FusedTopk {
  int mode;
  int64_t sgi;
  int parts;
  LongRowWs W;
  // optional: the latent cache [n_seq][n_max][288] and the queries' sequences,
  // for an L2 prefetch of the selected records (modes 2 and 3)
  const uint8_t *kv;
  const int32_t *q_seq;
  int n_seq;
  // SMs to leave to the grid that follows (the attention, whose CTAs are
  // placed while the collection runs), when that still leaves the collection
  // at least four CTAs per row
  int reserve;
};

// The KV pack's fix-up list (m = 2): the (row, lane block) pairs, row * 32 +
// block, whose fp64 recomputation a second grid does; cnt zero on entry;
// next_cnt (optional) zeroed by that grid, for the next launch.
struct KvFix {
  uint32_t *cnt;
  uint32_t *list;
  uint32_t cap;
  uint32_t *next_cnt;
};
// pooled (KV, m = 2, optional): also write the pooled bf16 latents, [rows / 2][512];
// fix (KV, m = 2, optional): defer the fp64 recomputations to a fix-up grid
cudaError_t launch_pack(int kind, const void *src, int64_t rows, int m, const float *gate, void *dst,
                        void *dst_scales, cudaStream_t st, void *pooled = nullptr, const KvFix *fix = nullptr);

// csa2_decode_host's inputs from page-locked host memory (device-accessible
// addresses): the indexer query rows (bf16 [qidx_rows][128]) packed into qnib
// / qsc, and up to three segments copied (units[k] units of 16 B when wide[k],
// else of 4 B; src and dst aligned to the unit).  One grid; pack_ctas is set
// by the launch.
struct StageIn {
  const uint16_t *qidx;
  int64_t qidx_rows;
  uint8_t *qnib, *qsc;
  const void *src[3];
  void *dst[3];
  int64_t units[3];
  int wide[3];
  int pack_ctas;
};
cudaError_t launch_stage_host_inputs(StageIn S, cudaStream_t st);

// The indexer keys of rows bf16 latents under the 512 -> 128 bf16 weights
// w ([128][512]): out [rows][128] bf16 (tcgen05, fp32 accumulation).
cudaError_t launch_proj_keys(const void *x, int64_t rows, const void *w, void *out, int *status, cudaStream_t st);

// W / smax_mode: maxima for a fused top-k (smax_mode 0: none).
cudaError_t launch_index_score_tc(const uint8_t *key_nib, const uint8_t *key_scale, int64_t n_max, int n_seq,
                                  const uint8_t *q_nib, const uint8_t *q_scale, const float *w, const int32_t *q_seq,
                                  const int32_t *n_vis, int n_q, const int32_t *pool, float *scores, int64_t stride,
                                  int *status, cudaStream_t st, const LongRowWs *W = nullptr, int smax_mode = 0);

// Multi-query indexer: queries [g * group, g * group + group) share their
// sequence and are scored in one pass over its keys (group 1 .. 6).
constexpr int kMaxQueryGroup = 6;
cudaError_t launch_index_score_mq(const uint8_t *key_nib, const uint8_t *key_scale, int64_t n_max, int n_seq,
                                  const uint8_t *q_nib, const uint8_t *q_scale, const float *w, const int32_t *q_seq,
                                  const int32_t *n_vis, int n_q, int group, float *scores, int64_t stride,
                                  int *status, cudaStream_t st);

size_t topk_workspace_bytes(int n_q, int64_t n_items, int k);
bool topk_items_supported(int64_t n_items, int k);
// bmax (pool rows, optional): the pool-mode indexer's block maxima,
// [n_q][bstride] order keys (see csa2_decode_reindex)
cudaError_t launch_topk(const float *scores, int64_t stride, int n_q, const int32_t *n_valid, int64_t n_max, int k,
                        int block, const int32_t *pool, int32_t *out, void *ws, int *status, cudaStream_t st,
                        const uint32_t *bmax = nullptr, int64_t bstride = 0);
FusedTopk topk_fused_plan(void *ws, int n_q, int64_t n_max, int k);
size_t topk_fused_bytes(int n_q, int64_t n_max, int k);
cudaError_t launch_topk_fused(const float *scores, int64_t stride, int n_q, const int32_t *n_valid, int64_t n_max,
                              int k, const FusedTopk &F, int32_t *out, void *ws, int *status, cudaStream_t st);
// CTAs (one per SM) that the fused plan's collection grid holds while it runs,
// or -1 where that is not known (modes -1 and 0).
int topk_fused_ctas(const FusedTopk &F, int n_q, int64_t n_max);

// settled: the plan of a launch with inputs_settled (below)
size_t attn_workspace_bytes(int n_q, int sel_stride, bool settled = false);
// CTAs of the attention grid (one per SM) for n_q queries
int attn_ctas(int n_q, int sel_stride, bool settled = false);
// inputs_settled: q, the window cache and the per-query arrays were final
// before the grid ahead of this one on the stream started (so inside
// csa2_decode): the kernel then stages Q and runs its window-only chunks before
// it waits for the selection.  ahead_ctas: the SMs the grid ahead holds while
// it runs (one CTA each), or -1; when this grid fits beside it and a CTA has
// one chunk, CTAs that wait for the selection run a warm-up pass meanwhile.
// hand: the selection grid ahead hands its candidates over (csa2_decode, where
// attn_handoff_fits(n_q)); the attention then runs kHandCap / 128 chunks of
// candidates instead of sel_stride / 128 of selected entries, and reads sel only
// where the selection fell back.
cudaError_t launch_attn_tc(const void *q, const void *kv, int64_t n_max, int n_seq, const int32_t *sel,
                           int sel_stride, const void *swa, int swa_cap, const int32_t *q_seq, const int32_t *pos,
                           const int32_t *swa_first, const int32_t *swa_cnt, int n_q, void *out, int out_dtype,
                           float sm_scale, double rope_base, void *ws, int *status, cudaStream_t st,
                           bool inputs_settled = false, int ahead_ctas = -1, const Handoff *hand = nullptr);
// The handoff pays where every CTA holding candidates fits one wave beside the
// selection: one chunk per CTA for n_q queries.
bool attn_handoff_fits(int n_q);

cudaError_t launch_bounded_wait_check(int *status, unsigned long long limit_ns, cudaStream_t st);

int *status_word_ptr();

}  // namespace csa2
