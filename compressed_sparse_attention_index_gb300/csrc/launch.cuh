// Host-side launchers shared by the C ABI (api.cu, topk_noalloc.cu) and the
// kernel files that define them.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace csa2 {

// Scratch of a long-row top-k, per row q: smax[q][sstride] (supergroup maxima,
// or partial maxima), ctr[q][4] (candidates appended, collecting CTAs done),
// cand[q][8192] (64-bit candidate keys).
struct LongRowWs {
  uint32_t *smax, *ctr;
  uint64_t *cand;
  int64_t sstride;
};

// Top-k plan of the fused decode: mode -1 one CTA per row (no scratch); 0 the
// standalone passes; 1 / 2 the indexer's epilogue writes the maxima (512-entry
// units as four partials / 32-entry groups) and only the collection runs.
struct FusedTopk {
  int mode;
  int64_t sgi;
  int parts;
  LongRowWs W;
};

cudaError_t launch_pack(int kind, const void *src, int64_t rows, int m, const float *gate, void *dst,
                        void *dst_scales, cudaStream_t st);

// smax / sstride / smax_mode: maxima for a fused top-k (smax_mode 0: none);
// clear / n_clear: words zeroed by the kernel before anything else.
cudaError_t launch_index_score_tc(const uint8_t *key_nib, const uint8_t *key_scale, int64_t n_max, int n_seq,
                                  const uint8_t *q_nib, const uint8_t *q_scale, const float *w, const int32_t *q_seq,
                                  const int32_t *n_vis, int n_q, const int32_t *pool, float *scores, int64_t stride,
                                  int *status, cudaStream_t st, uint32_t *smax = nullptr, int64_t sstride = 0,
                                  int smax_mode = 0, uint32_t *clear = nullptr, int n_clear = 0);

size_t topk_workspace_bytes(int n_q, int64_t n_items, int k);
bool topk_items_supported(int64_t n_items, int k);
cudaError_t launch_topk(const float *scores, int64_t stride, int n_q, const int32_t *n_valid, int64_t n_max, int k,
                        int block, const int32_t *pool, int32_t *out, void *ws, int *status, cudaStream_t st);
FusedTopk topk_fused_plan(void *ws, int n_q, int64_t n_max, int k);
size_t topk_fused_bytes(int n_q, int64_t n_max, int k);
cudaError_t launch_topk_fused(const float *scores, int64_t stride, int n_q, const int32_t *n_valid, int64_t n_max,
                              int k, const FusedTopk &F, int32_t *out, void *ws, int *status, cudaStream_t st);

size_t attn_workspace_bytes(int n_q, int sel_stride);
cudaError_t launch_attn_tc(const void *q, const void *kv, int64_t n_max, int n_seq, const int32_t *sel,
                           int sel_stride, const void *swa, int swa_cap, const int32_t *q_seq, const int32_t *pos,
                           const int32_t *swa_first, const int32_t *swa_cnt, int n_q, void *out, int out_dtype,
                           float sm_scale, double rope_base, void *ws, int *status, cudaStream_t st);

int *status_word_ptr();

}  // namespace csa2
