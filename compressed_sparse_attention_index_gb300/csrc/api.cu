// C ABI of the CSA2 library: argument checks, workspace sizing, launches.
// The declarations and the contract of every entry point are in include/csa2.h.
#include <cuda_runtime.h>
#include <math.h>
#include <string.h>

#include "common.cuh"
#include "launch.cuh"

namespace csa2 {

// The sticky status word of each device (a file-scope device variable: the
// library makes no allocation for it).
__device__ int g_status_word;

static int *status_ptr() {
  static std::atomic<int *> ptrs[kMaxDevices];
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  int *p = ptrs[dev].load(std::memory_order_relaxed);
  if (p == nullptr) {
    void *a = nullptr;
    if (cudaGetSymbolAddress(&a, g_status_word) != cudaSuccess) return nullptr;
    p = static_cast<int *>(a);
    ptrs[dev].store(p, std::memory_order_relaxed);
  }
  return p;
}

// The status word's device address for entry points defined in other files.
int *status_word_ptr() { return status_ptr(); }

static bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

static bool params_ok(const csa2_params *p) {
  if (p == nullptr) return true;   // null = the pages' constants
  return p->heads == kHeads && p->dim == kDim && p->rope_dim == kRopeDim && p->rope_off == kRopeOff &&
         p->idx_heads == kIdxHeads && p->idx_dim == kIdxDim && p->topk == kTopK && p->swa == kSwa &&
         p->block == kBlock && p->pool_blocks == kPoolBlocks && p->rope_base > 0.0 && p->sm_scale > 0.f &&
         isfinite(p->sm_scale) && isfinite(p->rope_base);
}

static csa2_status from_cuda(cudaError_t e) { return e == cudaSuccess ? CSA2_OK : CSA2_ERR_CUDA; }

static size_t round256(size_t b) { return (b + 255) / 256 * 256; }

// csa2_profile_events: events recorded around the indexer launch of the
// decode steps, per host thread (null: off)
static thread_local cudaEvent_t g_prof_begin = nullptr, g_prof_end = nullptr;
static cudaError_t prof_mark(cudaEvent_t e, cudaStream_t s) { return e != nullptr ? cudaEventRecord(e, s) : cudaSuccess; }

// csa2_decode's workspace, each part 256-B aligned:
// scores [n_q][n_max] fp32 | top-k scratch | attention partials
// csa2_decode's workspace: scores | top-k scratch | attention partials | the
// indexer's claim counter (256 B, where the maxima come from the indexer) |
// the candidate handoff (flags, then keys), where the selection hands its
// candidates to the attention (the maxima come from the indexer and all
// attention CTAs holding candidates fit one wave).
static bool decode_handoff(int n_q, int64_t n_max) {
  return topk_fused_plan(nullptr, n_q, n_max, kTopK).mode > 0 && attn_handoff_fits(n_q);
}
static size_t decode_workspace_bytes(int n_q, int64_t n_max) {
  const bool hand = decode_handoff(n_q, n_max);
  size_t b = round256((size_t)n_q * (size_t)n_max * 4) + round256(topk_fused_bytes(n_q, n_max, kTopK)) +
             round256(attn_workspace_bytes(n_q, hand ? kHandCap : kTopK, true));
  if (topk_fused_plan(nullptr, n_q, n_max, kTopK).mode > 0) b += 256;
  if (hand) b += round256((size_t)n_q * kHandWords * 4) + round256((size_t)n_q * kHandCtas * kHandSeg * 8);
  return b;
}

}  // namespace csa2

using namespace csa2;

extern "C" {

csa2_status csa2_default_params(csa2_params *p) {
  if (p == nullptr) return CSA2_ERR_INVALID_ARG;
  p->heads = kHeads;
  p->dim = kDim;
  p->rope_dim = kRopeDim;
  p->rope_off = kRopeOff;
  p->rope_base = 10000.0;
  p->sm_scale = 1.0f / sqrtf((float)kDim);
  p->idx_heads = kIdxHeads;
  p->idx_dim = kIdxDim;
  p->topk = kTopK;
  p->swa = kSwa;
  p->block = kBlock;
  p->pool_blocks = kPoolBlocks;
  return CSA2_OK;
}

size_t csa2_entry_bytes(int kind) {
  switch (kind) {
    case CSA2_KV_NVFP4: return kKvBytes;
    case CSA2_IDX_MXFP4: return kIdxNibBytes + kIdxScaleBytes;
    case CSA2_SWA_MXFP8: return kSwaBytes;
    default: return 0;
  }
}

const char *csa2_status_string(csa2_status s) {
  switch (s) {
    case CSA2_OK: return "ok";
    case CSA2_ERR_INVALID_ARG: return "invalid argument";
    case CSA2_ERR_UNSUPPORTED: return "unsupported parameters";
    case CSA2_ERR_CUDA: return "CUDA runtime error";
    case CSA2_ERR_BOUNDS: return "device-side index out of range";
    case CSA2_ERR_TIMEOUT: return "device-side bounded wait ran out";
    case CSA2_ERR_WORKSPACE: return "workspace too small";
    default: return "unknown status";
  }
}

csa2_status csa2_fp4_pack(int kind, const void *src, int64_t rows, int m, const float *gate_logits, void *dst,
                          void *dst_scales, csa2_stream_t stream) {
  if (kind != CSA2_KV_NVFP4 && kind != CSA2_IDX_MXFP4 && kind != CSA2_SWA_MXFP8) return CSA2_ERR_INVALID_ARG;
  if (rows < 0 || (m != 1 && m != 2)) return CSA2_ERR_INVALID_ARG;
  if (m == 2 && (kind != CSA2_KV_NVFP4 || gate_logits == nullptr || rows % 2 != 0)) return CSA2_ERR_INVALID_ARG;
  if (m == 1 && gate_logits != nullptr) return CSA2_ERR_INVALID_ARG;
  if ((kind == CSA2_IDX_MXFP4) != (dst_scales != nullptr)) return CSA2_ERR_INVALID_ARG;
  if (rows == 0) return CSA2_OK;
  if (src == nullptr || dst == nullptr) return CSA2_ERR_INVALID_ARG;
  if (!aligned(src, 16) || !aligned(dst, 16) || (gate_logits && !aligned(gate_logits, 16)))
    return CSA2_ERR_INVALID_ARG;
  return from_cuda(launch_pack(kind, src, rows, m, gate_logits, dst, dst_scales, (cudaStream_t)stream));
}

csa2_status csa2_index_score(const void *key_nib, const void *key_scale, int64_t n_max, int n_seq, const void *q_nib,
                             const void *q_scale, const float *w, const int32_t *q_seq, const int32_t *n_vis, int n_q,
                             const int32_t *pool_blocks, float *scores, int64_t score_stride,
                             const csa2_params *params, csa2_stream_t stream) {
  if (!params_ok(params)) return CSA2_ERR_UNSUPPORTED;
  if (n_q < 0 || n_seq < 1 || n_max <= 0 || n_max % 128 != 0 || n_max > ((int64_t)1 << 31) - 128)
    return CSA2_ERR_INVALID_ARG;
  if (n_q > 65535) return CSA2_ERR_UNSUPPORTED;
  if (score_stride < (pool_blocks ? (int64_t)kPoolSlots : n_max)) return CSA2_ERR_INVALID_ARG;
  if (n_q == 0) return CSA2_OK;
  if (!key_nib || !key_scale || !q_nib || !q_scale || !w || !q_seq || !n_vis || !scores)
    return CSA2_ERR_INVALID_ARG;
  if (!aligned(key_nib, 512) || !aligned(key_scale, 16) || !aligned(q_nib, 512) || !aligned(q_scale, 16) ||
      !aligned(w, 16) || !aligned(scores, 4))
    return CSA2_ERR_INVALID_ARG;
  int *st = status_ptr();
  if (st == nullptr) return CSA2_ERR_CUDA;
  return from_cuda(launch_index_score_tc(
      static_cast<const uint8_t *>(key_nib), static_cast<const uint8_t *>(key_scale), n_max, n_seq,
      static_cast<const uint8_t *>(q_nib), static_cast<const uint8_t *>(q_scale), w, q_seq, n_vis, n_q, pool_blocks,
      scores, score_stride, st, (cudaStream_t)stream));
}

// csa2_decode_host's device staging, after the decode workspace (from a
// 512-B boundary on), each part 512-B aligned (csa2_decode wants its packed
// indexer query so): q | indexer query bf16 | its packed nibbles | its scales |
// w | descriptors [5][n_q] | sel | out (fp32-sized)
static size_t round512(size_t b) { return (b + 511) / 512 * 512; }
struct HostStage {
  size_t q, qidx, qnib, qsc, w, desc, sel, out, total;
};
static HostStage host_stage(int n_q) {
  HostStage h;
  size_t o = 0;
  auto take = [&](size_t b) { const size_t at = o; o += round512(b); return at; };
  h.q = take((size_t)n_q * kHeads * kDim * 2);
  h.qidx = take((size_t)n_q * kIdxHeads * kIdxDim * 2);
  h.qnib = take((size_t)n_q * kIdxHeads * kIdxNibBytes);
  h.qsc = take((size_t)n_q * kIdxHeads * kIdxScaleBytes);
  h.w = take((size_t)n_q * kIdxHeads * 4);
  h.desc = take((size_t)n_q * 5 * 4);
  h.sel = take((size_t)n_q * kTopK * 4);
  h.out = take((size_t)n_q * kHeads * kDim * 4);
  h.total = o;
  return h;
}

// csa2_build_cache's workspace for one chunk of entries: the keys (bf16
// [chunk][128]) and, for m = 2, the pooled latents (bf16 [chunk][512]), two
// counts (256 B) and the pooling's fix-up list (uint32 [chunk * 4]: up to
// four of an entry's 32 channel blocks on average).
constexpr int64_t kBuildChunk = 131072;
constexpr int kBuildFixPerEntry = 4;
static size_t build_cache_workspace_bytes(int64_t n_tokens, int m) {
  const int64_t entries = n_tokens / m;
  const int64_t c = entries < kBuildChunk ? entries : kBuildChunk;
  return round256((size_t)c * kIdxDim * 2) +
         (m == 2 ? round256((size_t)c * kDim * 2) + 256 + round256((size_t)c * kBuildFixPerEntry * 4) : 0);
}

// csa2_decode_reindex's workspace: pool scores [n_q][16384] fp32 | block
// maxima [n_q][2048] | top-k scratch | attention partials
static size_t decode_reindex_workspace_bytes(int n_q) {
  return round256((size_t)n_q * kPoolSlots * 4) + round256((size_t)n_q * kPoolBlocks * 4) +
         round256(topk_workspace_bytes(n_q, kPoolSlots, kTopK)) + round256(attn_workspace_bytes(n_q, kTopK, true));
}

// csa2_decode_mq's workspace: scores [n_q][n_max] | top-k scratch | attention partials
static size_t decode_mq_workspace_bytes(int n_q, int64_t n_max) {
  return round256((size_t)n_q * (size_t)n_max * 4) + round256(topk_workspace_bytes(n_q, n_max, kTopK)) +
         round256(attn_workspace_bytes(n_q, kTopK));
}

csa2_status csa2_profile_events(void *begin, void *end) {
  if ((begin == nullptr) != (end == nullptr)) return CSA2_ERR_INVALID_ARG;
  g_prof_begin = static_cast<cudaEvent_t>(begin);
  g_prof_end = static_cast<cudaEvent_t>(end);
  return CSA2_OK;
}

csa2_status csa2_workspace_size(int op, int n_q, int64_t n_items, int k, size_t *bytes) {
  if (bytes == nullptr || n_q < 0 || n_items < 0) return CSA2_ERR_INVALID_ARG;
  if (op == CSA2_OP_BUILD_CACHE) {
    if (n_items < 0 || (k != 1 && k != 2)) return CSA2_ERR_INVALID_ARG;
    *bytes = build_cache_workspace_bytes(n_items, k);
    return CSA2_OK;
  }
  if (op == CSA2_OP_DECODE_MQ) {
    if (n_items <= 0) return CSA2_ERR_INVALID_ARG;
    *bytes = decode_mq_workspace_bytes(n_q, n_items);
    return CSA2_OK;
  }
  if (op == CSA2_OP_DECODE_REINDEX) {
    if (n_items <= 0) return CSA2_ERR_INVALID_ARG;
    *bytes = decode_reindex_workspace_bytes(n_q);
    return CSA2_OK;
  }
  if (op == CSA2_OP_DECODE_HOST) {
    if (n_items <= 0) return CSA2_ERR_INVALID_ARG;
    *bytes = round512(decode_workspace_bytes(n_q, n_items)) + host_stage(n_q).total;
    return CSA2_OK;
  }
  if (op == CSA2_OP_TOPK) {
    if (k < 1 || k > 2048) return CSA2_ERR_UNSUPPORTED;
    *bytes = topk_workspace_bytes(n_q, n_items, k);
    return CSA2_OK;
  }
  if (op == CSA2_OP_DECODE) {
    if (n_items <= 0) return CSA2_ERR_INVALID_ARG;
    *bytes = decode_workspace_bytes(n_q, n_items);
    return CSA2_OK;
  }
  if (op == CSA2_OP_SPARSE_ATTN) {
    const int64_t sel_stride = n_items - kSwa;
    if (sel_stride < 1 || sel_stride > kTopK) return CSA2_ERR_INVALID_ARG;
    *bytes = attn_workspace_bytes(n_q, (int)sel_stride);
    return CSA2_OK;
  }
  return CSA2_ERR_INVALID_ARG;
}

csa2_status csa2_topk(const float *scores, int64_t score_stride, int n_q, const int32_t *n_valid, int64_t n_max,
                      int k, int block, const int32_t *pool_blocks, int32_t *out, void *workspace,
                      size_t workspace_bytes, csa2_stream_t stream) {
  if (k < 1 || k > 2048) return CSA2_ERR_UNSUPPORTED;
  if (n_q < 0 || n_max <= 0 || n_max > ((int64_t)1 << 31) - 8 || (block != 1 && block != kBlock))
    return CSA2_ERR_INVALID_ARG;
  if (block != 1 && pool_blocks != nullptr) return CSA2_ERR_INVALID_ARG;
  if (n_q > 65535) return CSA2_ERR_UNSUPPORTED;
  const int64_t row_len = pool_blocks ? (int64_t)kPoolSlots : n_max;
  if (score_stride < row_len) return CSA2_ERR_INVALID_ARG;
  if (n_q == 0) return CSA2_OK;
  if (!scores || !n_valid || !out) return CSA2_ERR_INVALID_ARG;
  const int64_t items = pool_blocks ? (int64_t)kPoolSlots : (block == 1 ? n_max : (n_max + kBlock - 1) / kBlock);
  if (!topk_items_supported(items, k)) return CSA2_ERR_UNSUPPORTED;
  const size_t need = topk_workspace_bytes(n_q, items, k);
  if (workspace_bytes < need || (need > 0 && (workspace == nullptr || !aligned(workspace, 256))))
    return CSA2_ERR_WORKSPACE;
  int *st = status_ptr();
  if (st == nullptr) return CSA2_ERR_CUDA;
  return from_cuda(launch_topk(scores, score_stride, n_q, n_valid, n_max, k, block, pool_blocks, out, workspace, st,
                               (cudaStream_t)stream));
}

csa2_status csa2_sparse_attn(const void *q, const void *kv_cache, int64_t n_max, int n_seq, const int32_t *sel,
                             int sel_stride, const void *swa_cache, int swa_cap, const int32_t *q_seq,
                             const int32_t *pos, const int32_t *swa_first, const int32_t *swa_cnt, int n_q, void *out,
                             int out_dtype, const csa2_params *params, void *workspace, size_t workspace_bytes,
                             csa2_stream_t stream) {
  if (!params_ok(params)) return CSA2_ERR_UNSUPPORTED;
  if (n_q < 0 || n_seq < 1 || n_max <= 0 || swa_cap < 0 || sel_stride < 1 || sel_stride > kTopK)
    return CSA2_ERR_INVALID_ARG;
  if (out_dtype != CSA2_OUT_BF16 && out_dtype != CSA2_OUT_F32) return CSA2_ERR_INVALID_ARG;
  if (n_q > 65535) return CSA2_ERR_UNSUPPORTED;
  if (n_q == 0) return CSA2_OK;
  if (!q || !kv_cache || !sel || !q_seq || !pos || !swa_first || !swa_cnt || !out) return CSA2_ERR_INVALID_ARG;
  if (swa_cap > 0 && swa_cache == nullptr) return CSA2_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(kv_cache, 16) || (swa_cache && !aligned(swa_cache, 16)) || !aligned(out, 16))
    return CSA2_ERR_INVALID_ARG;
  const size_t need = attn_workspace_bytes(n_q, sel_stride);
  if (workspace_bytes < need || (need > 0 && (workspace == nullptr || !aligned(workspace, 256))))
    return CSA2_ERR_WORKSPACE;
  int *st = status_ptr();
  if (st == nullptr) return CSA2_ERR_CUDA;
  const float sm_scale = params ? params->sm_scale : 1.0f / sqrtf((float)kDim);
  const double rope_base = params ? params->rope_base : 10000.0;
  return from_cuda(launch_attn_tc(q, kv_cache, n_max, n_seq, sel, sel_stride, swa_cache, swa_cap, q_seq, pos,
                                    swa_first, swa_cnt, n_q, out, out_dtype, sm_scale, rope_base, workspace, st,
                                    (cudaStream_t)stream));
}

csa2_status csa2_decode(const void *key_nib, const void *key_scale, int64_t n_max, int n_seq, const void *q_nib,
                        const void *q_scale, const float *w, const int32_t *q_seq, const int32_t *n_vis, int n_q,
                        const void *q, const void *kv_cache, const void *swa_cache, int swa_cap, const int32_t *pos,
                        const int32_t *swa_first, const int32_t *swa_cnt, int32_t *sel, void *out, int out_dtype,
                        const csa2_params *params, void *workspace, size_t workspace_bytes, csa2_stream_t stream) {
  if (!params_ok(params)) return CSA2_ERR_UNSUPPORTED;
  if (n_q < 0 || n_seq < 1 || n_max <= 0 || n_max % 128 != 0 || n_max > ((int64_t)1 << 31) - 128 || swa_cap < 0)
    return CSA2_ERR_INVALID_ARG;
  if (out_dtype != CSA2_OUT_BF16 && out_dtype != CSA2_OUT_F32) return CSA2_ERR_INVALID_ARG;
  if (n_q > 65535) return CSA2_ERR_UNSUPPORTED;
  if (n_q == 0) return CSA2_OK;
  if (!key_nib || !key_scale || !q_nib || !q_scale || !w || !q_seq || !n_vis || !q || !kv_cache || !pos ||
      !swa_first || !swa_cnt || !sel || !out)
    return CSA2_ERR_INVALID_ARG;
  if (swa_cap > 0 && swa_cache == nullptr) return CSA2_ERR_INVALID_ARG;
  if (!aligned(key_nib, 512) || !aligned(key_scale, 16) || !aligned(q_nib, 512) || !aligned(q_scale, 16) ||
      !aligned(w, 16) || !aligned(q, 16) || !aligned(kv_cache, 16) || (swa_cache && !aligned(swa_cache, 16)) ||
      !aligned(out, 16) || !aligned(sel, 4))
    return CSA2_ERR_INVALID_ARG;
  if (!topk_items_supported(n_max, kTopK)) return CSA2_ERR_UNSUPPORTED;
  if (workspace_bytes < decode_workspace_bytes(n_q, n_max) || workspace == nullptr || !aligned(workspace, 256))
    return CSA2_ERR_WORKSPACE;
  int *st = status_ptr();
  if (st == nullptr) return CSA2_ERR_CUDA;
  const cudaStream_t s = (cudaStream_t)stream;
  unsigned char *base = static_cast<unsigned char *>(workspace);
  float *scores = reinterpret_cast<float *>(base);
  void *ws_topk = base + round256((size_t)n_q * (size_t)n_max * 4);
  void *ws_attn = static_cast<unsigned char *>(ws_topk) + round256(topk_fused_bytes(n_q, n_max, kTopK));
  FusedTopk F = topk_fused_plan(ws_topk, n_q, n_max, kTopK);
  F.kv = static_cast<const uint8_t *>(kv_cache);
  F.q_seq = q_seq;
  F.n_seq = n_seq;
  const bool fused = F.mode > 0;
  const bool hand = decode_handoff(n_q, n_max);
  F.reserve = attn_ctas(n_q, hand ? kHandCap : kTopK, true);
  unsigned char *after_attn = static_cast<unsigned char *>(ws_attn) +
                              round256(attn_workspace_bytes(n_q, hand ? kHandCap : kTopK, true));
  if (fused) {
    // the indexer's claim counter, tagged per call (the tag is never 0)
    static std::atomic<uint32_t> calls{0};
    uint32_t id = calls.fetch_add(1, std::memory_order_relaxed) + 1u;
    if (id == 0u) id = calls.fetch_add(1, std::memory_order_relaxed) + 1u;
    F.W.steal = reinterpret_cast<unsigned long long *>(after_attn);
    F.W.call_id = id;
    after_attn += 256;
  }
  Handoff H = {nullptr, nullptr, 0};
  if (hand) {
    unsigned char *hb = after_attn;
    H.flag = reinterpret_cast<uint32_t *>(hb);
    H.cand = reinterpret_cast<uint64_t *>(hb + round256((size_t)n_q * kHandWords * 4));
    H.parts = topk_fused_ctas(F, n_q, n_max) / n_q;   // the selection's cluster size
    F.W.hand = H;
  }
  if (prof_mark(g_prof_begin, s) != cudaSuccess) return CSA2_ERR_CUDA;
  cudaError_t e = launch_index_score_tc(static_cast<const uint8_t *>(key_nib), static_cast<const uint8_t *>(key_scale),
                                        n_max, n_seq, static_cast<const uint8_t *>(q_nib),
                                        static_cast<const uint8_t *>(q_scale), w, q_seq, n_vis, n_q, nullptr, scores,
                                        n_max, st, s, fused ? &F.W : nullptr, fused ? F.mode : 0);
  if (e != cudaSuccess || prof_mark(g_prof_end, s) != cudaSuccess) return CSA2_ERR_CUDA;
  e = launch_topk_fused(scores, n_max, n_q, n_vis, n_max, kTopK, F, sel, ws_topk, st, s);
  if (e != cudaSuccess) return CSA2_ERR_CUDA;
  const float sm_scale = params ? params->sm_scale : 1.0f / sqrtf((float)kDim);
  const double rope_base = params ? params->rope_base : 10000.0;
  // the attention inputs were final before the indexer started (it waits for
  // every earlier grid), so the attention may stage them during the top-k
  return from_cuda(launch_attn_tc(q, kv_cache, n_max, n_seq, sel, kTopK, swa_cache, swa_cap, q_seq, pos, swa_first,
                                  swa_cnt, n_q, out, out_dtype, sm_scale, rope_base, ws_attn, st, s, true,
                                  topk_fused_ctas(F, n_q, n_max), hand ? &H : nullptr));
}

csa2_status csa2_decode_reindex(const void *key_nib, const void *key_scale, int64_t n_max, int n_seq,
                                const void *q_nib, const void *q_scale, const float *w, const int32_t *q_seq,
                                const int32_t *n_vis, int n_q, const int32_t *pool_blocks, const void *q,
                                const void *kv_cache, const void *swa_cache, int swa_cap, const int32_t *pos,
                                const int32_t *swa_first, const int32_t *swa_cnt, int32_t *sel, void *out,
                                int out_dtype, const csa2_params *params, void *workspace, size_t workspace_bytes,
                                csa2_stream_t stream) {
  if (!params_ok(params)) return CSA2_ERR_UNSUPPORTED;
  if (n_q < 0 || n_seq < 1 || n_max <= 0 || n_max % 128 != 0 || n_max > ((int64_t)1 << 31) - 128 || swa_cap < 0)
    return CSA2_ERR_INVALID_ARG;
  if (out_dtype != CSA2_OUT_BF16 && out_dtype != CSA2_OUT_F32) return CSA2_ERR_INVALID_ARG;
  if (n_q > 65535) return CSA2_ERR_UNSUPPORTED;
  if (n_q == 0) return CSA2_OK;
  if (!key_nib || !key_scale || !q_nib || !q_scale || !w || !q_seq || !n_vis || !pool_blocks || !q || !kv_cache ||
      !pos || !swa_first || !swa_cnt || !sel || !out)
    return CSA2_ERR_INVALID_ARG;
  if (swa_cap > 0 && swa_cache == nullptr) return CSA2_ERR_INVALID_ARG;
  if (!aligned(key_nib, 512) || !aligned(key_scale, 16) || !aligned(q_nib, 512) || !aligned(q_scale, 16) ||
      !aligned(w, 16) || !aligned(pool_blocks, 4) || !aligned(q, 16) || !aligned(kv_cache, 16) ||
      (swa_cache && !aligned(swa_cache, 16)) || !aligned(out, 16) || !aligned(sel, 4))
    return CSA2_ERR_INVALID_ARG;
  if (workspace_bytes < decode_reindex_workspace_bytes(n_q) || workspace == nullptr || !aligned(workspace, 256))
    return CSA2_ERR_WORKSPACE;
  int *st = status_ptr();
  if (st == nullptr) return CSA2_ERR_CUDA;
  const cudaStream_t s = (cudaStream_t)stream;
  unsigned char *base = static_cast<unsigned char *>(workspace);
  float *scores = reinterpret_cast<float *>(base);
  uint32_t *bmax = reinterpret_cast<uint32_t *>(base + round256((size_t)n_q * kPoolSlots * 4));
  void *ws_topk = reinterpret_cast<unsigned char *>(bmax) + round256((size_t)n_q * kPoolBlocks * 4);
  void *ws_attn = static_cast<unsigned char *>(ws_topk) + round256(topk_workspace_bytes(n_q, kPoolSlots, kTopK));
  // the pool-mode indexer also writes every block's largest order key
  LongRowWs W;
  W.smax = nullptr;
  W.sstride = 0;
  W.gmax = bmax;
  W.gstride = kPoolBlocks;
  if (prof_mark(g_prof_begin, s) != cudaSuccess) return CSA2_ERR_CUDA;
  cudaError_t e = launch_index_score_tc(static_cast<const uint8_t *>(key_nib), static_cast<const uint8_t *>(key_scale),
                                        n_max, n_seq, static_cast<const uint8_t *>(q_nib),
                                        static_cast<const uint8_t *>(q_scale), w, q_seq, n_vis, n_q, pool_blocks, scores,
                                        kPoolSlots, st, s, &W, 1);
  if (e != cudaSuccess || prof_mark(g_prof_end, s) != cudaSuccess) return CSA2_ERR_CUDA;
  e = launch_topk(scores, kPoolSlots, n_q, n_vis, n_max, kTopK, 1, pool_blocks, sel, ws_topk, st, s, bmax,
                  kPoolBlocks);
  if (e != cudaSuccess) return CSA2_ERR_CUDA;
  const float sm_scale = params ? params->sm_scale : 1.0f / sqrtf((float)kDim);
  const double rope_base = params ? params->rope_base : 10000.0;
  // the attention inputs were final before the indexer started, so the
  // attention may stage them during the selection (one CTA per pool row)
  return from_cuda(launch_attn_tc(q, kv_cache, n_max, n_seq, sel, kTopK, swa_cache, swa_cap, q_seq, pos, swa_first,
                                  swa_cnt, n_q, out, out_dtype, sm_scale, rope_base, ws_attn, st, s, true, n_q,
                                  nullptr));
}

csa2_status csa2_index_score_mq(const void *key_nib, const void *key_scale, int64_t n_max, int n_seq,
                                const void *q_nib, const void *q_scale, const float *w, const int32_t *q_seq,
                                const int32_t *n_vis, int n_q, int q_group, float *scores, int64_t score_stride,
                                const csa2_params *params, csa2_stream_t stream) {
  if (!params_ok(params)) return CSA2_ERR_UNSUPPORTED;
  if (n_q < 0 || n_seq < 1 || n_max <= 0 || n_max % 128 != 0 || n_max > ((int64_t)1 << 31) - 256)
    return CSA2_ERR_INVALID_ARG;
  if (q_group < 1 || q_group > kMaxQueryGroup) return CSA2_ERR_UNSUPPORTED;
  if (n_q % q_group != 0) return CSA2_ERR_INVALID_ARG;
  if (n_q > 65535) return CSA2_ERR_UNSUPPORTED;
  if (score_stride < n_max) return CSA2_ERR_INVALID_ARG;
  if (n_q == 0) return CSA2_OK;
  if (!key_nib || !key_scale || !q_nib || !q_scale || !w || !q_seq || !n_vis || !scores) return CSA2_ERR_INVALID_ARG;
  if (!aligned(key_nib, 512) || !aligned(key_scale, 16) || !aligned(q_nib, 512) || !aligned(q_scale, 16) ||
      !aligned(w, 16) || !aligned(scores, 4))
    return CSA2_ERR_INVALID_ARG;
  int *st = status_ptr();
  if (st == nullptr) return CSA2_ERR_CUDA;
  return from_cuda(launch_index_score_mq(static_cast<const uint8_t *>(key_nib), static_cast<const uint8_t *>(key_scale),
                                         n_max, n_seq, static_cast<const uint8_t *>(q_nib),
                                         static_cast<const uint8_t *>(q_scale), w, q_seq, n_vis, n_q, q_group, scores,
                                         score_stride, st, (cudaStream_t)stream));
}

csa2_status csa2_decode_mq(const void *key_nib, const void *key_scale, int64_t n_max, int n_seq, const void *q_nib,
                           const void *q_scale, const float *w, const int32_t *q_seq, const int32_t *n_vis, int n_q,
                           int q_group, const void *q, const void *kv_cache, const void *swa_cache, int swa_cap,
                           const int32_t *pos, const int32_t *swa_first, const int32_t *swa_cnt, int32_t *sel,
                           void *out, int out_dtype, const csa2_params *params, void *workspace,
                           size_t workspace_bytes, csa2_stream_t stream) {
  if (!params_ok(params)) return CSA2_ERR_UNSUPPORTED;
  if (n_q < 0 || n_seq < 1 || n_max <= 0 || n_max % 128 != 0 || n_max > ((int64_t)1 << 31) - 256 || swa_cap < 0)
    return CSA2_ERR_INVALID_ARG;
  if (q_group < 1 || q_group > kMaxQueryGroup) return CSA2_ERR_UNSUPPORTED;
  if (n_q % q_group != 0 || (out_dtype != CSA2_OUT_BF16 && out_dtype != CSA2_OUT_F32)) return CSA2_ERR_INVALID_ARG;
  if (n_q > 65535) return CSA2_ERR_UNSUPPORTED;
  if (n_q == 0) return CSA2_OK;
  if (!key_nib || !key_scale || !q_nib || !q_scale || !w || !q_seq || !n_vis || !q || !kv_cache || !pos ||
      !swa_first || !swa_cnt || !sel || !out)
    return CSA2_ERR_INVALID_ARG;
  if (swa_cap > 0 && swa_cache == nullptr) return CSA2_ERR_INVALID_ARG;
  if (!aligned(key_nib, 512) || !aligned(key_scale, 16) || !aligned(q_nib, 512) || !aligned(q_scale, 16) ||
      !aligned(w, 16) || !aligned(q, 16) || !aligned(kv_cache, 16) || (swa_cache && !aligned(swa_cache, 16)) ||
      !aligned(out, 16) || !aligned(sel, 4))
    return CSA2_ERR_INVALID_ARG;
  if (!topk_items_supported(n_max, kTopK)) return CSA2_ERR_UNSUPPORTED;
  if (workspace_bytes < decode_mq_workspace_bytes(n_q, n_max) || workspace == nullptr || !aligned(workspace, 256))
    return CSA2_ERR_WORKSPACE;
  int *st = status_ptr();
  if (st == nullptr) return CSA2_ERR_CUDA;
  const cudaStream_t s = (cudaStream_t)stream;
  unsigned char *base = static_cast<unsigned char *>(workspace);
  float *scores = reinterpret_cast<float *>(base);
  void *ws_topk = base + round256((size_t)n_q * (size_t)n_max * 4);
  void *ws_attn = static_cast<unsigned char *>(ws_topk) + round256(topk_workspace_bytes(n_q, n_max, kTopK));
  cudaError_t e = launch_index_score_mq(static_cast<const uint8_t *>(key_nib), static_cast<const uint8_t *>(key_scale),
                                        n_max, n_seq, static_cast<const uint8_t *>(q_nib),
                                        static_cast<const uint8_t *>(q_scale), w, q_seq, n_vis, n_q, q_group, scores,
                                        n_max, st, s);
  if (e != cudaSuccess) return CSA2_ERR_CUDA;
  e = launch_topk(scores, n_max, n_q, n_vis, n_max, kTopK, 1, nullptr, sel, ws_topk, st, s);
  if (e != cudaSuccess) return CSA2_ERR_CUDA;
  const float sm_scale = params ? params->sm_scale : 1.0f / sqrtf((float)kDim);
  const double rope_base = params ? params->rope_base : 10000.0;
  return from_cuda(launch_attn_tc(q, kv_cache, n_max, n_seq, sel, kTopK, swa_cache, swa_cap, q_seq, pos, swa_first,
                                  swa_cnt, n_q, out, out_dtype, sm_scale, rope_base, ws_attn, st, s));
}

// The device address of page-locked host memory (under unified addressing
// the same as the host's, for memory from cudaHostAlloc / cudaMallocHost or
// registered with cudaHostRegister); false for pageable memory.
static bool device_accessible_host(const void *h, const void **d) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, h) != cudaSuccess) {
    (void)cudaGetLastError();                      // (an unknown pointer: not an error of the call)
    return false;
  }
  if (a.type != cudaMemoryTypeHost || a.devicePointer == nullptr) return false;
  *d = a.devicePointer;
  return true;
}

csa2_status csa2_decode_host(const void *key_nib, const void *key_scale, int64_t n_max, int n_seq, const void *kv_cache,
                             const void *swa_cache, int swa_cap, const void *h_q, const void *h_qidx, const float *h_w,
                             const int32_t *h_desc, int n_q, int32_t *h_sel, void *h_out, int out_dtype,
                             const csa2_params *params, void *workspace, size_t workspace_bytes, csa2_stream_t stream) {
  if (!params_ok(params)) return CSA2_ERR_UNSUPPORTED;
  if (n_q < 0 || n_seq < 1 || n_max <= 0 || n_max % 128 != 0 || n_max > ((int64_t)1 << 31) - 128 || swa_cap < 0)
    return CSA2_ERR_INVALID_ARG;
  if (out_dtype != CSA2_OUT_BF16 && out_dtype != CSA2_OUT_F32) return CSA2_ERR_INVALID_ARG;
  if (n_q > 65535) return CSA2_ERR_UNSUPPORTED;
  if (n_q == 0) return CSA2_OK;
  if (!h_q || !h_qidx || !h_w || !h_desc || !h_out) return CSA2_ERR_INVALID_ARG;
  const size_t dec = round512(decode_workspace_bytes(n_q, n_max));
  const HostStage H = host_stage(n_q);
  if (workspace == nullptr || !aligned(workspace, 256) || workspace_bytes < dec + H.total) return CSA2_ERR_WORKSPACE;
  const cudaStream_t s = (cudaStream_t)stream;
  unsigned char *st = static_cast<unsigned char *>(workspace) + dec;
  const size_t b_q = (size_t)n_q * kHeads * kDim * 2, b_qidx = (size_t)n_q * kIdxHeads * kIdxDim * 2;
  const size_t b_w = (size_t)n_q * kIdxHeads * 4, b_desc = (size_t)n_q * 5 * 4;
  const size_t b_out = (size_t)n_q * kHeads * kDim * (out_dtype == CSA2_OUT_F32 ? 4 : 2);
  const size_t b_sel = (size_t)n_q * kTopK * 4;
  // the step's inputs: from page-locked host memory, read by one grid that
  // also packs the indexer query (no copy engine round trip per buffer);
  // from pageable memory, one copy per host buffer and the packing kernel
  const void *dq = nullptr, *dqidx = nullptr, *dw = nullptr, *ddesc = nullptr;
  if (device_accessible_host(h_q, &dq) && device_accessible_host(h_qidx, &dqidx) &&
      device_accessible_host(h_w, &dw) && device_accessible_host(h_desc, &ddesc) && aligned(dqidx, 16) &&
      aligned(dq, 4) && aligned(dw, 4) && aligned(ddesc, 4)) {
    StageIn S;
    S.qidx = static_cast<const uint16_t *>(dqidx);
    S.qidx_rows = (int64_t)n_q * kIdxHeads;
    S.qnib = st + H.qnib;
    S.qsc = st + H.qsc;
    const void *src[3] = {dq, dw, ddesc};
    void *dst[3] = {st + H.q, st + H.w, st + H.desc};
    const size_t bytes[3] = {b_q, b_w, b_desc};
    for (int k = 0; k < 3; k++) {
      S.src[k] = src[k];
      S.dst[k] = dst[k];
      S.wide[k] = aligned(src[k], 16) && bytes[k] % 16 == 0 ? 1 : 0;
      S.units[k] = (int64_t)(bytes[k] / (S.wide[k] ? 16 : 4));
    }
    if (launch_stage_host_inputs(S, s) != cudaSuccess) return CSA2_ERR_CUDA;
  } else {
    if (cudaMemcpyAsync(st + H.q, h_q, b_q, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaMemcpyAsync(st + H.qidx, h_qidx, b_qidx, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaMemcpyAsync(st + H.w, h_w, b_w, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaMemcpyAsync(st + H.desc, h_desc, b_desc, cudaMemcpyHostToDevice, s) != cudaSuccess)
      return CSA2_ERR_CUDA;
    const csa2_status r = csa2_fp4_pack(CSA2_IDX_MXFP4, st + H.qidx, (int64_t)n_q * kIdxHeads, 1, nullptr,
                                        st + H.qnib, st + H.qsc, stream);
    if (r != CSA2_OK) return r;
  }
  const int32_t *d = reinterpret_cast<const int32_t *>(st + H.desc);
  // a page-locked output buffer takes the output straight from the grid that
  // finishes it; otherwise the output goes through the staging and a copy
  const void *dout = nullptr;
  const bool out_direct = device_accessible_host(h_out, &dout) && aligned(dout, 16);
  const csa2_status r =
      csa2_decode(key_nib, key_scale, n_max, n_seq, st + H.qnib, st + H.qsc, reinterpret_cast<const float *>(st + H.w),
                  d, d + n_q, n_q, st + H.q, kv_cache, swa_cache, swa_cap, d + 2 * n_q, d + 3 * n_q, d + 4 * n_q,
                  reinterpret_cast<int32_t *>(st + H.sel), out_direct ? const_cast<void *>(dout) : st + H.out,
                  out_dtype, params, workspace, dec, stream);
  if (r != CSA2_OK) return r;
  // the step's other outputs: one copy per host buffer
  if (!out_direct && cudaMemcpyAsync(h_out, st + H.out, b_out, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return CSA2_ERR_CUDA;
  if (h_sel != nullptr && cudaMemcpyAsync(h_sel, st + H.sel, b_sel, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return CSA2_ERR_CUDA;
  return CSA2_OK;
}

csa2_status csa2_index_key_proj(const void *latent, int64_t rows, const void *w_idx, void *keys,
                                csa2_stream_t stream) {
  if (rows < 0 || rows > ((int64_t)1 << 40)) return CSA2_ERR_INVALID_ARG;
  if (rows == 0) return CSA2_OK;
  if (!latent || !w_idx || !keys) return CSA2_ERR_INVALID_ARG;
  if (!aligned(latent, 16) || !aligned(w_idx, 16) || !aligned(keys, 16)) return CSA2_ERR_INVALID_ARG;
  int *st = status_ptr();
  if (st == nullptr) return CSA2_ERR_CUDA;
  return from_cuda(launch_proj_keys(latent, rows, w_idx, keys, st, (cudaStream_t)stream));
}

csa2_status csa2_build_cache(const void *tokens, int64_t n_tokens, int m, const float *gate_logits,
                             const void *w_idx, void *kv, void *idx_nib, void *idx_scale, void *workspace,
                             size_t workspace_bytes, csa2_stream_t stream) {
  if (n_tokens < 0 || (m != 1 && m != 2) || n_tokens % (8 * m) != 0 || n_tokens > ((int64_t)1 << 40))
    return CSA2_ERR_INVALID_ARG;
  if ((m == 2) != (gate_logits != nullptr)) return CSA2_ERR_INVALID_ARG;
  if (n_tokens == 0) return CSA2_OK;
  if (!tokens || !w_idx || !kv || !idx_nib || !idx_scale) return CSA2_ERR_INVALID_ARG;
  if (!aligned(tokens, 16) || !aligned(w_idx, 16) || !aligned(kv, 16) || !aligned(idx_nib, 512) ||
      !aligned(idx_scale, 4) || (gate_logits && !aligned(gate_logits, 16)))
    return CSA2_ERR_INVALID_ARG;
  if (workspace == nullptr || !aligned(workspace, 256) || workspace_bytes < build_cache_workspace_bytes(n_tokens, m))
    return CSA2_ERR_WORKSPACE;
  int *st = status_ptr();
  if (st == nullptr) return CSA2_ERR_CUDA;
  const cudaStream_t s = (cudaStream_t)stream;
  const int64_t entries = n_tokens / m;
  uint16_t *keys = static_cast<uint16_t *>(workspace);
  const int64_t c = entries < kBuildChunk ? entries : kBuildChunk;   // (the workspace's chunk)
  uint16_t *pooled = m == 2 ? reinterpret_cast<uint16_t *>(static_cast<unsigned char *>(workspace) +
                                                           round256((size_t)c * kIdxDim * 2))
                            : nullptr;
  // m = 2: the pooling's fix-up list and its two counts (one per parity of the
  // chunk; each chunk's fix-up grid zeroes the next chunk's)
  uint32_t *fix_cnt = m == 2 ? reinterpret_cast<uint32_t *>(pooled + (size_t)round256((size_t)c * kDim * 2) / 2)
                             : nullptr;
  uint32_t *fix_list = m == 2 ? fix_cnt + 64 : nullptr;
  if (m == 2 && cudaMemsetAsync(fix_cnt, 0, 2 * sizeof(uint32_t), s) != cudaSuccess) return CSA2_ERR_CUDA;
  const uint16_t *tok = static_cast<const uint16_t *>(tokens);
  for (int64_t e0 = 0, k = 0; e0 < entries; e0 += kBuildChunk, k++) {
    const int64_t ne = entries - e0 < kBuildChunk ? entries - e0 : kBuildChunk;
    // the chunk's latents (m = 2: pooled into the workspace) and main-cache records
    const KvFix fix = {fix_cnt + (k & 1), fix_list, (uint32_t)(c * kBuildFixPerEntry), fix_cnt + ((k + 1) & 1)};
    cudaError_t e = launch_pack(CSA2_KV_NVFP4, tok + e0 * m * kDim, ne * m, m,
                                m == 2 ? gate_logits + e0 * 2 * kDim : nullptr,
                                static_cast<uint8_t *>(kv) + e0 * kKvBytes, nullptr, s, pooled, m == 2 ? &fix : nullptr);
    if (e != cudaSuccess) return CSA2_ERR_CUDA;
    // their keys, then the keys' records (e0 is a multiple of 8: the key plane's swizzle holds per chunk)
    e = launch_proj_keys(m == 2 ? static_cast<const void *>(pooled) : static_cast<const void *>(tok + e0 * kDim), ne,
                         w_idx, keys, st, s);
    if (e != cudaSuccess) return CSA2_ERR_CUDA;
    e = launch_pack(CSA2_IDX_MXFP4, keys, ne, 1, nullptr, static_cast<uint8_t *>(idx_nib) + e0 * (kIdxDim / 2),
                    static_cast<uint8_t *>(idx_scale) + e0 * 4, s);
    if (e != cudaSuccess) return CSA2_ERR_CUDA;
  }
  return CSA2_OK;
}

csa2_status csa2_check_bounded_wait(unsigned limit_us, csa2_stream_t stream) {
  if (limit_us < 1 || limit_us > 2000000) return CSA2_ERR_INVALID_ARG;
  int *st = status_ptr();
  if (st == nullptr) return CSA2_ERR_CUDA;
  return from_cuda(launch_bounded_wait_check(st, 1000ull * limit_us, (cudaStream_t)stream));
}

csa2_status csa2_get_device_status(csa2_stream_t stream, csa2_status *out) {
  if (out == nullptr) return CSA2_ERR_INVALID_ARG;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return CSA2_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_status_word, sizeof(int)) != cudaSuccess) return CSA2_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof(int)) != cudaSuccess) return CSA2_ERR_CUDA;
  *out = (csa2_status)v;
  return CSA2_OK;
}

}  // extern "C"
