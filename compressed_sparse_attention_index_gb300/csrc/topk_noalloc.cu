// csa2_topk_noalloc: the top-k selection of csa2_topk for callers that cannot
// allocate device memory.  The only scratch the selection needs (one group
// maximum per group of scores, for rows longer than 16,384 items) lives in a
// fixed array compiled into the library instead of a caller-provided buffer.
#include <cuda_runtime.h>

#include "common.cuh"
#include "launch.cuh"

namespace csa2 {

// Fixed scratch of CSA2_TOPK_NOALLOC_SCRATCH_BYTES (4 MiB) on every device that
// loads the library, held until the process exits.
static __device__ __align__(256) uint32_t g_topk_scratch[CSA2_TOPK_NOALLOC_SCRATCH_BYTES / 4];

// Device address of the scratch array on the current device, looked up once
// per device with that device current (the host-side name of a __device__
// array is not a device address).  nullptr if the lookup failed.
static void *topk_scratch_ptr() {
  static std::atomic<void *> ptrs[kMaxDevices];
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  void *p = ptrs[dev].load(std::memory_order_relaxed);
  if (p == nullptr) {
    if (cudaGetSymbolAddress(&p, g_topk_scratch) != cudaSuccess) return nullptr;
    ptrs[dev].store(p, std::memory_order_relaxed);
  }
  return p;
}

}  // namespace csa2

using namespace csa2;

extern "C" csa2_status csa2_topk_noalloc(const float *scores, int64_t score_stride, int n_q, const int32_t *n_valid,
                                         int64_t n_max, int k, int block, const int32_t *pool_blocks, int32_t *out,
                                         csa2_stream_t stream) {
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
  // the whole scratch requirement must fit the fixed array
  if (topk_workspace_bytes(n_q, items, k) > (size_t)CSA2_TOPK_NOALLOC_SCRATCH_BYTES) return CSA2_ERR_WORKSPACE;
  void *ws = topk_scratch_ptr();
  int *st = status_word_ptr();
  if (ws == nullptr || st == nullptr) return CSA2_ERR_CUDA;
  // every slot of the scratch that the selection reads is written earlier in
  // the same call, so nothing has to be cleared between calls
  const cudaError_t e = launch_topk(scores, score_stride, n_q, n_valid, n_max, k, block, pool_blocks, out, ws, st,
                                    (cudaStream_t)stream);
  return e == cudaSuccess ? CSA2_OK : CSA2_ERR_CUDA;
}
