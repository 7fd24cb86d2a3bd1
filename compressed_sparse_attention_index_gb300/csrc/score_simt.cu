// Lightning-indexer scores on CUDA cores (csa2_index_score, small-batch path).
//
// "32 FP4 query heads of 128 dims against one shared key per entry, ReLU'd
// scores summed with per-head weights" ("An infra-oriented diagram of the
// DeepSeek-V4.1-Flash architecture", reading notes, lightning-indexer note):
//     s_j = sum_h w_h * max(0, sum_b 2^(eq_hb + ek_jb) * sum_{c in block b} q_hc k_jc)
// where q, k are E2M1 codes and eq, ek the E8M0 exponents of the 32-channel
// blocks.  Codes are doubled into int8 (all E2M1 values are halves), each
// 32-channel block dot is an exact int32 from dp4a, and the block results are
// scaled by 2^(eq + ek - 2) and summed in fp32.
//
// One thread per cache entry, 256 entries per CTA; the query's codes sit in
// shared memory and are read as warp-wide broadcasts.
#include "common.cuh"

namespace csa2 {

// Four E2M1 nibbles (the low 16 bits of w) -> four int8 holding 2 x value.
__device__ __forceinline__ uint32_t nib4_to_i8x4(uint32_t w) {
  const uint32_t mag = __byte_perm(0x03020100u, 0x0C080604u, w & 0x7777u);
  const uint32_t s = (w >> 3) & 0x1111u;
  const uint32_t sb = (s & 1u) | ((s & 0x10u) << 4) | ((s & 0x100u) << 8) | ((s & 0x1000u) << 12);
  const uint32_t mask = sb * 0xFFu;
  return (mag & ~mask) | (__vsub4(0u, mag) & mask);
}

__global__ void __launch_bounds__(256) index_score_simt_kernel(
    const uint8_t *__restrict__ key_nib, const uint8_t *__restrict__ key_scale, int64_t n_max, int n_seq,
    const uint8_t *__restrict__ q_nib, const uint8_t *__restrict__ q_scale, const float *__restrict__ w,
    const int32_t *__restrict__ q_seq, const int32_t *__restrict__ n_vis, const int32_t *__restrict__ pool,
    float *__restrict__ scores, int64_t stride, int *status) {
  __shared__ uint32_t qs[kIdxHeads][32];   // int8 codes x2, 4 per word
  __shared__ int qe[kIdxHeads][4];         // E8M0 exponents
  __shared__ float ws[kIdxHeads];
  const int qi = blockIdx.y;
  const int t = threadIdx.x;
  const int seq = __ldg(q_seq + qi);
  int nv = __ldg(n_vis + qi);
  if (seq < 0 || seq >= n_seq || nv < 0 || (int64_t)nv > n_max) {
    if (t == 0 && blockIdx.x == 0) record_error(status, CSA2_ERR_BOUNDS);
    return;
  }
  const int64_t item = (int64_t)blockIdx.x * blockDim.x + t;
  if (pool == nullptr && (int64_t)blockIdx.x * blockDim.x >= nv) return;   // whole tile beyond n_vis

  // stage the query: 32 heads x 64 nibble bytes -> int8 words; exponents; weights
  for (int i = t; i < kIdxHeads * 16; i += blockDim.x) {      // 16 words of nibbles per head
    const int h = i >> 4, wd = i & 15;
    const uint32_t v = __ldg(reinterpret_cast<const uint32_t *>(q_nib + ((int64_t)qi * kIdxHeads + h) * 64) + wd);
    qs[h][2 * wd] = nib4_to_i8x4(v);
    qs[h][2 * wd + 1] = nib4_to_i8x4(v >> 16);
  }
  if (t < kIdxHeads * 4) qe[t >> 2][t & 3] = (int)__ldg(q_scale + ((int64_t)qi * kIdxHeads) * 4 + t) - 127;
  if (t < kIdxHeads) ws[t] = __ldg(w + (int64_t)qi * kIdxHeads + t);
  __syncthreads();

  int64_t j;
  if (pool != nullptr) {
    if (item >= kPoolSlots) return;
    const int blk = __ldg(pool + (int64_t)qi * kPoolBlocks + (item >> 3));
    j = (int64_t)blk * kBlock + (item & 7);
    if (blk < 0 || j >= nv) {
      if (blk >= 0 && (int64_t)blk * kBlock >= n_max) record_error(status, CSA2_ERR_BOUNDS);
      scores[(int64_t)qi * stride + item] = -INFINITY;
      return;
    }
  } else {
    j = item;
    if (j >= nv) return;
  }
  const int64_t row = (int64_t)seq * n_max + j;
  const uint4 *kp = reinterpret_cast<const uint4 *>(key_nib + row * 64);
  uint32_t kw[32];
#pragma unroll
  for (int v = 0; v < 4; v++) {
    const uint4 a = __ldg(kp + v);
    const uint32_t x[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int u = 0; u < 4; u++) {
      kw[8 * v + 2 * u] = nib4_to_i8x4(x[u]);
      kw[8 * v + 2 * u + 1] = nib4_to_i8x4(x[u] >> 16);
    }
  }
  const uint32_t ksw = __ldg(reinterpret_cast<const uint32_t *>(key_scale) + row);
  int ke[4];
#pragma unroll
  for (int b = 0; b < 4; b++) ke[b] = (int)((ksw >> (8 * b)) & 0xFFu) - 127;

  float s = 0.f;
#pragma unroll 4
  for (int h = 0; h < kIdxHeads; h++) {
    float d = 0.f;
#pragma unroll
    for (int b = 0; b < 4; b++) {
      int acc = 0;
#pragma unroll
      for (int u = 0; u < 8; u++) acc = __dp4a((int)kw[8 * b + u], (int)qs[h][8 * b + u], acc);
      d += ldexpf((float)acc, qe[h][b] + ke[b] - 2);
    }
    s = fmaf(ws[h], fmaxf(d, 0.f), s);
  }
  scores[(int64_t)qi * stride + item] = s;
}

cudaError_t launch_index_score_simt(const uint8_t *key_nib, const uint8_t *key_scale, int64_t n_max, int n_seq,
                                    const uint8_t *q_nib, const uint8_t *q_scale, const float *w,
                                    const int32_t *q_seq, const int32_t *n_vis, int n_q, const int32_t *pool,
                                    float *scores, int64_t stride, int *status, cudaStream_t st) {
  const int64_t items = pool ? kPoolSlots : n_max;
  dim3 grid((unsigned)((items + 255) / 256), (unsigned)n_q);
  index_score_simt_kernel<<<grid, 256, 0, st>>>(key_nib, key_scale, n_max, n_seq, q_nib, q_scale, w, q_seq, n_vis,
                                                pool, scores, stride, status);
  return cudaGetLastError();
}

}  // namespace csa2
