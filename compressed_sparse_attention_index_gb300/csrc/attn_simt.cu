// Sparse MQA attention on CUDA cores (csa2_sparse_attn), split over the entry
// list with a log-sum-exp merge.
//
// "There is one KV latent per token and it is shared by all 64 query heads
// (k = v, 512-wide)"; "Every other layer attends over that window plus 512
// selected entries"; "RoPE touches 64 of the 512 dims, and is un-rotated on the
// attention output" ("An infra-oriented diagram of the DeepSeek-V4.1-Flash
// architecture", reading notes).
//
// Entry slots of a query: slot e < sel_stride is cache entry sel[q][e] (-1 =
// empty), slot sel_stride + t is the window's ring slot (swa_first + t) % swa_cap
// for t < swa_cnt.  Slots are processed in chunks of 32: the chunk is gathered
// and dequantised to bf16 in shared memory (exact: an E2M1 x E4M3 product has at
// most 6 significant bits; E4M3 x 2^e fits bf16's exponent range), scored
// against the 64 heads, and folded into an online softmax.  A CTA handles a
// range of chunks of one query; with one range per query it finishes the output
// itself, otherwise it leaves (O, m, l) partials that the merge kernel combines.
#include <cuda_bf16.h>

#include "common.cuh"

namespace csa2 {

constexpr int kAChunk = 32;           // entries per chunk
constexpr int kAThreads = 256;
constexpr int kQStride = kDim + 8;    // bf16 row stride in smem (pad against bank conflicts)
constexpr float kLog2e = 1.4426950408889634f;

struct AttnArgs {
  const uint16_t *q;
  const uint8_t *kv;
  int64_t n_max;
  int n_seq;
  const int32_t *sel;
  int sel_stride;
  const uint8_t *swa;
  int swa_cap;
  const int32_t *q_seq, *pos, *swa_first, *swa_cnt;
  void *out;
  int out_f32;
  float scale_log2;      // sm_scale * log2(e)
  double rope_base;
  int nsplit, chunks_per_split;
  float *part;           // [n_q][nsplit][64][512] partial O
  float *part_ml;        // [n_q][nsplit][2][64]  (m, l)
  int *status;
};

// rotate (a, b) by -pos * base^(-2i/64), computed in fp64 (pos reaches 2^20)
__device__ __forceinline__ void unrotate_pair(float &a, float &b, int pair, int pos, double base) {
  const double th = (double)pos * pow(base, -2.0 * (double)pair / (double)kRopeDim);
  double sn, cs;
  sincos(th, &sn, &cs);
  const float c = (float)cs, s = (float)sn;
  const float x = a, y = b;
  a = x * c + y * s;
  b = -x * s + y * c;
}

__global__ void __launch_bounds__(kAThreads) attn_simt_kernel(AttnArgs A) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  uint16_t *qs = reinterpret_cast<uint16_t *>(smem_raw);                 // [64][kQStride]
  uint16_t *ks = qs + kHeads * kQStride;                                 // [32][kQStride]
  float *ps = reinterpret_cast<float *>(ks + kAChunk * kQStride);        // [64][32]
  __shared__ float m_run[kHeads], l_run[kHeads], alpha[kHeads];
  __shared__ int valid[kAChunk];

  const int qi = blockIdx.y, split = blockIdx.x, t = threadIdx.x;
  const int seq = __ldg(A.q_seq + qi);
  const int swa_cnt = __ldg(A.swa_cnt + qi), swa_first = __ldg(A.swa_first + qi);
  const bool bad = seq < 0 || seq >= A.n_seq || swa_cnt < 0 || swa_cnt > kSwa ||
                   (swa_cnt > 0 && (swa_first < 0 || swa_first >= A.swa_cap));
  if (bad && t == 0 && split == 0) record_error(A.status, CSA2_ERR_BOUNDS);
  const int n_slots = A.sel_stride + (bad ? 0 : swa_cnt);
  const int c0 = split * A.chunks_per_split;
  const int c1 = min((n_slots + kAChunk - 1) / kAChunk, c0 + A.chunks_per_split);

  // stage q (64 x 512 bf16)
  const uint4 *qsrc = reinterpret_cast<const uint4 *>(A.q + (int64_t)qi * kHeads * kDim);
  for (int i = t; i < kHeads * kDim / 8; i += kAThreads) {
    const int h = i >> 6, c = (i & 63) * 8;
    *reinterpret_cast<uint4 *>(qs + h * kQStride + c) = __ldg(qsrc + i);
  }
  if (t < kHeads) { m_run[t] = -INFINITY; l_run[t] = 0.f; }

  // O-phase ownership: heads 4*hg .. 4*hg+3, dims 2*dg + 32*i (+1), i < 16
  const int hg = t >> 4, dg = t & 15;
  float o[4][32];
#pragma unroll
  for (int a = 0; a < 4; a++)
#pragma unroll
    for (int b = 0; b < 32; b++) o[a][b] = 0.f;
  // S-phase ownership: heads 2*hp, 2*hp+1; entries 4*eq .. 4*eq+3
  const int hp = t >> 3, eq = t & 7;

  for (int c = c0; c < c1 && !bad; c++) {
    __syncthreads();   // previous chunk fully consumed
    // ---- gather + dequantise 32 entries (8 threads per entry, 64 dims each)
    {
      const int e = t >> 3, part = t & 7;
      const int slot = c * kAChunk + e;
      uint16_t *dst = ks + e * kQStride + part * 64;
      int ok = 0;
      if (slot < A.sel_stride) {
        const int j = __ldg(A.sel + (int64_t)qi * A.sel_stride + slot);
        if (j >= 0 && (int64_t)j < A.n_max) {
          ok = 1;
          const uint8_t *rec = A.kv + ((int64_t)seq * A.n_max + j) * kKvBytes;
          const uint4 nb0 = __ldg(reinterpret_cast<const uint4 *>(rec + part * 32));
          const uint4 nb1 = __ldg(reinterpret_cast<const uint4 *>(rec + part * 32 + 16));
          const uint32_t sc = __ldg(reinterpret_cast<const uint32_t *>(rec + 256 + part * 4));
          const uint32_t nw[8] = {nb0.x, nb0.y, nb0.z, nb0.w, nb1.x, nb1.y, nb1.z, nb1.w};
#pragma unroll
          for (int wi = 0; wi < 8; wi++) {            // 8 channels per word
            const float s = e4m3_to_float((sc >> (8 * (wi >> 1))) & 0xFFu) * 0.5f;   // codes are 2x
            uint32_t packed[4];
#pragma unroll
            for (int u = 0; u < 4; u++) {
              const float lo = (float)e2m1_x2((nw[wi] >> (8 * u)) & 15u) * s;
              const float hi = (float)e2m1_x2((nw[wi] >> (8 * u + 4)) & 15u) * s;
              packed[u] = (__float_as_uint(lo) >> 16) | (__float_as_uint(hi) & 0xFFFF0000u);
            }
            *reinterpret_cast<uint4 *>(dst + wi * 8) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
          }
        } else if (j >= 0) {
          record_error(A.status, CSA2_ERR_BOUNDS);
        }
      } else if (slot < n_slots) {
        ok = 1;
        const int ring = (swa_first + (slot - A.sel_stride)) % A.swa_cap;
        const uint8_t *rec = A.swa + ((int64_t)seq * A.swa_cap + ring) * kSwaBytes;
        const uint32_t sc = __ldg(reinterpret_cast<const uint32_t *>(rec + 512 + (part * 2 & ~3)));
#pragma unroll
        for (int v = 0; v < 4; v++) {                  // 16 channels per 16-B load
          const uint4 b = __ldg(reinterpret_cast<const uint4 *>(rec + part * 64 + v * 16));
          const int g = (part * 64 + v * 16) / 32;     // E8M0 group
          const float s = e8m0_to_float((sc >> (8 * (g & 3))) & 0xFFu);
          const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
          uint32_t packed[8];
#pragma unroll
          for (int u = 0; u < 8; u++) {
            const float lo = e4m3_to_float((bw[u >> 1] >> (16 * (u & 1))) & 0xFFu) * s;
            const float hi = e4m3_to_float((bw[u >> 1] >> (16 * (u & 1) + 8)) & 0xFFu) * s;
            packed[u] = (__float_as_uint(lo) >> 16) | (__float_as_uint(hi) & 0xFFFF0000u);
          }
          *reinterpret_cast<uint4 *>(dst + v * 16) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
          *reinterpret_cast<uint4 *>(dst + v * 16 + 8) = make_uint4(packed[4], packed[5], packed[6], packed[7]);
        }
      }
      if (!ok) {
#pragma unroll
        for (int v = 0; v < 8; v++) *reinterpret_cast<uint4 *>(dst + v * 8) = make_uint4(0, 0, 0, 0);
      }
      if (part == 0) valid[e] = ok;
    }
    __syncthreads();
    // ---- scores for heads 2hp, 2hp+1 x entries 4eq..4eq+3
    float sc[2][4];
#pragma unroll
    for (int a = 0; a < 2; a++)
#pragma unroll
      for (int b = 0; b < 4; b++) sc[a][b] = 0.f;
    const uint32_t *q0 = reinterpret_cast<const uint32_t *>(qs + (2 * hp) * kQStride);
    const uint32_t *q1 = reinterpret_cast<const uint32_t *>(qs + (2 * hp + 1) * kQStride);
#pragma unroll 4
    for (int d2 = 0; d2 < kDim / 2; d2++) {
      const uint32_t qa = q0[d2], qb = q1[d2];
      const float qa0 = bf16_lo(qa), qa1 = bf16_hi(qa), qb0 = bf16_lo(qb), qb1 = bf16_hi(qb);
#pragma unroll
      for (int b = 0; b < 4; b++) {
        const uint32_t kw = reinterpret_cast<const uint32_t *>(ks + (4 * eq + b) * kQStride)[d2];
        const float k0 = bf16_lo(kw), k1 = bf16_hi(kw);
        sc[0][b] = fmaf(qa0, k0, fmaf(qa1, k1, sc[0][b]));
        sc[1][b] = fmaf(qb0, k0, fmaf(qb1, k1, sc[1][b]));
      }
    }
    // ---- online softmax update (log2 domain)
#pragma unroll
    for (int a = 0; a < 2; a++) {
      float mx = -INFINITY;
#pragma unroll
      for (int b = 0; b < 4; b++) {
        sc[a][b] = valid[4 * eq + b] ? sc[a][b] * A.scale_log2 : -INFINITY;
        mx = fmaxf(mx, sc[a][b]);
      }
      mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
      mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 4));
      const int h = 2 * hp + a;
      const float m_old = m_run[h];
      const float m_new = fmaxf(m_old, mx);
      float sum = 0.f;
#pragma unroll
      for (int b = 0; b < 4; b++) {
        const float p = (sc[a][b] == -INFINITY) ? 0.f : exp2f(sc[a][b] - m_new);
        ps[h * kAChunk + 4 * eq + b] = p;
        sum += p;
      }
      sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 1);
      sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 2);
      sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 4);
      __syncwarp();
      if (eq == 0) {
        const float al = (m_old == -INFINITY) ? 0.f : exp2f(m_old - m_new);
        alpha[h] = al;
        l_run[h] = l_run[h] * al + sum;
        m_run[h] = m_new;
      }
    }
    __syncthreads();
    // ---- O += P K
#pragma unroll
    for (int a = 0; a < 4; a++) {
      const float al = alpha[4 * hg + a];
#pragma unroll
      for (int b = 0; b < 32; b++) o[a][b] *= al;
    }
    for (int e = 0; e < kAChunk; e++) {
      float p[4];
#pragma unroll
      for (int a = 0; a < 4; a++) p[a] = ps[(4 * hg + a) * kAChunk + e];
      const uint32_t *kr = reinterpret_cast<const uint32_t *>(ks + e * kQStride);
#pragma unroll
      for (int i = 0; i < 16; i++) {
        const uint32_t kw = kr[dg + 16 * i];
        const float k0 = bf16_lo(kw), k1 = bf16_hi(kw);
#pragma unroll
        for (int a = 0; a < 4; a++) {
          o[a][2 * i] = fmaf(p[a], k0, o[a][2 * i]);
          o[a][2 * i + 1] = fmaf(p[a], k1, o[a][2 * i + 1]);
        }
      }
    }
  }
  __syncthreads();

  if (A.nsplit == 1) {
    const int pos = __ldg(A.pos + qi);
#pragma unroll
    for (int a = 0; a < 4; a++) {
      const int h = 4 * hg + a;
      const float l = l_run[h];
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
      for (int i = 0; i < 16; i++) {
        const int d = 2 * dg + 32 * i;
        float x = o[a][2 * i] * inv, y = o[a][2 * i + 1] * inv;
        if (d >= kRopeOff) unrotate_pair(x, y, (d - kRopeOff) >> 1, pos, A.rope_base);
        const int64_t off = ((int64_t)qi * kHeads + h) * kDim + d;
        if (A.out_f32) {
          *reinterpret_cast<float2 *>(static_cast<float *>(A.out) + off) = make_float2(x, y);
        } else {
          *reinterpret_cast<__nv_bfloat162 *>(static_cast<uint16_t *>(A.out) + off) = __floats2bfloat162_rn(x, y);
        }
      }
    }
  } else {
    float *P = A.part + ((int64_t)qi * A.nsplit + split) * kHeads * kDim;
#pragma unroll
    for (int a = 0; a < 4; a++) {
      const int h = 4 * hg + a;
#pragma unroll
      for (int i = 0; i < 16; i++) {
        const int d = 2 * dg + 32 * i;
        *reinterpret_cast<float2 *>(P + h * kDim + d) = make_float2(o[a][2 * i], o[a][2 * i + 1]);
      }
    }
    if (t < kHeads) {
      float *ml = A.part_ml + ((int64_t)qi * A.nsplit + split) * 2 * kHeads;
      ml[t] = m_run[t];
      ml[kHeads + t] = l_run[t];
    }
  }
}

// Combine the split partials of one (query, head) row: 256 threads, one dim pair each.
__global__ void __launch_bounds__(256) attn_merge_kernel(AttnArgs A) {
  const int qi = blockIdx.y, h = blockIdx.x, t = threadIdx.x;
  const float *ml = A.part_ml + (int64_t)qi * A.nsplit * 2 * kHeads;
  float M = -INFINITY;
  for (int s = 0; s < A.nsplit; s++) M = fmaxf(M, ml[s * 2 * kHeads + h]);
  float L = 0.f, x = 0.f, y = 0.f;
  const int d = 2 * t;
  if (M != -INFINITY) {
    for (int s = 0; s < A.nsplit; s++) {
      const float m = ml[s * 2 * kHeads + h];
      if (m == -INFINITY) continue;
      const float wgt = exp2f(m - M);
      L += wgt * ml[s * 2 * kHeads + kHeads + h];
      const float2 v = *reinterpret_cast<const float2 *>(A.part + (((int64_t)qi * A.nsplit + s) * kHeads + h) * kDim + d);
      x += wgt * v.x;
      y += wgt * v.y;
    }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  x *= inv;
  y *= inv;
  if (d >= kRopeOff) unrotate_pair(x, y, (d - kRopeOff) >> 1, __ldg(A.pos + qi), A.rope_base);
  const int64_t off = ((int64_t)qi * kHeads + h) * kDim + d;
  if (A.out_f32)
    *reinterpret_cast<float2 *>(static_cast<float *>(A.out) + off) = make_float2(x, y);
  else
    *reinterpret_cast<__nv_bfloat162 *>(static_cast<uint16_t *>(A.out) + off) = __floats2bfloat162_rn(x, y);
}

int attn_nsplit(int n_q, int sel_stride) {
  const int chunks = (sel_stride + kSwa + kAChunk - 1) / kAChunk;
  int ns = (4 * 152 + n_q - 1) / n_q;
  return ns < 1 ? 1 : (ns > chunks ? chunks : ns);
}

size_t attn_workspace_bytes(int n_q, int sel_stride) {
  const int ns = attn_nsplit(n_q, sel_stride);
  if (ns == 1) return 0;
  return (size_t)n_q * ns * (kHeads * kDim + 2 * kHeads) * sizeof(float);
}

cudaError_t launch_attn_simt(const void *q, const void *kv, int64_t n_max, int n_seq, const int32_t *sel,
                             int sel_stride, const void *swa, int swa_cap, const int32_t *q_seq, const int32_t *pos,
                             const int32_t *swa_first, const int32_t *swa_cnt, int n_q, void *out, int out_dtype,
                             float sm_scale, double rope_base, void *ws, int *status, cudaStream_t st) {
  AttnArgs A;
  A.q = static_cast<const uint16_t *>(q);
  A.kv = static_cast<const uint8_t *>(kv);
  A.n_max = n_max;
  A.n_seq = n_seq;
  A.sel = sel;
  A.sel_stride = sel_stride;
  A.swa = static_cast<const uint8_t *>(swa);
  A.swa_cap = swa_cap;
  A.q_seq = q_seq;
  A.pos = pos;
  A.swa_first = swa_first;
  A.swa_cnt = swa_cnt;
  A.out = out;
  A.out_f32 = out_dtype == CSA2_OUT_F32;
  A.scale_log2 = sm_scale * kLog2e;
  A.rope_base = rope_base;
  const int chunks = (sel_stride + kSwa + kAChunk - 1) / kAChunk;
  A.nsplit = attn_nsplit(n_q, sel_stride);
  A.chunks_per_split = (chunks + A.nsplit - 1) / A.nsplit;
  A.nsplit = (chunks + A.chunks_per_split - 1) / A.chunks_per_split;
  A.part = static_cast<float *>(ws);
  A.part_ml = A.part + (size_t)n_q * A.nsplit * kHeads * kDim;
  A.status = status;
  const size_t smem = (size_t)(kHeads + kAChunk) * kQStride * 2 + (size_t)kHeads * kAChunk * 4;
  int dev = 0;
  cudaGetDevice(&dev);
  static bool attr_done[64] = {};
  if (dev >= 0 && dev < 64 && !attr_done[dev]) {
    cudaFuncSetAttribute(attn_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    attr_done[dev] = true;
  }
  attn_simt_kernel<<<dim3(A.nsplit, n_q), kAThreads, smem, st>>>(A);
  if (A.nsplit > 1) attn_merge_kernel<<<dim3(kHeads, n_q), 256, 0, st>>>(A);
  return cudaGetLastError();
}

}  // namespace csa2
