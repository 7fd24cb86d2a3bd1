// Sparse MQA attention on the 5th-generation tensor cores (csa2_sparse_attn).
//
// Each token keeps one 512-wide latent that serves as key and value for all 64
// query heads; a query attends over its 512 selected entries plus the sliding
// window; RoPE acts on 64 of the 512 dimensions and is undone on the output
// (An infra-oriented diagram of the DeepSeek-V4.1-Flash architecture, reading
// notes).
//
// The entry slots of a query (sel_stride selected entries, -1 = empty, then the
// swa_cnt window entries) are processed in chunks of 128.  Per chunk:
//   1. gather + dequantise the 128 records in shared memory, exactly: a chunk
//      of FP4 latents only to f16 (an E2M1 x E4M3 product has <= 6 significant
//      bits and lies in [2^-10, 2688] or is 0), a chunk holding window entries
//      to bf16 (E4M3 x 2^e fits bf16); Q is staged in the chunk's type;
//   2. S^T[entry][head] = Khat . Q^T     tcgen05 kind::f16, M=128 entries, N=64
//      heads, K=512 (both operands K-major, 128B-swizzled);
//   3. softmax numerators p = 2^(l*log2e - m_ref) per (entry, head), stored as
//      f16 (chunks of FP4 latents, see below; 11 significant bits) or as bf16
//      hi + lo parts (together ~16 significant bits);
//   4. O^T[dim][head] += Vhat^T . P^T     M=128 dims (4 blocks), N=64, K=128
//      entries; Vhat^T is the same shared-memory chunk read MN-major (k = v).
//      A fifth block multiplies an all-ones tile, so its rows accumulate the
//      softmax denominator sum_e p[e][h] with exactly the same weights.
// m_ref is the running per-head maximum, raised lazily: the accumulators in
// TMEM are rescaled only when a chunk's maximum exceeds m_ref by more than 8
// (factor 256), otherwise the larger numerators are simply accumulated.
// A CTA handles a range of chunks of one query; with a single range it
// finishes the output (normalise, un-rotate, store), otherwise it writes
// (O, m, l) partials that attn_tc_merge_kernel combines.  Started ahead of the
// selection (settled inputs), a CTA stages Q, runs window-only chunks, and may
// run a discarded warm-up pass of its first chunk before it waits.
//
// 256 threads: all of them gather/dequantise and run the softmax (warp w reads
// TMEM lane quarter w%4, heads 32*(w/4) ..); lane 0 of warps 0-1 issues the QK
// MMAs and lane 0 of warps 0-4 the PV MMAs; all 8 warps share the final
// read-out of the 5 x 64 accumulator columns.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "launch.cuh"
#include "tc_ptx.cuh"

namespace csa2 {

constexpr int kTcChunk = 128;
static_assert(kHandCap > kTcChunk, "with the handoff a query always has several chunks (splits)");
constexpr int kTcThreads = 256;
// shared-memory layout (bytes; the big regions are 1024-aligned)
constexpr int kSmK = 0;                         // 128 entries x 512 dims bf16  (128 KB)
constexpr int kSmQ = kSmK + 128 * 1024;         // 64 heads  x 512 dims bf16    (64 KB)
constexpr int kSmPhi = kSmQ + 64 * 1024;        // 64 heads  x 128 entries bf16 (16 KB)
constexpr int kSmPlo = kSmPhi + 16 * 1024;      //                              (16 KB)
constexpr int kSmOnes = kSmPlo + 16 * 1024;     // one 8 x 16-B core matrix of bf16 ones (128 B)
constexpr int kSmOnes16 = kSmOnes + 128;        // the same of f16 ones (128 B)
constexpr int kSmMref = kSmOnes16 + 128;        // float[64] running maxima
constexpr int kSmAlpha = kSmMref + 256;         // float[64] rescale factors
constexpr int kSmValid = kSmAlpha + 256;        // uint8[128] slot validity
constexpr int kSmBars = kSmValid + 128;         // 2 mbarriers, tmem base, flags
constexpr int kSmTotal = kSmBars + 48;            // + the drain barrier at kSmBars + 32
constexpr int kSmAlloc = kSmTotal + 1024;       // + alignment slack (<= 227 KB)
constexpr uint32_t kAttTmemCols = 512;
constexpr uint32_t kColS = 0;                   // S^T, dims 0..255 of the dot products: 64 columns
constexpr uint32_t kColO = 64;                  // O^T: 5 blocks x 64 columns (block 4 = denominators)
constexpr uint32_t kColS2 = 384;                // S^T, dims 256..511: 64 columns (a second issuer)
constexpr float kRescaleLog2 = 8.0f;

// Eight E2M1 codes (one per nibble of w, channel i in nibble i) -> eight bf16
// values as four bf16x2 words, by table lookups with __byte_perm: the high and
// low bytes of the bf16 magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6}, then the sign.
__device__ __forceinline__ void e2m1x8_to_bf16(uint32_t w, uint32_t (&out)[4]) {
#pragma unroll
  for (int hw = 0; hw < 2; hw++) {
    const uint32_t n = w >> (16 * hw);               // nibbles of channels 4hw .. 4hw+3
    const uint32_t sel = n & 0x7777u;
    const uint32_t hi = __byte_perm(0x3F3F3F00u, 0x40404040u, sel);
    const uint32_t lo = __byte_perm(0xC0800000u, 0xC0804000u, sel);
    uint32_t a = __byte_perm(lo, hi, 0x5140u);       // channels 4hw, 4hw+1
    uint32_t b = __byte_perm(lo, hi, 0x7362u);       // channels 4hw+2, 4hw+3
    a |= ((n << 12) & 0x8000u) | ((n << 24) & 0x80000000u);
    b |= ((n << 4) & 0x8000u) | ((n << 16) & 0x80000000u);
    out[2 * hw] = a;
    out[2 * hw + 1] = b;
  }
}

// Two E4M3 codes (low byte first) -> their values as f16x2 (exact: E4M3 is a
// subset of f16), by the hardware converter.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t two) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((unsigned short)two));
  return __half22float2(*reinterpret_cast<__half2 *>(&h));
}

// byte offset of 16-B chunk `ch` (0..7) in row r of a 128B-swizzled 1024-B atom
__device__ __forceinline__ uint32_t sw128(uint32_t r, uint32_t ch) { return r * 128u + ((ch ^ (r & 7u)) << 4); }

// kind::f16 instruction descriptor: bf16 x bf16 (or f16 x f16) -> f32, M=128,
// N = n (a multiple of 16), A K- or MN-major.
__host__ __device__ constexpr uint32_t idesc_m128(uint32_t a_mn_major, bool f16, uint32_t n) {
  return (1u << 4)                     // D format f32
         | ((f16 ? 0u : 1u) << 7)      // A: f16 0, bf16 1
         | ((f16 ? 0u : 1u) << 10)     // B: f16 0, bf16 1
         | (a_mn_major << 15)          // A major-ness
         | ((n >> 3) << 17)            // N / 8
         | ((128u >> 4) << 24);        // M / 16
}

// Eight E2M1 codes (channel i in nibble i of w) -> eight f16 values as four
// f16x2 words, by the hardware converter (exact: E2M1 is a subset of f16).
__device__ __forceinline__ void e2m1x8_to_f16(uint32_t w, uint32_t (&out)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(out[0]), "=r"(out[1]), "=r"(out[2]), "=r"(out[3])
      : "r"(w));
}

// Two E4M3 codes (low byte first) -> f16x2 bits (exact).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((unsigned short)two));
  return h;
}

struct AttnTcArgs {
  const uint16_t *q;
  const uint8_t *kv;
  int64_t n_max;
  int n_seq;
  const int32_t *sel;
  int sel_stride;
  // entry slots ahead of the window: sel_stride, or kHandCap with the handoff
  int n_sel;
  // optional: the selection grid ahead hands its candidates over (null: off)
  const uint32_t *hflag;
  const uint64_t *hcand;
  int hparts;       // selection CTAs per query (each publishes one segment of candidates)
  const uint8_t *swa;
  int swa_cap;
  const int32_t *q_seq, *pos, *swa_first, *swa_cnt;
  void *out;
  int out_f32;
  float scale_log2;
  double inv_freq[kRopeDim / 2];   // rope_base^(-2i/64)
  int nsplit, chunks_per_split;
  int merge_tail;   // the last split also runs the window-only chunks, first (settled inputs: during the selection)
  int hsplit;       // CTAs sharing a chunk, each with 64 / hsplit of the heads
  float *part;      // [n_q][nsplit][64][512]: unnormalised O
  float *part_ml;   // [n_q][nsplit][2][64]
  int *status;
  int settled;      // q, the window cache and the per-query arrays may be read before the grid ahead completes
  int warm;         // settled, one chunk per CTA, all CTAs resident beside the grid ahead: warm-up pass
};

// cos and sin of theta = pos * inv_freq (inv_freq = rope_base^(-2i/64), computed
// on the host in fp64): the product and its reduction modulo 2 pi are done in
// fp64 (pos reaches 2^20, so theta reaches ~1e6 rad), the sine and cosine of the
// reduced angle in fp32.
__device__ __forceinline__ void rope_cs(double inv_freq, int pos, float &c, float &s) {
  const double th = (double)pos * inv_freq;
  const double k = rint(th * 0.15915494309189535);            // 1 / (2 pi)
  const double r = fma(-k, 6.283185307179586, th);
  sincosf((float)r, &s, &c);
}

// NH: the heads one CTA handles (64, or 32 when two CTAs share each chunk:
// the gather is repeated, the MMAs, the softmax and the read-out are halved).
// HAND: the selection grid ahead hands its candidates over (A.hflag set).
template <int NH, bool HAND>
__global__ void __launch_bounds__(kTcThreads, 1) attn_tc_kernel(AttnTcArgs A) {
  static_assert(NH == 64 || NH == 32, "heads per CTA");
  constexpr int HS = kHeads / NH;                 // CTAs per chunk
  constexpr int HW = NH / 2;                      // heads per softmax warp (two warps per TMEM lane quarter)
  extern __shared__ __align__(1024) unsigned char at_smem_raw[];
  unsigned char *sm = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(at_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  float *m_ref = reinterpret_cast<float *>(sm + kSmMref);
  float *alpha_sh = reinterpret_cast<float *>(sm + kSmAlpha);
  float(*red)[kHeads] = reinterpret_cast<float(*)[kHeads]>(sm + kSmPhi);   // [4][64], during the max only
  uint8_t *valid_sh = sm + kSmValid;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kSmBars);
  uint64_t &bar_s = bars[0], &bar_o = bars[1], &bar_drain = bars[4];
  uint32_t &tmem_sh = *reinterpret_cast<uint32_t *>(sm + kSmBars + 16);
  volatile int &bad_sh = *reinterpret_cast<volatile int *>(sm + kSmBars + 24);

  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  // grid (n_q, nsplit x HS), the last split first: the window-only chunks,
  // which need no selection, are the first CTAs to be placed; heads [h0, h0 + NH)
  const int qi = blockIdx.x, split = A.nsplit - 1 - (int)blockIdx.y / HS, h0 = ((int)blockIdx.y % HS) * NH;
  // The selection (sel) comes from the grid ahead.  With settled inputs the
  // wait is put off until the first chunk that holds selected entries: Q is
  // staged and window-only chunks run while the selection finishes.  (TMEM is
  // taken before the wait only then, when the grid ahead is the top-k, which
  // holds no TMEM.)  With the handoff, that chunk waits only for the
  // candidates, and the softmax for the smallest selected key; the grid
  // completion wait moves to the end (no data of the grid ahead is read after
  // it), and the grid that follows may be placed at once.
  __shared__ uint32_t hand_sh;
  __shared__ uint64_t kth_sh;
  __shared__ int hoff_sh[kHandCtas + 1];           // first candidate slot of each segment
  bool waited = false;
  if (HAND) griddep_launch();
  if (!HAND && !A.settled) {                       // (the handoff runs inside csa2_decode: settled)
    griddep_wait();
    griddep_launch();
    waited = true;
  }
  const int seq = __ldg(A.q_seq + qi);
  const int swa_cnt = __ldg(A.swa_cnt + qi), swa_first = __ldg(A.swa_first + qi);
  // the position is needed only by the read-out: loaded now, kept in shared
  // memory once Q is staged
  __shared__ int pos_sh;
  const int pos0 = t == 0 ? __ldg(A.pos + qi) : 0;
  const bool bad = seq < 0 || seq >= A.n_seq || swa_cnt < 0 || swa_cnt > kSwa || swa_cnt > A.swa_cap ||
                   (swa_cnt > 0 && (swa_first < 0 || swa_first >= A.swa_cap));
  if (bad && t == 0 && split == 0 && h0 == 0) record_error(A.status, CSA2_ERR_BOUNDS);
  const int n_slots = A.n_sel + (bad ? 0 : swa_cnt);
  // A merged last split (settled inputs) runs the window-only chunks first,
  // while the selection finishes, then its chunks of selected entries
  const bool merged = A.merge_tail && split == A.nsplit - 1;
  const int c0 = split * A.chunks_per_split;
  const int c1 = bad ? c0 : min((n_slots + kTcChunk - 1) / kTcChunk, merged ? 1 << 20 : c0 + A.chunks_per_split);
  const int sel_end = (A.n_sel + kTcChunk - 1) / kTcChunk;      // the first window-only chunk
  const int n_w = merged ? max(0, c1 - max(c0, sel_end)) : 0;  // window-only chunks run first

  if (t == 0) {
    ptx::mbar_init(&bar_s, 2);                       // two S issuers
    ptx::mbar_init(&bar_o, 5);                       // five O issuers
    ptx::mbar_init(&bar_drain, 5);                   // the MMA issuers, once each, after a wait ran out
    bad_sh = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0) ptx::tmem_alloc(&tmem_sh, kAttTmemCols);
  if (t < NH) m_ref[t] = -INFINITY;
  // start the first chunk's record reads (L2 prefetch) while Q is staged
  if (waited && c0 < c1) {
    const int e = t >> 1, half = t & 1, slot = c0 * kTcChunk + e;
    const uint8_t *rec = nullptr;
    int bytes = 0;
    if (slot < A.n_sel) {
      const int j = slot < A.sel_stride ? __ldg(A.sel + (int64_t)qi * A.sel_stride + slot) : -1;
      if (j >= 0 && (int64_t)j < A.n_max) { rec = A.kv + ((int64_t)seq * A.n_max + j) * kKvBytes; bytes = kKvBytes; }
    } else if (slot < n_slots) {
      const int ring = (swa_first + (slot - A.n_sel)) % A.swa_cap;
      rec = A.swa + ((int64_t)seq * A.swa_cap + ring) * kSwaBytes;
      bytes = kSwaBytes;
    }
    for (int o = half * 128; rec != nullptr && o < bytes; o += 256)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(rec + o));
  }
  // Stage Q (K-major, 128B swizzle: [head/8][dim/64][head%8][128 B]) in the
  // operand type of the chunk ahead: bf16, or f16 for a chunk of FP4 latents
  // only (their dequantised values are exact in f16 and the hardware converts
  // E2M1 straight to f16).  In f16, Q is scaled by 2^-qs, the power of two
  // that brings max |q| into [2^14, 2^15) (qs >= -100): exact but for elements
  // below 2^-24 of that range, and folded back into the softmax scale.
  // Returns 2^qs.
  __shared__ uint32_t qmax_sh[kTcThreads / 32];
  constexpr int kQv = NH * kDim / 8 / kTcThreads;    // 16-B loads per thread
  auto stage_q = [&](bool f16) -> float {
    const uint4 *src = reinterpret_cast<const uint4 *>(A.q + ((int64_t)qi * kHeads + h0) * kDim);
    uint4 qv[kQv];                                   // all loads in flight before any store
#pragma unroll
    for (int j = 0; j < kQv; j++) qv[j] = __ldg(src + t + j * kTcThreads);
    float qscale = 1.f;
    if (f16) {
      uint32_t m = 0u;                               // max |q| as bf16 bits, two lanes per word
#pragma unroll
      for (int j = 0; j < kQv; j++) {
        m = __vmaxu2(m, qv[j].x & 0x7FFF7FFFu);
        m = __vmaxu2(m, qv[j].y & 0x7FFF7FFFu);
        m = __vmaxu2(m, qv[j].z & 0x7FFF7FFFu);
        m = __vmaxu2(m, qv[j].w & 0x7FFF7FFFu);
      }
      m = __reduce_max_sync(0xFFFFFFFFu, max(m & 0xFFFFu, m >> 16));
      if (lane == 0) qmax_sh[warp] = m;
      __syncthreads();
      uint32_t mm = 0u;
#pragma unroll
      for (int w = 0; w < kTcThreads / 32; w++) mm = max(mm, qmax_sh[w]);
      const int ex = (int)((mm >> 7) & 0xFFu) - 127;  // max |q| in [2^ex, 2^(ex + 1)) if normal
      const int qs = mm == 0u ? 0 : max(ex - 14, -100);
      qscale = ldexpf(1.f, qs);
      const float inv = ldexpf(1.f, -qs);
#pragma unroll
      for (int j = 0; j < kQv; j++) {
        uint32_t wd[4] = {qv[j].x, qv[j].y, qv[j].z, qv[j].w};
#pragma unroll
        for (int k = 0; k < 4; k++) {
          const __half2 h2 = __floats2half2_rn(bf16_lo(wd[k]) * inv, bf16_hi(wd[k]) * inv);
          wd[k] = *reinterpret_cast<const uint32_t *>(&h2);
        }
        qv[j] = make_uint4(wd[0], wd[1], wd[2], wd[3]);
      }
    }
#pragma unroll
    for (int j = 0; j < kQv; j++) {
      const int i = t + j * kTcThreads;
      const int h = i >> 6, ch = i & 63;               // 16-B chunk ch of row h (8 dims)
      const uint32_t off = (h >> 3) * 8192 + (ch >> 3) * 1024 + sw128(h & 7, ch & 7);
      *reinterpret_cast<uint4 *>(sm + kSmQ + off) = qv[j];
    }
    return qscale;
  };
  // the chunks of FP4 latents only (the first n_sel / 128 ones) run in f16
  auto chunk_f16 = [&](int c) { return (c + 1) * kTcChunk <= A.n_sel; };
  bool q16 = c0 < c1 && chunk_f16(n_w > 0 ? c1 - n_w : c0);   // the type of the first chunk run
  float qscale = stage_q(q16);
  // all-ones A operands: one 8 x 16-B core matrix of 1.0 in bf16 and in f16,
  // read for every row group and K chunk (both descriptor strides 0)
  if (t < 8)
    *reinterpret_cast<uint4 *>(sm + kSmOnes + t * 16) = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
  else if (t < 16)
    *reinterpret_cast<uint4 *>(sm + kSmOnes16 + (t - 8) * 16) =
        make_uint4(0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u);
  if (t == 0) pos_sh = pos0;
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = tmem_sh;
  const uint32_t sK = ptx::smem_u32(sm + kSmK), sQ = ptx::smem_u32(sm + kSmQ);
  const uint32_t sPhi = ptx::smem_u32(sm + kSmPhi), sPlo = ptx::smem_u32(sm + kSmPlo);
  const uint32_t sOnes = ptx::smem_u32(sm + kSmOnes), sOnes16 = ptx::smem_u32(sm + kSmOnes16);
  uint32_t phase = 0;
  bool any_chunk = false;

  // A CTA that has to wait for the selection first runs its first chunk's
  // pipeline once over the sequence's first 128 entries (settled inputs) and
  // discards the result (wp: the warm-up pass): the real pass then finds its
  // instructions in the SM's caches instead of fetching each phase's code as
  // it first runs.
  const int warm = A.warm && !waited && c0 < c1 && c0 * kTcChunk < A.n_sel ? 1 : 0;
  uint32_t hnc = 0;                                  // handoff: candidates + 1, or kHandFallback
  bool got_sel = false;
  // A CTA with several chunks of selected entries reads the records of the
  // next one into registers while the current one runs its MMAs and softmax
  // (pre_c: the chunk whose records rec_sc / rec_nb hold; the gather of a
  // chunk without them loads them itself)
  int pre_c = -1, pre_j = -1;
  uint32_t rec_sc[4];                                // this thread's half-record: 16 E4M3 scales
  uint4 rec_nb[8];                                   //   and 256 E2M1 latents
  auto load_rec = [&](int j) {
    const int half = t & 1;
    const uint8_t *rec = A.kv + ((int64_t)seq * A.n_max + j) * kKvBytes;
#pragma unroll
    for (int k = 0; k < 4; k++) rec_sc[k] = __ldg(reinterpret_cast<const uint32_t *>(rec + 256 + half * 16 + 4 * k));
#pragma unroll
    for (int v = 0; v < 8; v++) rec_nb[v] = __ldg(reinterpret_cast<const uint4 *>(rec + half * 128 + v * 16));
  };
  for (int kc = c0, wp = warm; kc < c1; kc += 1 - wp, wp = 0) {
    const int c = kc - c0 < n_w ? c1 - n_w + (kc - c0) : kc - n_w;   // (merged: window-only chunks first)
    const bool sel_chunk = !wp && c * kTcChunk < A.n_sel;   // the chunk holds selected entries (or candidates)
    if (sel_chunk && !got_sel) {
      got_sel = true;
      if (!HAND) {
        if (!waited) {
          griddep_wait();
          griddep_launch();
          waited = true;
        }
      } else {
        // every selection CTA of the query has published its segment: the
        // segments' counts give each candidate slot; too many candidates, or a
        // segment that could not be handed over, and the chunk waits for the
        // final selection instead
        const uint32_t *hf = A.hflag + (int64_t)qi * kHandWords;
        if (t == 0) {
          uint32_t v = 1u;                           // candidates + 1
          if (!ptx::poll_at_least_u32(hf, (uint32_t)A.hparts)) {
            record_error(A.status, CSA2_ERR_TIMEOUT);
            bad_sh = 1;                              // (v = 1: no candidates)
          } else {
            uint32_t cnt[kHandCtas];                 // all counts in one round trip
            const uint4 *c4 = reinterpret_cast<const uint4 *>(hf + 8);
#pragma unroll
            for (int v4 = 0; v4 < kHandCtas / 4; v4++) {
              const uint4 x = __ldcg(c4 + v4);
              cnt[4 * v4] = x.x;
              cnt[4 * v4 + 1] = x.y;
              cnt[4 * v4 + 2] = x.z;
              cnt[4 * v4 + 3] = x.w;
            }
            int o = 0;
            bool fb = false;
#pragma unroll
            for (int p = 0; p < kHandCtas; p++) {
              if (p < A.hparts) {
                hoff_sh[p] = o;
                fb = fb || cnt[p] == kHandFallback;
                o += fb ? 0 : (int)cnt[p];
              }
            }
            hoff_sh[A.hparts] = o;
            v = (fb || o > kHandCap) ? kHandFallback : (uint32_t)o + 1u;
          }
          if (v == kHandFallback && !ptx::poll_at_least_u32(hf + 1, 1u)) {   // the final selection
            record_error(A.status, CSA2_ERR_TIMEOUT);
            bad_sh = 1;
            v = 1u;
          }
          hand_sh = v;
        }
        __syncthreads();
        hnc = hand_sh;
      }
    }
    // handoff: candidates to be masked once the smallest selected key is out
    const bool hand_live = HAND && sel_chunk && hnc != kHandFallback;
    if (HAND && sel_chunk && c * kTcChunk >= (hand_live ? (int)hnc - 1 : A.sel_stride))
      continue;                                      // uniform: the chunk holds no entry
    // a chunk of selected entries only whose 128 slots are all empty (a query
    // with fewer visible entries than k: a prefill's early positions) is
    // skipped; the slot indices read here serve its gather too
    int sel_j = -1;
    if (sel_chunk && !hand_live) {                   // (the handoff's fallback reads the selection too)
      const int slot = c * kTcChunk + (t >> 1);
      sel_j = pre_c == c ? pre_j : (slot < A.sel_stride ? __ldcg(A.sel + (int64_t)qi * A.sel_stride + slot) : -1);
      if (!__syncthreads_or(sel_j >= 0) && (c + 1) * kTcChunk <= A.n_sel) continue;
    }
    const bool f16c = chunk_f16(c);
    if (f16c != q16) {                                // the last chunk's MMAs are complete
      qscale = stage_q(f16c);
      q16 = f16c;
      ptx::fence_proxy_async_smem();
      __syncthreads();
    }
    const uint32_t id_qk = idesc_m128(0, f16c, NH), id_pv = idesc_m128(1, f16c, NH);
    const float sl2 = A.scale_log2 * (f16c ? qscale : 1.f);   // S was computed with Q x 2^-qs
    // ---------------------------------------------------------- gather + dequantise
    uint64_t hk = 0ull;                              // handoff: this slot's candidate key
    {
      const int e = t >> 1, half = t & 1;             // entry slot e, dims [256*half, 256*half+256)
      const int slot = c * kTcChunk + e;
      const uint32_t rowbase = (e >> 3) * 8192;        // 8-entry group
      int ok = 0;
      if (slot < A.n_sel) {
        int j = -1;
        if (wp) {
          j = (int64_t)e < A.n_max ? e : -1;
        } else if (hand_live) {
          if (slot < (int)hnc - 1) {                  // the key's low half is ~index
            int p = 0;
            while (slot >= hoff_sh[p + 1]) p++;
            hk = __ldcg(A.hcand + ((int64_t)qi * kHandCtas + p) * kHandSeg + (slot - hoff_sh[p]));
            j = (int)~(uint32_t)hk;
          }
        } else {
          j = sel_j;                                  // (read above)
        }
        if (j >= 0 && (int64_t)j < A.n_max) {
          ok = 1;
          if (pre_c != c) load_rec(j);
          const uint32_t(&sc4)[4] = rec_sc;
          const uint4(&nbv)[8] = rec_nb;
          if (f16c) {
            // f16: E2M1 pairs and E4M3 scale pairs by the hardware converter
            uint32_t sh[8];                           // the half-row's 16 scales as f16x2 pairs
#pragma unroll
            for (int k = 0; k < 8; k++) sh[k] = e4m3x2_to_f16x2(sc4[k >> 1] >> (16 * (k & 1)));
#pragma unroll
            for (int v = 0; v < 8; v++) {
              const uint32_t nw[4] = {nbv[v].x, nbv[v].y, nbv[v].z, nbv[v].w};
#pragma unroll
              for (int u = 0; u < 4; u++) {
                const int d0 = half * 256 + v * 32 + u * 8;
                const int g = 2 * v + (u >> 1);       // scale group within this half (0..15)
                const uint32_t sg = (sh[g >> 1] >> (16 * (g & 1))) & 0xFFFFu;
                const uint32_t s2w = sg | (sg << 16);
                uint32_t pk[4];
                e2m1x8_to_f16(nw[u], pk);
#pragma unroll
                for (int b = 0; b < 4; b++) {
                  __half2 x = *reinterpret_cast<__half2 *>(&pk[b]);
                  x = __hmul2(x, *reinterpret_cast<const __half2 *>(&s2w));   // exact: <= 10 significant bits, <= 2688
                  pk[b] = *reinterpret_cast<uint32_t *>(&x);
                }
                const uint32_t off = rowbase + (d0 >> 6) * 1024 + sw128(e & 7, (d0 >> 3) & 7);
                *reinterpret_cast<uint4 *>(sm + kSmK + off) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
              }
            }
          } else
#pragma unroll
          for (int v = 0; v < 8; v++) {               // 16-B nibble load = 32 dims
            const uint32_t nw[4] = {nbv[v].x, nbv[v].y, nbv[v].z, nbv[v].w};
#pragma unroll
            for (int u = 0; u < 4; u++) {             // 8 dims per word -> one 16-B smem chunk
              const int d0 = half * 256 + v * 32 + u * 8;
              const int g = (d0 >> 4) - half * 16;    // scale group within this half (0..15)
              const __nv_bfloat16 sb = __float2bfloat16_rn(e4m3_to_float((sc4[g >> 2] >> (8 * (g & 3))) & 0xFFu));
              const __nv_bfloat162 s2 = __halves2bfloat162(sb, sb);
              uint32_t pk[4];
              e2m1x8_to_bf16(nw[u], pk);
#pragma unroll
              for (int b = 0; b < 4; b++) {
                __nv_bfloat162 x = *reinterpret_cast<__nv_bfloat162 *>(&pk[b]);
                x = __hmul2(x, s2);                   // exact: <= 6 significant bits, in range
                pk[b] = *reinterpret_cast<uint32_t *>(&x);
              }
              const uint32_t off = rowbase + (d0 >> 6) * 1024 + sw128(e & 7, (d0 >> 3) & 7);
              *reinterpret_cast<uint4 *>(sm + kSmK + off) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
          }
        } else if (j >= 0) {
          record_error(A.status, CSA2_ERR_BOUNDS);
        }
      } else if (slot < n_slots) {
        ok = 1;
        const int ring = (swa_first + (slot - A.n_sel)) % A.swa_cap;
        const uint8_t *rec = A.swa + ((int64_t)seq * A.swa_cap + ring) * kSwaBytes;
        const uint2 scw = __ldg(reinterpret_cast<const uint2 *>(rec + 512 + half * 8));
        const uint32_t sc2[2] = {scw.x, scw.y};
        uint4 bv[16];
#pragma unroll
        for (int v = 0; v < 16; v++) bv[v] = __ldg(reinterpret_cast<const uint4 *>(rec + half * 256 + v * 16));
#pragma unroll
        for (int v = 0; v < 16; v++) {                // 16 B = 16 dims per load
          const uint4 b = bv[v];
          const int g = v >> 1;                       // E8M0 group (32 dims) within this half
          const float s = e8m0_to_float((sc2[g >> 2] >> (8 * (g & 3))) & 0xFFu);
          const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
          for (int hf = 0; hf < 2; hf++) {            // two 8-dim smem chunks
            uint32_t pk[4];
#pragma unroll
            for (int u = 0; u < 4; u++) {
              const uint32_t word = bw[hf * 2 + (u >> 1)];
              const float2 f = e4m3x2_to_float2(word >> (16 * (u & 1)));   // exact; x the power-of-two scale: exact
              const __nv_bfloat162 bb = __floats2bfloat162_rn(f.x * s, f.y * s);
              pk[u] = *reinterpret_cast<const uint32_t *>(&bb);
            }
            const int d0 = half * 256 + v * 16 + hf * 8;
            const uint32_t off = rowbase + (d0 >> 6) * 1024 + sw128(e & 7, (d0 >> 3) & 7);
            *reinterpret_cast<uint4 *>(sm + kSmK + off) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          }
        }
      }
      if (!ok) {
#pragma unroll 4
        for (int ch = 0; ch < 32; ch++) {
          const int d0 = half * 256 + ch * 8;
          const uint32_t off = rowbase + (d0 >> 6) * 1024 + sw128(e & 7, (d0 >> 3) & 7);
          *reinterpret_cast<uint4 *>(sm + kSmK + off) = make_uint4(0, 0, 0, 0);
        }
      }
      if (half == 0) valid_sh[e] = (uint8_t)ok;
    }
    ptx::fence_proxy_async_smem();
    __syncthreads();
    // ---------------------------------------------------------- S^T = Khat Q^T
    // two issuers (lane 0 of warps 0 and 1), dims 0..255 and 256..511 into two
    // tiles that the softmax adds: tcgen05 issue cost is per thread
    if (lane == 0 && warp < 2) {
      ptx::tc_fence_after();
      const uint32_t col = warp == 0 ? kColS : kColS2;
#pragma unroll 1
      for (int k2 = 0; k2 < kDim / 32; k2++) {
        const int kk = warp * (kDim / 32) + k2;
        const uint32_t koff = (kk >> 2) * 1024 + (kk & 3) * 32;
        const uint64_t ad = ptx::smem_desc(sK + koff, 16, 8192, 2);
        const uint64_t bd = ptx::smem_desc(sQ + koff, 16, 8192, 2);
        ptx::tc_mma_bf16(tmem + col, ad, bd, id_qk, k2 > 0 ? 1u : 0u);
      }
      ptx::tc_commit(&bar_s);
    }
    // the next chunk's records, if it holds selected entries only (its smem
    // stores wait for this chunk's PV)
    if (!HAND && got_sel && !wp && c + 1 < c1 && chunk_f16(c + 1)) {
      const int slot = (c + 1) * kTcChunk + (t >> 1);
      pre_c = c + 1;
      pre_j = slot < A.sel_stride ? __ldcg(A.sel + (int64_t)qi * A.sel_stride + slot) : -1;
      if (pre_j >= 0 && (int64_t)pre_j < A.n_max) load_rec(pre_j);
    }
    // ---------------------------------------------------------- handoff mask
    // while S is computed: candidates below the smallest selected key drop out
    if (hand_live) {
      if (t == 0) {
        uint64_t K = 0ull;
        if (!ptx::poll_nonzero_u64(reinterpret_cast<const uint64_t *>(A.hflag + (int64_t)qi * kHandWords + 2), K)) {
          record_error(A.status, CSA2_ERR_TIMEOUT);
          bad_sh = 1;
          K = ~0ull;
        }
        kth_sh = K;
      }
      __syncthreads();
      if ((t & 1) == 0 && valid_sh[t >> 1] != 0) valid_sh[t >> 1] = hk >= kth_sh ? 1 : 0;
      __syncthreads();
    }
    // ---------------------------------------------------------- softmax (all 8 warps)
    int need_rescale = 0;
    // warp w: TMEM lane quarter w%4 (entries 32*(w%4) ..), heads HW*(w/4) .. +HW-1
    {
      const int quarter = warp & 3, hb = (warp >> 2) * HW;
      if (!ptx::mbar_wait(&bar_s, phase)) { record_error(A.status, CSA2_ERR_TIMEOUT); bad_sh = 1; }
      ptx::tc_fence_after();
      const int e = quarter * 32 + lane;               // TMEM lane = entry
      const uint32_t s_addr = tmem + ((uint32_t)(quarter * 32) << 16) + kColS + hb;
      const bool ev = valid_sh[e] != 0;
      // S (two K halves, summed) for this warp's HW heads
      auto load_s = [&](float (&x)[HW]) {
        if constexpr (HW == 32) {
          uint32_t r[32], r2[32];
          ptx::tmem_ld_32x32b_x32(s_addr, r);
          ptx::tmem_ld_32x32b_x32(s_addr + (kColS2 - kColS), r2);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int h = 0; h < 32; h++) x[h] = (__uint_as_float(r[h]) + __uint_as_float(r2[h])) * sl2;
        } else {
          uint32_t r[16], r2[16];
          ptx::tmem_ld_32x32b_x16(s_addr, r);
          ptx::tmem_ld_32x32b_x16(s_addr + (kColS2 - kColS), r2);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int h = 0; h < 16; h++) x[h] = (__uint_as_float(r[h]) + __uint_as_float(r2[h])) * sl2;
        }
      };
      // per-head max over the warp's 32 entries: transpose-reduce (HW - 1
      // shuffles, one more when HW = 16); afterwards lane L holds the max of
      // head hb + L % HW
      float v[HW];
      load_s(v);
#pragma unroll
      for (int h = 0; h < HW; h++) v[h] = ev ? v[h] : -INFINITY;
#pragma unroll
      for (int w = HW / 2; w >= 1; w >>= 1) {          // w = values kept, partner distance w
        const bool upper = (lane & w) != 0;
#pragma unroll
        for (int i = 0; i < HW / 2; i++) {
          if (i < w) {
            const float mine = upper ? v[i + w] : v[i];
            const float send = upper ? v[i] : v[i + w];
            v[i] = fmaxf(mine, __shfl_xor_sync(0xFFFFFFFFu, send, w));
          }
        }
      }
      if (HW == 16) v[0] = fmaxf(v[0], __shfl_xor_sync(0xFFFFFFFFu, v[0], 16));
      red[quarter][hb + (lane & (HW - 1))] = v[0];
      __syncthreads();
      int rs = 0;                                      // some head's accumulators need rescaling
      if (t < NH) {
        const float cm = fmaxf(fmaxf(red[0][t], red[1][t]), fmaxf(red[2][t], red[3][t]));
        const float mo = m_ref[t];
        float al = 1.f;
        if (cm != -INFINITY && (mo == -INFINITY || cm > mo + kRescaleLog2)) {
          al = (mo == -INFINITY) ? 0.f : exp2f(mo - cm);
          m_ref[t] = cm;
        }
        alpha_sh[t] = al;
        rs = al != 1.f && al != 0.f;
      }
      need_rescale = __syncthreads_or(rs);
      // numerators, bf16 hi + lo, into P[head][entry] (K-major, 128B swizzle);
      // S is read from TMEM again rather than kept live through the reduction
      const uint32_t pe = (e >> 6) * 1024;             // entry atom
      const uint32_t pcol = (uint32_t)(e & 63) * 2;    // byte within the 128-B row
      float l2v[HW];
      load_s(l2v);
      // f16 chunks: the numerator rounded to f16 (11 significant bits); bf16
      // chunks: bf16 hi + lo parts (~16 bits).  One loop per type.
      auto off_of = [&](int i) {
        const int h = hb + i;
        return (h >> 3) * 2048 + pe + sw128(h & 7, pcol >> 4) + (pcol & 15);
      };
      auto put = [&](int i, uint16_t hi, uint16_t lo) {
        const uint32_t off = off_of(i);
        *reinterpret_cast<uint16_t *>(sm + kSmPhi + off) = hi;
        *reinterpret_cast<uint16_t *>(sm + kSmPlo + off) = lo;
      };
      if (f16c) {
#pragma unroll
        for (int i = 0; i < HW; i++) {
          const float p = ev ? exp2f(l2v[i] - m_ref[hb + i]) : 0.f;
          *reinterpret_cast<__half *>(sm + kSmPhi + off_of(i)) = __float2half_rn(p);
        }
      } else {
#pragma unroll
        for (int i = 0; i < HW; i++) {
          const float p = ev ? exp2f(l2v[i] - m_ref[hb + i]) : 0.f;
          const __nv_bfloat16 ph = __float2bfloat16_rn(p);
          put(i, __bfloat16_as_ushort(ph), __bfloat16_as_ushort(__float2bfloat16_rn(p - __bfloat162float(ph))));
        }
      }
      ptx::tc_fence_before();
    }
    ptx::fence_proxy_async_smem();
    __syncthreads();
    // ---------------------------------------------------------- lazy rescale of O^T
    if (need_rescale && any_chunk) {
      ptx::tc_fence_after();
      // warp w: lane quarter w%4, blocks {w/4, w/4 + 2} (+ block 4 for warps 0-3)
      const int quarter = warp & 3;
      for (int blk = warp >> 2; blk < 5; blk += 2) {
        if (blk == 4 && warp >= 4) break;
        for (int half = 0; half < NH / 32; half++) {
          uint32_t r[32];
          const uint32_t ta = tmem + ((uint32_t)(quarter * 32) << 16) + kColO + blk * NH + half * 32;
          ptx::tmem_ld_32x32b_x32(ta, r);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; i++) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha_sh[half * 32 + i]);
          ptx::tmem_st_32x32b_x32(ta, r);
        }
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncthreads();
    }
    // ---------------------------------------------------------- O^T += Vhat^T P^T
    // five issuers (lane 0 of warps 0..4): dim blocks 0..3, then the
    // denominators (ones x P^T)
    if (lane == 0 && warp < 5) {
      ptx::tc_fence_after();
      const int mb = warp;
#pragma unroll 1
      for (int ks = 0; ks < kTcChunk / 16; ks++) {
        const uint32_t poff = (ks >> 2) * 1024 + (ks & 3) * 32;
        const uint64_t bhi = ptx::smem_desc(sPhi + poff, 16, 2048, 2);
        const uint64_t blo = ptx::smem_desc(sPlo + poff, 16, 2048, 2);
        const uint32_t acc0 = (any_chunk || ks > 0) ? 1u : 0u;
        if (mb < 4) {
          // Vhat^T block: dims [128 mb, 128 mb + 128), entries [16 ks, 16 ks + 16), MN-major
          const uint64_t ad = ptx::smem_desc(sK + (2 * ks) * 8192 + (2 * mb) * 1024, 1024, 8192, 2);
          ptx::tc_mma_bf16(tmem + kColO + mb * NH, ad, bhi, id_pv, acc0);
          if (!f16c) ptx::tc_mma_bf16(tmem + kColO + mb * NH, ad, blo, id_pv, 1u);
        } else {
          const uint64_t ones = ptx::smem_desc(f16c ? sOnes16 : sOnes, 0, 0, 0);
          ptx::tc_mma_bf16(tmem + kColO + 4 * NH, ones, bhi, id_qk, acc0);
          if (!f16c) ptx::tc_mma_bf16(tmem + kColO + 4 * NH, ones, blo, id_qk, 1u);
        }
      }
      ptx::tc_commit(&bar_o);
    }
    if (!ptx::mbar_wait(&bar_o, phase)) { record_error(A.status, CSA2_ERR_TIMEOUT); bad_sh = 1; }
    ptx::tc_fence_after();
    phase ^= 1;
    if (wp) {
      if (t < NH) m_ref[t] = -INFINITY;               // the real pass starts afresh (any_chunk stays false)
    } else {
      any_chunk = true;
    }
    __syncthreads();
    if (bad_sh) break;
  }

  if (bad_sh) {
    // A wait ran out: before the tensor memory is read and given back, every
    // MMA this CTA issued must have finished.  Each issuer commits once more
    // (the commit completes when all of that thread's earlier MMAs have) and
    // all threads wait on it, bounded.
    if (lane == 0 && warp < 5) ptx::tc_commit(&bar_drain);
    ptx::mbar_wait(&bar_drain, 0);
    ptx::tc_fence_after();
  }
  if (!waited && !HAND) {
    griddep_wait();
    griddep_launch();
  }
  // ---------------------------------------------------------- read-out
  {
    // one split: the CTA finishes the output; else it writes its partials
    // (always so with the handoff: a query's candidates take five chunks)
    const bool one_split = !HAND && A.nsplit == 1;
    const int quarter = warp & 3;
    const int pos = pos_sh;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    for (int blk = warp >> 2; blk < 4; blk += 2) {
      const int d = blk * 128 + quarter * 32 + lane;   // TMEM lane = dim within block
      float rc = 1.f, rs = 0.f;                        // cos t, sin t of the pair holding d
      if (d >= kRopeOff && one_split) rope_cs(A.inv_freq[(d - kRopeOff) >> 1], pos, rc, rs);
#pragma unroll
      for (int half = 0; half < NH / 32; half++) {
        uint32_t r[32], lr[32];
        if (any_chunk) {
          ptx::tmem_ld_32x32b_x32(lane_base + kColO + blk * NH + half * 32, r);
          ptx::tmem_ld_32x32b_x32(lane_base + kColO + 4 * NH + half * 32, lr);
          ptx::tmem_wait_ld();
        } else {
#pragma unroll
          for (int i = 0; i < 32; i++) r[i] = lr[i] = 0u;
        }
        if (one_split) {
#pragma unroll
          for (int i = 0; i < 32; i++) {
            const int h = h0 + half * 32 + i;
            const float l = __uint_as_float(lr[i]);
            float x = l > 0.f ? __fdividef(__uint_as_float(r[i]), l) : 0.f;   // (within 2 ulp)
            if (d >= kRopeOff) {
              // rotate the pair (a, b) = (o[d & ~1], o[d | 1]) by -pos:
              // a' = a c + b s,  b' = -a s + b c; the partner lives in the next lane
              const float y = __shfl_xor_sync(0xFFFFFFFFu, x, 1);
              x = (d & 1) ? (x * rc - y * rs) : (x * rc + y * rs);
            }
            const int64_t off = ((int64_t)qi * kHeads + h) * kDim + d;
            if (A.out_f32) static_cast<float *>(A.out)[off] = x;
            else reinterpret_cast<__nv_bfloat16 *>(A.out)[off] = __float2bfloat16_rn(x);
          }
        } else {
          // partial O[head][dim]: for each head the warp writes one 128-B line
          float *P = A.part + ((int64_t)qi * A.nsplit + split) * kHeads * kDim;
#pragma unroll
          for (int i = 0; i < 32; i++) P[(h0 + half * 32 + i) * kDim + d] = __uint_as_float(r[i]);
          if (blk == (warp >> 2) && quarter == 0 && lane == 0 && warp < 4) {
            float *ml = A.part_ml + ((int64_t)qi * A.nsplit + split) * 2 * kHeads;
#pragma unroll
            for (int i = 0; i < 32; i++) ml[kHeads + h0 + half * 32 + i] = __uint_as_float(lr[i]);
          }
        }
      }
    }
    if (!one_split && t < NH) {
      // (the denominators, replicated over all 128 lanes, were written by lane 0 of warp 0)
      float *ml = A.part_ml + ((int64_t)qi * A.nsplit + split) * 2 * kHeads;
      ml[h0 + t] = any_chunk ? m_ref[t] : -INFINITY;
    }
  }
  // handoff: this grid completes after the selection grid ahead of it, as
  // without it (the grids that follow rely on that)
  if (HAND) griddep_wait();
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kAttTmemCols);
  }
}

// Combine the split partials of one query over 32 output dims: grid
// (kDim / 32, n_q), 256 threads, thread = (head, 8 consecutive dims).
// Weights w_s = 2^(m_s - max_s m_s) per head, O = sum_s w_s O_s / sum_s w_s l_s,
// then the RoPE pairs are rotated by -pos.  The rotation angles (fp64 range
// reduction) depend on pos alone, an input of the call that no grid of it
// writes, so they are computed before the wait, while the attention runs.
constexpr int kMaxSplit = 8;
__global__ void __launch_bounds__(256) attn_tc_merge_kernel(AttnTcArgs A) {
  const int qi = blockIdx.y, t = threadIdx.x, ns = A.nsplit;
  const int h = t >> 2, d = blockIdx.x * 32 + (t & 3) * 8;
  float rc[4] = {1.f, 1.f, 1.f, 1.f}, rsn[4] = {0.f, 0.f, 0.f, 0.f};
  if (d >= kRopeOff) {
    const int pos = __ldg(A.pos + qi);
#pragma unroll
    for (int j = 0; j < 4; j++) rope_cs(A.inv_freq[(d + 2 * j - kRopeOff) >> 1], pos, rc[j], rsn[j]);
  }
  griddep_wait();
  griddep_launch();
  const float *ml = A.part_ml + (int64_t)qi * ns * 2 * kHeads;
  float4 v[kMaxSplit][2];                            // every split's loads in flight at once
  float m[kMaxSplit], l[kMaxSplit];
#pragma unroll
  for (int s = 0; s < kMaxSplit; s++) {
    if (s < ns) {
      const float4 *src = reinterpret_cast<const float4 *>(A.part + (((int64_t)qi * ns + s) * kHeads + h) * kDim + d);
      v[s][0] = __ldcg(src);
      v[s][1] = __ldcg(src + 1);
      m[s] = __ldcg(ml + s * 2 * kHeads + h);
      l[s] = __ldcg(ml + s * 2 * kHeads + kHeads + h);
    }
  }
  float M = -INFINITY;
#pragma unroll
  for (int s = 0; s < kMaxSplit; s++)
    if (s < ns) M = fmaxf(M, m[s]);
  float L = 0.f, y[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int s = 0; s < kMaxSplit; s++) {
    if (s < ns && M != -INFINITY && m[s] != -INFINITY) {
      const float w = exp2f(m[s] - M);
      L += w * l[s];
      const float e[8] = {v[s][0].x, v[s][0].y, v[s][0].z, v[s][0].w, v[s][1].x, v[s][1].y, v[s][1].z, v[s][1].w};
#pragma unroll
      for (int j = 0; j < 8; j++) y[j] += w * e[j];
    }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
  for (int j = 0; j < 8; j++) y[j] *= inv;
  if (d >= kRopeOff) {
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
      const float c = rc[j >> 1], sn = rsn[j >> 1], a = y[j], b = y[j + 1];
      y[j] = a * c + b * sn;
      y[j + 1] = -a * sn + b * c;
    }
  }
  const int64_t off = ((int64_t)qi * kHeads + h) * kDim + d;
  if (A.out_f32) {
    float4 *o = reinterpret_cast<float4 *>(static_cast<float *>(A.out) + off);
    o[0] = make_float4(y[0], y[1], y[2], y[3]);
    o[1] = make_float4(y[4], y[5], y[6], y[7]);
  } else {
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; j++) {
      const __nv_bfloat162 b2 = __floats2bfloat162_rn(y[2 * j], y[2 * j + 1]);
      w[j] = *reinterpret_cast<const uint32_t *>(&b2);
    }
    *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(A.out) + off) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

static int attn_chunks(int sel_stride) { return (sel_stride + kSwa + kTcChunk - 1) / kTcChunk; }

// How the chunks of a query are spread over CTAs (one CTA per SM): one chunk
// per CTA while the CTAs whose chunks hold selected entries fit one wave on the
// current device's n_sm SMs (the window-only chunks are placed first and run
// while the selection finishes); else contiguous runs of chunks, at least one
// CTA per query.  With settled inputs, where the chunks of selected entries
// alone, in runs of fewer chunks, fit one wave (64 queries: two runs of two
// instead of a run of three beside one of two), the last split also takes the
// window-only chunk and runs it first, while the selection finishes.
struct AttnPlan {
  int nsplit, cps, hs;   // splits of a query's chunks, chunks per split, CTAs per chunk (head halves)
  int merge;             // the last split also runs the window-only chunks (first)
};
static AttnPlan attn_plan(int n_q, int sel_stride, int n_sm, bool settled = false) {
  const int chunks = attn_chunks(sel_stride);
  const int sel_ch = (sel_stride + kTcChunk - 1) / kTcChunk;
  if (n_q * sel_ch <= n_sm) {
    // one chunk per CTA; two CTAs per chunk (32 heads each) while all of them
    // fit one wave: the gather is repeated, the rest of the chunk is halved
    return AttnPlan{chunks, 1, n_q * chunks * 2 <= n_sm ? 2 : 1, 0};
  }
  const int ns = std::max(1, std::min(chunks, n_sm / n_q));
  const int cps = (chunks + ns - 1) / ns;
  if (settled && sel_stride % kTcChunk == 0 && chunks > sel_ch) {
    const int ns_s = std::max(1, std::min(sel_ch, n_sm / n_q));
    const int cps_s = (sel_ch + ns_s - 1) / ns_s;
    const int nsp = (sel_ch + cps_s - 1) / cps_s;
    if (cps_s < cps && n_q * nsp <= n_sm) return AttnPlan{nsp, cps_s, 1, 1};
  }
  return AttnPlan{(chunks + cps - 1) / cps, cps, 1, 0};
}

int attn_ctas(int n_q, int sel_stride, bool settled) {
  const AttnPlan p = attn_plan(n_q, sel_stride, device_sm_count(current_device()), settled);
  return n_q * p.nsplit * p.hs;
}

bool attn_handoff_fits(int n_q) {
  return attn_plan(n_q, kHandCap, device_sm_count(current_device())).cps == 1;
}

size_t attn_workspace_bytes(int n_q, int sel_stride, bool settled) {
  const AttnPlan p = attn_plan(n_q, sel_stride, device_sm_count(current_device()), settled);
  if (p.nsplit == 1) return 0;
  return (size_t)n_q * p.nsplit * (kHeads * kDim + 2 * kHeads) * sizeof(float);
}

cudaError_t launch_attn_tc(const void *q, const void *kv, int64_t n_max, int n_seq, const int32_t *sel, int sel_stride,
                           const void *swa, int swa_cap, const int32_t *q_seq, const int32_t *pos,
                           const int32_t *swa_first, const int32_t *swa_cnt, int n_q, void *out, int out_dtype,
                           float sm_scale, double rope_base, void *ws, int *status, cudaStream_t st,
                           bool inputs_settled, int ahead_ctas, const Handoff *hand) {
  AttnTcArgs A;
  A.settled = inputs_settled ? 1 : 0;
  A.q = static_cast<const uint16_t *>(q);
  A.kv = static_cast<const uint8_t *>(kv);
  A.n_max = n_max;
  A.n_seq = n_seq;
  A.sel = sel;
  A.sel_stride = sel_stride;
  A.n_sel = hand != nullptr ? kHandCap : sel_stride;
  A.hflag = hand != nullptr ? hand->flag : nullptr;
  A.hcand = hand != nullptr ? hand->cand : nullptr;
  A.hparts = hand != nullptr ? hand->parts : 0;
  A.swa = static_cast<const uint8_t *>(swa);
  A.swa_cap = swa_cap;
  A.q_seq = q_seq;
  A.pos = pos;
  A.swa_first = swa_first;
  A.swa_cnt = swa_cnt;
  A.out = out;
  A.out_f32 = out_dtype == CSA2_OUT_F32;
  A.scale_log2 = sm_scale * 1.4426950408889634f;
  for (int i = 0; i < kRopeDim / 2; i++) A.inv_freq[i] = pow(rope_base, -2.0 * i / (double)kRopeDim);
  const int dev = current_device();
  const int n_sm = device_sm_count(dev);
  const AttnPlan plan = attn_plan(n_q, A.n_sel, n_sm, inputs_settled);
  A.nsplit = plan.nsplit;
  A.chunks_per_split = plan.cps;
  A.merge_tail = plan.merge;
  A.hsplit = plan.hs;
  A.part = static_cast<float *>(ws);
  A.part_ml = A.part + (size_t)n_q * A.nsplit * kHeads * kDim;
  A.status = status;
  static std::atomic<int> attr_done[kMaxDevices];
  cudaError_t e = once_per_device(attr_done, dev, [&] {
    const cudaError_t es[4] = {
        cudaFuncSetAttribute(attn_tc_kernel<64, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmAlloc),
        cudaFuncSetAttribute(attn_tc_kernel<32, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmAlloc),
        cudaFuncSetAttribute(attn_tc_kernel<64, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmAlloc),
        cudaFuncSetAttribute(attn_tc_kernel<32, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmAlloc)};
    for (cudaError_t x : es)
      if (x != cudaSuccess) return x;
    return cudaSuccess;
  });
  if (e != cudaSuccess) return e;
  // the warm-up pays only where every CTA is resident while the grid ahead runs
  const int n_ctas = n_q * plan.nsplit * plan.hs;
  A.warm = inputs_settled && plan.cps == 1 && ahead_ctas >= 0 && ahead_ctas + n_ctas <= n_sm ? 1 : 0;
  const dim3 grid(n_q, A.nsplit * plan.hs);
  const bool h = A.hflag != nullptr;
  e = plan.hs == 2 ? (h ? launch_pdl(attn_tc_kernel<32, true>, grid, dim3(kTcThreads), kSmAlloc, st, 1u, A)
                        : launch_pdl(attn_tc_kernel<32, false>, grid, dim3(kTcThreads), kSmAlloc, st, 1u, A))
                   : (h ? launch_pdl(attn_tc_kernel<64, true>, grid, dim3(kTcThreads), kSmAlloc, st, 1u, A)
                        : launch_pdl(attn_tc_kernel<64, false>, grid, dim3(kTcThreads), kSmAlloc, st, 1u, A));
  if (e != cudaSuccess || A.nsplit == 1) return e;
  return launch_pdl(attn_tc_merge_kernel, dim3(kDim / 32, n_q), dim3(256), 0, st, 1u, A);
}

}  // namespace csa2
