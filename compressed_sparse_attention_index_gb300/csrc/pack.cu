// Cache-write kernels: bf16 rows -> FP4 / FP8 cache records (csa2_fp4_pack).
//
// Formats ("An infra-oriented diagram of the DeepSeek-V4.1-Flash architecture",
// reading notes and section "The KV cache"):
//   KV  : 512 FP4 E2M1 + one E4M3 scale per 16 channels   (288 B)
//   IDX : 128 FP4 E2M1 + one E8M0 scale per 32 channels    (68 B, two planes)
//   SWA : 512 E4M3 + one E8M0 scale per 32 channels        (528 B)
// m=2 entries pool two tokens with a per-channel softmax gate (same notes).
//
// Rounding is done by the hardware converters (cvt.rn.satfinite to e2m1x2 /
// e4m3x2: nearest-even, saturating).  Each converter input is a correctly
// rounded fp32 quotient or an exact power-of-two scaling of a bf16 value, and a
// tie of the exact quotient cannot move under fp32 rounding (the quotient of an
// 8-bit by a 4-bit significand is either exact or at least 2^-12 relative away
// from every tie point), so the codes equal those of the exact real quotient.
//
// All three kernels are HBM-bound streams: one warp per row (KV, SWA) or eight
// lanes per row (IDX), 16-B vector loads of the bf16 row, 8- or 16-B stores.
#include <cuda_bf16.h>

#include "common.cuh"
#include "launch.cuh"

namespace csa2 {

// Eight floats -> four bytes of E2M1 pairs; byte i = code(v[2i+1]) << 4 | code(v[2i]).
__device__ __forceinline__ uint32_t cvt_e2m1x8(float v0, float v1, float v2, float v3, float v4, float v5,
                                               float v6, float v7) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(v0), "f"(v1), "f"(v2), "f"(v3), "f"(v4), "f"(v5), "f"(v6), "f"(v7));
  return r;
}

__device__ __forceinline__ uint32_t cvt_e4m3x2(float hi, float lo) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return (uint32_t)r;
}

// fp64 -> bf16 bits, one rounding (nearest-even), for finite values of bf16 range.
__device__ __forceinline__ uint32_t bf16_from_f64(double v) {
  unsigned long long u = (unsigned long long)__double_as_longlong(v);
  uint32_t sign = (uint32_t)(u >> 63) << 15;
  unsigned long long a = u & 0x7FFFFFFFFFFFFFFFull;
  if (a == 0) return sign;
  int ex = (int)(a >> 52) - 1023;                 // unbiased exponent of a normal double
  uint32_t bits;
  if (ex >= -126) {
    // keep 7 of the 52 fraction bits: round away 45 bits, nearest-even
    unsigned long long r = a + ((1ull << 44) - 1) + ((a >> 45) & 1ull);
    r >>= 45;                                     // (exponent_d << 7) | frac7, may carry
    int e_bf = (int)(r >> 7) - 1023 + 127;
    bits = ((uint32_t)e_bf << 7) | (uint32_t)(r & 0x7F);
  } else {
    // bf16 subnormal: multiple of 2^-133; |v| < 2^-126 so the count is <= 128
    double m = fabs(v) * 0x1p133;                 // exact power-of-two scaling
    bits = (uint32_t)__double2ull_rn(m);          // nearest-even to an integer
  }
  return sign | bits;
}

// ------------------------------------------------------------------ KV (S1)
// One warp per output row; lane g packs channels [16g, 16g+16).  pooled
// (M = 2, optional): the pooled bf16 latents as well, [rows_out][512].
//
// M = 2: gated pooling of tokens 2*row and 2*row+1, rounded once to bf16: the
// exact value's rounding.  With the larger logit's token t_m, the other t_o,
// e = exp(-|z_a - z_b|) and s = e / (1 + e), the value is t_m + (t_o - t_m) s.
// fp32 first, one FMA: expf is within 2 ulps, the argument, 1 + e, the
// quotient and t_o - t_m round once each, so its error is below
// |t_o - t_m| (1.75 s 2^-22 + 0.28 2^-24) + 2^-24 |v| (s |dz| <= 0.28); with d
// twice that or more, when v - d and v + d round to the same bf16 so does the
// exact value.  The rest (about one element in a thousand, near a rounding
// boundary) are recomputed in fp64 as (e_a t_a + e_b t_b) / (e_a + e_b).  fp64
// is slow on this part, and a warp recomputing an element stalls its row: with
// a fix-up list (csa2_build_cache), a lane with such elements appends its
// (row, lane) and leaves, and a second grid recomputes those 16-channel blocks
// densely, one per thread; without one (or once the list is full), the warp's
// lanes recompute theirs together, each taking its next element.

// The 16 channels of lane block g of output row `row`: the fp32 values (x,
// rounded down where ambiguous) and the mask of channels to recompute, with
// the inputs the recomputation needs.
struct Kv2Block {
  float x[16], t0[16], t1[16], za[16], zb[16];
  uint32_t redo;
};
__device__ __forceinline__ void kv2_block(const uint16_t *__restrict__ src, const float *__restrict__ gate,
                                          int64_t row, int g, Kv2Block &B) {
  const uint4 *p0 = reinterpret_cast<const uint4 *>(src + (2 * row) * kDim + g * 16);
  const uint4 *p1 = reinterpret_cast<const uint4 *>(src + (2 * row + 1) * kDim + g * 16);
  const float *z0 = gate + (2 * row) * kDim + g * 16;
  const float *z1 = gate + (2 * row + 1) * kDim + g * 16;
  uint4 a0 = __ldg(p0), b0 = __ldg(p0 + 1), a1 = __ldg(p1), b1 = __ldg(p1 + 1);
  uint32_t w0[8] = {a0.x, a0.y, a0.z, a0.w, b0.x, b0.y, b0.z, b0.w};
  uint32_t w1[8] = {a1.x, a1.y, a1.z, a1.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
  for (int v = 0; v < 4; v++) {                     // the logits, 16-B loads
    const float4 ga = __ldg(reinterpret_cast<const float4 *>(z0) + v);
    const float4 gb = __ldg(reinterpret_cast<const float4 *>(z1) + v);
    B.za[4 * v] = ga.x; B.za[4 * v + 1] = ga.y; B.za[4 * v + 2] = ga.z; B.za[4 * v + 3] = ga.w;
    B.zb[4 * v] = gb.x; B.zb[4 * v + 1] = gb.y; B.zb[4 * v + 2] = gb.z; B.zb[4 * v + 3] = gb.w;
  }
  B.redo = 0u;
#pragma unroll
  for (int i = 0; i < 16; i++) {
    B.t0[i] = (i & 1) ? bf16_hi(w0[i >> 1]) : bf16_lo(w0[i >> 1]);
    B.t1[i] = (i & 1) ? bf16_hi(w1[i >> 1]) : bf16_lo(w1[i >> 1]);
    const float fa = B.za[i], fb = B.zb[i];
    const float tm = fa >= fb ? B.t0[i] : B.t1[i], to = fa >= fb ? B.t1[i] : B.t0[i];
    const float e = expf(-fabsf(fa - fb));
    const float sg = e / (1.0f + e);
    const float dl = to - tm;
    const float vf = fmaf(dl, sg, tm);
    const float d = fabsf(dl) * fmaf(sg, 0x1p-20f, 0x1p-24f) + fabsf(vf) * 0x1p-23f;
    const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(vf - d));
    const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(vf + d));
    B.x[i] = __uint_as_float(lo << 16);
    B.redo |= (lo != hi ? 1u : 0u) << i;
  }
}

// channel c of the block, recomputed in fp64 and rounded once to bf16
__device__ __forceinline__ void kv2_recompute(Kv2Block &B, int c) {
  float t0 = 0.f, t1 = 0.f, fa = 0.f, fb = 0.f;
#pragma unroll
  for (int i = 0; i < 16; i++)
    if (i == c) { t0 = B.t0[i]; t1 = B.t1[i]; fa = B.za[i]; fb = B.zb[i]; }
  const double za = (double)fa, zb = (double)fb;
  const double e = exp(-fabs(za - zb));
  const double v = za >= zb ? ((double)t0 + e * (double)t1) / (1.0 + e) : (e * (double)t0 + (double)t1) / (e + 1.0);
  const float xv = __uint_as_float(bf16_from_f64(v) << 16);
#pragma unroll
  for (int i = 0; i < 16; i++)
    if (i == c) B.x[i] = xv;
}

// the pooled latents of the block (bf16, 32 B)
__device__ __forceinline__ void kv2_store_pooled(const float (&x)[16], uint16_t *__restrict__ pooled, int64_t row,
                                                 int g) {
  uint32_t b[8];
#pragma unroll
  for (int i = 0; i < 8; i++) b[i] = (__float_as_uint(x[2 * i]) >> 16) | (__float_as_uint(x[2 * i + 1]) & 0xFFFF0000u);
  uint4 *po = reinterpret_cast<uint4 *>(pooled + row * kDim + g * 16);
  po[0] = make_uint4(b[0], b[1], b[2], b[3]);
  po[1] = make_uint4(b[4], b[5], b[6], b[7]);
}

// the block's 16 channels -> one E4M3 scale and 8 bytes of E2M1 codes of the
// record of `row`
__device__ __forceinline__ void kv_store_record(const float (&x)[16], uint8_t *__restrict__ dst, int64_t row, int g) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; i++) amax = fmaxf(amax, fabsf(x[i]));
  const uint32_t sc = cvt_e4m3x2(0.f, __fdiv_rn(amax, 6.0f)) & 0xFFu;
  const float s = e4m3_to_float(sc);
  uint32_t nib[2] = {0u, 0u};
  if (s != 0.f) {
    float y[16];
#pragma unroll
    for (int i = 0; i < 16; i++) y[i] = __fdiv_rn(x[i], s);
    nib[0] = cvt_e2m1x8(y[0], y[1], y[2], y[3], y[4], y[5], y[6], y[7]);
    nib[1] = cvt_e2m1x8(y[8], y[9], y[10], y[11], y[12], y[13], y[14], y[15]);
  }
  uint8_t *rec = dst + row * kKvBytes;
  *reinterpret_cast<uint2 *>(rec + g * 8) = make_uint2(nib[0], nib[1]);
  rec[256 + g] = (uint8_t)sc;
}

template <int M>
__global__ void __launch_bounds__(256) pack_kv_kernel(const uint16_t *__restrict__ src,
                                                       const float *__restrict__ gate, int64_t rows_out,
                                                       uint8_t *__restrict__ dst, uint16_t *__restrict__ pooled,
                                                       KvFix F) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= rows_out) return;
  if (M == 1) {
    float x[16];
    const uint4 *p = reinterpret_cast<const uint4 *>(src + row * kDim + lane * 16);
    uint4 a = __ldg(p), b = __ldg(p + 1);
    uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; i++) { x[2 * i] = bf16_lo(w[i]); x[2 * i + 1] = bf16_hi(w[i]); }
    kv_store_record(x, dst, row, lane);
  } else {
    Kv2Block B;
    kv2_block(src, gate, row, lane, B);
    bool deferred = false;
    if (F.list != nullptr && B.redo != 0u) {
      const uint32_t i = atomicAdd(F.cnt, 1u);
      if (i < F.cap) {
        F.list[i] = (uint32_t)row * 32u + (uint32_t)lane;
        deferred = true;
        B.redo = 0u;
      }
    }
    while (__any_sync(0xFFFFFFFFu, B.redo != 0u)) {
      if (B.redo != 0u) {
        const int c = __ffs(B.redo) - 1;
        B.redo &= B.redo - 1u;
        kv2_recompute(B, c);
      }
    }
    if (deferred) return;                            // (the fix-up grid writes this block)
    if (pooled != nullptr) kv2_store_pooled(B.x, pooled, row, lane);
    kv_store_record(B.x, dst, row, lane);
  }
}

// The deferred blocks of one pack_kv_kernel<2> launch, one per thread; then
// the next launch's list count is zeroed (none of this grid reads it).
__global__ void __launch_bounds__(256) pack_kv2_fix_kernel(const uint16_t *__restrict__ src,
                                                            const float *__restrict__ gate, uint8_t *__restrict__ dst,
                                                            uint16_t *__restrict__ pooled, KvFix F) {
  const uint32_t n = min(*F.cnt, F.cap);
  for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    const uint32_t e = F.list[i];
    const int64_t row = e >> 5;
    const int g = (int)(e & 31u);
    Kv2Block B;
    kv2_block(src, gate, row, g, B);
    while (B.redo != 0u) {
      const int c = __ffs(B.redo) - 1;
      B.redo &= B.redo - 1u;
      kv2_recompute(B, c);
    }
    if (pooled != nullptr) kv2_store_pooled(B.x, pooled, row, g);
    kv_store_record(B.x, dst, row, g);
  }
  if (blockIdx.x == 0 && threadIdx.x == 0 && F.next_cnt != nullptr) *F.next_cnt = 0u;
}

// smallest e with lim * 2^e >= amax (amax > 0), for lim = 1.5 * 2^p, 1.75 * 2^p
__device__ __forceinline__ int pow2_exp_fp4(float amax) {   // lim = 6 = 1.5 * 2^2
  int ex;
  frexpf(amax, &ex);                     // amax in [2^(ex-1), 2^ex)
  int e0 = ex - 1;
  int e = (amax <= ldexpf(6.0f, e0 - 2)) ? e0 - 2 : e0 - 1;
  return max(-127, min(127, e));
}
__device__ __forceinline__ int pow2_exp_fp8(float amax) {   // lim = 448 = 1.75 * 2^8
  int ex;
  frexpf(amax, &ex);
  int e0 = ex - 1;
  int e = (amax <= ldexpf(448.0f, e0 - 8)) ? e0 - 8 : e0 - 7;
  return max(-127, min(127, e));
}

// ------------------------------------------------------------------ IDX (S2, S4)
// Eight lanes per 128-wide row; lane part p packs channels [16p, 16p+16), the
// lane pair (2g, 2g+1) shares E8M0 group g.  The nibble row is stored in the
// 64-byte swizzled order (see include/csa2.h) so that the indexer can move
// whole tiles with one bulk copy.
// The part of one thread t (row t / 8, channels 16 (t % 8) ..): HOST reads
// the row from page-locked host memory (fetched anew, not from a cache).
template <bool HOST>
__device__ __forceinline__ void pack_idx_part(const uint16_t *__restrict__ src, int64_t rows, int64_t t,
                                              uint8_t *__restrict__ nib_out, uint8_t *__restrict__ sc_out) {
  const int64_t row = t >> 3;
  const int part = (int)(t & 7);
  const bool live = row < rows;
  float x[16];
  float amax = 0.f;
  if (live) {
    const uint4 *p = reinterpret_cast<const uint4 *>(src + row * kIdxDim + part * 16);
    uint4 a = HOST ? __ldcv(p) : __ldg(p), b = HOST ? __ldcv(p + 1) : __ldg(p + 1);
    uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; i++) { x[2 * i] = bf16_lo(w[i]); x[2 * i + 1] = bf16_hi(w[i]); }
#pragma unroll
    for (int i = 0; i < 16; i++) amax = fmaxf(amax, fabsf(x[i]));
  }
  amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
  if (!live) return;
  uint32_t scale_byte = 0, nib[2] = {0u, 0u};
  if (amax > 0.f) {
    const int e = pow2_exp_fp4(amax);
    scale_byte = (uint32_t)(e + 127);
    float y[16];
#pragma unroll
    for (int i = 0; i < 16; i++) y[i] = ldexpf(x[i], -e);
    nib[0] = cvt_e2m1x8(y[0], y[1], y[2], y[3], y[4], y[5], y[6], y[7]);
    nib[1] = cvt_e2m1x8(y[8], y[9], y[10], y[11], y[12], y[13], y[14], y[15]);
  }
  // 64-byte-swizzled row: 16-B chunk c of the row at address A goes to chunk
  // c ^ ((A >> 7) & 3), the order the tensor-core operand reads it in
  uint8_t *rowp = nib_out + row * kIdxNibBytes;
  const uint32_t chunk = ((uint32_t)part >> 1) ^ (uint32_t)((reinterpret_cast<uintptr_t>(rowp) >> 7) & 3u);
  *reinterpret_cast<uint2 *>(rowp + chunk * 16 + (part & 1) * 8) = make_uint2(nib[0], nib[1]);
  if ((part & 1) == 0) sc_out[row * kIdxScaleBytes + (part >> 1)] = (uint8_t)scale_byte;
}

__global__ void __launch_bounds__(256) pack_idx_kernel(const uint16_t *__restrict__ src, int64_t rows,
                                                        uint8_t *__restrict__ nib_out,
                                                        uint8_t *__restrict__ sc_out) {
  pack_idx_part<false>(src, rows, (int64_t)blockIdx.x * blockDim.x + threadIdx.x, nib_out, sc_out);
}

// ------------------------------------------------------------------ host-input staging
// csa2_decode_host's per-step inputs read straight from page-locked host
// memory (device-accessible at the same address under unified addressing),
// in one grid instead of one copy per buffer plus the packing kernel: the
// first pack_ctas CTAs pack the indexer query (as pack_idx_kernel), the rest
// copy the other segments (16-B units; 4-B units where a segment's size or
// address is not a multiple of 16).  Every thread loads its first unit before
// the grid-dependency wait and stores it after.
__global__ void __launch_bounds__(256) stage_host_inputs_kernel(StageIn S) {
  if ((int)blockIdx.x < S.pack_ctas) {
    griddep_wait();
    pack_idx_part<true>(S.qidx, S.qidx_rows, (int64_t)blockIdx.x * blockDim.x + threadIdx.x, S.qnib, S.qsc);
    return;
  }
  const int64_t total = S.units[0] + S.units[1] + S.units[2];
  const int64_t stride = (int64_t)(gridDim.x - S.pack_ctas) * blockDim.x;
  auto locate = [&](int64_t i, int &k, int64_t &u) {
    k = 0;
    u = i;
    while (k < 2 && u >= S.units[k]) { u -= S.units[k]; k++; }
  };
  auto load = [&](int k, int64_t u) -> uint4 {
    if (S.wide[k]) return __ldcv(static_cast<const uint4 *>(S.src[k]) + u);
    return make_uint4(__ldcv(static_cast<const unsigned int *>(S.src[k]) + u), 0u, 0u, 0u);
  };
  auto store = [&](int k, int64_t u, uint4 v) {
    if (S.wide[k]) static_cast<uint4 *>(S.dst[k])[u] = v;
    else static_cast<unsigned int *>(S.dst[k])[u] = v.x;
  };
  int64_t i = (int64_t)(blockIdx.x - S.pack_ctas) * blockDim.x + threadIdx.x;
  int k0 = 0;
  int64_t u0 = 0;
  uint4 v0 = make_uint4(0u, 0u, 0u, 0u);
  if (i < total) {
    locate(i, k0, u0);
    v0 = load(k0, u0);
  }
  griddep_wait();
  if (i < total) store(k0, u0, v0);
  for (i += stride; i < total; i += stride) {
    int k;
    int64_t u;
    locate(i, k, u);
    store(k, u, load(k, u));
  }
}

// ------------------------------------------------------------------ SWA (S3)
// One warp per row; lane l packs channels [16l, 16l+16), lanes (2g, 2g+1) share group g.
__global__ void __launch_bounds__(256) pack_swa_kernel(const uint16_t *__restrict__ src, int64_t rows,
                                                        uint8_t *__restrict__ dst) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= rows) return;
  const uint4 *p = reinterpret_cast<const uint4 *>(src + row * kDim + lane * 16);
  uint4 a = __ldg(p), b = __ldg(p + 1);
  uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  float x[16];
#pragma unroll
  for (int i = 0; i < 8; i++) { x[2 * i] = bf16_lo(w[i]); x[2 * i + 1] = bf16_hi(w[i]); }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; i++) amax = fmaxf(amax, fabsf(x[i]));
  amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
  uint32_t scale_byte = 0, v[4] = {0u, 0u, 0u, 0u};
  if (amax > 0.f) {
    const int e = pow2_exp_fp8(amax);
    scale_byte = (uint32_t)(e + 127);
#pragma unroll
    for (int i = 0; i < 8; i++) {
      uint32_t two = cvt_e4m3x2(ldexpf(x[2 * i + 1], -e), ldexpf(x[2 * i], -e));
      v[i >> 1] |= two << (16 * (i & 1));
    }
  }
  uint8_t *rec = dst + row * kSwaBytes;
  *reinterpret_cast<uint4 *>(rec + lane * 16) = make_uint4(v[0], v[1], v[2], v[3]);
  if ((lane & 1) == 0) rec[512 + (lane >> 1)] = (uint8_t)scale_byte;
}

// ------------------------------------------------------------------ launchers
cudaError_t launch_pack(int kind, const void *src, int64_t rows, int m, const float *gate, void *dst,
                        void *dst_scales, cudaStream_t st, void *pooled, const KvFix *fix) {
  const uint16_t *s = static_cast<const uint16_t *>(src);
  if (kind == CSA2_KV_NVFP4) {
    const int64_t out_rows = rows / m;
    const int64_t blocks = (out_rows + 7) / 8;
    const KvFix none = {nullptr, nullptr, 0u, nullptr};
    if (m == 1) {
      pack_kv_kernel<1><<<(unsigned)blocks, 256, 0, st>>>(s, nullptr, out_rows, (uint8_t *)dst, nullptr, none);
    } else {
      const KvFix F = fix != nullptr && out_rows * 32 < ((int64_t)1 << 32) ? *fix : none;
      pack_kv_kernel<2><<<(unsigned)blocks, 256, 0, st>>>(s, gate, out_rows, (uint8_t *)dst,
                                                          static_cast<uint16_t *>(pooled), F);
      if (F.list != nullptr) {
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        pack_kv2_fix_kernel<<<(unsigned)(2 * device_sm_count(current_device())), 256, 0, st>>>(
            s, gate, (uint8_t *)dst, static_cast<uint16_t *>(pooled), F);
      }
    }
  } else if (kind == CSA2_IDX_MXFP4) {
    const int64_t blocks = (rows * 8 + 255) / 256;
    pack_idx_kernel<<<(unsigned)blocks, 256, 0, st>>>(s, rows, (uint8_t *)dst, (uint8_t *)dst_scales);
  } else {
    const int64_t blocks = (rows + 7) / 8;
    pack_swa_kernel<<<(unsigned)blocks, 256, 0, st>>>(s, rows, (uint8_t *)dst);
  }
  return cudaGetLastError();
}

cudaError_t launch_stage_host_inputs(StageIn S, cudaStream_t st) {
  S.pack_ctas = (int)((S.qidx_rows * 8 + 255) / 256);
  int64_t units = 0;
  for (int k = 0; k < 3; k++) units += S.units[k];
  const int64_t copy_ctas = (units + 255) / 256;
  const int64_t cap = 8 * (int64_t)device_sm_count(current_device());
  const int64_t grid = S.pack_ctas + (copy_ctas < cap ? copy_ctas : cap);
  return launch_pdl(stage_host_inputs_kernel, dim3((unsigned)grid), dim3(256), 0, st, 1u, S);
}

}  // namespace csa2
