// Device twin of gen/inputs.py: the same counter-based draws, bit for bit.
// Integer hashing (SplitMix64 output function), a table lookup for normal
// variates (the table bytes come from the host), a Feistel permutation for
// Zipf ranks, and correctly rounded fp32 multiply / divide.  None of the CSA2
// method's arithmetic is here.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ull;

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ uint16_t normal_at(const uint16_t *table, uint64_t key, uint64_t ctr) {
  return table[mix64(key + (ctr + 1) * kGolden) >> 44];
}

__device__ __forceinline__ uint16_t f32_to_bf16_rne(float x) {
  const uint32_t b = __float_as_uint(x);
  return (uint16_t)((b + 0x7FFFu + ((b >> 16) & 1u)) >> 16);
}

__device__ __forceinline__ uint64_t feistel(uint64_t x, uint64_t key, int bits) {
  const int half = bits / 2;
  const uint64_t mask = (1ull << half) - 1;
  uint64_t L = (x >> half) & mask, R = x & mask;
  for (int r = 0; r < 4; r++) {
    const uint64_t f = mix64(key ^ ((uint64_t)r << 56) ^ R) & mask;
    const uint64_t nl = R;
    R = L ^ f;
    L = nl;
  }
  return (L << half) | R;
}

__global__ void normal_kernel(const uint16_t *table, uint64_t key, int64_t row0, int64_t nrows, int ncols,
                              uint16_t *out) {
  const int64_t n = nrows * ncols;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    out[i] = normal_at(table, key, (uint64_t)(row0 * ncols + i));
  }
}

__global__ void zipf_keys_kernel(const uint16_t *table, uint64_t key_normal, uint64_t key_perm, int64_t n_entries,
                                 int bits, int64_t row0, int64_t nrows, int ncols, uint16_t *out, int *walk_fail) {
  const int64_t n = nrows * ncols;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = row0 + i / ncols;
    uint64_t x = feistel((uint64_t)r, key_perm, bits);
    int it = 0;
    while (x >= (uint64_t)n_entries && it < 100000) { x = feistel(x, key_perm, bits); it++; }
    if (x >= (uint64_t)n_entries) { atomicExch(walk_fail, 1); x = 0; }
    const float g = __uint_as_float((uint32_t)normal_at(table, key_normal, (uint64_t)(r * ncols + i % ncols)) << 16);
    const float inv = __fdiv_rn(1.0f, (float)(x + 1));
    out[i] = f32_to_bf16_rne(__fmul_rn(g, inv));
  }
}

__global__ void scaled_normal_f32_kernel(const uint16_t *table, uint64_t key, int64_t row0, int64_t nrows, int ncols,
                                         float scale, float *out) {
  const int64_t n = nrows * ncols;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const float g = __uint_as_float((uint32_t)normal_at(table, key, (uint64_t)(row0 * ncols + i)) << 16);
    out[i] = __fmul_rn(g, scale);
  }
}

unsigned grid_for(int64_t n) {
  int64_t b = (n + 255) / 256;
  return (unsigned)(b > 152 * 32 ? 152 * 32 : (b < 1 ? 1 : b));
}

}  // namespace

extern "C" {

int gen_normal_bf16(const void *table, uint64_t key, int64_t row0, int64_t nrows, int ncols, void *out,
                    cudaStream_t st) {
  if (nrows <= 0) return 0;
  normal_kernel<<<grid_for(nrows * ncols), 256, 0, st>>>((const uint16_t *)table, key, row0, nrows, ncols,
                                                         (uint16_t *)out);
  return (int)cudaGetLastError();
}

int gen_zipf_keys_bf16(const void *table, uint64_t key_normal, uint64_t key_perm, int64_t n_entries, int bits,
                       int64_t row0, int64_t nrows, int ncols, void *out, int *walk_fail, cudaStream_t st) {
  if (nrows <= 0) return 0;
  zipf_keys_kernel<<<grid_for(nrows * ncols), 256, 0, st>>>((const uint16_t *)table, key_normal, key_perm, n_entries,
                                                            bits, row0, nrows, ncols, (uint16_t *)out, walk_fail);
  return (int)cudaGetLastError();
}

int gen_scaled_normal_f32(const void *table, uint64_t key, int64_t row0, int64_t nrows, int ncols, float scale,
                          void *out, cudaStream_t st) {
  if (nrows <= 0) return 0;
  scaled_normal_f32_kernel<<<grid_for(nrows * ncols), 256, 0, st>>>((const uint16_t *)table, key, row0, nrows, ncols,
                                                                    scale, (float *)out);
  return (int)cudaGetLastError();
}

}  // extern "C"
