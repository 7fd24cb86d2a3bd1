// Indexer-key projection on the 5th-generation tensor cores (csa2_index_key_proj).
//
// The indexer's 128-wide key is a 512 -> 128 projection of the latent the
// main cache stores ("An infra-oriented diagram of the DeepSeek-V4.1-Flash
// architecture", reading notes on the Full layer's global KV):
//     key[r][n] = bf16( sum_c latent[r][c] * w[n][c] )
// with bf16 latents and weights and an fp32 accumulator (tcgen05 kind::f16).
//
// Per entry the kernel reads 1 KB and writes 256 B for 256 KFLOP, below the
// GPU's FLOP/byte ridge: it is bound by HBM.  Persistent CTAs, one per SM,
// take tiles of 128 entries (the MMA's M); the 128 x 512 weights (128 KB) stay
// in shared memory as the B operand for the whole kernel, and a tile's
// latents stream through a 6-stage ring of 64-wide K slices (16 KB: 128 rows
// x 128 B), each slice four MMAs of K = 16 into the tile's TMEM accumulator
// (128 lanes x 128 columns, two accumulators so that the epilogue of one tile
// overlaps the MMAs of the next).  Both operands are K-major with the 128-byte
// swizzle: 8-row groups of 128-B rows, the 16-B chunk c of row r at c ^ (r & 7).
// Roles (384 threads): warps 0-3 load the slices (warp p: rows 32p..32p+31,
// 16-B asynchronous copies, eight lanes per 128-B slice), lane 0 of warp 4 issues the
// MMAs (warp 4 owns the tensor memory), warps 8-11 read the accumulator (one
// row per thread), round to bf16 and store.  Every wait is bounded.
#include <cuda_bf16.h>

#include "common.cuh"
#include "launch.cuh"
#include "tc_ptx.cuh"

namespace csa2 {

constexpr int kPjRows = 128;                       // entries per tile (MMA M)
constexpr int kPjIn = 512, kPjOut = 128;           // K, N
constexpr int kPjAtoms = kPjIn / 64;               // 64-wide (128-B) K slices
constexpr int kPjStages = 6;
constexpr int kPjStageBytes = kPjRows * 128;       // 16 KB
constexpr int kPjSmW = 0;                          // weights: [n/8][atom][n%8][128 B]  (128 KB)
constexpr int kPjSmA = kPjOut * kPjIn * 2;         // slices: [stage][row/8][row%8][128 B]
constexpr int kPjSmem = kPjSmA + kPjStages * kPjStageBytes;
constexpr int kPjThreads = 384;
constexpr uint32_t kPjTmemCols = 256;              // two 128-column accumulators
static_assert(kPjSmem + 1024 <= 227 * 1024, "shared memory");

__device__ __forceinline__ uint32_t pj_sw128(uint32_t r, uint32_t ch) { return r * 128u + ((ch ^ (r & 7u)) << 4); }

// kind::f16 instruction descriptor: bf16 x bf16 -> f32, M = 128, N = 128, both K-major
constexpr uint32_t kPjIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((128u >> 3) << 17) | ((128u >> 4) << 24);

__global__ void __launch_bounds__(kPjThreads, 1)
    proj_keys_kernel(const uint16_t *__restrict__ x, int64_t rows, const uint16_t *__restrict__ w,
                     uint16_t *__restrict__ out, int *status) {
  extern __shared__ __align__(1024) unsigned char pj_smem_raw[];
  unsigned char *sm = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(pj_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t full_bar[kPjStages], empty_bar[kPjStages], acc_full[2], acc_empty[2], drain_bar;
  __shared__ uint32_t tmem_sh;
  __shared__ volatile int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kPjStages; s++) {
      ptx::mbar_init(&full_bar[s], 4 * 32);        // every loading lane, when its copies have landed
      ptx::mbar_init(&empty_bar[s], 1);            // the MMAs reading the slice
    }
    for (int a = 0; a < 2; a++) {
      ptx::mbar_init(&acc_full[a], 1);
      ptx::mbar_init(&acc_empty[a], 4);            // the four epilogue warps
    }
    ptx::mbar_init(&drain_bar, 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 4) ptx::tmem_alloc(&tmem_sh, kPjTmemCols);
  griddep_wait();
  griddep_launch();
  // the weights, once, into their swizzled K-major layout
  for (int i = threadIdx.x; i < kPjOut * kPjIn / 8; i += blockDim.x) {
    const int n = i >> 6, ch = i & 63;             // 16-B chunk ch of row n (8 inputs)
    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(w) + i);
    *reinterpret_cast<uint4 *>(sm + kPjSmW + (n >> 3) * 8192 + (ch >> 3) * 1024 + pj_sw128(n & 7, ch & 7)) = v;
  }
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = tmem_sh;
  auto fail = [&]() {
    record_error(status, CSA2_ERR_TIMEOUT);
    abort_flag = 1;
  };
  const int64_t n_tiles = (rows + kPjRows - 1) / kPjRows;

  if (warp < 4) {
    // ------------------------------------------------------------ loaders
    // eight lanes per 128-B row slice, so that each instruction moves four
    // whole slices (lane: row 4j + lane / 8 of the warp's 32, chunk lane % 8)
    uint32_t it = 0;
    const int c = lane & 7;
    for (int64_t t = blockIdx.x; t < n_tiles && !abort_flag; t += gridDim.x) {
      for (int a = 0; a < kPjAtoms; a++, it++) {
        const uint32_t s = it % kPjStages, ph = (it / kPjStages) & 1;
        if (!ptx::mbar_wait(&empty_bar[s], ph ^ 1)) { fail(); break; }
        unsigned char *dst = sm + kPjSmA + s * kPjStageBytes;
#pragma unroll
        for (int j = 0; j < 8; j++) {
          const int r = warp * 32 + j * 4 + (lane >> 3);
          const int64_t row = t * kPjRows + r;
          if (row < rows)
            ptx::cp_async16(dst + (r >> 3) * 1024 + pj_sw128(r & 7, c),
                            reinterpret_cast<const unsigned char *>(x + row * kPjIn) + a * 128 + c * 16);
        }
        ptx::cp_async_arrive_noinc(&full_bar[s]);
      }
    }
  } else if (warp == 4) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t it = 0, k = 0;
      const uint32_t sW = ptx::smem_u32(sm + kPjSmW), sA = ptx::smem_u32(sm + kPjSmA);
      for (int64_t t = blockIdx.x; t < n_tiles && !abort_flag; t += gridDim.x, k++) {
        const uint32_t acc = k & 1;
        if (!ptx::mbar_wait(&acc_empty[acc], ((k >> 1) & 1) ^ 1)) { fail(); break; }
        bool ok = true;
        for (int a = 0; a < kPjAtoms; a++, it++) {
          const uint32_t s = it % kPjStages, ph = (it / kPjStages) & 1;
          if (!ptx::mbar_wait(&full_bar[s], ph)) { fail(); ok = false; break; }
          ptx::fence_proxy_async_smem();            // the slice came by ordinary asynchronous copies
          ptx::tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; kk++) {
            const uint64_t ad = ptx::smem_desc(sA + s * kPjStageBytes + kk * 32, 16, 1024, 2);
            const uint64_t bd = ptx::smem_desc(sW + a * 1024 + kk * 32, 16, 8192, 2);
            ptx::tc_mma_bf16(tmem + acc * kPjOut, ad, bd, kPjIdesc, (a > 0 || kk > 0) ? 1u : 0u);
          }
          ptx::tc_commit(&empty_bar[s]);
        }
        if (!ok) break;
        ptx::tc_commit(&acc_full[acc]);
      }
    }
    __syncwarp();
  } else if (warp >= 8) {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;
    uint32_t k = 0;
    for (int64_t t = blockIdx.x; t < n_tiles && !abort_flag; t += gridDim.x, k++) {
      const uint32_t acc = k & 1;
      if (!ptx::mbar_wait(&acc_full[acc], (k >> 1) & 1)) { fail(); break; }
      ptx::tc_fence_after();
      const int64_t row = t * kPjRows + quarter * 32 + lane;
      uint4 *o = reinterpret_cast<uint4 *>(out + row * kPjOut);
#pragma unroll 1
      for (int c0 = 0; c0 < kPjOut / 32; c0++) {
        uint32_t d[32];
        ptx::tmem_ld_32x32b_x32(tmem + ((uint32_t)(quarter * 32) << 16) + acc * kPjOut + c0 * 32, d);
        ptx::tmem_wait_ld();
        uint32_t p[16];
#pragma unroll
        for (int i = 0; i < 16; i++) {
          const __nv_bfloat162 b = __floats2bfloat162_rn(__uint_as_float(d[2 * i]), __uint_as_float(d[2 * i + 1]));
          p[i] = *reinterpret_cast<const uint32_t *>(&b);
        }
        if (row < rows) {
#pragma unroll
          for (int j = 0; j < 4; j++) o[c0 * 4 + j] = make_uint4(p[4 * j], p[4 * j + 1], p[4 * j + 2], p[4 * j + 3]);
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&acc_empty[acc]);
    }
  }
  __syncthreads();
  if (abort_flag) {
    // a wait ran out: the loading lanes' copies and the MMAs finish before
    // the tensor memory goes back (bounded)
    if (warp < 4) asm volatile("cp.async.wait_all;" ::: "memory");
    if (warp == 4 && lane == 0) ptx::tc_commit(&drain_bar);
    ptx::mbar_wait(&drain_bar, 0);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kPjTmemCols);
  }
}

cudaError_t launch_proj_keys(const void *x, int64_t rows, const void *w, void *out, int *status, cudaStream_t st) {
  const int dev = current_device();
  static std::atomic<int> attr_done[kMaxDevices];
  const size_t smem = (size_t)kPjSmem + 1024;
  cudaError_t e = once_per_device(attr_done, dev, [&] {
    return cudaFuncSetAttribute(proj_keys_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  });
  if (e != cudaSuccess) return e;
  const int64_t n_tiles = (rows + kPjRows - 1) / kPjRows;
  const int n_sm = device_sm_count(dev);
  const int64_t grid = n_tiles < n_sm ? n_tiles : n_sm;
  return launch_pdl(proj_keys_kernel, dim3((unsigned)grid), dim3(kPjThreads), smem, st, 1u,
                    static_cast<const uint16_t *>(x), rows, static_cast<const uint16_t *>(w),
                    static_cast<uint16_t *>(out), status);
}

}  // namespace csa2
