// Lightning-indexer scores on the 5th-generation tensor cores (csa2_index_score).
//
// "32 FP4 query heads of 128 dims against one shared key per entry, ReLU'd
// scores summed with per-head weights" and the keys are "128 FP4 values with one
// E8M0 scale per 32" ("An infra-oriented diagram of the DeepSeek-V4.1-Flash
// architecture", lightning-indexer note and section "The KV cache").  That is
// exactly the MXFP4 block-scaled format the tcgen05 MMA consumes, so
//     D[entry][head] = sum_c khat[entry][c] * qhat[head][c]
// is one  M=128 (entries) x N=32 (heads) x K=128  product per tile, issued as two
// tcgen05.mma.kind::mxf4.block_scale.scale_vec::2X (K=64 each) into TMEM, and the
// epilogue computes s = sum_h w_h * max(0, D[entry][h]) per row.
//
// The kernel is HBM-bound (68 B of key per entry, 8 FLOP/B of FP4 MMA): a
// persistent CTA per SM streams tiles through a 20-stage shared-memory ring.
// Warp roles (320 threads):
//   warp 0      producer: bulk copies (cp.async.bulk) of the 128 x 64 B nibble
//               tile (or 16 gathered 8-entry blocks of 512 B in pool mode) and of
//               its E8M0 scales into the stage ring; the query's 32 x 64 B and its
//               scales only when the CTA moves to another query (two query slots),
//               so that 152 CTAs do not re-read the same few L2 lines per tile.
//               The nibble planes are stored 64B-swizzled, so a plain contiguous
//               copy lands in the layout the MMA reads;
//   warp 1      TMEM owner + MMA issuer: rearranges the scales in shared memory
//               into the 32-lane x 16-B layout tcgen05.cp expects, copies them
//               into TMEM, issues the two MMAs, commits to the stage's "empty"
//               barrier and to the accumulator's "full" barrier;
//   warps 2..9  epilogue, two groups of four warps taking alternate tiles: one
//               TMEM lane (= one entry) per thread, 32 columns (= heads) per
//               tcgen05.ld, ReLU + weighted sum, coalesced store.
// Four TMEM accumulators let the epilogue of earlier tiles overlap the MMAs of
// later ones.
// Every mbarrier wait is bounded (CSA2_ERR_TIMEOUT instead of a hang).
#include "common.cuh"
#include "tc_ptx.cuh"

namespace csa2 {

constexpr int kScStages = 20;
constexpr int kScStageBytes = 9216;
constexpr int kOffA = 0;          // 128 rows x 64 B nibble tile, 64B-swizzled as stored
constexpr int kOffSFA = 8192;     // 512 B key scales: staged [row][4], rearranged in place
constexpr int kScQBytes = 2560;   // per query slot: 32 x 64 B nibbles + 512 B scales
constexpr int kQOffB = 0, kQOffSFB = 2048;
constexpr int kScSmem = kScStages * kScStageBytes + 2 * kScQBytes;
constexpr int kScThreads = 320;
constexpr int kScAcc = 4;               // TMEM accumulator stages
constexpr uint32_t kScTmemCols = 256;   // 4 x 32 accumulator columns + 4 x 4 SFA + 2 x 4 SFB
constexpr uint32_t kColSFA = 128, kColSFB = 144;

// Instruction descriptor of kind::mxf4 block-scaled MMA, M=128, N=32, both
// operands E2M1 and K-major, UE8M0 scales; sf_id picks the scale byte pair.
__host__ __device__ constexpr uint32_t idesc_mxf4_m128n32(uint32_t sf_id) {
  return (sf_id << 4)            // B scale-factor id
         | (1u << 7)             // A format: E2M1
         | (1u << 10)            // B format: E2M1
         | ((32u >> 3) << 17)    // N / 8
         | (1u << 23)            // scale format UE8M0
         | ((128u >> 4) << 24)   // M / 16
         | (sf_id << 29);        // A scale-factor id
}

struct ScoreTcArgs {
  const uint8_t *key_nib;
  const uint8_t *q_nib;
  const uint8_t *key_scale;
  const uint8_t *q_scale;
  const float *w;
  const int32_t *q_seq;
  const int32_t *n_vis;
  const int32_t *pool;
  float *scores;
  int64_t stride;
  int64_t n_max;
  int n_seq;
  int n_q;
  int tiles_per_q;
  int64_t total_tiles;
  int *status;
};

struct TileInfo {
  int q, tile, seq, nv;
};

// Shared tile schedule of every role: tile T = blockIdx.x + k * gridDim.x over
// (query, 128-entry tile); tiles past a query's visible length are skipped.
__device__ __forceinline__ bool next_tile(const ScoreTcArgs &P, int64_t &T, TileInfo &t) {
  for (; T < P.total_tiles; T += gridDim.x) {
    t.q = (int)(T / P.tiles_per_q);
    t.tile = (int)(T % P.tiles_per_q);
    t.seq = __ldg(P.q_seq + t.q);
    t.nv = __ldg(P.n_vis + t.q);
    if (t.seq < 0 || t.seq >= P.n_seq || t.nv < 0 || (int64_t)t.nv > P.n_max) {
      if (t.tile == 0 && threadIdx.x == 0) record_error(P.status, CSA2_ERR_BOUNDS);
      continue;
    }
    if (P.pool == nullptr && (int64_t)t.tile * 128 >= t.nv) continue;
    T += gridDim.x;
    return true;
  }
  return false;
}

__global__ void __launch_bounds__(kScThreads, 1) index_score_tc_kernel(ScoreTcArgs P) {
  extern __shared__ __align__(1024) unsigned char sc_smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(sc_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  unsigned char *qslots = smem + kScStages * kScStageBytes;
  __shared__ __align__(8) uint64_t full_bar[kScStages], empty_bar[kScStages], acc_full[kScAcc], acc_empty[kScAcc];
  __shared__ __align__(8) uint64_t qfull[2], qempty[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kScStages; s++) {
      ptx::mbar_init(&full_bar[s], 1);
      ptx::mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < kScAcc; a++) {
      ptx::mbar_init(&acc_full[a], 1);
      ptx::mbar_init(&acc_empty[a], 4);
    }
    for (int q = 0; q < 2; q++) {
      ptx::mbar_init(&qfull[q], 1);
      ptx::mbar_init(&qempty[q], 1);
    }
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) ptx::tmem_alloc(&tmem_base_sh, kScTmemCols);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  auto fail = [&]() {
    record_error(P.status, CSA2_ERR_TIMEOUT);
    abort_flag = 1;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t policy = ptx::policy_evict_first();
    int64_t T = blockIdx.x;
    TileInfo t;
    int cur_q = -1;
    uint32_t qsw = 0;                                   // query switches so far
    for (uint32_t it = 0; next_tile(P, T, t); it++) {
      if (abort_flag) break;
      if (t.q != cur_q) {
        const uint32_t slot = qsw & 1, rnd = qsw >> 1;
        if (!ptx::mbar_wait(&qempty[slot], (rnd & 1) ^ 1)) { fail(); break; }
        if (lane == 0) {
          unsigned char *qs = qslots + slot * kScQBytes;
          ptx::mbar_arrive_expect_tx(&qfull[slot], 2048 + 128);
          ptx::bulk_load(qs + kQOffB, P.q_nib + (int64_t)t.q * kIdxHeads * 64, 2048, &qfull[slot]);
          ptx::bulk_load(qs + kQOffSFB, P.q_scale + (int64_t)t.q * kIdxHeads * 4, 128, &qfull[slot]);
        }
        cur_q = t.q;
        qsw++;
      }
      const uint32_t s = it % kScStages, r = it / kScStages;
      if (!ptx::mbar_wait(&empty_bar[s], (r & 1) ^ 1)) { fail(); break; }
      unsigned char *st = smem + s * kScStageBytes;
      const int64_t row0 = (int64_t)t.seq * P.n_max;
      if (P.pool == nullptr) {
        if (lane == 0) {
          ptx::mbar_arrive_expect_tx(&full_bar[s], 8192 + 512);
          const int64_t r0 = row0 + (int64_t)t.tile * 128;
          ptx::bulk_load_hint(st + kOffA, P.key_nib + r0 * 64, 8192, &full_bar[s], policy);
          ptx::bulk_load(st + kOffSFA, P.key_scale + r0 * 4, 512, &full_bar[s]);
        }
      } else {
        int blk = -1;
        bool ok = false;
        if (lane < 16) {
          blk = __ldg(P.pool + (int64_t)t.q * kPoolBlocks + t.tile * 16 + lane);
          ok = blk >= 0 && (int64_t)blk * kBlock < P.n_max;
          if (blk >= 0 && !ok) record_error(P.status, CSA2_ERR_BOUNDS);
        }
        const unsigned m = __ballot_sync(0xFFFFFFFFu, ok);
        // an all-empty tile still arrives once, so its phase completes
        if (lane == 0) ptx::mbar_arrive_expect_tx(&full_bar[s], (uint32_t)__popc(m) * (512 + 32));
        __syncwarp();
        if (ok) {
          const int64_t r0 = row0 + (int64_t)blk * kBlock;
          ptx::bulk_load_hint(st + kOffA + lane * 512, P.key_nib + r0 * 64, 512, &full_bar[s], policy);
          ptx::bulk_load(st + kOffSFA + lane * 32, P.key_scale + r0 * 4, 32, &full_bar[s]);
        }
      }
      __syncwarp();
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    int64_t T = blockIdx.x;
    TileInfo t;
    int cur_q = -1;
    uint32_t qsw = 0, slot = 0;
    const uint32_t idesc0 = idesc_mxf4_m128n32(0), idesc1 = idesc_mxf4_m128n32(2);
    for (uint32_t it = 0; next_tile(P, T, t); it++) {
      if (abort_flag) break;
      if (t.q != cur_q) {
        // release the previous query slot once every MMA issued so far is done
        if (qsw > 0 && lane == 0) ptx::tc_commit(&qempty[(qsw - 1) & 1]);
        slot = qsw & 1;
        const uint32_t rnd = qsw >> 1;
        if (!ptx::mbar_wait(&qfull[slot], rnd & 1)) { fail(); break; }
        uint32_t *sfb = reinterpret_cast<uint32_t *>(qslots + slot * kScQBytes + kQOffSFB);
        const uint32_t vb = sfb[lane];
        __syncwarp();
        sfb[lane * 4 + 0] = vb;          // head `lane` -> 16-B line `lane` (tcgen05.cp layout)
        sfb[lane * 4 + 1] = 0u;
        sfb[lane * 4 + 2] = 0u;
        sfb[lane * 4 + 3] = 0u;
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          ptx::tc_fence_after();
          ptx::tc_cp_32x128b_warpx4(tmem + kColSFB + slot * 4, ptx::smem_desc(ptx::smem_u32(sfb), 0, 128, 0));
        }
        cur_q = t.q;
        qsw++;
      }
      const uint32_t s = it % kScStages, r = it / kScStages, a = it % kScAcc, ra = it / kScAcc;
      if (!ptx::mbar_wait(&full_bar[s], r & 1)) { fail(); break; }
      unsigned char *st = smem + s * kScStageBytes;
      // key scales -> tcgen05.cp layout: 16-B line m0 holds rows m0, m0+32, m0+64, m0+96
      uint32_t *sfa = reinterpret_cast<uint32_t *>(st + kOffSFA);
      uint32_t va[4];
#pragma unroll
      for (int i = 0; i < 4; i++) va[i] = sfa[i * 32 + lane];
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 4; i++) sfa[lane * 4 + i] = va[i];
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        if (!ptx::mbar_wait(&acc_empty[a], (ra & 1) ^ 1)) {
          fail();
        } else {
          ptx::tc_fence_after();
          const uint32_t t_sfa = tmem + kColSFA + a * 4, t_sfb = tmem + kColSFB + slot * 4;
          ptx::tc_cp_32x128b_warpx4(t_sfa, ptx::smem_desc(ptx::smem_u32(sfa), 0, 128, 0));
          const uint64_t ad = ptx::smem_desc(ptx::smem_u32(st + kOffA), 16, 512, 4);
          const uint64_t bd = ptx::smem_desc(ptx::smem_u32(qslots + slot * kScQBytes + kQOffB), 16, 512, 4);
          ptx::tc_mma_mxf4(tmem + a * 32, ad, bd, idesc0, t_sfa, t_sfb, 0u);
          ptx::tc_mma_mxf4(tmem + a * 32, ad + 2, bd + 2, idesc1, t_sfa, t_sfb, 1u);   // +32 B along K
          ptx::tc_commit(&empty_bar[s]);
          ptx::tc_commit(&acc_full[a]);
        }
      }
      __syncwarp();
      if (abort_flag) break;
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;
    const uint32_t group = (uint32_t)(warp - 2) >> 2;     // warps 2..5 -> 0, 6..9 -> 1
    const int row = quarter * 32 + lane;
    int64_t T = blockIdx.x;
    TileInfo t;
    int cur_q = -1;
    float wv[kIdxHeads];
    for (uint32_t it = 0; next_tile(P, T, t); it++) {
      if (abort_flag) break;
      if ((it & 1) != group) continue;
      const uint32_t a = it % kScAcc, ra = it / kScAcc;
      if (t.q != cur_q) {
        const float4 *wp = reinterpret_cast<const float4 *>(P.w + (int64_t)t.q * kIdxHeads);
#pragma unroll
        for (int i = 0; i < 8; i++) {
          const float4 v = __ldg(wp + i);
          wv[4 * i] = v.x;
          wv[4 * i + 1] = v.y;
          wv[4 * i + 2] = v.z;
          wv[4 * i + 3] = v.w;
        }
        cur_q = t.q;
      }
      if (!ptx::mbar_wait(&acc_full[a], ra & 1)) { fail(); break; }
      ptx::tc_fence_after();
      uint32_t d[32];
      ptx::tmem_ld_32x32b_x32(tmem + ((uint32_t)(quarter * 32) << 16) + a * 32, d);
      ptx::tmem_wait_ld();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&acc_empty[a]);
      float s = 0.f;
#pragma unroll
      for (int h = 0; h < kIdxHeads; h++) s = fmaf(wv[h], fmaxf(__uint_as_float(d[h]), 0.f), s);
      const int64_t item = (int64_t)t.tile * 128 + row;
      if (P.pool == nullptr) {
        if (item < t.nv) P.scores[(int64_t)t.q * P.stride + item] = s;
      } else {
        const int blk = __ldg(P.pool + (int64_t)t.q * kPoolBlocks + (item >> 3));
        const int64_t j = (int64_t)blk * kBlock + (item & 7);
        const bool ok = blk >= 0 && (int64_t)blk * kBlock < P.n_max && j < t.nv;
        P.scores[(int64_t)t.q * P.stride + item] = ok ? s : -INFINITY;
      }
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kScTmemCols);
  }
}

// ---------------------------------------------------------------- host side
static int sm_count() {
  static int counts[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 148;
  if (counts[dev] == 0) cudaDeviceGetAttribute(&counts[dev], cudaDevAttrMultiProcessorCount, dev);
  return counts[dev] > 0 ? counts[dev] : 148;
}

cudaError_t launch_index_score_tc(const uint8_t *key_nib, const uint8_t *key_scale, int64_t n_max, int n_seq,
                                  const uint8_t *q_nib, const uint8_t *q_scale, const float *w, const int32_t *q_seq,
                                  const int32_t *n_vis, int n_q, const int32_t *pool, float *scores, int64_t stride,
                                  int *status, cudaStream_t st) {
  ScoreTcArgs P;
  P.key_nib = key_nib;
  P.q_nib = q_nib;
  P.key_scale = key_scale;
  P.q_scale = q_scale;
  P.w = w;
  P.q_seq = q_seq;
  P.n_vis = n_vis;
  P.pool = pool;
  P.scores = scores;
  P.stride = stride;
  P.n_max = n_max;
  P.n_seq = n_seq;
  P.n_q = n_q;
  P.tiles_per_q = pool ? kPoolSlots / 128 : (int)(n_max / 128);
  P.total_tiles = (int64_t)n_q * P.tiles_per_q;
  P.status = status;
  const size_t smem = (size_t)kScSmem + 1024;
  int dev = 0;
  cudaGetDevice(&dev);
  static bool attr_done[64] = {};
  if (dev >= 0 && dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(index_score_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  const int64_t grid = P.total_tiles < sm_count() ? P.total_tiles : sm_count();
  index_score_tc_kernel<<<(unsigned)grid, kScThreads, smem, st>>>(P);
  return cudaGetLastError();
}

}  // namespace csa2
