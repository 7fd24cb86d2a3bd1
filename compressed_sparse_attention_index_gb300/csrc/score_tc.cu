// Lightning-indexer scores on the 5th-generation tensor cores (csa2_index_score).
//
// The indexer compares 32 FP4 query heads of width 128 with one key per entry,
// clamps each head's dot product at zero and sums them with per-head weights;
// a key is 128 FP4 values with one E8M0 scale per 32 (An infra-oriented diagram
// of the DeepSeek-V4.1-Flash architecture, lightning-indexer note and section
// "The KV cache").  That is
// exactly the MXFP4 block-scaled format the tcgen05 MMA consumes, so
//     D[entry][head] = sum_c khat[entry][c] * qhat[head][c]
// is one  M=128 (entries) x N=32 (heads) x K=128  product per 128 entries,
// issued as two tcgen05.mma.kind::mxf4.block_scale.scale_vec::2X (K=64 each)
// into TMEM; the epilogue computes s = sum_h w_h * max(0, D[entry][h]) per row.
//
// The kernel is HBM-bound (68 B of key per entry, 8 FLOP/B of FP4 MMA): a
// persistent CTA per SM streams work units of 512 entries (four 128-row
// sub-tiles, 34 KB) through a 6-stage shared-memory ring.  Every tcgen05
// instruction and every barrier wait costs its issuing thread tens of cycles,
// so the design keeps those per byte low: big units, one commit per unit, and
// two MMA issuers.  Warp roles (480 threads):
//   warp 0      producer: one bulk copy (cp.async.bulk) of the unit's 32 KB of
//               nibbles, and its 2 KB of E8M0 scales by the lanes' 16-B
//               asynchronous copies (pool mode: 8 of the 64 gathered 8-entry
//               blocks of 512 B + 32 B, by 16-B asynchronous copies; warps
//               12..14 and 7..10 gather the other 56); with the first unit of each run
//               of one query, its 2 KB of nibbles and 128 B of scales (lanes'
//               copies too) into the next of six query slots (so a CTA may
//               switch query on every unit without a stall).  The nibble planes are stored
//               64B-swizzled, so a plain contiguous copy lands in the layout the
//               MMA reads;
//   warp 2      scale-factor warp: rearranges the unit's key scales in shared
//               memory into the 32-lane x 16-B layout tcgen05.cp expects, copies
//               them into TMEM and signals the MMA issuers through tcgen05.commit;
//   warps 1, 11 MMA issuers (lane 0; warp 1 also owns TMEM), even and odd
//               units: eight MMAs per unit into the unit's accumulator, then one
//               commit to the stage's done barrier, which both frees the stage
//               and marks the accumulator full;
//   warps 3..10 epilogue, two groups of four warps taking alternate units (pool
//               mode: warps 3..6 take every unit, warps 7..10 gather): one
//               TMEM lane (= one entry of each sub-tile) per thread, 32 columns
//               (= heads) per sub-tile, ReLU + weighted sum, coalesced store.
// The producer walks the CTA's units (a fixed stride over all of them, or
// over runs of consecutive units) and hands each to the other roles through
// a small shared-memory ring; the
// per-query sequence id / visible length are cached.  Every wait is bounded (CSA2_ERR_TIMEOUT
// instead of a hang).
#include "common.cuh"
#include "tc_ptx.cuh"
#include "launch.cuh"

namespace csa2 {

constexpr int kScStages = 6;
constexpr int kSub = 4;                   // 128-row sub-tiles per work unit
constexpr int kUnit = kSub * 128;         // entries per work unit
constexpr int kOffA = 0;                  // sub-tile j at j * 8192: 128 rows x 64 B, 64B-swizzled as stored
constexpr int kOffSFA = kSub * 8192;      // kSub x 512 B key scales: staged [row][4], rearranged in place
constexpr int kScStageBytes = kOffSFA + kSub * 512;
constexpr int kQSlots = 6;                // query slots, used round-robin, one per run of units of a query
constexpr int kScQBytes = 2560;           // per slot: 32 heads x 64 B nibbles + 128 B scales spread to 512 B
constexpr int kQOffB = 0, kQOffSFB = 2048;
constexpr int kScSmem = kScStages * kScStageBytes + kQSlots * kScQBytes;
static_assert(kScStageBytes % 1024 == 0, "64B-swizzled tiles need 512-B aligned stages and slots");
constexpr int kScGather0 = 12;            // warps 12..14: extra gathering warps (pool mode)
constexpr int kScGather1 = 7;             // warps 7..10: gathering warps too in pool mode (one epilogue group there)
constexpr int kPoolGatherWarps = 8;       // warp 0, warps 12..14 and 7..10, 8 of a unit's 64 blocks each
constexpr int kPoolWarpBlocks = 64 / kPoolGatherWarps;
constexpr int kScThreads = 480;
constexpr int kScMmaWarp2 = 11;          // second MMA issuer (odd units)
constexpr int kScAcc = 2;                 // TMEM accumulators (kSub x 32 columns each), one per epilogue group
constexpr uint32_t kScTmemCols = 512;
constexpr uint32_t kColSFA = kScAcc * kSub * 32;              // per stage: kSub x 4 columns
constexpr uint32_t kColSFB = kColSFA + kScStages * kSub * 4;  // per query slot: 4 columns
static_assert(kColSFB + kQSlots * 4 <= kScTmemCols, "TMEM columns");
static_assert(kScStages % kScAcc == 0, "a stage's done barrier also marks its accumulator full");

// Instruction descriptor of kind::mxf4 block-scaled MMA, M=128, N=n (a
// multiple of 16, <= 256), both operands E2M1 and K-major, UE8M0 scales;
// sf_id picks the scale byte pair.
__host__ __device__ constexpr uint32_t idesc_mxf4_m128(uint32_t sf_id, uint32_t n) {
  return (sf_id << 4)            // B scale-factor id
         | (1u << 7)             // A format: E2M1
         | (1u << 10)            // B format: E2M1
         | ((n >> 3) << 17)      // N / 8
         | (1u << 23)            // scale format UE8M0
         | ((128u >> 4) << 24)   // M / 16
         | (sf_id << 29);        // A scale-factor id
}
__host__ __device__ constexpr uint32_t idesc_mxf4_m128n32(uint32_t sf_id) { return idesc_mxf4_m128(sf_id, 32); }

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
  int units_per_q;
  int *status;
  // optional: maxima of the order keys of the scores, for the top-k that
  // follows.  Full mode: smax_mode 2: per 32 consecutive entries at
  // smax[q * sstride + entry / 32]; smax_mode 3: per work unit u, four partial
  // maxima (one per TMEM lane quarter, over its rows of the four sub-tiles) at
  // smax[q * sstride + 4u + quarter], and per 32 consecutive entries at
  // gmax[q * gstride + entry / 32].  Pool mode: smax_mode 1: per gathered
  // 8-entry block b at gmax[q * gstride + b].  Invalid entries count as key 0.
  uint32_t *smax;
  int64_t sstride;
  uint32_t *gmax;
  int64_t gstride;
  int smax_mode;
  // optional: the candidate-handoff flags of the selection and attention
  // grids that follow ([n_q][kHandWords] words; words 0-3 zeroed here)
  uint32_t *hflag;
  // optional (Full mode): the claim counter of the last kStealRounds rounds of
  // units, tagged with call_id in its upper 32 bits (see the producer)
  unsigned long long *steal;
  uint32_t call_id;
  int run;          // Full mode without claims: consecutive units a CTA takes at a time (set by the launch)
};

// Full mode inside csa2_decode: a CTA takes the units T = blockIdx.x + k gridDim.x
// up to the last kStealRounds rounds, then claims units one at a time from a
// counter, so that the SMs that stream faster take more of the tail.
// Only where a CTA has many rounds (measured: 8 x 1M, 108 rounds, -2 us per
// step; 32 x 64K, 27 rounds, +4.7 us: there a claimed unit is a fresh query
// almost every time).
constexpr int kStealRounds = 4;
constexpr int kMaxRun = 16;
constexpr uint32_t kStealMinRounds = 32;

// Work units are T = (query, unit) in query-major order, T < n_q * units_per_q;
// a CTA takes T = blockIdx.x, blockIdx.x + gridDim.x, ... (or runs of P.run
// consecutive units at a stride of gridDim.x runs; inside csa2_decode the last
// rounds may be claimed, see kStealRounds).  The producer walks that sequence,
// skips units past a query's visible length, and publishes the unit of each
// of its iterations `it` in a ring of shared-memory words (it << 32 | T;
// T = kDone after the last unit); every other role reads the ring in
// iteration order instead of walking the sequence itself.  A slot is
// rewritten 16 iterations later, which needs the MMA of iteration it + 10
// done, so every role has read it by then.  (Claiming every unit from a
// global counter measured slower: its atomics queue up.)
constexpr int kRing = 16;
constexpr uint32_t kDone = 0xFFFFFFFFu;

// Bounded wait for the ring entry of iteration it (a ring of R entries); false
// on timeout or abort.
template <int R = kRing>
__device__ __forceinline__ bool ring_get(const volatile unsigned long long *ring, uint32_t it, uint32_t &T,
                                         const volatile int &abort_flag) {
  for (long long n = 0; n < kSpinLimit; n++) {
    const unsigned long long e = ring[it % R];
    if ((uint32_t)(e >> 32) == it) { T = (uint32_t)e; return true; }
    if ((n & 63) == 63 && abort_flag) return false;
  }
  return false;
}

// Sequence id and visible length of a query, re-read when the query changes
// (from the CTA's shared-memory copy of every query's pair when there is one:
// qcache, for up to kQCache queries); nv = -1 marks a query whose values are
// out of range (recorded once, by the producer of its unit 0).
constexpr int kQCache = 256;
struct QueryInfo {
  int q = -1, seq = 0, nv = -1;
  int pre_q = -1, pre_seq = 0, pre_nv = 0;   // values loaded ahead (prefetch)
  const int2 *cache = nullptr;
  __device__ void prefetch(const ScoreTcArgs &P, int nq) {
    if (cache != nullptr || nq == q || nq == pre_q) return;
    pre_q = nq;
    pre_seq = __ldg(P.q_seq + nq);
    pre_nv = __ldg(P.n_vis + nq);
  }
  __device__ void set(const ScoreTcArgs &P, int nq, int u, bool record) {
    if (nq == q) return;
    q = nq;
    if (cache != nullptr) {
      const int2 c = cache[q];
      seq = c.x;
      nv = c.y;
    } else {
      seq = nq == pre_q ? pre_seq : __ldg(P.q_seq + q);
      nv = nq == pre_q ? pre_nv : __ldg(P.n_vis + q);
    }
    if (seq < 0 || seq >= P.n_seq || nv < 0 || (int64_t)nv > P.n_max) {
      if (record && u == 0) record_error(P.status, CSA2_ERR_BOUNDS);
      nv = -1;
    }
  }
};

// Query slots as seen by one role walking the schedule.  A run of consecutive
// units of one query (an epoch) takes the next slot round-robin; the slot's
// previous user was the last unit of the epoch kQSlots earlier.  Registers
// only: the ring of epoch starts is shifted, never indexed.
template <int NS>
struct QuerySlotsT {
  int cur_q = -1;
  uint32_t slot = NS - 1;
  int start[NS];                         // first unit of the last NS epochs, oldest first
  __device__ QuerySlotsT() {
#pragma unroll
    for (int i = 0; i < NS; i++) start[i] = -1;
  }
  // call once per unit in schedule order; true when unit `it` starts an epoch
  __device__ bool step(int q, int it) {
    if (q == cur_q) return false;
    cur_q = q;
    slot = slot + 1 == (uint32_t)NS ? 0u : slot + 1;
#pragma unroll
    for (int i = 0; i + 1 < NS; i++) start[i] = start[i + 1];
    start[NS - 1] = it;
    return true;
  }
  // after step() returned true: the last unit that used this slot (< 0 if none)
  __device__ int prev_user() const { return start[0] - 1; }
};
using QuerySlots = QuerySlotsT<kQSlots>;

// Pool mode: a unit is 64 gathered 8-entry blocks (512 B of nibbles + 32 B of
// scales each).  Small bulk copies cost the copy engine more than their bytes
// (measured, also as tile::gather4 tensor copies), and a warp takes a
// microsecond or more to issue a unit's asynchronous copies, so eight warps
// each move 8 blocks in 16-B pieces: one block's nibbles per instruction (16 B
// per lane), then the 8 blocks' scales in one.  Each lane arrives on the
// stage's barrier when its copies have landed (the barrier expects 1 + 32 x 8
// arrivals: the producer's lane 0 and every gathering lane).  A CTA has few units in
// pool mode (2,048 for 64 queries over 152 SMs), so the block ids are loaded
// kPoolAhead units ahead (the CTA's units T, T + gridDim.x, ...): a unit's
// copies then never wait for its ids to come back from memory.
constexpr int kPoolAhead = 6;
struct PoolGather {
  uint32_t pre_T[kPoolAhead];
  int pre_b[kPoolAhead];
  __device__ int load_b(const ScoreTcArgs &P, int g, uint32_t T) const {
    const int lane = threadIdx.x & 31;
    constexpr uint32_t upq = kPoolSlots / kUnit;   // (pool mode: a power of two)
    const int q = (int)(T / upq), u = (int)(T - (uint32_t)q * upq);
    return __ldg(P.pool + (int64_t)q * kPoolBlocks + u * (kUnit / kBlock) + g * kPoolWarpBlocks +
                 (lane & (kPoolWarpBlocks - 1)));
  }
  // ids of the units T0, T0 + gridDim.x, ... (kPoolAhead of them)
  __device__ void start(const ScoreTcArgs &P, int g, uint32_t T0, uint32_t total_units) {
#pragma unroll
    for (int d = 0; d < kPoolAhead; d++) {
      const uint32_t T = T0 + (uint32_t)d * gridDim.x;
      pre_T[d] = T < total_units ? T : kDone;
      pre_b[d] = T < total_units ? load_b(P, g, T) : -1;
    }
  }
  // the ids of unit T (normally the oldest prefetched); the ring then moves on
  __device__ int take(const ScoreTcArgs &P, int g, uint32_t T, uint32_t total_units) {
    if (pre_T[0] != T) start(P, g, T, total_units);   // a unit was skipped: restart the look-ahead at T
    const int b = pre_b[0];
#pragma unroll
    for (int d = 0; d + 1 < kPoolAhead; d++) {
      pre_T[d] = pre_T[d + 1];
      pre_b[d] = pre_b[d + 1];
    }
    const uint32_t Tn = T + (uint32_t)kPoolAhead * gridDim.x;
    pre_T[kPoolAhead - 1] = Tn < total_units ? Tn : kDone;
    pre_b[kPoolAhead - 1] = Tn < total_units ? load_b(P, g, Tn) : -1;
    return b;
  }
  __device__ void gather(const ScoreTcArgs &P, int g, uint32_t T, int64_t row0, unsigned char *st, uint64_t *full,
                         uint32_t total_units) {
    const int lane = threadIdx.x & 31;
    const int b = take(P, g, T, total_units);
    const bool ok = b >= 0 && (int64_t)b * kBlock < P.n_max;
    if (lane < kPoolWarpBlocks && b >= 0 && !ok) record_error(P.status, CSA2_ERR_BOUNDS);
#pragma unroll
    for (int j = 0; j < kPoolWarpBlocks; j++) {
      const int bj = __shfl_sync(0xFFFFFFFFu, b, j);
      if (bj >= 0 && (int64_t)bj * kBlock < P.n_max)
        ptx::cp_async16(st + kOffA + (g * kPoolWarpBlocks + j) * 512 + lane * 16,
                        P.key_nib + (row0 + (int64_t)bj * kBlock) * 64 + lane * 16);
    }
    const int bs = __shfl_sync(0xFFFFFFFFu, b, (lane >> 1) & (kPoolWarpBlocks - 1));
    if (lane < 2 * kPoolWarpBlocks && bs >= 0 && (int64_t)bs * kBlock < P.n_max)
      ptx::cp_async16(st + kOffSFA + (g * kPoolWarpBlocks + (lane >> 1)) * 32 + (lane & 1) * 16,
                      P.key_scale + (row0 + (int64_t)bs * kBlock) * 4 + (lane & 1) * 16);
    ptx::cp_async_arrive_noinc(full);
  }
};

// POOL: pool mode (P.pool set: units of gathered 8-entry blocks); SMAX: the
// maxima the epilogue writes (P.smax_mode: 0, 2 or 3 in Full mode, 0 or 1 in
// pool mode).
template <bool POOL, int SMAX>
__global__ void __launch_bounds__(kScThreads, 1) index_score_tc_kernel(ScoreTcArgs P) {
  extern __shared__ __align__(1024) unsigned char sc_smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(sc_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  unsigned char *qslots = smem + kScStages * kScStageBytes;
  // done_bar[s]: the MMAs of the unit in stage s have completed, so the stage
  // may be refilled and the unit's accumulator may be read (one commit serves both)
  __shared__ __align__(8) uint64_t full_bar[kScStages], sf_bar[kScStages], done_bar[kScStages];
  __shared__ __align__(8) uint64_t acc_empty[kScAcc];
  __shared__ __align__(8) uint64_t drain_bar;      // after a wait ran out: the tcgen05 issuers' last commits
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_flag;
  __shared__ int armed_sh;                         // iterations whose copies the producer issued
  __shared__ volatile unsigned long long unit_ring[kRing];
  __shared__ int2 qcache[POOL ? kQCache : 1];      // pool mode: (q_seq, n_vis) of every query, when n_q <= kQCache

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // The barriers and the tensor memory are set up before the wait for the
  // grid ahead: neither touches memory that grid writes, and this CTA is
  // placed only where no CTA holding tensor memory remains.
  if (threadIdx.x == 0) {
    for (int s = 0; s < kScStages; s++) {
      ptx::mbar_init(&full_bar[s], POOL ? 1 + 32 * kPoolGatherWarps : 1);   // pool: see PoolGather
      ptx::mbar_init(&sf_bar[s], 1);
      ptx::mbar_init(&done_bar[s], 1);
    }
    for (int a = 0; a < kScAcc; a++) ptx::mbar_init(&acc_empty[a], 4);
    ptx::mbar_init(&drain_bar, 3);                  // MMA issuers (warps 1, 11) and the scale-factor warp
    for (int i = 0; i < kRing; i++) unit_ring[i] = ~0ull;   // no iteration's tag
    abort_flag = 0;
    armed_sh = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) ptx::tmem_alloc(&tmem_base_sh, kScTmemCols);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  // everything below reads inputs: after the grid ahead
  griddep_wait();
  griddep_launch();
  // (pool mode only, where the query changes on every unit; elsewhere the
  // first unit would wait for the table)
  const int2 *qc = POOL && P.n_q <= kQCache ? qcache : nullptr;
  if (qc != nullptr) {
    for (int i = threadIdx.x; i < P.n_q; i += blockDim.x) qcache[i] = make_int2(__ldg(P.q_seq + i), __ldg(P.n_vis + i));
    __syncthreads();
  }
  // (the previous call's attention, which read these flags, has completed:
  // the grid ahead waited for it)
  if (P.hflag != nullptr)
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < 4 * P.n_q; i += gridDim.x * blockDim.x)
      P.hflag[(i >> 2) * kHandWords + (i & 3)] = 0u;
  const uint32_t tmem = tmem_base_sh;

  auto fail = [&]() {
    record_error(P.status, CSA2_ERR_TIMEOUT);
    abort_flag = 1;
  };

  // units per query: in pool mode a compile-time power of two (the divisions
  // below become shifts; each role divides on every unit, the query changing
  // on nearly every one there)
  const uint32_t upq = POOL ? (uint32_t)(kPoolSlots / kUnit) : (uint32_t)P.units_per_q;
  const uint32_t total_units = (uint32_t)P.n_q * upq;
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t policy = ptx::policy_evict_first();
    QuerySlots qs;
    QueryInfo sc;
    sc.cache = qc;
    // Claims (Full mode with a counter): the counter holds this call's tag
    // in its upper half and the next claim index in its lower half.  A value
    // with another tag is left from an earlier call (or is the workspace's
    // initial contents).  Before its first claim each CTA makes sure the tag
    // is this call's, by compare-and-swap alone (no CTA adds before it has
    // seen the tag, so every failed swap means another CTA installed it).
    // One claim is then always in flight (lane 0), issued a unit ahead of its
    // use, so that the atomic's latency hides behind the unit's copies.
    const bool steal = !POOL && P.steal != nullptr && total_units >= kStealMinRounds * gridDim.x;
    const uint32_t s_static =
        steal ? (uint32_t)max(0, (int)(total_units / gridDim.x) - kStealRounds) * gridDim.x : total_units;
    unsigned long long claim_v = 0ull;
    if (steal && lane == 0) {
      unsigned long long v = *reinterpret_cast<volatile unsigned long long *>(P.steal);
      int tries = 0;
      for (; tries < 4096 && (uint32_t)(v >> 32) != P.call_id; tries++) {
        const unsigned long long w = atomicCAS(P.steal, v, (unsigned long long)P.call_id << 32);
        if (w == v) break;                                             // installed: index 0 is next
        v = w;
      }
      if (tries == 4096) record_error(P.status, CSA2_ERR_TIMEOUT);   // (never seen)
      claim_v = atomicAdd(P.steal, 1ull);
    }
    auto claim_next = [&]() -> uint32_t {
      uint32_t idx = kDone;
      if (lane == 0) {
        if ((uint32_t)(claim_v >> 32) == P.call_id) idx = (uint32_t)claim_v;
        claim_v = atomicAdd(P.steal, 1ull);                            // the next claim goes out now
      }
      return __shfl_sync(0xFFFFFFFFu, idx, 0);
    };
    // Full mode without claims: the CTA takes runs of P.run consecutive units
    // at a stride of gridDim.x runs, so that where queries have few units
    // each (many short sequences, or a prefill's queries) a new query's data
    // and bookkeeping come once per run instead of on nearly every unit (the
    // launch picks the run length, never more units for the busiest CTA)
    const uint32_t run = !POOL && !steal && P.run > 1 ? (uint32_t)P.run : 1u;
    uint32_t grp = blockIdx.x, rin = 0;            // the current unit: grp * run + rin
    // the unit after Tc in this CTA's sequence (total_units: none left)
    auto advance = [&](uint32_t Tc) -> uint32_t {
      if (run > 1) {
        if (++rin < run && Tc + 1 < total_units) return Tc + 1;
        rin = 0;
        grp += gridDim.x;
        return (uint64_t)grp * run < total_units ? grp * run : total_units;
      }
      if (!steal || Tc + gridDim.x < s_static) return Tc + gridDim.x;
      const uint32_t i = claim_next();
      return i < total_units - s_static ? s_static + i : total_units;
    };
    uint32_t T = (uint64_t)blockIdx.x * run < total_units ? blockIdx.x * run : total_units;
    if (steal && T >= s_static) {
      const uint32_t i = claim_next();
      T = i < total_units - s_static ? s_static + i : total_units;
    }
    PoolGather pg;
    if (POOL) pg.start(P, 0, T, total_units);
    for (uint32_t it = 0;; it++) {
      if (abort_flag) break;
      // this iteration's unit: the next one inside its query's visible length
      int uq = 0;
      for (;;) {
        if (T >= total_units) { T = kDone; break; }
        const int q = (int)(T / upq);
        uq = (int)(T - (uint32_t)q * upq);
        sc.set(P, q, uq, lane == 0);
        if (sc.nv >= 0 && (POOL || uq * kUnit < sc.nv)) break;
        T = advance(T);
      }
      if (lane == 0) unit_ring[it % kRing] = ((unsigned long long)it << 32) | T;
      if (T == kDone) break;
      const int cur_u = uq;
      const uint32_t s = it % kScStages, r = it / kScStages;
      const bool fresh = qs.step(sc.q, (int)it);
      if (!ptx::mbar_wait(&done_bar[s], (r & 1) ^ 1)) { fail(); break; }
      if (fresh) {
        // the slot's previous users must be done: its last unit and the one
        // before (the two issuers complete independently; each in order).
        // Units up to it - kScStages are (the wait above); a later one is
        // waited for on its own stage barrier, whose next phase needs a unit
        // not yet loaded, so the parity is unambiguous.
        bool ok = true;
        for (int u = qs.prev_user(), k = 0; k < 2 && ok; k++, u--)
          if (u >= 0 && u + kScStages > (int)it)
            ok = ptx::mbar_wait(&done_bar[u % kScStages], (uint32_t)(u / kScStages) & 1);
        if (!ok) { fail(); break; }
      }
      unsigned char *st = smem + s * kScStageBytes;
      // a new run of units of one query: its data travel with this unit
      unsigned char *qd = qslots + qs.slot * kScQBytes;
      const int64_t row0 = (int64_t)sc.seq * P.n_max;
      if (!POOL) {
        // A new query's 2 KB of nibbles and 128 B of scales, and the unit's
        // key scales, go as 16-B asynchronous copies of the warp's lanes, each
        // lane counted into the stage's barrier (before the expected bytes of
        // the nibbles' bulk copy), not as more bulk copies: the bulk-copy unit
        // spends a fixed time per instruction (measured: -1.5 us per step at
        // 32 x 64K, where the query changes on nearly every unit).
        // Sub-tiles that start before n_vis end within n_max (n_max % 128 == 0).
        const int left = sc.nv - cur_u * kUnit;
        const int nsub = left >= kUnit ? kSub : (left + 127) >> 7;
        const int64_t r0 = row0 + (int64_t)cur_u * kUnit;
        if (fresh) {
          const unsigned char *qn = P.q_nib + (int64_t)sc.q * kIdxHeads * 64;
#pragma unroll
          for (int k = 0; k < 4; k++) ptx::cp_async16(qd + kQOffB + (k * 32 + lane) * 16, qn + (k * 32 + lane) * 16);
          if (lane < 8) ptx::cp_async16(qd + kQOffSFB + lane * 16, P.q_scale + (int64_t)sc.q * kIdxHeads * 4 + lane * 16);
        }
        // the unit's key scales (nsub x 512 B) the same way
#pragma unroll
        for (int k = 0; k < 4; k++)
          if (k * 32 + lane < nsub * 32)
            ptx::cp_async16(st + kOffSFA + (k * 32 + lane) * 16, P.key_scale + r0 * 4 + (k * 32 + lane) * 16);
        ptx::cp_async_arrive(&full_bar[s]);
        __syncwarp();
        if (lane == 0) {
          ptx::mbar_arrive_expect_tx(&full_bar[s], (uint32_t)nsub * 8192);
          ptx::bulk_load_hint(st + kOffA, P.key_nib + r0 * 64, (uint32_t)nsub * 8192, &full_bar[s], policy);
        }
      } else {
        // pool: this warp gathers blocks 0..15 of the unit, warps 12..14 the
        // rest (see PoolGather); its lanes also bring the query data, if any,
        // as asynchronous copies that the gather's arrivals cover
        if (fresh) {
          const unsigned char *qn = P.q_nib + (int64_t)sc.q * kIdxHeads * 64;
#pragma unroll
          for (int k = 0; k < 4; k++) ptx::cp_async16(qd + kQOffB + (k * 32 + lane) * 16, qn + (k * 32 + lane) * 16);
          if (lane < 8) ptx::cp_async16(qd + kQOffSFB + lane * 16, P.q_scale + (int64_t)sc.q * kIdxHeads * 4 + lane * 16);
        }
        if (lane == 0) ptx::mbar_arrive(&full_bar[s]);
        pg.gather(P, 0, T, row0, st, &full_bar[s], total_units);
        if (T + gridDim.x < total_units) sc.prefetch(P, (int)((T + gridDim.x) / upq));
      }
      __syncwarp();
      if (lane == 0) armed_sh = (int)it + 1;
      T = advance(T);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ scale-factor warp
    QuerySlots qs;
    for (uint32_t it = 0;; it++) {
      if (abort_flag) break;
      uint32_t T;
      if (!ring_get(unit_ring, it, T, abort_flag)) { fail(); break; }
      if (T == kDone) break;
      const uint32_t s = it % kScStages, r = it / kScStages;
      const bool fresh = qs.step((int)(T / upq), (int)it);
      if (!ptx::mbar_wait(&full_bar[s], r & 1)) { fail(); break; }
      unsigned char *st = smem + s * kScStageBytes;
      unsigned char *qd = qslots + qs.slot * kScQBytes;
      if (fresh) {
        uint32_t *sfb = reinterpret_cast<uint32_t *>(qd + kQOffSFB);
        const uint32_t vb = sfb[lane];
        __syncwarp();
        sfb[lane * 4 + 0] = vb;          // head `lane` -> 16-B line `lane` (tcgen05.cp layout)
        sfb[lane * 4 + 1] = 0u;
        sfb[lane * 4 + 2] = 0u;
        sfb[lane * 4 + 3] = 0u;
      }
      // key scales -> tcgen05.cp layout: 16-B line m0 of sub-tile j holds rows
      // m0, m0+32, m0+64, m0+96 of that sub-tile
      uint32_t *sfa = reinterpret_cast<uint32_t *>(st + kOffSFA);
      uint32_t va[4 * kSub];
#pragma unroll
      for (int i = 0; i < 4 * kSub; i++) va[i] = sfa[i * 32 + lane];
      __syncwarp();
#pragma unroll
      for (int j = 0; j < kSub; j++)
#pragma unroll
        for (int i = 0; i < 4; i++) sfa[j * 128 + lane * 4 + i] = va[j * 4 + i];
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        ptx::tc_fence_after();
        if (fresh)
          ptx::tc_cp_32x128b_warpx4(tmem + kColSFB + qs.slot * 4, ptx::smem_desc(ptx::smem_u32(qd + kQOffSFB), 0, 128, 0));
        const uint32_t sa = ptx::smem_u32(sfa);
#pragma unroll
        for (int j = 0; j < kSub; j++)
          ptx::tc_cp_32x128b_warpx4(tmem + kColSFA + s * (kSub * 4) + j * 4, ptx::smem_desc(sa + j * 512, 0, 128, 0));
        ptx::tc_commit(&sf_bar[s]);
      }
      __syncwarp();
    }
  } else if (warp == 1 || warp == kScMmaWarp2) {
    // ------------------------------------------------------------ MMA issuers (lane 0 of warps 1, 11)
    // A lone issuing thread spends most of a unit's time on its own instruction
    // latency (waits, descriptors, schedule), so two warps issue alternate units,
    // each into its own accumulator, with one commit per unit.
    if (lane == 0) {
      const uint32_t par = warp == 1 ? 0u : 1u;
      const uint32_t idesc0 = idesc_mxf4_m128n32(0), idesc1 = idesc_mxf4_m128n32(2);
      QuerySlots qs;
      for (uint32_t it = 0;; it++) {
        if (abort_flag) break;
        uint32_t T;
        if (!ring_get(unit_ring, it, T, abort_flag)) { fail(); break; }
        if (T == kDone) break;
        qs.step((int)(T / upq), (int)it);
        if ((it & 1) != par) continue;
        const uint32_t s = it % kScStages, r = it / kScStages, a = it % kScAcc, ra = it / kScAcc;
        if (!ptx::mbar_wait(&sf_bar[s], r & 1) || !ptx::mbar_wait(&acc_empty[a], (ra & 1) ^ 1)) { fail(); break; }
        // the query data (and, in pool mode, the stage) came by ordinary
        // asynchronous copies, which the MMA (async proxy) reads only after a
        // proxy fence
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_after();
        const uint32_t sa = ptx::smem_u32(smem + s * kScStageBytes + kOffA);
        const uint64_t bd = ptx::smem_desc(ptx::smem_u32(qslots + qs.slot * kScQBytes + kQOffB), 16, 512, 4);
        const uint32_t t_sfb = tmem + kColSFB + qs.slot * 4;
#pragma unroll
        for (int j = 0; j < kSub; j++) {
          const uint64_t ad = ptx::smem_desc(sa + j * 8192, 16, 512, 4);
          const uint32_t t_sfa = tmem + kColSFA + s * (kSub * 4) + j * 4;
          const uint32_t d = tmem + a * (kSub * 32) + j * 32;
          ptx::tc_mma_mxf4(d, ad, bd, idesc0, t_sfa, t_sfb, 0u);
          ptx::tc_mma_mxf4(d, ad + 2, bd + 2, idesc1, t_sfa, t_sfb, 1u);   // +32 B along K
        }
        ptx::tc_commit(&done_bar[s]);
      }
    }
    __syncwarp();
  } else if (warp >= kScGather0 || (POOL && warp >= kScGather1 && warp < kScGather1 + 4)) {
    // ------------------------------------------------------------ gathering warps (pool mode only)
    if (POOL) {
      const int g = warp >= kScGather0 ? warp - kScGather0 + 1 : warp - kScGather1 + 4;
      QueryInfo gq;
      gq.cache = qc;
      PoolGather pg;
      pg.start(P, g, blockIdx.x, total_units);
      for (uint32_t it = 0;; it++) {
        if (abort_flag) break;
        uint32_t T;
        if (!ring_get(unit_ring, it, T, abort_flag)) { fail(); break; }
        if (T == kDone) break;
        const uint32_t s = it % kScStages, r = it / kScStages;
        const int q = (int)(T / upq), u = (int)(T % upq);
        gq.set(P, q, u, false);                       // published units are valid
        if (!ptx::mbar_wait(&done_bar[s], (r & 1) ^ 1)) { fail(); break; }
        pg.gather(P, g, T, (int64_t)gq.seq * P.n_max, smem + s * kScStageBytes, &full_bar[s], total_units);
        if (T + gridDim.x < total_units) gq.prefetch(P, (int)((T + gridDim.x) / upq));
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // group g (warps 3+4g .. 6+4g) takes the units with it % 2 == g and owns
    // accumulator g; in pool mode, whose units are few and gathered by more
    // warps, group 0 alone takes every unit, accumulator it % 2 (warps 7..10
    // gather).  Waiting on done_bar is unambiguous: the stage's next phase
    // needs the MMA of unit it+kScStages, which needs the unit it+kScStages-2
    // (same accumulator) released, i.e. this group to have passed unit it.
    const int quarter = warp & 3;
    const uint32_t group = (uint32_t)(warp - 3) >> 2;     // warps 3..6 -> 0, 7..10 -> 1
    const int row = quarter * 32 + lane;
    int cur_q = -1;
    float wv[kIdxHeads];
    QueryInfo sc;
    sc.cache = qc;
    for (uint32_t it = 0;; it++) {
      if (abort_flag) break;
      uint32_t T;
      if (!ring_get(unit_ring, it, T, abort_flag)) { fail(); break; }   // every entry: the last may be either parity
      if (T == kDone) break;
      if (!POOL && (it & 1) != group) continue;
      const uint32_t acc = POOL ? (it & 1) : group;
      const int cur_u = (int)(T % upq), nq = (int)(T / upq);
      const uint32_t s = it % kScStages, r = it / kScStages;
      auto load_w = [&]() {
        const float4 *wp = reinterpret_cast<const float4 *>(P.w + (int64_t)nq * kIdxHeads);
#pragma unroll
        for (int i = 0; i < 8; i++) {
          const float4 v = __ldg(wp + i);
          wv[4 * i] = v.x;
          wv[4 * i + 1] = v.y;
          wv[4 * i + 2] = v.z;
          wv[4 * i + 3] = v.w;
        }
        cur_q = nq;
      };
      int pb[kSub] = {};
      if constexpr (POOL) {
        // Pool mode changes query on every unit: every global load the unit's
        // epilogue needs (the query's weights, the block id of each of this
        // lane's four entries; its sequence and length are in shared memory)
        // goes out before the wait for its MMA, so that their latencies
        // overlap it and one another.
        sc.prefetch(P, nq);
        if (nq != cur_q) load_w();
        const int32_t *pl = P.pool + (int64_t)nq * kPoolBlocks;
#pragma unroll
        for (int j = 0; j < kSub; j++) pb[j] = __ldg(pl + ((cur_u * kUnit + row + j * 128) >> 3));
        if (!ptx::mbar_wait(&done_bar[s], r & 1)) { fail(); break; }
        sc.set(P, nq, cur_u, false);
      } else {
        sc.set(P, nq, cur_u, false);
        if (nq != cur_q) load_w();
        if (!ptx::mbar_wait(&done_bar[s], r & 1)) { fail(); break; }
      }
      ptx::tc_fence_after();
      const uint32_t ta = tmem + ((uint32_t)(quarter * 32) << 16) + acc * (kSub * 32);
      float *out = P.scores + (int64_t)sc.q * P.stride;
      // entry i = i0 + 128 j of the unit (j = 0..3)
      // stores the score of entry i (sub-tile j); true if the entry is valid
      auto store = [&](int64_t i, int j, float v) -> bool {
        if (!POOL) {
          if (i < sc.nv) out[i] = v;
          return i < sc.nv;
        } else {
          const int b = j == 0 ? pb[0] : j == 1 ? pb[1] : j == 2 ? pb[2] : pb[3];   // (registers)
          const bool ok = b >= 0 && (int64_t)b * kBlock < P.n_max && (int64_t)b * kBlock + (i & 7) < sc.nv;
          out[i] = ok ? v : -INFINITY;
          return ok;
        }
      };
      const int64_t i0 = (int64_t)cur_u * kUnit + row;
      uint32_t umax = 0u;                             // smax_mode 3: the quarter's maximum key
#pragma unroll 1
      for (int h2 = 0; h2 < kSub / 2; h2++) {         // two sub-tiles (64 columns) at a time
        uint32_t d0[32], d1[32];
        ptx::tmem_ld_32x32b_x32(ta + h2 * 64, d0);
        ptx::tmem_ld_32x32b_x32(ta + h2 * 64 + 32, d1);
        ptx::tmem_wait_ld();
        if (h2 == kSub / 2 - 1) {
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&acc_empty[acc]);
        }
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int h = 0; h < kIdxHeads; h++) {
          s0 = fmaf(wv[h], fmaxf(__uint_as_float(d0[h]), 0.f), s0);
          s1 = fmaf(wv[h], fmaxf(__uint_as_float(d1[h]), 0.f), s1);
        }
        const bool ok0 = store(i0 + h2 * 256, 2 * h2, s0);
        const bool ok1 = store(i0 + h2 * 256 + 128, 2 * h2 + 1, s1);
        if constexpr (POOL && SMAX == 1) {
          // pool mode: the maximum order key of each gathered 8-entry block
          // (8 consecutive TMEM lanes; 0 when none of its entries is valid),
          // for the selection in the pool that follows
          uint32_t k0 = ok0 ? order_key(s0) : 0u, k1 = ok1 ? order_key(s1) : 0u;
#pragma unroll
          for (int o = 1; o < kBlock; o <<= 1) {
            k0 = max(k0, __shfl_xor_sync(0xFFFFFFFFu, k0, o));
            k1 = max(k1, __shfl_xor_sync(0xFFFFFFFFu, k1, o));
          }
          if ((lane & (kBlock - 1)) == 0) {
            uint32_t *bm = P.gmax + (int64_t)sc.q * P.gstride + (int64_t)cur_u * (kUnit / kBlock);
            bm[(2 * h2) * (128 / kBlock) + quarter * (32 / kBlock) + lane / kBlock] = k0;
            bm[(2 * h2 + 1) * (128 / kBlock) + quarter * (32 / kBlock) + lane / kBlock] = k1;
          }
        } else if constexpr (SMAX != 0) {
          // order keys of this lane's two entries (0 if not visible)
          const uint32_t k0 = i0 + h2 * 256 < sc.nv ? order_key(s0) : 0u;
          const uint32_t k1 = i0 + h2 * 256 + 128 < sc.nv ? order_key(s1) : 0u;
          // 32 consecutive entries per warp and sub-tile
          uint32_t *gm = SMAX == 2 ? P.smax + (int64_t)sc.q * P.sstride : P.gmax + (int64_t)sc.q * P.gstride;
          const uint32_t g0 = __reduce_max_sync(0xFFFFFFFFu, k0), g1 = __reduce_max_sync(0xFFFFFFFFu, k1);
          if (lane == 0) {
            const int64_t e0 = (int64_t)cur_u * kUnit + h2 * 256 + quarter * 32;
            gm[e0 >> 5] = g0;
            gm[(e0 + 128) >> 5] = g1;
          }
          umax = max(umax, max(g0, g1));
        }
      }
      if (SMAX == 3 && lane == 0) P.smax[(int64_t)sc.q * P.sstride + (int64_t)cur_u * 4 + quarter] = umax;
    }
  }
  __syncthreads();
  if (abort_flag) {
    // A wait ran out.  Before the CTA gives its tensor memory back and exits,
    // nothing it started may still be running: the copies of the last
    // kScStages iterations the producer issued (waited on their barriers;
    // pool mode: every gathering lane waits for its own asynchronous copies)
    // and the MMAs and scale-factor copies (each issuer commits once more).
    // All bounded.
    if (warp == 0 && lane == 0) {
      for (int i = max(0, armed_sh - kScStages); i < armed_sh; i++)
        ptx::mbar_wait(&full_bar[i % kScStages], (uint32_t)(i / kScStages) & 1);
    }
    if (warp == 0 || (POOL && (warp >= kScGather0 || (warp >= kScGather1 && warp < kScGather1 + 4))))
      asm volatile("cp.async.wait_all;" ::: "memory");
    if (lane == 0 && (warp == 1 || warp == 2 || warp == kScMmaWarp2)) ptx::tc_commit(&drain_bar);
    ptx::mbar_wait(&drain_bar, 0);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kScTmemCols);
  }
}

// ---------------------------------------------------------------- multi-query
// Several queries of one sequence decoded together (draft positions of one
// step: helix.ml, DeepSeek V4.1 Flash, section on DSpark, which proposes five
// future positions at once) see the same keys, so a group of G consecutive
// queries of one sequence is scored in one pass over the keys: the G queries'
// 32 heads each are the MMA's N = 32 G columns, and every key unit is read once
// per group instead of once per query.  The accumulators are G times wider, so
// units are 128 entries, with two accumulators of 32 G <= 192 TMEM columns
// (MMA and epilogue overlap) and 20 stages of 8.5 KB in flight; a CTA takes
// its units in adjacent pairs, each pair one bulk copy.
// Roles (384 threads): warp 0 producer, warp 1 MMA issuer (lane 0) and TMEM
// owner, warp 2 scale factors, warp 3 idle, warps 4..11 epilogue in two groups
// of four taking alternate units (warp w: TMEM lane quarter w % 4), each group
// reading only its own units' entries of the ring.  A query's
// scale factors sit in TMEM as rows of B: head h of the group's query g (row
// 32 g + h) at lane h, 32-bit word g (words 4..7 in the next four columns), as
// the key rows of A do.
constexpr int kMqUnit = 128;
constexpr int kMqStages = 20;
constexpr int kMqNibBytes = 8192;                             // a stage's nibbles: [stage][8 KB]
constexpr int kMqStageBytes = kMqNibBytes + 512;               // and its key scales, after all nibbles
constexpr int kMqSfaBase = kMqStages * kMqNibBytes;
constexpr int kMqMaxG = 6;                                   // N = 32 G <= 192
constexpr int kMqSlots = 2;
constexpr int kMqQOffSFB = kMqMaxG * 2048;                    // then two 32 x 16-B scale blocks
constexpr int kMqSlotBytes = kMqQOffSFB + 1024;
constexpr int kMqSmem = kMqStages * kMqStageBytes + kMqSlots * kMqSlotBytes;
constexpr int kMqThreads = 384;
// ring of published units: the producer, gated by the MMA of the unit
// kMqStages back, may run that far ahead of the MMA, and the epilogue trails
// the MMA by up to two units, so the ring holds more than kMqStages + 2
constexpr int kMqRing = 32;
static_assert(kMqRing > kMqStages + 3, "ring of published units (and the second end mark)");
constexpr uint32_t kMqColSFA = 2 * kMqMaxG * 32;              // after the two accumulators
constexpr uint32_t kMqColSFB = kMqColSFA + kMqStages * 4;
static_assert(kMqNibBytes % 512 == 0 && kMqSlotBytes % 512 == 0, "64B-swizzled tiles need 512-B alignment");
static_assert(kMqStages % 2 == 0, "unit pairs take stages s, s + 1 with s even");
static_assert(kMqColSFB + kMqSlots * 8 <= kScTmemCols, "TMEM columns");
static_assert(kMqSmem + 1024 <= 227 * 1024, "shared memory");
static_assert(kMqStages % 2 == 0, "a stage's done barrier also marks its accumulator full");
static_assert(kMqMaxG == kMaxQueryGroup, "the query-group limit of the C ABI");

// The group and unit of a schedule position T, for positions that only grow:
// the division runs only when T leaves the current group (every role runs
// this per unit, on sub-partitions shared with the epilogue's arithmetic).
struct GroupOf {
  uint32_t upq, base = 0;
  int g = -1;
  __device__ explicit GroupOf(uint32_t units_per_q) : upq(units_per_q) {}
  __device__ int group(uint32_t T) {
    if (g < 0 || T - base >= upq) {
      g = (int)(T / upq);
      base = (uint32_t)g * upq;
    }
    return g;
  }
  __device__ int unit(uint32_t T) const { return (int)(T - base); }
};

// G (the queries of a group) is a template parameter so that the epilogue's
// loops over the queries unroll into independent running sums.
template <int G>
__global__ void __launch_bounds__(kMqThreads, 1) index_score_mq_kernel(ScoreTcArgs P) {
  extern __shared__ __align__(1024) unsigned char mq_smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(mq_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  unsigned char *qslots = smem + kMqStages * kMqStageBytes;
  __shared__ __align__(8) uint64_t full_bar[kMqStages], sf_bar[kMqStages], done_bar[kMqStages];
  __shared__ __align__(8) uint64_t acc_empty[2];
  __shared__ __align__(8) uint64_t drain_bar;      // after a wait ran out: the tcgen05 issuers' last commits
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_flag;
  __shared__ int armed_sh;                         // iterations whose copies the producer issued
  __shared__ volatile unsigned long long unit_ring[kMqRing];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t N = 32u * (uint32_t)G;
  griddep_wait();
  griddep_launch();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kMqStages; s++) {
      ptx::mbar_init(&full_bar[s], 1);
      ptx::mbar_init(&sf_bar[s], 1);
      ptx::mbar_init(&done_bar[s], 1);
    }
    ptx::mbar_init(&acc_empty[0], 4);
    ptx::mbar_init(&acc_empty[1], 4);
    ptx::mbar_init(&drain_bar, 2);                  // the MMA issuer and the scale-factor warp
    for (int i = 0; i < kMqRing; i++) unit_ring[i] = ~0ull;
    abort_flag = 0;
    armed_sh = 0;
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
  const int n_groups = P.n_q / G;
  const uint32_t total_units = (uint32_t)n_groups * (uint32_t)P.units_per_q;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The CTA's units come in adjacent pairs (2b, 2b + 1 for b = blockIdx.x,
    // blockIdx.x + gridDim.x, ...), so that one bulk copy (16 KB) and one
    // 16-B asynchronous copy per lane bring both, into stages s, s + 1 (s
    // even), counted on stage s's barrier; the second stage's barrier then
    // takes a plain arrival (its consumers wait on stage s's first, in order).
    // The producer shares its sub-partition with two epilogue warps, and its
    // instructions per unit set the kernel's pace when they are many (units of
    // one at a time, a division per unit and two bulk copies: 312 us per
    // 8 x 1M x 5 launch, against 261 us with the pairs and the steps below
    // together), so it looks one unit ahead and does little per unit.
    const uint64_t policy = ptx::policy_evict_first();
    QuerySlotsT<kMqSlots> qs;
    GroupOf go((uint32_t)P.units_per_q);
    int cur_g = -1;
    int64_t row_g = 0;                             // the looked-at group's first key row
    int nv_max = -1;
    struct Found {
      uint32_t T;
      int g;
      int64_t r0;                                  // the unit's first key row
    };
    // the first valid unit at or after schedule position T
    auto find = [&](uint32_t T) -> Found {
      for (;;) {
        if (T >= total_units) return Found{kDone, -1, 0};
        const int gi = go.group(T), u = go.unit(T);
        if (gi != cur_g) {
          // the group's sequence (all G queries must share it) and its
          // longest visible length; a group breaking this is skipped
          cur_g = gi;
          int sq = -1, nm = -1, ok = 1;
          for (int g = 0; g < G; g++) {
            const int q = gi * G + g, s_ = __ldg(P.q_seq + q), v = __ldg(P.n_vis + q);
            if (g == 0) sq = s_;
            if (s_ != sq || v < 0 || (int64_t)v > P.n_max) ok = 0;
            nm = max(nm, v);
          }
          if (sq < 0 || sq >= P.n_seq) ok = 0;
          if (!ok && lane == 0 && u == 0) record_error(P.status, CSA2_ERR_BOUNDS);
          row_g = (int64_t)sq * P.n_max;
          nv_max = ok ? nm : -1;
        }
        // a unit that starts before n_vis ends within n_max (n_max % 128 == 0)
        if (nv_max >= 0 && u * kMqUnit < nv_max) return Found{T, gi, row_g + (int64_t)u * kMqUnit};
        T = (T & 1u) ? T + 2u * gridDim.x - 1u : T + 1u;
      }
    };
    Found nx = find(2u * blockIdx.x);
    bool second = false;                           // this unit's data came with the previous one's
    for (uint32_t it = 0;; it++) {
      if (abort_flag) break;
      const Found cu = nx;
      if (lane == 0) unit_ring[it % kMqRing] = ((unsigned long long)it << 32) | cu.T;
      if (cu.T == kDone) {
        // the end, also for the epilogue group that reads only the other entries
        if (lane == 0) unit_ring[(it + 1) % kMqRing] = ((unsigned long long)(it + 1) << 32) | kDone;
        break;
      }
      nx = find((cu.T & 1u) ? cu.T + 2u * gridDim.x - 1u : cu.T + 1u);
      const uint32_t s = it % kMqStages, r = it / kMqStages;
      const bool fresh = qs.step(cu.g, (int)it);
      if (second) {
        second = false;
        if (lane == 0) {
          ptx::mbar_arrive(&full_bar[s]);
          armed_sh = (int)it + 1;
        }
        __syncwarp();
        continue;
      }
      // a pair: the next unit is adjacent, in the same group (so not a fresh one)
      const bool pair = (s & 1u) == 0u && nx.T == cu.T + 1u && nx.g == cu.g;
      // stage s (and s + 1) free: MMAs complete in order, so the later suffices
      if (!ptx::mbar_wait(&done_bar[pair ? s + 1 : s], (r & 1) ^ 1)) { fail(); break; }
      if (fresh) {
        // the slot's previous user (MMAs complete in order: its last unit)
        const int pu = qs.prev_user();
        if (pu >= 0 && pu + kMqStages > (int)it &&
            !ptx::mbar_wait(&done_bar[pu % kMqStages], (uint32_t)(pu / kMqStages) & 1)) { fail(); break; }
      }
      unsigned char *qd = qslots + qs.slot * kMqSlotBytes;
      // the units' key scales (512 B each) come as the lanes' 16-B asynchronous
      // copies, each lane counted into the stage's barrier, not as more bulk
      // copies: the bulk-copy unit spends a fixed time per instruction
      const unsigned char *ks = P.key_scale + cu.r0 * 4;
      ptx::cp_async16(smem + kMqSfaBase + s * 512 + lane * 16, ks + lane * 16);
      if (pair) ptx::cp_async16(smem + kMqSfaBase + s * 512 + 512 + lane * 16, ks + 512 + lane * 16);
      ptx::cp_async_arrive(&full_bar[s]);
      __syncwarp();
      if (lane == 0) {
        const uint32_t nbytes = pair ? 16384u : 8192u;
        const uint32_t qbytes = fresh ? (uint32_t)G * (2048 + 128) : 0u;
        ptx::mbar_arrive_expect_tx(&full_bar[s], nbytes + qbytes);
        if (fresh) {
          const int64_t q0 = (int64_t)cu.g * G;
          ptx::bulk_load(qd, P.q_nib + q0 * kIdxHeads * 64, (uint32_t)G * 2048, &full_bar[s]);
          ptx::bulk_load(qd + kMqQOffSFB, P.q_scale + q0 * kIdxHeads * 4, (uint32_t)G * 128, &full_bar[s]);
        }
        ptx::bulk_load_hint(smem + s * kMqNibBytes, P.key_nib + cu.r0 * 64, nbytes, &full_bar[s], policy);
        armed_sh = (int)it + 1;
      }
      __syncwarp();
      second = pair;
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ scale-factor warp
    QuerySlotsT<kMqSlots> qs;
    GroupOf go((uint32_t)P.units_per_q);
    for (uint32_t it = 0;; it++) {
      if (abort_flag) break;
      uint32_t T;
      if (!ring_get<kMqRing>(unit_ring, it, T, abort_flag)) { fail(); break; }
      if (T == kDone) break;
      const uint32_t s = it % kMqStages, r = it / kMqStages;
      const bool fresh = qs.step(go.group(T), (int)it);
      if (!ptx::mbar_wait(&full_bar[s], r & 1)) { fail(); break; }
      unsigned char *qd = qslots + qs.slot * kMqSlotBytes;
      if (fresh) {
        // the queries' scales, [g][head] words as loaded -> block g / 4, line
        // head, word g % 4 (zero for g >= G)
        uint32_t *sfb = reinterpret_cast<uint32_t *>(qd + kMqQOffSFB);
        uint32_t vb[8];
#pragma unroll
        for (int g = 0; g < 8; g++) vb[g] = g < G ? sfb[g * 32 + lane] : 0u;
        __syncwarp();
#pragma unroll
        for (int g = 0; g < 8; g++) sfb[(g >> 2) * 128 + lane * 4 + (g & 3)] = vb[g];
      }
      // key scales -> tcgen05.cp layout: 16-B line m0 holds rows m0, m0+32, m0+64, m0+96
      uint32_t *sfa = reinterpret_cast<uint32_t *>(smem + kMqSfaBase + s * 512);
      uint32_t va[4];
#pragma unroll
      for (int i = 0; i < 4; i++) va[i] = sfa[i * 32 + lane];
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 4; i++) sfa[lane * 4 + i] = va[i];
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        ptx::tc_fence_after();
        if (fresh) {
          const uint32_t sb = ptx::smem_u32(qd + kMqQOffSFB);
          ptx::tc_cp_32x128b_warpx4(tmem + kMqColSFB + qs.slot * 8, ptx::smem_desc(sb, 0, 128, 0));
          if (G > 4) ptx::tc_cp_32x128b_warpx4(tmem + kMqColSFB + qs.slot * 8 + 4, ptx::smem_desc(sb + 512, 0, 128, 0));
        }
        ptx::tc_cp_32x128b_warpx4(tmem + kMqColSFA + s * 4, ptx::smem_desc(ptx::smem_u32(sfa), 0, 128, 0));
        ptx::tc_commit(&sf_bar[s]);
      }
      __syncwarp();
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (lane 0)
    if (lane == 0) {
      const uint32_t idesc0 = idesc_mxf4_m128(0, N), idesc1 = idesc_mxf4_m128(2, N);
      QuerySlotsT<kMqSlots> qs;
      GroupOf go((uint32_t)P.units_per_q);
      for (uint32_t it = 0;; it++) {
        if (abort_flag) break;
        uint32_t T;
        if (!ring_get<kMqRing>(unit_ring, it, T, abort_flag)) { fail(); break; }
        if (T == kDone) break;
        qs.step(go.group(T), (int)it);
        const uint32_t s = it % kMqStages, r = it / kMqStages, a = it & 1, ra = it >> 1;
        if (!ptx::mbar_wait(&sf_bar[s], r & 1) || !ptx::mbar_wait(&acc_empty[a], (ra & 1) ^ 1)) { fail(); break; }
        ptx::tc_fence_after();
        const uint64_t ad = ptx::smem_desc(ptx::smem_u32(smem + s * kMqNibBytes), 16, 512, 4);
        const uint64_t bd = ptx::smem_desc(ptx::smem_u32(qslots + qs.slot * kMqSlotBytes), 16, 512, 4);
        const uint32_t t_sfa = tmem + kMqColSFA + s * 4, t_sfb = tmem + kMqColSFB + qs.slot * 8;
        const uint32_t d = tmem + a * N;
        ptx::tc_mma_mxf4(d, ad, bd, idesc0, t_sfa, t_sfb, 0u);
        ptx::tc_mma_mxf4(d, ad + 2, bd + 2, idesc1, t_sfa, t_sfb, 1u);   // +32 B along K
        ptx::tc_commit(&done_bar[s]);
      }
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ epilogue
    // group grp (warps 4+4 grp .. 7+4 grp) takes the units with it % 2 == grp
    // and owns accumulator grp (see the single-query kernel for why waiting on
    // done_bar is unambiguous)
    // Each warp keeps its group's G x 32 weights in shared memory (read back
    // four at a time, the same address in every lane) and the queries'
    // visible lengths in registers, both reloaded when the group changes.
    const int quarter = warp & 3;
    const uint32_t grp = (uint32_t)(warp - 4) >> 2;
    __shared__ __align__(16) float w_sm[8][kMqMaxG * 32];
    float *wsm = w_sm[warp - 4];
    int cur_gi = -1;
    int nvq[G];
    GroupOf go((uint32_t)P.units_per_q);
    for (uint32_t it = grp;; it += 2) {             // this group's units only
      if (abort_flag) break;
      uint32_t T;
      if (!ring_get<kMqRing>(unit_ring, it, T, abort_flag)) { fail(); break; }
      if (T == kDone) break;
      const int gi = go.group(T), u = go.unit(T);
      const uint32_t s = it % kMqStages, r = it / kMqStages;
      if (gi != cur_gi) {
        for (int i = lane; i < G * 32; i += 32) wsm[i] = __ldg(P.w + (int64_t)gi * G * kIdxHeads + i);
#pragma unroll
        for (int g = 0; g < G; g++) nvq[g] = __ldg(P.n_vis + gi * G + g);
        __syncwarp();
        cur_gi = gi;
      }
      if (!ptx::mbar_wait(&done_bar[s], r & 1)) { fail(); break; }
      ptx::tc_fence_after();
      const int64_t e = (int64_t)u * kMqUnit + quarter * 32 + lane;
      const uint32_t ta = tmem + ((uint32_t)(quarter * 32) << 16) + grp * N;
      // up to three queries at a time: their 32 columns each in one load
      // apiece and one wait (each TMEM round trip costs hundreds of cycles),
      // then four running sums per query
#pragma unroll
      for (int g0 = 0; g0 < G; g0 += 3) {
        constexpr int kB = 3;
        const int nb = G - g0 < kB ? G - g0 : kB;
        uint32_t d[kB][32];
#pragma unroll
        for (int b = 0; b < kB; b++)
          if (b < nb) ptx::tmem_ld_32x32b_x32(ta + (g0 + b) * 32, d[b]);
        ptx::tmem_wait_ld();
        // four running sums per query (heads i mod 4), as two pairs: the
        // packed two-lane FMA halves the FMA instructions (the epilogue's
        // arithmetic, 160 ReLU-weight-add steps per entry at G = 5, is what
        // the units wait on once the producer keeps ahead)
        float2 acc[kB][2];
#pragma unroll
        for (int b = 0; b < kB; b++) acc[b][0] = acc[b][1] = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < 8; i++) {
#pragma unroll
          for (int b = 0; b < kB; b++) {
            if (b < nb) {
              const float4 wv = reinterpret_cast<const float4 *>(wsm + (g0 + b) * kIdxHeads)[i];
              const float2 r01 = make_float2(fmaxf(__uint_as_float(d[b][4 * i]), 0.f),
                                             fmaxf(__uint_as_float(d[b][4 * i + 1]), 0.f));
              const float2 r23 = make_float2(fmaxf(__uint_as_float(d[b][4 * i + 2]), 0.f),
                                             fmaxf(__uint_as_float(d[b][4 * i + 3]), 0.f));
              acc[b][0] = __ffma2_rn(make_float2(wv.x, wv.y), r01, acc[b][0]);
              acc[b][1] = __ffma2_rn(make_float2(wv.z, wv.w), r23, acc[b][1]);
            }
          }
        }
#pragma unroll
        for (int b = 0; b < kB; b++) {
          if (b < nb) {
            const int q = gi * G + g0 + b;
            if (e < nvq[g0 + b])
              P.scores[(int64_t)q * P.stride + e] = (acc[b][0].x + acc[b][0].y) + (acc[b][1].x + acc[b][1].y);
          }
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&acc_empty[grp]);
    }
  }
  __syncthreads();
  if (abort_flag) {
    // a wait ran out: as in the single-query kernel, the producer's last
    // copies and the issuers' tcgen05 operations finish before TMEM goes back
    if (warp == 0) asm volatile("cp.async.wait_all;" ::: "memory");
    if (warp == 0 && lane == 0) {
      for (int i = max(0, armed_sh - kMqStages); i < armed_sh; i++)
        ptx::mbar_wait(&full_bar[i % kMqStages], (uint32_t)(i / kMqStages) & 1);
    }
    if (lane == 0 && (warp == 1 || warp == 2)) ptx::tc_commit(&drain_bar);
    ptx::mbar_wait(&drain_bar, 0);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kScTmemCols);
  }
}

// ---------------------------------------------------------------- bounded-wait check
// One warp takes tensor memory, waits on a barrier that nothing completes with
// a short wall-time limit, records CSA2_ERR_TIMEOUT, gives the memory back and
// exits: the path every kernel here takes when a wait runs out, with nothing
// asynchronous in flight.
__global__ void __launch_bounds__(32, 1) bounded_wait_check_kernel(int *status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t never;
  __shared__ uint32_t tmem_sh;
  griddep_wait();
  griddep_launch();
  if (threadIdx.x == 0) {
    ptx::mbar_init(&never, 1);                       // its one arrival never comes
    ptx::fence_mbar_init();
  }
  ptx::tmem_alloc(&tmem_sh, 32);
  ptx::tc_fence_before();
  __syncwarp();
  ptx::tc_fence_after();
  const uint32_t tmem = tmem_sh;
  if (!ptx::mbar_wait(&never, 0, limit_ns) && threadIdx.x == 0) record_error(status, CSA2_ERR_TIMEOUT);
  ptx::tc_fence_before();
  __syncwarp();
  ptx::tc_fence_after();
  ptx::tmem_dealloc(tmem, 32);
}

cudaError_t launch_bounded_wait_check(int *status, unsigned long long limit_ns, cudaStream_t st) {
  return launch_pdl(bounded_wait_check_kernel, dim3(1), dim3(32), 0, st, 1u, status, limit_ns);
}

// ---------------------------------------------------------------- host side
cudaError_t launch_index_score_tc(const uint8_t *key_nib, const uint8_t *key_scale, int64_t n_max, int n_seq,
                                  const uint8_t *q_nib, const uint8_t *q_scale, const float *w, const int32_t *q_seq,
                                  const int32_t *n_vis, int n_q, const int32_t *pool, float *scores, int64_t stride,
                                  int *status, cudaStream_t st, const LongRowWs *W, int smax_mode) {
  ScoreTcArgs P;
  P.smax = W ? W->smax : nullptr;
  P.sstride = W ? W->sstride : 0;
  P.gmax = W ? W->gmax : nullptr;
  P.gstride = W ? W->gstride : 0;
  P.hflag = W && pool == nullptr ? W->hand.flag : nullptr;
  P.steal = W && pool == nullptr ? W->steal : nullptr;
  P.call_id = W ? W->call_id : 0u;
  P.smax_mode = pool == nullptr && W != nullptr && (smax_mode == 2 || (smax_mode == 3 && W->gmax != nullptr))
                    ? smax_mode : 0;
  if (pool != nullptr && W != nullptr && smax_mode == 1 && W->gmax != nullptr) P.smax_mode = 1;   // block maxima
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
  P.units_per_q = pool ? kPoolSlots / kUnit : (int)((n_max + kUnit - 1) / kUnit);
  const int64_t total_units = (int64_t)n_q * P.units_per_q;
  P.status = status;
  const size_t smem = (size_t)kScSmem + 1024;
  const int dev = current_device();
  static std::atomic<int> attr_done[kMaxDevices];
  const cudaError_t e = once_per_device(attr_done, dev, [&] {
    const cudaError_t es[5] = {
        cudaFuncSetAttribute(index_score_tc_kernel<false, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem),
        cudaFuncSetAttribute(index_score_tc_kernel<false, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem),
        cudaFuncSetAttribute(index_score_tc_kernel<false, 3>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem),
        cudaFuncSetAttribute(index_score_tc_kernel<true, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem),
        cudaFuncSetAttribute(index_score_tc_kernel<true, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)};
    for (cudaError_t x : es)
      if (x != cudaSuccess) return x;
    return cudaSuccess;
  });
  if (e != cudaSuccess) return e;
  const int n_sm = device_sm_count(dev);
  const int64_t grid = total_units < n_sm ? total_units : n_sm;
  // runs of consecutive units (Full mode without claims): the longest run,
  // up to kMaxRun, that leaves the busiest CTA no more units than a stride of
  // single units would
  P.run = 1;
  const bool steal = pool == nullptr && P.steal != nullptr && total_units >= (int64_t)kStealMinRounds * grid;
  if (pool == nullptr && !steal && grid > 0) {
    const int64_t most = (total_units + grid - 1) / grid;
    for (int r = kMaxRun; r > 1; r--) {
      const int64_t groups = (total_units + r - 1) / r;
      if ((groups + grid - 1) / grid * r <= most) {
        P.run = r;
        break;
      }
    }
  }
  const dim3 g((unsigned)grid), b(kScThreads);
  if (pool != nullptr && P.smax_mode == 1) return launch_pdl(index_score_tc_kernel<true, 1>, g, b, smem, st, 1u, P);
  if (pool != nullptr) return launch_pdl(index_score_tc_kernel<true, 0>, g, b, smem, st, 1u, P);
  if (P.smax_mode == 3) return launch_pdl(index_score_tc_kernel<false, 3>, g, b, smem, st, 1u, P);
  if (P.smax_mode == 2) return launch_pdl(index_score_tc_kernel<false, 2>, g, b, smem, st, 1u, P);
  return launch_pdl(index_score_tc_kernel<false, 0>, g, b, smem, st, 1u, P);
}

}  // namespace csa2

namespace csa2 {

cudaError_t launch_index_score_mq(const uint8_t *key_nib, const uint8_t *key_scale, int64_t n_max, int n_seq,
                                  const uint8_t *q_nib, const uint8_t *q_scale, const float *w, const int32_t *q_seq,
                                  const int32_t *n_vis, int n_q, int group, float *scores, int64_t stride,
                                  int *status, cudaStream_t st) {
  ScoreTcArgs P = {};
  P.key_nib = key_nib;
  P.q_nib = q_nib;
  P.key_scale = key_scale;
  P.q_scale = q_scale;
  P.w = w;
  P.q_seq = q_seq;
  P.n_vis = n_vis;
  P.pool = nullptr;
  P.scores = scores;
  P.stride = stride;
  P.n_max = n_max;
  P.n_seq = n_seq;
  P.n_q = n_q;
  P.units_per_q = (int)((n_max + kMqUnit - 1) / kMqUnit);
  P.status = status;
  const int64_t total_units = (int64_t)(n_q / group) * P.units_per_q;
  const size_t smem = (size_t)kMqSmem + 1024;
  const int dev = current_device();
  static std::atomic<int> attr_done[kMaxDevices];
  const cudaError_t e = once_per_device(attr_done, dev, [&] {
    cudaError_t r = cudaSuccess, ri;
    ri = cudaFuncSetAttribute(index_score_mq_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    r = r == cudaSuccess ? ri : r;
    ri = cudaFuncSetAttribute(index_score_mq_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    r = r == cudaSuccess ? ri : r;
    ri = cudaFuncSetAttribute(index_score_mq_kernel<3>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    r = r == cudaSuccess ? ri : r;
    ri = cudaFuncSetAttribute(index_score_mq_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    r = r == cudaSuccess ? ri : r;
    ri = cudaFuncSetAttribute(index_score_mq_kernel<5>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    r = r == cudaSuccess ? ri : r;
    ri = cudaFuncSetAttribute(index_score_mq_kernel<6>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    return r == cudaSuccess ? ri : r;
  });
  if (e != cudaSuccess) return e;
  const int n_sm = device_sm_count(dev);
  const dim3 grid((unsigned)(total_units < n_sm ? total_units : n_sm)), block(kMqThreads);
  switch (group) {
    case 1: return launch_pdl(index_score_mq_kernel<1>, grid, block, smem, st, 1u, P);
    case 2: return launch_pdl(index_score_mq_kernel<2>, grid, block, smem, st, 1u, P);
    case 3: return launch_pdl(index_score_mq_kernel<3>, grid, block, smem, st, 1u, P);
    case 4: return launch_pdl(index_score_mq_kernel<4>, grid, block, smem, st, 1u, P);
    case 5: return launch_pdl(index_score_mq_kernel<5>, grid, block, smem, st, 1u, P);
    default: return launch_pdl(index_score_mq_kernel<6>, grid, block, smem, st, 1u, P);
  }
}

}  // namespace csa2
