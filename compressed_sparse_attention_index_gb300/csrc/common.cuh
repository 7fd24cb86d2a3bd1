// Shared device helpers of the CSA2 GB300 library (internal header).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "csa2.h"

namespace csa2 {

constexpr int kHeads = 64, kDim = 512, kRopeDim = 64, kRopeOff = 448;
constexpr int kIdxHeads = 32, kIdxDim = 128, kTopK = 512, kSwa = 128, kBlock = 8, kPoolBlocks = 2048;
constexpr int kPoolSlots = kPoolBlocks * kBlock;   // 16,384 candidate positions
constexpr int kKvBytes = 288, kIdxNibBytes = 64, kIdxScaleBytes = 4, kSwaBytes = 528;

// Sticky device status word (one per device, owned by api.cu and passed to the
// kernels as a pointer): the first error code recorded wins.
__device__ __forceinline__ void record_error(int *status, int code) { atomicCAS(status, 0, code); }

// ---- bf16 bit helpers (host-independent, exact) ----
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// E4M3 byte -> float (exact).  Codes 0x7F/0xFF (NaN) are never produced by the packers.
__device__ __forceinline__ float e4m3_to_float(uint32_t b) {
  uint32_t e = (b >> 3) & 15u, m = b & 7u;
  float v = (e == 0) ? (float)m * 0.001953125f                      // m * 2^-9
                     : __uint_as_float(((e + 120u) << 23) | (m << 20));  // (1+m/8) 2^(e-7)
  return (b & 0x80u) ? -v : v;
}

// E8M0 byte -> 2^(b-127) as float (exact, including the fp32 subnormal 2^-127).
__device__ __forceinline__ float e8m0_to_float(uint32_t b) {
  return b == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(b << 23);
}

// E2M1 nibble -> twice its value as a small integer in [-12, 12].
__device__ __forceinline__ int e2m1_x2(uint32_t nib) {
  // magnitudes x2: 0,1,2,3,4,6,8,12 packed as bytes
  const uint32_t lo = 0x03020100u, hi = 0x0C080604u;
  uint32_t m = nib & 7u;
  int v = (int)(((m < 4 ? lo : hi) >> (8 * (m & 3))) & 0xFFu);
  return (nib & 8u) ? -v : v;
}

// Order-preserving 32-bit key of a float score (-0 treated as +0).
__device__ __forceinline__ uint32_t order_key(float s) {
  uint32_t u = __float_as_uint(s == 0.0f ? 0.0f : s);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Programmatic dependent launch.  A kernel launched with the programmatic
// stream-serialisation attribute may start before the grid ahead of it on the
// stream has finished; griddep_wait() returns once that grid has completed and
// its memory is visible (at once when there is no such grid).  griddep_launch()
// lets the next grid on the stream start early.  Every kernel of this library
// waits before it reads anything that a grid still running may write, and
// signals only after its own wait, so a grid that starts early finds every
// grid two or more places ahead of it complete.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Iteration limit of a spin-wait on shared memory written by another warp.
constexpr long long kSpinLimit = 1LL << 26;


}  // namespace csa2
