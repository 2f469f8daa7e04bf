// Phase-level device helpers shared by the persistent engines: waiting for
// the end-of-phase flags of every CTA, sums of squares for the RMSNorm
// prologues, and the SiLU gate of the feed-forward epilogue.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "q4_device.cuh"

namespace q4 {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Wait until every CTA has published phase `tag`'s flag (or a later one)
// and return the sum of the sums of squares they carry, in a fixed order
// (the same in every CTA).  One warp per CTA polls; after the flags are
// seen, a fence orders later loads after the producers' writes.  Gives up
// after `limit` polls (status bit set).
static __device__ float wait_phase_flags(const unsigned long long* flags, unsigned tag, int lane, uint32_t limit,
                                  Control* ctl) {
  const int G = static_cast<int>(gridDim.x);
  float part[kMaxGrid / 32];
  bool ok = false;
  for (uint32_t it = 0; it < limit; ++it) {
    bool mine = true;
#pragma unroll
    for (int i = 0; i < kMaxGrid / 32; ++i) {
      part[i] = 0.f;
      if (lane + 32 * i < G) {
        const unsigned long long f = ld_relaxed_u64(flags + lane + 32 * i);
        mine &= static_cast<int>(static_cast<unsigned>(f >> 32) - tag) >= 0;
        part[i] = __uint_as_float(static_cast<unsigned>(f));
      }
    }
    if (__all_sync(0xffffffffu, mine)) {
      ok = true;
      break;
    }
    if (it > 16) __nanosleep(64);
  }
  if (!ok && lane == 0) atomicOr(&ctl->status, ST_FLAG_TIMEOUT);
  __threadfence();
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < kMaxGrid / 32; ++i) ss += part[i];
  return warp_sum(ss);
}

// Sum of a per-CTA sums-of-squares array written by an earlier launch.
__device__ __forceinline__ float sum_ss_array(const float* ss, int lane) {
  const int G = static_cast<int>(gridDim.x);
  float part = 0.f;
#pragma unroll
  for (int i = 0; i < kMaxGrid / 32; ++i)
    if (lane + 32 * i < G) part += __ldcg(ss + lane + 32 * i);
  return warp_sum(part);
}

// Sum of squares of a binary16 input vector (every warp on its own).
__device__ __forceinline__ float input_sumsq16(const Phase& ph, int lane) {
  float ss = 0.f;
  const uint4* p = reinterpret_cast<const uint4*>(ph.x_src);
  for (int i = lane; i < ph.k / 8; i += 32) {
    const uint4 u = __ldcg(p + i);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[t]));
      ss = fmaf(f.x, f.x, ss);
      ss = fmaf(f.y, f.y, ss);
    }
  }
  return warp_sum(ss);
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

}  // namespace q4
