// Tensor-core fragments of Q4_0 blocks (mma.sync m16n8k16, binary16 in,
// fp32 accumulate): exact binary16 values (q - 8) built in registers from
// the staged code bytes, and the matching order of the input x.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "q4_device.cuh"

namespace q4 {

// Programmatic dependent launch.  griddep_launch_dependents lets the next
// kernel of the stream (launched with programmatic stream serialisation) be
// scheduled once every CTA of this one has issued it; griddep_wait blocks
// until the kernels this one depends on have completed and their memory is
// visible.  Without that launch attribute both are no-ops.
__device__ __forceinline__ void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" :::); }
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void mma16816(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Exact binary16 (q - 8) for the 8 codes of one code word w (bytes 4t..4t+3
// of a block's code bytes: elements 4t..4t+3 low nibbles, 4t+16..4t+19 high).
// The code in the low mantissa bits of 1024 gives 1024 + q (or 1024 + 16 q for
// a high nibble); subtracting 1032 (or scaling by 1/16 and subtracting 72) is
// exact.  Output half2 pairs, elements (4t, 4t+2), (4t+1, 4t+3),
// (4t+16, 4t+18), (4t+17, 4t+19).
__device__ __forceinline__ void unpack_word(uint32_t w, uint32_t magic, uint32_t& l02, uint32_t& l13,
                                            uint32_t& h02, uint32_t& h13) {
  const uint32_t w8 = w >> 8;
  uint32_t a, b, c, d;
  asm("lop3.b32 %0, %1, 0x000F000F, %2, 0xEA;" : "=r"(a) : "r"(w), "r"(magic));
  asm("lop3.b32 %0, %1, 0x000F000F, %2, 0xEA;" : "=r"(b) : "r"(w8), "r"(magic));
  asm("lop3.b32 %0, %1, 0x00F000F0, %2, 0xEA;" : "=r"(c) : "r"(w), "r"(magic));
  asm("lop3.b32 %0, %1, 0x00F000F0, %2, 0xEA;" : "=r"(d) : "r"(w8), "r"(magic));
  const __half2 k1032 = __floats2half2_rn(1032.f, 1032.f);
  const __half2 k16 = __floats2half2_rn(0.0625f, 0.0625f);
  const __half2 k72 = __floats2half2_rn(-72.f, -72.f);
  __half2 A = __hsub2(*reinterpret_cast<__half2*>(&a), k1032);
  __half2 B = __hsub2(*reinterpret_cast<__half2*>(&b), k1032);
  __half2 C = __hfma2(*reinterpret_cast<__half2*>(&c), k16, k72);
  __half2 D = __hfma2(*reinterpret_cast<__half2*>(&d), k16, k72);
  l02 = *reinterpret_cast<uint32_t*>(&A);
  l13 = *reinterpret_cast<uint32_t*>(&B);
  h02 = *reinterpret_cast<uint32_t*>(&C);
  h13 = *reinterpret_cast<uint32_t*>(&D);
}

__device__ __forceinline__ float lo_half_f(uint32_t w) { return __low2float(*reinterpret_cast<const __half2*>(&w)); }
__device__ __forceinline__ float hi_half_f(uint32_t w) { return __high2float(*reinterpret_cast<const __half2*>(&w)); }

// One block pair (even block, odd block after it) of tile rows g and g + 8:
// rg, rh point at the pair's 36 bytes in the two staged rows.  ee/eh collect
// the even block (valid in lane quarter 0), og/oh the odd one (quarter 3).
__device__ __forceinline__ void pair_mma(const uint8_t* rg, const uint8_t* rh, int t, const uint4& xe, const uint4& xo,
                                         uint32_t magic, float& eg, float& eh, float& og, float& oh) {
  const uint32_t* pg = reinterpret_cast<const uint32_t*>(rg);
  const uint32_t* ph = reinterpret_cast<const uint32_t*>(rh);
  const uint32_t g0 = pg[t], g1 = pg[t + 1], go = pg[5 + t];
  const uint32_t h0 = ph[t], h1 = ph[t + 1], ho = ph[5 + t];
  uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
  // even block: its code bytes start 2 bytes into the pair, word t is a funnel of words t, t+1
  unpack_word(__funnelshift_r(g0, g1, 16), magic, a0, a1, a2, a3);
  unpack_word(__funnelshift_r(h0, h1, 16), magic, b0, b1, b2, b3);
  float c[4] = {0.f, 0.f, 0.f, 0.f};
  mma16816(c, a0, b0, a1, b1, xe.x, xe.y);
  mma16816(c, a2, b2, a3, b3, xe.z, xe.w);
  eg = fmaf(lo_half_f(g0), c[0], eg);   // quarter 0: word 0 starts with the even block's d
  eh = fmaf(lo_half_f(h0), c[2], eh);
  // odd block: code words 5..8 of the pair, 4-byte aligned
  unpack_word(go, magic, a0, a1, a2, a3);
  unpack_word(ho, magic, b0, b1, b2, b3);
  float e[4] = {0.f, 0.f, 0.f, 0.f};
  mma16816(e, a0, b0, a1, b1, xo.x, xo.y);
  mma16816(e, a2, b2, a3, b3, xo.z, xo.w);
  og = fmaf(hi_half_f(g1), e[0], og);   // quarter 3: word 4 ends with the odd block's d
  oh = fmaf(hi_half_f(h1), e[2], oh);
}

// The B fragments of one block for batch column `col`: x elements in the
// k order of unpack_word (zero for columns beyond the batch).
__device__ __forceinline__ void x_frags(const __half* x, int k, int batch, int col, int blk, int t, uint32_t& s0b0,
                                        uint32_t& s0b1, uint32_t& s1b0, uint32_t& s1b1) {
  if (col < batch) {
    const uint2 lo = *reinterpret_cast<const uint2*>(x + static_cast<size_t>(col) * k + blk * 32 + 4 * t);
    const uint2 hi = *reinterpret_cast<const uint2*>(x + static_cast<size_t>(col) * k + blk * 32 + 16 + 4 * t);
    s0b0 = __byte_perm(lo.x, lo.y, 0x5410);   // elements 4t, 4t+2
    s0b1 = __byte_perm(lo.x, lo.y, 0x7632);   // elements 4t+1, 4t+3
    s1b0 = __byte_perm(hi.x, hi.y, 0x5410);
    s1b1 = __byte_perm(hi.x, hi.y, 0x7632);
  } else {
    s0b0 = s0b1 = s1b0 = s1b1 = 0u;
  }
}

// Code word t of block b of a staged row and its scale.
__device__ __forceinline__ uint32_t code_word(const uint8_t* row, int b, int t) {
  const uint8_t* p = row + b * kBlockBytes + 2 + 4 * t;
  if (b & 1) return *reinterpret_cast<const uint32_t*>(p);   // 4-byte aligned for odd blocks
  const uint32_t lo = *reinterpret_cast<const uint32_t*>(p - 2);
  const uint32_t hi = *reinterpret_cast<const uint32_t*>(p + 2);
  return __funnelshift_r(lo, hi, 16);
}

__device__ __forceinline__ float row_scale(const uint8_t* row, int b) {
  return __half2float(*reinterpret_cast<const __half*>(row + b * kBlockBytes));
}

}  // namespace q4
