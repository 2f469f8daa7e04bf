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
