// Device-side filler for seeded synthetic inputs (libq4synth.so).  It draws
// random numbers and lays them out; it computes nothing of the decode step.
// The same recipe is written in numpy in synth.py; the two are checked
// against each other bit for bit and against the published Philox4x32-10
// known-answer vectors.
//
// Generator: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11).
//   block b of tensor `tid` under `seed`:
//     codes   = the 16 bytes of philox(ctr = (b_lo, b_hi, 0x51, 0), key = (seed, tid))
//     scale   = binary16(|sigma * z|), z = sum of the 12 words of
//               philox(ctr = (b_lo, b_hi, 0xD0 + r, 0)), r = 0..2, times 2^-32, minus 6
//   activation e of vector `tid`: binary16(sigma * z) with tags 0xA0..0xA2.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

struct U4 {
  uint32_t x, y, z, w;
};

__device__ __forceinline__ U4 philox4x32_10(U4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = U4{hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0};
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c;
}

__device__ __forceinline__ double irwin_hall12(uint64_t idx, uint32_t tag, uint32_t seed, uint32_t tid) {
  unsigned long long total = 0;
#pragma unroll
  for (int r = 0; r < 3; ++r) {
    const U4 o = philox4x32_10(U4{static_cast<uint32_t>(idx), static_cast<uint32_t>(idx >> 32), tag + r, 0u}, seed, tid);
    total += static_cast<unsigned long long>(o.x) + o.y + o.z + o.w;
  }
  const long long centered = static_cast<long long>(total) - (6ll << 32);
  return static_cast<double>(centered) * 0x1p-32;
}

__global__ void fill_q4_kernel(uint8_t* dst, uint64_t n_blocks, uint64_t block0, uint32_t seed, uint32_t tid,
                               double sigma) {
  for (uint64_t i = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n_blocks;
       i += static_cast<uint64_t>(gridDim.x) * blockDim.x) {
    const uint64_t b = block0 + i;
    const U4 o = philox4x32_10(U4{static_cast<uint32_t>(b), static_cast<uint32_t>(b >> 32), 0x51u, 0u}, seed, tid);
    const double z = irwin_hall12(b, 0xD0u, seed, tid);
    const unsigned short d = __half_as_ushort(__double2half(fabs(z * sigma)));
    unsigned short* p = reinterpret_cast<unsigned short*>(dst + i * 18);   // blocks are 2-byte aligned
    p[0] = d;
    const uint32_t w[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      p[1 + 2 * t] = static_cast<unsigned short>(w[t] & 0xFFFFu);
      p[2 + 2 * t] = static_cast<unsigned short>(w[t] >> 16);
    }
  }
}

__global__ void fill_normal_kernel(uint16_t* dst, uint64_t n, uint64_t start, uint32_t seed, uint32_t tid,
                                   double sigma) {
  for (uint64_t i = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<uint64_t>(gridDim.x) * blockDim.x) {
    const double z = irwin_hall12(start + i, 0xA0u, seed, tid);
    dst[i] = __half_as_ushort(__double2half(z * sigma));
  }
}

__global__ void philox_kernel(uint32_t* out, uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0, uint32_t k1) {
  const U4 o = philox4x32_10(U4{c0, c1, c2, c3}, k0, k1);
  out[0] = o.x;
  out[1] = o.y;
  out[2] = o.z;
  out[3] = o.w;
}

}  // namespace

extern "C" {

// Fill n_blocks Q4_0 blocks (18 bytes each, dst 2-byte aligned) with blocks
// block0 .. block0+n_blocks-1 of tensor `tid`.  Returns a cudaError_t.
int q4s_fill_q4_0(void* dst, uint64_t n_blocks, uint64_t block0, uint32_t seed, uint32_t tid, double sigma,
                  void* stream) {
  if (n_blocks == 0) return 0;
  fill_q4_kernel<<<4096, 256, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<uint8_t*>(dst), n_blocks, block0,
                                                                      seed, tid, sigma);
  return static_cast<int>(cudaGetLastError());
}

// Fill n binary16 values: element start+i of activation vector `tid`.
int q4s_fill_normal_f16(uint16_t* dst, uint64_t n, uint64_t start, uint32_t seed, uint32_t tid, double sigma,
                        void* stream) {
  if (n == 0) return 0;
  fill_normal_kernel<<<1024, 256, 0, static_cast<cudaStream_t>(stream)>>>(dst, n, start, seed, tid, sigma);
  return static_cast<int>(cudaGetLastError());
}

// One Philox4x32-10 evaluation into out[4] (device), for known-answer checks.
int q4s_philox(uint32_t* out, uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0, uint32_t k1,
               void* stream) {
  philox_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(out, c0, c1, c2, c3, k0, k1);
  return static_cast<int>(cudaGetLastError());
}

}  // extern "C"
