// Plain kernels beside the persistent engine: a one-warp-per-row product for
// any shape and batch, the dequantise-only debug kernel that checks the block
// layout bit for bit, and the scale poisoner used by the streaming ring's
// race check.
#include <cuda_fp16.h>
#include <stdint.h>

#include "q4_device.cuh"

namespace q4 {

__device__ __forceinline__ float load_scale(const uint8_t* blk) {
  return __half2float(__ushort_as_half(*reinterpret_cast<const unsigned short*>(blk)));
}

// y[b][n] = sum_k W[n][k] x[b][k]: one warp per row, lanes stride over the
// row's blocks; each product (q - 8) * x is exact in fp32, each block sum is
// scaled by d once, and the lane sums are reduced with shuffles.
__global__ void __launch_bounds__(256) simple_kernel(const uint8_t* __restrict__ w,
                                                     const __half* __restrict__ x,
                                                     float* __restrict__ y, int n_rows, int k,
                                                     int batch) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= n_rows) return;
  const int nb = k / kQK;
  const uint8_t* row = w + static_cast<size_t>(warp) * nb * kBlockBytes;
  float tot[kMaxBatch];
#pragma unroll
  for (int b = 0; b < kMaxBatch; ++b) tot[b] = 0.f;
  for (int i = lane; i < nb; i += 32) {
    const uint8_t* blk = row + static_cast<size_t>(i) * kBlockBytes;
    const float d = load_scale(blk);
    const unsigned short* qs = reinterpret_cast<const unsigned short*>(blk + 2);
    float qv[32];
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const unsigned short two = qs[t];   // code bytes 2t, 2t+1
      qv[2 * t] = static_cast<float>(static_cast<int>(two & 0xF) - 8);
      qv[2 * t + 1] = static_cast<float>(static_cast<int>((two >> 8) & 0xF) - 8);
      qv[2 * t + 16] = static_cast<float>(static_cast<int>((two >> 4) & 0xF) - 8);
      qv[2 * t + 17] = static_cast<float>(static_cast<int>(two >> 12) - 8);
    }
#pragma unroll
    for (int b = 0; b < kMaxBatch; ++b) {
      if (b < batch) {
        const __half* xb = x + static_cast<size_t>(b) * k + i * kQK;
        float s = 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j) s = fmaf(qv[j], __half2float(xb[j]), s);
        tot[b] = fmaf(d, s, tot[b]);
      }
    }
  }
#pragma unroll
  for (int b = 0; b < kMaxBatch; ++b) {
    if (b < batch) {
      float v = tot[b];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) y[static_cast<size_t>(b) * n_rows + warp] = v;
    }
  }
}

// out[n][k] = (q - 8) * d for every weight.
__global__ void dequant_kernel(const uint8_t* __restrict__ w, float* __restrict__ out, int n_rows, int k) {
  const size_t idx = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const size_t total = static_cast<size_t>(n_rows) * k;
  if (idx >= total) return;
  const size_t blk = idx / kQK;   // rows are whole blocks, so the flat block index is row-major
  const int j = static_cast<int>(idx % kQK);
  const uint8_t* p = w + blk * kBlockBytes;
  const uint8_t byte = p[2 + (j & 15)];
  const int q = (j < 16) ? (byte & 0xF) : (byte >> 4);
  out[idx] = static_cast<float>(q - 8) * load_scale(p);
}

// Overwrite the scale of every block of a merged layer buffer with a NaN.
__global__ void poison_kernel(uint8_t* buf, size_t n_blocks) {
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n_blocks;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    *reinterpret_cast<unsigned short*>(buf + i * kBlockBytes) = 0x7E00u;
  }
}

cudaError_t simple_launch(const uint8_t* w, const uint16_t* x, float* y, int n, int k, int batch,
                          cudaStream_t stream) {
  const int threads = 256;
  const long long warps = n;
  const int grid = static_cast<int>((warps * 32 + threads - 1) / threads);
  simple_kernel<<<grid, threads, 0, stream>>>(w, reinterpret_cast<const __half*>(x), y, n, k, batch);
  return cudaGetLastError();
}

cudaError_t dequant_launch(const uint8_t* w, float* out, int n, int k, cudaStream_t stream) {
  const size_t total = static_cast<size_t>(n) * k;
  const int threads = 256;
  const size_t grid = (total + threads - 1) / threads;
  if (grid > 0x7FFFFFFFull) return cudaErrorInvalidValue;
  dequant_kernel<<<static_cast<unsigned>(grid), threads, 0, stream>>>(w, out, n, k);
  return cudaGetLastError();
}

cudaError_t poison_launch(uint8_t* buf, size_t n_blocks, cudaStream_t stream) {
  poison_kernel<<<1024, 256, 0, stream>>>(buf, n_blocks);
  return cudaGetLastError();
}

// The GPU's global nanosecond timer, written when the stream reaches this
// point (copy/compute timelines of the ring: stamps on both streams share
// one clock).
__global__ void stamp_kernel(unsigned long long* out) {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  *out = t;
}

cudaError_t stamp_launch(unsigned long long* out, cudaStream_t stream) {
  stamp_kernel<<<1, 1, 0, stream>>>(out);
  return cudaGetLastError();
}

}  // namespace q4
