// Decoder-layer glue between the projections, for batches of more than one
// row.  The context-1 attention gather and the SiLU-gated product are written
// by the epilogues of the q|k|v and gate|up products themselves; the batch-1
// path folds the same steps into the prologues and epilogues of the
// persistent engine.  These kernels are the RMSNorms, as separate launches
// around the tensor-core products:
//   norm          z  = f16(t / sqrt(mean(t^2) + eps))        (t binary16 or fp32)
//   resid_norm    t  = z + o (fp32);  z' = f16(t / sqrt(mean(t^2) + eps))
// Reductions run in a fixed order, so results do not depend on timing.
#include <cuda_fp16.h>
#include <stdint.h>

#include "q4_device.cuh"
#include "q4_frag.cuh"

namespace q4 {

constexpr int kGlueThreads = 256;    // element-wise kernels
constexpr int kNormThreads = 1024;   // one CTA per batch row for the RMSNorms
constexpr int kNormKeep = 4;          // 4-value steps a thread keeps in registers

// Sum of v over the CTA (T threads), the same fixed order in every CTA.
template <int T>
__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[w] = v;
  __syncthreads();
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < T / 32; ++i) s += red[i];
  __syncthreads();
  return s;
}

__device__ __forceinline__ float4 load_h4(const __half* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

__device__ __forceinline__ void store_h4(__half* p, float4 v, float r) {
  const __half2 a = __floats2half2_rn(v.x * r, v.y * r);
  const __half2 b = __floats2half2_rn(v.z * r, v.w * r);
  uint2 u;
  u.x = *reinterpret_cast<const uint32_t*>(&a);
  u.y = *reinterpret_cast<const uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = u;
}

// z[b] = f16(t[b] * rsqrt(mean(t[b]^2) + eps)); t is binary16 (src16) or fp32
// (src32); dim a multiple of 4.  One CTA per batch row, 4 values per thread
// and step.
__global__ void __launch_bounds__(kNormThreads) norm_kernel(const __half* src16, const float* src32, int dim, float eps,
                                                            __half* z) {
  griddep_launch_dependents();
  griddep_wait();
  __shared__ float red[kNormThreads / 32];
  const size_t base = static_cast<size_t>(blockIdx.x) * dim;
  float ss = 0.f;
  for (int i = 4 * threadIdx.x; i < dim; i += 4 * kNormThreads) {
    const float4 v = src16 ? load_h4(src16 + base + i) : *reinterpret_cast<const float4*>(src32 + base + i);
    ss = fmaf(v.x, v.x, ss);
    ss = fmaf(v.y, v.y, ss);
    ss = fmaf(v.z, v.z, ss);
    ss = fmaf(v.w, v.w, ss);
  }
  const float r = rsqrtf(block_sum<kNormThreads>(ss, red) / static_cast<float>(dim) + eps);
  for (int i = 4 * threadIdx.x; i < dim; i += 4 * kNormThreads) {
    const float4 v = src16 ? load_h4(src16 + base + i) : *reinterpret_cast<const float4*>(src32 + base + i);
    store_h4(z + base + i, v, r);
  }
}

// t[b] = z[b] + o[b] (fp32); z_out[b] = f16(t[b] * rsqrt(mean(t[b]^2) + eps)).
// dim a multiple of 4; one CTA per batch row.
__global__ void __launch_bounds__(kNormThreads) resid_norm_kernel(const __half* z, const float* o, int dim, float eps,
                                                                  float* t, __half* z_out) {
  griddep_launch_dependents();
  griddep_wait();
  __shared__ float red[kNormThreads / 32];
  const size_t base = static_cast<size_t>(blockIdx.x) * dim;
  // the thread's sums stay in registers for rows of up to kNormKeep steps
  // (16384 values); longer rows read them back
  float4 keep[kNormKeep];
  float ss = 0.f;
  int j = 0;
  for (int i = 4 * threadIdx.x; i < dim; i += 4 * kNormThreads, ++j) {
    const float4 a = load_h4(z + base + i);
    const float4 b = *reinterpret_cast<const float4*>(o + base + i);
    const float4 v = make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
    *reinterpret_cast<float4*>(t + base + i) = v;
    if (j < kNormKeep) keep[j] = v;
    ss = fmaf(v.x, v.x, ss);
    ss = fmaf(v.y, v.y, ss);
    ss = fmaf(v.z, v.z, ss);
    ss = fmaf(v.w, v.w, ss);
  }
  const float r = rsqrtf(block_sum<kNormThreads>(ss, red) / static_cast<float>(dim) + eps);
  j = 0;
  for (int i = 4 * threadIdx.x; i < dim; i += 4 * kNormThreads, ++j)
    store_h4(z_out + base + i, j < kNormKeep ? keep[j] : *reinterpret_cast<const float4*>(t + base + i), r);
}

template <typename... P, typename... A>
static cudaError_t glue_launch(void (*kern)(P...), unsigned grid, unsigned threads, cudaStream_t s, bool pdl,
                               A... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<P>(args)...);
}

cudaError_t glue_norm(const uint16_t* src16, const float* src32, int batch, int dim, float eps, uint16_t* z,
                      cudaStream_t s, bool pdl) {
  if (dim % 4) return cudaErrorInvalidValue;
  return glue_launch(norm_kernel, batch, kNormThreads, s, pdl, reinterpret_cast<const __half*>(src16), src32, dim, eps,
                     reinterpret_cast<__half*>(z));
}

cudaError_t glue_resid_norm(const uint16_t* z, const float* o, int batch, int dim, float eps, float* t,
                            uint16_t* z_out, cudaStream_t s, bool pdl) {
  if (dim % 4) return cudaErrorInvalidValue;
  return glue_launch(resid_norm_kernel, batch, kNormThreads, s, pdl, reinterpret_cast<const __half*>(z), o, dim, eps,
                     t, reinterpret_cast<__half*>(z_out));
}

}  // namespace q4
