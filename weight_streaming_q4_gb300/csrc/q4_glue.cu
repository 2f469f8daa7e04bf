// Decoder-layer glue between the projections, for batches of more than one
// row (one CTA per batch row).  The batch-1 path folds the same steps into the
// prologues and epilogues of the persistent engine; these kernels give the
// same arithmetic as separate launches around the tensor-core product:
//   norm          z  = f16(t / sqrt(mean(t^2) + eps))        (t binary16 or fp32)
//   attention     a  = f16(v of the value head each query head is grouped with)
//   resid_norm    t  = z + o (fp32);  z' = f16(t / sqrt(mean(t^2) + eps))
//   silu_mul      act = f16(silu(g) * u)
// Reductions run in a fixed order, so results do not depend on timing.
#include <cuda_fp16.h>
#include <stdint.h>

#include "q4_device.cuh"

namespace q4 {

constexpr int kGlueThreads = 256;

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[w] = v;
  __syncthreads();
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < kGlueThreads / 32; ++i) s += red[i];
  __syncthreads();
  return s;
}

// z[b] = f16(t[b] * rsqrt(mean(t[b]^2) + eps)); t is binary16 (src16) or fp32 (src32).
__global__ void __launch_bounds__(kGlueThreads) norm_kernel(const __half* src16, const float* src32, int dim, float eps,
                                                            __half* z) {
  griddep_launch_dependents();
  griddep_wait();
  __shared__ float red[kGlueThreads / 32];
  const size_t base = static_cast<size_t>(blockIdx.x) * dim;
  float ss = 0.f;
  for (int i = threadIdx.x; i < dim; i += kGlueThreads) {
    const float v = src16 ? __half2float(src16[base + i]) : src32[base + i];
    ss = fmaf(v, v, ss);
  }
  const float r = rsqrtf(block_sum(ss, red) / static_cast<float>(dim) + eps);
  for (int i = threadIdx.x; i < dim; i += kGlueThreads) {
    const float v = src16 ? __half2float(src16[base + i]) : src32[base + i];
    z[base + i] = __float2half_rn(v * r);
  }
}

// t[b] = z[b] + o[b] (fp32); z_out[b] = f16(t[b] * rsqrt(mean(t[b]^2) + eps)).
__global__ void __launch_bounds__(kGlueThreads) resid_norm_kernel(const __half* z, const float* o, int dim, float eps,
                                                                  float* t, __half* z_out) {
  griddep_launch_dependents();
  griddep_wait();
  __shared__ float red[kGlueThreads / 32];
  const size_t base = static_cast<size_t>(blockIdx.x) * dim;
  float ss = 0.f;
  for (int i = threadIdx.x; i < dim; i += kGlueThreads) {
    const float v = __half2float(z[base + i]) + o[base + i];
    t[base + i] = v;
    ss = fmaf(v, v, ss);
  }
  const float r = rsqrtf(block_sum(ss, red) / static_cast<float>(dim) + eps);
  for (int i = threadIdx.x; i < dim; i += kGlueThreads) z_out[base + i] = __float2half_rn(t[base + i] * r);
}

// a[b][i] = f16(qkv[b][v_off + (i / hd / group) * hd + i % hd]), i < q_dim.
__global__ void __launch_bounds__(kGlueThreads) attn_kernel(const float* qkv, int ld, int q_dim, int v_off, int hd,
                                                            int group, __half* a) {
  griddep_launch_dependents();
  griddep_wait();
  const size_t base = static_cast<size_t>(blockIdx.x);
  for (int i = threadIdx.x; i < q_dim; i += kGlueThreads) {
    const int src = v_off + ((i / hd) / group) * hd + (i % hd);
    a[base * q_dim + i] = __float2half_rn(qkv[base * ld + src]);
  }
}

// act = f16(g / (1 + exp(-g)) * u) over n values.
__global__ void __launch_bounds__(kGlueThreads) silu_kernel(const float* g, const float* u, size_t n, __half* act) {
  griddep_launch_dependents();
  griddep_wait();
  for (size_t i = static_cast<size_t>(blockIdx.x) * kGlueThreads + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * kGlueThreads) {
    const float gv = g[i];
    act[i] = __float2half_rn(gv / (1.0f + expf(-gv)) * u[i]);
  }
}

template <typename... P, typename... A>
static cudaError_t glue_launch(void (*kern)(P...), unsigned grid, cudaStream_t s, bool pdl, A... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kGlueThreads);
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
  return glue_launch(norm_kernel, batch, s, pdl, reinterpret_cast<const __half*>(src16), src32, dim, eps,
                     reinterpret_cast<__half*>(z));
}

cudaError_t glue_resid_norm(const uint16_t* z, const float* o, int batch, int dim, float eps, float* t,
                            uint16_t* z_out, cudaStream_t s, bool pdl) {
  return glue_launch(resid_norm_kernel, batch, s, pdl, reinterpret_cast<const __half*>(z), o, dim, eps, t,
                     reinterpret_cast<__half*>(z_out));
}

cudaError_t glue_attn(const float* qkv, int batch, int ld, int q_dim, int v_off, int hd, int group, uint16_t* a,
                      cudaStream_t s, bool pdl) {
  return glue_launch(attn_kernel, batch, s, pdl, qkv, ld, q_dim, v_off, hd, group, reinterpret_cast<__half*>(a));
}

cudaError_t glue_silu(const float* g, const float* u, size_t n, uint16_t* act, cudaStream_t s, bool pdl) {
  const size_t blocks = (n + kGlueThreads - 1) / kGlueThreads;
  return glue_launch(silu_kernel, static_cast<unsigned>(blocks < 1024 ? blocks : 1024), s, pdl, g, u, n,
                     reinterpret_cast<__half*>(act));
}

}  // namespace q4
