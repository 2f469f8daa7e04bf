// Decode attention of one token over a binary16 KV cache (sm_103a).
//
// The decode loop attends the new token's queries to every cached position:
// PipeLLM captures that loop as a static graph per context-length bucket
// ("Layer 1: CUDA Graph Compilation": buckets of 512, 1024, 2048 and 4096
// positions), and PIPO moves each layer's KV cache with the layer ("PIPO:
// Pipelined Offloading for Efficient Inference on Consumer Devices", Method,
// "Offloading architecture").  The work reads every cached key and value
// once, so it is bound by HBM bandwidth, not arithmetic: CUDA cores, no
// tensor cores.
//
// Two kernels, split over the context (so a short query still spreads over
// the whole GPU):
//   attn_partial: one CTA per (value head g, chunk of 128 positions).  The
//     chunk's keys and values of head g are copied to shared memory with
//     16-byte asynchronous copies (all in flight at once); every thread takes
//     one position and forms its scores with the group's query heads
//     (q pre-scaled by 1/sqrt(head_dim)); per head, the chunk's maximum m,
//     l = sum exp(s - m) and o[i] = sum exp(s - m) v[i] are written out.
//   attn_combine: one CTA per query head, one thread per output element:
//     M = max m_c, L = sum l_c exp(m_c - M), out = f16(sum o_c exp(m_c - M) / L).
// The number of positions in use is read from device memory, so one
// captured graph serves every length up to its bucket's capacity.  All
// reductions run in a fixed order.
#include <cuda_fp16.h>
#include <math.h>
#include <stdint.h>

#include "q4_device.cuh"

namespace q4 {

constexpr int kAttnChunk = 128;    // positions per CTA (one per thread)
constexpr int kAttnThreads = 128;

struct AttnArgs {
  const float* q;        // fp32 [n_q][hd]
  const __half* k;       // binary16 [capacity][n_kv * hd]
  const __half* v;
  const int* ctx_len;    // positions in use
  float* part;           // fp32 [n_q][n_chunks][hd + 2]: m, l, o[0..hd)
  int n_q, n_kv, hd, n_chunks, capacity;
  float scale;           // 1 / sqrt(hd)
};

extern __shared__ __align__(16) unsigned char g_attn_smem[];

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

__device__ __forceinline__ float attn_block_reduce(float v, float* red, bool is_max) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float w = __shfl_xor_sync(0xffffffffu, v, o);
    v = is_max ? fmaxf(v, w) : v + w;
  }
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[w] = v;
  __syncthreads();
  float r = red[0];
#pragma unroll
  for (int i = 1; i < kAttnThreads / 32; ++i) r = is_max ? fmaxf(r, red[i]) : r + red[i];
  __syncthreads();
  return r;
}

// Clamp the positions in use to [1, capacity].
__device__ __forceinline__ int attn_ctx(const AttnArgs& a) {
  const int c = *a.ctx_len;
  return c < 1 ? 1 : (c > a.capacity ? a.capacity : c);
}

__global__ void __launch_bounds__(kAttnThreads) attn_partial_kernel(const __grid_constant__ AttnArgs a) {
  const int g = blockIdx.x, c = blockIdx.y, tid = threadIdx.x;
  const int group = a.n_q / a.n_kv, hd = a.hd, kv_dim = a.n_kv * hd;
  const int ctx = attn_ctx(a);
  const int t0 = c * kAttnChunk;
  const int nt = min(kAttnChunk, ctx - t0);
  const size_t head_stride = static_cast<size_t>(a.n_chunks) * (hd + 2);
  float* part = a.part + static_cast<size_t>(g * group) * head_stride + static_cast<size_t>(c) * (hd + 2);
  if (nt <= 0) {   // chunk past the context: contributes nothing
    for (int j = 0; j < group; ++j)
      if (tid == 0) {
        part[j * head_stride] = -INFINITY;
        part[j * head_stride + 1] = 0.f;
      }
    return;
  }
  // shared memory: keys [128][hd] (16-byte chunks swizzled by position), values [128][hd],
  // q [group][hd], scores [group][128], reduction scratch
  __half* ks = reinterpret_cast<__half*>(g_attn_smem);
  __half* vs = ks + kAttnChunk * hd;
  float* qs = reinterpret_cast<float*>(vs + kAttnChunk * hd);
  float* ps = qs + group * hd;
  float* red = ps + group * kAttnChunk;
  const int cpr = hd / 8;            // 16-byte chunks per row (8, 16 or 32)
  for (int i = tid; i < nt * cpr; i += kAttnThreads) {
    const int t = i / cpr, cc = i % cpr;
    const size_t src = static_cast<size_t>(t0 + t) * kv_dim + static_cast<size_t>(g) * hd + cc * 8;
    cp_async16(ks + t * hd + ((cc ^ (t & 7)) * 8), a.k + src);
    cp_async16(vs + t * hd + cc * 8, a.v + src);
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
  for (int i = tid; i < group * hd; i += kAttnThreads)
    qs[i] = a.q[static_cast<size_t>(g * group) * hd + i] * a.scale;
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  __syncthreads();

  // scores: thread t = position t of the chunk
  {
    const int t = tid;
    float s[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) s[j] = 0.f;
    if (t < nt) {
      for (int cc = 0; cc < cpr; ++cc) {
        const uint4 raw = *reinterpret_cast<const uint4*>(ks + t * hd + ((cc ^ (t & 7)) * 8));
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
        float kf[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
          kf[2 * e] = f.x;
          kf[2 * e + 1] = f.y;
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          if (j < group) {
            const float* qj = qs + j * hd + cc * 8;
#pragma unroll
            for (int e = 0; e < 8; ++e) s[j] = fmaf(qj[e], kf[e], s[j]);
          }
        }
      }
    }
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (j < group) ps[j * kAttnChunk + t] = t < nt ? s[j] : -INFINITY;
  }
  __syncthreads();
  // per head: chunk maximum, weights exp(s - m), their sum
  for (int j = 0; j < group; ++j) {
    const float sv = ps[j * kAttnChunk + tid];
    const float m = attn_block_reduce(sv, red, true);
    const float p = tid < nt ? expf(sv - m) : 0.f;
    ps[j * kAttnChunk + tid] = p;
    const float l = attn_block_reduce(p, red, false);
    if (tid == 0) {
      part[j * head_stride] = m;
      part[j * head_stride + 1] = l;
    }
  }
  __syncthreads();
  // weighted values: thread i = output element i (and i + 128, ... for wide heads)
  for (int i = tid; i < hd; i += kAttnThreads) {
    for (int j = 0; j < group; ++j) {
      float o = 0.f;
      for (int t = 0; t < nt; ++t) o = fmaf(ps[j * kAttnChunk + t], __half2float(vs[t * hd + i]), o);
      part[j * head_stride + 2 + i] = o;
    }
  }
}

__global__ void attn_combine_kernel(const __grid_constant__ AttnArgs a, __half* out) {
  const int h = blockIdx.x, hd = a.hd;
  const int used = (attn_ctx(a) + kAttnChunk - 1) / kAttnChunk;
  const float* part = a.part + static_cast<size_t>(h) * a.n_chunks * (hd + 2);
  float M = -INFINITY;
  for (int c = 0; c < used; ++c) M = fmaxf(M, part[c * (hd + 2)]);
  for (int i = threadIdx.x; i < hd; i += blockDim.x) {
    float L = 0.f, O = 0.f;
    for (int c = 0; c < used; ++c) {
      const float w = expf(part[c * (hd + 2)] - M);
      L = fmaf(part[c * (hd + 2) + 1], w, L);
      O = fmaf(part[c * (hd + 2) + 2 + i], w, O);
    }
    out[static_cast<size_t>(h) * hd + i] = __float2half_rn(O / L);
  }
}

// k_cache[pos][i] = f16(k[i]), v_cache[pos][i] = f16(v[i]), pos read from device memory.
__global__ void kv_append_kernel(const float* k, const float* v, __half* kc, __half* vc, const int* pos,
                                 int capacity, int kv_dim) {
  const int p = *pos;
  if (p < 0 || p >= capacity) return;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < kv_dim; i += gridDim.x * blockDim.x) {
    kc[static_cast<size_t>(p) * kv_dim + i] = __float2half_rn(k[i]);
    vc[static_cast<size_t>(p) * kv_dim + i] = __float2half_rn(v[i]);
  }
}

size_t attn_smem_bytes(int group, int hd) {
  return static_cast<size_t>(2) * kAttnChunk * hd * sizeof(__half) + static_cast<size_t>(group) * hd * sizeof(float) +
         static_cast<size_t>(group) * kAttnChunk * sizeof(float) + 32 * sizeof(float);
}

cudaError_t attn_prepare() {
  return cudaFuncSetAttribute(attn_partial_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(attn_smem_bytes(16, 256)));
}

cudaError_t attn_launch(const float* q, const uint16_t* k, const uint16_t* v, const int* ctx_len, int capacity,
                        int n_q, int n_kv, int hd, uint16_t* out, float* part, cudaStream_t s) {
  AttnArgs a;
  a.q = q;
  a.k = reinterpret_cast<const __half*>(k);
  a.v = reinterpret_cast<const __half*>(v);
  a.ctx_len = ctx_len;
  a.part = part;
  a.n_q = n_q;
  a.n_kv = n_kv;
  a.hd = hd;
  a.capacity = capacity;
  a.n_chunks = capacity / kAttnChunk;
  a.scale = 1.0f / sqrtf(static_cast<float>(hd));
  attn_partial_kernel<<<dim3(n_kv, a.n_chunks), kAttnThreads, attn_smem_bytes(n_q / n_kv, hd), s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  attn_combine_kernel<<<n_q, hd < 256 ? hd : 256, 0, s>>>(a, reinterpret_cast<__half*>(out));
  return cudaGetLastError();
}

cudaError_t kv_append_launch(const float* k, const float* v, uint16_t* kc, uint16_t* vc, const int* pos, int capacity,
                             int kv_dim, cudaStream_t s) {
  const int threads = 256, blocks = (kv_dim + threads - 1) / threads;
  kv_append_kernel<<<blocks < 64 ? blocks : 64, threads, 0, s>>>(k, v, reinterpret_cast<__half*>(kc),
                                                                  reinterpret_cast<__half*>(vc), pos, capacity, kv_dim);
  return cudaGetLastError();
}

}  // namespace q4
