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
// One kernel, split over the context (so a short query still spreads over
// the whole GPU): one CTA per (value head g, chunk of 32/64/128 positions,
// chosen per bucket so that there is a CTA for every SM), 256 threads.  The chunk's keys
// and values of head g are copied to shared memory with 16-byte asynchronous
// copies (all in flight at once); 256/chunk threads form each position's
// scores with the group's query heads (q pre-scaled by 1/sqrt(head_dim));
// per head, the chunk's maximum m, l = sum exp(s - m) and
// o[i] = sum exp(s - m) v[i] are written out.  The last chunk of a value head
// to finish (an arrival counter) combines them for the group's query heads:
// M = max m_c, L = sum l_c exp(m_c - M), out = f16(sum o_c exp(m_c - M) / L),
// chunks in order, and resets the counter.
// The number of positions in use is read from device memory, so one
// captured graph serves every length up to its bucket's capacity.  All
// reductions run in a fixed order.
#include <cuda_fp16.h>
#include <math.h>
#include <stdint.h>

#include "q4_device.cuh"

namespace q4 {

constexpr int kAttnThreads = 256;
constexpr int kAttnWarps = kAttnThreads / 32;
constexpr int kAttnMaxChunk = 128;   // positions per CTA: 32, 64 or 128 (chosen per bucket)
constexpr int kAttnMaxGroup = 16;

struct AttnArgs {
  const float* q;        // fp32 [n_q][hd]
  const __half* k;       // binary16 [capacity][n_kv * hd]
  const __half* v;
  const int* ctx_len;    // positions in use (plus ctx_add)
  int ctx_add;
  // with new_k set, the token's own key and value (fp32 [n_kv * hd]) go into
  // row *pos of the caches (kw, vw: the same arrays as k, v) as part of this
  // kernel: the CTA whose chunk holds that row uses them directly and stores
  // them; *pos outside 0..capacity-1 sets ST_KV_POS in *status and stores nothing
  const float* new_k;
  const float* new_v;
  const int* pos;
  __half* kw;
  __half* vw;
  int* status;
  float* part;           // fp32 [n_q][n_chunks][hd + 2]: m, l, o[0..hd)
  unsigned* arrive;      // [n_kv] chunks of the value head done (the last one combines and resets it)
  __half* out;           // binary16 [n_q][hd]
  int n_q, n_kv, hd, n_chunks, capacity, chunk;
  float scale;           // 1 / sqrt(hd)
};

extern __shared__ __align__(16) unsigned char g_attn_smem[];

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

// Clamp the positions in use to [1, capacity].
__device__ __forceinline__ int attn_ctx(const AttnArgs& a) {
  const int c = *a.ctx_len + a.ctx_add;
  return c < 1 ? 1 : (c > a.capacity ? a.capacity : c);
}

// Block-wide max (or sum) of v[0..group) for every head at once: one
// shuffle tree per head, one shared-memory exchange, a fixed order.
// GMAX (a power of two >= group) bounds the unrolled loops.
template <bool kMax, int GMAX>
__device__ __forceinline__ void attn_reduce_heads(float* v, int group, float* red) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int j = 0; j < GMAX; ++j) {
    if (j < group) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float x = __shfl_xor_sync(0xffffffffu, v[j], o);
        v[j] = kMax ? fmaxf(v[j], x) : v[j] + x;
      }
      if (lane == 0) red[j * kAttnWarps + w] = v[j];
    }
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < GMAX; ++j) {
    if (j < group) {
      float r = red[j * kAttnWarps];
#pragma unroll
      for (int i = 1; i < kAttnWarps; ++i) r = kMax ? fmaxf(r, red[j * kAttnWarps + i]) : r + red[j * kAttnWarps + i];
      v[j] = r;
    }
  }
  __syncthreads();
}

// One CTA per (value head g, chunk c of `chunk` positions), 256 threads;
// tp = 256 / chunk threads share a position's scores (each a slice of the
// head dimension, summed with shuffles).
template <int GMAX>
__global__ void __launch_bounds__(kAttnThreads) attn_kernel(const __grid_constant__ AttnArgs a) {
  const int g = blockIdx.x, c = blockIdx.y, tid = threadIdx.x;
  const int group = a.n_q / a.n_kv, hd = a.hd, kv_dim = a.n_kv * hd, P = a.chunk;
  const int ctx = attn_ctx(a);
  const int used = (ctx + P - 1) / P;
  if (c >= used) return;   // chunk past the context: no work, not counted
  const int t0 = c * P;
  const int nt = min(P, ctx - t0);
  const size_t head_stride = static_cast<size_t>(a.n_chunks) * (hd + 2);
  float* part = a.part + static_cast<size_t>(g * group) * head_stride + static_cast<size_t>(c) * (hd + 2);
  // shared memory: keys [P][hd] (16-byte chunks swizzled by position), values [P][hd],
  // q [group][hd], weights [group][P], reduction scratch
  __half* ks = reinterpret_cast<__half*>(g_attn_smem);
  __half* vs = ks + P * hd;
  float* qs = reinterpret_cast<float*>(vs + P * hd);
  float* ps = qs + group * hd;
  float* red = ps + group * P;
  __shared__ int is_last;
  const int cpr = hd / 8;            // 16-byte chunks per row
  // the row of this token's own key and value, when this kernel appends them
  int own = -1;
  if (a.new_k) {
    const int p = *a.pos;
    if (p < 0 || p >= a.capacity) {
      if (g == 0 && c == 0 && tid == 0) atomicOr(a.status, ST_KV_POS);
    } else if (p >= t0 && p < t0 + nt) {
      own = p - t0;
    }
  }
  for (int i = tid; i < nt * cpr; i += kAttnThreads) {
    const int t = i / cpr, cc = i % cpr;
    const size_t src = static_cast<size_t>(t0 + t) * kv_dim + static_cast<size_t>(g) * hd + cc * 8;
    if (t == own) {
      // f16 of the fp32 key and value, into shared memory and the caches
      const float* kf = a.new_k + static_cast<size_t>(g) * hd + cc * 8;
      const float* vf = a.new_v + static_cast<size_t>(g) * hd + cc * 8;
      uint4 kh, vh;
      __half2* k2 = reinterpret_cast<__half2*>(&kh);
      __half2* v2 = reinterpret_cast<__half2*>(&vh);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        k2[e] = __floats2half2_rn(kf[2 * e], kf[2 * e + 1]);
        v2[e] = __floats2half2_rn(vf[2 * e], vf[2 * e + 1]);
      }
      *reinterpret_cast<uint4*>(ks + t * hd + ((cc ^ (t & 7)) * 8)) = kh;
      *reinterpret_cast<uint4*>(vs + t * hd + cc * 8) = vh;
      *reinterpret_cast<uint4*>(a.kw + src) = kh;
      *reinterpret_cast<uint4*>(a.vw + src) = vh;
    } else {
      cp_async16(ks + t * hd + ((cc ^ (t & 7)) * 8), a.k + src);
      cp_async16(vs + t * hd + cc * 8, a.v + src);
    }
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
  for (int i = tid; i < group * hd; i += kAttnThreads)
    qs[i] = a.q[static_cast<size_t>(g * group) * hd + i] * a.scale;
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  __syncthreads();

  // scores of position t = tid / tp over dims [sub * hd / tp, (sub + 1) * hd / tp)
  const int tp = kAttnThreads / P, t = tid / tp, sub = tid % tp;
  float s[GMAX];
#pragma unroll
  for (int j = 0; j < GMAX; ++j) s[j] = 0.f;
  if (t < nt) {
    const int c_lo = sub * (cpr / tp), c_hi = c_lo + cpr / tp;
#pragma unroll 2
    for (int cc = c_lo; cc < c_hi; ++cc) {
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
      for (int j = 0; j < GMAX; ++j) {
        if (j < group) {
          const float4 qa = *reinterpret_cast<const float4*>(qs + j * hd + cc * 8);
          const float4 qb = *reinterpret_cast<const float4*>(qs + j * hd + cc * 8 + 4);
          s[j] = fmaf(qa.x, kf[0], s[j]);
          s[j] = fmaf(qa.y, kf[1], s[j]);
          s[j] = fmaf(qa.z, kf[2], s[j]);
          s[j] = fmaf(qa.w, kf[3], s[j]);
          s[j] = fmaf(qb.x, kf[4], s[j]);
          s[j] = fmaf(qb.y, kf[5], s[j]);
          s[j] = fmaf(qb.z, kf[6], s[j]);
          s[j] = fmaf(qb.w, kf[7], s[j]);
        }
      }
    }
  }
  // the tp partial sums of a position are adjacent lanes
#pragma unroll
  for (int j = 0; j < GMAX; ++j)
    if (j < group)
      for (int o = tp >> 1; o > 0; o >>= 1) s[j] += __shfl_xor_sync(0xffffffffu, s[j], o);
  // chunk maximum and weights, all heads at once (positions past the context get weight 0)
  float m[GMAX];
#pragma unroll
  for (int j = 0; j < GMAX; ++j) m[j] = (t < nt) ? s[j] : -INFINITY;
  attn_reduce_heads<true, GMAX>(m, group, red);
  float l[GMAX];
#pragma unroll
  for (int j = 0; j < GMAX; ++j) {
    const float p = (t < nt && sub == 0) ? expf(s[j] - m[j]) : 0.f;
    if (j < group && sub == 0) ps[j * P + t] = p;
    l[j] = p;
  }
  attn_reduce_heads<false, GMAX>(l, group, red);   // (its barriers also publish ps)
  if (tid == 0)
    for (int j = 0; j < group; ++j) {
      part[j * head_stride] = m[j];
      part[j * head_stride + 1] = l[j];
    }
  // weighted values: work item (pair of elements, head); positions four at a
  // time (loads issued together), two accumulator sets summed at the end
  const int pairs = hd / 2;
  for (int it = tid; it < pairs * group; it += kAttnThreads) {
    const int e2 = it % pairs, j = it / pairs;
    const float* pj = ps + j * P;
    const __half* vp = vs + 2 * e2;
    float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
    int tt = 0;
    for (; tt + 4 <= nt; tt += 4) {
      const float4 p4 = *reinterpret_cast<const float4*>(pj + tt);
      const float2 v0 = __half22float2(*reinterpret_cast<const __half2*>(vp + tt * hd));
      const float2 v1 = __half22float2(*reinterpret_cast<const __half2*>(vp + (tt + 1) * hd));
      const float2 v2 = __half22float2(*reinterpret_cast<const __half2*>(vp + (tt + 2) * hd));
      const float2 v3 = __half22float2(*reinterpret_cast<const __half2*>(vp + (tt + 3) * hd));
      a0 = fmaf(p4.x, v0.x, a0);
      a1 = fmaf(p4.x, v0.y, a1);
      b0 = fmaf(p4.y, v1.x, b0);
      b1 = fmaf(p4.y, v1.y, b1);
      a0 = fmaf(p4.z, v2.x, a0);
      a1 = fmaf(p4.z, v2.y, a1);
      b0 = fmaf(p4.w, v3.x, b0);
      b1 = fmaf(p4.w, v3.y, b1);
    }
    for (; tt < nt; ++tt) {
      const float2 v0 = __half22float2(*reinterpret_cast<const __half2*>(vp + tt * hd));
      a0 = fmaf(pj[tt], v0.x, a0);
      a1 = fmaf(pj[tt], v0.y, a1);
    }
    *reinterpret_cast<float2*>(part + j * head_stride + 2 + 2 * e2) = make_float2(a0 + b0, a1 + b1);
  }
  // the last chunk of this value head to finish combines the group's heads
  __threadfence();
  __syncthreads();
  if (tid == 0) is_last = atomicAdd(&a.arrive[g], 1u) == static_cast<unsigned>(used - 1);
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  // chunk maxima and sums of the group's heads -> shared memory (reusing the key buffer)
  float* cm = reinterpret_cast<float*>(ks);            // [group][used] m, then the weights exp(m - M)
  float* cl = cm + group * used;                        // [group][used] l
  float* hM = cl + group * used;                        // [group] L
  for (int i = tid; i < group * used; i += kAttnThreads) {
    const int j = i / used, cc = i % used;
    const float* ph = a.part + static_cast<size_t>(g * group + j) * head_stride + static_cast<size_t>(cc) * (hd + 2);
    cm[i] = __ldcg(ph);
    cl[i] = __ldcg(ph + 1);
  }
  __syncthreads();
  if (tid < group) {
    float M = -INFINITY;
    for (int cc = 0; cc < used; ++cc) M = fmaxf(M, cm[tid * used + cc]);
    float L = 0.f;
    for (int cc = 0; cc < used; ++cc) {
      const float w = expf(cm[tid * used + cc] - M);
      cm[tid * used + cc] = w;
      L = fmaf(cl[tid * used + cc], w, L);
    }
    hM[tid] = L;
  }
  __syncthreads();
  for (int it = tid; it < group * hd; it += kAttnThreads) {
    const int j = it / hd, i = it % hd;
    const float* ph = a.part + static_cast<size_t>(g * group + j) * head_stride + 2 + i;
    const float* wj = cm + j * used;
    float O = 0.f;
    // 16 chunks' values loaded before they are summed (one round trip per 16 chunks), in chunk order
    for (int c0 = 0; c0 < used; c0 += 16) {
      float ov[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) ov[e] = c0 + e < used ? __ldcg(ph + static_cast<size_t>(c0 + e) * (hd + 2)) : 0.f;
#pragma unroll
      for (int e = 0; e < 16; ++e)
        if (c0 + e < used) O = fmaf(ov[e], wj[c0 + e], O);
    }
    a.out[static_cast<size_t>(g * group + j) * hd + i] = __float2half_rn(O / hM[j]);
  }
  if (tid == 0) a.arrive[g] = 0u;   // reusable by the next call
}

// k_cache[pos][i] = f16(k[i]), v_cache[pos][i] = f16(v[i]), pos read from device memory.
__global__ void kv_append_kernel(const float* k, const float* v, __half* kc, __half* vc, const int* pos,
                                 int capacity, int kv_dim, int* status) {
  const int p = *pos;
  if (p < 0 || p >= capacity) {
    if (status && blockIdx.x == 0 && threadIdx.x == 0) atomicOr(status, ST_KV_POS);
    return;
  }
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < kv_dim; i += gridDim.x * blockDim.x) {
    kc[static_cast<size_t>(p) * kv_dim + i] = __float2half_rn(k[i]);
    vc[static_cast<size_t>(p) * kv_dim + i] = __float2half_rn(v[i]);
  }
}

// Positions per CTA for a bucket: enough CTAs to cover the GPU at small
// contexts, 128 at large ones.
int attn_chunk(int capacity, int n_kv) {
  int p = kAttnMaxChunk;
  while (p > 32 && static_cast<long>(n_kv) * (capacity / p) < 152) p >>= 1;
  return p;
}

size_t attn_smem_bytes(int group, int hd, int chunk) {
  return static_cast<size_t>(2) * chunk * hd * sizeof(__half) + static_cast<size_t>(group) * hd * sizeof(float) +
         static_cast<size_t>(group) * chunk * sizeof(float) + kAttnMaxGroup * kAttnWarps * sizeof(float);
}

size_t attn_workspace_bytes(int n_q, int n_kv, int hd, int capacity) {
  const int chunk = attn_chunk(capacity, n_kv);
  return static_cast<size_t>(n_q) * (capacity / chunk) * (hd + 2) * sizeof(float) +
         static_cast<size_t>(n_kv) * sizeof(unsigned) + 16;
}

cudaError_t attn_prepare() {
  const int bytes = static_cast<int>(attn_smem_bytes(kAttnMaxGroup, 256, kAttnMaxChunk));
  cudaError_t e = cudaFuncSetAttribute(attn_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(attn_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(attn_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(attn_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(attn_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  return e;
}

cudaError_t attn_launch(const float* q, const uint16_t* k, const uint16_t* v, const int* ctx_len, int capacity,
                        int n_q, int n_kv, int hd, uint16_t* out, void* ws, cudaStream_t s, int ctx_add,
                        const AttnAppend* app) {
  AttnArgs a;
  a.ctx_add = ctx_add;
  a.new_k = app ? app->k : nullptr;
  a.new_v = app ? app->v : nullptr;
  a.pos = app ? app->pos : nullptr;
  a.kw = reinterpret_cast<__half*>(const_cast<uint16_t*>(k));
  a.vw = reinterpret_cast<__half*>(const_cast<uint16_t*>(v));
  a.status = app ? app->status : nullptr;
  a.q = q;
  a.k = reinterpret_cast<const __half*>(k);
  a.v = reinterpret_cast<const __half*>(v);
  a.ctx_len = ctx_len;
  a.n_q = n_q;
  a.n_kv = n_kv;
  a.hd = hd;
  a.capacity = capacity;
  a.chunk = attn_chunk(capacity, n_kv);
  a.n_chunks = capacity / a.chunk;
  a.part = static_cast<float*>(ws);
  a.arrive = reinterpret_cast<unsigned*>(static_cast<char*>(ws) +
                                         static_cast<size_t>(n_q) * a.n_chunks * (hd + 2) * sizeof(float));
  a.out = reinterpret_cast<__half*>(out);
  a.scale = 1.0f / sqrtf(static_cast<float>(hd));
  const int group = n_q / n_kv;
  const dim3 grid(n_kv, a.n_chunks);
  const size_t smem = attn_smem_bytes(group, hd, a.chunk);
  // the loops over the group's heads are unrolled to the next power of two
  if (group <= 1)
    attn_kernel<1><<<grid, kAttnThreads, smem, s>>>(a);
  else if (group <= 2)
    attn_kernel<2><<<grid, kAttnThreads, smem, s>>>(a);
  else if (group <= 4)
    attn_kernel<4><<<grid, kAttnThreads, smem, s>>>(a);
  else if (group <= 8)
    attn_kernel<8><<<grid, kAttnThreads, smem, s>>>(a);
  else
    attn_kernel<16><<<grid, kAttnThreads, smem, s>>>(a);
  return cudaGetLastError();
}

// The decoder's position counter advances by one after a token.
__global__ void pos_advance_kernel(int* pos) { *pos += 1; }

cudaError_t pos_advance_launch(int* pos, cudaStream_t s) {
  pos_advance_kernel<<<1, 1, 0, s>>>(pos);
  return cudaGetLastError();
}

cudaError_t kv_append_launch(const float* k, const float* v, uint16_t* kc, uint16_t* vc, const int* pos, int capacity,
                             int kv_dim, cudaStream_t s, int* status) {
  const int threads = 256, blocks = (kv_dim + threads - 1) / threads;
  kv_append_kernel<<<blocks < 64 ? blocks : 64, threads, 0, s>>>(k, v, reinterpret_cast<__half*>(kc),
                                                                  reinterpret_cast<__half*>(vc), pos, capacity, kv_dim,
                                                                  status);
  return cudaGetLastError();
}

}  // namespace q4
