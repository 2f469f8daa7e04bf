// Decode attention entry points and the KV-cache helpers (sm_103a).
//
// The attention itself is the cluster kernel of q4_attn_cluster.cu (one
// thread-block cluster per value head, the partial softmax states combined
// through distributed shared memory).  This file holds the calls the rest of
// the library makes: the append of a token's key and value to a cache, the
// decoder's position counter, and the attention launch.
#include <cuda_fp16.h>
#include <math.h>
#include <stdint.h>

#include "q4_device.cuh"

namespace q4 {

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

// The decoder's position counter advances by one after a token.
__global__ void pos_advance_kernel(int* pos) { *pos += 1; }

// The cluster kernel keeps its partial results in shared memory; the
// workspace of the attention call is reserved (16 bytes, unused).
size_t attn_workspace_bytes(int, int, int, int) { return 16; }

cudaError_t attn_prepare() { return attn_cluster_prepare(); }

cudaError_t attn_launch(const float* q, const uint16_t* k, const uint16_t* v, const int* ctx_len, int capacity,
                        int n_q, int n_kv, int hd, uint16_t* out, void*, cudaStream_t s, int ctx_add,
                        const AttnAppend* app) {
  return attn_cluster_launch(q, k, v, ctx_len, ctx_add, capacity, n_q, n_kv, hd, out, app, s);
}

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
