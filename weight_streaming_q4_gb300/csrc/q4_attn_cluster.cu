// Decode attention of one token over a binary16 KV cache (sm_103a), one
// thread-block cluster per value head.
//
// The decode loop attends the new token's queries to every cached position:
// PipeLLM captures that loop as a static graph per context-length bucket
// ("Layer 1: CUDA Graph Compilation": buckets of 512, 1024, 2048 and 4096
// positions), and PIPO moves each layer's KV cache with the layer ("PIPO:
// Pipelined Offloading for Efficient Inference on Consumer Devices", Method,
// "Offloading architecture").  The work reads every cached key and value once,
// so it is bound by HBM bandwidth: CUDA cores, no tensor cores.
//
// Value head g is one cluster of C CTAs (16 where the GPU schedules clusters
// that large, else 8); CTA r takes positions [r * span, (r + 1) * span) of the
// context, span = capacity / C.  A CTA copies its keys and values into shared
// memory with 16-byte asynchronous copies, a round of 64 KB (128 positions at
// head_dim 128) at a time with every copy of the round in flight at once, and
// keeps a running softmax state per query head of the
// group: the maximum m, l = sum exp(s - m) and o = sum exp(s - m) v, rescaled
// when a later round raises m.  Scores use q pre-scaled by 1/sqrt(head_dim).
// The C states of a head then meet through distributed shared memory: each
// CTA of the cluster finishes a slice of the group's outputs, reading every
// CTA's m, l and o, M = max m_r, L = sum l_r exp(m_r - M),
// out = f16(sum o_r exp(m_r - M) / L), ranks in order.  Nothing goes through
// global memory between the CTAs and every sum runs in a fixed order.
//
// The number of positions in use is read from device memory, so one captured
// graph serves every length up to its bucket's capacity.  With the append
// arguments set, the kernel also stores the token's own key and value in row
// *pos of the caches: the CTA whose span holds that row converts them to
// binary16, attends to them and writes them out.
#include <cooperative_groups.h>
#include <cuda_fp16.h>
#include <math.h>
#include <stdint.h>

#include "q4_device.cuh"

namespace cg = cooperative_groups;

namespace q4 {

namespace {

constexpr int kAcThreads = 256;
constexpr int kAcWarps = kAcThreads / 32;
constexpr int kAcMaxGroup = 16;
constexpr size_t kAcSmemMax = 112 * 1024;

struct AcArgs {
  const float* q;        // fp32 [n_q][hd]
  const __half* k;       // binary16 [capacity][n_kv * hd]
  const __half* v;
  const int* ctx_len;    // positions in use, plus ctx_add
  int ctx_add;
  const float* new_k;    // append: the token's fp32 key and value [n_kv * hd], or null
  const float* new_v;
  const int* pos;        // append: the row they go to
  __half* kw;            // the caches, written by the append
  __half* vw;
  int* status;           // append: ST_KV_POS when *pos is outside the bucket
  __half* out;           // binary16 [n_q][hd]
  int n_q, n_kv, hd, capacity;
  int span;              // positions per CTA
  int round;             // positions per round (64 KB of keys and values)
  float scale;           // 1 / sqrt(hd)
};

__device__ __forceinline__ void ac_cp16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

// Block-wide max (or sum) of v[0..group) for every head at once: one
// shuffle tree per head, one shared-memory exchange, warps in order.
template <bool kMax, int GMAX>
__device__ __forceinline__ void ac_reduce(float* v, int group, float* red) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int j = 0; j < GMAX; ++j) {
    if (j < group) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float x = __shfl_xor_sync(0xffffffffu, v[j], o);
        v[j] = kMax ? fmaxf(v[j], x) : v[j] + x;
      }
      if (lane == 0) red[j * kAcWarps + w] = v[j];
    }
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < GMAX; ++j) {
    if (j < group) {
      float r = red[j * kAcWarps];
#pragma unroll
      for (int i = 1; i < kAcWarps; ++i) r = kMax ? fmaxf(r, red[j * kAcWarps + i]) : r + red[j * kAcWarps + i];
      v[j] = r;
    }
  }
  __syncthreads();
}

}  // namespace

// One CTA per (rank r of the cluster, value head g), 256 threads.  GMAX (a
// power of two >= group) bounds the unrolled loops over the group's heads.
template <int GMAX>
__global__ void __launch_bounds__(kAcThreads) attn_cluster_kernel(const __grid_constant__ AcArgs a) {
  extern __shared__ __align__(16) unsigned char sm[];
  __shared__ float red[kAcMaxGroup * kAcWarps];
  __shared__ float st_m[kAcMaxGroup], st_l[kAcMaxGroup], st_c[kAcMaxGroup];
  cg::cluster_group cluster = cg::this_cluster();
  const int C = static_cast<int>(cluster.num_blocks());
  const int r = static_cast<int>(cluster.block_rank());
  const int g = blockIdx.y, tid = threadIdx.x;
  const int group = a.n_q / a.n_kv, hd = a.hd, kv_dim = a.n_kv * hd, R = a.round;
  const int cpr = hd / 8;   // 16-byte chunks per row
  // shared memory: keys [R][hd] (16-byte chunks swizzled by position), values
  // [R][hd], q [group][hd], weights [group][R], this CTA's o [group][hd]
  __half* ks = reinterpret_cast<__half*>(sm);
  __half* vs = ks + R * hd;
  float* qs = reinterpret_cast<float*>(vs + R * hd);
  float* ps = qs + group * hd;
  float* osm = ps + group * R;

  int ctx = *a.ctx_len + a.ctx_add;
  ctx = ctx < 1 ? 1 : (ctx > a.capacity ? a.capacity : ctx);
  const int lo = r * a.span;
  const int hi = lo + a.span < ctx ? lo + a.span : ctx;   // empty when lo >= ctx
  int own = -1;   // the row of the token's own key and value, when this CTA holds it
  if (a.new_k) {
    const int p = *a.pos;
    if (p < 0 || p >= a.capacity) {
      if (r == 0 && g == 0 && tid == 0) atomicOr(a.status, ST_KV_POS);
    } else if (p >= lo && p < hi) {
      own = p;
    }
  }
  for (int i = tid; i < group * hd; i += kAcThreads) qs[i] = a.q[static_cast<size_t>(g * group) * hd + i] * a.scale;

  // running softmax state: per head m, l (all threads hold the same values);
  // o [group][hd] in shared memory (osm)
  const int pairs = hd / 2;
  const int Q = kAcThreads / pairs;   // position subsets of the value pass
  float m_run[GMAX], l_run[GMAX];
#pragma unroll
  for (int j = 0; j < GMAX; ++j) {
    m_run[j] = -INFINITY;
    l_run[j] = 0.f;
  }
  for (int i = tid; i < group * hd; i += kAcThreads) osm[i] = 0.f;

  const int tp = kAcThreads / R;   // threads per position (1, 2 or 4)
  const int t = tid / tp, sub = tid % tp;
  for (int r0 = lo; r0 < hi; r0 += R) {
    const int np = hi - r0 < R ? hi - r0 : R;
    // keys, then values, all copies of the round in flight
    for (int i = tid; i < np * cpr; i += kAcThreads) {
      const int tt = i / cpr, cc = i % cpr;
      const size_t src = static_cast<size_t>(r0 + tt) * kv_dim + static_cast<size_t>(g) * hd + cc * 8;
      __half* dst = ks + tt * hd + ((cc ^ (tt & 7)) * 8);
      if (r0 + tt == own) {
        const float* f = a.new_k + static_cast<size_t>(g) * hd + cc * 8;
        uint4 h;
        __half2* h2 = reinterpret_cast<__half2*>(&h);
#pragma unroll
        for (int e = 0; e < 4; ++e) h2[e] = __floats2half2_rn(f[2 * e], f[2 * e + 1]);
        *reinterpret_cast<uint4*>(dst) = h;
        *reinterpret_cast<uint4*>(a.kw + src) = h;
      } else {
        ac_cp16(dst, a.k + src);
      }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    for (int i = tid; i < np * cpr; i += kAcThreads) {
      const int tt = i / cpr, cc = i % cpr;
      const size_t src = static_cast<size_t>(r0 + tt) * kv_dim + static_cast<size_t>(g) * hd + cc * 8;
      __half* dst = vs + tt * hd + cc * 8;
      if (r0 + tt == own) {
        const float* f = a.new_v + static_cast<size_t>(g) * hd + cc * 8;
        uint4 h;
        __half2* h2 = reinterpret_cast<__half2*>(&h);
#pragma unroll
        for (int e = 0; e < 4; ++e) h2[e] = __floats2half2_rn(f[2 * e], f[2 * e + 1]);
        *reinterpret_cast<uint4*>(dst) = h;
        *reinterpret_cast<uint4*>(a.vw + src) = h;
      } else {
        ac_cp16(dst, a.v + src);
      }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_group 1;" ::: "memory");   // the keys
    __syncthreads();

    // scores of position t over dims [sub * hd / tp, (sub + 1) * hd / tp)
    float s[GMAX];
#pragma unroll
    for (int j = 0; j < GMAX; ++j) s[j] = 0.f;
    if (t < np) {
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
    // the tp slices of a position are adjacent lanes
    for (int o = tp >> 1; o > 0; o >>= 1) {
#pragma unroll
      for (int j = 0; j < GMAX; ++j) s[j] += __shfl_xor_sync(0xffffffffu, s[j], o);
    }
    // the round's maximum, the new running maximum, the rescale of the old state
    float m_new[GMAX], corr[GMAX], l_r[GMAX];
#pragma unroll
    for (int j = 0; j < GMAX; ++j) m_new[j] = t < np ? s[j] : -INFINITY;
    ac_reduce<true, GMAX>(m_new, group, red);
#pragma unroll
    for (int j = 0; j < GMAX; ++j) {
      m_new[j] = fmaxf(m_new[j], m_run[j]);
      corr[j] = expf(m_run[j] - m_new[j]);   // 0 on the first round (m_run = -inf)
      const float p = (t < np && sub == 0) ? expf(s[j] - m_new[j]) : 0.f;
      if (j < group && sub == 0 && t < R) ps[j * R + t] = p;
      l_r[j] = p;
    }
    ac_reduce<false, GMAX>(l_r, group, red);   // its barriers also publish ps
#pragma unroll
    for (int j = 0; j < GMAX; ++j) {
      l_run[j] = fmaf(l_run[j], corr[j], l_r[j]);
      m_run[j] = m_new[j];
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");   // the values
    __syncthreads();
    // weighted values: thread (element pair e2, position subset qq) sums
    // positions qq, qq + Q, ... for every head of the group (each value pair
    // is loaded once), into the key buffer (free now) as part[qq][j][hd]
    float* part = reinterpret_cast<float*>(ks);
    if (tid < group) {
      float cj = corr[0];
#pragma unroll
      for (int jj = 1; jj < GMAX; ++jj)
        if (jj == tid) cj = corr[jj];
      st_c[tid] = cj;
    }
    {
      const int e2 = tid % pairs, qq = tid / pairs;
      if (qq < Q) {
        float a0[GMAX], a1[GMAX];
#pragma unroll
        for (int jj = 0; jj < GMAX; ++jj) a0[jj] = a1[jj] = 0.f;
        const __half* vp = vs + 2 * e2;
#pragma unroll 4
        for (int tt = qq; tt < np; tt += Q) {
          const float2 v2 = __half22float2(*reinterpret_cast<const __half2*>(vp + tt * hd));
#pragma unroll
          for (int jj = 0; jj < GMAX; ++jj) {
            if (jj < group) {
              const float p = ps[jj * R + tt];
              a0[jj] = fmaf(p, v2.x, a0[jj]);
              a1[jj] = fmaf(p, v2.y, a1[jj]);
            }
          }
        }
#pragma unroll
        for (int jj = 0; jj < GMAX; ++jj) {
          if (jj < group)
            *reinterpret_cast<float2*>(part + (qq * group + jj) * hd + 2 * e2) = make_float2(a0[jj], a1[jj]);
        }
      }
    }
    __syncthreads();
    // the subsets in order, then the running state: o = o * corr + round
    for (int it = tid; it < group * hd; it += kAcThreads) {
      float sum = part[it];
      for (int qq = 1; qq < Q; ++qq) sum += part[qq * group * hd + it];
      osm[it] = fmaf(osm[it], st_c[it / hd], sum);
    }
    __syncthreads();   // the round's buffers are free for the next one
  }

  // this CTA's m and l into its shared memory (o is there already), for the cluster
  if (tid < group) {
    float mj = m_run[0], lj = l_run[0];
#pragma unroll
    for (int j = 1; j < GMAX; ++j)
      if (j == tid) {
        mj = m_run[j];
        lj = l_run[j];
      }
    st_m[tid] = mj;
    st_l[tid] = lj;
  }
  cluster.sync();
  // (1) every rank's m and l of the group's heads, loaded together;
  // (2) per head M = max m_r, the weights w_r = exp(m_r - M) and L = sum l_r w_r,
  //     ranks in order (rank 0 always holds position 0, so M is finite);
  // (3) rank r finishes outputs [r * per, (r + 1) * per) of the group * hd:
  //     every rank's o of them loaded together, then summed in rank order
  float* rm = reinterpret_cast<float*>(ks);   // [C][group] m, then the weights
  float* rl = rm + C * group;                  // [C][group] l
  float* rL = rl + C * group;                  // [group] L
  float* ro = rL + kAcMaxGroup;                // [per][C] o
  if (tid < C * group) {
    const int rr = tid / group, j = tid % group;
    rm[tid] = *cluster.map_shared_rank(st_m + j, rr);
    rl[tid] = *cluster.map_shared_rank(st_l + j, rr);
  }
  const int total = group * hd, per = (total + C - 1) / C;
  const int i0 = r * per, n_out = i0 + per < total ? per : (total > i0 ? total - i0 : 0);
  for (int x = tid; x < n_out * C; x += kAcThreads) {
    const int ii = x / C, rr = x % C;
    ro[x] = *cluster.map_shared_rank(osm + i0 + ii, rr);
  }
  __syncthreads();
  if (tid < group) {
    float M = -INFINITY;
    for (int rr = 0; rr < C; ++rr) M = fmaxf(M, rm[rr * group + tid]);
    float L = 0.f;
    for (int rr = 0; rr < C; ++rr) {
      const float w = expf(rm[rr * group + tid] - M);
      rm[rr * group + tid] = w;
      L = fmaf(rl[rr * group + tid], w, L);
    }
    rL[tid] = L;
  }
  __syncthreads();
  for (int ii = tid; ii < n_out; ii += kAcThreads) {
    const int j = (i0 + ii) / hd;
    float O = 0.f;
    for (int rr = 0; rr < C; ++rr) O = fmaf(ro[ii * C + rr], rm[rr * group + j], O);
    a.out[static_cast<size_t>(g * group) * hd + i0 + ii] = __float2half_rn(O / rL[j]);
  }
  cluster.sync();   // no CTA leaves while another reads its shared memory
}

namespace {

int g_ac_cluster = 0;   // cluster size chosen by attn_cluster_prepare: 16 or 8

template <int GMAX>
cudaError_t ac_set_attrs(bool nonportable) {
  cudaError_t e = cudaFuncSetAttribute(attn_cluster_kernel<GMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kAcSmemMax));
  if (e == cudaSuccess && nonportable)
    e = cudaFuncSetAttribute(attn_cluster_kernel<GMAX>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return e;
}

}  // namespace

// Positions per round: 64 KB of keys and values (256 positions at head_dim
// 64, 128 at 128, 64 above), so that a cluster's CTAs use about 70 KB of
// shared memory at the common shapes and every value head's cluster is
// resident at once (at 139 KB per CTA a GB300 holds only 7 clusters of 16).
int attn_cluster_round(int hd) { return hd <= 64 ? 256 : hd <= 128 ? 128 : 64; }

size_t attn_cluster_smem(int group, int hd) {
  const int R = attn_cluster_round(hd);
  return static_cast<size_t>(2) * R * hd * sizeof(__half) + static_cast<size_t>(group) * hd * 4 * 2 +
         static_cast<size_t>(group) * R * 4;
}

// Cluster size: 16 when one such cluster with the largest shared memory fits
// on the GPU, else the portable 8.
cudaError_t attn_cluster_prepare() {
  cudaError_t e = cudaSuccess;
  bool big = ac_set_attrs<1>(true) == cudaSuccess && ac_set_attrs<2>(true) == cudaSuccess &&
             ac_set_attrs<4>(true) == cudaSuccess && ac_set_attrs<8>(true) == cudaSuccess &&
             ac_set_attrs<16>(true) == cudaSuccess;
  cudaGetLastError();   // a refused attribute is not an error of the library
  if (big) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(16, 1);
    cfg.blockDim = dim3(kAcThreads);
    cfg.dynamicSmemBytes = kAcSmemMax;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 16;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    big = cudaOccupancyMaxActiveClusters(&n, attn_cluster_kernel<16>, &cfg) == cudaSuccess && n >= 1;
    cudaGetLastError();
  }
  if (!big) {
    e = ac_set_attrs<1>(false);
    if (e == cudaSuccess) e = ac_set_attrs<2>(false);
    if (e == cudaSuccess) e = ac_set_attrs<4>(false);
    if (e == cudaSuccess) e = ac_set_attrs<8>(false);
    if (e == cudaSuccess) e = ac_set_attrs<16>(false);
  }
  g_ac_cluster = big ? 16 : 8;
  return e;
}

int attn_cluster_size() { return g_ac_cluster; }

cudaError_t attn_cluster_launch(const float* q, const uint16_t* k, const uint16_t* v, const int* ctx_len, int ctx_add,
                                int capacity, int n_q, int n_kv, int hd, uint16_t* out, const AttnAppend* app,
                                cudaStream_t s) {
  const int C = g_ac_cluster;
  if (C != 8 && C != 16) return cudaErrorInitializationError;
  AcArgs a;
  a.q = q;
  a.k = reinterpret_cast<const __half*>(k);
  a.v = reinterpret_cast<const __half*>(v);
  a.ctx_len = ctx_len;
  a.ctx_add = ctx_add;
  a.new_k = app ? app->k : nullptr;
  a.new_v = app ? app->v : nullptr;
  a.pos = app ? app->pos : nullptr;
  a.kw = reinterpret_cast<__half*>(const_cast<uint16_t*>(k));
  a.vw = reinterpret_cast<__half*>(const_cast<uint16_t*>(v));
  a.status = app ? app->status : nullptr;
  a.out = reinterpret_cast<__half*>(out);
  a.n_q = n_q;
  a.n_kv = n_kv;
  a.hd = hd;
  a.capacity = capacity;
  a.span = (capacity + C - 1) / C;
  a.round = attn_cluster_round(hd);
  a.scale = 1.0f / sqrtf(static_cast<float>(hd));
  const int group = n_q / n_kv;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C, n_kv);
  cfg.blockDim = dim3(kAcThreads);
  cfg.dynamicSmemBytes = attn_cluster_smem(group, hd);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // the loops over the group's heads are unrolled to the next power of two
  if (group <= 1) return cudaLaunchKernelEx(&cfg, attn_cluster_kernel<1>, a);
  if (group <= 2) return cudaLaunchKernelEx(&cfg, attn_cluster_kernel<2>, a);
  if (group <= 4) return cudaLaunchKernelEx(&cfg, attn_cluster_kernel<4>, a);
  if (group <= 8) return cudaLaunchKernelEx(&cfg, attn_cluster_kernel<8>, a);
  return cudaLaunchKernelEx(&cfg, attn_cluster_kernel<16>, a);
}

}  // namespace q4
