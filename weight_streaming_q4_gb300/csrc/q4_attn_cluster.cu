// Decode attention of one token over a binary16 KV cache (sm_103a), one
// thread-block cluster per value head.
//
// The decode loop attends the new token's queries to every cached position:
// PipeLLM captures that loop as a static graph per context-length bucket
// ("Layer 1: CUDA Graph Compilation": buckets of 512, 1024, 2048 and 4096
// positions), and PIPO moves each layer's KV cache with the layer ("PIPO:
// Pipelined Offloading for Efficient Inference on Consumer Devices", Method,
// "Offloading architecture").  The work reads every cached key and value once
// and should be bound by HBM bandwidth; on CUDA cores its score and value
// steps were long dependent chains (latency-bound), hence the tensor cores.
//
// Value head g is one cluster of C CTAs (16 where the GPU schedules clusters
// that large and the bucket holds more than 1024 positions, else 8); CTA r
// takes positions [r * span, (r + 1) * span) of the
// context, span = capacity / C.  A CTA copies its keys and values into shared
// memory with 16-byte asynchronous copies, a round of 64 KB (128 positions at
// head_dim 128) at a time with every copy of the round in flight, and keeps a
// running softmax state per query head of the group: the maximum m,
// l = sum exp(s - m) and o = sum exp(s - m) v, rescaled when a later round
// raises m.  The scores q . k / sqrt(head_dim) and the products of the weights
// with the values run on the tensor cores, with the fp32 query and the fp32
// weights each split into two binary16 parts (about 22 bits kept; keys and
// values are binary16 already), fp32 accumulation.  The C states of a head
// then meet through distributed shared memory: each CTA of the cluster
// finishes a slice of the group's outputs, reading every CTA's m, l and o,
// M = max m_r, L = sum l_r exp(m_r - M), out = f16(sum o_r exp(m_r - M) / L),
// ranks in order.  Nothing goes through global memory between the CTAs and
// every sum runs in a fixed order.
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
#include "q4_frag.cuh"

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
  int pdl;               // launched as a programmatic dependent of the kernel that wrote q and the
                         // token's key and value: the first round's cached rows are copied
                         // before waiting for it
};

// The token's own key or value chunk cc (8 values) as binary16: into the
// staged row (swizzled chunk) and the cache.
__device__ __forceinline__ void ac_put_own(const float* f, __half* dst_smem, __half* dst_cache) {
  uint4 h;
  __half2* h2 = reinterpret_cast<__half2*>(&h);
#pragma unroll
  for (int e = 0; e < 4; ++e) h2[e] = __floats2half2_rn(f[2 * e], f[2 * e + 1]);
  *reinterpret_cast<uint4*>(dst_smem) = h;
  *reinterpret_cast<uint4*>(dst_cache) = h;
}

__device__ __forceinline__ void ac_cp16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

// ldmatrix: 8x8 binary16 matrices from shared memory, one row address per
// lane (lanes 8i..8i+7: the rows of matrix i); .trans delivers each matrix
// transposed.
__device__ __forceinline__ void ldsm_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x2(uint32_t& r0, uint32_t& r1, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x2_t(uint32_t& r0, uint32_t& r1, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];"
               : "=r"(r0), "=r"(r1)
               : "r"(smem_u32(p)));
}
// d += a * b, binary16 in, fp32 accumulate (m16n8k16).
__device__ __forceinline__ void ac_mma(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                       uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// A value split into two binary16 parts (hi = f16(v), lo = f16(v - hi)), so
// that a pair of binary16 products carries about 22 bits of v.
__device__ __forceinline__ void split_half(float v, __half& hi, __half& lo) {
  hi = __float2half_rn(v);
  lo = __float2half_rn(v - __half2float(hi));
}

}  // namespace

// One CTA per (rank r of the cluster, value head g), 256 threads, the score
// and value steps on the tensor cores (mma.sync m16n8k16, binary16 in, fp32
// accumulate).  Scores:
// A = a tile of 16 positions x 16 dimensions of keys (ldmatrix from the
// swizzled key rows), B = q as two binary16 parts (hi + lo, about 22 bits of
// the fp32 query), heads in the n dimension (NTS tiles of 8 heads).  Values:
// A = the weights exp(s - m) as two binary16 parts, heads x positions, B = a
// tile of values (ldmatrix.trans from the swizzled value rows), warp w taking
// NTV tiles of 8 dimensions; the running output stays in the accumulator
// registers and is rescaled when a round raises m.  Softmax maxima and sums
// per head by shuffles and one shared-memory exchange; positions past the
// context get weight 0 (their value rows in the last tile are zeroed while
// the round's copies are in flight, so no stale bits can make a NaN).  The
// first round's copies are issued before q is staged, so q's load overlaps
// them.
template <int NTS, int NTV>
__global__ void __launch_bounds__(kAcThreads) attn_mma_kernel(const __grid_constant__ AcArgs a) {
  extern __shared__ __align__(16) unsigned char sm[];
  __shared__ float wred[kAcWarps][kAcMaxGroup];
  __shared__ float hm[kAcMaxGroup], hl[kAcMaxGroup], hc[kAcMaxGroup];
  cg::cluster_group cluster = cg::this_cluster();
  const int C = static_cast<int>(cluster.num_blocks());
  const int r = static_cast<int>(cluster.block_rank());
  const int g = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const int group = a.n_q / a.n_kv, hd = a.hd, kv_dim = a.n_kv * hd, R = a.round;
  const int cpr = hd / 8;          // 16-byte chunks per row
  const int QS = hd + 8, PS = R + 8;   // padded rows of q and of the weights (conflict-free ldmatrix)
  // shared memory: keys, values [R][hd] (16-byte chunks swizzled by position),
  // q hi/lo [16][QS], weights hi/lo [16][PS], this CTA's o [group][hd]
  __half* ks = reinterpret_cast<__half*>(sm);
  __half* vs = ks + R * hd;
  __half* qh = vs + R * hd;
  __half* ql = qh + 16 * QS;
  __half* ph = ql + 16 * QS;
  __half* pl = ph + 16 * PS;
  float* osm = reinterpret_cast<float*>(pl + 16 * PS);

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
  if (tid < kAcMaxGroup) {
    hm[tid] = -INFINITY;
    hl[tid] = 0.f;
  }
  float oacc[NTV][4];
#pragma unroll
  for (int nt = 0; nt < NTV; ++nt) oacc[nt][0] = oacc[nt][1] = oacc[nt][2] = oacc[nt][3] = 0.f;
  const int d0 = warp * 8 * NTV;   // this warp's first value dimension

  for (int r0 = lo; r0 < hi; r0 += R) {
    const int np = hi - r0 < R ? hi - r0 : R;
    const int ntiles = (np + 15) >> 4;
    // a programmatic dependent launch writes the token's own row of its first
    // round after the wait (it comes from the kernel ahead of this one)
    const bool defer_own = a.pdl && r0 == lo;
    // keys, then values, all copies of the round in flight
    for (int i = tid; i < np * cpr; i += kAcThreads) {
      const int tt = i / cpr, cc = i % cpr;
      const size_t src = static_cast<size_t>(r0 + tt) * kv_dim + static_cast<size_t>(g) * hd + cc * 8;
      __half* dst = ks + tt * hd + ((cc ^ (tt & 7)) * 8);
      if (r0 + tt != own)
        ac_cp16(dst, a.k + src);
      else if (!defer_own)
        ac_put_own(a.new_k + static_cast<size_t>(g) * hd + cc * 8, dst, a.kw + src);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    for (int i = tid; i < np * cpr; i += kAcThreads) {
      const int tt = i / cpr, cc = i % cpr;
      const size_t src = static_cast<size_t>(r0 + tt) * kv_dim + static_cast<size_t>(g) * hd + cc * 8;
      __half* dst = vs + tt * hd + ((cc ^ (tt & 7)) * 8);
      if (r0 + tt != own)
        ac_cp16(dst, a.v + src);
      else if (!defer_own)
        ac_put_own(a.new_v + static_cast<size_t>(g) * hd + cc * 8, dst, a.vw + src);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    if (r0 == lo && a.pdl) {
      // the cached rows are on their way: now wait for the kernel that wrote q
      // and the token's key and value, and only then let the next kernel
      // start (so it cannot overlap that one)
      griddep_wait();
      griddep_launch_dependents();
      if (own >= r0 && own < r0 + np) {
        const int tt = own - r0;
        const size_t src = static_cast<size_t>(own) * kv_dim + static_cast<size_t>(g) * hd;
        for (int cc = tid; cc < cpr; cc += kAcThreads) {
          ac_put_own(a.new_k + static_cast<size_t>(g) * hd + cc * 8, ks + tt * hd + ((cc ^ (tt & 7)) * 8),
                     a.kw + src + cc * 8);
          ac_put_own(a.new_v + static_cast<size_t>(g) * hd + cc * 8, vs + tt * hd + ((cc ^ (tt & 7)) * 8),
                     a.vw + src + cc * 8);
        }
      }
    }
    // while the copies fly: value rows of the last tile past the context hold
    // 0 (never stale bits that could be NaN), and on the first round q and the
    // weights' rows of heads past the group are zeroed and q staged
    for (int i = tid; i < (ntiles * 16 - np) * cpr; i += kAcThreads)
      reinterpret_cast<uint4*>(vs + (np + i / cpr) * hd)[i % cpr] = make_uint4(0u, 0u, 0u, 0u);
    if (r0 == lo) {
      uint4* z = reinterpret_cast<uint4*>(qh);
      for (int i = tid; i < (2 * 16 * QS + 2 * 16 * PS) / 8; i += kAcThreads) z[i] = make_uint4(0u, 0u, 0u, 0u);
      __syncthreads();
      for (int i = tid; i < group * hd; i += kAcThreads) {
        const int j = i / hd, d = i % hd;
        __half h, l;
        split_half(a.q[static_cast<size_t>(g * group) * hd + i] * a.scale, h, l);
        qh[j * QS + d] = h;
        ql[j * QS + d] = l;
      }
    }
    asm volatile("cp.async.wait_group 1;" ::: "memory");   // the keys
    __syncthreads();

    // scores of the warp's position tiles (tile = 16 positions): sc[slot][nt]
    // = rows: positions tile*16 + gq (+8), columns: heads nt*8 + 2tq (+1)
    float sc[2][NTS][4];
#pragma unroll
    for (int ti = 0; ti < 2; ++ti) {
#pragma unroll
      for (int nt = 0; nt < NTS; ++nt) sc[ti][nt][0] = sc[ti][nt][1] = sc[ti][nt][2] = sc[ti][nt][3] = 0.f;
      const int tl = warp + 8 * ti;
      if (tl < ntiles) {
        const int mi = lane >> 3;
        const int krow = tl * 16 + (lane & 7) + (mi & 1) * 8;
        for (int kk = 0; kk < hd / 16; ++kk) {
          uint32_t a0, a1, a2, a3;
          const int chunk = 2 * kk + (mi >> 1);
          ldsm_x4(a0, a1, a2, a3, ks + krow * hd + ((chunk ^ (krow & 7)) * 8));
#pragma unroll
          for (int nt = 0; nt < NTS; ++nt) {
            const int qoff = (nt * 8 + (lane & 7)) * QS + 16 * kk + (mi & 1) * 8;
            uint32_t b0, b1, c0, c1;
            ldsm_x2(b0, b1, qh + qoff);
            ldsm_x2(c0, c1, ql + qoff);
            ac_mma(sc[ti][nt], a0, a1, a2, a3, b0, b1);
            ac_mma(sc[ti][nt], a0, a1, a2, a3, c0, c1);
          }
        }
      }
    }
    // the round's maximum per head: the lane's positions, the warp (shuffles
    // over gq), then the warps in order
    float mx[NTS][2];
#pragma unroll
    for (int nt = 0; nt < NTS; ++nt) {
      mx[nt][0] = mx[nt][1] = -INFINITY;
#pragma unroll
      for (int ti = 0; ti < 2; ++ti) {
        const int p0 = (warp + 8 * ti) * 16 + gq;
        if (p0 < np) {
          mx[nt][0] = fmaxf(mx[nt][0], sc[ti][nt][0]);
          mx[nt][1] = fmaxf(mx[nt][1], sc[ti][nt][1]);
        }
        if (p0 + 8 < np) {
          mx[nt][0] = fmaxf(mx[nt][0], sc[ti][nt][2]);
          mx[nt][1] = fmaxf(mx[nt][1], sc[ti][nt][3]);
        }
      }
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        mx[nt][0] = fmaxf(mx[nt][0], __shfl_xor_sync(0xffffffffu, mx[nt][0], o));
        mx[nt][1] = fmaxf(mx[nt][1], __shfl_xor_sync(0xffffffffu, mx[nt][1], o));
      }
      if (gq == 0) {
        wred[warp][nt * 8 + 2 * tq] = mx[nt][0];
        wred[warp][nt * 8 + 2 * tq + 1] = mx[nt][1];
      }
    }
    __syncthreads();
    if (tid < group) {
      float bm = wred[0][tid];
      for (int w = 1; w < kAcWarps; ++w) bm = fmaxf(bm, wred[w][tid]);
      const float m_new = fmaxf(hm[tid], bm);
      hc[tid] = expf(hm[tid] - m_new);   // 0 on the first round (m = -inf)
      hm[tid] = m_new;
    }
    __syncthreads();
    // weights exp(s - m) of the group's heads (0 past the context), as binary16
    // hi + lo, and their sums per head
    float sm_[NTS][2];
#pragma unroll
    for (int nt = 0; nt < NTS; ++nt) {
      const int h0 = nt * 8 + 2 * tq;
      const float m0 = h0 < group ? hm[h0] : 0.f, m1 = h0 + 1 < group ? hm[h0 + 1] : 0.f;
      sm_[nt][0] = sm_[nt][1] = 0.f;
#pragma unroll
      for (int ti = 0; ti < 2; ++ti) {
        const int tl = warp + 8 * ti;
        if (tl < ntiles) {
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int pos = tl * 16 + gq + 8 * hh;
            const float p0 = (pos < np && h0 < group) ? expf(sc[ti][nt][2 * hh] - m0) : 0.f;
            const float p1 = (pos < np && h0 + 1 < group) ? expf(sc[ti][nt][2 * hh + 1] - m1) : 0.f;
            sm_[nt][0] += p0;
            sm_[nt][1] += p1;
            if (h0 < group) split_half(p0, ph[h0 * PS + pos], pl[h0 * PS + pos]);
            if (h0 + 1 < group) split_half(p1, ph[(h0 + 1) * PS + pos], pl[(h0 + 1) * PS + pos]);
          }
        }
      }
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        sm_[nt][0] += __shfl_xor_sync(0xffffffffu, sm_[nt][0], o);
        sm_[nt][1] += __shfl_xor_sync(0xffffffffu, sm_[nt][1], o);
      }
    }
    __syncthreads();   // every warp has read the maxima's exchange buffer
#pragma unroll
    for (int nt = 0; nt < NTS; ++nt) {
      if (gq == 0) {
        wred[warp][nt * 8 + 2 * tq] = sm_[nt][0];
        wred[warp][nt * 8 + 2 * tq + 1] = sm_[nt][1];
      }
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");   // the values
    __syncthreads();
    if (tid < group) {
      float ls = wred[0][tid];
      for (int w = 1; w < kAcWarps; ++w) ls += wred[w][tid];
      hl[tid] = fmaf(hl[tid], hc[tid], ls);
    }
    // weighted values: oacc = oacc * corr + P V over the round's positions
    {
      const float c0 = gq < group ? hc[gq] : 0.f, c1 = gq + 8 < group ? hc[gq + 8] : 0.f;
#pragma unroll
      for (int nt = 0; nt < NTV; ++nt) {
        oacc[nt][0] *= c0;
        oacc[nt][1] *= c0;
        oacc[nt][2] *= c1;
        oacc[nt][3] *= c1;
      }
      const int mi = lane >> 3;
      for (int kk = 0; kk < ntiles; ++kk) {
        uint32_t a0, a1, a2, a3, e0, e1, e2, e3;
        const int poff = ((lane & 7) + (mi & 1) * 8) * PS + 16 * kk + (mi >> 1) * 8;
        ldsm_x4(a0, a1, a2, a3, ph + poff);
        ldsm_x4(e0, e1, e2, e3, pl + poff);
        const int vrow = 16 * kk + (lane & 7) + (mi & 1) * 8;
#pragma unroll
        for (int nt = 0; nt + 1 < NTV; nt += 2) {
          const int chunk = ((d0 + nt * 8) >> 3) + (mi >> 1);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(b0, b1, b2, b3, vs + vrow * hd + ((chunk ^ (vrow & 7)) * 8));
          ac_mma(oacc[nt], a0, a1, a2, a3, b0, b1);
          ac_mma(oacc[nt], e0, e1, e2, e3, b0, b1);
          ac_mma(oacc[nt + 1], a0, a1, a2, a3, b2, b3);
          ac_mma(oacc[nt + 1], e0, e1, e2, e3, b2, b3);
        }
        if (NTV & 1) {
          const int chunk = (d0 + (NTV - 1) * 8) >> 3;
          uint32_t b0, b1;
          ldsm_x2_t(b0, b1, vs + vrow * hd + ((chunk ^ (vrow & 7)) * 8));
          ac_mma(oacc[NTV - 1], a0, a1, a2, a3, b0, b1);
          ac_mma(oacc[NTV - 1], e0, e1, e2, e3, b0, b1);
        }
      }
    }
    __syncthreads();   // the round's buffers are free for the next one
  }

  if (a.pdl && lo >= hi) {   // a CTA past the context: nothing was copied early
    griddep_wait();
    griddep_launch_dependents();
  }
  // this CTA's state for the cluster: m and l (hm, hl) and o [group][hd]
#pragma unroll
  for (int nt = 0; nt < NTV; ++nt) {
    const int d = d0 + nt * 8 + 2 * tq;
    if (gq < group) {
      osm[gq * hd + d] = oacc[nt][0];
      osm[gq * hd + d + 1] = oacc[nt][1];
    }
    if (gq + 8 < group) {
      osm[(gq + 8) * hd + d] = oacc[nt][2];
      osm[(gq + 8) * hd + d + 1] = oacc[nt][3];
    }
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
    rm[tid] = *cluster.map_shared_rank(hm + j, rr);
    rl[tid] = *cluster.map_shared_rank(hl + j, rr);
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

template <int NTS, int NTV>
cudaError_t ac_set_attr(bool nonportable) {
  cudaError_t e = cudaFuncSetAttribute(attn_mma_kernel<NTS, NTV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kAcSmemMax));
  if (e == cudaSuccess && nonportable)
    e = cudaFuncSetAttribute(attn_mma_kernel<NTS, NTV>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return e;
}

cudaError_t ac_set_attrs(bool nonportable) {
  cudaError_t e = ac_set_attr<1, 1>(nonportable);
  if (e == cudaSuccess) e = ac_set_attr<1, 2>(nonportable);
  if (e == cudaSuccess) e = ac_set_attr<1, 3>(nonportable);
  if (e == cudaSuccess) e = ac_set_attr<1, 4>(nonportable);
  if (e == cudaSuccess) e = ac_set_attr<2, 1>(nonportable);
  if (e == cudaSuccess) e = ac_set_attr<2, 2>(nonportable);
  if (e == cudaSuccess) e = ac_set_attr<2, 3>(nonportable);
  if (e == cudaSuccess) e = ac_set_attr<2, 4>(nonportable);
  return e;
}

}  // namespace

// Positions per round: 64 KB of keys and values (256 positions at head_dim
// 64, 128 at 128, 64 above), so that a cluster's CTAs use under 105 KB of
// shared memory, two fit on an SM, and every value head's cluster is resident
// at once (at 139 KB per CTA a GB300 holds only 7 clusters of 16).
int attn_cluster_round(int hd) { return hd <= 64 ? 256 : hd <= 128 ? 128 : 64; }

size_t attn_cluster_smem(int group, int hd) {
  const int R = attn_cluster_round(hd);
  return static_cast<size_t>(2) * R * hd * 2 + static_cast<size_t>(2) * 16 * (hd + 8) * 2 +
         static_cast<size_t>(2) * 16 * (R + 8) * 2 + static_cast<size_t>(group) * hd * 4;
}

// Cluster size: 16 when one such cluster with the largest shared memory fits
// on the GPU, else the portable 8.
cudaError_t attn_cluster_prepare() {
  cudaError_t e = cudaSuccess;
  bool big = ac_set_attrs(true) == cudaSuccess;
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
    big = cudaOccupancyMaxActiveClusters(&n, attn_mma_kernel<2, 4>, &cfg) == cudaSuccess && n >= 1;
    cudaGetLastError();
  }
  if (!big) e = ac_set_attrs(false);
  g_ac_cluster = big ? 16 : 8;
  return e;
}

cudaError_t attn_cluster_launch(const float* q, const uint16_t* k, const uint16_t* v, const int* ctx_len, int ctx_add,
                                int capacity, int n_q, int n_kv, int hd, uint16_t* out, const AttnAppend* app,
                                cudaStream_t s) {
  // 16 CTAs per value head where the GPU schedules such clusters, except up to
  // 1024 positions: there 8 (fewer partial states to combine outweighs the
  // copies' parallelism; measured on the 8B heads at 512, 1024 and 2048)
  const int C = g_ac_cluster == 16 && capacity <= 1024 ? 8 : g_ac_cluster;
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
  a.pdl = app && app->pdl ? 1 : 0;
  const int group = n_q / n_kv;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C, n_kv);
  cfg.blockDim = dim3(kAcThreads);
  cfg.dynamicSmemBytes = attn_cluster_smem(group, hd);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.pdl ? 2 : 1;
  // score tiles of 8 heads: 1 up to 8 query heads per value head, else 2;
  // value tiles of 8 dimensions per warp: head_dim / 64
  const int ntv = hd / 64;
  if (group <= 8) {
    if (ntv == 1) return cudaLaunchKernelEx(&cfg, attn_mma_kernel<1, 1>, a);
    if (ntv == 2) return cudaLaunchKernelEx(&cfg, attn_mma_kernel<1, 2>, a);
    if (ntv == 3) return cudaLaunchKernelEx(&cfg, attn_mma_kernel<1, 3>, a);
    return cudaLaunchKernelEx(&cfg, attn_mma_kernel<1, 4>, a);
  }
  if (ntv == 1) return cudaLaunchKernelEx(&cfg, attn_mma_kernel<2, 1>, a);
  if (ntv == 2) return cudaLaunchKernelEx(&cfg, attn_mma_kernel<2, 2>, a);
  if (ntv == 3) return cudaLaunchKernelEx(&cfg, attn_mma_kernel<2, 3>, a);
  return cudaLaunchKernelEx(&cfg, attn_mma_kernel<2, 4>, a);
}

}  // namespace q4
