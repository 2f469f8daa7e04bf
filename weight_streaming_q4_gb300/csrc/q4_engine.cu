// Persistent, warp-specialised Q4_0 matrix-vector engine for sm_103a.
//
// One CTA per SM.  Warp 15 is the producer: one lane streams the CTA's work
// units (consecutive weight rows, contiguous in the GGUF row-major layout)
// from HBM into a 5- or 6-deep ring of 31.5 KB shared-memory stages with 1-D bulk
// TMA copies (cp.async.bulk) whose completion is counted on one mbarrier
// per stage.  Warps 0-14 are the consumers: each thread keeps a fixed slice
// of 64 columns of the input vector x in registers, reads its slice of two
// staged rows per unit, unpacks the 4-bit codes in registers and
// accumulates the exact products (q - 8) * x in fp32.  Row sums are reduced
// with warp shuffles; rows wider than one warp's slice leave one partial per
// warp in shared memory, summed in a fixed order when the phase ends (no
// barrier per unit).  The work of a launch is a list of phases
// (matrix-vector products with an input prologue and an output epilogue),
// while the producer keeps streaming the next phase's weights, which never
// depend on the activations.  Two instantiations synchronise the phases
// differently: engine_kernel<false> meets at a flag barrier after every
// phase; engine_kernel<true> (tagged programs) passes every value one phase
// hands to the next as a tagged word and has each CTA poll the words of its
// own input, with one flag exchange per layer.
//
// The method: PIPO's dequantisation-free 4-bit matrix-vector product
// ("PIPO: Pipelined Offloading for Efficient Inference on Consumer
// Devices", Method, "Computation optimization") run layer by layer (same
// page, "Offloading architecture"), with the weights of the next unit
// prefetched while the current one computes (PipeLLM page, "Layer 2:
// Asynchronous Weight Prefetching").
//
// Exactness of the block dot product: a code q is placed in the mantissa of
// 2^23 (bits p..p+3 for p in {0,4,8,12}), so the float equals 2^23 + q*2^p
// exactly; subtracting 2^23 + 8*2^p gives (q - 8)*2^p exactly, and the matching
// x was stored pre-multiplied by 2^-p (exact).  Each product (q - 8) * x is
// therefore exact, a block of all-8 codes contributes exactly zero, and a
// block with one non-8 code contributes exactly fl(d * (q - 8) * x).
#include <cuda_fp16.h>
#include <stdint.h>

#include "q4_device.cuh"
#include "q4_phase.cuh"

namespace q4 {

__device__ int g_status;   // status bits of launches without a control block


// Column order of the 8 codes of one 32-bit word of a block's code bytes
// (bytes 4m..4m+3 hold elements 4m..4m+3 low and 4m+16..4m+19 high).  The
// word and the word shifted right by 16 give the codes in pairs that sit at
// the same bit position p: (4m, 4m+2) at p=0, (4m+16, 4m+18) at p=4,
// (4m+1, 4m+3) at p=8, (4m+17, 4m+19) at p=12.
__device__ __forceinline__ constexpr int elem_off(int e) {
  return e == 0 ? 0 : e == 1 ? 2 : e == 2 ? 16 : e == 3 ? 18 : e == 4 ? 1 : e == 5 ? 3 : e == 6 ? 17 : 19;
}
__device__ __forceinline__ constexpr int elem_shift(int e) { return 4 * (e >> 1); }

typedef unsigned long long u64;

// (a & MASK) | magic as one three-input logic op, the magic held in a register.
template <uint32_t MASK>
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t magic) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "n"(MASK), "r"(magic));
  return d;
}
__device__ __forceinline__ u64 pack2(uint32_t lo, uint32_t hi) {
  u64 d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "r"(lo), "r"(hi));
  return d;
}
__device__ __forceinline__ u64 add2(u64 a, u64 b) {
  u64 d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ u64 fma2(u64 a, u64 b, u64 c) {
  u64 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ float hsum2(u64 a) {
  return __uint_as_float(static_cast<uint32_t>(a)) + __uint_as_float(static_cast<uint32_t>(a >> 32));
}

// Constants of the exact unpack, kept in registers: the magic 2^23 and the
// four bias pairs 2^23 + 8 * 2^p.
struct Unpack {
  uint32_t magic;
  u64 bias[4];
};

__device__ __forceinline__ Unpack make_unpack() {
  Unpack u;
  asm volatile("mov.b32 %0, 0x4B000000;" : "=r"(u.magic));   // opaque: stays a register operand
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float b = -(8388608.0f + 8.0f * static_cast<float>(1 << (4 * i)));
    const uint32_t bb = __float_as_uint(b);
    asm volatile("mov.b64 %0, {%1, %1};" : "=l"(u.bias[i]) : "r"(bb));
  }
  return u;
}

// Accumulate the 8 exact products of one code word into acc (two lanes).
__device__ __forceinline__ u64 word_dot(uint32_t w, const u64* xs, u64 acc, const Unpack& k) {
  const uint32_t h = w >> 16;
  u64 v0 = pack2(and_or<0xFu>(w, k.magic), and_or<0xFu>(h, k.magic));
  u64 v1 = pack2(and_or<0xF0u>(w, k.magic), and_or<0xF0u>(h, k.magic));
  u64 v2 = pack2(and_or<0xF00u>(w, k.magic), and_or<0xF00u>(h, k.magic));
  u64 v3 = pack2(and_or<0xF000u>(w, k.magic), and_or<0xF000u>(h, k.magic));
  v0 = add2(v0, k.bias[0]);
  v1 = add2(v1, k.bias[1]);
  v2 = add2(v2, k.bias[2]);
  v3 = add2(v3, k.bias[3]);
  acc = fma2(v0, xs[0], acc);
  acc = fma2(v1, xs[1], acc);
  acc = fma2(v2, xs[2], acc);
  acc = fma2(v3, xs[3], acc);
  return acc;
}

// Dot product of one 64-column slice (two blocks = 36 bytes starting at a
// 4-byte aligned shared-memory address) with the thread's 32 pairs of x.
__device__ __forceinline__ float pair_dot(const uint8_t* p, const u64* xs, float tot, const Unpack& k) {
  const uint32_t* pw = reinterpret_cast<const uint32_t*>(p);
  uint32_t W[9];
#pragma unroll
  for (int i = 0; i < 9; ++i) W[i] = pw[i];
  const float d0 = __half2float(__ushort_as_half(static_cast<unsigned short>(W[0] & 0xFFFFu)));
  const float d1 = __half2float(__ushort_as_half(static_cast<unsigned short>(W[4] >> 16)));
  u64 a0 = 0, a1 = 0, b0 = 0, b1 = 0;
  // block 0: code bytes start 2 bytes into word 0
  a0 = word_dot(__funnelshift_r(W[0], W[1], 16), xs + 0, a0, k);
  a1 = word_dot(__funnelshift_r(W[1], W[2], 16), xs + 4, a1, k);
  a0 = word_dot(__funnelshift_r(W[2], W[3], 16), xs + 8, a0, k);
  a1 = word_dot(__funnelshift_r(W[3], W[4], 16), xs + 12, a1, k);
  // block 1: code bytes are words 5..8
  b0 = word_dot(W[5], xs + 16, b0, k);
  b1 = word_dot(W[6], xs + 20, b1, k);
  b0 = word_dot(W[7], xs + 24, b0, k);
  b1 = word_dot(W[8], xs + 28, b1, k);
  tot = fmaf(d0, hsum2(a0) + hsum2(a1), tot);
  tot = fmaf(d1, hsum2(b0) + hsum2(b1), tot);
  return tot;
}

// The dot products of two rows' 64-column slices with the same x, word by
// word for both rows so that the two rows' dependency chains interleave.
__device__ __forceinline__ void pair_dot2(const uint8_t* pa, const uint8_t* pb, const u64* xs, float& ta, float& tb,
                                          const Unpack& k) {
  const uint32_t* qa = reinterpret_cast<const uint32_t*>(pa);
  const uint32_t* qb = reinterpret_cast<const uint32_t*>(pb);
  uint32_t A[9], B[9];
#pragma unroll
  for (int i = 0; i < 9; ++i) {
    A[i] = qa[i];
    B[i] = qb[i];
  }
  u64 a0 = 0, a1 = 0, b0 = 0, b1 = 0, c0 = 0, c1 = 0, e0 = 0, e1 = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t wa = __funnelshift_r(A[i], A[i + 1], 16), wb = __funnelshift_r(B[i], B[i + 1], 16);
    if (i & 1) {
      a1 = word_dot(wa, xs + 4 * i, a1, k);
      c1 = word_dot(wb, xs + 4 * i, c1, k);
    } else {
      a0 = word_dot(wa, xs + 4 * i, a0, k);
      c0 = word_dot(wb, xs + 4 * i, c0, k);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (i & 1) {
      b1 = word_dot(A[5 + i], xs + 16 + 4 * i, b1, k);
      e1 = word_dot(B[5 + i], xs + 16 + 4 * i, e1, k);
    } else {
      b0 = word_dot(A[5 + i], xs + 16 + 4 * i, b0, k);
      e0 = word_dot(B[5 + i], xs + 16 + 4 * i, e0, k);
    }
  }
  const float da0 = __half2float(__ushort_as_half(static_cast<unsigned short>(A[0] & 0xFFFFu)));
  const float da1 = __half2float(__ushort_as_half(static_cast<unsigned short>(A[4] >> 16)));
  const float db0 = __half2float(__ushort_as_half(static_cast<unsigned short>(B[0] & 0xFFFFu)));
  const float db1 = __half2float(__ushort_as_half(static_cast<unsigned short>(B[4] >> 16)));
  ta = fmaf(da1, hsum2(b0) + hsum2(b1), fmaf(da0, hsum2(a0) + hsum2(a1), 0.f));
  tb = fmaf(db1, hsum2(e0) + hsum2(e1), fmaf(db0, hsum2(c0) + hsum2(c1), 0.f));
}

__device__ __forceinline__ void set_status(Control* ctl, int bits) {
  atomicOr(ctl ? &ctl->status : &g_status, bits);
}

// Load the thread's 64 consecutive columns [c0, c0 + 64) of the phase input
// (before any normalisation) as floats, with 16-byte loads through L1: the
// row teams of a CTA share the same slices, so one line fill serves them all.
// The data was written by other CTAs before this phase's flags were seen.
// For the attention gather the 64 columns lie in one query head (head_dim is
// a multiple of 64), so they map to 64 consecutive values of one value head.
__device__ __forceinline__ void load_x_slice(const Phase& ph, int c0, float* v) {
  if (ph.x_kind == X_F16 || ph.x_kind == X_NORM16) {
    // natural layout: the thread's 128 bytes; slice-transposed: chunk i of
    // slice j at (i * T + j) * 16 bytes, so a warp's loads are contiguous
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const __half*>(ph.x_src) + (ph.x_t ? 0 : c0));
    const int step = ph.x_t ? ph.x_ld : 1;
    if (ph.x_t) p += c0 / kKT;
#pragma unroll
    for (int i = 0; i < kKT / 8; ++i) {
      const uint4 u = p[i * step];
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[t]));
        v[8 * i + 2 * t] = f.x;
        v[8 * i + 2 * t + 1] = f.y;
      }
    }
  } else {
    int src0 = c0;
    if (ph.x_kind == X_ATTN) {
      const int hd = ph.head_dim;
      src0 = (ph.x_t ? 0 : ph.attn_off) + ((c0 / hd) / ph.group) * hd + (c0 % hd);
    }
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(ph.x_src)) +
                      (ph.x_t ? src0 / kKT : src0 / 4);
    const int step = ph.x_t ? ph.x_ld : 1;
#pragma unroll
    for (int i = 0; i < kKT / 4; ++i) {
      const float4 f = p[i * step];
      v[4 * i] = f.x;
      v[4 * i + 1] = f.y;
      v[4 * i + 2] = f.z;
      v[4 * i + 3] = f.w;
    }
  }
}

// Geometry of a phase as the consumers see it.
struct Tile {
  int team_threads, teams, team, j, tw, spu, rpu, w_in_team;
  bool active, dual;
  uint32_t row_bytes;
};

__device__ __forceinline__ Tile tile_of(const Phase& ph, int tid) {
  Tile t;
  t.team_threads = ph.k / kKT;
  t.teams = ph.teams;
  t.team = tid / t.team_threads;
  t.j = tid % t.team_threads;
  t.active = t.team < t.teams;
  t.tw = t.team_threads >= 32 ? t.team_threads / 32 : 1;   // partials per row (one per warp)
  t.w_in_team = t.team_threads >= 32 ? (tid / 32 - t.team * t.tw) : 0;
  t.spu = 2 * t.teams;                                     // row slots per unit
  t.dual = ph.epi_kind == EPI_SILU;
  t.rpu = ph.rows_per_unit;
  t.row_bytes = static_cast<uint32_t>(ph.k / kQK) * kBlockBytes;
  return t;
}

// xs2 from the thread's 64 binary16 inputs: 32 float2 in the order pair_dot
// expects, each value pre-scaled by 2^-shift (exact).
__device__ __forceinline__ void xs2_from_halves(const __half* xv, u64* xs2) {
#pragma unroll
  for (int blk = 0; blk < kKT / 32; ++blk) {
#pragma unroll
    for (int m = 0; m < 4; ++m) {
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        const float a =
            __half2float(xv[blk * 32 + 4 * m + elem_off(e)]) * (1.0f / static_cast<float>(1 << elem_shift(e)));
        const float b = __half2float(xv[blk * 32 + 4 * m + elem_off(e + 1)]) *
                        (1.0f / static_cast<float>(1 << elem_shift(e + 1)));
        xs2[blk * 16 + m * 4 + e / 2] = pack2(__float_as_uint(a), __float_as_uint(b));
      }
    }
  }
}

// Team 0 of CTA 0 leaves the formed x of a phase: plain binary16 in x_dbg,
// and tagged binary16 words in xr_out (the residual base a later phase reads).
__device__ __forceinline__ void store_formed_x(const Phase& ph, int k0, const __half* xv, uint32_t tag16) {
  if (ph.x_dbg) {
    uint4* d = reinterpret_cast<uint4*>(ph.x_dbg + k0);
#pragma unroll
    for (int i = 0; i < kKT / 8; ++i) d[i] = reinterpret_cast<const uint4*>(xv)[i];
  }
  if (ph.xr_out) {
    const uint32_t t = tag16 << 16;
#pragma unroll
    for (int i = 0; i < kKT / 4; ++i)
      st_relaxed_v4(ph.xr_out + k0 + 4 * i,
                    make_uint4(__half_as_ushort(xv[4 * i]) | t, __half_as_ushort(xv[4 * i + 1]) | t,
                               __half_as_ushort(xv[4 * i + 2]) | t, __half_as_ushort(xv[4 * i + 3]) | t));
  }
}

// Form the thread's slice of x for a phase with an untagged input: columns
// [64 j, 64 j + 64) belong to the thread.  All loads are issued before any
// dependent arithmetic, so the prologue costs one round trip to L2.
__device__ void form_x(const Phase& ph, int j, int lane, u64* xs2, bool team0_cta0, float sumsq, uint32_t tag16) {
  const bool norm = ph.x_kind == X_NORM16 || ph.x_kind == X_NORM32;
  const int k0 = j * kKT;
  float v[kKT];
  load_x_slice(ph, k0, v);
  if (ph.x_kind == X_NORM16) sumsq = input_sumsq16(ph, lane);
  const float r = norm ? rsqrtf(sumsq / static_cast<float>(ph.k) + ph.eps) : 1.0f;
  __half xv[kKT];
#pragma unroll
  for (int e = 0; e < kKT; e += 2) {
    const __half2 hp = norm ? __floats2half2_rn(v[e] * r, v[e + 1] * r) : __floats2half2_rn(v[e], v[e + 1]);
    xv[e] = __low2half(hp);
    xv[e + 1] = __high2half(hp);
  }
  if (team0_cta0) store_formed_x(ph, k0, xv, tag16);   // before xs2 is formed: fewer live registers
  xs2_from_halves(xv, xs2);
}

// ------------------------------------------------------------ tagged inputs
//
// A tagged input is staged once per CTA: every consumer thread polls a share
// of its 16-byte chunks (all of them in flight at once) until the tags match,
// and writes the values to shared memory; each thread then reads its own 64
// columns from there.  Nothing is read from L2 twice by one CTA.  Binary16
// inputs are staged as binary16; the RMSNorm inputs are staged as fp32 with
// the scale returned, and normalised when each thread reads its columns.

// Positions in the stage.  binary16: the 16-byte chunk q of the 64-value slice
// s sits at chunk q ^ (s & 7) of that slice; fp32: chunk q of slice s at
// q ^ (s & 15).  Either way the 16-byte loads with which consecutive threads
// read consecutive slices fall in different banks.
__device__ __forceinline__ int stage_pos16(int e) { return (e & ~63) | ((((e >> 3) ^ (e >> 6)) & 7) << 3) | (e & 7); }
__device__ __forceinline__ int stage_pos32(int e) {
  return (e & ~63) | ((((e >> 2) ^ (e >> 6)) & 15) << 2) | (e & 3);
}

// The n values of a tagged binary16 input into the stage (n a multiple of 4,
// at most kTag16MaxValues).  All consumer threads.  Each pass loads all of the
// thread's chunks at once and stores them; the thread repeats the pass until
// every tag was the expected one (a pass keeps no values across iterations,
// which keeps the registers of the poll few).
__device__ __forceinline__ void stage_tag16(const uint32_t* src, int n, uint16_t* stage, uint32_t tag16, uint32_t limit,
                                            Control* ctl, int tid) {
  constexpr int kC = (kTag16MaxValues / 4 + kConsumerThreads - 1) / kConsumerThreads;
  const int nch = n >> 2;
  const uint32_t want = tag16 << 16;
  for (uint32_t it = 0; it < limit; ++it) {
    bool ok = true;
#pragma unroll
    for (int c = 0; c < kC; ++c) {
      const int i = tid + c * kConsumerThreads;
      if (i < nch) {
        const uint4 w = ld_relaxed_v4(src + 4 * i);
        ok &= (((w.x ^ want) | (w.y ^ want) | (w.z ^ want) | (w.w ^ want)) >> 16) == 0u;
        *reinterpret_cast<uint2*>(stage + stage_pos16(4 * i)) = make_uint2(__byte_perm(w.x, w.y, 0x5410),
                                                                            __byte_perm(w.z, w.w, 0x5410));
      }
    }
    if (ok) return;
    if (it >= 2) __nanosleep(32);
  }
  set_status(ctl, ST_DATA_TIMEOUT);
}

// The RMSNorm scale of a staged fp32 input: the sum of squares of each
// thread's chunks (2 values each, chunk i = tid + c * kConsumerThreads) in
// order, then over the warps in order -- a fixed order that depends only on
// n, so every CTA computes the same scale.  One CTA barrier inside.
__device__ __forceinline__ float stage_norm_scale(const float* xf, int n, int per, float eps, float* red_cta, int tid,
                                                  int warp, int lane) {
  float ss = 0.f;
  for (int i = tid * per; i < n; i += kConsumerThreads * per)
    for (int q = 0; q < per; ++q) {
      const float v = xf[stage_pos32(i + q)];
      ss = fmaf(v, v, ss);
    }
  ss = warp_sum(ss);
  if (lane == 0) red_cta[warp] = ss;
  named_bar_sync(1, kConsumerThreads);
  float tot = 0.f;
  for (int w = 0; w < kConsumerWarps; ++w) tot += red_cta[w];
  return rsqrtf(tot / static_cast<float>(n) + eps);
}

// A tagged fp32 input of n values (n even, at most kNormMaxValues) into the
// stage, polled as in stage_tag16; returns its RMSNorm scale.  All consumer
// threads.
__device__ __forceinline__ float stage_tag32_norm(const unsigned long long* src, int n, float eps, float* xf,
                                                  uint32_t tag, uint32_t limit, Control* ctl, float* red_cta,
                                                  int tid, int warp, int lane) {
  constexpr int kC = (kNormMaxValues / 2 + kConsumerThreads - 1) / kConsumerThreads;
  const int nch = n >> 1;
  bool ok = false;
  for (uint32_t it = 0; it < limit && !ok; ++it) {
    ok = true;
#pragma unroll
    for (int c = 0; c < kC; ++c) {
      const int i = tid + c * kConsumerThreads;
      if (i < nch) {
        const uint4 w = ld_relaxed_v4(src + 2 * i);
        ok &= w.y == tag && w.w == tag;
        *reinterpret_cast<float2*>(xf + stage_pos32(2 * i)) = make_float2(__uint_as_float(w.x), __uint_as_float(w.z));
      }
    }
    if (!ok && it >= 2) __nanosleep(32);
  }
  if (!ok) set_status(ctl, ST_DATA_TIMEOUT);
  return stage_norm_scale(xf, n, 2, eps, red_cta, tid, warp, lane);
}

// An untagged binary16 input of n values (the first layer's input, written
// before the launch; n a multiple of 8, at most kNormMaxValues) into the stage as
// fp32; returns its RMSNorm scale.  All consumer threads.
__device__ __forceinline__ float stage_plain16_norm(const uint16_t* src, int n, float eps, float* xf, float* red_cta,
                                                 int tid, int warp, int lane) {
  for (int i = tid; i < (n >> 3); i += kConsumerThreads) {
    const uint4 u = __ldcg(reinterpret_cast<const uint4*>(src) + i);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[h]));
      *reinterpret_cast<float2*>(xf + stage_pos32(8 * i + 2 * h)) = f;
    }
  }
  return stage_norm_scale(xf, n, 8, eps, red_cta, tid, warp, lane);
}

// The prologue of a phase of a tagged program for a CTA that reads its input:
// wait for the previous phase's flags where the phase asks for it, stage the
// whole input (fp32 with its RMSNorm scale for the norms, which it returns),
// and meet at a CTA barrier.  Kept out of line so that the unit loop's
// registers are allocated without the staging loads in flight.
__device__ __noinline__ float tagged_prologue(const Phase& ph, unsigned tag, uint32_t lim, Control* ctl,
                                             const unsigned long long* flags, float* xbuf, float* red_cta, int tid,
                                             int warp, int lane) {
  float r = 1.f;
  if (ph.sync == SYNC_WAIT && warp == 0) wait_phase_flags(flags, tag - 1u, lane, lim, ctl);
  if (ph.x_kind == X_NORM16)
    r = stage_plain16_norm(static_cast<const uint16_t*>(ph.x_src), ph.k, ph.eps, xbuf, red_cta, tid, warp, lane);
  else if (ph.x_kind == X_TAG32_NORM)
    r = stage_tag32_norm(static_cast<const unsigned long long*>(ph.x_src), ph.k, ph.eps, xbuf, tag - 1u, lim, ctl,
                         red_cta, tid, warp, lane);
  else
    stage_tag16(static_cast<const uint32_t*>(ph.x_src), ph.x_kind == X_TAG16_ATTN ? ph.xt_n : ph.k,
                reinterpret_cast<uint16_t*>(xbuf), (tag - 1u) & 0xFFFFu, lim, ctl, tid);
  named_bar_sync(1, kConsumerThreads);
  return r;
}

// Sum the buffered per-warp partials of n_buf units (the CTA's units
// u_first, u_first + G, ...) and run the epilogue of their rows.  All
// consumer threads take part.  Returns the thread's sum of squares of the
// residual sums it wrote (EPI_RESID), for the next phase's RMSNorm.
__device__ float flush_rows(const Phase& ph, const Tile& t, const float* red, int n_buf, int u_first, int G,
                            int tid, bool reuse) {
  constexpr int kPre = 4;   // residual inputs prefetched per thread (the rest load in the loop)
  const int n_slots = n_buf * t.spu;
  float ss = 0.f;
  if (!t.dual) {
    // residual inputs are loaded before the barrier so their latency overlaps it
    unsigned short res[kPre];
    if (ph.epi_kind == EPI_RESID) {
#pragma unroll
      for (int c = 0; c < kPre; ++c) {
        const int s = tid + c * kConsumerThreads;
        res[c] = 0;
        if (s < n_slots) {
          const int n = (u_first + (s / t.spu) * G) * t.rpu + s % t.spu;
          if (n < ph.n_rows) res[c] = ph.res[n];
        }
      }
    }
    named_bar_sync(1, kConsumerThreads);
    for (int c = 0, s = tid; s < n_slots; ++c, s += kConsumerThreads) {
      float v = 0.f;
      for (int w = 0; w < t.tw; ++w) v += red[s * t.tw + w];
      const int i = s / t.spu, rem = s % t.spu;
      const int n = (u_first + i * G) * t.rpu + rem;   // rem = 2 * team + row of the team
      if (n < ph.n_rows) {
        ph.y[n] = v;
        float out = v;
        if (ph.epi_kind == EPI_RESID) {
          const unsigned short rv = c < kPre ? res[c < kPre ? c : 0] : ph.res[n];
          const float tv = __half2float(__ushort_as_half(rv)) + v;
          ph.y2[n] = tv;
          ss = fmaf(tv, tv, ss);
          out = tv;
        }
        const int e = n - ph.yt_off;
        if (ph.yt && e >= 0 && e < ph.yt_n) static_cast<float*>(ph.yt)[slice_t32(e, ph.yt_n / kKT)] = out;
      }
    }
  } else {
    named_bar_sync(1, kConsumerThreads);
    for (int q = tid; q < n_slots / 2; q += kConsumerThreads) {
      float g = 0.f, u = 0.f;
      for (int w = 0; w < t.tw; ++w) {
        g += red[(2 * q) * t.tw + w];
        u += red[(2 * q + 1) * t.tw + w];
      }
      const int i = (2 * q) / t.spu, tm = ((2 * q) % t.spu) / 2;
      const int n = (u_first + i * G) * t.rpu + tm;
      if (n < ph.n_rows) {
        ph.y[n] = g;
        ph.y2[n] = u;
        const unsigned short a16 = __half_as_ushort(__float2half_rn(silu_mul(g, u)));
        ph.aux16[n] = a16;
        if (ph.yt) static_cast<unsigned short*>(ph.yt)[slice_t16(n, ph.yt_n / kKT)] = a16;
      }
    }
  }
  if (reuse) named_bar_sync(1, kConsumerThreads);   // red is written again in this phase
  return ss;
}

// A tagged residual input word, polled until it carries tag16.
__device__ __forceinline__ unsigned short tagged_res(const uint32_t* p, uint32_t w, uint32_t tag16, uint32_t limit,
                                                     Control* ctl) {
  for (uint32_t it = 0; (w >> 16) != tag16 && it < limit; ++it) {
    __nanosleep(32);
    w = ld_relaxed_b32(p);
  }
  if ((w >> 16) != tag16) set_status(ctl, ST_DATA_TIMEOUT);
  return static_cast<unsigned short>(w & 0xFFFFu);
}

// The epilogue of flush_rows in a tagged program: the same sums, with the
// residual base read from tagged words (the previous phase's tag), the plain
// outputs written where the phase has them (the last layer), and the value
// the next phase reads stored as a tagged word with this phase's tag.
__device__ void flush_rows_tagged(const Phase& ph, const Tile& t, const float* red, int n_buf, int u_first, int G,
                                  int tid, bool reuse, uint32_t tag, uint32_t limit, Control* ctl) {
  constexpr int kPre = 4;   // residual words loaded before the barrier (the rest in the loop)
  const int n_slots = n_buf * t.spu;
  const uint32_t tag16 = tag & 0xFFFFu, prev16 = (tag - 1u) & 0xFFFFu;
  if (!t.dual) {
    const bool resid = ph.epi_kind == EPI_RESID;
    uint32_t res[kPre];
    if (resid) {
#pragma unroll
      for (int c = 0; c < kPre; ++c) {
        const int s = tid + c * kConsumerThreads;
        res[c] = prev16 << 16;
        if (s < n_slots) {
          const int n = (u_first + (s / t.spu) * G) * t.rpu + s % t.spu;
          if (n < ph.n_rows) res[c] = ld_relaxed_b32(ph.res_t + n);
        }
      }
    }
    named_bar_sync(1, kConsumerThreads);
    for (int c = 0, s = tid; s < n_slots; ++c, s += kConsumerThreads) {
      float v = 0.f;
      for (int w = 0; w < t.tw; ++w) v += red[s * t.tw + w];
      const int i = s / t.spu, rem = s % t.spu;
      const int n = (u_first + i * G) * t.rpu + rem;
      if (n >= ph.n_rows) continue;
      if (ph.y) ph.y[n] = v;
      if (resid) {
        const uint32_t w0 = c < kPre ? res[c < kPre ? c : 0] : ld_relaxed_b32(ph.res_t + n);
        const unsigned short rv = tagged_res(ph.res_t + n, w0, prev16, limit, ctl);
        const float tv = __half2float(__ushort_as_half(rv)) + v;
        if (ph.y2) ph.y2[n] = tv;
        st_relaxed_b64(static_cast<unsigned long long*>(ph.yt) + n,
                       (static_cast<unsigned long long>(tag) << 32) | __float_as_uint(tv));
      } else {
        const int e = n - ph.yt_off;
        if (ph.yt && e >= 0 && e < ph.yt_n)
          st_relaxed_b32(static_cast<uint32_t*>(ph.yt) + e, (tag16 << 16) | __half_as_ushort(__float2half_rn(v)));
      }
    }
  } else {
    named_bar_sync(1, kConsumerThreads);
    for (int q = tid; q < n_slots / 2; q += kConsumerThreads) {
      float g = 0.f, u = 0.f;
      for (int w = 0; w < t.tw; ++w) {
        g += red[(2 * q) * t.tw + w];
        u += red[(2 * q + 1) * t.tw + w];
      }
      const int i = (2 * q) / t.spu, tm = ((2 * q) % t.spu) / 2;
      const int n = (u_first + i * G) * t.rpu + tm;
      if (n >= ph.n_rows) continue;
      if (ph.y) ph.y[n] = g;
      if (ph.y2) ph.y2[n] = u;
      const unsigned short a16 = __half_as_ushort(__float2half_rn(silu_mul(g, u)));
      if (ph.aux16) ph.aux16[n] = a16;
      st_relaxed_b32(static_cast<uint32_t*>(ph.yt) + n, (tag16 << 16) | a16);
    }
  }
  if (reuse) named_bar_sync(1, kConsumerThreads);   // red is written again in this phase
}

// flush_rows_tagged for the rare flush in the middle of a phase (its partial
// buffer is full).  Kept inline: an out-of-line call inside the unit loop
// would add register saves around it.
__device__ __forceinline__ void flush_rows_tagged_mid(const Phase& ph, const Tile& t, const float* red, int n_buf,
                                                   int u_first, int G, int tid, uint32_t tag, uint32_t limit,
                                                   Control* ctl) {
  flush_rows_tagged(ph, t, red, n_buf, u_first, G, tid, true, tag, limit, ctl);
}

extern __shared__ __align__(128) uint8_t g_ring[];

// TAGGED selects the synchronisation of a multi-phase launch: tagged words
// between phases (EngineArgs::tagged set), or a flag barrier after every phase.
template <bool TAGGED>
__global__ void __launch_bounds__(kThreads, 1) engine_kernel(const __grid_constant__ EngineArgs a) {
  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ __align__(8) uint64_t empty_bar[kStages];
  // ring depth; row partials (a tagged program keeps them in the staging
  // buffer after the ring: the prologue is over before the first partial is
  // written)
  const int S = TAGGED ? a.stages : kStages;
  __shared__ __align__(16) float red_static[TAGGED ? 4 : kRedFloats];
  float* const red = TAGGED ? reinterpret_cast<float*>(g_ring + static_cast<size_t>(S) * kStageBytes) : red_static;
  uint16_t* const stage = reinterpret_cast<uint16_t*>(red);
  const int red_floats = TAGGED ? a.xbuf_floats : kRedFloats;
  __shared__ float red_cta[kConsumerWarps];
  __shared__ volatile int abort_flag;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, cta = blockIdx.x;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kConsumerWarps);
    }
    fence_mbar_init();
    abort_flag = 0;
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t it = 0;
      int slot = 0;      // it % S: ring stage of the next copy
      uint32_t use = 0;  // it / S: earlier uses of that stage
      for (int p = 0; p < a.n_phases && !abort_flag; ++p) {
        const Phase& ph = a.phases ? a.phases[p] : a.one;
        const uint32_t row_bytes = static_cast<uint32_t>(ph.k / kQK) * kBlockBytes;
        const bool dual = ph.epi_kind == EPI_SILU;
        const int u0 = (cta - ph.base % G + G) % G;
        for (int u = u0; u < ph.units; u += G) {
          if (use > 0 && !mbar_wait_bounded(&empty_bar[slot], (use - 1) & 1, a.wait_limit)) {
            set_status(a.ctl, ST_EMPTY_TIMEOUT);
            abort_flag = 1;
            break;
          }
          if (abort_flag) break;
          const int row0 = u * ph.rows_per_unit;
          const int rows = min(ph.rows_per_unit, ph.n_rows - row0);
          const uint32_t bytes = static_cast<uint32_t>(rows) * row_bytes;
          uint8_t* dst = g_ring + static_cast<size_t>(slot) * kStageBytes;
          mbar_arrive_expect_tx(&full_bar[slot], dual ? 2 * bytes : bytes);
          bulk_g2s(dst, ph.w0 + static_cast<size_t>(row0) * row_bytes, bytes, &full_bar[slot]);
          if (dual)
            bulk_g2s(dst + static_cast<size_t>(ph.rows_per_unit) * row_bytes,
                     ph.w1 + static_cast<size_t>(row0) * row_bytes, bytes, &full_bar[slot]);
          ++it;
          if (++slot == S) {
            slot = 0;
            ++use;
          }
        }
      }
      // Drain: no copy may still be in flight when the CTA exits.
      const uint32_t issued = it;
      for (int s = 0; s < S && static_cast<uint32_t>(s) < issued; ++s) {
        const uint32_t last = (issued - 1 - s) / S;   // uses of stage s minus one
        if (!mbar_wait_bounded(&full_bar[s], last & 1, a.wait_limit)) set_status(a.ctl, ST_DRAIN_TIMEOUT);
      }
    }
  } else {
    // ------------------------------------------------------------ consumers
    int slot = 0;      // ring stage of the next unit and its earlier uses
    uint32_t use = 0;
    // flag protocol: tag of the launch's phase 0; tagged: tag of the program's phase 0
    const unsigned tag0 = (TAGGED || a.n_phases > 1) ? a.ctl->epoch * kPhasesPerEpoch + 1u : 0u;
    uint32_t lim = a.wait_limit;   // polls a tagged wait may take
    const uint32_t st0 = TAGGED ? ld_relaxed_b32(&a.ctl->status) : 0u;   // status bits at launch
    for (int p = 0; p < a.n_phases; ++p) {
      const Phase& ph = a.phases ? a.phases[p] : a.one;
      u64 xs2[kKT / 2];   // this phase's x slice (formed below when the CTA has units)
      unsigned tag = 0;
      float rscale = 1.f;   // tagged: RMSNorm scale of a staged fp32 input
      if (TAGGED) {
        // Tagged program: no barrier between phases.  A CTA with units here (or
        // CTA 0, which leaves the formed x) polls the tagged words of its input;
        // one flag exchange per layer keeps a fast CTA from overwriting words
        // that a slow one has yet to read (see SyncKind).
        // Once a wait of this launch has run out (a new status bit), the others
        // give up at once, so that a failed launch still ends promptly.
        tag = tag0 + static_cast<unsigned>(ph.gidx);
        lim = ld_relaxed_b32(&a.ctl->status) != st0 ? 0u : a.wait_limit;
        {
          const bool team0_cta0 = cta == 0 && (ph.x_dbg || ph.xr_out);
          if ((cta - ph.base % G + G) % G < ph.units || team0_cta0) {
            rscale = tagged_prologue(ph, tag, lim, a.ctl, a.flags, red, red_cta, tid, warp, lane);
          }
          if (ph.sync == SYNC_PUBLISH) {
            named_bar_sync(1, kConsumerThreads);   // every input read of this CTA is done
            if (tid == 0) st_release_u64(a.flags + cta, static_cast<unsigned long long>(tag) << 32);
          }
        }
        // nothing of the staging code stays in registers past this point
        asm volatile("" ::: "memory");
      }
      const Tile t = tile_of(ph, tid);
      const int units = ph.units, n_rows = ph.n_rows;
      const int u0 = (cta - ph.base % G + G) % G;
      if (TAGGED) {
        // the thread's 64 columns from the stage (for the attention gather, the
        // 64 values of v its query-head columns read).  Done by every CTA, also
        // one that staged nothing (its xs2 is then never used): xs2 is written
        // on every path, so no earlier phase's xs2 stays live across the
        // prologue.
        const int c0 = (t.active ? t.j : 0) * kKT;
        const int e0 =
            ph.x_kind == X_TAG16_ATTN ? ((c0 / ph.head_dim) / ph.group) * ph.head_dim + c0 % ph.head_dim : c0;
        const int sl = e0 >> 6;
        __half xv[kKT];
        if (ph.x_kind == X_NORM16 || ph.x_kind == X_TAG32_NORM) {
#pragma unroll
          for (int i = 0; i < kKT / 4; ++i) {
            const float4 f = *reinterpret_cast<const float4*>(red + (sl << 6) + ((i ^ (sl & 15)) << 2));
            const __half2 h0 = __floats2half2_rn(f.x * rscale, f.y * rscale);
            const __half2 h1 = __floats2half2_rn(f.z * rscale, f.w * rscale);
            xv[4 * i] = __low2half(h0);
            xv[4 * i + 1] = __high2half(h0);
            xv[4 * i + 2] = __low2half(h1);
            xv[4 * i + 3] = __high2half(h1);
          }
        } else {
#pragma unroll
          for (int i = 0; i < kKT / 8; ++i) {
            const uint4 u = *reinterpret_cast<const uint4*>(stage + (sl << 6) + ((i ^ (sl & 7)) << 3));
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              xv[8 * i + 2 * h] = __ushort_as_half(static_cast<unsigned short>(w[h] & 0xFFFFu));
              xv[8 * i + 2 * h + 1] = __ushort_as_half(static_cast<unsigned short>(w[h] >> 16));
            }
          }
        }
        if (cta == 0 && t.active && t.team == 0) store_formed_x(ph, c0, xv, tag & 0xFFFFu);
        xs2_from_halves(xv, xs2);
      }
      // the stage shares its memory with the row partials written from here on
      if (TAGGED) named_bar_sync(1, kConsumerThreads);
      // Every CTA waits for all CTAs' flags of the previous phase, even with no
      // units of its own here: a CTA may never publish phase p's flag while
      // another can still be reading phase p - 2's flags from the same slot
      // (the slots alternate), or that reader would take the wrong sum of squares.
      float sumsq = 0.f;
      if (!TAGGED && p > 0) {
        // one warp polls every CTA's flag, the CTA barrier releases the others
        if (warp == 0) {
          const float v = wait_phase_flags(a.flags + ((p - 1) & 1) * kMaxGrid, tag0 + (p - 1), lane,
                                           a.wait_limit, a.ctl);
          if (lane == 0) red_cta[0] = v;
        }
        named_bar_sync(1, kConsumerThreads);
        sumsq = red_cta[0];
      }
      if (!TAGGED && (u0 < units || (ph.x_dbg && cta == 0))) {
        if (p == 0 && ph.x_kind == X_NORM32) sumsq = sum_ss_array(ph.ss_in, lane);   // from an earlier launch
        form_x(ph, t.active ? t.j : 0, lane, xs2, ph.x_dbg != nullptr && cta == 0 && t.team == 0, sumsq, 0u);
      }
      // the unpack constants live in registers from here to the phase end only,
      // which leaves the prologue room for its loads
      const Unpack kk = make_unpack();
      const int cap = red_floats / (t.spu * t.tw);   // units buffered before a flush
      int n_buf = 0, u_first = u0;
      float ss = 0.f;
      for (int u = u0; u < units; u += G) {
        if (n_buf == cap) {
          if (TAGGED)
            flush_rows_tagged_mid(ph, t, red, n_buf, u_first, G, tid, tag, lim, a.ctl);
          else
            ss += flush_rows(ph, t, red, n_buf, u_first, G, tid, true);
          n_buf = 0;
          u_first = u;
        }
        // After a failed wait the CTA keeps walking its units without waiting
        // (reading whatever the stage holds) so that every barrier is still
        // reached; the launch then reports the failure in its status.
        if (!abort_flag && !mbar_wait_bounded(&full_bar[slot], use & 1, a.wait_limit)) {
          set_status(a.ctl, ST_FULL_TIMEOUT);
          abort_flag = 1;
        }
        const uint8_t* sb = g_ring + static_cast<size_t>(slot) * kStageBytes;
        const int row0 = u * t.rpu;
        float t0 = 0.f, t1 = 0.f;
        if (t.active) {
          const uint8_t *pa, *pb;
          int ra, rb;
          if (t.dual) {
            ra = rb = row0 + t.team;
            pa = sb + static_cast<size_t>(t.team) * t.row_bytes;
            pb = sb + static_cast<size_t>(t.rpu + t.team) * t.row_bytes;
          } else {
            ra = row0 + 2 * t.team;
            rb = ra + 1;
            pa = sb + static_cast<size_t>(2 * t.team) * t.row_bytes;
            pb = pa + t.row_bytes;
          }
          if (rb < n_rows) {
            pair_dot2(pa + static_cast<size_t>(t.j) * 36, pb + static_cast<size_t>(t.j) * 36, xs2, t0, t1, kk);
          } else if (ra < n_rows) {
            t0 = pair_dot(pa + static_cast<size_t>(t.j) * 36, xs2, 0.f, kk);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[slot]);
        if (++slot == S) {
          slot = 0;
          ++use;
        }
        if (t.active) {
          // both rows' sums over the width-lane group in one tree: the first
          // exchange leaves row 0 partials in the lower half-group and row 1
          // partials in the upper one, the remaining steps reduce each half
          const int width = t.team_threads < 32 ? t.team_threads : 32;
          const int half = width >> 1;
          const bool upper = (lane & half) != 0;
          float r = (upper ? t1 : t0) + __shfl_xor_sync(0xffffffffu, upper ? t0 : t1, half);
          if (width == 32) {   // the common case (teams of 32 or more threads), unrolled
            r += __shfl_xor_sync(0xffffffffu, r, 8);
            r += __shfl_xor_sync(0xffffffffu, r, 4);
            r += __shfl_xor_sync(0xffffffffu, r, 2);
            r += __shfl_xor_sync(0xffffffffu, r, 1);
          } else {
            for (int o = half >> 1; o > 0; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
          }
          if (((lane & (width - 1)) & ~half) == 0) {   // lane 0 (row 0) and lane `half` (row 1) of the group
            const int slot = n_buf * t.spu + 2 * t.team + (upper ? 1 : 0);
            red[slot * t.tw + t.w_in_team] = r;
          }
        }
        ++n_buf;
      }
      if (TAGGED) {
        flush_rows_tagged(ph, t, red, n_buf, u_first, G, tid, false, tag, lim, a.ctl);
        continue;
      }
      ss += flush_rows(ph, t, red, n_buf, u_first, G, tid, false);
      // phase end: publish this CTA's flag (its outputs are written; the sum of
      // squares of its residual sums rides along for the next RMSNorm)
      const bool resid = ph.epi_kind == EPI_RESID && ph.ss_out != nullptr;
      if (p + 1 < a.n_phases || resid) {
        ss = warp_sum(ss);
        if (lane == 0) red_cta[warp] = ss;
        named_bar_sync(1, kConsumerThreads);
        if (tid == 0) {
          float tot = 0.f;
          for (int w = 0; w < kConsumerWarps; ++w) tot += red_cta[w];
          if (resid) ph.ss_out[cta] = tot;
          if (p + 1 < a.n_phases) {
            const unsigned long long f =
                (static_cast<unsigned long long>(tag0 + p) << 32) | __float_as_uint(tot);
            st_release_u64(a.flags + (p & 1) * kMaxGrid + cta, f);
          }
        }
        named_bar_sync(1, kConsumerThreads);   // red_cta is read again at the next phase start
      }
    }
  }

  __syncthreads();
  if ((TAGGED || a.n_phases > 1) && tid == 0) {
    // The last CTA to leave advances the epoch (so the next launch's, or in a
    // tagged program the next program's, tags are new) and resets the
    // departure count.
    __threadfence();
    const unsigned long long left = atomicAdd(&a.ctl->depart, 1ull);
    if (left == static_cast<unsigned long long>(G) - 1) {
      a.ctl->depart = 0ull;
      if (!TAGGED || a.end_of_program) atomicAdd(&a.ctl->epoch, 1u);
    }
  }
}

cudaError_t engine_prepare() {
  cudaError_t e = cudaFuncSetAttribute(engine_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kStages * kStageBytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(engine_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kDynSmemMax);
}

cudaError_t engine_launch(const EngineArgs& a, int grid, bool cooperative, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = a.tagged ? static_cast<size_t>(a.stages) * kStageBytes + 4 * static_cast<size_t>(a.xbuf_floats)
                                  : static_cast<size_t>(kStages) * kStageBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = cooperative ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (a.tagged && (a.stages < 1 || a.stages > kStages || cfg.dynamicSmemBytes > static_cast<size_t>(kDynSmemMax)))
    return cudaErrorInvalidValue;
  return a.tagged ? cudaLaunchKernelEx(&cfg, engine_kernel<true>, a) : cudaLaunchKernelEx(&cfg, engine_kernel<false>, a);
}

cudaError_t engine_occupancy(int* blocks_per_sm) {
  int b0 = 0, b1 = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b0, engine_kernel<false>, kThreads,
                                                                kStages * kStageBytes);
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b1, engine_kernel<true>, kThreads, kDynSmemMax);
  *blocks_per_sm = b0 < b1 ? b0 : b1;
  return e;
}

cudaError_t engine_read_status(int* out) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_status, sizeof(int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_status, &zero, sizeof(int));
}

}  // namespace q4
