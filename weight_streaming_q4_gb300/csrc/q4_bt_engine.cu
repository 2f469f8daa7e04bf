// Persistent, warp-specialised Q4_0 engine on the tensor cores for batches of
// 2..8 rows (sm_103a): a whole decoder stack in one launch.
//
// The products are the batch-1 engine's (q4_tc_engine.cu): exact binary16
// values (q - 8) unpacked in registers, mma.sync m16n8k16 with fp32
// accumulation, each block's sum scaled by its d once in fp32.  Here the 8
// columns of the instruction are 8 batch rows instead of 8 copies of one x,
// so every lane keeps a different output and the input of a phase is 16 bytes
// per value of k: 64 KB for a 4096-wide row, 229 KB for a 14336-wide one,
// more than a CTA can hold beside its ring.  So the input travels with the
// weights: the producer copies each stage's 32 x 2048 weight tile with a 2-D
// tensor copy and the matching 32 KB chunk of input fragments with a 1-D bulk
// copy from global memory (an L2 hit: every CTA reads the same input).
//
// Warps 0-7 compute (four block pairs of every chunk, both 16-row halves of a
// 32-row unit), warp 8 is the epilogue (sums the 8 warps' partials in a fixed
// order, writes the outputs and the next phase's fragments), warp 9 the
// producer (weights run ahead across phase boundaries; a stage's input chunk
// is copied once every CTA has published the previous phase).
//
// Phases (per layer): q|k|v (v also gathered per head as the context-1
// attention output; value rows first, published once they are stored), o
// (+ residual), RMSNorm, gate|up (+ SiLU product), down (+ residual),
// RMSNorm; and one RMSNorm of the caller's binary16 state before the first
// layer.  Every phase ends with each CTA publishing a flag.  An RMSNorm after
// a residual phase (BT_FORM) is the epilogue warp's: once every CTA has
// published the residual phase it sums their sums of squares in CTA order and
// normalises the rows its own CTA produced; the first one is the consumers',
// each CTA normalising a slice of the rows.
//
// The method: PIPO's dequantisation-free 4-bit matrix-vector product for
// small batches ("PIPO: Pipelined Offloading for Efficient Inference on
// Consumer Devices", Method, "Computation optimization" and "Automatic
// configuration": the INT4 kernel serves batches below 16), layer by layer
// ("Offloading architecture").
#include <cuda.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "q4_device.cuh"
#include "q4_frag.cuh"
#include "q4_phase.cuh"

namespace q4 {

namespace {

constexpr int kBtWarps = 8;                        // consumer warps
constexpr int kBtConsumers = kBtWarps * 32;
constexpr int kBtEpiWarp = kBtWarps;               // warp 8
constexpr int kBtProdWarp = kBtWarps + 1;          // warp 9
constexpr int kBtThreads = (kBtWarps + 2) * 32;
constexpr int kBtMaxStages = 6;
constexpr int kBtRedSlots = 2;                     // unit partial slots between consumers and epilogue
constexpr int kBtRedFloats = kBtWarps * kTcUnitRows * kBtCols;   // one slot: 8 warps x 32 rows x 8 columns
constexpr int kBtRedBytes = kBtRedSlots * kBtRedFloats * 4;
constexpr int kBtDynSmemMax = 231424;
static_assert(kBtWarps == kBtCols, "an RMSNorm phase sums batch column b in consumer warp b");

extern __shared__ __align__(128) uint8_t g_bt_smem[];

}  // namespace

// Timeline build (-DQ4_TIMELINE, libq4_tl.so): the GPU's global timer at six
// points of every phase of every CTA, indexed by the phase's place in the
// program.  Product phases: 0 consumers reach the phase, 1 the producer issues
// its first weights, 2 the first stage has landed, 3 the consumers hand the
// last unit to the epilogue, 4 the epilogue publishes the phase, 5 the producer
// issues its first input chunk (every CTA has published the phase before).
// RMSNorm phases: 0 reached, 1 the previous phase seen from every CTA, 2 the
// rows formed, 4 published.  Other builds compile the stamps away.
#ifdef Q4_TIMELINE
constexpr int kBtTlCtas = 256, kBtTlPhases = 64, kBtTlEvents = 6;
__device__ unsigned long long g_bt_tl[kBtTlCtas * kBtTlPhases * kBtTlEvents];
__device__ __forceinline__ void bt_stamp(int phase, int event) {
  if (phase < kBtTlPhases && blockIdx.x < kBtTlCtas) {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    g_bt_tl[(blockIdx.x * kBtTlPhases + phase) * kBtTlEvents + event] = t;
  }
}
#else
__device__ __forceinline__ void bt_stamp(int, int) {}
#endif

namespace {

__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

__device__ __forceinline__ int bt_first_unit(const BtPhase& ph, int cta, int G) { return (cta - ph.base % G + G) % G; }
// First row of unit u of a 32-row phase, after the phase's row rotation.
__device__ __forceinline__ int bt_row0(const BtPhase& ph, int u) {
  const int r = u * kTcUnitRows + ph.row_rot;
  return r >= ph.n_rows ? r - ph.n_rows : r;
}

// Four consecutive values e..e+3 (e % 4 == 0) of batch row b as binary16
// pairs h01 = (x_e, x_e+1), h23 = (x_e+2, x_e+3): one 8-byte store.
__device__ __forceinline__ void bt_frag_store4(uint8_t* f, int b, int e, int cols, uint32_t h01, uint32_t h23) {
  *reinterpret_cast<uint2*>(f + bt_frag_off(b, e, cols)) =
      make_uint2(__byte_perm(h01, h23, 0x5410), __byte_perm(h01, h23, 0x7632));
}

// Whether every CTA's flag carries `tag` or a later one (the whole warp polls once).
__device__ __forceinline__ bool bt_flags_seen(const unsigned long long* flags, unsigned tag, int lane) {
  const int G = static_cast<int>(gridDim.x);
  bool mine = true;
  for (int i = lane; i < G; i += 32)
    mine &= static_cast<int>(static_cast<unsigned>(ld_relaxed_u64(flags + i) >> 32) - tag) >= 0;
  return __all_sync(0xffffffffu, mine);
}

// The whole warp waits (bounded) for every CTA's flag of `tag`; afterwards the
// CTA's later loads, and its later bulk copies, see what the CTAs wrote
// before their flags.
__device__ __forceinline__ void bt_wait_flags(const unsigned long long* flags, unsigned tag, int lane,
                                              uint32_t limit, Control* ctl) {
  bool ok = false;
  for (uint32_t it = 0; it < limit && !ok; ++it) {
    ok = bt_flags_seen(flags, tag, lane);
    if (!ok && it > 16) __nanosleep(64);
  }
  if (!ok && lane == 0) atomicOr(&ctl->status, ST_FLAG_TIMEOUT);
  fence_acq_rel_gpu();
  fence_proxy_async_global();
}

// Publish the CTA's flag of local phase p (tag), after the flags of the
// earlier phases of the launch (two warps publish: the epilogue after a unit
// phase or an RMSNorm of its rows, the consumers after the first RMSNorm;
// *pub is the last local phase published).  The writes of the phase by the
// other threads of the warp (or of the consumer warps) were ordered before
// the caller's by a warp or CTA barrier, and the release store is cumulative:
// a CTA that sees the flag with acquire semantics sees them all.
__device__ __forceinline__ void bt_publish(unsigned long long* flags, unsigned tag, volatile int* pub, int p,
                                           uint32_t limit, Control* ctl) {
  for (uint32_t it = 0; *pub != p - 1 && it < limit; ++it) __nanosleep(32);
  if (*pub != p - 1) atomicOr(&ctl->status, ST_FLAG_TIMEOUT);
  st_release_u64(flags + blockIdx.x, static_cast<unsigned long long>(tag) << 32);
  *pub = p;
}

// Wait for a stage: as the batch-1 engine, one non-blocking test in the
// common case; after a failed wait the CTA walks on without waiting.
__device__ __forceinline__ void bt_stage_wait(uint64_t* bar, uint32_t parity, uint32_t limit, volatile int* abort_flag,
                                              Control* ctl) {
  if (mbar_test_wait(bar, parity)) return;
  if (!*abort_flag && !mbar_wait_bounded(bar, parity, limit)) {
    atomicOr(&ctl->status, ST_FULL_TIMEOUT);
    *abort_flag = 1;
  }
}

// One block pair (even block, odd block after it) of tile rows g and g + 8
// against the 8 batch columns: rg, rh point at the pair's 36 bytes in the two
// staged rows; xe, xo are the lane's fragments of the two blocks.  acc: rows
// g, g (columns 2t, 2t + 1), g + 8, g + 8.
__device__ __forceinline__ void bt_pair(const uint8_t* rg, const uint8_t* rh, int t, const uint4& xe, const uint4& xo,
                                        uint32_t magic, float (&acc)[4]) {
  const uint32_t* pg = reinterpret_cast<const uint32_t*>(rg);
  const uint32_t* ph = reinterpret_cast<const uint32_t*>(rh);
  const uint32_t g0 = pg[t], g1 = pg[t + 1], go = pg[5 + t];
  const uint32_t h0 = ph[t], h1 = ph[t + 1], ho = ph[5 + t];
  // the blocks' scales: the even block's d opens word 0, the odd block's closes word 4
  const float dge = lo_half_f(pg[0]), dhe = lo_half_f(ph[0]);
  const float dgo = hi_half_f(pg[4]), dho = hi_half_f(ph[4]);
  uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
  unpack_word(__funnelshift_r(g0, g1, 16), magic, a0, a1, a2, a3);
  unpack_word(__funnelshift_r(h0, h1, 16), magic, b0, b1, b2, b3);
  float c[4] = {0.f, 0.f, 0.f, 0.f};
  mma16816(c, a0, b0, a1, b1, xe.x, xe.y);
  mma16816(c, a2, b2, a3, b3, xe.z, xe.w);
  acc[0] = fmaf(dge, c[0], acc[0]);
  acc[1] = fmaf(dge, c[1], acc[1]);
  acc[2] = fmaf(dhe, c[2], acc[2]);
  acc[3] = fmaf(dhe, c[3], acc[3]);
  unpack_word(go, magic, a0, a1, a2, a3);
  unpack_word(ho, magic, b0, b1, b2, b3);
  float e[4] = {0.f, 0.f, 0.f, 0.f};
  mma16816(e, a0, b0, a1, b1, xo.x, xo.y);
  mma16816(e, a2, b2, a3, b3, xo.z, xo.w);
  acc[0] = fmaf(dgo, e[0], acc[0]);
  acc[1] = fmaf(dgo, e[1], acc[1]);
  acc[2] = fmaf(dho, e[2], acc[2]);
  acc[3] = fmaf(dho, e[3], acc[3]);
}

// One unit's products for one consumer warp, chunk by chunk as the stages
// land (WIDE: 64-block chunks, 1168-byte staged rows, as constants).
template <bool WIDE>
__device__ __forceinline__ void bt_unit(const uint8_t* ring, uint32_t SB, uint32_t x_off, int S, int& slot,
                                        uint32_t& use, uint64_t* full_bar, uint64_t* empty_bar,
                                        volatile int* abort_flag, int chunks, int cb_rt, int pitch_rt, int warp,
                                        int lane, uint32_t magic, uint32_t limit, Control* ctl, float (&acc)[2][4],
                                        int stamp_gidx, int cols) {
  const int cb = WIDE ? 64 : cb_rt;
  const int pitch = WIDE ? 64 * kBlockBytes + 16 : pitch_rt;
  const int g = lane >> 2, t = lane & 3;
  for (int c = 0; c < chunks; ++c) {
    bt_stage_wait(&full_bar[slot], use & 1, limit, abort_flag, ctl);
    if (stamp_gidx >= 0 && c == 0 && warp == 0 && lane == 0) bt_stamp(stamp_gidx, 2);
    const uint8_t* sb = ring + static_cast<size_t>(slot) * SB;
    const uint4* xs = reinterpret_cast<const uint4*>(sb + x_off);
#pragma unroll(WIDE ? 4 : 1)
    for (int q = 0; q < 4; ++q) {
      const int pp = warp + kBtWarps * q;   // block pair of the chunk
      if (WIDE || 2 * pp < cb) {
        const uint4 z4 = make_uint4(0u, 0u, 0u, 0u);
        const uint4 xe = lane < 4 * cols ? xs[(2 * pp) * 4 * cols + lane] : z4;
        const uint4 xo = lane < 4 * cols ? xs[(2 * pp + 1) * 4 * cols + lane] : z4;
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          const uint8_t* rg = sb + (m * 16 + g) * pitch + 36 * pp;
          bt_pair(rg, rg + 8 * pitch, t, xe, xo, magic, acc[m]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_bar[slot]);
    if (++slot == S) {
      slot = 0;
      ++use;
    }
  }
}

}  // namespace

namespace {

// The first RMSNorm of a program (the caller's binary16 state), by the
// consumer warps: this CTA's slice of the batch rows' 4-value groups,
// z = f16(t * r_b), to out16 (natural order) and out_frag; r_b =
// 1 / sqrt(mean(t_b^2) + eps) summed here over the whole row in an order
// fixed by k (every CTA the same): each thread's chunks, the warp tree, the 8
// warps in order.
__device__ void bt_form16(const BtPhase& ph, int batch, int cols, float* rsm, float* red_cta, int tid) {
  const int G = static_cast<int>(gridDim.x), cta = static_cast<int>(blockIdx.x);
  const int k4 = ph.k >> 2;
  float s[kBtCols];
#pragma unroll
  for (int b = 0; b < kBtCols; ++b) s[b] = 0.f;
  for (int i = tid; i < k4; i += kBtConsumers) {
    uint2 u[kBtCols];   // the rows' loads in flight together
#pragma unroll
    for (int b = 0; b < kBtCols; ++b)
      u[b] = b < batch ? __ldcg(reinterpret_cast<const uint2*>(ph.src16 + static_cast<size_t>(b) * ph.k) + i)
                       : make_uint2(0u, 0u);
#pragma unroll
    for (int b = 0; b < kBtCols; ++b) {
      const float2 x0 = __half22float2(*reinterpret_cast<const __half2*>(&u[b].x));
      const float2 x1 = __half22float2(*reinterpret_cast<const __half2*>(&u[b].y));
      s[b] = fmaf(x0.x, x0.x, s[b]);
      s[b] = fmaf(x0.y, x0.y, s[b]);
      s[b] = fmaf(x1.x, x1.x, s[b]);
      s[b] = fmaf(x1.y, x1.y, s[b]);
    }
  }
#pragma unroll
  for (int b = 0; b < kBtCols; ++b) {
    const float v = warp_sum(s[b]);
    if ((tid & 31) == 0) red_cta[(tid >> 5) * kBtCols + b] = v;
  }
  named_bar_sync(1, kBtConsumers);
  if (tid < batch) {
    float t = 0.f;
    for (int w = 0; w < kBtWarps; ++w) t += red_cta[w * kBtCols + tid];
    rsm[tid] = rsqrtf(t / static_cast<float>(ph.k) + ph.eps);
  }
  named_bar_sync(1, kBtConsumers);
  const int total = batch * k4, per = (total + G - 1) / G;
  const int lo = cta * per, hi = lo + per < total ? lo + per : total;
  for (int i = lo + tid; i < hi; i += kBtConsumers) {
    const int b = i / k4, e = (i - b * k4) * 4;
    const uint2 u = __ldcg(reinterpret_cast<const uint2*>(ph.src16 + static_cast<size_t>(b) * ph.k + e));
    const float2 x0 = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
    const float2 x1 = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
    const float r = rsm[b];
    const __half2 h01 = __floats2half2_rn(x0.x * r, x0.y * r), h23 = __floats2half2_rn(x1.x * r, x1.y * r);
    const uint32_t w01 = *reinterpret_cast<const uint32_t*>(&h01), w23 = *reinterpret_cast<const uint32_t*>(&h23);
    *reinterpret_cast<uint2*>(ph.out16 + static_cast<size_t>(b) * ph.k + e) = make_uint2(w01, w23);
    bt_frag_store4(ph.out_frag, b, e, cols, w01, w23);
  }
}

// Item cursor of the producer: (phase p, unit u, chunk c) over this CTA's
// units of the unit phases, in the order the consumers take them.
__device__ __forceinline__ void bt_settle(const BtArgs& a, int cta, int G, int& p, int& u, int& c) {
  while (p < a.n_phases && u >= a.phases[p].units) {   // BT_FORM phases have no units
    if (++p < a.n_phases) {
      u = bt_first_unit(a.phases[p], cta, G);
      c = 0;
    }
  }
}
__device__ __forceinline__ void bt_next(const BtArgs& a, int cta, int G, int& p, int& u, int& c) {
  if (++c == tc_chunks(a.phases[p].k)) {
    c = 0;
    u += G;
  }
  bt_settle(a, cta, G, p, u, c);
}

// The warp's 32 rows of binary16 values for the 8 batch columns (h[b] of
// the lane's row, value e of the next phase's input) into the fragment
// buffer: lane L takes the four rows of its group (lanes 4(L/4) .. +3, values
// e_grp .. e_grp + 3, 4-aligned) for batch columns 2(L%4) and 2(L%4) + 1,
// gathers them with four shuffles and stores two 8-byte pieces.  A group
// stores when its rows are valid (ok, the same for the four lanes).
__device__ __forceinline__ void bt_frag_rows(uint8_t* frag, int e_grp, bool ok, int batch, int cols,
                                             const __half (&h)[kBtCols], int lane) {
  uint32_t packed[4];
#pragma unroll
  for (int q = 0; q < 4; ++q)
    packed[q] = static_cast<uint32_t>(__half_as_ushort(h[2 * q])) |
                (static_cast<uint32_t>(__half_as_ushort(h[2 * q + 1])) << 16);
  const int q = lane & 3;
  uint32_t row[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    // round r: lane j of a group offers its pair (j + r) % 4; lane q reads lane (q - r) % 4
    const int give = (q + r) & 3;
    const uint32_t mine = give == 0 ? packed[0] : give == 1 ? packed[1] : give == 2 ? packed[2] : packed[3];
    const uint32_t got = __shfl_sync(0xffffffffu, mine, (lane & ~3) | ((q - r) & 3));
    const int j = (q - r) & 3;
    row[0] = j == 0 ? got : row[0];
    row[1] = j == 1 ? got : row[1];
    row[2] = j == 2 ? got : row[2];
    row[3] = j == 3 ? got : row[3];
  }
  if (!ok) return;
  // batch column 2q: the low halves of the four rows; 2q + 1: the high halves
  if (2 * q < batch)
    bt_frag_store4(frag, 2 * q, e_grp, cols, __byte_perm(row[0], row[1], 0x5410), __byte_perm(row[2], row[3], 0x5410));
  if (2 * q + 1 < batch)
    bt_frag_store4(frag, 2 * q + 1, e_grp, cols, __byte_perm(row[0], row[1], 0x7632), __byte_perm(row[2], row[3], 0x7632));
}

// The epilogue of unit u for the warp (lane = row of the unit; v: its 8 batch
// columns; u2: the up row of a gate|up pair; rv: the residual base of a
// residual phase, whose sums go to t_out and their squares into ss).
// Natural-order outputs per lane, the next phase's fragments per group of
// four rows.
__device__ __forceinline__ void bt_epilogue_unit(const BtPhase& ph, int u, int lane, int batch, int cols,
                                                 const float (&v)[kBtCols], const float (&u2)[kBtCols],
                                                 const unsigned short (&rv)[kBtCols], float (&ss)[kBtCols],
                                                 float (&t_out)[kBtCols]) {
  const size_t N = static_cast<size_t>(ph.n_rows);
  if (ph.kind == BT_SILU) {
    const int n = u * (kTcUnitRows / 2) + lane;
    const bool ok = lane < kTcUnitRows / 2 && n < ph.n_rows;
    __half a16[kBtCols];
#pragma unroll
    for (int b = 0; b < kBtCols; ++b) {
      a16[b] = __float2half_rn(silu_mul(v[b], u2[b]));
      if (ok && b < batch) {
        ph.y[b * N + n] = v[b];
        ph.y2[b * N + n] = u2[b];
        ph.out16[b * N + n] = __half_as_ushort(a16[b]);
      }
    }
    bt_frag_rows(ph.out_frag, n & ~3, ok, batch, cols, a16, lane);
  } else if (ph.kind == BT_RESID) {
    const int n = u * kTcUnitRows + lane;
    if (n < ph.n_rows) {
#pragma unroll
      for (int b = 0; b < kBtCols; ++b) {
        if (b < batch) {
          ph.y[b * N + n] = v[b];
          const float tv = __half2float(__ushort_as_half(rv[b])) + v[b];
          ph.y2[b * N + n] = tv;
          ss[b] = fmaf(tv, tv, ss[b]);
          t_out[b] = tv;
        }
      }
    }
  } else {
    const int r0 = bt_row0(ph, u), n = r0 + lane;
#pragma unroll
    for (int b = 0; b < kBtCols; ++b)
      if (n < ph.n_rows && b < batch) ph.y[b * N + n] = v[b];
    // a unit with value rows (the range is 4-aligned, and so is head_dim):
    // value row i of value head vh is element i of query heads vh * group ..
    if (ph.out16 && r0 < ph.g_lo + ph.g_n && r0 + kTcUnitRows > ph.g_lo) {
      const bool ok = n >= ph.g_lo && n < ph.g_lo + ph.g_n;
      const int r = ok ? n - ph.g_lo : 0;
      const int vh = r / ph.head_dim, i = r % ph.head_dim;
      __half h16[kBtCols];
#pragma unroll
      for (int b = 0; b < kBtCols; ++b) h16[b] = __float2half_rn(v[b]);
      for (int h = 0; h < ph.group; ++h) {
        const int e = (vh * ph.group + h) * ph.head_dim + i;
#pragma unroll
        for (int b = 0; b < kBtCols; ++b)
          if (ok && b < batch) ph.out16[static_cast<size_t>(b) * ph.out_ld + e] = __half_as_ushort(h16[b]);
        bt_frag_rows(ph.out_frag, e & ~3, ok, batch, cols, h16, lane);
      }
    }
  }
}

}  // namespace

namespace {

// An RMSNorm phase after a residual phase, by the epilogue warp: the rows
// this CTA produced in that phase (its units), z = f16(t * r_b) into out16
// and the fragments.  r_b from every CTA's sums of squares (summed in CTA
// order: lane l the partials l, l + 32, ..., then the warp tree), once every
// CTA has published the residual phase.  A CTA without rows has nothing to
// wait for.  t0, t1: the values of the CTA's first two units of that phase.
__device__ void bt_form_rows(const BtArgs& a, int p, unsigned tag0, int lane, const float (&t0)[kBtCols],
                             const float (&t1)[kBtCols]) {
  const BtPhase& ph = a.phases[p];
  const BtPhase& rp = a.phases[p - 1];
  const int G = static_cast<int>(gridDim.x), cta = static_cast<int>(blockIdx.x);
  const int u0 = bt_first_unit(rp, cta, G);
  if (u0 >= rp.units) return;
  bt_wait_flags(a.flags, tag0 + a.stall + static_cast<unsigned>(rp.gidx), lane, a.wait_limit, a.ctl);
  if (lane == 0) bt_stamp(ph.gidx, 1);
  // the 8 partials of CTA c are contiguous: two 16-byte loads, all of the
  // lane's CTAs in flight together
  float4 lo[kMaxGrid / 32], hi[kMaxGrid / 32];
#pragma unroll
  for (int j = 0; j < kMaxGrid / 32; ++j) {
    const int c = lane + 32 * j;
    lo[j] = c < G ? __ldcg(reinterpret_cast<const float4*>(ph.ss + c * kBtCols)) : make_float4(0.f, 0.f, 0.f, 0.f);
    hi[j] = c < G ? __ldcg(reinterpret_cast<const float4*>(ph.ss + c * kBtCols + 4)) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float s[kBtCols];
#pragma unroll
  for (int b = 0; b < kBtCols; ++b) s[b] = 0.f;
#pragma unroll
  for (int j = 0; j < kMaxGrid / 32; ++j) {
    s[0] += lo[j].x;
    s[1] += lo[j].y;
    s[2] += lo[j].z;
    s[3] += lo[j].w;
    s[4] += hi[j].x;
    s[5] += hi[j].y;
    s[6] += hi[j].z;
    s[7] += hi[j].w;
  }
  float r[kBtCols];
#pragma unroll
  for (int b = 0; b < kBtCols; ++b) r[b] = rsqrtf(warp_sum(s[b]) / static_cast<float>(ph.k) + ph.eps);
  const size_t N = static_cast<size_t>(ph.k);
  int kept = 0;
  for (int u = u0; u < rp.units; u += G, ++kept) {
    const int n = u * kTcUnitRows + lane;
    const bool ok = n < rp.n_rows;
    __half z[kBtCols];
#pragma unroll
    for (int b = 0; b < kBtCols; ++b) {
      // t of this row: kept in registers for the first two units, else
      // reloaded (this lane stored it in the residual phase)
      const float t = !(ok && b < a.batch) ? 0.f
                      : kept == 0         ? t0[b]
                      : kept == 1         ? t1[b]
                                          : __ldcg(ph.src32 + b * N + n);
      z[b] = __float2half_rn(t * r[b]);
      if (ok && b < a.batch) ph.out16[b * N + n] = __half_as_ushort(z[b]);
    }
    bt_frag_rows(ph.out_frag, n & ~3, ok, a.batch, a.cols, z, lane);
  }
  if (lane == 0) bt_stamp(ph.gidx, 2);
}

}  // namespace

__global__ void __launch_bounds__(kBtThreads, 1) bt_engine_kernel(const __grid_constant__ BtArgs a) {
  __shared__ __align__(8) uint64_t full_bar[kBtMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kBtMaxStages];
  __shared__ __align__(8) uint64_t rfull_bar[kBtRedSlots];
  __shared__ __align__(8) uint64_t rempty_bar[kBtRedSlots];
  __shared__ float red_cta[kBtWarps * kBtCols];
  __shared__ float rsm[kBtCols];
  __shared__ volatile int abort_flag;
  __shared__ volatile int pub;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = static_cast<int>(gridDim.x), cta = static_cast<int>(blockIdx.x);
  const int S = a.stages;
  const uint32_t SB = a.stage_bytes;
  uint8_t* const ring = g_bt_smem;
  float* const red = reinterpret_cast<float*>(g_bt_smem + static_cast<size_t>(S) * SB);

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kBtWarps);
    }
    for (int s = 0; s < kBtRedSlots; ++s) {
      mbar_init(&rfull_bar[s], kBtWarps);
      mbar_init(&rempty_bar[s], 1);
    }
    fence_mbar_init();
    abort_flag = 0;
    pub = -1;
  }
  __syncthreads();
  const unsigned tag0 = a.ctl->epoch * kPhasesPerEpoch + 1u;

  if (warp == kBtProdWarp) {
    // ------------------------------------------------------------ producer
    // The whole warp walks two cursors over the CTA's items: the weights of
    // item nw go out as soon as its stage is free; its input chunk (item nx)
    // once every CTA has published the phase before the item's phase.
    int wp = 0, wu = bt_first_unit(a.phases[0], cta, G), wc = 0;
    bt_settle(a, cta, G, wp, wu, wc);
    int xp = wp, xu = wu, xc = wc;
    uint32_t nw = 0, nx = 0, idle = 0;
    int ready = 0, acquired = -1, x_stamped = -1;
    while (xp < a.n_phases) {
      if (__shfl_sync(0xffffffffu, static_cast<int>(abort_flag), 0)) break;
      bool moved = false;
      if (wp < a.n_phases) {
        const int slot = static_cast<int>(nw % S);
        const uint32_t use = nw / S;
        int free = 1;
        if (use > 0) {
          free = lane == 0 ? static_cast<int>(mbar_test_wait(&empty_bar[slot], (use - 1) & 1)) : 0;
          free = __shfl_sync(0xffffffffu, free, 0);
        }
        if (free) {
          if (lane == 0) {
            const BtPhase& ph = a.phases[wp];
            const bool dual = ph.kind == BT_SILU;
            if (wp != acquired) {
              // descriptors written by the host into global memory: order their use
              // through the tensor-map proxy after the generic-proxy writes
              tensormap_acquire(&ph.tm0);
              if (dual) tensormap_acquire(&ph.tm1);
              acquired = wp;
              bt_stamp(ph.gidx, 1);
            }
            const int pitch = tc_pitch(ph.k), cb = tc_chunk_blocks(ph.k), cx = cb * kBlockBytes / 8;
            uint8_t* dst = ring + static_cast<size_t>(slot) * SB;
            mbar_arrive_expect_tx(&full_bar[slot],
                                  static_cast<uint32_t>(pitch * kTcUnitRows + cb * 64 * a.cols));
            if (dual) {
              const int r0 = wu * (kTcUnitRows / 2);
              tma_load_2d(dst, &ph.tm0, wc * cx, r0, &full_bar[slot]);
              tma_load_2d(dst + (kTcUnitRows / 2) * pitch, &ph.tm1, wc * cx, r0, &full_bar[slot]);
            } else {
              tma_load_2d(dst, &ph.tm0, wc * cx, bt_row0(ph, wu), &full_bar[slot]);
            }
          }
          ++nw;
          bt_next(a, cta, G, wp, wu, wc);
          moved = true;
        }
      }
      if (nx < nw) {
        if (xp > ready &&
            bt_flags_seen(a.flags, tag0 + a.stall + static_cast<unsigned>(a.phases[xp - 1].gidx), lane)) {
          ready = xp;
          fence_acq_rel_gpu();
          fence_proxy_async_global();
        }
        if (xp <= ready) {
          if (lane == 0) {
            const BtPhase& ph = a.phases[xp];
            if (xp != x_stamped) {
              bt_stamp(ph.gidx, 5);
              x_stamped = xp;
            }
            const int slot = static_cast<int>(nx % S);
            const uint32_t cbytes = static_cast<uint32_t>(tc_chunk_blocks(ph.k) * 64 * a.cols);
            bulk_g2s(ring + static_cast<size_t>(slot) * SB + a.x_off, ph.x_frag + static_cast<size_t>(xc) * cbytes,
                     cbytes, &full_bar[slot]);
          }
          ++nx;
          bt_next(a, cta, G, xp, xu, xc);
          moved = true;
        }
      }
      if (moved) {
        idle = 0;
      } else if (++idle > a.wait_limit) {
        if (lane == 0) {
          atomicOr(&a.ctl->status, nx < nw ? ST_FLAG_TIMEOUT : ST_EMPTY_TIMEOUT);
          abort_flag = 1;
        }
        break;
      } else if (idle > 16) {
        __nanosleep(64);
      }
    }
    // Drain: no copy may still be in flight when the CTA exits.
    if (lane == 0) {
      for (int s = 0; s < S && static_cast<uint32_t>(s) < nw; ++s) {
        const uint32_t last = (nw - 1 - s) / S;
        if (!mbar_wait_bounded(&full_bar[s], last & 1, a.wait_limit)) atomicOr(&a.ctl->status, ST_DRAIN_TIMEOUT);
      }
    }
  } else if (warp == kBtEpiWarp) {
    // ------------------------------------------------------------ epilogue
    int rs = 0;
    uint32_t ruse = 0;
    // publish phase p: the warp's writes are ordered before lane 0's fence and flag
    auto publish = [&](const BtPhase& ph, int p) {
      __syncwarp();
      if (lane == 0) {
        bt_publish(a.flags, tag0 + static_cast<unsigned>(ph.gidx), &pub, p, a.wait_limit, a.ctl);
        bt_stamp(ph.gidx, 4);
      }
      __syncwarp();
    };
    float keep0[kBtCols], keep1[kBtCols];   // t of the last residual phase's first two units
#pragma unroll
    for (int b = 0; b < kBtCols; ++b) keep0[b] = keep1[b] = 0.f;
    for (int p = 0; p < a.n_phases; ++p) {
      const BtPhase& ph = a.phases[p];
      if (ph.kind == BT_FORM) {
        if (ph.src32) {
          bt_form_rows(a, p, tag0, lane, keep0, keep1);
          publish(ph, p);
        }
        continue;   // the first RMSNorm (binary16 source) is the consumers'
      }
      const bool dual = ph.kind == BT_SILU;
      float ss[kBtCols];
#pragma unroll
      for (int b = 0; b < kBtCols; ++b) ss[b] = 0.f;
      const int u0 = bt_first_unit(ph, cta, G);
      // q|k|v: once the CTA's units with value rows are stored (or at once when
      // it has none), the o phase may start; the q and k rows follow
      bool published = false;
      if (ph.early_units > 0 && u0 >= ph.early_units) {
        publish(ph, p);
        published = true;
      }
      // the residual base was written by other CTAs before they published the
      // phases up to the previous one: seen here, before its loads are issued
      if (ph.kind == BT_RESID && p > 0 && u0 < ph.units)
        bt_wait_flags(a.flags, tag0 + a.stall + static_cast<unsigned>(a.phases[p - 1].gidx), lane, a.wait_limit,
                      a.ctl);
      for (int u = u0, ord = 0; u < ph.units; u += G, ++ord) {
        const int n = dual ? u * (kTcUnitRows / 2) + lane : u * kTcUnitRows + lane;
        const bool row_ok = (!dual || lane < kTcUnitRows / 2) && n < ph.n_rows;
        // the residual base of this row: its loads overlap the wait for the
        // unit's partials
        unsigned short rv[kBtCols];
#pragma unroll
        for (int b = 0; b < kBtCols; ++b)
          rv[b] = ph.kind == BT_RESID && row_ok && b < a.batch ? __ldcg(ph.res + static_cast<size_t>(b) * ph.n_rows + n)
                                                               : static_cast<unsigned short>(0);
        if (!mbar_wait_bounded(&rfull_bar[rs], ruse & 1, a.wait_limit)) atomicOr(&a.ctl->status, ST_FULL_TIMEOUT);
        // row `lane` of the unit: the 8 warps' partials in warp order
        const float* pr = red + rs * kBtRedFloats + lane * kBtCols;
        float v[kBtCols], u2[kBtCols];
#pragma unroll
        for (int b = 0; b < kBtCols; ++b) v[b] = 0.f;
#pragma unroll
        for (int w = 0; w < kBtWarps; ++w) {
          const float4 x0 = *reinterpret_cast<const float4*>(pr + w * kTcUnitRows * kBtCols);
          const float4 x1 = *reinterpret_cast<const float4*>(pr + w * kTcUnitRows * kBtCols + 4);
          v[0] += x0.x;
          v[1] += x0.y;
          v[2] += x0.z;
          v[3] += x0.w;
          v[4] += x1.x;
          v[5] += x1.y;
          v[6] += x1.z;
          v[7] += x1.w;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&rempty_bar[rs]);
        if (++rs == kBtRedSlots) {
          rs = 0;
          ++ruse;
        }
        // a gate|up unit: rows 0-15 gate, rows 16-31 the same rows of up
#pragma unroll
        for (int b = 0; b < kBtCols; ++b) u2[b] = __shfl_down_sync(0xffffffffu, v[b], 16);
        float tv[kBtCols];
#pragma unroll
        for (int b = 0; b < kBtCols; ++b) tv[b] = 0.f;
        bt_epilogue_unit(ph, u, lane, a.batch, a.cols, v, u2, rv, ss, tv);
        if (ph.kind == BT_RESID) {
#pragma unroll
          for (int b = 0; b < kBtCols; ++b) {
            keep0[b] = ord == 0 ? tv[b] : keep0[b];
            keep1[b] = ord == 1 ? tv[b] : keep1[b];
          }
        }
        if (!published && ph.early_units > 0 && u + G >= ph.early_units) {
          publish(ph, p);
          published = true;
        }
      }
      if (ph.kind == BT_RESID) {
#pragma unroll
        for (int b = 0; b < kBtCols; ++b) {
          const float s = warp_sum(ss[b]);
          if (lane == 0) ph.ss[cta * kBtCols + b] = s;
        }
      }
      if (!published) publish(ph, p);
    }
  } else {
    // ------------------------------------------------------------ consumers
    uint32_t magic;
    asm volatile("mov.b32 %0, 0x64006400;" : "=r"(magic));
    const int g = lane >> 2, t = lane & 3;
    int slot = 0;
    uint32_t use = 0;
    int rs = 0;
    uint32_t ruse = 0;
    for (int p = 0; p < a.n_phases; ++p) {
      const BtPhase& ph = a.phases[p];
      if (tid == 0) bt_stamp(ph.gidx, 0);
      if (ph.kind == BT_FORM && ph.src32) continue;   // the epilogue warp's
      if (ph.kind == BT_FORM) {
        if (p > 0 && warp == 0)
          bt_wait_flags(a.flags, tag0 + a.stall + static_cast<unsigned>(a.phases[p - 1].gidx), lane, a.wait_limit,
                      a.ctl);
        named_bar_sync(1, kBtConsumers);
        if (tid == 0) bt_stamp(ph.gidx, 1);
        bt_form16(ph, a.batch, a.cols, rsm, red_cta, tid);
        named_bar_sync(1, kBtConsumers);
        if (tid == 0) {   // the consumers' writes are ordered before thread 0's fence and flag
          bt_stamp(ph.gidx, 2);
          bt_publish(a.flags, tag0 + static_cast<unsigned>(ph.gidx), &pub, p, a.wait_limit, a.ctl);
          bt_stamp(ph.gidx, 4);
        }
        continue;
      }
      const int chunks = tc_chunks(ph.k), cb = tc_chunk_blocks(ph.k), pitch = tc_pitch(ph.k);
      const bool wide = ph.k > 2048;
      const int u0 = bt_first_unit(ph, cta, G);
      for (int u = u0; u < ph.units; u += G) {
        float acc[2][4] = {};
        const int sg = u == u0 ? ph.gidx : -1;
        if (wide)
          bt_unit<true>(ring, SB, a.x_off, S, slot, use, full_bar, empty_bar, &abort_flag, chunks, cb, pitch, warp,
                        lane, magic, a.wait_limit, a.ctl, acc, sg, a.cols);
        else
          bt_unit<false>(ring, SB, a.x_off, S, slot, use, full_bar, empty_bar, &abort_flag, chunks, cb, pitch, warp,
                         lane, magic, a.wait_limit, a.ctl, acc, sg, a.cols);
        if (ruse > 0) {
          // slot rs's previous unit has been read by the epilogue
          if (lane == 0 && !mbar_wait_bounded(&rempty_bar[rs], (ruse - 1) & 1, a.wait_limit))
            atomicOr(&a.ctl->status, ST_EMPTY_TIMEOUT);
          __syncwarp();
        }
        float* pr = red + rs * kBtRedFloats + warp * (kTcUnitRows * kBtCols);
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          *reinterpret_cast<float2*>(pr + (m * 16 + g) * kBtCols + 2 * t) = make_float2(acc[m][0], acc[m][1]);
          *reinterpret_cast<float2*>(pr + (m * 16 + g + 8) * kBtCols + 2 * t) = make_float2(acc[m][2], acc[m][3]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&rfull_bar[rs]);
        if (tid == 0) bt_stamp(ph.gidx, 3);
        if (++rs == kBtRedSlots) {
          rs = 0;
          ++ruse;
        }
      }
    }
  }

  __syncthreads();
  if (tid == 0) {
    // The last CTA to leave advances the epoch when the launch ends the
    // program (so the next program's tags are new) and resets the count.
    __threadfence();
    const unsigned long long left = atomicAdd(&a.ctl->depart, 1ull);
    if (left == static_cast<unsigned long long>(G) - 1) {
      a.ctl->depart = 0ull;
      if (a.end_of_program) atomicAdd(&a.ctl->epoch, 1u);
    }
  }
}

cudaError_t bt_timeline_read(unsigned long long* out, size_t n, bool clear) {
#ifdef Q4_TIMELINE
  const size_t total = static_cast<size_t>(kBtTlCtas) * kBtTlPhases * kBtTlEvents;
  if (n < total) return cudaErrorInvalidValue;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_bt_tl, total * sizeof(unsigned long long));
  if (e == cudaSuccess && clear) {
    static unsigned long long zero[kBtTlCtas * kBtTlPhases * kBtTlEvents];
    e = cudaMemcpyToSymbol(g_bt_tl, zero, sizeof(zero));
  }
  return e;
#else
  (void)out;
  (void)n;
  (void)clear;
  return cudaErrorNotSupported;
#endif
}

cudaError_t bt_engine_prepare() {
  return cudaFuncSetAttribute(bt_engine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kBtDynSmemMax);
}

bool bt_geom(const int* ks, int n, int cols, int* stages, uint32_t* stage_bytes, uint32_t* x_off) {
  int pmax = 0, cbmax = 0;
  for (int i = 0; i < n; ++i) {
    const int k = ks[i];
    if (k < 256 || k % 256 || (k > 2048 && k % 2048)) return false;
    pmax = tc_pitch(k) > pmax ? tc_pitch(k) : pmax;
    cbmax = tc_chunk_blocks(k) > cbmax ? tc_chunk_blocks(k) : cbmax;
  }
  const uint32_t xo = (static_cast<uint32_t>(pmax) * kTcUnitRows + 127u) / 128u * 128u;
  const uint32_t sb = (xo + static_cast<uint32_t>(cbmax * 64 * cols) + 127u) / 128u * 128u;
  int s = kBtMaxStages;
  while (s > 0 && static_cast<size_t>(s) * sb + kBtRedBytes > static_cast<size_t>(kBtDynSmemMax)) --s;
  *stages = s;
  *stage_bytes = sb;
  *x_off = xo;
  return s >= 2;
}

cudaError_t bt_engine_launch(const BtArgs& a, int grid, cudaStream_t stream) {
  const size_t smem = static_cast<size_t>(a.stages) * a.stage_bytes + kBtRedBytes;
  if (a.stages < 2 || a.stages > kBtMaxStages || a.batch < 1 || a.batch > kBtCols || a.cols != bt_cols(a.batch) ||
      a.stage_bytes % 128 ||
      a.x_off % 16 || smem > static_cast<size_t>(kBtDynSmemMax) || grid < 1 || grid > kMaxGrid || !a.phases ||
      !a.ctl || !a.flags || a.n_phases < 1)
    return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kBtThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, bt_engine_kernel, a);
}

}  // namespace q4
