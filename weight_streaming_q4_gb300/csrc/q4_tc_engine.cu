// Persistent, warp-specialised Q4_0 matrix-vector engine on the tensor cores
// (batch 1, sm_103a): the default engine of batch-1 decoder stacks, streamed
// rings and single products.
//
// Work unit = a tile of 32 matrix rows (16 rows of gate and the same 16 rows
// of up for the paired feed-forward product) over the full width k, staged in
// column chunks of 64 blocks.  Three kinds of warps:
//
// * Warp 9, the producer: one lane walks the CTA's units of every phase of
//   the launch and copies each chunk of a unit with one 2-D tensor TMA copy
//   (box: 146 64-bit columns by 32 rows, so every staged row starts 1168 bytes
//   after the previous one and the code-word loads of the 8 row groups of a
//   tile fall in different banks) into a ring of shared-memory stages,
//   completion counted on one mbarrier per stage.  Weights never depend on
//   the activations, so the producer keeps streaming the next phase's weights
//   while the other warps wait at a phase boundary.
// * Warps 0-7, the consumers (two per SM sub-partition): each takes four
//   pairs of blocks (an even block and the odd one after it) of every chunk
//   and both 16-row halves of the tile, straight-line, so that the eight
//   products of a stage give every warp enough independent work.  Lane (g, t) turns code word t of rows g and g + 8 of a block into
//   exact binary16 values (q - 8) in registers (lop3 with the 0x6400 magic,
//   one subtraction or fused scale per pair) and issues two mma.sync
//   m16n8k16 (binary16 in, fp32 accumulate) against the input, which the
//   phase prologue stored once per phase in shared memory in fragment order
//   with x in every column of the instruction.  Each block's sum is scaled
//   by its d once, in fp32: the products (q - 8) * x are exact, a block of
//   all-8 codes contributes exactly zero and a block with one non-8 code
//   contributes exactly fl(d * (q - 8) * x).  The even block's d arrives with
//   lane 0's first code word and the odd block's with lane 3's second one, so
//   no load is spent on the scales; lane 0 accumulates the even blocks and
//   lane 3 the odd ones, and one shuffle adds them at the end of the unit.
// * Warp 8, the epilogue: sums the 8 consumer warps' partials of each row
//   of a unit in a fixed order as soon as the unit is done (eight partial slots
//   handed over with mbarriers) and stores the outputs, so the consumers
//   never wait for an epilogue.
//
// Phases pass their outputs to the next phase as tagged words (the same
// protocol as the CUDA-core engine's tagged programs, q4_engine.cu): a value
// travels with the tag of the phase that wrote it in one aligned word, and a
// CTA stages its whole input by polling the words until every tag matches;
// one flag exchange per layer guards the rewrite of the tagged buffers.  An
// RMSNorm input is staged in registers and its sum of squares taken in an
// order that depends only on its length, so every CTA forms the same input.
//
// The method: PIPO's dequantisation-free 4-bit matrix-vector product
// ("PIPO: Pipelined Offloading for Efficient Inference on Consumer
// Devices", Method, "Computation optimization"), layer by layer (same page,
// "Offloading architecture"), with the weights of later work prefetched
// while the current work computes (PipeLLM page, "Layer 2: Asynchronous
// Weight Prefetching").
#include <cuda.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "q4_device.cuh"
#include "q4_frag.cuh"
#include "q4_phase.cuh"

namespace q4 {

__device__ int g_status_tc;   // status bits of launches without a control block

// Timeline build (-DQ4_TIMELINE, libq4_tl.so): the GPU's global timer at six
// points of every phase of every CTA, indexed by the phase's place in the
// program: 0 consumers reach the phase, 1 after their barrier, 2 input staged,
// 3 last unit handed to the epilogue, 4 last unit stored by the epilogue,
// 5 last stage issued by the producer.  Other builds compile the stamps away.
#ifdef Q4_TIMELINE
constexpr int kTlCtas = 256, kTlPhases = 64, kTlEvents = 6;
__device__ unsigned long long g_tc_tl[kTlCtas * kTlPhases * kTlEvents];
__device__ __forceinline__ void tc_stamp(int phase, int event) {
  if (phase < kTlPhases) {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    g_tc_tl[(blockIdx.x * kTlPhases + phase) * kTlEvents + event] = t;
  }
}
#else
__device__ __forceinline__ void tc_stamp(int, int) {}
#endif

constexpr int kTcWarps = 8;                       // consumer warps (two per SM sub-partition)
constexpr int kTcConsumers = kTcWarps * 32;
constexpr int kTcPairsPerWarp = 32 / kTcWarps;    // block pairs of a 64-block chunk per warp
constexpr int kTcEpiWarp = kTcWarps;              // warp 8
constexpr int kTcProdWarp = kTcWarps + 1;         // warp 9
constexpr int kTcThreads = (kTcWarps + 2) * 32;
constexpr int kTcMaxStages = 8;
constexpr int kTcRedSlots = 8;                    // unit partial slots between consumers and epilogue
constexpr int kTcRedBytes = kTcRedSlots * kTcWarps * kTcUnitRows * 4;
constexpr int kTcNormChunks = 8;                  // 4-value chunks of an RMSNorm input per consumer thread
constexpr int kTcDynSmemMax = 231424;

extern __shared__ __align__(128) uint8_t g_tc_smem[];

__device__ __forceinline__ void tc_set_status(Control* ctl, int bits) {
  atomicOr(ctl ? &ctl->status : &g_status_tc, bits);
}

__device__ __forceinline__ const Phase& phase_at(const EngineArgs& a, int p) {
  return a.phases ? a.phases[p] : a.one;
}

__device__ __forceinline__ int first_unit(const Phase& ph, int cta, int G) { return (cta - ph.base % G + G) % G; }
// First row of unit u (rpu rows per unit), after the phase's row rotation.
__device__ __forceinline__ int unit_row0(const Phase& ph, int u, int rpu) {
  const int r = u * rpu + ph.row_rot;
  return r >= ph.n_rows ? r - ph.n_rows : r;
}

// ------------------------------------------------------------------ input

// Four consecutive input values e..e+3 (e % 4 == 0), as binary16 pairs
// h01 = (x_e, x_e+1) and h23 = (x_e+2, x_e+3), into the fragment-order buffer:
// lane quarter t of block b holds x[32b + 4t + {0, 2, 1, 3}] and the same 16
// further on, the k order in which unpack_word delivers the codes.
__device__ __forceinline__ void frag_store4(uint8_t* xf, int e, uint32_t h01, uint32_t h23) {
  const int b = e >> 5, i = e & 31;
  const int off = ((b << 2) + ((i & 15) >> 2)) * 16 + ((i >> 4) << 3);
  *reinterpret_cast<uint2*>(xf + off) = make_uint2(__byte_perm(h01, h23, 0x5410), __byte_perm(h01, h23, 0x7632));
}

// CTA 0 also leaves the formed input of a phase: natural binary16 in x_dbg and
// tagged binary16 words in xr_out (the residual base a later phase reads).
__device__ __forceinline__ void store_formed4(const Phase& ph, int e, uint32_t h01, uint32_t h23, uint32_t tag16) {
  if (ph.x_dbg) *reinterpret_cast<uint2*>(ph.x_dbg + e) = make_uint2(h01, h23);
  if (ph.xr_out) {
    const uint32_t t = tag16 << 16;
    st_relaxed_v4(ph.xr_out + e, make_uint4((h01 & 0xFFFFu) | t, (h01 >> 16) | t, (h23 & 0xFFFFu) | t, (h23 >> 16) | t));
  }
}

// The consumer threads together: wait until every CTA's phase flag carries
// `tag` or a later one.  Thread i reads flag i (one load per thread, all in
// flight at once) and the CTA decides by one barrier reduction per poll, so
// every thread polls as often as the others (a thread whose own limit has run
// out votes to stop); the longest limit bounds the wait.  Each thread fences
// after it, before any later access.
__device__ __forceinline__ void tc_wait_flags_cta(const unsigned long long* flags, unsigned tag, int tid,
                                                  uint32_t limit, Control* ctl) {
  const int G = static_cast<int>(gridDim.x);
  bool mine = false;
  for (uint32_t it = 0;; ++it) {
    mine = tid >= G || static_cast<int>(static_cast<unsigned>(ld_relaxed_u64(flags + tid) >> 32) - tag) >= 0;
    uint32_t stop;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.and.pred p, 1, %2, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(stop)
        : "r"(static_cast<uint32_t>(mine || it + 1 >= limit)), "n"(kTcConsumers)
        : "memory");
    if (stop) break;
    if (it > 16) __nanosleep(64);
  }
  if (!mine) tc_set_status(ctl, ST_FLAG_TIMEOUT);
  __threadfence();
}

// The RMSNorm input of a phase (k values, at most 8192): staged in
// registers, 4 consecutive values per chunk, chunk i = tid + c * 256.  Tagged
// fp32 words are polled until every tag is `want`; a plain binary16 input is
// read once.  The sum of squares runs over each thread's chunks in order,
// then the warp tree, then the 8 warps in order: an order fixed by k alone.
// With `flags` set, the consumers first wait for the layer's phase flags (tag
// flag_tag): the flags guard the phase's first tagged write, which follows
// the reduction's barrier.
// Returns the scale 1 / sqrt(mean(t^2) + eps); v holds the values.
__device__ __forceinline__ float stage_norm(const Phase& ph, uint32_t want, uint32_t limit, Control* ctl, float* red_cta,
                                            int tid, float (&v)[kTcNormChunks][4], const unsigned long long* flags,
                                            unsigned flag_tag) {
  const int n4 = ph.k >> 2;
  if (flags) tc_wait_flags_cta(flags, flag_tag, tid, limit, ctl);
  if (ph.x_kind == X_NORM16) {
#pragma unroll
    for (int c = 0; c < kTcNormChunks; ++c) {
      const int i = tid + c * kTcConsumers;
      if (i < n4) {
        const uint2 u = __ldcg(reinterpret_cast<const uint2*>(ph.x_src) + i);
        const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
        const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
        v[c][0] = a.x;
        v[c][1] = a.y;
        v[c][2] = b.x;
        v[c][3] = b.y;
      }
    }
  } else {   // X_TAG32_NORM: 64-bit words {fp32 value, tag}
    const uint4* src = static_cast<const uint4*>(ph.x_src);
    bool ok = false;
    for (uint32_t it = 0; it < limit && !ok; ++it) {
      ok = true;
#pragma unroll
      for (int c = 0; c < kTcNormChunks; ++c) {
        const int i = tid + c * kTcConsumers;
        if (i < n4) {
          const uint4 a = ld_relaxed_v4(src + 2 * i);
          const uint4 b = ld_relaxed_v4(src + 2 * i + 1);
          ok &= a.y == want && a.w == want && b.y == want && b.w == want;
          v[c][0] = __uint_as_float(a.x);
          v[c][1] = __uint_as_float(a.z);
          v[c][2] = __uint_as_float(b.x);
          v[c][3] = __uint_as_float(b.z);
        }
      }
      if (!ok && it >= 2) __nanosleep(32);
    }
    if (!ok) tc_set_status(ctl, ST_DATA_TIMEOUT);
  }
  float ss = 0.f;
#pragma unroll
  for (int c = 0; c < kTcNormChunks; ++c)
    if (tid + c * kTcConsumers < n4)
#pragma unroll
      for (int q = 0; q < 4; ++q) ss = fmaf(v[c][q], v[c][q], ss);
  ss = warp_sum(ss);
  if ((tid & 31) == 0) red_cta[tid >> 5] = ss;
  named_bar_sync(1, kTcConsumers);
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < kTcWarps; ++w) tot += red_cta[w];
  return rsqrtf(tot / static_cast<float>(ph.k) + ph.eps);
}

// Tagged binary16 words (X_TAG16: x = the k values; X_TAG16_ATTN: the xt_n
// values of v, each 4-value chunk of a value head copied to the `group` query
// heads that read it) polled until every tag is `want16`, into the fragment
// buffer.
__device__ __forceinline__ void stage_tag16(const Phase& ph, uint8_t* xf, uint32_t want16, uint32_t limit, Control* ctl,
                                            int tid, bool cta0) {
  const bool attn = ph.x_kind == X_TAG16_ATTN;
  const int n4 = (attn ? ph.xt_n : ph.k) >> 2;
  const uint4* src = static_cast<const uint4*>(ph.x_src);
  const uint32_t want = want16 << 16;
  // The thread's chunks in batches of 4, each batch polled until its tags
  // match before the next is read: the values arrive roughly in row order,
  // so once the last ones land only the last batches are still to be read.
  bool all_ok = true;
  for (int i0 = tid; i0 < n4; i0 += 4 * kTcConsumers) {
    uint32_t lo[4], hi[4];
    bool ok;
    uint32_t it = 0;
    do {   // at least one read, so lo and hi always hold the loaded words
      ok = true;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int i = i0 + j * kTcConsumers;
        if (i < n4) {
          const uint4 w = ld_relaxed_v4_nb(src + i);
          ok &= (((w.x ^ want) | (w.y ^ want) | (w.z ^ want) | (w.w ^ want)) >> 16) == 0u;
          lo[j] = __byte_perm(w.x, w.y, 0x5410);
          hi[j] = __byte_perm(w.z, w.w, 0x5410);
        }
      }
      if (!ok && it >= 2) __nanosleep(32);
    } while (!ok && ++it < limit);
    all_ok &= ok;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = i0 + j * kTcConsumers;
      if (i < n4) {
        const int e = 4 * i;
        if (!attn) {
          frag_store4(xf, e, lo[j], hi[j]);
        } else {
          const int hd = ph.head_dim;
          const int x0 = (e / hd) * ph.group * hd + e % hd;
          for (int h = 0; h < ph.group; ++h) frag_store4(xf, x0 + h * hd, lo[j], hi[j]);
        }
      }
    }
  }
  if (!all_ok) tc_set_status(ctl, ST_DATA_TIMEOUT);
  if (cta0 && (ph.x_dbg || ph.xr_out)) {
    // The formed x in natural order.  Its chunks were polled by other threads:
    // after the barrier every word carries its tag (re-checked, bounded).
    named_bar_sync(1, kTcConsumers);
    const int k4 = ph.k >> 2;
    for (int i = tid; i < k4; i += kTcConsumers) {
      int s = i;
      if (attn) {
        const int e = 4 * i, hd = ph.head_dim;
        s = (((e / hd) / ph.group) * hd + e % hd) >> 2;
      }
      uint4 w = ld_relaxed_v4(src + s);
      for (uint32_t it = 0; (((w.x ^ want) | (w.y ^ want) | (w.z ^ want) | (w.w ^ want)) >> 16) != 0u && it < limit;
           ++it)
        w = ld_relaxed_v4(src + s);
      store_formed4(ph, 4 * i, __byte_perm(w.x, w.y, 0x5410), __byte_perm(w.z, w.w, 0x5410), want16);
    }
  }
}

// A plain binary16 input (single products) into the fragment buffer.
__device__ __forceinline__ void stage_plain16(const Phase& ph, uint8_t* xf, int tid) {
  const int n4 = ph.k >> 2;
  for (int i = tid; i < n4; i += kTcConsumers) {
    const uint2 u = __ldcg(reinterpret_cast<const uint2*>(ph.x_src) + i);
    frag_store4(xf, 4 * i, u.x, u.y);
  }
}

// The prologue of a phase for a CTA that reads its input: wait for the
// previous layer's flags where the phase asks for it, stage the whole input
// in fragment order (normalised for the RMSNorm inputs), meet at a barrier of
// the consumer warps.  Out of line: the unit loop's registers are allocated
// without the staging loads.
__device__ __noinline__ void tc_prologue(const Phase& ph, unsigned tag, uint32_t lim, Control* ctl,
                                         const unsigned long long* flags, uint8_t* xf, float* red_cta, int tid,
                                         bool cta0) {
  const bool norm = ph.x_kind == X_NORM16 || ph.x_kind == X_TAG32_NORM;
  if (ph.sync == SYNC_WAIT && !norm) tc_wait_flags_cta(flags, tag - 1u, tid, lim, ctl);
  if (ph.sync == SYNC_WAIT && !norm) named_bar_sync(1, kTcConsumers);
  if (norm) {
    float v[kTcNormChunks][4];
    const float r = stage_norm(ph, tag - 1u, lim, ctl, red_cta, tid, v, ph.sync == SYNC_WAIT ? flags : nullptr,
                               tag - 1u);
    const int n4 = ph.k >> 2;
#pragma unroll
    for (int c = 0; c < kTcNormChunks; ++c) {
      const int i = tid + c * kTcConsumers;
      if (i < n4) {
        const __half2 a = __floats2half2_rn(v[c][0] * r, v[c][1] * r);
        const __half2 b = __floats2half2_rn(v[c][2] * r, v[c][3] * r);
        const uint32_t h01 = *reinterpret_cast<const uint32_t*>(&a), h23 = *reinterpret_cast<const uint32_t*>(&b);
        frag_store4(xf, 4 * i, h01, h23);
        if (cta0) store_formed4(ph, 4 * i, h01, h23, tag & 0xFFFFu);
      }
    }
  } else if (ph.x_kind == X_F16) {
    stage_plain16(ph, xf, tid);
  } else {
    stage_tag16(ph, xf, (tag - 1u) & 0xFFFFu, lim, ctl, tid, cta0);
  }
  named_bar_sync(1, kTcConsumers);
}

// ------------------------------------------------------------------ compute

// Wait for a stage to land.  The common case (the copy has landed) is one
// non-blocking test; after a failed wait the CTA keeps walking its units
// without waiting (reading whatever the stage holds) so that every barrier is
// still reached, and the launch reports the failure in its status.
__device__ __forceinline__ void stage_wait(uint64_t* bar, uint32_t parity, uint32_t limit, volatile int* abort_flag,
                                           Control* ctl) {
  if (mbar_test_wait(bar, parity)) return;
  if (!*abort_flag && !mbar_wait_bounded(bar, parity, limit)) {
    tc_set_status(ctl, ST_FULL_TIMEOUT);
    *abort_flag = 1;
  }
}

// The products of one unit for one consumer warp, chunk by chunk as the
// stages land: four block pairs of every chunk (pairs warp + 8q) and
// both 16-row halves of the tile.  WIDE: rows wider than 2048 columns (64-block
// chunks, 1168-byte staged rows), with the geometry as constants; otherwise
// the chunk is the whole row.  acc[m] = {even-block sums of rows g, g + 8,
// odd-block sums of rows g, g + 8} of half m.
template <bool WIDE>
__device__ __forceinline__ void unit_products(const uint8_t* ring, uint32_t SB, int S, int& slot, uint32_t& use,
                                              uint64_t* full_bar, uint64_t* empty_bar, volatile int* abort_flag,
                                              const uint4* xf4, int chunks, int cb_rt, int pitch_rt, int warp,
                                              int lane, uint32_t magic, uint32_t wait_limit, Control* ctl,
                                              float (&acc)[2][4]) {
  const int cb = WIDE ? 64 : cb_rt;
  const int pitch = WIDE ? 64 * kBlockBytes + 16 : pitch_rt;
  const int g = lane >> 2, t = lane & 3;
  for (int c = 0; c < chunks; ++c) {
    stage_wait(&full_bar[slot], use & 1, wait_limit, abort_flag, ctl);
    const uint8_t* sb = ring + static_cast<size_t>(slot) * SB;
#pragma unroll(WIDE ? kTcPairsPerWarp : 1)
    for (int q = 0; q < kTcPairsPerWarp; ++q) {
      const int pp = warp + kTcWarps * q;   // block pair of the chunk
      if (WIDE || 2 * pp < cb) {
        const int blk = c * cb + 2 * pp;
        const uint4 xe = xf4[blk * 4 + t], xo = xf4[(blk + 1) * 4 + t];
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          const uint8_t* rg = sb + (m * 16 + g) * pitch + 36 * pp;
          pair_mma(rg, rg + 8 * pitch, t, xe, xo, magic, acc[m][0], acc[m][1], acc[m][2], acc[m][3]);
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

// ------------------------------------------------------------------ epilogue

// A tagged residual input word (w: its value loaded earlier), polled until it
// carries tag16.
__device__ __forceinline__ unsigned short tc_tagged_res(const uint32_t* p, uint32_t w, uint32_t tag16, uint32_t limit,
                                                        Control* ctl) {
  for (uint32_t it = 0; (w >> 16) != tag16 && it < limit; ++it) {
    __nanosleep(32);
    w = ld_relaxed_b32(p);
  }
  if ((w >> 16) != tag16) tc_set_status(ctl, ST_DATA_TIMEOUT);
  return static_cast<unsigned short>(w & 0xFFFFu);
}

// The outputs of one row (lane) of a finished unit.  Tagged programs hand the
// next phase its input as tagged words with this phase's tag; the plain
// outputs are written where the phase has them.
__device__ __forceinline__ void tc_epilogue_row(const Phase& ph, int n, float v, float u2, uint32_t res_w, bool tagged,
                                                uint32_t tag, uint32_t lim, Control* ctl) {
  const uint32_t tag16 = tag & 0xFFFFu;
  if (ph.epi_kind == EPI_SILU) {
    if (ph.y) ph.y[n] = v;
    if (ph.y2) ph.y2[n] = u2;
    const unsigned short a16 = __half_as_ushort(__float2half_rn(silu_mul(v, u2)));
    if (ph.aux16) ph.aux16[n] = a16;
    if (tagged) st_relaxed_b32(static_cast<uint32_t*>(ph.yt) + n, (tag16 << 16) | a16);
  } else if (ph.epi_kind == EPI_RESID) {
    if (ph.y) ph.y[n] = v;
    const unsigned short rv = tc_tagged_res(ph.res_t + n, res_w, (tag - 1u) & 0xFFFFu, lim, ctl);
    const float tv = __half2float(__ushort_as_half(rv)) + v;
    if (ph.y2) ph.y2[n] = tv;
    st_relaxed_b64(static_cast<unsigned long long*>(ph.yt) + n,
                   (static_cast<unsigned long long>(tag) << 32) | __float_as_uint(tv));
  } else {
    if (ph.y) ph.y[n] = v;
    const int e = n - ph.yt_off;
    if (tagged && ph.yt && e >= 0 && e < ph.yt_n)
      st_relaxed_b32(static_cast<uint32_t*>(ph.yt) + e, (tag16 << 16) | __half_as_ushort(__float2half_rn(v)));
  }
}

// ------------------------------------------------------------------ kernel

__global__ void __launch_bounds__(kTcThreads, 1) tc_engine_kernel(const __grid_constant__ EngineArgs a) {
  __shared__ __align__(8) uint64_t full_bar[kTcMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kTcMaxStages];
  __shared__ __align__(8) uint64_t rfull_bar[kTcRedSlots];
  __shared__ __align__(8) uint64_t rempty_bar[kTcRedSlots];
  __shared__ float red_cta[kTcWarps];
  __shared__ volatile int abort_flag;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, cta = blockIdx.x;
  const int S = a.stages;
  const uint32_t SB = a.stage_bytes;
  uint8_t* const ring = g_tc_smem;
  uint8_t* const xf = g_tc_smem + static_cast<size_t>(S) * SB;
  float* const red = reinterpret_cast<float*>(xf + 4 * static_cast<size_t>(a.xbuf_floats));
  const bool tagged = a.tagged != 0;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kTcWarps);
    }
    for (int s = 0; s < kTcRedSlots; ++s) {
      mbar_init(&rfull_bar[s], kTcWarps);
      mbar_init(&rempty_bar[s], 1);
    }
    fence_mbar_init();
    abort_flag = 0;
  }
  __syncthreads();
  // programmatic dependent launch: the next launch may be scheduled (it waits
  // for this one before it reads anything this one writes); the weights need
  // nothing from the launch before this one, everything else does
  if (a.pdl & 2) griddep_launch_dependents();
  if ((a.pdl & 1) && warp != kTcProdWarp) griddep_wait();

  const unsigned tag0 = tagged ? a.ctl->epoch * kPhasesPerEpoch + 1u : 0u;

  if (warp == kTcProdWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t it = 0;
      int slot = 0;
      uint32_t use = 0;
      for (int p = 0; p < a.n_phases && !abort_flag; ++p) {
        const Phase& ph = phase_at(a, p);
        if (a.phases && ph.units > 0) {
          // descriptors written by the host into global memory: order their use
          // through the tensor-map proxy after the generic-proxy writes
          tensormap_acquire(&ph.tm0);
          if (ph.epi_kind == EPI_SILU) tensormap_acquire(&ph.tm1);
        }
        const int chunks = tc_chunks(ph.k);
        const int cx = tc_chunk_blocks(ph.k) * kBlockBytes / 8;   // chunk stride in 64-bit columns
        const int pitch = tc_pitch(ph.k);
        const bool dual = ph.epi_kind == EPI_SILU;
        const uint32_t bytes = static_cast<uint32_t>(pitch) * kTcUnitRows;
        const int units = ph.units;
        for (int u = first_unit(ph, cta, G); u < units && !abort_flag; u += G) {
          for (int c = 0; c < chunks; ++c) {
            if (use > 0 && !mbar_wait_bounded(&empty_bar[slot], (use - 1) & 1, a.wait_limit)) {
              tc_set_status(a.ctl, ST_EMPTY_TIMEOUT);
              abort_flag = 1;
              break;
            }
            uint8_t* dst = ring + static_cast<size_t>(slot) * SB;
            mbar_arrive_expect_tx(&full_bar[slot], bytes);
            if (dual) {
              const int r0 = unit_row0(ph, u, kTcUnitRows / 2);
              tma_load_2d(dst, &ph.tm0, c * cx, r0, &full_bar[slot]);
              tma_load_2d(dst + (kTcUnitRows / 2) * pitch, &ph.tm1, c * cx, r0, &full_bar[slot]);
            } else {
              tma_load_2d(dst, &ph.tm0, c * cx, unit_row0(ph, u, kTcUnitRows), &full_bar[slot]);
            }
            ++it;
            tc_stamp(ph.gidx, 5);
            if (++slot == S) {
              slot = 0;
              ++use;
            }
          }
        }
      }
      // Drain: no copy may still be in flight when the CTA exits.
      const uint32_t issued = it;
      for (int s = 0; s < S && static_cast<uint32_t>(s) < issued; ++s) {
        const uint32_t last = (issued - 1 - s) / S;
        if (!mbar_wait_bounded(&full_bar[s], last & 1, a.wait_limit)) tc_set_status(a.ctl, ST_DRAIN_TIMEOUT);
      }
    }
  } else if (warp == kTcEpiWarp) {
    // ------------------------------------------------------------ epilogue
    int rs = 0;
    uint32_t ruse = 0;
    const uint32_t st0 = tagged ? ld_relaxed_b32(&a.ctl->status) : 0u;
    for (int p = 0; p < a.n_phases; ++p) {
      const Phase& ph = phase_at(a, p);
      const unsigned tag = tag0 + static_cast<unsigned>(ph.gidx);
      const bool dual = ph.epi_kind == EPI_SILU;
      const int units = ph.units;
      for (int u = first_unit(ph, cta, G); u < units; u += G) {
        // once a wait of this launch has run out, the residual polls give up at once
        const uint32_t lim = tagged && ld_relaxed_b32(&a.ctl->status) != st0 ? 0u : a.wait_limit;
        const int n = unit_row0(ph, u, dual ? kTcUnitRows / 2 : kTcUnitRows) + lane;
        const bool row_ok = (!dual || lane < kTcUnitRows / 2) && n < ph.n_rows;
        // the residual base of this row was written phases ago: its load
        // overlaps the wait for the unit's partials
        const uint32_t res_w = row_ok && ph.epi_kind == EPI_RESID ? ld_relaxed_b32(ph.res_t + n) : 0u;
        if (!mbar_wait_bounded(&rfull_bar[rs], ruse & 1, a.wait_limit)) tc_set_status(a.ctl, ST_FULL_TIMEOUT);
        const float* pr = red + rs * (kTcWarps * kTcUnitRows);
        float v = 0.f, u2 = 0.f;
#pragma unroll
        for (int w = 0; w < kTcWarps; ++w) v += pr[w * kTcUnitRows + lane];
        if (dual) u2 = __shfl_down_sync(0xffffffffu, v, 16);   // up row r sits 16 rows below gate row r
        __syncwarp();
        if (lane == 0) mbar_arrive(&rempty_bar[rs]);
        if (++rs == kTcRedSlots) {
          rs = 0;
          ++ruse;
        }
        if (row_ok) tc_epilogue_row(ph, n, v, u2, res_w, tagged, tag, lim, a.ctl);
        if (lane == 0) tc_stamp(ph.gidx, 4);
      }
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int g = lane >> 2, t = lane & 3;
    uint32_t magic;
    asm volatile("mov.b32 %0, 0x64006400;" : "=r"(magic));
    int slot = 0;
    uint32_t use = 0;
    int rs = 0;
    uint32_t ruse = 0;
    const uint32_t st0 = tagged ? ld_relaxed_b32(&a.ctl->status) : 0u;
    for (int p = 0; p < a.n_phases; ++p) {
      const Phase& ph = phase_at(a, p);
      const unsigned tag = tag0 + static_cast<unsigned>(ph.gidx);
      const uint32_t lim = tagged && ld_relaxed_b32(&a.ctl->status) != st0 ? 0u : a.wait_limit;
      const int u0 = first_unit(ph, cta, G);
      const bool cta0 = cta == 0 && (ph.x_dbg || ph.xr_out);
      // every consumer warp is done with the previous phase's input
      if (tid == 0) tc_stamp(ph.gidx, 0);
      named_bar_sync(1, kTcConsumers);
      if (tid == 0) tc_stamp(ph.gidx, 1);
      if (u0 < ph.units || cta0) tc_prologue(ph, tag, lim, a.ctl, a.flags, xf, red_cta, tid, cta0);
      if (tid == 0) tc_stamp(ph.gidx, 2);
      if (ph.sync == SYNC_PUBLISH && tid == 0) st_release_u64(a.flags + cta, static_cast<unsigned long long>(tag) << 32);
      asm volatile("" ::: "memory");
      const int chunks = tc_chunks(ph.k);
      const int cb = tc_chunk_blocks(ph.k);
      const int pitch = tc_pitch(ph.k);
      const bool wide = ph.k > 2048;
      const int units = ph.units;
      const uint4* xf4 = reinterpret_cast<const uint4*>(xf);
      for (int u = u0; u < units; u += G) {
        float acc[2][4] = {};
        if (wide)
          unit_products<true>(ring, SB, S, slot, use, full_bar, empty_bar, &abort_flag, xf4, chunks, cb, pitch, warp,
                              lane, magic, a.wait_limit, a.ctl, acc);
        else
          unit_products<false>(ring, SB, S, slot, use, full_bar, empty_bar, &abort_flag, xf4, chunks, cb, pitch, warp,
                               lane, magic, a.wait_limit, a.ctl, acc);
        // lane (g, 0) adds the odd blocks of lane (g, 3); rows g and g + 8 of each half
        float r[2][2];
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
          for (int h = 0; h < 2; ++h) r[m][h] = acc[m][h] + __shfl_sync(0xffffffffu, acc[m][2 + h], lane | 3);
        if (ruse > 0) {
          // slot rs's previous unit (use ruse - 1) has been read by the epilogue
          if (lane == 0 && !mbar_wait_bounded(&rempty_bar[rs], (ruse - 1) & 1, a.wait_limit))
            tc_set_status(a.ctl, ST_EMPTY_TIMEOUT);
          __syncwarp();
        }
        float* pr = red + rs * (kTcWarps * kTcUnitRows) + warp * kTcUnitRows;
        if (t == 0) {
          pr[g] = r[0][0];
          pr[g + 8] = r[0][1];
          pr[16 + g] = r[1][0];
          pr[24 + g] = r[1][1];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&rfull_bar[rs]);
        if (tid == 0) tc_stamp(ph.gidx, 3);
        if (++rs == kTcRedSlots) {
          rs = 0;
          ++ruse;
        }
      }
    }
  }

  __syncthreads();
  if (tagged && tid == 0) {
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

// Copy the timeline of the last launches out (and clear it): Q4_ERR_ARG-like
// cudaErrorNotSupported in a build without stamps.
cudaError_t tc_timeline_read(unsigned long long* out, size_t n, bool clear) {
#ifdef Q4_TIMELINE
  const size_t total = static_cast<size_t>(kTlCtas) * kTlPhases * kTlEvents;
  if (n < total) return cudaErrorInvalidValue;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_tc_tl, total * sizeof(unsigned long long));
  if (e == cudaSuccess && clear) {
    static unsigned long long zero[kTlCtas * kTlPhases * kTlEvents];
    e = cudaMemcpyToSymbol(g_tc_tl, zero, sizeof(zero));
  }
  return e;
#else
  (void)out;
  (void)n;
  (void)clear;
  return cudaErrorNotSupported;
#endif
}

cudaError_t tc_engine_prepare() {
  return cudaFuncSetAttribute(tc_engine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcDynSmemMax);
}

size_t tc_smem_bytes(int stages, uint32_t stage_bytes, int xbuf_floats) {
  return static_cast<size_t>(stages) * stage_bytes + 4 * static_cast<size_t>(xbuf_floats) + kTcRedBytes;
}

cudaError_t tc_engine_launch(const EngineArgs& a, int grid, bool cooperative, cudaStream_t stream) {
  const size_t smem = tc_smem_bytes(a.stages, a.stage_bytes, a.xbuf_floats);
  if (a.stages < 2 || a.stages > kTcMaxStages || smem > static_cast<size_t>(kTcDynSmemMax) || a.stage_bytes % 128)
    return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  if ((a.pdl & 1) && cooperative) return cudaErrorInvalidValue;
  cudaLaunchAttribute attr[1];
  if (a.pdl & 1) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
  } else {
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = cooperative ? 1 : 0;
  }
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tc_engine_kernel, a);
}

cudaError_t tc_engine_occupancy(int* blocks_per_sm) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, tc_engine_kernel, kTcThreads, kTcDynSmemMax);
}

cudaError_t tc_engine_read_status(int* out) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_status_tc, sizeof(int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_status_tc, &zero, sizeof(int));
}

}  // namespace q4
