// Persistent, warp-specialised Q4_0 matrix-vector engine on the tensor cores
// (batch 1, sm_103a).
//
// Same phase programs as the CUDA-core engine (q4_engine.cu): a launch runs
// a list of matrix-vector products with input prologues and output
// epilogues, separated by per-CTA end-of-phase flags.  What differs is the
// inner product and the way weights reach it:
//
// * Work unit = a tile of 16 matrix rows (or 8 rows of each matrix of a
//   gate/up pair, stacked as one 16-row tile) over the full width k, staged
//   in column chunks of 64 blocks.  Warp 16 (the producer) copies each
//   chunk's 16 row segments with 1-D bulk TMA into an 8-deep ring of
//   shared-memory stages; rows are padded so the code-word loads of the 8
//   row groups fall in different banks.
// * The 16 consumer warps take 4 of a chunk's 64 blocks each.  A lane turns
//   its two code words (rows g and g+8) into exact binary16 (q - 8) values in
//   registers and issues two mma.sync m16n8k16 (binary16 in, fp32
//   accumulate) against the input, which the prologue stored once per phase
//   in shared memory in fragment order (every column of the instruction sees
//   the same x, so every lane ends with its rows' sums).  Each block's sum is
//   scaled by its d once, in fp32: the products (q - 8) * x are exact, a
//   block of all-8 codes contributes exactly zero and a block with one non-8
//   code contributes exactly fl(d * (q - 8) * x).
// * Besides the ring, the producer keeps up to `prefetch_bytes` of its
//   upcoming units requested into L2 (cp.async.bulk.prefetch), across phase
//   boundaries: weights never depend on the activations, so HBM keeps
//   streaming while the consumers wait at a phase boundary.
//
// The method: PIPO's dequantisation-free 4-bit matrix-vector product
// ("PIPO: Pipelined Offloading for Efficient Inference on Consumer
// Devices", Method, "Computation optimization"), layer by layer (same page,
// "Offloading architecture"), with the weights of later work prefetched
// while the current work computes (PipeLLM page, "Layer 2: Asynchronous
// Weight Prefetching").
#include <cuda_fp16.h>
#include <stdint.h>

#include "q4_device.cuh"
#include "q4_frag.cuh"
#include "q4_phase.cuh"

namespace q4 {

__device__ int g_status_tc;   // status bits of launches without a control block

constexpr int kTcWarps = 16;                          // consumer warps
constexpr int kTcConsumers = kTcWarps * 32;
constexpr int kTcThreads = kTcConsumers + 32;         // + the producer warp
constexpr int kTcChunk = 64;                          // blocks per staged row segment (2048 columns)
constexpr int kTcPitch = kTcChunk * kBlockBytes + 16; // 1168 B: rows 4 banks apart
constexpr int kTcStageBytes = 16 * kTcPitch;          // 18688 B
constexpr int kTcStages = 8;
constexpr int kTcMaxK = 30720;
constexpr int kTcXBytes = kTcMaxK * 2;                // the phase input in fragment order
constexpr int kTcRedUnits = 16;                       // units buffered before a flush
constexpr int kTcSmem = kTcStages * kTcStageBytes + kTcXBytes;
constexpr uint32_t kTcPrefetchPiece = 16384;          // bytes per L2 prefetch instruction

extern __shared__ __align__(128) uint8_t g_tc_smem[];

__device__ __forceinline__ void tc_set_status(Control* ctl, int bits) {
  atomicOr(ctl ? &ctl->status : &g_status_tc, bits);
}

__device__ __forceinline__ const Phase& phase_at(const EngineArgs& a, int p) {
  return a.phases ? a.phases[p] : a.one;
}

// This CTA's walk over its units of all phases (units u0, u0 + G, ... of each
// phase, u0 = (cta - base) mod G rotating so that the phases' first units go
// to different CTAs).
struct Walk {
  int p, u;
};

__device__ __forceinline__ int first_unit(const Phase& ph, int cta, int G) { return (cta - ph.base % G + G) % G; }

__device__ __forceinline__ void walk_settle(Walk& w, const EngineArgs& a, int cta, int G) {
  while (w.p < a.n_phases) {
    if (w.u < phase_at(a, w.p).units) return;
    ++w.p;
    if (w.p < a.n_phases) w.u = first_unit(phase_at(a, w.p), cta, G);
  }
}

// Request unit (p, u)'s rows into L2, the pieces spread over the warp's lanes.
__device__ __forceinline__ uint32_t prefetch_unit(const Phase& ph, int u, int lane) {
  const uint32_t row_bytes = static_cast<uint32_t>(ph.k / kQK) * kBlockBytes;
  const int row0 = u * ph.rows_per_unit;
  const int rows = min(ph.rows_per_unit, ph.n_rows - row0);
  const uint32_t bytes = static_cast<uint32_t>(rows) * row_bytes;   // rows of a unit are contiguous
  const int mats = ph.epi_kind == EPI_SILU ? 2 : 1;
  const uint32_t pieces = (bytes + kTcPrefetchPiece - 1) / kTcPrefetchPiece;
  for (uint32_t i = lane; i < mats * pieces; i += 32) {
    const uint8_t* base = (i < pieces ? ph.w0 : ph.w1) + static_cast<size_t>(row0) * row_bytes;
    const uint32_t off = (i % pieces) * kTcPrefetchPiece;
    bulk_prefetch_l2(base + off, min(kTcPrefetchPiece, bytes - off));
  }
  return bytes * mats;
}

// The phase input in fragment order: for block b and lane quarter t, 16
// bytes holding x[32b + 4t + {0, 2, 1, 3}] and x[32b + 16 + 4t + {0, 2, 1, 3}]
// (the k order in which unpack_word delivers the weights).  The values are
// formed per XKind; CTA 0 also stores the formed x in natural order to
// x_dbg when asked.  All loads of a pass are issued before its arithmetic.
__device__ void tc_form_x(const Phase& ph, uint4* xf, float sumsq, int tid, bool dbg) {
  const bool norm = ph.x_kind == X_NORM16 || ph.x_kind == X_NORM32;
  const float r = norm ? rsqrtf(sumsq / static_cast<float>(ph.k) + ph.eps) : 1.0f;
  const int nf = ph.k >> 3;
  constexpr int kPass = 4;
  for (int f0 = tid; f0 < nf; f0 += kPass * kTcConsumers) {
    float v[kPass][8];
#pragma unroll
    for (int q = 0; q < kPass; ++q) {
      const int f = f0 + q * kTcConsumers;
      if (f >= nf) break;
      const int e0 = 32 * (f >> 2) + 4 * (f & 3);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int e = e0 + 16 * h;
        if (ph.x_kind == X_F16 || ph.x_kind == X_NORM16) {
          const uint2 u = __ldcg(reinterpret_cast<const uint2*>(static_cast<const __half*>(ph.x_src) + e));
          const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
          const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
          v[q][4 * h] = a.x;
          v[q][4 * h + 1] = a.y;
          v[q][4 * h + 2] = b.x;
          v[q][4 * h + 3] = b.y;
        } else {
          int src = e;
          if (ph.x_kind == X_ATTN) src = ph.attn_off + ((e / ph.head_dim) / ph.group) * ph.head_dim + e % ph.head_dim;
          const float4 a = __ldcg(reinterpret_cast<const float4*>(static_cast<const float*>(ph.x_src) + src));
          v[q][4 * h] = a.x;
          v[q][4 * h + 1] = a.y;
          v[q][4 * h + 2] = a.z;
          v[q][4 * h + 3] = a.w;
        }
      }
    }
#pragma unroll
    for (int q = 0; q < kPass; ++q) {
      const int f = f0 + q * kTcConsumers;
      if (f >= nf) break;
      __half2 h[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        h[i] = norm ? __floats2half2_rn(v[q][2 * i] * r, v[q][2 * i + 1] * r)
                    : __floats2half2_rn(v[q][2 * i], v[q][2 * i + 1]);
      // natural order: h[0] = (e0, e0+1), h[1] = (e0+2, e0+3), h[2], h[3] the same 16 further
      uint4 o;
      o.x = __byte_perm(*reinterpret_cast<uint32_t*>(&h[0]), *reinterpret_cast<uint32_t*>(&h[1]), 0x5410);
      o.y = __byte_perm(*reinterpret_cast<uint32_t*>(&h[0]), *reinterpret_cast<uint32_t*>(&h[1]), 0x7632);
      o.z = __byte_perm(*reinterpret_cast<uint32_t*>(&h[2]), *reinterpret_cast<uint32_t*>(&h[3]), 0x5410);
      o.w = __byte_perm(*reinterpret_cast<uint32_t*>(&h[2]), *reinterpret_cast<uint32_t*>(&h[3]), 0x7632);
      xf[f] = o;
      if (dbg) {
        const int e0 = 32 * (f >> 2) + 4 * (f & 3);
        uint2 lo, hi;
        lo.x = *reinterpret_cast<uint32_t*>(&h[0]);
        lo.y = *reinterpret_cast<uint32_t*>(&h[1]);
        hi.x = *reinterpret_cast<uint32_t*>(&h[2]);
        hi.y = *reinterpret_cast<uint32_t*>(&h[3]);
        *reinterpret_cast<uint2*>(ph.x_dbg + e0) = lo;
        *reinterpret_cast<uint2*>(ph.x_dbg + e0 + 16) = hi;
      }
    }
  }
}

// Sum the 16 warps' partials of the n_buf buffered units (the CTA's units
// u_first, u_first + G, ...) in a fixed order and run the epilogue of their
// rows.  All consumer threads take part.  Returns the thread's sum of squares
// of the residual sums it wrote (EPI_RESID), for the next RMSNorm.
__device__ float tc_flush(const Phase& ph, const float* red, int n_buf, int u_first, int G, int tid, bool reuse) {
  named_bar_sync(1, kTcConsumers);
  float ss = 0.f;
  if (ph.epi_kind != EPI_SILU) {
    for (int o = tid; o < n_buf * 16; o += kTcConsumers) {
      const int s = o >> 4, m = o & 15;
      const float* pr = red + s * kTcWarps * 16 + m;
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < kTcWarps; ++w) v += pr[w * 16];
      const int n = (u_first + s * G) * 16 + m;
      if (n < ph.n_rows) {
        ph.y[n] = v;
        if (ph.epi_kind == EPI_RESID) {
          const float tv = __half2float(__ushort_as_half(ph.res[n])) + v;
          ph.y2[n] = tv;
          ss = fmaf(tv, tv, ss);
        }
      }
    }
  } else {
    for (int o = tid; o < n_buf * 8; o += kTcConsumers) {
      const int s = o >> 3, m = o & 7;
      const float* pr = red + s * kTcWarps * 16 + m;
      float g = 0.f, u = 0.f;
#pragma unroll
      for (int w = 0; w < kTcWarps; ++w) {
        g += pr[w * 16];
        u += pr[w * 16 + 8];
      }
      const int n = (u_first + s * G) * 8 + m;
      if (n < ph.n_rows) {
        ph.y[n] = g;
        ph.y2[n] = u;
        ph.aux16[n] = __half_as_ushort(__float2half_rn(silu_mul(g, u)));
      }
    }
  }
  if (reuse) named_bar_sync(1, kTcConsumers);   // red is written again in this phase
  return ss;
}

__global__ void __launch_bounds__(kTcThreads, 1) tc_engine_kernel(const __grid_constant__ EngineArgs a) {
  __shared__ __align__(8) uint64_t full_bar[kTcStages];
  __shared__ __align__(8) uint64_t empty_bar[kTcStages];
  __shared__ float red[kTcRedUnits * kTcWarps * 16];
  __shared__ float red_cta[kTcWarps];
  __shared__ volatile int abort_flag;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, cta = blockIdx.x;
  uint8_t* ring = g_tc_smem;
  uint4* xf = reinterpret_cast<uint4*>(g_tc_smem + kTcStages * kTcStageBytes);

  if (tid == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kTcWarps);
    }
    fence_mbar_init();
    abort_flag = 0;
  }
  __syncthreads();

  if (warp == kTcWarps) {
    // ------------------------------------------------------------ producer
    uint32_t it = 0;
    Walk pf{0, first_unit(phase_at(a, 0), cta, G)};   // the L2 prefetch cursor runs ahead of the copies
    walk_settle(pf, a, cta, G);
    unsigned long long copied = 0, requested = 0;
    bool stop = false;
    for (int p = 0; p < a.n_phases && !stop; ++p) {
      const Phase& ph = phase_at(a, p);
      const uint32_t row_bytes = static_cast<uint32_t>(ph.k / kQK) * kBlockBytes;
      const int nb = ph.k / kQK;
      const int chunks = (nb + kTcChunk - 1) / kTcChunk;
      const bool dual = ph.epi_kind == EPI_SILU;
      const int rpu = ph.rows_per_unit;
      for (int u = first_unit(ph, cta, G); u < ph.units && !stop; u += G) {
        const int row0 = u * rpu;
        const int rows = min(rpu, ph.n_rows - row0);
        if (a.prefetch_bytes) {
          while (pf.p < a.n_phases && requested < copied + a.prefetch_bytes) {
            requested += prefetch_unit(phase_at(a, pf.p), pf.u, lane);
            pf.u += G;
            walk_settle(pf, a, cta, G);
          }
        }
        for (int c = 0; c < chunks; ++c) {
          const int stage = it % kTcStages;
          const uint32_t n = it / kTcStages;
          int ok = 1;
          if (lane == 0 && n > 0 && !mbar_wait_bounded(&empty_bar[stage], (n - 1) & 1, a.wait_limit)) {
            tc_set_status(a.ctl, ST_EMPTY_TIMEOUT);
            abort_flag = 1;
            ok = 0;
          }
          ok = __shfl_sync(0xffffffffu, ok, 0) && !abort_flag;
          if (!ok) {
            stop = true;
            break;
          }
          const int blk0 = c * kTcChunk;
          const uint32_t seg = static_cast<uint32_t>(min(kTcChunk, nb - blk0)) * kBlockBytes;
          if (lane == 0) mbar_arrive_expect_tx(&full_bar[stage], seg * rows * (dual ? 2 : 1));
          __syncwarp();
          if (lane < 16) {
            const int r = dual ? (lane & 7) : lane;
            if (r < rows) {
              const uint8_t* src = (dual && lane >= 8 ? ph.w1 : ph.w0) + static_cast<size_t>(row0 + r) * row_bytes +
                                   static_cast<size_t>(blk0) * kBlockBytes;
              bulk_g2s(ring + static_cast<size_t>(stage) * kTcStageBytes + lane * kTcPitch, src, seg,
                       &full_bar[stage]);
            }
          }
          ++it;
        }
        copied += static_cast<unsigned long long>(rows) * row_bytes * (dual ? 2 : 1);
      }
    }
    // Drain: no copy may still be in flight when the CTA exits.
    if (lane == 0) {
      const uint32_t issued = it;
      for (int s = 0; s < kTcStages && static_cast<uint32_t>(s) < issued; ++s) {
        const uint32_t last = (issued - 1 - s) / kTcStages;
        if (!mbar_wait_bounded(&full_bar[s], last & 1, a.wait_limit)) tc_set_status(a.ctl, ST_DRAIN_TIMEOUT);
      }
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int g = lane >> 2, t = lane & 3;
    uint32_t magic;
    asm volatile("mov.b32 %0, 0x64006400;" : "=r"(magic));
    uint32_t it = 0;
    const unsigned tag0 = a.n_phases > 1 ? a.ctl->epoch * kPhasesPerEpoch + 1u : 0u;   // tag of phase 0
    for (int p = 0; p < a.n_phases; ++p) {
      const Phase& ph = phase_at(a, p);
      const int units = ph.units;
      const int nb = ph.k / kQK;
      const int chunks = (nb + kTcChunk - 1) / kTcChunk;
      const int u0 = first_unit(ph, cta, G);
      // Every CTA waits for all CTAs' flags of the previous phase, even with no
      // units of its own here: a CTA may never publish phase p's flag while
      // another can still be reading phase p - 2's flags from the same slot.
      float sumsq = 0.f;
      if (p > 0) {
        // one warp polls every CTA's flag, the CTA barrier releases the others
        if (warp == 0) {
          const float v = wait_phase_flags(a.flags + ((p - 1) & 1) * kMaxGrid, tag0 + (p - 1), lane,
                                           a.wait_limit, a.ctl);
          if (lane == 0) red_cta[0] = v;
        }
        named_bar_sync(1, kTcConsumers);
        sumsq = red_cta[0];
      }
      if (u0 < units || (ph.x_dbg && cta == 0)) {
        if (p == 0 && ph.x_kind == X_NORM32) sumsq = sum_ss_array(ph.ss_in, lane);   // from an earlier launch
        if (ph.x_kind == X_NORM16) sumsq = input_sumsq16(ph, lane);
        tc_form_x(ph, xf, sumsq, tid, ph.x_dbg != nullptr && cta == 0);
        named_bar_sync(1, kTcConsumers);   // xf complete before any warp reads it
      }
      int n_buf = 0, u_first = u0;
      float ss = 0.f;
      for (int u = u0; u < units; u += G) {
        if (n_buf == kTcRedUnits) {
          ss += tc_flush(ph, red, n_buf, u_first, G, tid, true);
          n_buf = 0;
          u_first = u;
        }
        float acc0 = 0.f, acc1 = 0.f;
        for (int c = 0; c < chunks; ++c) {
          const int stage = it % kTcStages;
          const uint32_t n = it / kTcStages;
          // After a failed wait the CTA keeps walking its units without
          // waiting so that every barrier is still reached; the launch then
          // reports the failure in its status.
          if (!abort_flag && !mbar_wait_bounded(&full_bar[stage], n & 1, a.wait_limit)) {
            tc_set_status(a.ctl, ST_FULL_TIMEOUT);
            abort_flag = 1;
          }
          const uint8_t* sb = ring + static_cast<size_t>(stage) * kTcStageBytes;
          const uint8_t* rg = sb + g * kTcPitch;
          const uint8_t* rh = sb + (g + 8) * kTcPitch;
          const int nblk = min(kTcChunk, nb - c * kTcChunk);
#pragma unroll
          for (int i = 0; i < kTcChunk / kTcWarps; ++i) {
            const int b = warp + kTcWarps * i;   // block within the chunk (parity = warp parity)
            if (b < nblk) {
              const uint4 xv = xf[(c * kTcChunk + b) * 4 + t];
              uint32_t gl02, gl13, gh02, gh13, hl02, hl13, hh02, hh13;
              unpack_word(code_word(rg, b, t), magic, gl02, gl13, gh02, gh13);
              unpack_word(code_word(rh, b, t), magic, hl02, hl13, hh02, hh13);
              const float dg = row_scale(rg, b), dh = row_scale(rh, b);
              float cb[4] = {0.f, 0.f, 0.f, 0.f};
              mma16816(cb, gl02, hl02, gl13, hl13, xv.x, xv.y);
              mma16816(cb, gh02, hh02, gh13, hh13, xv.z, xv.w);
              acc0 = fmaf(dg, cb[0], acc0);
              acc1 = fmaf(dh, cb[2], acc1);
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty_bar[stage]);
          ++it;
        }
        // lanes (g, 0) hold the sums of tile rows g and g + 8
        if (t == 0) {
          float* pr = red + (n_buf * kTcWarps + warp) * 16;
          pr[g] = acc0;
          pr[g + 8] = acc1;
        }
        ++n_buf;
      }
      ss += tc_flush(ph, red, n_buf, u_first, G, tid, false);
      // phase end: publish this CTA's flag (its outputs are written; the sum of
      // squares of its residual sums rides along for the next RMSNorm)
      const bool resid = ph.epi_kind == EPI_RESID && ph.ss_out != nullptr;
      if (p + 1 < a.n_phases || resid) {
        ss = warp_sum(ss);
        if (lane == 0) red_cta[warp] = ss;
        named_bar_sync(1, kTcConsumers);
        if (tid == 0) {
          float tot = 0.f;
          for (int w = 0; w < kTcWarps; ++w) tot += red_cta[w];
          if (resid) ph.ss_out[cta] = tot;
          if (p + 1 < a.n_phases) {
            const unsigned long long f =
                (static_cast<unsigned long long>(tag0 + p) << 32) | __float_as_uint(tot);
            st_release_u64(a.flags + (p & 1) * kMaxGrid + cta, f);
          }
        }
        named_bar_sync(1, kTcConsumers);   // red_cta is read again at the next phase start
      }
    }
  }

  __syncthreads();
  if (a.n_phases > 1 && tid == 0) {
    // The last CTA to leave advances the epoch (so the next launch's tags are
    // new) and resets the departure count.
    __threadfence();
    const unsigned long long left = atomicAdd(&a.ctl->depart, 1ull);
    if (left == static_cast<unsigned long long>(G) - 1) {
      a.ctl->depart = 0ull;
      atomicAdd(&a.ctl->epoch, 1u);
    }
  }
}

cudaError_t tc_engine_prepare() {
  return cudaFuncSetAttribute(tc_engine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
}

cudaError_t tc_engine_launch(const EngineArgs& a, int grid, bool cooperative, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = kTcSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = cooperative ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tc_engine_kernel, a);
}

cudaError_t tc_engine_read_status(int* out) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_status_tc, sizeof(int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_status_tc, &zero, sizeof(int));
}

}  // namespace q4
