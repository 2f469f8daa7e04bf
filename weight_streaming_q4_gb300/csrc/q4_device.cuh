// Device-side building blocks for the Q4_0 decode kernels (sm_103a):
// the phase descriptor shared by host and device, and thin inline-PTX
// wrappers for mbarriers, 1-D bulk TMA copies and bounded waits.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace q4 {

constexpr int kQK = 32;              // weights per Q4_0 block
constexpr int kBlockBytes = 18;      // binary16 scale + 16 code bytes
constexpr int kConsumerWarps = 15;   // warps doing the arithmetic (4 warps per SM sub-partition
                                     // with the producer, so up to 128 registers per thread)
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kThreads = kConsumerThreads + 32;   // + one producer warp
constexpr int kKT = 64;              // input columns each consumer thread keeps in registers
constexpr int kStageBytes = 32256;   // one work unit of weights in shared memory
constexpr int kStages = 6;           // ring depth (6 * 31.5 KB = 189 KB)
constexpr int kRedFloats = 6144;     // per-warp row partials buffered until the phase ends
// Tagged programs stage a phase input per CTA in dynamic shared memory after
// the ring (the buffer also holds the row partials): up to kNormMaxValues fp32
// RMSNorm inputs or kTag16MaxValues binary16 inputs.  The ring then has 6
// stages when the buffer takes at most kXBufMaxBytes6, else 5.
constexpr int kNormMaxValues = 8192;
constexpr int kTag16MaxValues = 28672;
constexpr int kXBufMaxBytes6 = 37888;     // 6 * 32256 + 37888 = 231424 bytes
constexpr int kXBufMaxBytes5 = 70144;     // 5 * 32256 + 70144 = 231424 bytes
constexpr int kDynSmemMax = 231424;
constexpr int kMaxGrid = 256;        // CTAs (one per SM) a launch may use
constexpr int kMaxBatch = 16;

// How the input vector x of a phase is formed (per batch row).
enum XKind : int {
  X_F16 = 0,      // x = src (binary16 [batch][k])
  X_NORM16 = 1,   // x = f16(t * rsqrt(mean(t^2) + eps)), t = src (binary16 [batch][k])
  X_ATTN = 2,     // context-1 attention: x[i] = f16(v[(i/hd)/group*hd + i%hd]), v = fp32 src
  X_NORM32 = 3,   // as X_NORM16 with an fp32 src
  // Tagged inputs (see TaggedWords): src holds one tagged word per value.
  X_TAG16 = 4,       // x = the binary16 values of 32-bit words, k of them
  X_TAG16_ATTN = 5,  // as X_ATTN over xt_n tagged binary16 values of v
  X_TAG32_NORM = 6,  // as X_NORM32 over k tagged fp32 values (64-bit words)
};

// How a CTA takes part in the one flag exchange of a tagged layer program.
enum SyncKind : int {
  SYNC_NONE = 0,
  SYNC_PUBLISH = 1,   // after its input is read, every CTA publishes the phase tag as its flag
  SYNC_WAIT = 2,      // before writing anything, a CTA waits until every flag carries the
                      // previous phase's tag (or a later one)
};

// Tagged words.  Inside a tagged layer program a value that one CTA hands to
// another travels with the tag of the phase that produced it in one aligned
// word: a binary16 value in the low half of a 32-bit word under the low 16
// bits of the tag, or an fp32 value in the low half of a 64-bit word under the
// 32-bit tag.  Aligned 32- and 64-bit accesses are single-copy atomic, so a
// reader that sees the tag it expects also sees the value stored with it;
// readers poll the words they need until every tag matches.

// What the epilogue does with the row sums.
enum EpiKind : int {
  EPI_F32 = 0,    // y[b][n] = sum
  EPI_RESID = 1,  // y[b][n] = sum; y2[b][n] = res[b][n] + sum (fp32 residual sum)
  EPI_SILU = 2,   // two matrices: y = g, y2 = u, act[b][n] = f16(silu(g) * u)
};

// One phase = one matrix-vector product over a row-major Q4_0 matrix
// (or two matrices with the same shape for EPI_SILU), with its input
// prologue and output epilogue.  Plain data, identical on host and device.
struct Phase {
  const uint8_t* w0;      // Q4_0 matrix [n_rows][k / 32] blocks
  const uint8_t* w1;      // second matrix (EPI_SILU only)
  const void* x_src;      // input per XKind
  float* y;               // fp32 [batch][n_rows]
  float* y2;              // fp32 [batch][n_rows]: EPI_SILU u, EPI_RESID the residual sum
  const uint16_t* res;    // EPI_RESID: residual input binary16 [batch][n_rows]
  uint16_t* aux16;        // EPI_SILU: act binary16 [batch][n_rows]
  float* ss_out;          // EPI_RESID: per-CTA sums of squares of y2 ([kMaxGrid] floats)
  const float* ss_in;     // X_NORM32 in a launch's first phase: the producing phase's ss_out
  uint16_t* x_dbg;        // if not null, CTA 0 stores the formed x here (binary16 [batch][k])
  int n_rows;
  int k;
  int x_kind;
  int epi_kind;
  int x_ld;               // row stride (elements) of x_src per batch row; with x_t, the
                          // chunk stride T of the transposed layout
  int attn_off;           // X_ATTN: element offset of v inside a row of x_src
  int head_dim;           // X_ATTN
  int group;              // X_ATTN: query heads per value head
  float eps;              // X_RMSNORM
  int teams;              // row teams of k/64 threads working side by side
  int units;              // work units in this phase
  int rows_per_unit;      // rows of each matrix per unit
  int x_t;                // 1: x_src is slice-transposed (see below), stride x_ld chunks
  // Slice-transposed copy written by the epilogue for the next phase's input
  // (CUDA-core engine): rows [yt_off, yt_off + yt_n) of the output (y for
  // EPI_F32, y2 for EPI_RESID, the SiLU product for EPI_SILU).  Element e of
  // that range sits where consumer thread e / 64 reads it with coalesced
  // 16-byte loads: fp32 at ((e % 64) / 4 * T + e / 64) * 4 + e % 4, binary16 at
  // ((e % 64) / 8 * T + e / 64) * 8 + e % 8, with T = yt_n / 64.
  void* yt;
  int yt_off;
  int yt_n;
  // Units of all earlier phases of the whole program: unit u of this phase
  // goes to CTA (base + u) mod G, the same in a fused, per-layer or
  // per-phase launch, so every schedule gives bit-identical results.
  int base;
  int pad_;
  // Tagged programs only.
  const uint32_t* res_t;  // EPI_RESID: tagged binary16 residual input [n_rows]
  uint32_t* xr_out;       // if not null, CTA 0 stores the formed x here as tagged binary16 [k]
  int gidx;               // index of the phase in the whole program (its tag offset)
  int sync;               // SyncKind
  int xt_n;               // X_TAG16_ATTN: tagged values of v in x_src
  int row_rot;            // tensor-core engine: unit u covers rows from (u * rows_per_unit +
                          // row_rot) mod n_rows (row_rot and n_rows multiples of the unit)
  // Tensor-core engine only: TMA descriptors of w0 and w1 (2-D, 64-bit elements:
  // columns = row bytes / 8, rows = n_rows; box = tc_pitch(k) / 8 columns by
  // the unit's rows), encoded on the host.
  CUtensorMap tm0;
  CUtensorMap tm1;
};

// Geometry of the tensor-core engine for rows of width k (k % 256 == 0 and
// either k <= 2048 or k % 2048 == 0): a stage holds one column chunk of a
// 32-row unit; a chunk is 64 blocks (the whole row when k <= 2048).  Staged
// rows of wide matrices are 1168 bytes apart, 16 more than the chunk, so that
// the 32-bit code-word loads of the 8 row groups of a tile fall in different
// banks (the copy box reads 16 bytes of the next chunk, or zero-fills past the
// row end); a row of at most 2048 columns is staged whole, unpadded.
__host__ __device__ __forceinline__ int tc_chunk_blocks(int k) { return k <= 2048 ? k / 32 : 64; }
__host__ __device__ __forceinline__ int tc_pitch(int k) { return k <= 2048 ? (k / 32) * 18 : 64 * 18 + 16; }
__host__ __device__ __forceinline__ int tc_chunks(int k) { return (k / 32) / tc_chunk_blocks(k); }
constexpr int kTcUnitRows = 32;   // rows of a unit (16 rows of each matrix of a gate|up pair)
constexpr int kTcMaxK = 30720;    // widest row the engine's input buffer takes

__host__ __device__ __forceinline__ int slice_t32(int e, int T) { return ((e & 63) >> 2) * T * 4 + (e >> 6) * 4 + (e & 3); }
__host__ __device__ __forceinline__ int slice_t16(int e, int T) { return ((e & 63) >> 3) * T * 8 + (e >> 6) * 8 + (e & 7); }

// Per-launch control block in device memory (decoder workspace).
struct Control {
  unsigned long long depart;    // CTAs that left the current launch (reset by the last one)
  unsigned int epoch;           // launches (tagged programs: whole programs) completed; the
                                // phase tags derive from it
  int status;                   // bit flags set by kernels on a failed wait
};

// A CTA's end-of-phase flag: its sum of squares of the residual sums it wrote
// (0 for other phases) in the low word, the phase tag in the high word.
// flags[(p & 1) * kMaxGrid + cta] holds phase p's flag of CTA cta.  Tagged
// programs use flags[cta] alone, with a zero low word.
constexpr unsigned kPhasesPerEpoch = 4096;

// ------------------------------------------------------------------ batched engine
//
// The persistent tensor-core engine for batches of 2..8 rows (q4_bt_engine.cu).
// The batch is the n dimension of the instruction (8 columns), so an input is
// 8 x k binary16 values: too many to keep a whole phase input in shared memory
// next to the ring.  Instead every phase input lives in global memory as
// fragments (column b of the instruction = batch row b, k in the order the
// code unpacking delivers it) and each ring stage carries the chunk of
// fragments its weights need, copied with one bulk copy.  The phases meet at a
// flag barrier (all CTAs), and each RMSNorm is its own small phase (BT_FORM):
// every CTA normalises rows' values into the next fragments (after a residual
// phase the rows it produced there; the first one a slice of the caller's).
enum BtKind : int {
  BT_PLAIN = 0,   // y = W x; optionally rows [g_lo, g_lo + g_n) gathered per head (context-1 attention)
  BT_RESID = 1,   // y = W x; y2 = t = res + y (fp32); sums of squares of t per CTA and batch row
  BT_SILU = 2,    // gate|up pair: y = g, y2 = u, act = f16(silu(g) * u)
  BT_FORM = 3,    // z = f16(t * rsqrt(mean(t^2) + eps)) for every batch row (no weights)
};
constexpr int kBtCols = 8;            // batch columns (one n-tile of the instruction)

// Fragment buffers hold `cols` columns (the batch rounded up to 2, 4 or 8;
// the instruction's other columns are zero): 64 * cols bytes per 32-value
// block.  Byte offset of value e of batch row b: block e / 32, lane
// (b, (e % 16) / 4), bytes 0-7 for e % 32 < 16 else 8-15, halves in the order
// 4t, 4t+2, 4t+1, 4t+3.
__host__ __device__ __forceinline__ int bt_cols(int batch) { return batch <= 2 ? 2 : batch <= 4 ? 4 : 8; }
__host__ __device__ __forceinline__ uint32_t bt_frag_off(int b, int e, int cols) {
  const int i = e & 31, j = e & 3;
  return static_cast<uint32_t>((e >> 5) * 64 * cols + (b * 4 + ((i & 15) >> 2)) * 16 + ((i >> 4) << 3) +
                               (((j & 1) << 1) | (j >> 1)) * 2);
}

struct BtPhase {
  CUtensorMap tm0;          // unit phases: the weights (descriptors as the batch-1 tensor-core engine's)
  CUtensorMap tm1;          // BT_SILU: up
  const uint8_t* x_frag;    // unit phases: input fragments, k * 16 bytes
  float* y;                 // fp32 [batch][n_rows] (BT_SILU: g)
  float* y2;                // BT_SILU: u; BT_RESID: t
  const uint16_t* res;      // BT_RESID: binary16 [batch][n_rows]
  uint16_t* out16;          // binary16 natural output: BT_PLAIN the gathered heads, BT_SILU act, BT_FORM z
  uint8_t* out_frag;        // the same values as fragments (the next phase's input)
  const float* src32;       // BT_FORM: fp32 t [batch][k], its sums of squares in ss
  const uint16_t* src16;    // BT_FORM: binary16 [batch][k] (sums of squares taken from it)
  float* ss;                // BT_RESID: out, BT_FORM: in; [grid][kBtCols]
  int kind;
  int gidx;                 // index of the phase in the whole program (its tag offset)
  int k;                    // unit phases: row width; BT_FORM: values per batch row
  int n_rows;
  int units;
  int base;                 // units of earlier phases: unit u goes to CTA (base + u) mod G
  int out_ld;               // BT_PLAIN: row stride of out16
  int g_lo, g_n, head_dim, group;
  float eps;
  int row_rot;              // unit u covers rows from (u * 32 + row_rot) mod n_rows (multiples of 32)
  int early_units;          // BT_PLAIN: units [0, early_units) hold the gathered rows; a CTA
                            // publishes the phase once its units among them are stored (0: at the end)
};

struct BtArgs {
  const BtPhase* phases;    // device array
  int n_phases;
  Control* ctl;
  unsigned long long* flags;   // [kMaxGrid] per-CTA flags, the phase tag in the high word
  uint32_t wait_limit;
  uint32_t stage_bytes;     // bytes between ring stages
  uint32_t x_off;           // offset of the fragment chunk inside a stage
  int stages;
  int batch;
  int cols;                 // bt_cols(batch): columns of the fragment buffers
  int end_of_program;       // the last CTA to leave advances the epoch
  uint32_t stall;           // failure-detection hook: added to every awaited flag tag (0 normally;
                            // kPhasesPerEpoch: a tag no CTA publishes, so every such wait runs out)
};

cudaError_t bt_engine_prepare();
// Ring geometry for phases of widths ks (each tc_chunk_blocks-compatible) and
// fragment buffers of `cols` columns: false if it does not fit.
bool bt_geom(const int* ks, int n, int cols, int* stages, uint32_t* stage_bytes, uint32_t* x_off);
cudaError_t bt_engine_launch(const BtArgs& a, int grid, cudaStream_t stream);
// Timeline of the batched engine's phases (libq4_tl.so only), laid out as
// tc_timeline_read's.
cudaError_t bt_timeline_read(unsigned long long* out, size_t n, bool clear);

// Arguments of one launch of the engine kernel: either a device array of
// phases or a single phase passed by value.
struct EngineArgs {
  const Phase* phases;     // device array, or null to run `one`
  int n_phases;
  Control* ctl;            // required when n_phases > 1
  unsigned long long* flags;  // [2][kMaxGrid] end-of-phase flags, required when n_phases > 1
  uint32_t wait_limit;     // polls of one wait before it is declared failed
  uint32_t stage_bytes;    // tensor-core engine: bytes between ring stages (32 rows of the
                           // widest pitch of the launch's phases)
  int tagged;              // CUDA-core engine: the phases exchange tagged words (phase tag =
                           // epoch * kPhasesPerEpoch + 1 + Phase::gidx) instead of meeting at
                           // a flag barrier after every phase
  int end_of_program;      // tagged: this launch runs the program's last phase, so the last
                           // CTA to leave advances the epoch
  int stages;              // tagged (and tensor-core engine): ring depth
  int xbuf_floats;         // tagged: floats of the staging buffer after the ring (tensor-core
                           // engine: of the fragment-order input buffer)
  int pdl;                 // tensor-core engine, programmatic dependent launch: bit 0 = this launch
                           // may start before the kernel ahead of it ends (the producer streams
                           // weights at once; the other warps wait for that kernel before they
                           // touch any data); bit 1 = let the next such launch start early
  Phase one;
};

enum StatusBits : int {
  ST_FLAG_TIMEOUT = 1,
  ST_FULL_TIMEOUT = 2,
  ST_EMPTY_TIMEOUT = 4,
  ST_DRAIN_TIMEOUT = 8,
  ST_DATA_TIMEOUT = 16,    // a tagged input word never carried the expected tag
  ST_KV_POS = 32,          // a KV decoder's position was outside 0..capacity-1
};

// ------------------------------------------------------------------ PTX

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// One bounded poll: the thread may be suspended in hardware until the phase
// completes or about kWaitHintNs nanoseconds pass, so a waiting warp takes no
// issue slots from the warps that compute.
constexpr uint32_t kWaitHintNs = 1000;

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "n"(kWaitHintNs)
      : "memory");
  return ok != 0;
}

// Non-blocking test of the given phase parity.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the given phase parity of an mbarrier, giving up after
// `limit` polls (each poll may suspend the thread for a short while).  A
// phase that has already completed is seen by one non-blocking test.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint32_t limit) {
  if (mbar_test_wait(bar, parity)) return true;
  for (uint32_t i = 0; i < limit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (i > 64) __nanosleep(64);
  }
  return false;
}

// 1-D bulk copy global -> shared, completion counted on an mbarrier.
// src, dst 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// 2-D tensor copy global -> shared of the box at column x (64-bit elements, x
// even so that the box starts 16-byte aligned) and row y of the tensor map,
// completion counted on an mbarrier.  Out-of-range rows and columns are
// filled with zeros (and still counted).
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Acquire a TMA descriptor that lives in global memory for the tensor-map proxy.
__device__ __forceinline__ void tensormap_acquire(const CUtensorMap* map) {
  asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(map) : "memory");
}

// Ask for `bytes` at src to be brought into L2 (no completion tracking).
// src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Relaxed (morally strong, gpu scope) accesses of tagged words.  A vector
// access is four independent 32-bit accesses, each single-copy atomic.
__device__ __forceinline__ uint4 ld_relaxed_v4(const void* p) {
  uint4 v;
  asm volatile("ld.relaxed.gpu.global.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

// As ld_relaxed_v4 without the compiler memory barrier (other memory
// accesses may move across it; the load itself is kept and not merged).
__device__ __forceinline__ uint4 ld_relaxed_v4_nb(const void* p) {
  uint4 v;
  asm volatile("ld.relaxed.gpu.global.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t ld_relaxed_b32(const void* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed_b32(void* p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void st_relaxed_b64(void* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void st_relaxed_v4(void* p, uint4 v) {
  asm volatile("st.relaxed.gpu.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// Packed fp32x2 arithmetic (sm_100 family).
__device__ __forceinline__ float2 f2_add(float2 a, float2 b) {
  unsigned long long ra = *reinterpret_cast<unsigned long long*>(&a);
  unsigned long long rb = *reinterpret_cast<unsigned long long*>(&b);
  unsigned long long rd;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(rd) : "l"(ra), "l"(rb));
  return *reinterpret_cast<float2*>(&rd);
}

__device__ __forceinline__ float2 f2_fma(float2 a, float2 b, float2 c) {
  unsigned long long ra = *reinterpret_cast<unsigned long long*>(&a);
  unsigned long long rb = *reinterpret_cast<unsigned long long*>(&b);
  unsigned long long rc = *reinterpret_cast<unsigned long long*>(&c);
  unsigned long long rd;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(rd) : "l"(ra), "l"(rb), "l"(rc));
  return *reinterpret_cast<float2*>(&rd);
}

// Host-side launchers (q4_engine.cu, q4_aux.cu).
cudaError_t engine_prepare();
cudaError_t engine_launch(const EngineArgs& a, int grid, bool cooperative, cudaStream_t stream);
cudaError_t engine_occupancy(int* blocks_per_sm);
cudaError_t engine_read_status(int* out);
cudaError_t simple_launch(const uint8_t* w, const uint16_t* x, float* y, int n, int k, int batch,
                          cudaStream_t stream);
cudaError_t dequant_launch(const uint8_t* w, float* out, int n, int k, cudaStream_t stream);
cudaError_t poison_launch(uint8_t* buf, size_t n_blocks, cudaStream_t stream);
cudaError_t stamp_launch(unsigned long long* out, cudaStream_t stream);
cudaError_t attn_prepare();
size_t attn_workspace_bytes(int n_q, int n_kv, int hd, int capacity);
// The cluster attention kernel (q4_attn_cluster.cu): prepare decides whether
// the GPU schedules clusters of 16 CTAs per value head (else 8).
cudaError_t attn_cluster_prepare();
// ctx_add: the positions in use are *ctx_len + ctx_add (the decoder passes its
// position counter and 1).  With `app`, the kernel also stores the token's key
// and value (fp32 app->k, app->v) as binary16 in row *app->pos of the caches
// (which must be row ctx - 1) and attends to them; *pos outside the bucket sets
// ST_KV_POS in *app->status.
struct AttnAppend {
  const float* k;
  const float* v;
  const int* pos;
  int* status;
  int pdl;   // launch as a programmatic dependent of the kernel that wrote q, k and v (the
             // cached rows of the first round are copied while that kernel finishes)
};
cudaError_t attn_launch(const float* q, const uint16_t* k, const uint16_t* v, const int* ctx_len, int capacity,
                        int n_q, int n_kv, int hd, uint16_t* out, void* ws, cudaStream_t s, int ctx_add = 0,
                        const AttnAppend* app = nullptr);
cudaError_t attn_cluster_launch(const float* q, const uint16_t* k, const uint16_t* v, const int* ctx_len, int ctx_add,
                                int capacity, int n_q, int n_kv, int hd, uint16_t* out, const AttnAppend* app,
                                cudaStream_t s);
cudaError_t pos_advance_launch(int* pos, cudaStream_t s);
// status (nullable): ST_KV_POS is or-ed in when *pos is outside 0..capacity-1.
cudaError_t kv_append_launch(const float* k, const float* v, uint16_t* kc, uint16_t* vc, const int* pos, int capacity,
                             int kv_dim, cudaStream_t s, int* status = nullptr);
// One-shot batch-1 product (q4_oneshot.cu): 16-row tiles, one CTA each.
constexpr int kOsSmemMax = 231424;   // dynamic bytes; with the static ones within the 227 KB a CTA may use
bool oneshot_ok(int n, int k);
size_t oneshot_smem_bytes(int k);
cudaError_t oneshot_prepare();
// chain: the launch may start before the kernel ahead of it on the stream
// ends (Q4_GEMV_CHAIN's contract), unless w or x overlap the y of a one-shot
// product on the stream that may still be running.
cudaError_t oneshot_launch(const uint8_t* w, const uint16_t* x, float* y, int n, int k, uint32_t wait_limit,
                           bool chain, cudaStream_t stream);
cudaError_t oneshot_read_status(int* out);
// A product of another kernel was launched on `stream`: the next one-shot
// product there does not start early.
void oneshot_chain_break(cudaStream_t stream);
// Timeline of the tensor-core engine's phases (libq4_tl.so only): per CTA,
// phase and event the global timer; n >= 256 * 64 * 6 values.
cudaError_t tc_timeline_read(unsigned long long* out, size_t n, bool clear);
cudaError_t tc_engine_prepare();
// With a.pdl bit 0 the launch carries programmatic stream serialisation (and
// must not be cooperative).
cudaError_t tc_engine_launch(const EngineArgs& a, int grid, bool cooperative, cudaStream_t stream);
cudaError_t tc_engine_read_status(int* out);
cudaError_t tc_engine_occupancy(int* blocks_per_sm);
// Dynamic shared memory of a tensor-core launch, and the largest allowed.
size_t tc_smem_bytes(int stages, uint32_t stage_bytes, int xbuf_floats);
constexpr size_t kTcSmemLimit = 231424;
cudaError_t mma_prepare();
// y2/split: rows from `split` on go to y2 ([batch][n - split]); rows before to y ([batch][split]).
// Rows [lo, lo + n_rows) of a product's output taken as value heads of head_dim
// rows each and also written, rounded to binary16, as the context-1 attention
// output: value row lo + vh * head_dim + i goes to out[b][(vh * group + h) *
// head_dim + i] for h < group (out has ld values per batch row).
struct MmaGather {
  uint16_t* out;
  int lo, n_rows, head_dim, group, ld;
};

// pdl: launch with programmatic stream serialisation (the weight copies start
// while the previous kernel of the stream finishes; x is read after it).
// gather: optional second output of some rows (see MmaGather).
// act: gate|up pairing.  The n rows are two matrices of n/2 rows (split =
// n/2, y2 given); each 16-row tile takes 8 rows of the first and the same 8
// rows of the second, and the epilogue also writes act = f16(silu(y) * y2).
cudaError_t mma_launch(const uint8_t* w, const uint16_t* x, float* y, int n, int k, int batch, int grid,
                       uint32_t wait_limit, int* status, cudaStream_t stream, float* y2 = nullptr, int split = 0,
                       bool pdl = false, const MmaGather* gather = nullptr, uint16_t* act = nullptr);
cudaError_t mma_read_status(int* out);
// Host: the TMA descriptor of a row-major Q4_0 matrix (n_rows x k; 64-bit
// elements, box tc_pitch(k) / 8 columns by box_rows rows); false if the
// driver cannot encode it.
bool encode_q4_rows(CUtensorMap* m, const uint8_t* w, int n_rows, int k, int box_rows);
// Glue launches; pdl as for mma_launch (each glue kernel waits for its inputs first).
cudaError_t glue_norm(const uint16_t* src16, const float* src32, int batch, int dim, float eps, uint16_t* z,
                      cudaStream_t s, bool pdl = false);
cudaError_t glue_resid_norm(const uint16_t* z, const float* o, int batch, int dim, float eps, float* t,
                            uint16_t* z_out, cudaStream_t s, bool pdl = false);

}  // namespace q4

struct q4_layer_shape;
namespace q4 {
// Host helper (q4_api.cu): keep a CUDA error for q4_last_cuda_error(); returns Q4_ERR_CUDA.
int record_cuda_error(cudaError_t e);
// Host helper (q4_api.cu): one eager run of a layer stack inside a given workspace.
int run_stack_in_workspace(const q4_layer_shape* shape, const void* const* layer_weights, int n_layers,
                           uint16_t* hidden_io, void* ws, size_t ws_bytes, cudaStream_t s);

}  // namespace q4
