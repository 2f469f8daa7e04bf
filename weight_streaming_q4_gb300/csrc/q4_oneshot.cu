// One-shot batch-1 Q4_0 matrix-vector product on the tensor cores: the
// launch path for a single product (q4_gemv), without the persistent
// engine's ring, warp roles or phase program.
//
// Each CTA takes a tile of 16 rows over the full width k.  As soon as the CTA
// starts, one thread puts all of the tile's bytes in flight: where the rows
// are whole 2048-column chunks (at least two), one 2-D tensor copy per chunk,
// each counted on its own mbarrier, the rows of a chunk landing at a padded
// 1168-byte pitch; otherwise every row as two 1-D bulk copies (its two
// halves, on two mbarriers) at a pitch of row bytes + 16.  Either padding puts
// the code-word loads of the 8 row groups in different banks.
// Meanwhile the 256 threads stage x in fragment order.  The 8 warps split the
// width: warp w takes block pairs [w * pp, (w + 1) * pp) and runs the exact
// binary16 (q - 8) unpack and mma.sync m16n8k16 of the persistent engine on
// them (q4_frag.cuh), waiting only for the chunks (or half) of the row its
// pairs lie in.
// The warps' partial sums meet in shared memory and are added in warp order
// (a fixed order: the result does not depend on timing).
//
// A chained call (Q4_GEMV_CHAIN) is launched with programmatic stream
// serialisation: it lets the next kernel of the stream start at once, and
// each CTA fetches its weights, stages x and computes before it waits for the
// kernel before it (griddepcontrol.wait) and stores y, so back-to-back
// products overlap almost entirely.  The caller vouches that nothing it
// enqueued since the last product writes w or x; the launcher itself starts a
// call early only when its w and x do not overlap the y of any one-shot
// product on the same stream that may still be running.  Any other call
// starts after its predecessor as usual (its wait then returns at once).
//
// The method: PIPO's dequantisation-free 4-bit matrix-vector product
// ("PIPO: Pipelined Offloading for Efficient Inference on Consumer Devices",
// Method, "Computation optimization").
#include <cuda_fp16.h>
#include <stdint.h>

#include <mutex>

#include "q4_device.cuh"
#include "q4_frag.cuh"

namespace q4 {

namespace {

constexpr int kOsWarps = 8;
constexpr int kOsThreads = kOsWarps * 32;
constexpr int kOsRows = 16;
// Rows of whole 2048-column chunks, more than one: the tile is staged chunk by
// chunk, each chunk one 2-D tensor copy of 16 rows at a padded 1168-byte
// pitch (the copy's box: 146 64-bit columns, the last 16 bytes of a row
// belonging to the next chunk or read as zeros past the row's end).
constexpr int kOsChunkPitch = 64 * kBlockBytes + 16;
constexpr int kOsChunkBytes = kOsRows * kOsChunkPitch;
constexpr int kOsMaxChunks = 12;

struct OsArgs {
  CUtensorMap tm;     // TM: the weights' descriptor (box 146 64-bit columns by 16 rows)
  const uint8_t* w;
  const __half* x;
  float* y;
  int n, k;
  uint32_t wait_limit;
};

__device__ int g_status_os;   // status bits (a copy that never landed)

// x (binary16, k values) into the fragment-order buffer: lane quarter t of
// block b holds x[32b + 4t + {0, 2, 1, 3}] and the same 16 further on.
__device__ __forceinline__ void os_stage_x(const __half* x, uint8_t* xf, int k, int tid) {
  for (int i = tid; i < (k >> 2); i += kOsThreads) {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(x) + i);
    const int e = 4 * i, b = e >> 5, j = e & 31;
    const int off = ((b << 2) + ((j & 15) >> 2)) * 16 + ((j >> 4) << 3);
    *reinterpret_cast<uint2*>(xf + off) = make_uint2(__byte_perm(u.x, u.y, 0x5410), __byte_perm(u.x, u.y, 0x7632));
  }
}

}  // namespace

template <bool TM>
__global__ void __launch_bounds__(kOsThreads, 2) oneshot_kernel(const __grid_constant__ OsArgs a) {
  extern __shared__ __align__(128) uint8_t sm[];
  __shared__ __align__(8) uint64_t bar[TM ? kOsMaxChunks : 2];
  const uint8_t* __restrict__ w = a.w;
  const __half* x = a.x;
  float* y = a.y;
  const int n = a.n, k = a.k;
  const uint32_t wait_limit = a.wait_limit;
  const int chunks = TM ? k >> 11 : 2;   // TM: 2048-column chunks; else the two halves of each row
  __shared__ float part[kOsWarps][kOsRows];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row_bytes = (k >> 5) * kBlockBytes, half = row_bytes >> 1, pitch = row_bytes + 16;
  const int n0 = blockIdx.x * kOsRows;
  const int rows = n - n0 < kOsRows ? n - n0 : kOsRows;
  uint8_t* xf = sm;                          // k * 2 bytes, fragment order
  uint8_t* tile = sm + 2 * k;                // 16 rows at `pitch` (TM: chunk by chunk)

  griddep_launch_dependents();
  // Everything but the store of y runs before the wait for the kernel before
  // this one: the only kernel that lets a successor start early is this one,
  // it writes nothing but its y, and the launcher starts this kernel early
  // only when w and x do not overlap that y.
  if (tid == 0) {
    for (int c = 0; c < chunks; ++c) mbar_init(&bar[c], 1);
    fence_mbar_init();
    if (TM) {
      // rows past n read as zeros and count in full
      for (int c = 0; c < chunks; ++c) {
        mbar_arrive_expect_tx(&bar[c], kOsChunkBytes);
        tma_load_2d(tile + c * kOsChunkBytes, &a.tm, c * (64 * kBlockBytes / 8), n0, &bar[c]);
      }
    } else {
      mbar_arrive_expect_tx(&bar[0], static_cast<uint32_t>(rows) * half);
      mbar_arrive_expect_tx(&bar[1], static_cast<uint32_t>(rows) * half);
      for (int r = 0; r < rows; ++r) {
        const uint8_t* src = w + static_cast<size_t>(n0 + r) * row_bytes;
        bulk_g2s(tile + r * pitch, src, half, &bar[0]);
        bulk_g2s(tile + r * pitch + half, src + half, half, &bar[1]);
      }
    }
  }
  os_stage_x(x, xf, k, tid);
  __syncthreads();

  // warp w: block pairs [p0, p1); rows of the tile beyond n hold stale bytes
  // and their outputs are not stored (each output row reads only its own row)
  const int pairs = k >> 6;
  const int pp = (pairs + kOsWarps - 1) / kOsWarps;
  const int p0 = warp * pp, p1 = p0 + pp < pairs ? p0 + pp : pairs;
  const int g = lane >> 2, t = lane & 3;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  bool ok = true;
  if (p0 < p1) {
    if (TM) {
      for (int c = p0 >> 5; c <= (p1 - 1) >> 5; ++c) ok &= mbar_wait_bounded(&bar[c], 0, wait_limit);
    } else {
      if (2 * p0 < pairs) ok &= mbar_wait_bounded(&bar[0], 0, wait_limit);
      if (2 * p1 > pairs) ok &= mbar_wait_bounded(&bar[1], 0, wait_limit);
    }
    uint32_t magic;
    asm volatile("mov.b32 %0, 0x64006400;" : "=r"(magic));
    const uint4* xf4 = reinterpret_cast<const uint4*>(xf);
#pragma unroll 2
    for (int p = p0; p < p1; ++p) {
      const uint4 xe = xf4[(2 * p) * 4 + t], xo = xf4[(2 * p + 1) * 4 + t];
      const uint8_t* rg = TM ? tile + (p >> 5) * kOsChunkBytes + g * kOsChunkPitch + 36 * (p & 31)
                             : tile + g * pitch + 36 * p;
      pair_mma(rg, rg + 8 * (TM ? kOsChunkPitch : pitch), t, xe, xo, magic, acc[0], acc[1], acc[2], acc[3]);
    }
  }
  // lane (g, 0) adds the odd blocks of lane (g, 3)
  const float r0 = acc[0] + __shfl_sync(0xffffffffu, acc[2], lane | 3);
  const float r1 = acc[1] + __shfl_sync(0xffffffffu, acc[3], lane | 3);
  if (t == 0) {
    part[warp][g] = r0;
    part[warp][g + 8] = r1;
  }
  if (!ok && lane == 0) atomicOr(&g_status_os, ST_FULL_TIMEOUT);
  __syncthreads();
  griddep_wait();   // y: after the kernel before this one (it may write the same y)
  if (tid < rows) {
    float v = 0.f;
#pragma unroll
    for (int q = 0; q < kOsWarps; ++q) v += part[q][tid];
    y[n0 + tid] = v;
  }
  // no copy may still be in flight into this CTA's shared memory at exit
  if (tid == 0 && !ok) {
    bool drained = true;
    for (int c = 0; c < chunks; ++c) drained &= mbar_wait_bounded(&bar[c], 0, wait_limit);
    if (!drained) atomicOr(&g_status_os, ST_DRAIN_TIMEOUT);
  }
}

// Whether a row of width k is staged chunk by chunk with tensor copies.
bool oneshot_tm(int k) { return k % 2048 == 0 && k / 2048 >= 2 && k / 2048 <= kOsMaxChunks; }

// Shared memory of a CTA for width k: x in fragment order and 16 padded rows
// (chunk by chunk when they are staged with tensor copies).
size_t oneshot_smem_bytes(int k) {
  if (oneshot_tm(k)) return 2 * static_cast<size_t>(k) + static_cast<size_t>(k / 2048) * kOsChunkBytes;
  return 2 * static_cast<size_t>(k) + static_cast<size_t>(kOsRows) * ((k >> 5) * kBlockBytes + 16);
}

bool oneshot_ok(int n, int k) {
  return n >= 1 && k >= 512 && k % 512 == 0 && oneshot_smem_bytes(k) <= static_cast<size_t>(kOsSmemMax);
}

cudaError_t oneshot_prepare() {
  cudaError_t e = cudaFuncSetAttribute(oneshot_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kOsSmemMax);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(oneshot_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kOsSmemMax);
}

namespace {

// Per stream, the y ranges of the one-shot products that may still be running
// when the next one starts early: a launch that starts early may overlap every
// such product before it (each started early in turn), so the chain is kept
// until a launch that waits for its predecessor as usual ends it.  A full
// chain ends too: 64 entries, so that a ring of a few dozen independent
// products runs without a drained launch between them (one every 8 launches
// cost 0.3 us per product on N = K = 4096).
constexpr int kOsChain = 64;
struct Chain {
  cudaStream_t stream;
  int n;
  uintptr_t lo[kOsChain], hi[kOsChain];
};
std::mutex g_chain_mu;
Chain g_chain[16];
int g_chain_n = 0;

bool overlaps(uintptr_t a, size_t na, uintptr_t lo, uintptr_t hi) { return a < hi && lo < a + na; }

}  // namespace

cudaError_t oneshot_launch(const uint8_t* w, const uint16_t* x, float* y, int n, int k, uint32_t wait_limit,
                           bool chain, cudaStream_t stream) {
  if (!oneshot_ok(n, k)) return cudaErrorInvalidValue;
  const uintptr_t wa = reinterpret_cast<uintptr_t>(w), xa = reinterpret_cast<uintptr_t>(x);
  const size_t w_bytes = static_cast<size_t>(n) * (k >> 5) * kBlockBytes, x_bytes = 2 * static_cast<size_t>(k);
  bool early = chain;   // only a chained call may start before the work ahead of it
  {
    std::lock_guard<std::mutex> lock(g_chain_mu);
    int i = 0;
    while (i < g_chain_n && g_chain[i].stream != stream) ++i;
    if (i == g_chain_n) {   // a new stream (or one that replaces a remembered one): no early start
      if (g_chain_n < 16) {
        ++g_chain_n;
      } else {
        i = static_cast<int>(reinterpret_cast<uintptr_t>(stream) % 16);
      }
      early = false;
      g_chain[i].stream = stream;
      g_chain[i].n = 0;
    }
    Chain& c = g_chain[i];
    if (c.n == kOsChain) early = false;
    for (int j = 0; j < c.n && early; ++j)
      if (overlaps(wa, w_bytes, c.lo[j], c.hi[j]) || overlaps(xa, x_bytes, c.lo[j], c.hi[j])) early = false;
    if (!early) c.n = 0;
    c.lo[c.n] = reinterpret_cast<uintptr_t>(y);
    c.hi[c.n] = reinterpret_cast<uintptr_t>(y) + 4 * static_cast<size_t>(n);
    ++c.n;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((n + kOsRows - 1) / kOsRows);
  cfg.blockDim = dim3(kOsThreads);
  cfg.dynamicSmemBytes = oneshot_smem_bytes(k);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = early ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  OsArgs a;
  a.w = w;
  a.x = reinterpret_cast<const __half*>(x);
  a.y = y;
  a.n = n;
  a.k = k;
  a.wait_limit = wait_limit;
  if (oneshot_tm(k) && encode_q4_rows(&a.tm, w, n, k, kOsRows)) return cudaLaunchKernelEx(&cfg, oneshot_kernel<true>, a);
  return cudaLaunchKernelEx(&cfg, oneshot_kernel<false>, a);
}

// Another kernel of the library's products was launched on the stream: the
// next one-shot product on it starts after it as usual (the list only knows
// one-shot products' outputs).
void oneshot_chain_break(cudaStream_t stream) {
  std::lock_guard<std::mutex> lock(g_chain_mu);
  for (int i = 0; i < g_chain_n; ++i)
    if (g_chain[i].stream == stream) {
      g_chain[i] = g_chain[--g_chain_n];
      return;
    }
}

cudaError_t oneshot_read_status(int* out) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_status_os, sizeof(int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_status_os, &zero, sizeof(int));
}

}  // namespace q4
