// Tensor-core Q4_0 matrix-vector product for batch 1..16 (sm_103a).
//
// y[b][n] = sum_k W[n][k] x[b][k] with the 4-bit codes turned into exact
// binary16 values (q - 8) in registers and multiplied by binary16 x on the
// tensor cores (mma.sync m16n8k16, fp32 accumulate): every product is exact,
// the 16-term sums of one instruction are accumulated in fp32, and each
// 32-weight block's sum is scaled by its d once, in fp32.  The batch is the
// n dimension of the instruction (one n-tile of 8 columns for batch <= 8, two
// for batch <= 16), so the weights are read once for every batch row
// (PIPO summary, Method, "Computation optimization": 4-bit matrix-vector
// products without dequantisation; "Automatic configuration": that kernel
// serves batch sizes below 16).
//
// Persistent, one CTA per SM, 17 warps: warp 16 streams 16-row x 2048-column
// tiles of the weights into a ring of shared-memory stages (rows padded to
// keep the code-word loads free of bank conflicts), with one 2-D tensor copy
// per stage and matrix where the rows are whole chunks, else a 1-D bulk copy
// per row segment; warps 0-15 each take 4 of the stage's 64 blocks.  A CTA
// takes its row tiles in groups (8 tiles at batch <= 8, 4 above): chunk by
// chunk, the x fragments of a warp's blocks are loaded once for the whole
// group, every tile's partial sums stay in registers, and each tile is summed
// over the 16 warps in a fixed order when the group ends.
#include <cuda_fp16.h>
#include <stdint.h>

#include "q4_device.cuh"
#include "q4_frag.cuh"

namespace q4 {

__device__ int g_status_mma;   // status bits of the tensor-core kernel's waits

constexpr int kMmaWarps = 16;                    // consumer warps
constexpr int kMmaThreads = (kMmaWarps + 1) * 32;
constexpr int kMmaChunkBlocks = 64;              // 2048 columns per stage
constexpr int kMmaRowPitch = kMmaChunkBlocks * kBlockBytes + 16;   // 1168 B: 292 words, rows 4 banks apart
constexpr int kMmaStageBytes = 16 * kMmaRowPitch;                  // 18688 B
constexpr int kMmaStages = 10;

struct MmaArgs {
  CUtensorMap tm;     // with use_tm: the weights' TMA descriptor (box 146 x 16 rows, 8 when paired)
  int use_tm;
  const uint8_t* w;   // Q4_0 [n][k/32]
  const __half* x;    // binary16 [batch][k]
  float* y;           // fp32 [batch][split]: rows below `split`
  float* y2;          // fp32 [batch][n - split]: rows from `split` on (two matrices stored back to back)
  int n, k, batch, split;
  uint32_t wait_limit;
  int* status;        // where timed-out waits are recorded (g_status_mma if none given)
  MmaGather gather;   // gather.out null: none
  __half* act;        // gate|up pairing (see mma_launch), or null
};

extern __shared__ __align__(128) uint8_t g_mma_ring[];

template <int NT>
__global__ void __launch_bounds__(kMmaThreads, 1) mma_kernel(const __grid_constant__ MmaArgs a) {
  __shared__ __align__(8) uint64_t full_bar[kMmaStages];
  __shared__ __align__(8) uint64_t empty_bar[kMmaStages];
  __shared__ float red[kMmaWarps][32][4 * NT];
  __shared__ volatile int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, cta = blockIdx.x;
  const int nb = a.k / kQK;                                   // blocks per row
  griddep_launch_dependents();
  const int chunks = (nb + kMmaChunkBlocks - 1) / kMmaChunkBlocks;
  // paired gate|up: tile t holds rows [8t, 8t + 8) of both halves
  const bool paired = a.act != nullptr;
  const int half = a.n / 2;
  const int tiles = paired ? (half + 7) / 8 : (a.n + 15) / 16;
  const uint32_t row_bytes = static_cast<uint32_t>(nb) * kBlockBytes;

  if (tid == 0) {
    for (int s = 0; s < kMmaStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kMmaWarps);
    }
    fence_mbar_init();
    abort_flag = 0;
  }
  __syncthreads();

  // The CTA's row tiles (cta, cta + G, ...) are taken in groups of TG: for
  // each column chunk the producer copies the chunk of every tile of the
  // group, so the consumers load that chunk's x fragments once per group and
  // keep every tile's partial sums in registers.
  constexpr int TG = NT == 1 ? 8 : 4;
  if (warp == kMmaWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t it = 0;
      for (int g0 = cta; g0 < tiles && !abort_flag; g0 += G * TG) {
        for (int c = 0; c < chunks && !abort_flag; ++c) {
          const int blk0 = c * kMmaChunkBlocks;
          const uint32_t seg = static_cast<uint32_t>(min(kMmaChunkBlocks, nb - blk0)) * kBlockBytes;
          for (int q = 0; q < TG; ++q) {
            const int tile = g0 + q * G;
            if (tile >= tiles) break;
            const int row0 = paired ? tile * 8 : tile * 16;
            const int rows = paired ? min(8, half - row0) : min(16, a.n - row0);
            const int stage = it % kMmaStages;
            const uint32_t n = it / kMmaStages;
            if (n > 0 && !mbar_wait_bounded(&empty_bar[stage], (n - 1) & 1, a.wait_limit)) {
              atomicOr(a.status, ST_EMPTY_TIMEOUT);
              abort_flag = 1;
              break;
            }
            uint8_t* dst = g_mma_ring + static_cast<size_t>(stage) * kMmaStageBytes;
            if (a.use_tm) {
              // one 2-D tensor copy per matrix: the whole padded stage (rows past
              // the matrix read as zeros, and count in full)
              const int cx = c * (kMmaChunkBlocks * kBlockBytes / 8);
              mbar_arrive_expect_tx(&full_bar[stage], kMmaStageBytes);
              tma_load_2d(dst, &a.tm, cx, row0, &full_bar[stage]);
              if (paired) tma_load_2d(dst + 8 * kMmaRowPitch, &a.tm, cx, half + row0, &full_bar[stage]);
              ++it;
              continue;
            }
            mbar_arrive_expect_tx(&full_bar[stage], seg * rows * (paired ? 2 : 1));
            for (int r = 0; r < rows; ++r)
              bulk_g2s(dst + r * kMmaRowPitch, a.w + static_cast<size_t>(row0 + r) * row_bytes + blk0 * kBlockBytes,
                       seg, &full_bar[stage]);
            if (paired)
              for (int r = 0; r < rows; ++r)
                bulk_g2s(dst + (8 + r) * kMmaRowPitch,
                         a.w + static_cast<size_t>(half + row0 + r) * row_bytes + blk0 * kBlockBytes, seg,
                         &full_bar[stage]);
            ++it;
          }
        }
      }
      const uint32_t issued = it;
      for (int s = 0; s < kMmaStages && static_cast<uint32_t>(s) < issued; ++s) {
        const uint32_t last = (issued - 1 - s) / kMmaStages;
        if (!mbar_wait_bounded(&full_bar[s], last & 1, a.wait_limit)) atomicOr(a.status, ST_DRAIN_TIMEOUT);
      }
    }
  } else {
    // ------------------------------------------------------------ consumers
    // the weights need nothing from the previous kernel; x and y do
    griddep_wait();
    const int g = lane >> 2, t = lane & 3;
    uint32_t magic;
    asm volatile("mov.b32 %0, 0x64006400;" : "=r"(magic));
    uint32_t it = 0;
    for (int g0 = cta; g0 < tiles; g0 += G * TG) {
      const int ntg = min(TG, (tiles - g0 + G - 1) / G);   // tiles in this group
      float acc[TG][NT][4];
#pragma unroll
      for (int q = 0; q < TG; ++q)
#pragma unroll
        for (int j = 0; j < NT; ++j) acc[q][j][0] = acc[q][j][1] = acc[q][j][2] = acc[q][j][3] = 0.f;
      for (int c = 0; c < chunks; ++c) {
        const int nblk = min(kMmaChunkBlocks, nb - c * kMmaChunkBlocks);
        // this warp's blocks of the chunk: their x fragments, once for the group
        uint32_t xf[kMmaChunkBlocks / kMmaWarps][NT][4];
#pragma unroll
        for (int i = 0; i < kMmaChunkBlocks / kMmaWarps; ++i) {
          const int b = warp + kMmaWarps * i;
#pragma unroll
          for (int j = 0; j < NT; ++j) {
            if (b < nblk)
              x_frags(a.x, a.k, a.batch, 8 * j + g, c * kMmaChunkBlocks + b, t, xf[i][j][0], xf[i][j][1],
                      xf[i][j][2], xf[i][j][3]);
            else
              xf[i][j][0] = xf[i][j][1] = xf[i][j][2] = xf[i][j][3] = 0u;
          }
        }
#pragma unroll
        for (int q = 0; q < TG; ++q) {
          if (q >= ntg) break;
          const int stage = it % kMmaStages;
          const uint32_t n = it / kMmaStages;
          if (!abort_flag && !mbar_wait_bounded(&full_bar[stage], n & 1, a.wait_limit)) {
            atomicOr(a.status, ST_FULL_TIMEOUT);
            abort_flag = 1;
          }
          const uint8_t* sb = g_mma_ring + static_cast<size_t>(stage) * kMmaStageBytes;
          const uint8_t* rg = sb + g * kMmaRowPitch;
          const uint8_t* rh = sb + (g + 8) * kMmaRowPitch;
#pragma unroll
          for (int i = 0; i < kMmaChunkBlocks / kMmaWarps; ++i) {
            const int b = warp + kMmaWarps * i;       // block within the chunk (parity = warp parity)
            if (b < nblk) {
              uint32_t gl02, gl13, gh02, gh13, hl02, hl13, hh02, hh13;
              unpack_word(code_word(rg, b, t), magic, gl02, gl13, gh02, gh13);
              unpack_word(code_word(rh, b, t), magic, hl02, hl13, hh02, hh13);
              const float dg = row_scale(rg, b), dh = row_scale(rh, b);
#pragma unroll
              for (int j = 0; j < NT; ++j) {
                float cb[4] = {0.f, 0.f, 0.f, 0.f};
                mma16816(cb, gl02, hl02, gl13, hl13, xf[i][j][0], xf[i][j][1]);
                mma16816(cb, gh02, hh02, gh13, hh13, xf[i][j][2], xf[i][j][3]);
                acc[q][j][0] = fmaf(dg, cb[0], acc[q][j][0]);
                acc[q][j][1] = fmaf(dg, cb[1], acc[q][j][1]);
                acc[q][j][2] = fmaf(dh, cb[2], acc[q][j][2]);
                acc[q][j][3] = fmaf(dh, cb[3], acc[q][j][3]);
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty_bar[stage]);
          ++it;
        }
      }
      // each tile's 16 warps' partial sums, summed in a fixed order
#pragma unroll
      for (int q = 0; q < TG; ++q) {
        if (q >= ntg) break;
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) red[warp][lane][4 * j + e] = acc[q][j][e];
        named_bar_sync(1, kMmaWarps * 32);
        if (paired) {
          // row m of the first half and row m of the second are rows m and m + 8 of the tile
          const int row0 = (g0 + q * G) * 8;
          for (int o = tid; o < 8 * 8 * NT; o += kMmaWarps * 32) {
            const int m = o % 8, col = o / 8;
            const int j = col / 8, cc = col % 8;
            const int ln = m * 4 + cc / 2, e = cc & 1;
            float gv = 0.f, uv = 0.f;
            for (int w = 0; w < kMmaWarps; ++w) {
              gv += red[w][ln][4 * j + e];
              uv += red[w][ln][4 * j + 2 + e];
            }
            const int r = row0 + m;
            if (col < a.batch && r < half) {
              const size_t i = static_cast<size_t>(col) * half + r;
              a.y[i] = gv;
              a.y2[i] = uv;
              a.act[i] = __float2half_rn(gv / (1.0f + expf(-gv)) * uv);
            }
          }
          named_bar_sync(1, kMmaWarps * 32);
          continue;
        }
        const int row0 = (g0 + q * G) * 16;
        for (int o = tid; o < 16 * 8 * NT; o += kMmaWarps * 32) {
          const int m = o % 16, col = o / 16;           // output row in the tile, batch column
          const int j = col / 8, cc = col % 8;
          // C fragment: lane (gm, tc) holds rows gm and gm+8, columns 2tc and 2tc+1
          const int ln = (m % 8) * 4 + cc / 2;
          const int e = (m >= 8 ? 2 : 0) + (cc & 1);
          float s = 0.f;
          for (int w = 0; w < kMmaWarps; ++w) s += red[w][ln][4 * j + e];
          const int r = row0 + m;
          if (col < a.batch && r < a.n) {
            if (r < a.split)
              a.y[static_cast<size_t>(col) * a.split + r] = s;
            else
              a.y2[static_cast<size_t>(col) * (a.n - a.split) + (r - a.split)] = s;
            const MmaGather& gt = a.gather;
            if (gt.out && r >= gt.lo && r < gt.lo + gt.n_rows) {
              const int vh = (r - gt.lo) / gt.head_dim, i = (r - gt.lo) % gt.head_dim;
              const unsigned short hv = __half_as_ushort(__float2half_rn(s));
              for (int h = 0; h < gt.group; ++h)
                gt.out[static_cast<size_t>(col) * gt.ld + (vh * gt.group + h) * gt.head_dim + i] = hv;
            }
          }
        }
        named_bar_sync(1, kMmaWarps * 32);
      }
    }
  }
  __syncthreads();
}

cudaError_t mma_read_status(int* out) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_status_mma, sizeof(int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_status_mma, &zero, sizeof(int));
}

cudaError_t mma_prepare() {
  cudaError_t e = cudaFuncSetAttribute(mma_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kMmaStages * kMmaStageBytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(mma_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kMmaStages * kMmaStageBytes);
}

cudaError_t mma_launch(const uint8_t* w, const uint16_t* x, float* y, int n, int k, int batch, int grid,
                       uint32_t wait_limit, int* status, cudaStream_t stream, float* y2, int split, bool pdl,
                       const MmaGather* gather, uint16_t* act) {
  MmaArgs a;
  a.gather = gather ? *gather : MmaGather{nullptr, 0, 0, 1, 0, 0};
  a.act = reinterpret_cast<__half*>(act);
  if (act && (!y2 || n % 2 || split != n / 2)) return cudaErrorInvalidValue;
  if (a.gather.out && (a.gather.head_dim < 1 || a.gather.group < 1)) return cudaErrorInvalidValue;
  a.y2 = y2;
  a.split = (y2 && split > 0 && split < n) ? split : n;
  if (!status) {
    cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&status), g_status_mma);
    if (e != cudaSuccess) return e;
  }
  a.status = status;
  a.w = w;
  a.x = reinterpret_cast<const __half*>(x);
  a.y = y;
  a.n = n;
  a.k = k;
  a.batch = batch;
  a.wait_limit = wait_limit;
  // rows of whole 2048-column chunks, more than one (the descriptor's box is
  // then the padded 1168-byte stage row), one n-tile: one tensor copy per
  // stage (and matrix) instead of a bulk copy per row, which bounded the
  // producer (at two n-tiles the consumers bound it and the row copies were
  // measured faster)
  a.use_tm = batch <= 8 && k % (kMmaChunkBlocks * kQK) == 0 && tc_pitch(k) == kMmaRowPitch &&
                     encode_q4_rows(&a.tm, w, n, k, act ? 8 : 16)
                 ? 1
                 : 0;
  const int tiles = act ? (n / 2 + 7) / 8 : (n + 15) / 16;
  if (grid > tiles) grid = tiles;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kMmaThreads);
  cfg.dynamicSmemBytes = kMmaStages * kMmaStageBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return batch <= 8 ? cudaLaunchKernelEx(&cfg, mma_kernel<1>, a) : cudaLaunchKernelEx(&cfg, mma_kernel<2>, a);
}

}  // namespace q4
