// C ABI of libq4.so (declared in include/q4.h): argument checks, launch
// configuration, the decoder (phase programs + CUDA-graph capture) and the
// double-buffered copy/compute ring.  Host code only; every arithmetic step
// of the decode runs in the kernels of q4_engine.cu and q4_aux.cu.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <stdlib.h>

#include <atomic>
#include <chrono>
#include <mutex>
#include <thread>
#include <algorithm>
#include <vector>

#include "q4.h"
#include "q4_device.cuh"

using q4::Control;
using q4::EngineArgs;
using q4::Phase;

namespace {

std::atomic<int> g_last_cuda{0};

int cuda_fail(cudaError_t e) {
  g_last_cuda.store(static_cast<int>(e));
  return Q4_ERR_CUDA;
}

#define Q4_CUDA(call)                              \
  do {                                             \
    cudaError_t e_ = (call);                       \
    if (e_ != cudaSuccess) return cuda_fail(e_);   \
  } while (0)

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Wait limit of one in-kernel wait, in polls (a poll suspends for tens to
// hundreds of nanoseconds): about a second, far above any legitimate wait.
constexpr uint32_t kWaitLimit = 1u << 22;

struct DeviceInfo {
  bool ready = false;
  int sm_count = 0;
  int engine_blocks_per_sm = 0;
};

std::mutex g_dev_mutex;
DeviceInfo g_dev[64];

int device_info(DeviceInfo** out) {
  int dev = 0;
  Q4_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return Q4_ERR_ARG;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    Q4_CUDA(cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev));
    Q4_CUDA(q4::engine_prepare());
    Q4_CUDA(q4::mma_prepare());
    Q4_CUDA(q4::tc_engine_prepare());
    Q4_CUDA(q4::oneshot_prepare());
    Q4_CUDA(q4::attn_prepare());
    Q4_CUDA(q4::bt_engine_prepare());
    Q4_CUDA(q4::engine_occupancy(&d.engine_blocks_per_sm));
    if (d.engine_blocks_per_sm < 1) return Q4_ERR_CUDA;
    int tc_blocks = 0;
    Q4_CUDA(q4::tc_engine_occupancy(&tc_blocks));
    if (tc_blocks < 1) return Q4_ERR_CUDA;
    d.ready = true;
  }
  *out = &d;
  return Q4_OK;
}

// Whether the streaming engine can run rows of width k: every consumer
// thread owns 64 columns, a row team is k/64 threads, and a team either fills
// whole warps or divides one; rows must start 16-byte aligned (k % 256 == 0).
bool engine_ok(int k) {
  if (k < 256 || k % 256 != 0) return false;
  const int team = k / q4::kKT;
  if (team > q4::kConsumerThreads) return false;
  // a unit holds two rows of every team: at least two rows must fit a stage
  if (2 * (k / q4::kQK) * q4::kBlockBytes > q4::kStageBytes) return false;
  return team % 32 == 0 || 32 % team == 0;
}

// The two persistent engines: exact CUDA-core products (q4_engine.cu) and
// tensor-core products (q4_tc_engine.cu).
enum Engine { ENG_CORE = 0, ENG_TC = 1, ENG_BT = 2 };

// Whether the tensor-core engine can run rows of width k: whole 8-block row
// segments (16-byte aligned), one column chunk or whole 64-block chunks, and
// an input that fits its fragment buffer.
bool tc_ok(int k) { return k >= 256 && k % 256 == 0 && (k <= 2048 || k % 2048 == 0) && k <= q4::kTcMaxK; }

// TMA descriptors are encoded with the driver's cuTensorMapEncodeTiled,
// reached through the runtime's entry-point query (no link-time dependency on
// the driver library).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static const EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeTiledFn>(nullptr);
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// Descriptor of a row-major Q4_0 matrix (n_rows x k) for the tensor-core
// engine: 64-bit elements, row_bytes / 8 columns, box tc_pitch(k) / 8 columns
// by box_rows rows.
bool encode_rows(CUtensorMap* m, const uint8_t* w, int n_rows, int k, int box_rows) {
  const EncodeTiledFn fn = encode_fn();
  if (!fn || !w || !aligned(w, 16) || n_rows < 1) return false;
  const cuuint64_t row_bytes = static_cast<cuuint64_t>(k / q4::kQK) * q4::kBlockBytes;
  const cuuint64_t gdim[2] = {row_bytes / 8, static_cast<cuuint64_t>(n_rows)};
  const cuuint64_t gstride[1] = {row_bytes};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(q4::tc_pitch(k) / 8), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estride[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<uint8_t*>(w), gdim, gstride, box, estride,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Fill the tiling fields of a phase.  CUDA-core engine: a work unit gives
// every team two rows (two rows of one matrix, or the same row of both
// matrices of a pair).  Tensor-core engine: a unit is one 32-row tile (16
// rows of each matrix of a pair), and with `encode` the phase's TMA
// descriptors are written (not for shape checks, which pass no weights).
bool tile_phase(Phase& ph, int engine = ENG_CORE, bool encode = true) {
  if (engine == ENG_TC) {
    if (!tc_ok(ph.k)) return false;
    ph.teams = 0;
    const bool dual = ph.epi_kind == q4::EPI_SILU;
    ph.rows_per_unit = dual ? q4::kTcUnitRows / 2 : q4::kTcUnitRows;
    ph.units = (ph.n_rows + ph.rows_per_unit - 1) / ph.rows_per_unit;
    if (encode && ph.n_rows > 0) {
      if (!encode_rows(&ph.tm0, ph.w0, ph.n_rows, ph.k, ph.rows_per_unit)) return false;
      if (dual && !encode_rows(&ph.tm1, ph.w1, ph.n_rows, ph.k, ph.rows_per_unit)) return false;
    }
    return true;
  }
  if (!engine_ok(ph.k)) return false;
  const int team = ph.k / q4::kKT;
  const int row_bytes = ph.k / q4::kQK * q4::kBlockBytes;
  int teams = q4::kConsumerThreads / team;
  const int fit = q4::kStageBytes / (2 * row_bytes);
  if (teams > fit) teams = fit;
  // teams narrower than a warp fill whole warps (their shuffles span the warp)
  if (team < 32) teams -= teams % (32 / team);
  if (teams < 1) return false;
  ph.teams = teams;
  ph.rows_per_unit = ph.epi_kind == q4::EPI_SILU ? teams : 2 * teams;
  ph.units = (ph.n_rows + ph.rows_per_unit - 1) / ph.rows_per_unit;
  return true;
}

// Ring and buffers of a tensor-core launch whose phases have widths in
// `ks`: stage stride = 32 rows of the widest pitch, fragment buffer = 2 bytes
// per value of the widest input, as many stages (up to 8) as fit.
struct TcGeom {
  int stages = 0;
  uint32_t stage_bytes = 0;
  int xbuf_floats = 0;
};

bool tc_geom(std::initializer_list<int> ks, TcGeom* g) {
  int kmax = 0, pmax = 0;
  for (int k : ks) {
    if (!tc_ok(k)) return false;
    kmax = std::max(kmax, k);
    pmax = std::max(pmax, q4::tc_pitch(k));
  }
  g->stage_bytes = static_cast<uint32_t>(pmax) * q4::kTcUnitRows;
  g->xbuf_floats = (2 * kmax + 15) / 16 * 4;
  int s = 8;
  while (s >= 2 && q4::tc_smem_bytes(s, g->stage_bytes, g->xbuf_floats) > q4::kTcSmemLimit) --s;
  g->stages = s;
  return s >= 3;
}

}  // namespace

namespace q4 {
bool encode_q4_rows(CUtensorMap* m, const uint8_t* w, int n_rows, int k, int box_rows) {
  return encode_rows(m, w, n_rows, k, box_rows);
}
}  // namespace q4

// ===================================================================== misc

extern "C" const char* q4_status_string(int s) {
  switch (s) {
    case Q4_OK: return "ok";
    case Q4_ERR_ARG: return "invalid argument";
    case Q4_ERR_ALIGN: return "pointer not 16-byte aligned";
    case Q4_ERR_CUDA: return "CUDA runtime error";
    case Q4_ERR_TIMEOUT: return "timed out";
    case Q4_ERR_OOM: return "workspace too small";
    case Q4_ERR_DEVICE: return "a kernel wait failed";
    default: return "unknown status";
  }
}

extern "C" int q4_last_cuda_error(void) { return g_last_cuda.exchange(0); }

extern "C" int q4_version(void) { return 100; }

extern "C" size_t q4_matrix_bytes(int n, int k) {
  if (n <= 0 || k <= 0 || k % q4::kQK) return 0;
  return static_cast<size_t>(n) * (k / q4::kQK) * q4::kBlockBytes;
}

// ===================================================================== one product

static int check_gemv(const void* w, const uint16_t* x, const float* y, int n, int k, int batch) {
  if (!w || !x || !y) return Q4_ERR_ARG;
  if (n < 1 || k < q4::kQK || k % q4::kQK || batch < 1 || batch > q4::kMaxBatch) return Q4_ERR_ARG;
  if (!aligned(w, 16) || !aligned(x, 16) || !aligned(y, 16)) return Q4_ERR_ALIGN;
  return Q4_OK;
}

extern "C" int q4_gemv_ex(const void* w, const uint16_t* x, float* y, int n, int k, int batch, int kernel,
                          void* stream) {
  int st = check_gemv(w, x, y, n, k, batch);
  if (st != Q4_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool chain = (kernel & Q4_GEMV_CHAIN) != 0;
  kernel &= ~Q4_GEMV_CHAIN;
  if (kernel == Q4_KERNEL_AUTO) {
    // batch 1: the one-shot kernel up to 64 MB of weights (it overlaps
    // consecutive launches), the persistent tensor-core engine above that (its
    // ring streams large matrices faster), else the CUDA-core engine or the
    // plain kernel for widths they cannot take; batch 2..16: tensor cores when
    // rows are 16-byte aligned
    const size_t bytes = static_cast<size_t>(n) * (k / q4::kQK) * q4::kBlockBytes;
    if (batch == 1)
      kernel = q4::oneshot_ok(n, k) && bytes <= (size_t(64) << 20) ? Q4_KERNEL_ONESHOT
               : tc_ok(k)                                          ? Q4_KERNEL_TC
               : engine_ok(k)                                      ? Q4_KERNEL_STREAM
                                                                   : Q4_KERNEL_SIMPLE;
    else if (k % 256 == 0) kernel = Q4_KERNEL_MMA;
    else kernel = Q4_KERNEL_SIMPLE;
  }
  // only one-shot products know how to follow one another early
  if (kernel != Q4_KERNEL_ONESHOT) q4::oneshot_chain_break(s);
  if (kernel == Q4_KERNEL_SIMPLE) {
    Q4_CUDA(q4::simple_launch(static_cast<const uint8_t*>(w), x, y, n, k, batch, s));
    return Q4_OK;
  }
  if (kernel == Q4_KERNEL_ONESHOT) {
    if (batch != 1 || !q4::oneshot_ok(n, k)) return Q4_ERR_ARG;
    DeviceInfo* dev = nullptr;
    if ((st = device_info(&dev)) != Q4_OK) return st;
    Q4_CUDA(q4::oneshot_launch(static_cast<const uint8_t*>(w), x, y, n, k, kWaitLimit, chain, s));
    return Q4_OK;
  }
  if (kernel == Q4_KERNEL_MMA) {
    if (k % 256 != 0) return Q4_ERR_ARG;   // row segments of a tile must start 16-byte aligned
    DeviceInfo* dev = nullptr;
    if ((st = device_info(&dev)) != Q4_OK) return st;
    Q4_CUDA(q4::mma_launch(static_cast<const uint8_t*>(w), x, y, n, k, batch, dev->sm_count, kWaitLimit, nullptr, s));
    return Q4_OK;
  }
  if ((kernel != Q4_KERNEL_STREAM && kernel != Q4_KERNEL_TC) || batch != 1) return Q4_ERR_ARG;
  const int engine = kernel == Q4_KERNEL_TC ? ENG_TC : ENG_CORE;
  if (!(engine == ENG_TC ? tc_ok(k) : engine_ok(k))) return Q4_ERR_ARG;
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev)) != Q4_OK) return st;
  EngineArgs a;
  memset(&a, 0, sizeof(a));
  Phase& ph = a.one;
  ph.w0 = static_cast<const uint8_t*>(w);
  ph.x_src = x;
  ph.y = y;
  ph.n_rows = n;
  ph.k = k;
  ph.x_kind = q4::X_F16;
  ph.epi_kind = q4::EPI_F32;
  ph.x_ld = k;
  if (!tile_phase(ph, engine)) return Q4_ERR_ARG;
  a.phases = nullptr;
  a.n_phases = 1;
  a.ctl = nullptr;
  a.wait_limit = kWaitLimit;
  const int grid = ph.units < dev->sm_count ? ph.units : dev->sm_count;
  if (engine == ENG_TC) {
    TcGeom g;
    if (!tc_geom({k}, &g)) return Q4_ERR_ARG;
    a.stages = g.stages;
    a.stage_bytes = g.stage_bytes;
    a.xbuf_floats = g.xbuf_floats;
    Q4_CUDA(q4::tc_engine_launch(a, grid, false, s));
  } else
    Q4_CUDA(q4::engine_launch(a, grid, false, s));
  return Q4_OK;
}

extern "C" int q4_gemv(const void* w, const uint16_t* x, float* y, int n, int k, int batch, void* stream) {
  return q4_gemv_ex(w, x, y, n, k, batch, Q4_KERNEL_AUTO, stream);
}

extern "C" int q4_timeline_read(unsigned long long* out, size_t n, int clear) {
  if (!out) return Q4_ERR_ARG;
  cudaError_t e = q4::tc_timeline_read(out, n, clear != 0);
  if (e == cudaErrorNotSupported || e == cudaErrorInvalidValue) return Q4_ERR_ARG;
  Q4_CUDA(e);
  // the batched engine keeps its own timeline: merged in (of two stamps of
  // one slot, only the engine that ran has written one)
  std::vector<unsigned long long> bt(n);
  e = q4::bt_timeline_read(bt.data(), n, clear != 0);
  if (e == cudaErrorNotSupported || e == cudaErrorInvalidValue) return Q4_ERR_ARG;
  Q4_CUDA(e);
  for (size_t i = 0; i < n; ++i) out[i] = std::max(out[i], bt[i]);
  return Q4_OK;
}

extern "C" int q4_device_status(void) {
  if (cudaDeviceSynchronize() != cudaSuccess) return cuda_fail(cudaGetLastError());
  int v = 0, m = 0;
  Q4_CUDA(q4::engine_read_status(&v));
  Q4_CUDA(q4::mma_read_status(&m));
  int tc = 0, os = 0;
  Q4_CUDA(q4::tc_engine_read_status(&tc));
  Q4_CUDA(q4::oneshot_read_status(&os));
  return v | m | tc | os;
}

extern "C" int q4_dequant_debug(const void* w, float* w_out, int n, int k, void* stream) {
  if (!w || !w_out || n < 1 || k < q4::kQK || k % q4::kQK) return Q4_ERR_ARG;
  if (!aligned(w, 16) || !aligned(w_out, 16)) return Q4_ERR_ALIGN;
  Q4_CUDA(q4::dequant_launch(static_cast<const uint8_t*>(w), w_out, n, k, static_cast<cudaStream_t>(stream)));
  return Q4_OK;
}

// ===================================================================== layers

static bool shape_ok(const q4_layer_shape* s) {
  if (!s) return false;
  if (s->hidden < 32 || s->q_dim < 32 || s->kv_dim < 32 || s->ffn < 32 || s->head_dim < 1) return false;
  if (s->hidden % 32 || s->q_dim % 32 || s->kv_dim % 32 || s->ffn % 32) return false;
  if (s->q_dim % s->head_dim || s->kv_dim % s->head_dim) return false;
  if ((s->q_dim / s->head_dim) % (s->kv_dim / s->head_dim)) return false;
  return s->eps >= 0.f;
}

extern "C" int q4_layer_offsets(const q4_layer_shape* s, size_t offsets[7], size_t* layer_bytes) {
  if (!shape_ok(s) || !offsets) return Q4_ERR_ARG;
  const int dims[7][2] = {{s->q_dim, s->hidden}, {s->kv_dim, s->hidden}, {s->kv_dim, s->hidden},
                          {s->hidden, s->q_dim}, {s->ffn, s->hidden},    {s->ffn, s->hidden},
                          {s->hidden, s->ffn}};
  size_t pos = 0;
  for (int p = 0; p < 7; ++p) {
    offsets[p] = pos;
    pos += q4_matrix_bytes(dims[p][0], dims[p][1]);
  }
  if (layer_bytes) *layer_bytes = pos;
  return Q4_OK;
}

extern "C" int q4_workspace_layout(const q4_layer_shape* s, int n_layers, int batch, size_t offsets[Q4_WS_COUNT],
                                   size_t* total_bytes) {
  if (!shape_ok(s) || n_layers < 1 || batch < 1 || batch > q4::kMaxBatch || !offsets) return Q4_ERR_ARG;
  const size_t B = static_cast<size_t>(batch);
  const size_t L = static_cast<size_t>(n_layers);
  // batch 2..16: the batched engine's program, its input fragments (z and the
  // attention output after the tagged-word regions' place, act after v's) and
  // its per-CTA sums of squares after the flags
  const size_t prog = std::max(sizeof(Phase) * (4 * L + 1), batch > 1 ? sizeof(q4::BtPhase) * (6 * L + 1) : 0);
  const size_t frag = 2 * static_cast<size_t>(q4::kBtCols);   // fragment bytes per value
  const size_t sizes[Q4_WS_COUNT] = {
      sizeof(Control),
      prog,
      4 * B * (s->q_dim + 2 * s->kv_dim),
      4 * B * s->hidden,
      4 * B * s->ffn,
      4 * B * s->ffn,
      4 * B * s->hidden,
      2 * B * s->ffn,
      2 * B * s->hidden,
      2 * B * s->q_dim,
      2 * B * s->hidden,
      4 * B * s->hidden,
      4 * B * s->hidden,
      8 * 2 * static_cast<size_t>(q4::kMaxGrid) + 4 * 2 * static_cast<size_t>(q4::kMaxGrid) +
          4 * static_cast<size_t>(q4::kBtCols) * q4::kMaxGrid,
      // batch-1 engine inputs: fp32 t1/t2 slice-transposed, or (tagged programs)
      // tagged t1 and t2 (64-bit words) and the tagged residual bases z and z1
      std::max(24 * static_cast<size_t>(s->hidden), batch > 1 ? frag * (s->hidden + s->q_dim) : 0),
      4 * static_cast<size_t>(s->kv_dim),
      std::max(4 * static_cast<size_t>(s->ffn), batch > 1 ? frag * s->ffn : 0),
  };
  size_t pos = 0;
  for (int i = 0; i < Q4_WS_COUNT; ++i) {
    offsets[i] = pos;
    pos += (sizes[i] + 255) / 256 * 256;
  }
  if (total_bytes) *total_bytes = pos;
  return Q4_OK;
}

namespace {

// Pointers into a workspace.
struct Work {
  Control* ctl;
  Phase* prog;
  float *qkv, *o, *g, *u, *dn, *t1, *t2;
  unsigned long long* flags;   // [2][kMaxGrid] end-of-phase flags
  float *ss1, *ss2;            // per-CTA sums of squares of t1 and t2
  uint16_t *act, *x, *attn, *x2;
  float *xt, *vt;              // slice-transposed t1/t2 and v (CUDA-core engine inputs)
  uint16_t* actt;              // slice-transposed act
  // the same regions in a tagged program: tagged t1, t2 (fp32), z, z1, v, act (binary16)
  unsigned long long *t1t, *t2t;
  uint32_t *zt, *z1t, *vtag, *acttag;
  // batched engine: input fragments of q|k|v and gate|up (z, z1), of o (the
  // attention output) and of down (act); per-CTA sums of squares
  uint8_t *zf, *af, *actf;
  float* ss8;
};

Work carve(void* ws, const size_t* off, int hidden) {
  char* b = static_cast<char*>(ws);
  Work w;
  w.ctl = reinterpret_cast<Control*>(b + off[Q4_WS_CONTROL]);
  w.prog = reinterpret_cast<Phase*>(b + off[Q4_WS_PROGRAM]);
  w.qkv = reinterpret_cast<float*>(b + off[Q4_WS_QKV]);
  w.o = reinterpret_cast<float*>(b + off[Q4_WS_O]);
  w.g = reinterpret_cast<float*>(b + off[Q4_WS_GATE]);
  w.u = reinterpret_cast<float*>(b + off[Q4_WS_UP]);
  w.dn = reinterpret_cast<float*>(b + off[Q4_WS_DOWN]);
  w.act = reinterpret_cast<uint16_t*>(b + off[Q4_WS_ACT]);
  w.x = reinterpret_cast<uint16_t*>(b + off[Q4_WS_X]);
  w.attn = reinterpret_cast<uint16_t*>(b + off[Q4_WS_ATTN]);
  w.x2 = reinterpret_cast<uint16_t*>(b + off[Q4_WS_X2]);
  w.t1 = reinterpret_cast<float*>(b + off[Q4_WS_T1]);
  w.t2 = reinterpret_cast<float*>(b + off[Q4_WS_T2]);
  w.flags = reinterpret_cast<unsigned long long*>(b + off[Q4_WS_FLAGS]);
  w.ss1 = reinterpret_cast<float*>(w.flags + 2 * q4::kMaxGrid);
  w.ss2 = w.ss1 + q4::kMaxGrid;
  w.xt = reinterpret_cast<float*>(b + off[Q4_WS_XT]);
  w.vt = reinterpret_cast<float*>(b + off[Q4_WS_VT]);
  w.actt = reinterpret_cast<uint16_t*>(b + off[Q4_WS_ACTT]);
  w.t1t = reinterpret_cast<unsigned long long*>(b + off[Q4_WS_XT]);
  w.t2t = w.t1t + hidden;
  w.zt = reinterpret_cast<uint32_t*>(w.t2t + hidden);
  w.z1t = w.zt + hidden;
  w.vtag = reinterpret_cast<uint32_t*>(b + off[Q4_WS_VT]);
  w.acttag = reinterpret_cast<uint32_t*>(b + off[Q4_WS_ACTT]);
  w.zf = reinterpret_cast<uint8_t*>(b + off[Q4_WS_XT]);
  w.af = w.zf + 2 * static_cast<size_t>(q4::kBtCols) * hidden;
  w.actf = reinterpret_cast<uint8_t*>(b + off[Q4_WS_ACTT]);
  w.ss8 = w.ss2 + q4::kMaxGrid;
  return w;
}

// The four phases of one decoder layer whose merged weight block is `wl`
// (PIPO summary, "Offloading architecture": the layer is the unit).  The
// layer input is normalised from `in16` (binary16, first layer) or from the
// previous layer's fp32 residual sum (`in32`); the normalised input is kept
// in w.x and is the residual base of the attention half, whose fp32 sum goes
// to w.t1; the normalised w.t1 (w.x2) is the residual base of the feed-forward
// half, whose fp32 sum goes to w.t2.
bool layer_phases(const q4_layer_shape& s, const uint8_t* wl, const uint16_t* in16, const Work& w, Phase out[4],
                  int engine) {
  size_t off[7];
  if (q4_layer_offsets(&s, off, nullptr) != Q4_OK) return false;
  memset(out, 0, 4 * sizeof(Phase));
  // q, k, v: one matrix of q_dim + 2 kv_dim rows (they are consecutive in the block)
  Phase& a = out[0];
  a.w0 = wl + off[Q4_PROJ_Q];
  a.x_src = in16 ? static_cast<const void*>(in16) : static_cast<const void*>(w.t2);
  a.y = w.qkv;
  a.n_rows = s.q_dim + 2 * s.kv_dim;
  a.k = s.hidden;
  a.x_kind = in16 ? q4::X_NORM16 : q4::X_NORM32;
  a.ss_in = w.ss2;
  a.epi_kind = q4::EPI_F32;
  a.x_ld = s.hidden;
  a.eps = s.eps;
  a.x_dbg = w.x;
  // o, with the context-1 attention as its input and the residual sum as its output
  Phase& b = out[1];
  b.w0 = wl + off[Q4_PROJ_O];
  b.x_src = w.qkv;
  b.y = w.o;
  b.y2 = w.t1;
  b.res = w.x;
  b.ss_out = w.ss1;
  b.n_rows = s.hidden;
  b.k = s.q_dim;
  b.x_kind = q4::X_ATTN;
  b.epi_kind = q4::EPI_RESID;
  b.x_ld = s.q_dim + 2 * s.kv_dim;
  b.attn_off = s.q_dim + s.kv_dim;
  b.head_dim = s.head_dim;
  b.group = (s.q_dim / s.head_dim) / (s.kv_dim / s.head_dim);
  b.x_dbg = w.attn;
  // gate and up together, SiLU-gated product as the output
  Phase& c = out[2];
  c.w0 = wl + off[Q4_PROJ_GATE];
  c.w1 = wl + off[Q4_PROJ_UP];
  c.x_src = w.t1;
  c.y = w.g;
  c.y2 = w.u;
  c.aux16 = w.act;
  c.n_rows = s.ffn;
  c.k = s.hidden;
  c.x_kind = q4::X_NORM32;
  c.ss_in = w.ss1;
  c.epi_kind = q4::EPI_SILU;
  c.x_ld = s.hidden;
  c.eps = s.eps;
  c.x_dbg = w.x2;
  // down, with the residual sum
  Phase& d = out[3];
  d.w0 = wl + off[Q4_PROJ_DOWN];
  d.x_src = w.act;
  d.y = w.dn;
  d.y2 = w.t2;
  d.res = w.x2;
  d.ss_out = w.ss2;
  d.n_rows = s.hidden;
  d.k = s.ffn;
  d.x_kind = q4::X_F16;
  d.epi_kind = q4::EPI_RESID;
  d.x_ld = s.ffn;
  if (engine == ENG_CORE) {
    // each phase also leaves the next phase's input slice-transposed, so that
    // the consumer threads' x-slice loads are coalesced
    if (!in16) {
      a.x_src = w.xt;
      a.x_t = 1;
      a.x_ld = s.hidden / q4::kKT;
    }
    a.yt = w.vt;
    a.yt_off = s.q_dim + s.kv_dim;
    a.yt_n = s.kv_dim;
    b.x_src = w.vt;
    b.x_t = 1;
    b.x_ld = s.kv_dim / q4::kKT;
    b.yt = w.xt;
    b.yt_n = s.hidden;
    c.x_src = w.xt;
    c.x_t = 1;
    c.x_ld = s.hidden / q4::kKT;
    c.yt = w.actt;
    c.yt_n = s.ffn;
    d.x_src = w.actt;
    d.x_t = 1;
    d.x_ld = s.ffn / q4::kKT;
    d.yt = w.xt;
    d.yt_n = s.hidden;
  }
  for (int i = 0; i < 4; ++i)
    if (!tile_phase(out[i], engine)) return false;
  return true;
}

// The closing phase of a stack: no product, CTA 0 writes the normalised last
// residual sum to the caller's hidden-state buffer.
bool final_phase(const q4_layer_shape& s, uint16_t* h_out, const Work& w, Phase* out, int engine) {
  memset(out, 0, sizeof(Phase));
  out->x_src = w.t2;
  out->ss_in = w.ss2;
  out->n_rows = 0;
  out->k = s.hidden;
  out->x_kind = q4::X_NORM32;
  out->epi_kind = q4::EPI_F32;
  out->x_ld = s.hidden;
  out->eps = s.eps;
  out->x_dbg = h_out;
  if (engine == ENG_CORE) {
    out->x_src = w.xt;
    out->x_t = 1;
    out->x_ld = s.hidden / q4::kKT;
  }
  return tile_phase(*out, engine);
}

// Whether the CUDA-core engine can run a layer shape as a tagged program:
// every phase input fits the per-CTA staging buffer and the chunk budget of
// the staging loops.
// Staging buffer of a tagged program (bytes): the widest phase input (fp32
// hidden values for the norms, binary16 kv_dim and ffn values), and room for
// the row partials.
size_t tagged_xbuf_bytes(const q4_layer_shape& s) {
  size_t b = 4 * static_cast<size_t>(q4::kRedFloats);
  b = std::max(b, 4 * static_cast<size_t>(s.hidden));
  b = std::max(b, 2 * static_cast<size_t>(s.kv_dim));
  b = std::max(b, 2 * static_cast<size_t>(s.ffn));
  return (b + 15) / 16 * 16;
}

// Ring depth of a tagged program: 6 stages when the staging buffer fits next
// to them, else 5.
int tagged_stages(const q4_layer_shape& s) {
  return tagged_xbuf_bytes(s) <= static_cast<size_t>(q4::kXBufMaxBytes6) ? 6 : 5;
}

bool tagged_ok(const q4_layer_shape& s) {
  return s.hidden <= q4::kNormMaxValues && s.kv_dim <= q4::kTag16MaxValues && s.ffn <= q4::kTag16MaxValues &&
         tagged_xbuf_bytes(s) <= static_cast<size_t>(q4::kXBufMaxBytes5);
}

// The four phases of one layer as a tagged program (CUDA-core engine, batch
// 1).  The same arithmetic as layer_phases; the values one phase hands to the
// next travel as tagged words (t1, t2 fp32; v, act and the residual bases z, z1
// binary16), so no phase waits at a barrier.  The plain intermediates are
// written for the last layer only (the workspace keeps the last layer's).
// Phase 1 publishes the flags that phase 2 waits for (SyncKind): every
// tagged buffer is rewritten once per layer, and that single exchange, with
// the data dependences between the phases, orders each rewrite after every
// read of the previous values.
bool layer_phases_tagged(const q4_layer_shape& s, const uint8_t* wl, const uint16_t* in16, const Work& w,
                         Phase out[4], bool last, int engine, bool kv = false) {
  size_t off[7];
  if (q4_layer_offsets(&s, off, nullptr) != Q4_OK) return false;
  memset(out, 0, 4 * sizeof(Phase));
  Phase& a = out[0];   // q, k, v
  a.w0 = wl + off[Q4_PROJ_Q];
  a.x_src = in16 ? static_cast<const void*>(in16) : static_cast<const void*>(w.t2t);
  a.x_kind = in16 ? q4::X_NORM16 : q4::X_TAG32_NORM;
  a.x_ld = s.hidden;
  a.k = s.hidden;
  a.eps = s.eps;
  a.n_rows = s.q_dim + 2 * s.kv_dim;
  a.epi_kind = q4::EPI_F32;
  a.y = last ? w.qkv : nullptr;
  a.x_dbg = last ? w.x : nullptr;
  a.xr_out = w.zt;
  a.yt = w.vtag;
  a.yt_off = s.q_dim + s.kv_dim;
  a.yt_n = s.kv_dim;
  Phase& b = out[1];   // o, input: the context-1 attention of v, output: t1 = z + Wo a
  b.w0 = wl + off[Q4_PROJ_O];
  b.x_src = w.vtag;
  b.x_kind = q4::X_TAG16_ATTN;
  b.xt_n = s.kv_dim;
  b.k = s.q_dim;
  b.head_dim = s.head_dim;
  b.group = (s.q_dim / s.head_dim) / (s.kv_dim / s.head_dim);
  b.n_rows = s.hidden;
  b.epi_kind = q4::EPI_RESID;
  b.res_t = w.zt;
  b.y = last ? w.o : nullptr;
  b.y2 = last ? w.t1 : nullptr;
  b.yt = w.t1t;
  b.yt_n = s.hidden;
  b.x_dbg = last ? w.attn : nullptr;
  b.sync = q4::SYNC_PUBLISH;
  Phase& c = out[2];   // gate | up, input z1 = f16(norm(t1)), output the SiLU-gated product
  c.w0 = wl + off[Q4_PROJ_GATE];
  c.w1 = wl + off[Q4_PROJ_UP];
  c.x_src = w.t1t;
  c.x_kind = q4::X_TAG32_NORM;
  c.k = s.hidden;
  c.eps = s.eps;
  c.n_rows = s.ffn;
  c.epi_kind = q4::EPI_SILU;
  c.y = last ? w.g : nullptr;
  c.y2 = last ? w.u : nullptr;
  c.aux16 = last ? w.act : nullptr;
  c.yt = w.acttag;
  c.yt_n = s.ffn;
  c.x_dbg = last ? w.x2 : nullptr;
  c.xr_out = w.z1t;
  c.sync = q4::SYNC_WAIT;
  Phase& d = out[3];   // down, output t2 = z1 + Wdown act
  d.w0 = wl + off[Q4_PROJ_DOWN];
  d.x_src = w.acttag;
  d.x_kind = q4::X_TAG16;
  d.k = s.ffn;
  d.n_rows = s.hidden;
  d.epi_kind = q4::EPI_RESID;
  d.res_t = w.z1t;
  d.y = last ? w.dn : nullptr;
  d.y2 = last ? w.t2 : nullptr;
  d.yt = w.t2t;
  d.yt_n = s.hidden;
  // Tensor-core engine: the v rows, the only ones the context-1 o phase reads,
  // are the phase's first units, so they are done in the first round of
  // units and the CTAs with a second q|k|v unit do it while the o phase starts.
  if (engine == ENG_TC && !kv && a.n_rows % q4::kTcUnitRows == 0 && (s.q_dim + s.kv_dim) % q4::kTcUnitRows == 0)
    a.row_rot = s.q_dim + s.kv_dim;
  if (kv) {
    // decode attention over the layer's KV cache runs between the q|k|v phase
    // and the o phase (separate launches): q, k, v go out in plain fp32 for
    // every layer, and the o phase reads the attention output, binary16, plain
    a.y = w.qkv;
    a.yt = nullptr;
    b.x_src = w.attn;
    b.x_kind = q4::X_F16;
    b.x_dbg = nullptr;
  }
  for (int i = 0; i < 4; ++i)
    if (!tile_phase(out[i], engine, wl != nullptr)) return false;
  return true;
}

// The closing phase of a tagged program: CTA 0 writes f16(norm(t2)) to the
// caller's hidden-state buffer.
bool final_phase_tagged(const q4_layer_shape& s, uint16_t* h_out, const Work& w, Phase* out, int engine) {
  memset(out, 0, sizeof(Phase));
  out->x_src = w.t2t;
  out->x_kind = q4::X_TAG32_NORM;
  out->k = s.hidden;
  out->eps = s.eps;
  out->n_rows = 0;
  out->epi_kind = q4::EPI_F32;
  out->x_dbg = h_out;
  return tile_phase(*out, engine, false);
}

// Phase program of a whole stack: 4 phases per layer and the closing phase.
bool stack_program(const q4_layer_shape& s, const std::vector<const uint8_t*>& layers, uint16_t* h,
                   const Work& w, std::vector<Phase>& prog, int engine, bool tagged, bool kv = false) {
  const int L = static_cast<int>(layers.size());
  prog.assign(4 * static_cast<size_t>(L) + 1, Phase());
  for (int l = 0; l < L; ++l) {
    const uint16_t* in16 = l == 0 ? h : nullptr;
    if (!(tagged ? layer_phases_tagged(s, layers[l], in16, w, &prog[4 * l], l == L - 1, engine, kv)
                 : layer_phases(s, layers[l], in16, w, &prog[4 * l], engine)))
      return false;
  }
  if (!(tagged ? final_phase_tagged(s, h, w, &prog[4 * L], engine) : final_phase(s, h, w, &prog[4 * L], engine)))
    return false;
  // unit rotation over the whole program, so that any split into launches
  // (fused, per layer, per phase) gives every CTA the same rows; the phase
  // index fixes a tagged program's tags the same way
  int base = 0, gidx = 0;
  for (Phase& ph : prog) {
    ph.base = base;
    ph.gidx = gidx++;
    base += ph.units;
  }
  return true;
}

// Ring and buffer geometry of a tensor-core layer program.
bool tc_layer_geom(const q4_layer_shape& s, TcGeom* g) { return tc_geom({s.hidden, s.q_dim, s.ffn}, g); }

int check_layer_shape_for_engine(const q4_layer_shape& s, int engine) {
  Phase tmp[5];
  Work w;
  memset(&w, 0, sizeof(w));
  if (engine == ENG_TC) {
    // tensor-core engine (tagged programs only): the RMSNorm inputs are staged
    // in registers (hidden <= 8192), values move in runs of 4 that stay
    // within one attention head
    TcGeom g;
    if (s.head_dim % 4 || s.kv_dim % 4 || s.hidden > 8192 || !tc_layer_geom(s, &g)) return Q4_ERR_ARG;
    return layer_phases_tagged(s, nullptr, nullptr, w, tmp, false, ENG_TC) &&
                   final_phase_tagged(s, nullptr, w, &tmp[4], ENG_TC)
               ? Q4_OK
               : Q4_ERR_ARG;
  }
  // CUDA-core engine: a thread's 64 attention columns stay in one head
  if (s.head_dim % q4::kKT) return Q4_ERR_ARG;
  return layer_phases(s, nullptr, nullptr, w, tmp, engine) && final_phase(s, nullptr, w, &tmp[4], engine)
             ? Q4_OK
             : Q4_ERR_ARG;
}

// The batch-1 engine of a decoder or ring: the tensor-core engine unless the
// CUDA-core one is asked for (or the flag barrier, which only it has) or the
// shape does not fit the tensor-core engine.  -1 if the asked engine cannot
// run the shape.
int pick_engine(const q4_layer_shape& s, bool want_tc, bool want_core) {
  if (want_tc && want_core) return -1;
  if (!want_core && check_layer_shape_for_engine(s, ENG_TC) == Q4_OK) return ENG_TC;
  if (want_tc) return -1;
  return check_layer_shape_for_engine(s, ENG_CORE) == Q4_OK ? ENG_CORE : -1;
}

// One layer for a batch of more than one row: the tensor-core product for each
// projection and the glue kernels between them (the same arithmetic as the
// batch-1 engine's phases).  The layer's input is the caller's binary16
// state (first layer) or the previous layer's z in w.x; `out` receives the
// normalised output of the last layer.
int launch_layer_batched(const q4_layer_shape& sh, const uint8_t* wl, int layer, int n_layers, uint16_t* h,
                         const Work& w, int batch, int grid, cudaStream_t s, const cudaEvent_t* chunk = nullptr) {
  size_t off[7];
  if (q4_layer_offsets(&sh, off, nullptr) != Q4_OK) return Q4_ERR_ARG;
  const int H = sh.hidden, Q = sh.q_dim, KV = sh.kv_dim, F = sh.ffn;
  const int nqkv = Q + 2 * KV;
  const int group = (Q / sh.head_dim) / (KV / sh.head_dim);
  // chunk c of the layer block (q|k|v, o, gate|up, down) must have landed before its product
  auto wait = [&](int c) { return chunk ? cudaStreamWaitEvent(s, chunk[c], 0) : cudaSuccess; };
  // resident weights: each launch may start (the products' weight copies)
  // while the previous one finishes; a streamed layer waits on its copy events
  const bool pdl = chunk == nullptr;
  if (layer == 0) Q4_CUDA(q4::glue_norm(h, nullptr, batch, H, sh.eps, w.x, s, pdl));
  Q4_CUDA(wait(0));
  // the v rows of q|k|v also go out as the context-1 attention output a (binary16, gathered per head)
  const q4::MmaGather gather{w.attn, Q + KV, KV, sh.head_dim, group, Q};
  Q4_CUDA(q4::mma_launch(wl + off[Q4_PROJ_Q], w.x, w.qkv, nqkv, H, batch, grid, kWaitLimit, &w.ctl->status, s,
                         nullptr, 0, pdl, &gather));
  Q4_CUDA(wait(1));
  Q4_CUDA(q4::mma_launch(wl + off[Q4_PROJ_O], w.attn, w.o, H, Q, batch, grid, kWaitLimit, &w.ctl->status, s, nullptr,
                         0, pdl));
  Q4_CUDA(q4::glue_resid_norm(w.x, w.o, batch, H, sh.eps, w.t1, w.x2, s, pdl));
  Q4_CUDA(wait(2));
  // gate and up are consecutive in the block: one product of 2 ffn rows, split into g and u
  // (each tile pairs 8 rows of gate with the same 8 rows of up, so its epilogue also forms act)
  Q4_CUDA(q4::mma_launch(wl + off[Q4_PROJ_GATE], w.x2, w.g, 2 * F, H, batch, grid, kWaitLimit, &w.ctl->status, s,
                         w.u, F, pdl, nullptr, w.act));
  Q4_CUDA(wait(3));
  Q4_CUDA(q4::mma_launch(wl + off[Q4_PROJ_DOWN], w.act, w.dn, H, F, batch, grid, kWaitLimit, &w.ctl->status, s,
                         nullptr, 0, pdl));
  // the next layer's z goes to w.x; the last layer's to the caller's buffer
  Q4_CUDA(q4::glue_resid_norm(w.x2, w.dn, batch, H, sh.eps, w.t2, layer + 1 == n_layers ? h : w.x, s, pdl));
  return Q4_OK;
}

bool batched_shape_ok(const q4_layer_shape& s) {
  return s.hidden % 256 == 0 && s.q_dim % 256 == 0 && s.ffn % 256 == 0 && (s.q_dim + 2 * s.kv_dim) > 0 &&
         s.kv_dim % 4 == 0 && s.head_dim % 4 == 0;   // the glue moves 4 values at a time
}

// ---------------------------------------------------------------- batched engine
//
// Batch 2..8: one persistent launch of q4_bt_engine.cu runs the stack (the
// same layer arithmetic as launch_layer_batched, within the product error
// bound of it: the sums run in another order).  The program has 6 phases per
// layer (q|k|v, o, RMSNorm, gate|up, down, RMSNorm) after one RMSNorm of the
// caller's binary16 state.

bool bt_fits(const q4_layer_shape& s, int batch, int* stages, uint32_t* stage_bytes, uint32_t* x_off) {
  const int ks[3] = {s.hidden, s.q_dim, s.ffn};
  return q4::bt_geom(ks, 3, q4::bt_cols(batch), stages, stage_bytes, x_off);
}

bool bt_shape_ok(const q4_layer_shape& s, int n_layers) {
  int st = 0;
  uint32_t sb = 0, xo = 0;
  return 6 * n_layers + 1 <= static_cast<int>(q4::kPhasesPerEpoch) && batched_shape_ok(s) &&
         bt_fits(s, q4::kBtCols, &st, &sb, &xo);
}

bool bt_stack_program(const q4_layer_shape& s, const std::vector<const uint8_t*>& layers, uint16_t* h, const Work& w,
                      std::vector<q4::BtPhase>& prog) {
  size_t off[7];
  if (q4_layer_offsets(&s, off, nullptr) != Q4_OK) return false;
  const int L = static_cast<int>(layers.size());
  const int H = s.hidden, Q = s.q_dim, KV = s.kv_dim, F = s.ffn;
  prog.assign(6 * static_cast<size_t>(L) + 1, q4::BtPhase{});
  int base = 0;
  // an RMSNorm of H values per batch row into z (natural) and the z fragments
  auto form = [&](q4::BtPhase& f, const float* src32, const uint16_t* src16, uint16_t* out16) {
    f.kind = q4::BT_FORM;
    f.k = H;
    f.src32 = src32;
    f.src16 = src16;
    f.ss = w.ss8;
    f.out16 = out16;
    f.out_frag = w.zf;
    f.eps = s.eps;
  };
  // a product phase: 32-row units (16 rows of each matrix of a gate|up pair)
  auto unit = [&](q4::BtPhase& p, int kind, const uint8_t* w0, const uint8_t* w1, int n, int k,
                  const uint8_t* xf) -> bool {
    p.kind = kind;
    p.n_rows = n;
    p.k = k;
    p.x_frag = xf;
    const int rows = kind == q4::BT_SILU ? q4::kTcUnitRows / 2 : q4::kTcUnitRows;
    p.units = (n + rows - 1) / rows;
    p.base = base;
    base += p.units;
    if (!encode_rows(&p.tm0, w0, n, k, rows)) return false;
    return kind != q4::BT_SILU || encode_rows(&p.tm1, w1, n, k, rows);
  };
  form(prog[0], nullptr, h, w.x);
  for (int l = 0; l < L; ++l) {
    const uint8_t* wl = layers[l];
    q4::BtPhase* P = &prog[1 + 6 * static_cast<size_t>(l)];
    // q, k, v: one matrix of q_dim + 2 kv_dim rows; the v rows also go out as
    // the context-1 attention output a (binary16, gathered per head)
    if (!unit(P[0], q4::BT_PLAIN, wl + off[Q4_PROJ_Q], nullptr, Q + 2 * KV, H, w.zf)) return false;
    P[0].y = w.qkv;
    P[0].out16 = w.attn;
    P[0].out_frag = w.af;
    P[0].out_ld = Q;
    P[0].g_lo = Q + KV;
    P[0].g_n = KV;
    P[0].head_dim = s.head_dim;
    P[0].group = (Q / s.head_dim) / (KV / s.head_dim);
    if ((Q + 2 * KV) % q4::kTcUnitRows == 0 && (Q + KV) % q4::kTcUnitRows == 0) {
      // value rows first: a CTA publishes q|k|v (the o phase's input is
      // ready) once its units among the first KV / 32 are stored
      P[0].row_rot = Q + KV;
      P[0].early_units = (KV + q4::kTcUnitRows - 1) / q4::kTcUnitRows;
    }
    // o with the residual base z: t1
    if (!unit(P[1], q4::BT_RESID, wl + off[Q4_PROJ_O], nullptr, H, Q, w.af)) return false;
    P[1].y = w.o;
    P[1].y2 = w.t1;
    P[1].res = w.x;
    P[1].ss = w.ss8;
    form(P[2], w.t1, nullptr, w.x2);
    if (!unit(P[3], q4::BT_SILU, wl + off[Q4_PROJ_GATE], wl + off[Q4_PROJ_UP], F, H, w.zf)) return false;
    P[3].y = w.g;
    P[3].y2 = w.u;
    P[3].out16 = w.act;
    P[3].out_frag = w.actf;
    // down with the residual base z1: t2, normalised into the next layer's z
    // (the last layer's into the caller's buffer)
    if (!unit(P[4], q4::BT_RESID, wl + off[Q4_PROJ_DOWN], nullptr, H, F, w.actf)) return false;
    P[4].y = w.dn;
    P[4].y2 = w.t2;
    P[4].res = w.x2;
    P[4].ss = w.ss8;
    form(P[5], w.t2, nullptr, l + 1 == L ? h : w.x);
  }
  for (size_t i = 0; i < prog.size(); ++i) prog[i].gidx = static_cast<int>(i);
  return true;
}

// Phases [first, first + n) of the batched program in the workspace (stall:
// BtArgs::stall, with its own wait limit).
int launch_bt(const Work& w, int first, int n, int grid, int batch, bool end, const q4_layer_shape& s,
              cudaStream_t st, uint32_t stall = 0, uint32_t wait_limit = kWaitLimit) {
  q4::BtArgs a;
  memset(&a, 0, sizeof(a));
  a.phases = reinterpret_cast<const q4::BtPhase*>(w.prog) + first;
  a.n_phases = n;
  a.ctl = w.ctl;
  a.flags = w.flags;
  a.wait_limit = wait_limit;
  a.stall = stall;
  a.batch = batch;
  a.cols = q4::bt_cols(batch);
  a.end_of_program = end ? 1 : 0;
  if (!bt_fits(s, batch, &a.stages, &a.stage_bytes, &a.x_off)) return Q4_ERR_ARG;
  Q4_CUDA(q4::bt_engine_launch(a, grid, st));
  return Q4_OK;
}

// Launch phases [first_phase, first_phase + n_phases) of the program in the
// workspace; `end` = they include the program's last phase.
// pdl (tensor-core engine): EngineArgs::pdl; with bit 0 the launch is not
// cooperative (it may start while the kernel ahead of it still runs).
int launch_layers(const Work& w, int first_phase, int n_phases, int grid, cudaStream_t s, int engine, bool tagged,
                  bool end, const q4_layer_shape& shape, uint32_t wait_limit = kWaitLimit, int pdl = 0) {
  EngineArgs a;
  memset(&a, 0, sizeof(a));
  a.pdl = engine == ENG_TC ? pdl : 0;
  a.phases = w.prog + first_phase;
  a.n_phases = n_phases;
  a.ctl = w.ctl;
  a.flags = w.flags;
  a.wait_limit = wait_limit;
  a.tagged = tagged ? 1 : 0;
  a.end_of_program = end ? 1 : 0;
  if (tagged) {
    a.stages = tagged_stages(shape);
    a.xbuf_floats = static_cast<int>(tagged_xbuf_bytes(shape) / 4);
  }
  if (engine == ENG_TC) {
    TcGeom g;
    if (!tc_layer_geom(shape, &g)) return Q4_ERR_ARG;
    a.tagged = 1;
    a.stages = g.stages;
    a.stage_bytes = g.stage_bytes;
    a.xbuf_floats = g.xbuf_floats;
    Q4_CUDA(q4::tc_engine_launch(a, grid, (a.pdl & 1) == 0, s));
  } else {
    Q4_CUDA(q4::engine_launch(a, grid, true, s));
  }
  return Q4_OK;
}

int read_status(Control* ctl, cudaStream_t s, int* out) {
  int v = 0;
  Q4_CUDA(cudaMemcpyAsync(&v, &ctl->status, sizeof(int), cudaMemcpyDeviceToHost, s));
  Q4_CUDA(cudaStreamSynchronize(s));
  if (v) Q4_CUDA(cudaMemsetAsync(&ctl->status, 0, sizeof(int), s));
  Q4_CUDA(cudaStreamSynchronize(s));
  *out = v;
  return Q4_OK;
}

}  // namespace

struct q4_decoder {
  q4_layer_shape shape;
  int n_layers = 0, batch = 1, mode = Q4_DEC_FUSED, grid = 0, engine = ENG_CORE;
  bool tagged = false;   // batch-1 CUDA-core engine with tagged words between phases
  // decode attention over per-layer KV caches (q4_decoder_create_kv)
  bool kv = false;
  int capacity = 0;
  std::vector<uint16_t*> kc, vc;
  int* pos = nullptr;
  void* attn_ws = nullptr;
  std::vector<const uint8_t*> layers;
  Work w;
  uint16_t* cur_h = nullptr;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
};

static int decoder_write_program(q4_decoder* d, uint16_t* h, cudaStream_t s) {
  if (d->engine == ENG_BT) {
    std::vector<q4::BtPhase> prog;
    if (!bt_stack_program(d->shape, d->layers, h, d->w, prog)) return Q4_ERR_ARG;
    Q4_CUDA(cudaMemcpyAsync(d->w.prog, prog.data(), prog.size() * sizeof(q4::BtPhase), cudaMemcpyHostToDevice, s));
    d->cur_h = h;
    return Q4_OK;
  }
  if (d->batch > 1) {   // the per-product path passes pointers as launch arguments
    d->cur_h = h;
    if (d->exec) {        // re-capture with the new buffer
      cudaGraphExecDestroy(d->exec);
      cudaGraphDestroy(d->graph);
      d->exec = nullptr;
      d->graph = nullptr;
    }
    return Q4_OK;
  }
  std::vector<Phase> prog;
  if (!stack_program(d->shape, d->layers, h, d->w, prog, d->engine, d->tagged, d->kv)) return Q4_ERR_ARG;
  // pageable source: the runtime stages it before returning, so `prog` may go
  Q4_CUDA(cudaMemcpyAsync(d->w.prog, prog.data(), prog.size() * sizeof(Phase), cudaMemcpyHostToDevice, s));
  d->cur_h = h;
  return Q4_OK;
}

static int decoder_enqueue(q4_decoder* d, cudaStream_t s) {
  const int L = d->n_layers;
  if (d->engine == ENG_BT) {
    if (d->mode == Q4_DEC_FUSED) return launch_bt(d->w, 0, 6 * L + 1, d->grid, d->batch, true, d->shape, s);
    for (int l = 0; l < L; ++l) {   // the first launch also runs the first RMSNorm
      int st = launch_bt(d->w, l == 0 ? 0 : 6 * l + 1, l == 0 ? 7 : 6, d->grid, d->batch, l == L - 1, d->shape, s);
      if (st != Q4_OK) return st;
    }
    return Q4_OK;
  }
  if (d->batch > 1) {
    for (int l = 0; l < L; ++l) {
      int st = launch_layer_batched(d->shape, d->layers[l], l, L, d->cur_h, d->w, d->batch, d->grid, s);
      if (st != Q4_OK) return st;
    }
    return Q4_OK;
  }
  if (d->kv) {
    // layer l: the q|k|v phase; one attention kernel that stores this token's
    // k and v in row *pos of the layer's caches and attends over rows
    // 0..*pos; then one engine launch runs the o, gate|up and down phases of
    // layer l and the q|k|v phase of layer l + 1 (or the closing phase).
    // After the last layer the position advances.  Programmatic dependent
    // launches chain them: an engine launch lets the attention after it start
    // (copying cached keys and values) as its CTAs leave; the attention, once
    // it has waited for that engine launch, lets the next engine launch start
    // (streaming weights) while it computes.
    const q4_layer_shape& sh = d->shape;
    int st = launch_layers(d->w, 0, 1, d->grid, s, d->engine, true, false, sh, kWaitLimit, 2);
    if (st != Q4_OK) return st;
    for (int l = 0; l < L; ++l) {
      const float* qkv = d->w.qkv;
      const q4::AttnAppend app = {qkv + sh.q_dim, qkv + sh.q_dim + sh.kv_dim, d->pos, &d->w.ctl->status, 1};
      Q4_CUDA(q4::attn_launch(qkv, d->kc[l], d->vc[l], d->pos, d->capacity, sh.q_dim / sh.head_dim,
                              sh.kv_dim / sh.head_dim, sh.head_dim, d->w.attn, d->attn_ws, s, 1, &app));
      st = launch_layers(d->w, 4 * l + 1, 4, d->grid, s, d->engine, true, l == L - 1, sh, kWaitLimit,
                         l == L - 1 ? 1 : 3);
      if (st != Q4_OK) return st;
    }
    Q4_CUDA(q4::pos_advance_launch(d->pos, s));
    return Q4_OK;
  }
  if (d->mode == Q4_DEC_FUSED) return launch_layers(d->w, 0, 4 * L + 1, d->grid, s, d->engine, d->tagged, true, d->shape);
  for (int l = 0; l < L; ++l) {   // the last launch also runs the closing phase
    int st = launch_layers(d->w, 4 * l, l == L - 1 ? 5 : 4, d->grid, s, d->engine, d->tagged, l == L - 1, d->shape);
    if (st != Q4_OK) return st;
  }
  return Q4_OK;
}

extern "C" int q4_decoder_create(q4_decoder** out, const q4_layer_shape* shape, const void* const* layer_weights,
                                 int n_layers, int batch, void* workspace, size_t workspace_bytes, int mode,
                                 void* stream) {
  if (!out || !shape_ok(shape) || !layer_weights || n_layers < 1 || !workspace) return Q4_ERR_ARG;
  if (batch < 1 || batch > q4::kMaxBatch) return Q4_ERR_ARG;
  if (4 * n_layers + 1 > static_cast<int>(q4::kPhasesPerEpoch)) return Q4_ERR_ARG;
  const int kind = mode & ~(Q4_DEC_TENSOR_CORE | Q4_DEC_BARRIER | Q4_DEC_CUDA_CORE | Q4_DEC_BATCH_ENGINE);
  if (kind != Q4_DEC_FUSED && kind != Q4_DEC_PER_LAYER) return Q4_ERR_ARG;
  // batch 1: a persistent engine; larger batches: tensor-core products +
  // glue, or (asked for, batch 2..8) the persistent batched engine
  const bool bt = batch > 1 && (mode & Q4_DEC_BATCH_ENGINE);
  if (bt && (batch > q4::kBtCols || !bt_shape_ok(*shape, n_layers))) return Q4_ERR_ARG;
  const int engine = batch == 1 ? pick_engine(*shape, (mode & Q4_DEC_TENSOR_CORE) != 0,
                                              (mode & (Q4_DEC_CUDA_CORE | Q4_DEC_BARRIER)) != 0)
                                : (bt ? ENG_BT : ENG_CORE);
  if (batch == 1 ? engine < 0 : !batched_shape_ok(*shape)) return Q4_ERR_ARG;
  if (!aligned(workspace, 256)) return Q4_ERR_ALIGN;
  for (int l = 0; l < n_layers; ++l) {
    if (!layer_weights[l]) return Q4_ERR_ARG;
    if (!aligned(layer_weights[l], 256)) return Q4_ERR_ALIGN;
  }
  size_t off[Q4_WS_COUNT], need = 0;
  int st = q4_workspace_layout(shape, n_layers, batch, off, &need);
  if (st != Q4_OK) return st;
  if (workspace_bytes < need) return Q4_ERR_OOM;
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev)) != Q4_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  q4_decoder* d = new q4_decoder();
  d->shape = *shape;
  d->n_layers = n_layers;
  d->batch = batch;
  d->mode = kind;
  d->engine = engine;
  d->tagged = batch == 1 && (engine == ENG_TC || (!(mode & Q4_DEC_BARRIER) && tagged_ok(*shape)));
  d->grid = dev->sm_count < q4::kMaxGrid ? dev->sm_count : q4::kMaxGrid;   // one CTA per SM, co-resident
  d->layers.assign(reinterpret_cast<const uint8_t* const*>(layer_weights),
                   reinterpret_cast<const uint8_t* const*>(layer_weights) + n_layers);
  d->w = carve(workspace, off, shape->hidden);
  cudaError_t e = cudaMemsetAsync(workspace, 0, need, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    delete d;
    return cuda_fail(e);
  }
  *out = d;
  return Q4_OK;
}

extern "C" int q4_decoder_create_kv(q4_decoder** out, const q4_layer_shape* shape, const void* const* layer_weights,
                                    int n_layers, const q4_kv_cache* kv, void* workspace, size_t workspace_bytes,
                                    void* stream) {
  if (!out || !shape_ok(shape) || !kv || !kv->k_layers || !kv->v_layers || !kv->pos || !kv->attn_workspace)
    return Q4_ERR_ARG;
  const int n_q = shape->q_dim / shape->head_dim, n_kv = shape->kv_dim / shape->head_dim;
  const size_t aws = q4_attn_workspace_bytes(n_q, n_kv, shape->head_dim, kv->capacity);
  if (aws == 0) return Q4_ERR_ARG;   // bucket or head shape the attention does not take
  if (check_layer_shape_for_engine(*shape, ENG_TC) != Q4_OK) return Q4_ERR_ARG;
  if (kv->attn_workspace_bytes < aws) return Q4_ERR_OOM;
  if (!aligned(kv->pos, 4) || !aligned(kv->attn_workspace, 16)) return Q4_ERR_ALIGN;
  for (int l = 0; l < n_layers; ++l) {
    if (!kv->k_layers[l] || !kv->v_layers[l]) return Q4_ERR_ARG;
    if (!aligned(kv->k_layers[l], 16) || !aligned(kv->v_layers[l], 16)) return Q4_ERR_ALIGN;
  }
  q4_decoder* d = nullptr;
  int st = q4_decoder_create(&d, shape, layer_weights, n_layers, 1, workspace, workspace_bytes,
                             Q4_DEC_PER_LAYER | Q4_DEC_TENSOR_CORE, stream);
  if (st != Q4_OK) return st;
  d->kv = true;
  d->capacity = kv->capacity;
  d->kc.assign(kv->k_layers, kv->k_layers + n_layers);
  d->vc.assign(kv->v_layers, kv->v_layers + n_layers);
  d->pos = kv->pos;
  d->attn_ws = kv->attn_workspace;
  // the attention's arrival counters start at zero (each call leaves them so)
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(kv->attn_workspace, 0, aws, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    q4_decoder_destroy(d);
    return cuda_fail(e);
  }
  *out = d;
  return Q4_OK;
}

static int decoder_capture(q4_decoder* d) {
  cudaStream_t cap = nullptr;
  Q4_CUDA(cudaStreamCreateWithFlags(&cap, cudaStreamNonBlocking));
  cudaError_t e = cudaStreamBeginCapture(cap, cudaStreamCaptureModeThreadLocal);
  int st = Q4_OK;
  if (e == cudaSuccess) {
    st = decoder_enqueue(d, cap);
    cudaGraph_t g = nullptr;
    e = cudaStreamEndCapture(cap, &g);
    if (e == cudaSuccess && st == Q4_OK) {
      d->graph = g;
      e = cudaGraphInstantiateWithFlags(&d->exec, g, 0);
    } else if (g) {
      cudaGraphDestroy(g);
    }
  }
  cudaStreamDestroy(cap);
  if (st != Q4_OK) return st;
  if (e != cudaSuccess) return cuda_fail(e);
  return Q4_OK;
}

static int decoder_prepare(q4_decoder* d, uint16_t* h, cudaStream_t s) {
  if (!d || !h) return Q4_ERR_ARG;
  if (!aligned(h, 16)) return Q4_ERR_ALIGN;
  if (h != d->cur_h) {
    int st = decoder_write_program(d, h, s);
    if (st != Q4_OK) return st;
  }
  return Q4_OK;
}

extern "C" int q4_layer_decode(q4_decoder* d, uint16_t* hidden_io, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int st = decoder_prepare(d, hidden_io, s);
  if (st != Q4_OK) return st;
  if (!d->exec && (st = decoder_capture(d)) != Q4_OK) return st;
  Q4_CUDA(cudaGraphLaunch(d->exec, s));
  return Q4_OK;
}

extern "C" int q4_layer_decode_eager(q4_decoder* d, uint16_t* hidden_io, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int st = decoder_prepare(d, hidden_io, s);
  if (st != Q4_OK) return st;
  return decoder_enqueue(d, s);
}

namespace q4 {

// Run an n_layers stack once, eagerly, with every scratch region inside the
// given workspace (q4_workspace_layout order): phase program written
// stream-ordered from host memory, control block cleared, one persistent
// launch.  Allocates nothing.
int run_stack_in_workspace(const q4_layer_shape* shape, const void* const* layer_weights, int n_layers,
                           uint16_t* hidden_io, void* ws, size_t ws_bytes, cudaStream_t s) {
  if (!shape_ok(shape) || !layer_weights || n_layers < 1 || !hidden_io || !ws) return Q4_ERR_ARG;
  if (4 * n_layers + 1 > static_cast<int>(kPhasesPerEpoch)) return Q4_ERR_ARG;
  const int engine = pick_engine(*shape, false, false);
  if (engine < 0) return Q4_ERR_ARG;
  if (!aligned(hidden_io, 16)) return Q4_ERR_ALIGN;
  for (int l = 0; l < n_layers; ++l) {
    if (!layer_weights[l]) return Q4_ERR_ARG;
    if (!aligned(layer_weights[l], 256)) return Q4_ERR_ALIGN;
  }
  size_t off[Q4_WS_COUNT], need = 0;
  int st = q4_workspace_layout(shape, n_layers, 1, off, &need);
  if (st != Q4_OK) return st;
  if (ws_bytes < need) return Q4_ERR_OOM;
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev)) != Q4_OK) return st;
  const Work w = carve(ws, off, shape->hidden);
  std::vector<const uint8_t*> layers(reinterpret_cast<const uint8_t* const*>(layer_weights),
                                     reinterpret_cast<const uint8_t* const*>(layer_weights) + n_layers);
  std::vector<Phase> prog;
  const bool tagged = engine == ENG_TC || tagged_ok(*shape);
  if (!stack_program(*shape, layers, hidden_io, w, prog, engine, tagged)) return Q4_ERR_ARG;
  Q4_CUDA(cudaMemcpyAsync(w.prog, prog.data(), prog.size() * sizeof(Phase), cudaMemcpyHostToDevice, s));
  // control block, phase flags and tagged words start from zero: earlier calls
  // left their tags, and the epoch starts again at 0
  Q4_CUDA(cudaMemsetAsync(w.ctl, 0, sizeof(Control), s));
  Q4_CUDA(cudaMemsetAsync(w.flags, 0, 2 * kMaxGrid * sizeof(unsigned long long), s));
  Q4_CUDA(cudaMemsetAsync(static_cast<char*>(ws) + off[Q4_WS_XT], 0, off[Q4_WS_COUNT - 1] - off[Q4_WS_XT] +
                                                                       4 * static_cast<size_t>(shape->ffn), s));
  const int grid = dev->sm_count < kMaxGrid ? dev->sm_count : kMaxGrid;
  return launch_layers(w, 0, static_cast<int>(prog.size()), grid, s, engine, tagged, true, *shape);
}

int record_cuda_error(cudaError_t e) { return cuda_fail(e); }

}  // namespace q4

extern "C" int q4_decoder_status(q4_decoder* d, void* stream, int* status_out) {
  if (!d || !status_out) return Q4_ERR_ARG;
  return read_status(d->w.ctl, static_cast<cudaStream_t>(stream), status_out);
}

extern "C" int q4_decoder_debug_stall(q4_decoder* d, uint32_t wait_limit, void* stream, int* status_out) {
  if (!d || !status_out || !d->cur_h || wait_limit < 1) return Q4_ERR_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (d->engine == ENG_BT) {
    // the first layer's q|k|v and o phases alone, every awaited flag tag an
    // epoch ahead: the o phase's input is never released, every wait runs out
    int st = launch_bt(d->w, 1, 2, d->grid, d->batch, false, d->shape, s, q4::kPhasesPerEpoch, wait_limit);
    if (st != Q4_OK) return st;
    if ((st = read_status(d->w.ctl, s, status_out)) != Q4_OK) return st;
    // the launch published flags of this epoch: clear them
    Q4_CUDA(cudaMemsetAsync(d->w.flags, 0, 2 * q4::kMaxGrid * sizeof(unsigned long long), s));
    Q4_CUDA(cudaStreamSynchronize(s));
    return Q4_OK;
  }
  if (!d->tagged) return Q4_ERR_ARG;
  int st;
  if (d->engine == ENG_TC) {
    // the gate|up phase alone first: it waits for the o phase's flags of this
    // epoch, which no CTA has published, and for its tagged input (t1)
    st = launch_layers(d->w, 2, 1, d->grid, s, d->engine, true, false, d->shape, wait_limit);
    if (st != Q4_OK) return st;
  }
  // the o-projection phase alone: its tagged input (v) was written under an
  // earlier epoch, so no word ever carries the tag it waits for
  st = launch_layers(d->w, 1, 1, d->grid, s, d->engine, true, false, d->shape, wait_limit);
  if (st != Q4_OK) return st;
  if ((st = read_status(d->w.ctl, s, status_out)) != Q4_OK) return st;
  // the launch left words under live tags: clear them and the flags
  size_t off[Q4_WS_COUNT];
  if (q4_workspace_layout(&d->shape, d->n_layers, 1, off, nullptr) != Q4_OK) return Q4_ERR_ARG;
  char* base = reinterpret_cast<char*>(d->w.ctl) - off[Q4_WS_CONTROL];
  Q4_CUDA(cudaMemsetAsync(base + off[Q4_WS_XT], 0,
                          off[Q4_WS_COUNT - 1] - off[Q4_WS_XT] + 4 * static_cast<size_t>(d->shape.ffn), s));
  Q4_CUDA(cudaMemsetAsync(d->w.flags, 0, 2 * q4::kMaxGrid * sizeof(unsigned long long), s));
  Q4_CUDA(cudaStreamSynchronize(s));
  return Q4_OK;
}

extern "C" int q4_decoder_tagged(const q4_decoder* d, int* tagged_out) {
  if (!d || !tagged_out) return Q4_ERR_ARG;
  *tagged_out = d->tagged ? 1 : 0;
  return Q4_OK;
}

extern "C" int q4_decoder_destroy(q4_decoder* d) {
  if (!d) return Q4_OK;
  if (d->exec) cudaGraphExecDestroy(d->exec);
  if (d->graph) cudaGraphDestroy(d->graph);
  delete d;
  return Q4_OK;
}

// ===================================================================== streamed layers

struct q4_stream {
  q4_layer_shape shape;
  int n_layers = 0, batch = 1, flags = 0, grid = 0, engine = ENG_CORE;
  bool tagged = false;
  std::vector<const void*> host;
  std::vector<const uint8_t*> resident;   // per layer: device block, or null if streamed
  std::vector<int> slot;                  // per layer: staging buffer (0/1), or -1 if resident
  uint8_t* buf[2] = {nullptr, nullptr};
  size_t layer_bytes = 0;
  size_t chunk_off[5] = {0, 0, 0, 0, 0};  // q|k|v, o, gate|up, down, end
  Work w;
  uint16_t* cur_h = nullptr;
  cudaStream_t copy = nullptr;
  cudaEvent_t loaded[2][4] = {}, freed[2] = {nullptr, nullptr};
  cudaEvent_t start = nullptr, done = nullptr;
  bool used[2] = {false, false};   // a buffer's `freed` event has been recorded
  unsigned long long* stamps = nullptr;   // Q4_STREAM_TIMELINE: [layer][copy begin, copy end,
                                          // compute begin, compute end], globaltimer ns
};

extern "C" int q4_stream_create(q4_stream** out, const q4_layer_shape* shape, const void* const* host_layers,
                                int n_layers, int batch, void* dev_buf0, void* dev_buf1, size_t buf_bytes,
                                void* workspace, size_t workspace_bytes, int flags) {
  return q4_stream_create_ex(out, shape, host_layers, nullptr, n_layers, batch, dev_buf0, dev_buf1, buf_bytes,
                             workspace, workspace_bytes, flags);
}

extern "C" int q4_stream_create_ex(q4_stream** out, const q4_layer_shape* shape, const void* const* host_layers,
                                   const void* const* resident_layers, int n_layers, int batch, void* dev_buf0,
                                   void* dev_buf1, size_t buf_bytes, void* workspace, size_t workspace_bytes,
                                   int flags) {
  const bool single = (flags & Q4_STREAM_SINGLE_BUFFER) != 0;
  if (!out || !shape_ok(shape) || !host_layers || n_layers < 1 || !dev_buf0 || (!dev_buf1 && !single) || !workspace)
    return Q4_ERR_ARG;
  if (batch < 1 || batch > q4::kMaxBatch ||
      (flags & ~(Q4_STREAM_POISON | Q4_STREAM_TENSOR_CORE | Q4_STREAM_CHUNKED | Q4_STREAM_BARRIER |
                 Q4_STREAM_CUDA_CORE | Q4_STREAM_SINGLE_BUFFER | Q4_STREAM_TIMELINE)))
    return Q4_ERR_ARG;
  if (4 * n_layers + 1 > static_cast<int>(q4::kPhasesPerEpoch)) return Q4_ERR_ARG;
  const int engine = batch == 1 ? pick_engine(*shape, (flags & Q4_STREAM_TENSOR_CORE) != 0,
                                              (flags & (Q4_STREAM_CUDA_CORE | Q4_STREAM_BARRIER)) != 0)
                                : ENG_CORE;
  if (batch == 1 ? engine < 0 : !batched_shape_ok(*shape)) return Q4_ERR_ARG;
  if (!aligned(dev_buf0, 256) || (!single && !aligned(dev_buf1, 256)) || !aligned(workspace, 256))
    return Q4_ERR_ALIGN;
  size_t lo[7], layer_bytes = 0;
  q4_layer_offsets(shape, lo, &layer_bytes);
  if (buf_bytes < layer_bytes) return Q4_ERR_OOM;
  for (int l = 0; l < n_layers; ++l) {
    const void* res = resident_layers ? resident_layers[l] : nullptr;
    if (res) {
      if (!aligned(res, 256)) return Q4_ERR_ALIGN;
    } else {
      if (!host_layers[l]) return Q4_ERR_ARG;
      if (!aligned(host_layers[l], 16)) return Q4_ERR_ALIGN;
    }
  }
  size_t off[Q4_WS_COUNT], need = 0;
  int st = q4_workspace_layout(shape, n_layers, batch, off, &need);
  if (st != Q4_OK) return st;
  if (workspace_bytes < need) return Q4_ERR_OOM;
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev)) != Q4_OK) return st;

  q4_stream* r = new q4_stream();
  r->resident.assign(n_layers, nullptr);
  r->slot.assign(n_layers, -1);
  for (int l = 0, si = 0; l < n_layers; ++l) {
    const void* res = resident_layers ? resident_layers[l] : nullptr;
    if (res)
      r->resident[l] = static_cast<const uint8_t*>(res);
    else
      r->slot[l] = single ? 0 : (si++) & 1;   // streamed layers alternate between the two buffers
  }
  r->chunk_off[0] = 0;
  r->chunk_off[1] = lo[Q4_PROJ_O];
  r->chunk_off[2] = lo[Q4_PROJ_GATE];
  r->chunk_off[3] = lo[Q4_PROJ_DOWN];
  r->chunk_off[4] = layer_bytes;
  r->shape = *shape;
  r->n_layers = n_layers;
  r->batch = batch;
  r->flags = flags;
  r->engine = engine;
  r->tagged = batch == 1 && (engine == ENG_TC || (!(flags & Q4_STREAM_BARRIER) && tagged_ok(*shape)));
  r->grid = dev->sm_count < q4::kMaxGrid ? dev->sm_count : q4::kMaxGrid;
  r->host.assign(host_layers, host_layers + n_layers);
  r->buf[0] = static_cast<uint8_t*>(dev_buf0);
  r->buf[1] = single ? nullptr : static_cast<uint8_t*>(dev_buf1);
  r->layer_bytes = layer_bytes;
  r->w = carve(workspace, off, shape->hidden);
  cudaError_t e = cudaStreamCreateWithFlags(&r->copy, cudaStreamNonBlocking);
  for (int i = 0; i < 2 && e == cudaSuccess; ++i) {
    for (int c = 0; c < 4 && e == cudaSuccess; ++c) e = cudaEventCreateWithFlags(&r->loaded[i][c], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&r->freed[i], cudaEventDisableTiming);
  }
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&r->start, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&r->done, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaMemset(workspace, 0, need);
  if (e == cudaSuccess && (flags & Q4_STREAM_TIMELINE)) {
    const size_t sb = 4 * static_cast<size_t>(n_layers) * sizeof(unsigned long long);
    e = cudaMalloc(&r->stamps, sb);
    if (e == cudaSuccess) e = cudaMemset(r->stamps, 0, sb);
  }
  if (e != cudaSuccess) {
    q4_stream_destroy(r);
    return cuda_fail(e);
  }
  *out = r;
  return Q4_OK;
}

extern "C" int q4_stream_layers(q4_stream* r, uint16_t* hidden_io, void* compute_stream, int64_t timeout_us) {
  if (!r || !hidden_io) return Q4_ERR_ARG;
  if (!aligned(hidden_io, 16)) return Q4_ERR_ALIGN;
  cudaStream_t cs = static_cast<cudaStream_t>(compute_stream);
  if (hidden_io != r->cur_h && r->batch == 1) {
    // layer i computes on staging buffer i % 2
    std::vector<const uint8_t*> bufs(r->n_layers);
    for (int i = 0; i < r->n_layers; ++i) bufs[i] = r->resident[i] ? r->resident[i] : r->buf[r->slot[i]];
    std::vector<Phase> prog;
    if (!stack_program(r->shape, bufs, hidden_io, r->w, prog, r->engine, r->tagged)) return Q4_ERR_ARG;
    Q4_CUDA(cudaMemcpyAsync(r->w.prog, prog.data(), prog.size() * sizeof(Phase), cudaMemcpyHostToDevice, cs));
    r->cur_h = hidden_io;
  }
  if (r->batch > 1) r->cur_h = hidden_io;
  // The copy stream may only overwrite a buffer once the compute that last read
  // it (in this call or an earlier one) has finished: its `freed` event.  No
  // wait on the whole previous token, so the next token's first copies overlap
  // the end of this token and the compute of any resident layers before them.
  const size_t n_blocks = r->layer_bytes / q4::kBlockBytes;
  const bool chunked = (r->flags & Q4_STREAM_CHUNKED) != 0;
  const int n_chunks = chunked ? 4 : 1;
  for (int i = 0; i < r->n_layers; ++i) {
    const int b = r->slot[i];
    const uint8_t* wl = b < 0 ? r->resident[i] : r->buf[b];
    unsigned long long* ts = r->stamps ? r->stamps + 4 * static_cast<size_t>(i) : nullptr;
    if (b >= 0) {
      // copy stream: layer i into buffer b once the last layer computed on b has released it
      if (r->used[b]) Q4_CUDA(cudaStreamWaitEvent(r->copy, r->freed[b], 0));
      r->used[b] = true;
      if (ts) Q4_CUDA(q4::stamp_launch(ts + 0, r->copy));
      for (int c = 0; c < n_chunks; ++c) {
        const size_t lo = chunked ? r->chunk_off[c] : 0, hi = chunked ? r->chunk_off[c + 1] : r->layer_bytes;
        Q4_CUDA(cudaMemcpyAsync(r->buf[b] + lo, static_cast<const uint8_t*>(r->host[i]) + lo, hi - lo,
                                cudaMemcpyHostToDevice, r->copy));
        // the copy-end stamp precedes the last chunk's event, so the compute
        // that waits for that event stamps its start after it
        if (ts && c == n_chunks - 1) Q4_CUDA(q4::stamp_launch(ts + 1, r->copy));
        Q4_CUDA(cudaEventRecord(r->loaded[b][c], r->copy));
      }
    }
    const bool last = i == r->n_layers - 1;
    int st = Q4_OK;
    if (r->batch > 1) {
      // batched: each projection waits for its own chunk (or the whole block)
      cudaEvent_t ev[4];
      for (int c = 0; c < 4; ++c) ev[c] = r->loaded[b < 0 ? 0 : b][chunked ? c : 0];
      if (ts) {   // the layer's compute starts once its first chunk (or block) has landed
        if (b >= 0) Q4_CUDA(cudaStreamWaitEvent(cs, ev[0], 0));
        Q4_CUDA(q4::stamp_launch(ts + 2, cs));
      }
      st = launch_layer_batched(r->shape, wl, i, r->n_layers, hidden_io, r->w, r->batch, r->grid, cs,
                                b < 0 ? nullptr : ev);
    } else if (b < 0 || !chunked) {
      if (b >= 0) Q4_CUDA(cudaStreamWaitEvent(cs, r->loaded[b][0], 0));
      if (ts) Q4_CUDA(q4::stamp_launch(ts + 2, cs));
      st = launch_layers(r->w, 4 * i, last ? 5 : 4, r->grid, cs, r->engine, r->tagged, last, r->shape);
    } else {
      // chunked: phase p of the layer starts once chunk p has landed (one launch per phase)
      for (int p = 0; p < 4 && st == Q4_OK; ++p) {
        Q4_CUDA(cudaStreamWaitEvent(cs, r->loaded[b][p], 0));
        if (ts && p == 0) Q4_CUDA(q4::stamp_launch(ts + 2, cs));
        st = launch_layers(r->w, 4 * i + p, (last && p == 3) ? 2 : 1, r->grid, cs, r->engine, r->tagged,
                           last && p == 3, r->shape);
      }
    }
    if (st != Q4_OK) return st;
    if (ts) Q4_CUDA(q4::stamp_launch(ts + 3, cs));
    if (b >= 0) {
      if (r->flags & Q4_STREAM_POISON) Q4_CUDA(q4::poison_launch(r->buf[b], n_blocks, cs));
      Q4_CUDA(cudaEventRecord(r->freed[b], cs));
    }
  }
  // the next call's copies wait on the `freed` events recorded above
  if (timeout_us > 0) {
    Q4_CUDA(cudaEventRecord(r->done, cs));
    const auto t0 = std::chrono::steady_clock::now();
    for (;;) {
      cudaError_t q = cudaEventQuery(r->done);
      if (q == cudaSuccess) break;
      if (q != cudaErrorNotReady) return cuda_fail(q);
      const auto us = std::chrono::duration_cast<std::chrono::microseconds>(std::chrono::steady_clock::now() - t0).count();
      if (us > timeout_us) return Q4_ERR_TIMEOUT;
      std::this_thread::sleep_for(std::chrono::microseconds(20));
    }
  }
  return Q4_OK;
}

extern "C" int q4_stream_status(q4_stream* r, void* compute_stream, int* status_out) {
  if (!r || !status_out) return Q4_ERR_ARG;
  return read_status(r->w.ctl, static_cast<cudaStream_t>(compute_stream), status_out);
}

extern "C" int q4_stream_timeline(q4_stream* r, unsigned long long* out_ns, int n, void* compute_stream) {
  if (!r || !out_ns || !r->stamps || n < 4 * r->n_layers) return Q4_ERR_ARG;
  Q4_CUDA(cudaStreamSynchronize(static_cast<cudaStream_t>(compute_stream)));
  Q4_CUDA(cudaStreamSynchronize(r->copy));
  Q4_CUDA(cudaMemcpy(out_ns, r->stamps, 4 * static_cast<size_t>(r->n_layers) * sizeof(unsigned long long),
                     cudaMemcpyDeviceToHost));
  return Q4_OK;
}

extern "C" int q4_stream_tagged(const q4_stream* r, int* tagged_out) {
  if (!r || !tagged_out) return Q4_ERR_ARG;
  *tagged_out = r->tagged ? 1 : 0;
  return Q4_OK;
}

extern "C" int q4_stream_destroy(q4_stream* r) {
  if (!r) return Q4_OK;
  if (r->copy) cudaStreamSynchronize(r->copy);
  for (int i = 0; i < 2; ++i) {
    for (int c = 0; c < 4; ++c)
      if (r->loaded[i][c]) cudaEventDestroy(r->loaded[i][c]);
    if (r->freed[i]) cudaEventDestroy(r->freed[i]);
  }
  if (r->start) cudaEventDestroy(r->start);
  if (r->done) cudaEventDestroy(r->done);
  if (r->stamps) cudaFree(r->stamps);
  if (r->copy) cudaStreamDestroy(r->copy);
  delete r;
  return Q4_OK;
}

// ===================================================================== decode attention

static bool attn_shape_ok(int capacity, int n_q, int n_kv, int hd) {
  if (capacity < 128 || capacity % 128 || capacity > 65536) return false;
  if (n_kv < 1 || n_q < n_kv || n_q % n_kv || n_q / n_kv > 16) return false;
  return hd >= 64 && hd <= 256 && hd % 64 == 0;
}

extern "C" size_t q4_attn_workspace_bytes(int n_q_heads, int n_kv_heads, int head_dim, int capacity) {
  if (!attn_shape_ok(capacity, n_q_heads, n_kv_heads, head_dim)) return 0;
  return q4::attn_workspace_bytes(n_q_heads, n_kv_heads, head_dim, capacity);
}

extern "C" int q4_attn_decode(const float* q, const uint16_t* k_cache, const uint16_t* v_cache, const int* ctx_len,
                              int capacity, int n_q_heads, int n_kv_heads, int head_dim, uint16_t* out,
                              void* workspace, size_t workspace_bytes, void* stream) {
  if (!q || !k_cache || !v_cache || !ctx_len || !out || !workspace) return Q4_ERR_ARG;
  if (!attn_shape_ok(capacity, n_q_heads, n_kv_heads, head_dim)) return Q4_ERR_ARG;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
      !aligned(workspace, 16) || !aligned(ctx_len, 4))
    return Q4_ERR_ALIGN;
  if (workspace_bytes < q4_attn_workspace_bytes(n_q_heads, n_kv_heads, head_dim, capacity)) return Q4_ERR_OOM;
  DeviceInfo* dev = nullptr;
  int st = device_info(&dev);
  if (st != Q4_OK) return st;
  Q4_CUDA(q4::attn_launch(q, k_cache, v_cache, ctx_len, capacity, n_q_heads, n_kv_heads, head_dim, out,
                          workspace, static_cast<cudaStream_t>(stream)));
  return Q4_OK;
}

extern "C" int q4_kv_append(const float* k, const float* v, uint16_t* k_cache, uint16_t* v_cache, const int* pos,
                            int capacity, int kv_dim, void* stream) {
  if (!k || !v || !k_cache || !v_cache || !pos || capacity < 1 || kv_dim < 1) return Q4_ERR_ARG;
  if (!aligned(pos, 4)) return Q4_ERR_ALIGN;
  Q4_CUDA(q4::kv_append_launch(k, v, k_cache, v_cache, pos, capacity, kv_dim, static_cast<cudaStream_t>(stream)));
  return Q4_OK;
}
