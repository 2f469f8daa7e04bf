/*
 * q4.h -- C ABI of libq4.so: the decode-step matrix-vector product over
 * GGUF Q4_0 weights on one GB300 GPU (sm_103a), run one matrix, one decoder
 * layer stack, or a stack streamed from pinned host memory.
 *
 * Sources of the operations (the pages this library follows):
 *   - "PIPO: Pipelined Offloading for Efficient Inference on Consumer
 *     Devices" (paper summary page), Method: "Computation optimization"
 *     (matrix-vector products computed directly on 4-bit weights, without
 *     dequantisation, at small batch), "Automatic configuration" (that kernel
 *     is used for batch sizes below 16), "Offloading architecture" and
 *     "Pipeline design" (only one or a few layers resident, per-layer
 *     schedule: load the next layer, synchronise the current one, compute),
 *     "Two pipeline modes" (performance-optimised mode keeps two layers in
 *     GPU memory), "Data transfer suite" (a layer's tensors merged into one
 *     buffer and one transfer).
 *   - "PipeLLM: Faster Local LLM Inference Than llama.cpp via System-Level
 *     Optimizations" (forum post), "Layer 1: CUDA Graph Compilation" (the
 *     decode loop captured as a static graph) and "Layer 2: Asynchronous
 *     Weight Prefetching" (two CUDA streams, a fixed pinned buffer pool,
 *     double-buffered weight staging).
 *   - The GGUF file format both pages load (PipeLLM, compatibility
 *     paragraph).  Q4_0 block: 32 weights as a little-endian IEEE binary16
 *     scale d followed by 16 code bytes; byte j holds element j in its low
 *     nibble and element j+16 in its high nibble; weight = (q - 8) * d.
 *     18 bytes per block, blocks of a row consecutive, rows consecutive.
 *
 * Conventions for every call:
 *   - Pointers named "device" are CUDA device (or managed) memory of the
 *     current device; the caller allocates and owns every buffer.  Handles
 *     own only CUDA streams, events and graphs, which destroy() releases.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default).
 *     Calls are asynchronous on it unless stated otherwise.
 *   - Return value: Q4_OK or a negative Q4_ERR_* code; nothing is launched
 *     when an argument check fails.  A CUDA error seen by the library is
 *     kept for q4_last_cuda_error().  Kernels never trap: a wait that runs
 *     out sets a status bit that q4_device_status() / the *_status() calls
 *     report, and the kernel returns.
 *   - Weight, x and y pointers must be 16-byte aligned (Q4_ERR_ALIGN).
 *   - k must be a multiple of 32 (one block); the streaming kernel needs k in
 *     {256, 512, 1024} or a multiple of 2048 up to 28672; other k use a
 *     plain (slower) kernel.
 *   - x is binary16 [batch][k] row-major, y is fp32 [batch][n] row-major and
 *     is overwritten, not accumulated.  1 <= batch <= 16.
 *   - Accuracy: |y - sum_k w*x| <= 1e-3 * sum_k |w*x| + 1e-5 per element;
 *     every product (q - 8) * x is formed exactly, so a block whose codes are
 *     all 8 contributes exactly zero.
 */
#ifndef Q4_H
#define Q4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ----------------------------------------------------------------- status */

#define Q4_OK 0
#define Q4_ERR_ARG (-1)      /* bad size, null pointer, unsupported shape */
#define Q4_ERR_ALIGN (-2)    /* pointer not 16-byte aligned */
#define Q4_ERR_CUDA (-3)     /* a CUDA runtime call failed; see q4_last_cuda_error() */
#define Q4_ERR_TIMEOUT (-4)  /* a host-side wait ran out */
#define Q4_ERR_OOM (-5)      /* the caller's workspace is too small */
#define Q4_ERR_DEVICE (-6)   /* a kernel reported a failed wait in its status word */

/* Text for a status code (static storage). */
const char *q4_status_string(int status);

/* The last cudaError_t value the library saw (0 if none); reading clears it. */
int q4_last_cuda_error(void);

/* Library version: major * 10000 + minor * 100 + patch. */
int q4_version(void);

/* Bytes of one row-major Q4_0 matrix with n rows and k columns: n * k / 32 * 18. */
size_t q4_matrix_bytes(int n, int k);

/* ------------------------------------------------------- one product */

/* Kernel choice for q4_gemv_ex. */
#define Q4_KERNEL_AUTO 0     /* what q4_gemv uses */
#define Q4_KERNEL_STREAM 1   /* persistent TMA-ring kernel, CUDA-core exact products (batch 1) */
#define Q4_KERNEL_SIMPLE 2   /* one warp per row, plain loads (any k % 32 == 0, any batch) */
#define Q4_KERNEL_MMA 3      /* persistent TMA-ring kernel, tensor-core products (batch 1..16) */
#define Q4_KERNEL_TC 4       /* persistent tensor-core engine, one phase (batch 1, k % 256 == 0 and
                                k <= 2048 or k % 2048 == 0, k <= 30720); what q4_gemv uses at
                                batch 1 for those widths above 64 MB of weights */
#define Q4_KERNEL_ONESHOT 5  /* one-shot tensor-core kernel for a single product: a CTA per 16
                                rows, the whole tile fetched at once by tensor or bulk copies
                                (batch 1, k % 512 == 0, shared memory within 231424 bytes: k <=
                                20992); what q4_gemv uses at batch 1 for those widths up to 64 MB
                                of weights */

/* Flag for q4_gemv_ex's kernel argument (OR it in): a chained call.  A
 * one-shot product launched with it may start before the kernel before it on
 * the stream has ended: it fetches its weights, reads x and computes while
 * that kernel finishes, and stores y only after it (programmatic stream
 * serialisation), so that back-to-back independent products overlap.  The
 * caller promises that no kernel it enqueued since the last q4_gemv call on
 * the stream writes this call's w or x (their reads may run ahead of that
 * kernel's end); the library itself never starts a call early whose w or x
 * overlap the y of a one-shot product on the same stream that may still be
 * running, and a product that another kernel computes on the stream ends that
 * list (the next chained call starts after it).  Without the flag every call
 * starts after the work before it, as usual.  Other kernels ignore the flag. */
#define Q4_GEMV_CHAIN 0x100

/*
 * y[b][n] = sum_k W[n][k] * x[b][k], W dequantisation-free from its Q4_0 blocks
 * (PIPO summary, Method, "Computation optimization").
 *   w      device, Q4_0 [n][k/32] blocks (q4_matrix_bytes(n, k) bytes), read only
 *   x      device, binary16 [batch][k], read only
 *   y      device, fp32 [batch][n], written
 *   n      rows (>= 1); k columns (>= 32, multiple of 32); 1 <= batch <= 16
 * Errors: Q4_ERR_ARG, Q4_ERR_ALIGN, Q4_ERR_CUDA (launch failure).
 */
int q4_gemv(const void *w, const uint16_t *x, float *y, int n, int k, int batch, void *stream);

/* q4_gemv with an explicit kernel (Q4_KERNEL_*); Q4_ERR_ARG if that kernel
 * cannot run the shape (see the conventions above). */
int q4_gemv_ex(const void *w, const uint16_t *x, float *y, int n, int k, int batch, int kernel,
               void *stream);

/* Status bits set by q4_gemv kernels whose internal waits ran out since the
 * last call (0 = none); synchronises the device and clears the bits. */
int q4_device_status(void);

/*
 * Tracing: the phase timeline of the tensor-core engine's last launches, in
 * the timeline build of the library only (libq4_tl.so, compiled with
 * Q4_TIMELINE; the Python module weight_streaming_q4_gb300.timeline builds,
 * runs and summarises it).  For CTA c (< 256), program phase p (< 64) and event
 * e (< 6), out[(c * 64 + p) * 6 + e] = the GPU's global timer (ns) when
 *   e = 0 the CTA's consumers reached the phase, 1 passed their barrier,
 *       2 had staged the phase's input, 3 handed their last unit to the
 *       epilogue, 4 the epilogue stored the last unit, 5 the producer issued
 *       the phase's last copy (0 = the event did not happen).
 *   out, n   host, n >= 256 * 64 * 6 values
 *   clear    nonzero: zero the timeline after the copy
 * Synchronous.  Errors: Q4_ERR_ARG (n too small, or a build without the
 * timeline), Q4_ERR_CUDA.
 */
int q4_timeline_read(unsigned long long *out, size_t n, int clear);

/*
 * Debug: w_out[n][k] = (q - 8) * d as fp32 for every weight (exact: every
 * such value is a float).  Checks the block layout bit for bit.
 *   w      device, Q4_0 [n][k/32] blocks; w_out device, fp32 [n][k]
 * Errors: Q4_ERR_ARG, Q4_ERR_ALIGN, Q4_ERR_CUDA.
 */
int q4_dequant_debug(const void *w, float *w_out, int n, int k, void *stream);

/* ------------------------------------------------------- decoder layers */

/*
 * Shape of one Llama-shaped decoder layer.  The pages name the projections
 * only by the model families they run, so the glue between them is this
 * library's reading, per batch row, with z the layer's normalised binary16
 * input (RMSNorm with unit weight: norm(t) = t / sqrt(mean(t^2) + eps)):
 *   q, k, v = Wq z, Wk z, Wv z                                       (fp32)
 *   a   = f16(v of the value head each query head is grouped with)
 *         (attention over a context of one token: softmax of one score is 1,
 *          rotary position 0 is the identity)
 *   t1  = z + Wo a            (fp32)      z1  = f16(norm(t1))
 *   act = f16(silu(Wgate z1) * (Wup z1))
 *   t2  = z1 + Wdown act      (fp32)      next layer's z = f16(norm(t2))
 * The residual sum is normalised after each add (post-norm): the specified
 * synthetic weights have a nonzero mean, and a pre-norm residual stream
 * overflows binary16 within two 8B-shaped layers.  The first layer's z is
 * f16(norm(h)) of the caller's hidden state h; after the last layer the
 * caller's buffer receives the last z.
 */
typedef struct q4_layer_shape {
  int hidden;     /* model width (4096 for 8B, 8192 for 70B) */
  int q_dim;      /* rows of Wq, columns of Wo */
  int kv_dim;     /* rows of Wk and Wv */
  int ffn;        /* rows of Wgate and Wup, columns of Wdown */
  int head_dim;   /* 128 */
  float eps;      /* RMSNorm epsilon (1e-5) */
} q4_layer_shape;

#define Q4_PROJ_Q 0
#define Q4_PROJ_K 1
#define Q4_PROJ_V 2
#define Q4_PROJ_O 3
#define Q4_PROJ_GATE 4
#define Q4_PROJ_UP 5
#define Q4_PROJ_DOWN 6

/*
 * Layout of one merged layer block (PIPO summary, "Data transfer suite":
 * data merging): the seven projections q, k, v, o, gate, up, down, each a
 * row-major Q4_0 matrix, back to back in that order.  offsets[7] receives
 * each projection's byte offset and *layer_bytes the block's size.
 * Errors: Q4_ERR_ARG (null or inconsistent shape).
 */
int q4_layer_offsets(const q4_layer_shape *shape, size_t offsets[7], size_t *layer_bytes);

/* Regions of a decoder or stream workspace (index into offsets[]). */
#define Q4_WS_CONTROL 0   /* barrier count and status word (zeroed at create) */
#define Q4_WS_PROGRAM 1   /* phase descriptors */
#define Q4_WS_QKV 2       /* fp32 [batch][q_dim + 2 kv_dim]: q, k, v of the last layer run */
#define Q4_WS_O 3         /* fp32 [batch][hidden]: Wo a */
#define Q4_WS_GATE 4      /* fp32 [batch][ffn] */
#define Q4_WS_UP 5        /* fp32 [batch][ffn] */
#define Q4_WS_DOWN 6      /* fp32 [batch][hidden] */
#define Q4_WS_ACT 7       /* binary16 [batch][ffn] */
#define Q4_WS_X 8         /* binary16 [batch][hidden]: z, the layer's normalised input */
#define Q4_WS_ATTN 9      /* binary16 [batch][q_dim]: attention output a */
#define Q4_WS_X2 10       /* binary16 [batch][hidden]: z1 = f16(norm(t1)) */
#define Q4_WS_T1 11       /* fp32 [batch][hidden]: t1 = z + Wo a */
#define Q4_WS_T2 12       /* fp32 [batch][hidden]: t2 = z1 + Wdown act */
#define Q4_WS_FLAGS 13    /* u64 [2][256] per-CTA end-of-phase flags (tag, sum of squares), then
                             fp32 [2][256] per-CTA sums of squares of t1 and t2 */
#define Q4_WS_XT 14       /* batch-1 engine inputs: t1 then t2 as tagged words (24 * hidden bytes:
                             t1, t2 as 64-bit {fp32, tag}, z, z1 as 32-bit {binary16, tag}), or,
                             with Q4_DEC_BARRIER, fp32 t1 / t2 slice-transposed */
#define Q4_WS_VT 15       /* batch-1 engine input: v as 32-bit tagged words, or fp32 slice-transposed */
#define Q4_WS_ACTT 16     /* batch-1 engine input: act as 32-bit tagged words, or binary16
                             slice-transposed */
#define Q4_WS_COUNT 17

/*
 * Byte offsets of the workspace regions for a decoder or a stream ring of
 * n_layers layers and the total size needed.  The intermediate regions hold
 * the values of the last layer run (for checks).
 * Errors: Q4_ERR_ARG.
 */
int q4_workspace_layout(const q4_layer_shape *shape, int n_layers, int batch,
                        size_t offsets[Q4_WS_COUNT], size_t *total_bytes);

typedef struct q4_decoder q4_decoder;

#define Q4_DEC_FUSED 0      /* the whole stack is one persistent launch (one graph node) */
#define Q4_DEC_PER_LAYER 1  /* one launch per layer (one graph node per layer) */
#define Q4_DEC_TENSOR_CORE 2  /* or-ed into the mode: batch 1 must run the tensor-core engine
                                 (the default whenever the shape allows it; Q4_ERR_ARG if not) */
#define Q4_DEC_BARRIER 4    /* or-ed into the mode: batch 1 runs the CUDA-core engine meeting at a
                               flag barrier after every phase instead of passing tagged words */
#define Q4_DEC_CUDA_CORE 8  /* or-ed into the mode: batch 1 runs the exact CUDA-core engine
                               (tagged words between phases when the shape allows) instead of
                               the tensor-core engine.  The engines and the two phase
                               synchronisations agree within the product error bound, not bit
                               for bit */
#define Q4_DEC_BATCH_ENGINE 16  /* or-ed into the mode: batch 2..8 runs the persistent batched
                                   tensor-core engine (the whole stack in one launch, phases
                                   meeting at flag barriers) instead of one product launch per
                                   projection; Q4_ERR_ARG for shapes it does not take.  The two
                                   agree within the product error bound, not bit for bit; on a
                                   GB300 the per-product launches are the faster */

/*
 * Create a decoder over n_layers HBM-resident layers and capture its CUDA
 * graph (PipeLLM, "Layer 1: CUDA Graph Compilation").
 *   shape          layer shape; layer_weights[i] = device pointer of layer
 *                  i's merged block (q4_layer_offsets layout), 256-byte aligned
 *   n_layers       1..1023; batch: 1 <= batch <= 16
 *   workspace      device, >= q4_workspace_layout() bytes, 256-byte aligned;
 *                  owned by the caller, must outlive the decoder
 *   mode           Q4_DEC_FUSED or Q4_DEC_PER_LAYER, optionally | Q4_DEC_TENSOR_CORE,
 *                  | Q4_DEC_CUDA_CORE or | Q4_DEC_BARRIER.
 *                  Batch 1 runs one persistent engine: tensor-core by default
 *                  (hidden, q_dim, ffn widths of Q4_KERNEL_TC, hidden <= 8192,
 *                  kv_dim and head_dim multiples of 4), else the CUDA-core one
 *                  (head_dim % 64 == 0 and the widths of Q4_KERNEL_STREAM);
 *                  batch 2..16 runs one tensor-core product launch per
 *                  projection with glue launches between them (hidden, q_dim,
 *                  ffn multiples of 256; kv_dim, head_dim multiples of 4), or,
 *                  with Q4_DEC_BATCH_ENGINE at batch 2..8, the persistent
 *                  batched engine: the whole stack in one launch
 *                  (Q4_DEC_FUSED) or one per layer, the batch rows as the
 *                  columns of the instruction, each stage carrying its weights
 *                  and its chunk of the input (hidden, q_dim, ffn of the widths
 *                  of Q4_KERNEL_TC, n_layers <= 682).  In every case the rows
 *                  of a batch do not affect one another
 *   stream         used for the workspace initialisation (synchronised)
 * Errors: Q4_ERR_ARG, Q4_ERR_ALIGN, Q4_ERR_OOM (workspace too small), Q4_ERR_CUDA.
 */
int q4_decoder_create(q4_decoder **out, const q4_layer_shape *shape, const void *const *layer_weights,
                      int n_layers, int batch, void *workspace, size_t workspace_bytes, int mode,
                      void *stream);

/*
 * Run all layers once on hidden_io (device, binary16 [batch][hidden]: read as
 * the first layer's input, overwritten with the last layer's normalised
 * output) by replaying the captured graph on `stream`.  The first call with
 * a new hidden_io pointer rewrites the phase descriptors (stream-ordered).
 * Errors: Q4_ERR_ARG, Q4_ERR_ALIGN, Q4_ERR_CUDA.
 */
int q4_layer_decode(q4_decoder *dec, uint16_t *hidden_io, void *stream);

/* The same launches as q4_layer_decode, issued directly (no graph). */
int q4_layer_decode_eager(q4_decoder *dec, uint16_t *hidden_io, void *stream);

/* Status word of the decoder's kernels (synchronises `stream`): 0 = every
 * wait completed; otherwise bit flags, clears it.  Bits: 1 a phase flag never
 * came, 2 a weight copy never landed, 4 a ring stage was never released, 8 a
 * copy was still in flight at exit, 16 a tagged input word never carried its
 * tag, 32 a KV decoder's position was outside its bucket.  Results of a call
 * that set a bit are not valid.  Errors: Q4_ERR_CUDA. */
int q4_decoder_status(q4_decoder *dec, void *stream, int *status_out);

/* *tagged_out = 1 if the decoder's batch-1 engine passes tagged words
 * between phases (always for the tensor-core engine), 0 if it meets at a flag
 * barrier after every phase (or runs another batch).  Host only.
 * Errors: Q4_ERR_ARG. */
int q4_decoder_tagged(const q4_decoder *dec, int *tagged_out);

/*
 * Failure-detection hook for tests (tagged decoders and the batched engine,
 * after one decode call): runs the decoder's o-projection phase alone with a
 * wait limit of wait_limit polls.  Its tagged input was written under an
 * earlier epoch, so no word ever carries the tag it waits for: every wait
 * gives up after wait_limit polls, the kernel sets status bit 16 (a tagged
 * input never arrived) and returns.  The tensor-core engine first runs the
 * gate|up phase alone: its wait for the o phase's flags of the current epoch
 * (never published) gives up too (bit 1).  The batched engine runs its first
 * layer's q|k|v and o phases with every awaited flag tag one epoch ahead:
 * the flag waits give up (status bit 1) and the stage waits behind them
 * (bits 2 and 8).  The call synchronises `stream`, reads and clears the status
 * word into *status_out, and clears the tagged words (the flags) so that the
 * next decode call runs normally.  Errors: Q4_ERR_ARG (neither kind of
 * decoder, no decode call yet, wait_limit 0), Q4_ERR_CUDA.
 */
int q4_decoder_debug_stall(q4_decoder *dec, uint32_t wait_limit, void *stream, int *status_out);

int q4_decoder_destroy(q4_decoder *dec);

/* ------------------------------------------------------- decoder with KV caches */

/*
 * Per-layer KV caches for decoding a sequence (the decode loop PipeLLM
 * captures per context-length bucket, "Layer 1: CUDA Graph Compilation";
 * the per-layer KV cache PIPO moves with the layer, Method, "Offloading
 * architecture").  All device memory, owned by the caller.
 *   capacity     the bucket: positions per cache (a multiple of 128, as for
 *                q4_attn_decode)
 *   k_layers[l], v_layers[l]   binary16 [capacity][kv_dim] caches of layer l,
 *                16-byte aligned
 *   pos          device int: the position of the next token (0 for the first);
 *                every decode call reads it and advances it by one
 *   attn_workspace, attn_workspace_bytes   >= q4_attn_workspace_bytes(n_q,
 *                n_kv, head_dim, capacity); zeroed by q4_decoder_create_kv and
 *                left reusable by every call
 */
typedef struct q4_kv_cache {
  int capacity;
  uint16_t *const *k_layers;
  uint16_t *const *v_layers;
  int *pos;
  void *attn_workspace;
  size_t attn_workspace_bytes;
} q4_kv_cache;

/*
 * A batch-1 decoder whose layers attend over their KV caches instead of the
 * context-1 stand-in: per layer, the q|k|v product; the token's k and v
 * rounded to binary16 into row *pos of the layer's caches (q4_kv_append); the
 * attention of every query head over rows 0..*pos (q4_attn_decode, output
 * binary16); the o, gate|up and down products as in q4_layer_decode.  After
 * the last layer *pos advances by one.  With *pos = 0 the result equals the
 * context-1 decoder's bit for bit.  Keys are cached without a position
 * encoding (the library applies none).  The tensor-core engine runs the
 * products (shape as for Q4_DEC_TENSOR_CORE; head_dim 64, 128, 192 or 256);
 * each layer is two engine launches around the two attention kernels, and
 * q4_layer_decode replays them from one CUDA graph (one graph serves every
 * position of the bucket: the kernels read *pos).  *pos must stay below
 * capacity: otherwise the cache row is not written, the attention covers the
 * capacity only, and the decoder's status word (q4_decoder_status) gets bit
 * 32; the caller moves to a larger bucket before that.
 *   other arguments as for q4_decoder_create (batch 1)
 * Errors: Q4_ERR_ARG, Q4_ERR_ALIGN, Q4_ERR_OOM, Q4_ERR_CUDA.
 */
int q4_decoder_create_kv(q4_decoder **out, const q4_layer_shape *shape, const void *const *layer_weights,
                         int n_layers, const q4_kv_cache *kv, void *workspace, size_t workspace_bytes,
                         void *stream);

/* ------------------------------------------------------- decoder without allocation */

/*
 * For callers that cannot allocate device memory -- code running where
 * cudaMalloc is not allowed or not wanted (inside an allocator's own
 * callbacks, in a process whose device memory is fully reserved up front,
 * or a plugin host that hands out no workspace) -- the decoder stack can run
 * with its scratch (phase program, control block, intermediate activations)
 * in one array that the library holds in static device memory.  The paper
 * has no counterpart to this entry point; it is a deployment convenience.
 *
 * The array is Q4_NOALLOC_SCRATCH_BYTES (1 MiB) on every GPU that loads the
 * library, held until the process exits; it fits a batch-1 stack of the
 * 70B shape with up to 106 layers (an 8B-shaped one with 304).  Larger
 * stacks return Q4_ERR_OOM.
 * The first call on a device looks up the array's device address on that
 * device (make that first call before any stream capture).  Every call
 * shares the one array and overwrites it, so calls whose work overlaps on
 * the GPU (different streams, or different threads without ordering) race:
 * issue them on one stream.  The control block is cleared by every call.
 * Nothing is allocated: no cudaMalloc, cudaFree or allocating library call.
 * The call copies its phase program from host memory that lives only for the
 * call, so it runs eagerly: on a stream that is being captured it returns
 * Q4_ERR_ARG and enqueues nothing.
 *   shape, layer_weights, n_layers   as for q4_decoder_create (batch 1)
 *   hidden_io  device, binary16 [1][hidden], updated as by q4_layer_decode
 *   stream     the work is enqueued asynchronously on it (eager launches)
 * Errors: Q4_ERR_ARG, Q4_ERR_ALIGN, Q4_ERR_OOM (stack too large for the
 * array), Q4_ERR_CUDA.
 */
#define Q4_NOALLOC_SCRATCH_BYTES (1u << 20)
int q4_layer_decode_noalloc(const q4_layer_shape *shape, const void *const *layer_weights, int n_layers,
                            uint16_t *hidden_io, void *stream);

/* Status word of the kernels of the last q4_layer_decode_noalloc call on the
 * current device (bits as for q4_decoder_status; 0 = every wait completed):
 * synchronises `stream`, reads the word from the static array's control
 * block and clears it.  Read it after each call: the next call clears it.
 * Errors: Q4_ERR_ARG, Q4_ERR_CUDA. */
int q4_noalloc_status(void *stream, int *status_out);

/* Size in bytes of the static scratch array used by q4_layer_decode_noalloc. */
size_t q4_noalloc_scratch_bytes(void);

/* ------------------------------------------------------- decode attention */

/*
 * Decode attention of one token over a binary16 KV cache, the work PipeLLM
 * captures per context-length bucket ("Layer 1: CUDA Graph Compilation":
 * buckets of 512, 1024, 2048, 4096 positions) over the per-layer KV cache
 * PIPO moves with the layer (PIPO summary, Method, "Offloading
 * architecture").  For query head h and its value head g = h / (n_q/n_kv):
 *   s_t = q[h] . k[t][g] / sqrt(head_dim) for t < ctx,
 *   out[h] = f16(sum_t softmax(s)_t v[t][g]),
 * scores and weights in fp32: one thread-block cluster per value head (16
 * CTAs where the GPU schedules clusters that large, else 8) splits the context,
 * each CTA keeps a running max-shifted softmax state over rounds of up to 256
 * positions, and the states are combined through distributed shared memory in
 * rank order (a fixed order).  Keys are stored as the model uses them (any
 * position encoding already applied).
 *   q                 device, fp32 [n_q_heads * head_dim]
 *   k_cache, v_cache  device, binary16 [capacity][n_kv_heads * head_dim], read only
 *   ctx_len           device int, the positions in use (clamped to 1..capacity);
 *                     read by the kernels, so a graph captured for one bucket
 *                     serves every length up to its capacity
 *   capacity          the bucket: a multiple of 128, at most 65536
 *   n_q_heads, n_kv_heads  n_q a multiple of n_kv, at most 16 query heads per value head
 *   head_dim          64, 128, 192 or 256
 *   out               device, binary16 [n_q_heads * head_dim], written
 *   workspace         device, >= q4_attn_workspace_bytes(...) (16 bytes, reserved:
 *                     the partial results stay in the cluster's shared memory)
 * Pointers 16-byte aligned (ctx_len 4).  Asynchronous on `stream`.
 * Errors: Q4_ERR_ARG, Q4_ERR_ALIGN, Q4_ERR_OOM, Q4_ERR_CUDA.
 */
int q4_attn_decode(const float *q, const uint16_t *k_cache, const uint16_t *v_cache, const int *ctx_len,
                   int capacity, int n_q_heads, int n_kv_heads, int head_dim, uint16_t *out,
                   void *workspace, size_t workspace_bytes, void *stream);

/* Bytes of the workspace of q4_attn_decode (0 for invalid sizes). */
size_t q4_attn_workspace_bytes(int n_q_heads, int n_kv_heads, int head_dim, int capacity);

/* Store the current token's key and value (fp32 [kv_dim], device) as
 * binary16 at row *pos (device int, ignored outside 0..capacity-1) of the
 * caches.  Errors: Q4_ERR_ARG, Q4_ERR_ALIGN, Q4_ERR_CUDA. */
int q4_kv_append(const float *k, const float *v, uint16_t *k_cache, uint16_t *v_cache, const int *pos,
                 int capacity, int kv_dim, void *stream);

/* ------------------------------------------------------- streamed layers */

typedef struct q4_stream q4_stream;

#define Q4_STREAM_POISON 1   /* after a layer's compute, overwrite its staging buffer's
                                scales with NaN before the next copy lands (race check) */
#define Q4_STREAM_TENSOR_CORE 2 /* batch 1 must run the tensor-core engine (as Q4_DEC_TENSOR_CORE) */
#define Q4_STREAM_CHUNKED 4   /* copy each streamed layer as four chunks (q|k|v, o, gate|up,
                                 down), one event each; each of the layer's products starts as
                                 soon as its own chunk has landed (PIPO, "Data transfer suite":
                                 blockwise transfer) instead of after the whole block */
#define Q4_STREAM_BARRIER 8   /* as Q4_DEC_BARRIER for the ring's batch-1 engine */
#define Q4_STREAM_CUDA_CORE 16  /* as Q4_DEC_CUDA_CORE for the ring's batch-1 engine */
#define Q4_STREAM_SINGLE_BUFFER 32 /* memory-efficient mode (PIPO, Method, "Two pipeline modes"):
                                   one staging buffer (dev_buf0; dev_buf1 may be null); the copy
                                   of a streamed layer starts once the compute of the layer before
                                   it has released the buffer.  With Q4_STREAM_CHUNKED a layer's
                                   products still start as their own chunks land */
#define Q4_STREAM_TIMELINE 64 /* record per layer the GPU's global timer (ns) when the copy
                                 stream starts and ends the layer's copy and when the compute
                                 stream starts and ends its compute (one-thread stamp kernels on
                                 both streams); read with q4_stream_timeline */

/*
 * Create a double-buffered copy/compute ring (PipeLLM, "Layer 2"; PIPO,
 * "Pipeline design" and the performance-optimised mode of "Two pipeline
 * modes"): every layer's merged block lives in pinned host memory and only
 * two layer buffers live in HBM.
 *   host_layers[i]   pinned host pointer (cudaHostAlloc or registered) of
 *                    layer i's merged block, 16-byte aligned, read only
 *   n_layers >= 1;  batch 1..16
 *   dev_buf0/1       device, buf_bytes >= one layer block each, 256-byte aligned
 *                    (dev_buf1 unused and may be null with Q4_STREAM_SINGLE_BUFFER)
 *   workspace        device, >= q4_workspace_layout(shape, n_layers, batch) bytes
 *   flags            0, or Q4_STREAM_POISON | Q4_STREAM_TENSOR_CORE | Q4_STREAM_CHUNKED |
 *                    Q4_STREAM_BARRIER | Q4_STREAM_CUDA_CORE | Q4_STREAM_SINGLE_BUFFER |
 *                    Q4_STREAM_TIMELINE
 * The handle creates its own copy stream and events.
 * Errors: Q4_ERR_ARG, Q4_ERR_ALIGN, Q4_ERR_OOM, Q4_ERR_CUDA.
 */
int q4_stream_create(q4_stream **out, const q4_layer_shape *shape, const void *const *host_layers,
                     int n_layers, int batch, void *dev_buf0, void *dev_buf1, size_t buf_bytes,
                     void *workspace, size_t workspace_bytes, int flags);

/*
 * q4_stream_create with partial residency (PIPO, "Two pipeline modes" and its
 * Experiments, where part of a model stays in GPU memory and the rest is
 * offloaded): resident_layers is null or holds n_layers device pointers;
 * entry i non-null = layer i's merged block is resident in HBM at that address
 * (256-byte aligned, caller-owned, read only) and is never copied, and
 * host_layers[i] may then be null.  The streamed layers alternate between the
 * two staging buffers in their own order; copies of the first streamed layers
 * overlap the compute of the resident layers before them.
 * Errors: as q4_stream_create.
 */
int q4_stream_create_ex(q4_stream **out, const q4_layer_shape *shape, const void *const *host_layers,
                        const void *const *resident_layers, int n_layers, int batch, void *dev_buf0,
                        void *dev_buf1, size_t buf_bytes, void *workspace, size_t workspace_bytes, int flags);

/*
 * Run all layers once on hidden_io (device, binary16 [batch][hidden]) while
 * the copy stream prefetches layer i+1 into the other buffer as layer i
 * computes on `compute_stream`.  Everything is enqueued asynchronously; if
 * timeout_us > 0 the call then waits for completion, polling, and returns
 * Q4_ERR_TIMEOUT if it has not finished after timeout_us microseconds (the
 * work stays queued).  Errors: Q4_ERR_ARG, Q4_ERR_ALIGN, Q4_ERR_CUDA, Q4_ERR_TIMEOUT.
 */
int q4_stream_layers(q4_stream *st, uint16_t *hidden_io, void *compute_stream, int64_t timeout_us);

/* Status word of the ring's kernels (synchronises compute_stream); clears it. */
int q4_stream_status(q4_stream *st, void *compute_stream, int *status_out);

/* The copy/compute timeline of the last q4_stream_layers call of a ring
 * created with Q4_STREAM_TIMELINE (PipeLLM, "Layer 2: Asynchronous Weight
 * Prefetching": the copy of layer i+1 overlaps the compute of layer i).
 * Synchronises compute_stream and the ring's copy stream, then writes
 * out_ns[4 i .. 4 i + 3] = copy begin, copy end, compute begin, compute end of
 * layer i (GPU global timer, ns; the copy pair is 0 for a resident layer).
 * n >= 4 * n_layers.  Errors: Q4_ERR_ARG (no timeline, n too small), Q4_ERR_CUDA. */
int q4_stream_timeline(q4_stream *st, unsigned long long *out_ns, int n, void *compute_stream);

/* As q4_decoder_tagged for a ring.  Host only.  Errors: Q4_ERR_ARG. */
int q4_stream_tagged(const q4_stream *st, int *tagged_out);

int q4_stream_destroy(q4_stream *st);

#ifdef __cplusplus
}
#endif

#endif /* Q4_H */
