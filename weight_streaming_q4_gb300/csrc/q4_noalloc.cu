// q4_layer_decode_noalloc: the decoder stack for callers that cannot
// allocate device memory (see include/q4.h).  Its scratch (phase program,
// control block, intermediate activations) lives in one statically sized
// device array that every GPU loading this library holds until the process
// exits.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "q4.h"
#include "q4_device.cuh"

namespace {

// Scratch of the no-alloc decoder.  In host code this name is only a
// stand-in for the device symbol; its device address is looked up per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[Q4_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Once per device, with that device current: the device address of the array.
int scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return q4::record_cuda_error(e);
  if (dev < 0 || dev >= kMaxDevices) return Q4_ERR_ARG;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return q4::record_cuda_error(e);
    if (!ptr) return Q4_ERR_CUDA;
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return Q4_OK;
}

}  // namespace

extern "C" size_t q4_noalloc_scratch_bytes(void) { return Q4_NOALLOC_SCRATCH_BYTES; }

extern "C" int q4_layer_decode_noalloc(const q4_layer_shape* shape, const void* const* layer_weights, int n_layers,
                                       uint16_t* hidden_io, void* stream) {
  if (!shape || !layer_weights || n_layers < 1 || !hidden_io) return Q4_ERR_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The phase program is copied from host memory that lives only for this
  // call, so the call runs eagerly and refuses to be captured into a graph.
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(s, &cap);
  if (e != cudaSuccess) return q4::record_cuda_error(e);
  if (cap != cudaStreamCaptureStatusNone) return Q4_ERR_ARG;
  size_t off[Q4_WS_COUNT], need = 0;
  int st = q4_workspace_layout(shape, n_layers, 1, off, &need);
  if (st != Q4_OK) return st;
  if (need > Q4_NOALLOC_SCRATCH_BYTES) return Q4_ERR_OOM;   // beyond the array's fixed size
  void* scratch = nullptr;
  if ((st = scratch_for_current_device(&scratch)) != Q4_OK) return st;
  return q4::run_stack_in_workspace(shape, layer_weights, n_layers, hidden_io, scratch, Q4_NOALLOC_SCRATCH_BYTES, s);
}

extern "C" int q4_noalloc_status(void* stream, int* status_out) {
  if (!status_out) return Q4_ERR_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* scratch = nullptr;
  int st = scratch_for_current_device(&scratch);
  if (st != Q4_OK) return st;
  // the control block is the first region of the scratch (q4_workspace_layout order)
  q4::Control* ctl = static_cast<q4::Control*>(scratch);
  int v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, &ctl->status, sizeof(int), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess && v) e = cudaMemsetAsync(&ctl->status, 0, sizeof(int), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return q4::record_cuda_error(e);
  *status_out = v;
  return Q4_OK;
}
