"""ctypes binding of libq4.so with the C ABI's own names (include/q4.h).

Argument marshalling only: tensors become their data pointers, streams their
cudaStream_t handles, and a negative status becomes a Q4Error.  Every step of
the computation runs in the library's CUDA kernels; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import re

from . import build as _build

_lib = None

c_p = ctypes.c_void_p
c_int = ctypes.c_int
c_size = ctypes.c_size_t
c_i64 = ctypes.c_int64

Q4_OK = 0
Q4_ERR_ARG = -1
Q4_ERR_ALIGN = -2
Q4_ERR_CUDA = -3
Q4_ERR_TIMEOUT = -4
Q4_ERR_OOM = -5
Q4_ERR_DEVICE = -6

Q4_KERNEL_AUTO = 0
Q4_KERNEL_STREAM = 1
Q4_KERNEL_SIMPLE = 2
Q4_KERNEL_MMA = 3
Q4_KERNEL_TC = 4
Q4_KERNEL_ONESHOT = 5
Q4_GEMV_CHAIN = 0x100      # OR into q4_gemv_ex's kernel: a chained one-shot call

Q4_DEC_FUSED = 0
Q4_DEC_PER_LAYER = 1
Q4_DEC_TENSOR_CORE = 2
Q4_DEC_BARRIER = 4
Q4_DEC_CUDA_CORE = 8
Q4_DEC_BATCH_ENGINE = 16
Q4_STREAM_POISON = 1
Q4_STREAM_TENSOR_CORE = 2
Q4_STREAM_CHUNKED = 4
Q4_STREAM_BARRIER = 8
Q4_STREAM_CUDA_CORE = 16
Q4_STREAM_SINGLE_BUFFER = 32
Q4_STREAM_TIMELINE = 64

WS_NAMES = ("control", "program", "qkv", "o", "gate", "up", "down", "act", "x", "attn", "x2", "t1", "t2", "flags", "xt", "vt", "actt")
WS_COUNT = len(WS_NAMES)


class Q4Error(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = status_string(status) if _lib is not None else str(status)
        extra = ""
        if status == Q4_ERR_CUDA and _lib is not None:
            extra = f" (cudaError {_lib.q4_last_cuda_error()})"
        super().__init__(f"{what}: {msg}{extra}")


class LayerShape(ctypes.Structure):
    """q4_layer_shape."""
    _fields_ = [("hidden", c_int), ("q_dim", c_int), ("kv_dim", c_int), ("ffn", c_int),
                ("head_dim", c_int), ("eps", ctypes.c_float)]

    @classmethod
    def of(cls, hidden, q_dim, kv_dim, ffn, head_dim=128, eps=1e-5, **_):
        return cls(hidden, q_dim, kv_dim, ffn, head_dim, eps)


class KVCache(ctypes.Structure):
    """q4_kv_cache."""
    _fields_ = [("capacity", c_int), ("k_layers", ctypes.POINTER(c_p)), ("v_layers", ctypes.POINTER(c_p)),
                ("pos", c_p), ("attn_workspace", c_p), ("attn_workspace_bytes", c_size)]


def _declare(lib):
    sig = {
        "q4_status_string": ([c_int], ctypes.c_char_p),
        "q4_last_cuda_error": ([], c_int),
        "q4_version": ([], c_int),
        "q4_matrix_bytes": ([c_int, c_int], c_size),
        "q4_gemv": ([c_p, c_p, c_p, c_int, c_int, c_int, c_p], c_int),
        "q4_gemv_ex": ([c_p, c_p, c_p, c_int, c_int, c_int, c_int, c_p], c_int),
        "q4_device_status": ([], c_int),
        "q4_dequant_debug": ([c_p, c_p, c_int, c_int, c_p], c_int),
        "q4_layer_offsets": ([ctypes.POINTER(LayerShape), ctypes.POINTER(c_size), ctypes.POINTER(c_size)], c_int),
        "q4_workspace_layout": ([ctypes.POINTER(LayerShape), c_int, c_int, ctypes.POINTER(c_size),
                                 ctypes.POINTER(c_size)], c_int),
        "q4_decoder_create": ([ctypes.POINTER(c_p), ctypes.POINTER(LayerShape), ctypes.POINTER(c_p), c_int, c_int,
                               c_p, c_size, c_int, c_p], c_int),
        "q4_layer_decode": ([c_p, c_p, c_p], c_int),
        "q4_layer_decode_eager": ([c_p, c_p, c_p], c_int),
        "q4_decoder_status": ([c_p, c_p, ctypes.POINTER(c_int)], c_int),
        "q4_decoder_tagged": ([c_p, ctypes.POINTER(c_int)], c_int),
        "q4_decoder_debug_stall": ([c_p, ctypes.c_uint32, c_p, ctypes.POINTER(c_int)], c_int),
        "q4_decoder_destroy": ([c_p], c_int),
        "q4_decoder_create_kv": ([ctypes.POINTER(c_p), ctypes.POINTER(LayerShape), ctypes.POINTER(c_p), c_int,
                                  ctypes.POINTER(KVCache), c_p, c_size, c_p], c_int),
        "q4_layer_decode_noalloc": ([ctypes.POINTER(LayerShape), ctypes.POINTER(c_p), c_int, c_p, c_p], c_int),
        "q4_noalloc_scratch_bytes": ([], c_size),
        "q4_noalloc_status": ([c_p, ctypes.POINTER(c_int)], c_int),
        "q4_stream_create": ([ctypes.POINTER(c_p), ctypes.POINTER(LayerShape), ctypes.POINTER(c_p), c_int, c_int,
                              c_p, c_p, c_size, c_p, c_size, c_int], c_int),
        "q4_stream_create_ex": ([ctypes.POINTER(c_p), ctypes.POINTER(LayerShape), ctypes.POINTER(c_p),
                                 ctypes.POINTER(c_p), c_int, c_int, c_p, c_p, c_size, c_p, c_size, c_int], c_int),
        "q4_stream_layers": ([c_p, c_p, c_p, c_i64], c_int),
        "q4_attn_decode": ([c_p, c_p, c_p, c_p, c_int, c_int, c_int, c_int, c_p, c_p, c_size, c_p], c_int),
        "q4_attn_workspace_bytes": ([c_int, c_int, c_int, c_int], c_size),
        "q4_kv_append": ([c_p, c_p, c_p, c_p, c_p, c_int, c_int, c_p], c_int),
        "q4_stream_status": ([c_p, c_p, ctypes.POINTER(c_int)], c_int),
        "q4_stream_tagged": ([c_p, ctypes.POINTER(c_int)], c_int),
        "q4_stream_timeline": ([c_p, c_p, c_int, c_p], c_int),
        "q4_timeline_read": ([c_p, c_size, c_int], c_int),
        "q4_stream_destroy": ([c_p], c_int),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    return lib


def lib():
    """The loaded libq4.so; raises if it has not been built (no fallback exists)."""
    global _lib
    if _lib is None:
        path = _build.lib_path("libq4.so")
        if not os.path.exists(path):
            raise ImportError(f"libq4.so is not built ({path}); run weight_streaming_q4_gb300.build.build()")
        _lib = _declare(ctypes.CDLL(path))
    return _lib


def use_library(path: str):
    """Bind every call to another build of the library (the timeline build)."""
    global _lib
    _lib = _declare(ctypes.CDLL(path))
    return _lib


def header_functions() -> list:
    """Names of the functions include/q4.h declares."""
    text = open(os.path.join(_build.INCLUDE, "q4.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(q4_[a-z0-9_]+)\s*\(", text)))


# ------------------------------------------------------------------ marshalling

def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(st: int, what: str):
    if st < 0:
        raise Q4Error(st, what)
    return st


def status_string(st: int) -> str:
    return lib().q4_status_string(st).decode()


def q4_last_cuda_error() -> int:
    return lib().q4_last_cuda_error()


def q4_version() -> int:
    return lib().q4_version()


def q4_matrix_bytes(n: int, k: int) -> int:
    return lib().q4_matrix_bytes(n, k)


def q4_gemv(w, x, y, n: int, k: int, batch: int = 1, stream=None, chain: bool = False):
    if chain:   # Q4_GEMV_CHAIN: may overlap the product before it on the stream
        _check(lib().q4_gemv_ex(_ptr(w), _ptr(x), _ptr(y), n, k, batch, Q4_KERNEL_AUTO | Q4_GEMV_CHAIN,
                                _stream(stream)), "q4_gemv_ex")
        return
    _check(lib().q4_gemv(_ptr(w), _ptr(x), _ptr(y), n, k, batch, _stream(stream)), "q4_gemv")


def q4_gemv_ex(w, x, y, n: int, k: int, batch: int, kernel: int, stream=None):
    _check(lib().q4_gemv_ex(_ptr(w), _ptr(x), _ptr(y), n, k, batch, kernel, _stream(stream)), "q4_gemv_ex")


def q4_device_status() -> int:
    return _check(lib().q4_device_status(), "q4_device_status")


def q4_dequant_debug(w, out, n: int, k: int, stream=None):
    _check(lib().q4_dequant_debug(_ptr(w), _ptr(out), n, k, _stream(stream)), "q4_dequant_debug")


def q4_layer_offsets(shape: LayerShape):
    offs = (c_size * 7)()
    total = c_size(0)
    _check(lib().q4_layer_offsets(ctypes.byref(shape), offs, ctypes.byref(total)), "q4_layer_offsets")
    return list(offs), total.value


def q4_workspace_layout(shape: LayerShape, n_layers: int, batch: int):
    offs = (c_size * WS_COUNT)()
    total = c_size(0)
    _check(lib().q4_workspace_layout(ctypes.byref(shape), n_layers, batch, offs, ctypes.byref(total)),
           "q4_workspace_layout")
    return dict(zip(WS_NAMES, list(offs))), total.value


def q4_decoder_create_kv(shape: LayerShape, layer_ptrs, capacity: int, k_layers, v_layers, pos, attn_workspace,
                         attn_workspace_bytes: int, workspace, workspace_bytes: int, stream=None):
    """Batch-1 decoder with decode attention over per-layer KV caches (device
    pointers or tensors; ``pos`` a device int32)."""
    h = c_p()
    arr = (c_p * len(layer_ptrs))(*[int(p) for p in layer_ptrs])
    ks = (c_p * len(k_layers))(*[_ptr(t) for t in k_layers])
    vs = (c_p * len(v_layers))(*[_ptr(t) for t in v_layers])
    kv = KVCache(capacity, ks, vs, _ptr(pos), _ptr(attn_workspace), attn_workspace_bytes)
    kv._keep = (ks, vs)
    _check(lib().q4_decoder_create_kv(ctypes.byref(h), ctypes.byref(shape), arr, len(layer_ptrs), ctypes.byref(kv),
                                      _ptr(workspace), workspace_bytes, _stream(stream)), "q4_decoder_create_kv")
    return h


def q4_decoder_create(shape: LayerShape, layer_ptrs, batch: int, workspace, workspace_bytes: int,
                      mode: int = Q4_DEC_FUSED, stream=None):
    h = c_p()
    arr = (c_p * len(layer_ptrs))(*[int(p) for p in layer_ptrs])
    _check(lib().q4_decoder_create(ctypes.byref(h), ctypes.byref(shape), arr, len(layer_ptrs), batch,
                                   _ptr(workspace), workspace_bytes, mode, _stream(stream)), "q4_decoder_create")
    return h


def q4_layer_decode(dec, hidden, stream=None):
    _check(lib().q4_layer_decode(dec, _ptr(hidden), _stream(stream)), "q4_layer_decode")


def q4_layer_decode_eager(dec, hidden, stream=None):
    _check(lib().q4_layer_decode_eager(dec, _ptr(hidden), _stream(stream)), "q4_layer_decode_eager")


def q4_decoder_status(dec, stream=None) -> int:
    v = c_int(0)
    _check(lib().q4_decoder_status(dec, _stream(stream), ctypes.byref(v)), "q4_decoder_status")
    return v.value


def q4_decoder_tagged(dec) -> bool:
    v = c_int(0)
    _check(lib().q4_decoder_tagged(dec, ctypes.byref(v)), "q4_decoder_tagged")
    return bool(v.value)


def q4_decoder_debug_stall(dec, wait_limit, stream=None) -> int:
    v = c_int(0)
    _check(lib().q4_decoder_debug_stall(dec, wait_limit, _stream(stream), ctypes.byref(v)), "q4_decoder_debug_stall")
    return v.value


def q4_decoder_destroy(dec):
    _check(lib().q4_decoder_destroy(dec), "q4_decoder_destroy")


def q4_layer_decode_noalloc(shape: LayerShape, layer_ptrs, hidden, stream=None):
    """The decoder stack with its scratch in the library's static device array (no allocation)."""
    arr = (c_p * len(layer_ptrs))(*[int(p) for p in layer_ptrs])
    _check(lib().q4_layer_decode_noalloc(ctypes.byref(shape), arr, len(layer_ptrs), _ptr(hidden), _stream(stream)),
           "q4_layer_decode_noalloc")


def q4_noalloc_scratch_bytes() -> int:
    return lib().q4_noalloc_scratch_bytes()


def q4_noalloc_status(stream=None) -> int:
    v = c_int(0)
    _check(lib().q4_noalloc_status(_stream(stream), ctypes.byref(v)), "q4_noalloc_status")
    return v.value


def q4_stream_create(shape: LayerShape, host_ptrs, batch: int, buf0, buf1, buf_bytes: int, workspace,
                     workspace_bytes: int, flags: int = 0):
    h = c_p()
    arr = (c_p * len(host_ptrs))(*[int(p) for p in host_ptrs])
    _check(lib().q4_stream_create(ctypes.byref(h), ctypes.byref(shape), arr, len(host_ptrs), batch, _ptr(buf0),
                                  _ptr(buf1), buf_bytes, _ptr(workspace), workspace_bytes, flags),
           "q4_stream_create")
    return h


def q4_stream_create_ex(shape: LayerShape, host_ptrs, resident_ptrs, batch: int, buf0, buf1, buf_bytes: int,
                        workspace, workspace_bytes: int, flags: int = 0):
    """host_ptrs[i] / resident_ptrs[i]: pinned host block or device block of layer i (0 = none)."""
    h = c_p()
    n = len(host_ptrs)
    harr = (c_p * n)(*[int(p) if p else None for p in host_ptrs])
    rarr = None if resident_ptrs is None else (c_p * n)(*[int(p) if p else None for p in resident_ptrs])
    _check(lib().q4_stream_create_ex(ctypes.byref(h), ctypes.byref(shape), harr, rarr, n, batch, _ptr(buf0),
                                     _ptr(buf1), buf_bytes, _ptr(workspace), workspace_bytes, flags),
           "q4_stream_create_ex")
    return h


def q4_attn_decode(q, k_cache, v_cache, ctx_len, capacity: int, n_q_heads: int, n_kv_heads: int, head_dim: int,
                   out, workspace, workspace_bytes: int, stream=None):
    _check(lib().q4_attn_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(ctx_len), capacity, n_q_heads,
                                n_kv_heads, head_dim, _ptr(out), _ptr(workspace), workspace_bytes, _stream(stream)),
           "q4_attn_decode")


def q4_attn_workspace_bytes(n_q_heads: int, n_kv_heads: int, head_dim: int, capacity: int) -> int:
    return lib().q4_attn_workspace_bytes(n_q_heads, n_kv_heads, head_dim, capacity)


def q4_kv_append(k, v, k_cache, v_cache, pos, capacity: int, kv_dim: int, stream=None):
    _check(lib().q4_kv_append(_ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache), _ptr(pos), capacity, kv_dim,
                              _stream(stream)), "q4_kv_append")


def q4_stream_layers(st, hidden, stream=None, timeout_us: int = 0):
    return _check(lib().q4_stream_layers(st, _ptr(hidden), _stream(stream), timeout_us), "q4_stream_layers")


def q4_stream_timeline(st, n_layers: int, stream=None):
    """[n_layers][4] globaltimer ns: copy begin, copy end, compute begin, compute end."""
    import numpy as np
    out = np.zeros(4 * n_layers, dtype=np.uint64)
    _check(lib().q4_stream_timeline(st, out.ctypes.data_as(ctypes.c_void_p), out.size, _stream(stream)),
           "q4_stream_timeline")
    return out.reshape(n_layers, 4)


TIMELINE_CTAS, TIMELINE_PHASES, TIMELINE_EVENTS = 256, 64, 6


def q4_timeline_read(clear: bool = True):
    """[CTA][phase][event] globaltimer ns of the engine's last launches (timeline build only)."""
    import numpy as np
    out = np.zeros(TIMELINE_CTAS * TIMELINE_PHASES * TIMELINE_EVENTS, dtype=np.uint64)
    _check(lib().q4_timeline_read(out.ctypes.data_as(ctypes.c_void_p), out.size, 1 if clear else 0),
           "q4_timeline_read")
    return out.reshape(TIMELINE_CTAS, TIMELINE_PHASES, TIMELINE_EVENTS)


def q4_stream_tagged(st) -> bool:
    v = c_int(0)
    _check(lib().q4_stream_tagged(st, ctypes.byref(v)), "q4_stream_tagged")
    return bool(v.value)


def q4_stream_status(st, stream=None) -> int:
    v = c_int(0)
    _check(lib().q4_stream_status(st, _stream(stream), ctypes.byref(v)), "q4_stream_status")
    return v.value


def q4_stream_destroy(st):
    _check(lib().q4_stream_destroy(st), "q4_stream_destroy")
