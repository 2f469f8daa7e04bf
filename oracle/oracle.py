"""ctypes front end of the plain C oracle in ``q4_oracle.c``.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke``
and by the CPU-baseline leg of ``bench.py``.  Nothing here is shared with the
GPU library.  Every function forwards to the C file, which states what each
step computes and which passage of the pages it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q4_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

# -ffp-contract=off: no fused multiply-add contraction, so the oracle gives
# the same doubles on every host architecture.
CFLAGS = ["-O2", "-fPIC", "-shared", "-std=c11", "-ffp-contract=off", "-fno-fast-math"]


def compile_oracle(src: str = _SRC, out: str = _LIB, extra_flags=()) -> str:
    """Compile the C oracle with gcc into a shared library and return its path."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", *CFLAGS, *extra_flags, src, "-o", out + ".tmp", "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    os.replace(out + ".tmp", out)
    return out


def build() -> str:
    """Build the oracle library if it is missing or older than its source."""
    with _lock:
        if not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            compile_oracle()
    return _LIB


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_INT = ctypes.c_int
_DBL = ctypes.c_double


def _declare(lib):
    lib.ora_half_to_double.argtypes = [ctypes.c_uint16]
    lib.ora_half_to_double.restype = _DBL
    lib.ora_double_to_half.argtypes = [_DBL]
    lib.ora_double_to_half.restype = ctypes.c_uint16
    lib.ora_half_to_double_n.argtypes = [_P, _I64, _P]
    lib.ora_double_to_half_n.argtypes = [_P, _I64, _P]
    lib.ora_dequant.argtypes = [_P, _I64, _I64, _P]
    lib.ora_gemv.argtypes = [_P, _P, _I64, _I64, _INT, _I64, _I64, _P, _P]
    lib.ora_gemv_rows.argtypes = [_P, _P, _I64, _I64, _INT, _P, _I64, _P, _P]
    lib.ora_rmsnorm.argtypes = [_P, _INT, _I64, _DBL, _P]
    lib.ora_attn_ctx1.argtypes = [_P, _INT, _I64, _I64, _I64, _P]
    lib.ora_attn_decode.argtypes = [_P, _P, _P, _I64, _I64, _I64, _I64, _P, _P, _P]
    lib.ora_rmsnorm_d.argtypes = [_P, _INT, _I64, _DBL, _P]
    lib.ora_add.argtypes = [_P, _P, _I64, _P]
    lib.ora_silu_mul.argtypes = [_P, _P, _I64, _P]
    lib.ora_layer.argtypes = [_P, _P, _INT, _I64, _I64, _I64, _I64, _I64, _DBL, _P, _P, _P, _P]
    lib.ora_layer_kv.argtypes = [_P, _P, _I64, _I64, _I64, _I64, _I64, _DBL, _P, _P, _I64, _P, _P, _P, _P]
    for name in ("ora_half_to_double_n", "ora_double_to_half_n", "ora_dequant", "ora_gemv",
                 "ora_gemv_rows", "ora_rmsnorm", "ora_rmsnorm_d", "ora_attn_ctx1", "ora_attn_decode", "ora_add",
                 "ora_silu_mul", "ora_layer", "ora_layer_kv"):
        getattr(lib, name).restype = None
    return lib


def load(path: str | None = None):
    """Load (building first if needed) the oracle library; ``path`` loads another build."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    if _lib is None:
        build()
        _lib = _declare(ctypes.CDLL(_LIB))
    return _lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _u8(w) -> np.ndarray:
    if isinstance(w, np.ndarray):
        return np.ascontiguousarray(w).view(np.uint8).reshape(-1)
    return np.frombuffer(memoryview(w), dtype=np.uint8)


def _u16(x) -> np.ndarray:
    a = np.ascontiguousarray(x)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    assert a.dtype == np.uint16
    return a


# ---------------------------------------------------------------- binary16

def half_to_double(bits, lib=None) -> np.ndarray:
    lib = lib or load()
    b = _u16(bits)
    out = np.empty(b.shape, dtype=np.float64)
    lib.ora_half_to_double_n(_ptr(b), b.size, _ptr(out))
    return out


def double_to_half(v, lib=None) -> np.ndarray:
    """Round doubles to binary16 (RNE); returns the uint16 bit patterns."""
    lib = lib or load()
    a = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(a.shape, dtype=np.uint16)
    lib.ora_double_to_half_n(_ptr(a), a.size, _ptr(out))
    return out


# ---------------------------------------------------------------- Q4_0

def dequant(w, n_rows: int, k_dim: int, lib=None) -> np.ndarray:
    lib = lib or load()
    wb = _u8(w)
    assert wb.size >= n_rows * k_dim // 32 * 18
    out = np.empty((n_rows, k_dim), dtype=np.float64)
    lib.ora_dequant(_ptr(wb), n_rows, k_dim, _ptr(out))
    return out


def gemv(w, x, n_rows: int, k_dim: int, batch: int = 1, threads: int = 1, lib=None):
    """Full product: returns (y, s), each float64 [batch, n_rows]."""
    lib = lib or load()
    wb = _u8(w)
    xb = _u16(x).reshape(batch, k_dim)
    y = np.empty((batch, n_rows), dtype=np.float64)
    s = np.empty((batch, n_rows), dtype=np.float64)
    if threads <= 1 or n_rows < 2 * threads:
        lib.ora_gemv(_ptr(wb), _ptr(xb), n_rows, k_dim, batch, 0, n_rows, _ptr(y), _ptr(s))
        return y, s
    # Row ranges on separate threads (ctypes drops the GIL during the call).
    bounds = np.linspace(0, n_rows, threads + 1).astype(np.int64)
    ths = [threading.Thread(target=lib.ora_gemv,
                            args=(_ptr(wb), _ptr(xb), n_rows, k_dim, batch, int(bounds[i]),
                                  int(bounds[i + 1]), _ptr(y), _ptr(s)))
           for i in range(threads)]
    for t in ths:
        t.start()
    for t in ths:
        t.join()
    return y, s


def gemv_rows(w, x, n_rows: int, k_dim: int, rows, batch: int = 1, lib=None):
    """Product on selected rows only: returns (y, s), each float64 [batch, len(rows)]."""
    lib = lib or load()
    wb = _u8(w)
    xb = _u16(x).reshape(batch, k_dim)
    r = np.ascontiguousarray(rows, dtype=np.int64)
    y = np.empty((batch, r.size), dtype=np.float64)
    s = np.empty((batch, r.size), dtype=np.float64)
    lib.ora_gemv_rows(_ptr(wb), _ptr(xb), n_rows, k_dim, batch, _ptr(r), r.size, _ptr(y), _ptr(s))
    return y, s


# ---------------------------------------------------------------- glue

def rmsnorm(h, batch: int, dim: int, eps: float = 1e-5, lib=None) -> np.ndarray:
    lib = lib or load()
    hb = _u16(h).reshape(batch, dim)
    out = np.empty((batch, dim), dtype=np.uint16)
    lib.ora_rmsnorm(_ptr(hb), batch, dim, eps, _ptr(out))
    return out


def attn_ctx1(v, batch: int, q_dim: int, kv_dim: int, head_dim: int, lib=None) -> np.ndarray:
    lib = lib or load()
    vb = np.ascontiguousarray(v, dtype=np.float64).reshape(batch, kv_dim)
    out = np.empty((batch, q_dim), dtype=np.uint16)
    lib.ora_attn_ctx1(_ptr(vb), batch, q_dim, kv_dim, head_dim, _ptr(out))
    return out


def attn_decode(q, k_cache, v_cache, ctx: int, n_q: int, n_kv: int, head_dim: int, lib=None):
    """Decode attention of one token over the first ctx rows of a binary16 KV
    cache ([positions][n_kv * head_dim]); q double [n_q * head_dim].
    Returns (o, sabs), each double [n_q * head_dim]."""
    lib = lib or load()
    qd = np.ascontiguousarray(q, dtype=np.float64).reshape(-1)
    kc = _u16(k_cache).reshape(-1)
    vc = _u16(v_cache).reshape(-1)
    assert qd.size == n_q * head_dim and kc.size >= ctx * n_kv * head_dim and vc.size >= ctx * n_kv * head_dim
    o = np.empty(n_q * head_dim, dtype=np.float64)
    sabs = np.empty(n_q * head_dim, dtype=np.float64)
    work = np.empty(max(ctx, 1), dtype=np.float64)
    lib.ora_attn_decode(_ptr(qd), _ptr(kc), _ptr(vc), ctx, n_q, n_kv, head_dim, _ptr(o), _ptr(sabs), _ptr(work))
    return o, sabs


def rmsnorm_d(t, batch: int, dim: int, eps: float = 1e-5, lib=None) -> np.ndarray:
    """RMSNorm of double vectors (residual sums), rounded to binary16 bits."""
    lib = lib or load()
    tb = np.ascontiguousarray(t, dtype=np.float64).reshape(batch, dim)
    out = np.empty((batch, dim), dtype=np.uint16)
    lib.ora_rmsnorm_d(_ptr(tb), batch, dim, eps, _ptr(out))
    return out


def add(z, o, lib=None) -> np.ndarray:
    """Residual sum t = z + o (z binary16 bits, o double) in double."""
    lib = lib or load()
    zb = _u16(z)
    ob = np.ascontiguousarray(o, dtype=np.float64)
    assert zb.size == ob.size
    out = np.empty(zb.shape, dtype=np.float64)
    lib.ora_add(_ptr(zb), _ptr(ob), zb.size, _ptr(out))
    return out


def silu_mul(g, u, lib=None) -> np.ndarray:
    lib = lib or load()
    gb = np.ascontiguousarray(g, dtype=np.float64)
    ub = np.ascontiguousarray(u, dtype=np.float64)
    out = np.empty(gb.shape, dtype=np.uint16)
    lib.ora_silu_mul(_ptr(gb), _ptr(ub), gb.size, _ptr(out))
    return out


def layer(weights, z, batch: int, hidden: int, q_dim: int, kv_dim: int, ffn: int,
          head_dim: int = 128, eps: float = 1e-5, lib=None):
    """One decoder layer from its normalised binary16 input z; ``weights`` = 7
    byte arrays (q, k, v, o, gate, up, down).  Returns (z_out bits, t2 doubles)."""
    lib = lib or load()
    ws = [_u8(w) for w in weights]
    arr = (ctypes.c_void_p * 7)(*[w.ctypes.data for w in ws])
    zb = _u16(z).reshape(batch, hidden)
    work = np.empty(batch * (q_dim + 2 * kv_dim + 3 * hidden + 2 * ffn), dtype=np.float64)
    work16 = np.empty(batch * (hidden + q_dim + ffn), dtype=np.uint16)
    t2 = np.empty((batch, hidden), dtype=np.float64)
    out = np.empty((batch, hidden), dtype=np.uint16)
    lib.ora_layer(arr, _ptr(zb), batch, hidden, q_dim, kv_dim, ffn, head_dim, eps,
                  _ptr(work), _ptr(work16), _ptr(t2), _ptr(out))
    return out, t2


def layer_kv(weights, z, k_cache, v_cache, pos: int, hidden: int, q_dim: int, kv_dim: int, ffn: int,
             head_dim: int = 128, eps: float = 1e-5, lib=None):
    """One decoder layer of one token at position ``pos`` over a binary16 KV
    cache (arrays [capacity][kv_dim] of uint16, updated in row ``pos``).
    Returns (z_out bits, t2 doubles)."""
    lib = lib or load()
    ws = [_u8(w) for w in weights]
    arr = (ctypes.c_void_p * 7)(*[w.ctypes.data for w in ws])
    zb = _u16(z).reshape(-1)
    assert k_cache.dtype == np.uint16 and v_cache.dtype == np.uint16
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous and pos < k_cache.shape[0]
    work = np.empty(q_dim + 2 * kv_dim + 3 * hidden + 2 * ffn + 2 * q_dim + pos + 1, dtype=np.float64)
    work16 = np.empty(hidden + q_dim + ffn, dtype=np.uint16)
    t2 = np.empty(hidden, dtype=np.float64)
    out = np.empty(hidden, dtype=np.uint16)
    lib.ora_layer_kv(arr, _ptr(zb), hidden, q_dim, kv_dim, ffn, head_dim, eps, _ptr(k_cache), _ptr(v_cache), pos,
                     _ptr(work), _ptr(work16), _ptr(t2), _ptr(out))
    return out, t2


def tolerance(s) -> np.ndarray:
    """Per-element bound of the accepted error: 1e-3 * sum|w*x| + 1e-5."""
    return 1e-3 * np.asarray(s) + 1e-5
