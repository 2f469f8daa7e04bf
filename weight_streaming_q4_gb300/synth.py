"""Seeded synthetic inputs: Q4_0 weight matrices and binary16 activations.

This module draws random numbers and lays them out; it computes nothing of
the decode step itself.  Both the GPU path's tests and benchmark and the CPU
oracle are fed from it.

Generator: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random
numbers: as easy as 1, 2, 3", SC'11), a counter-based generator, so any block
of any tensor can be regenerated on its own.  The same generator is written a
second time in CUDA (``csrc/synth.cu``) to fill large models on the device;
both are checked against the published known-answer vector and against each
other bit for bit.

Value recipe (the workloads' stated distributions):
  * 4-bit codes q: i.i.d. uniform on {0..15} (one Philox output = 16 bytes
    of codes for one block);
  * block scale d = binary16(|sigma * z|), sigma = 0.02;
  * activations x = binary16(z);
  where z is the Irwin-Hall sum of twelve uniforms minus six, a textbook
  approximation of N(0, 1) (unit variance, tails cut at +-6) that needs no
  transcendental function, so the CPU and the GPU draw bit-identical values.
"""
from __future__ import annotations

import numpy as np

# Philox4x32 constants from the published definition.
_M0 = np.uint64(0xD2511F53)
_M1 = np.uint64(0xCD9E8D57)
_W0 = 0x9E3779B9
_W1 = 0xBB67AE85
_MASK = np.uint64(0xFFFFFFFF)

TAG_QS = 0x51      # counter word 2 for the codes of a block
TAG_D = 0xD0       # 0xD0..0xD2: the twelve uniforms of a block scale
TAG_X = 0xA0       # 0xA0..0xA2: the twelve uniforms of an activation

SCALE_SIGMA = 0.02
X_SIGMA = 1.0

PROJ_NAMES = ("q", "k", "v", "o", "gate", "up", "down")
BLOCK_BYTES = 18
QK = 32


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Philox4x32 with 10 rounds on uint32 counter words and a 2-word key.

    Arguments broadcast; returns four uint32 arrays.
    """
    c0 = np.asarray(c0, dtype=np.uint64) & _MASK
    c1 = np.asarray(c1, dtype=np.uint64) & _MASK
    c2 = np.asarray(c2, dtype=np.uint64) & _MASK
    c3 = np.asarray(c3, dtype=np.uint64) & _MASK
    k0 = np.uint64(int(k0) & 0xFFFFFFFF)
    k1 = np.uint64(int(k1) & 0xFFFFFFFF)
    for _ in range(10):
        p0 = _M0 * c0
        p1 = _M1 * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
        k0 = np.uint64((int(k0) + _W0) & 0xFFFFFFFF)
        k1 = np.uint64((int(k1) + _W1) & 0xFFFFFFFF)
    return (c0.astype(np.uint32), c1.astype(np.uint32), c2.astype(np.uint32),
            c3.astype(np.uint32))


def _irwin_hall12(idx: np.ndarray, tag: int, seed: int, tid: int) -> np.ndarray:
    """z = (sum of 12 uniform 32-bit words) * 2^-32 - 6, exact in double."""
    lo = idx & np.uint64(0xFFFFFFFF)
    hi = idx >> np.uint64(32)
    total = np.zeros(idx.shape, dtype=np.uint64)
    for r in range(3):
        words = philox4x32_10(lo, hi, tag + r, 0, seed, tid)
        for wd in words:
            total += wd.astype(np.uint64)
    centered = total.astype(np.int64) - np.int64(6 << 32)
    return centered.astype(np.float64) * (2.0 ** -32)


def tensor_id(layer: int, proj: int) -> int:
    """Key word of projection ``proj`` (0..6: q,k,v,o,gate,up,down) of ``layer``."""
    return ((layer & 0x0FFFFFFF) << 4) | (proj & 0xF)


GEMV_TID = 0x7FFF0000   # the stand-alone matrix of the single-product workload
X_TID = 0x80000000      # activations (bit 31 set keeps them apart from weights)


def q4_blocks(block_idx, seed: int, tid: int) -> np.ndarray:
    """The 18-byte Q4_0 blocks with the given flat indices: uint8 [n, 18]."""
    idx = np.asarray(block_idx, dtype=np.uint64).reshape(-1)
    lo = idx & np.uint64(0xFFFFFFFF)
    hi = idx >> np.uint64(32)
    out = np.empty((idx.size, BLOCK_BYTES), dtype=np.uint8)
    words = philox4x32_10(lo, hi, TAG_QS, 0, seed, tid)
    out[:, 2:] = np.stack(words, axis=1).astype("<u4").view(np.uint8).reshape(-1, 16)
    z = _irwin_hall12(idx, TAG_D, seed, tid)
    d = np.abs(z * SCALE_SIGMA).astype(np.float16)   # numpy rounds double -> half to nearest even
    out[:, 0:2] = d.view(np.uint16).astype("<u2").view(np.uint8).reshape(-1, 2)
    return out


def q4_matrix(n_rows: int, k_dim: int, seed: int, tid: int) -> np.ndarray:
    """A whole row-major Q4_0 matrix as uint8 [n_rows * k_dim / 32 * 18]."""
    assert k_dim % QK == 0
    nb = n_rows * (k_dim // QK)
    return q4_blocks(np.arange(nb, dtype=np.uint64), seed, tid).reshape(-1)


def q4_rows(rows, k_dim: int, seed: int, tid: int) -> np.ndarray:
    """Selected rows of the matrix ``q4_matrix(., k_dim, seed, tid)``, packed: uint8 [len(rows), row_bytes]."""
    bpr = k_dim // QK
    r = np.asarray(rows, dtype=np.uint64).reshape(-1, 1)
    idx = r * np.uint64(bpr) + np.arange(bpr, dtype=np.uint64)[None, :]
    return q4_blocks(idx.reshape(-1), seed, tid).reshape(len(r), bpr * BLOCK_BYTES)


def normal_f16(n: int, seed: int, tid: int, sigma: float = X_SIGMA, start: int = 0) -> np.ndarray:
    """n binary16 values ~ binary16(sigma * z); returns the uint16 bit patterns."""
    idx = np.arange(start, start + n, dtype=np.uint64)
    z = _irwin_hall12(idx, TAG_X, seed, tid)
    return (z * sigma).astype(np.float16).view(np.uint16)


def activations(batch: int, dim: int, seed: int, tid: int = X_TID) -> np.ndarray:
    """Activation rows x [batch, dim] as binary16 bit patterns."""
    return normal_f16(batch * dim, seed, tid).reshape(batch, dim)


# ------------------------------------------------------------------ shapes

def q4_bytes(n_rows: int, k_dim: int) -> int:
    return n_rows * (k_dim // QK) * BLOCK_BYTES


def layer_dims(hidden: int, q_dim: int, kv_dim: int, ffn: int):
    """(rows, cols) of q, k, v, o, gate, up, down."""
    return ((q_dim, hidden), (kv_dim, hidden), (kv_dim, hidden), (hidden, q_dim),
            (ffn, hidden), (ffn, hidden), (hidden, ffn))


def layer_offsets(hidden: int, q_dim: int, kv_dim: int, ffn: int):
    """Byte offsets of the seven projections inside one merged layer block, and its size.

    Each projection is a contiguous GGUF-order Q4_0 matrix, and they follow
    one another with no gap (the library's q4_layer_offsets layout).
    """
    offs, pos = [], 0
    for (n, k) in layer_dims(hidden, q_dim, kv_dim, ffn):
        offs.append(pos)
        pos += q4_bytes(n, k)
    return offs, pos


def layer_block(layer: int, hidden: int, q_dim: int, kv_dim: int, ffn: int, seed: int) -> np.ndarray:
    """The merged weight block of one layer (host, numpy): uint8 [layer_bytes]."""
    offs, total = layer_offsets(hidden, q_dim, kv_dim, ffn)
    out = np.zeros(total, dtype=np.uint8)
    for p, (n, k) in enumerate(layer_dims(hidden, q_dim, kv_dim, ffn)):
        m = q4_matrix(n, k, seed, tensor_id(layer, p))
        out[offs[p]:offs[p] + m.size] = m
    return out


LLAMA_8B = dict(hidden=4096, q_dim=4096, kv_dim=1024, ffn=14336, head_dim=128, n_layers=32)
LLAMA_70B = dict(hidden=8192, q_dim=8192, kv_dim=1024, ffn=28672, head_dim=128, n_layers=80)


# ------------------------------------------------------------------ device filler

_synth_lib = None


def _device_lib():
    global _synth_lib
    if _synth_lib is None:
        import ctypes
        import os

        from . import build as _build
        path = _build.lib_path("libq4synth.so")
        if not os.path.exists(path):
            raise ImportError(f"libq4synth.so is not built ({path})")
        lib = ctypes.CDLL(path)
        u64, u32, vp = ctypes.c_uint64, ctypes.c_uint32, ctypes.c_void_p
        lib.q4s_fill_q4_0.argtypes = [vp, u64, u64, u32, u32, ctypes.c_double, vp]
        lib.q4s_fill_normal_f16.argtypes = [vp, u64, u64, u32, u32, ctypes.c_double, vp]
        lib.q4s_philox.argtypes = [vp, u32, u32, u32, u32, u32, u32, vp]
        for f in (lib.q4s_fill_q4_0, lib.q4s_fill_normal_f16, lib.q4s_philox):
            f.restype = ctypes.c_int
        _synth_lib = lib
    return _synth_lib


def _cur_stream(stream):
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def device_fill_q4(dst_ptr: int, n_blocks: int, seed: int, tid: int, block0: int = 0, stream=None):
    """Write blocks block0.. of tensor ``tid`` (same bytes as ``q4_blocks``) to device memory."""
    e = _device_lib().q4s_fill_q4_0(dst_ptr, n_blocks, block0, seed & 0xFFFFFFFF, tid & 0xFFFFFFFF,
                                    SCALE_SIGMA, _cur_stream(stream))
    if e != 0:
        raise RuntimeError(f"q4s_fill_q4_0 failed: cudaError {e}")


def device_fill_normal_f16(dst_ptr: int, n: int, seed: int, tid: int, sigma: float = X_SIGMA, start: int = 0,
                           stream=None):
    e = _device_lib().q4s_fill_normal_f16(dst_ptr, n, start, seed & 0xFFFFFFFF, tid & 0xFFFFFFFF, sigma,
                                          _cur_stream(stream))
    if e != 0:
        raise RuntimeError(f"q4s_fill_normal_f16 failed: cudaError {e}")


def device_philox(out_ptr: int, c0, c1, c2, c3, k0, k1, stream=None):
    e = _device_lib().q4s_philox(out_ptr, c0, c1, c2, c3, k0, k1, _cur_stream(stream))
    if e != 0:
        raise RuntimeError(f"q4s_philox failed: cudaError {e}")
