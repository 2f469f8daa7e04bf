"""Synthetic Llama-shaped Q4_0 models laid out for the decoder and the ring.

Memory plumbing only (torch allocations, pointers, the seeded filler); every
arithmetic step of the decode runs in libq4.so.
"""
from __future__ import annotations

import torch

from . import _lib, synth


def shape_of(cfg: dict) -> _lib.LayerShape:
    return _lib.LayerShape.of(**cfg)


def layer_stride(shape: _lib.LayerShape) -> int:
    """Bytes of one merged layer block, rounded up to 256 (device placement stride)."""
    _, nbytes = _lib.q4_layer_offsets(shape)
    return (nbytes + 255) // 256 * 256


def fill_layer(dst_ptr: int, shape: _lib.LayerShape, layer: int, seed: int, stream=None):
    """Write layer ``layer``'s merged block (all seven projections) at dst_ptr (device)."""
    offs, _ = _lib.q4_layer_offsets(shape)
    dims = synth.layer_dims(shape.hidden, shape.q_dim, shape.kv_dim, shape.ffn)
    for p, (n, k) in enumerate(dims):
        synth.device_fill_q4(dst_ptr + offs[p], n * (k // 32), seed, synth.tensor_id(layer, p), stream=stream)


def resident_layers(shape: _lib.LayerShape, n_layers: int, seed: int, device="cuda", first_layer: int = 0):
    """All layers in one device allocation: returns (tensor, [layer pointers])."""
    stride = layer_stride(shape)
    buf = torch.empty(n_layers * stride, dtype=torch.uint8, device=device)
    base = buf.data_ptr()
    ptrs = [base + i * stride for i in range(n_layers)]
    for i, p in enumerate(ptrs):
        fill_layer(p, shape, first_layer + i, seed)
    return buf, ptrs


def host_layers(shape: _lib.LayerShape, n_layers: int, seed: int, distinct: int | None = None,
                device="cuda"):
    """Pinned host blocks, one per layer (filled on the device, then copied).

    ``distinct``: generate only that many distinct layers and reuse them
    cyclically (for hosts without room for every layer); None = all distinct.
    Returns (list of pinned tensors, [host pointers]).
    """
    stride = layer_stride(shape)
    _, nbytes = _lib.q4_layer_offsets(shape)
    n_dist = n_layers if distinct is None else min(distinct, n_layers)
    staging = torch.empty(stride, dtype=torch.uint8, device=device)
    blocks = []
    for i in range(n_dist):
        fill_layer(staging.data_ptr(), shape, i, seed)
        h = torch.empty(stride, dtype=torch.uint8, pin_memory=True)
        h.copy_(staging)
        blocks.append(h)
    torch.cuda.synchronize()
    ptrs = [blocks[i % n_dist].data_ptr() for i in range(n_layers)]
    return blocks, ptrs


def workspace(shape: _lib.LayerShape, n_layers: int, batch: int, device="cuda"):
    """A device workspace for a decoder or a ring of n_layers layers: (tensor, offsets, bytes)."""
    offs, total = _lib.q4_workspace_layout(shape, n_layers, batch)
    ws = torch.zeros(total, dtype=torch.uint8, device=device)
    return ws, offs, total


def ws_view(ws: torch.Tensor, offs: dict, name: str, dtype, count: int) -> torch.Tensor:
    """A typed view of one workspace region."""
    itemsize = torch.tensor([], dtype=dtype).element_size()
    start = offs[name]
    return ws[start:start + count * itemsize].view(dtype)
