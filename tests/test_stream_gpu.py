"""q4_stream_layers: the double-buffered copy/compute ring from pinned host memory."""
import numpy as np
import pytest
import torch

import weight_streaming_q4_gb300 as q4
from weight_streaming_q4_gb300 import build, model, synth
from gpu_util import dev_u16, host_u16

pytestmark = pytest.mark.gpu

TINY = dict(hidden=256, q_dim=256, kv_dim=128, ffn=1024, head_dim=64)
SMALL = dict(hidden=2048, q_dim=2048, kv_dim=512, ffn=4096, head_dim=128)


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


class Ring:
    def __init__(self, cfg, n_layers, seed, flags=0, distinct=None, batch=1):
        self.shape = q4.LayerShape.of(**cfg)
        self.blocks, self.hptrs = model.host_layers(self.shape, n_layers, seed, distinct=distinct)
        stride = model.layer_stride(self.shape)
        single = bool(flags & q4.Q4_STREAM_SINGLE_BUFFER)
        self.bufs = [torch.empty(stride, dtype=torch.uint8, device="cuda") for _ in range(1 if single else 2)]
        self.ws, self.offs, self.ws_bytes = model.workspace(self.shape, n_layers, batch)
        self.h = q4.q4_stream_create(self.shape, self.hptrs, batch, self.bufs[0], None if single else self.bufs[1],
                                     stride, self.ws, self.ws_bytes, flags)

    def run(self, h_np, tokens=1, timeout_us=0):
        h = dev_u16(h_np.reshape(-1))
        for _ in range(tokens):
            q4.q4_stream_layers(self.h, h, timeout_us=timeout_us)
        torch.cuda.synchronize()
        assert q4.q4_stream_status(self.h) == 0
        return host_u16(h).reshape(1, -1)

    def close(self):
        q4.q4_stream_destroy(self.h)


def resident(cfg, n_layers, seed, h_np, tokens=1, core=False, barrier=False, batch=1):
    shape = q4.LayerShape.of(**cfg)
    wbuf, ptrs = model.resident_layers(shape, n_layers, seed)
    ws, offs, nb = model.workspace(shape, n_layers, batch)
    mode = q4.Q4_DEC_PER_LAYER | (q4.Q4_DEC_CUDA_CORE if core else 0) | (q4.Q4_DEC_BARRIER if barrier else 0)
    dec = q4.q4_decoder_create(shape, ptrs, batch, ws, nb, mode)
    h = dev_u16(h_np.reshape(-1))
    for _ in range(tokens):
        q4.q4_layer_decode(dec, h)
    torch.cuda.synchronize()
    q4.q4_decoder_destroy(dec)
    return host_u16(h).reshape(batch, -1)


@pytest.mark.parametrize("cfg,n_layers", [(TINY, 5), (SMALL, 4)], ids=["tiny5", "small4"])
@pytest.mark.parametrize("flags", [0, q4.Q4_STREAM_POISON, q4.Q4_STREAM_POISON | q4.Q4_STREAM_CUDA_CORE,
                                   q4.Q4_STREAM_POISON | q4.Q4_STREAM_BARRIER],
                         ids=["plain", "poison", "poison-core", "poison-barrier"])
def test_streamed_equals_resident(cfg, n_layers, flags):
    h0 = synth.activations(1, cfg["hidden"], 50)
    ring = Ring(cfg, n_layers, seed=51, flags=flags)
    got = ring.run(h0, tokens=2)
    ref = resident(cfg, n_layers, 51, h0, tokens=2, core=bool(flags & q4.Q4_STREAM_CUDA_CORE),
                   barrier=bool(flags & q4.Q4_STREAM_BARRIER))
    assert np.array_equal(got, ref)
    assert np.all(np.isfinite(got.view(np.float16).astype(np.float64)))
    ring.close()


def test_streamed_70b_layers_equal_resident():
    cfg = dict(synth.LLAMA_70B)
    cfg.pop("n_layers")
    h0 = synth.activations(1, cfg["hidden"], 60)
    ring = Ring(cfg, 3, seed=61, flags=q4.Q4_STREAM_POISON)
    got = ring.run(h0)
    ref = resident(cfg, 3, 61, h0)
    assert np.array_equal(got, ref)
    ring.close()


def test_host_timeout_returns_and_work_completes():
    cfg = SMALL
    ring = Ring(cfg, 6, seed=70)
    h = dev_u16(synth.activations(1, cfg["hidden"], 71).reshape(-1))
    with pytest.raises(q4.Q4Error) as e:
        q4.q4_stream_layers(ring.h, h, timeout_us=1)
    assert e.value.status == q4.Q4_ERR_TIMEOUT
    torch.cuda.synchronize()                     # the queued work still finishes
    assert q4.q4_stream_status(ring.h) == 0
    ring.close()


def _mixed_ring(cfg, n_layers, seed, resident_mask, flags, batch=1, single=False):
    """A ring where layer i is resident (device block) when resident_mask[i], else streamed."""
    shape = q4.LayerShape.of(**cfg)
    blocks, hptrs = model.host_layers(shape, n_layers, seed)
    wbuf, dptrs = model.resident_layers(shape, n_layers, seed)
    stride = model.layer_stride(shape)
    bufs = [torch.empty(stride, dtype=torch.uint8, device="cuda") for _ in range(1 if single else 2)]
    ws, offs, nb = model.workspace(shape, n_layers, batch)
    host = [0 if m else hptrs[i] for i, m in enumerate(resident_mask)]
    res = [dptrs[i] if m else 0 for i, m in enumerate(resident_mask)]
    h = q4.q4_stream_create_ex(shape, host, res, batch, bufs[0], None if single else bufs[1], stride, ws, nb,
                               flags)
    return h, (blocks, wbuf, bufs, ws)


@pytest.mark.parametrize("flags", [q4.Q4_STREAM_CHUNKED, q4.Q4_STREAM_CHUNKED | q4.Q4_STREAM_POISON,
                                   q4.Q4_STREAM_CHUNKED | q4.Q4_STREAM_CUDA_CORE,
                                   q4.Q4_STREAM_CHUNKED | q4.Q4_STREAM_BARRIER],
                         ids=["chunked", "chunked-poison", "chunked-core", "chunked-barrier"])
def test_chunked_copies_equal_resident(flags):
    cfg, L = SMALL, 4
    h0 = synth.activations(1, cfg["hidden"], 80)
    ring = Ring(cfg, L, seed=81, flags=flags)
    got = ring.run(h0, tokens=2)
    ref = resident(cfg, L, 81, h0, tokens=2, core=bool(flags & q4.Q4_STREAM_CUDA_CORE),
                   barrier=bool(flags & q4.Q4_STREAM_BARRIER))
    assert np.array_equal(got, ref)
    ring.close()


@pytest.mark.parametrize("mask", [(1, 1, 0, 0, 0), (0, 1, 0, 1, 0), (1, 1, 1, 1, 1), (0, 0, 0, 0, 1)],
                         ids=["prefix", "alternate", "all", "last"])
@pytest.mark.parametrize("flags", [0, q4.Q4_STREAM_CHUNKED | q4.Q4_STREAM_POISON], ids=["merged", "chunked"])
def test_partial_residency_equals_resident(mask, flags):
    cfg, L = SMALL, 5
    h0 = synth.activations(1, cfg["hidden"], 82)
    st, keep = _mixed_ring(cfg, L, 83, mask, flags)
    h = dev_u16(h0.reshape(-1))
    for _ in range(2):
        q4.q4_stream_layers(st, h)
    torch.cuda.synchronize()
    assert q4.q4_stream_status(st) == 0
    got = host_u16(h).reshape(1, -1)
    q4.q4_stream_destroy(st)
    assert np.array_equal(got, resident(cfg, L, 83, h0, tokens=2))


def test_partial_residency_batch8_chunked():
    cfg, L, B = SMALL, 4, 8
    h0 = synth.activations(B, cfg["hidden"], 84)
    st, keep = _mixed_ring(cfg, L, 85, (1, 0, 0, 1), q4.Q4_STREAM_CHUNKED | q4.Q4_STREAM_POISON, batch=B)
    h = dev_u16(h0.reshape(-1))
    for _ in range(2):
        q4.q4_stream_layers(st, h)
    torch.cuda.synchronize()
    assert q4.q4_stream_status(st) == 0
    got = host_u16(h).reshape(B, -1)
    q4.q4_stream_destroy(st)
    shape = q4.LayerShape.of(**cfg)
    wbuf, ptrs = model.resident_layers(shape, L, 85)
    ws, offs, nb = model.workspace(shape, L, B)
    dec = q4.q4_decoder_create(shape, ptrs, B, ws, nb)
    hr = dev_u16(h0.reshape(-1))
    for _ in range(2):
        q4.q4_layer_decode(dec, hr)
    torch.cuda.synchronize()
    q4.q4_decoder_destroy(dec)
    assert np.array_equal(got, host_u16(hr).reshape(B, -1))


@pytest.mark.parametrize("cfg", [SMALL, dict(hidden=1024, q_dim=1024, kv_dim=256, ffn=14336, head_dim=128)],
                         ids=["small", "wide"])
def test_fused_per_layer_and_per_phase_schedules_identical(cfg):
    # one launch for the stack, one per layer, one per phase (chunked ring): same rows on the same CTAs
    h0 = synth.activations(1, cfg["hidden"], 86)
    shape = q4.LayerShape.of(**cfg)
    wbuf, ptrs = model.resident_layers(shape, 3, 87)
    outs = []
    for mode in (q4.Q4_DEC_FUSED, q4.Q4_DEC_PER_LAYER):
        ws, offs, nb = model.workspace(shape, 3, 1)
        dec = q4.q4_decoder_create(shape, ptrs, 1, ws, nb, mode)
        h = dev_u16(h0.reshape(-1))
        q4.q4_layer_decode(dec, h)
        torch.cuda.synchronize()
        q4.q4_decoder_destroy(dec)
        outs.append(host_u16(h).reshape(1, -1))
    ring = Ring(cfg, 3, seed=87, flags=q4.Q4_STREAM_CHUNKED)
    outs.append(ring.run(h0))
    ring.close()
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


SB = q4.Q4_STREAM_SINGLE_BUFFER


@pytest.mark.parametrize("flags", [SB | q4.Q4_STREAM_POISON, SB | q4.Q4_STREAM_POISON | q4.Q4_STREAM_CHUNKED,
                                   SB | q4.Q4_STREAM_POISON | q4.Q4_STREAM_CUDA_CORE,
                                   SB | q4.Q4_STREAM_POISON | q4.Q4_STREAM_BARRIER],
                         ids=["single", "single-chunked", "single-core", "single-barrier"])
def test_single_buffer_equals_resident(flags):
    """One staging buffer: every streamed layer overwrites the block the layer
    before it computed on (poisoned after each compute), over three tokens."""
    cfg, L = SMALL, 5
    h0 = synth.activations(1, cfg["hidden"], 90)
    ring = Ring(cfg, L, seed=91, flags=flags)
    got = ring.run(h0, tokens=3)
    ref = resident(cfg, L, 91, h0, tokens=3, core=bool(flags & q4.Q4_STREAM_CUDA_CORE),
                   barrier=bool(flags & q4.Q4_STREAM_BARRIER))
    assert np.array_equal(got, ref)
    ring.close()


def test_single_buffer_partial_residency_and_batch():
    """Single buffer with every other layer resident, batch 1 and batch 4."""
    cfg, L = SMALL, 6
    mask = [i % 2 == 1 for i in range(L)]
    for batch in (1, 4):
        h0 = synth.activations(batch, cfg["hidden"], 92)
        flags = SB | q4.Q4_STREAM_POISON
        h, keep = _mixed_ring(cfg, L, 93, mask, flags, batch=batch, single=True)
        x = dev_u16(h0.reshape(-1))
        for _ in range(2):
            q4.q4_stream_layers(h, x)
        torch.cuda.synchronize()
        assert q4.q4_stream_status(h) == 0
        got = host_u16(x).reshape(batch, -1)
        h2, keep2 = _mixed_ring(cfg, L, 93, [True] * L, 0, batch=batch)
        y = dev_u16(h0.reshape(-1))
        for _ in range(2):
            q4.q4_stream_layers(h2, y)
        torch.cuda.synchronize()
        assert np.array_equal(got, host_u16(y).reshape(batch, -1))
        q4.q4_stream_destroy(h)
        q4.q4_stream_destroy(h2)


@pytest.mark.parametrize("batch", [1, 4])
@pytest.mark.parametrize("single", [False, True], ids=["double", "single"])
def test_timeline_orders_copies_and_compute(single, batch):
    """The ring's GPU timestamps obey its synchronisation: a layer computes
    after its copy ended; a buffer is overwritten only after the compute that
    read it ended (layer i + 2 with two buffers, i + 1 with one); layers
    compute in order.  Results stay equal to the resident stack (batch 4: the
    per-product path)."""
    cfg, L = SMALL, 6
    flags = q4.Q4_STREAM_TIMELINE | (SB if single else 0)
    h0 = synth.activations(batch, cfg["hidden"], 94)
    ring = Ring(cfg, L, seed=95, flags=flags, batch=batch)
    got = ring.run(h0, tokens=2)
    tl = q4.q4_stream_timeline(ring.h, L).astype(np.int64)
    assert (tl > 0).all()
    cb, ce, kb, ke = tl[:, 0], tl[:, 1], tl[:, 2], tl[:, 3]
    assert (ce >= cb).all() and (ke >= kb).all()
    assert (kb >= ce).all()                      # compute waits for its own copy
    assert (kb[1:] >= ke[:-1]).all()             # one compute stream
    step = 1 if single else 2
    assert (cb[step:] >= ke[:-step]).all()       # buffer reuse after its reader finished
    assert np.array_equal(got.reshape(batch, -1), resident(cfg, L, 95, h0, tokens=2, batch=batch))
    with pytest.raises(q4.Q4Error):
        q4.q4_stream_timeline(ring.h, L - 1)      # buffer too small
    ring.close()
