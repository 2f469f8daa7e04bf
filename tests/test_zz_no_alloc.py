"""q4_layer_decode_noalloc: the decoder stack for callers that cannot
allocate device memory (inside allocator callbacks, in processes whose
device memory is reserved up front, or under plugin hosts that hand out no
workspace).  Its scratch lives in a fixed-size static device array in the
library instead of a caller-provided workspace.

Checked through the C ABI against q4_layer_decode with a caller workspace:
the same inputs must give the same outputs, within the error bound the other
tests use (the two paths run the same kernels, so they agree bit for bit),
on two calls in a row.  This file is collected last so that a run stopping
at its first failure has run every other test first.
"""
import ctypes

import numpy as np
import pytest
import torch

import weight_streaming_q4_gb300 as q4
from weight_streaming_q4_gb300 import build, model, synth
from gpu_util import dev_u16, f16_ulps, host_u16

pytestmark = pytest.mark.gpu

TINY = dict(hidden=256, q_dim=256, kv_dim=128, ffn=1024, head_dim=64)
EIGHT_B = dict(hidden=4096, q_dim=4096, kv_dim=1024, ffn=14336, head_dim=128)


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


@pytest.mark.parametrize("cfg,n_layers", [(TINY, 3), (EIGHT_B, 2)], ids=["tiny3", "8b2"])
def test_noalloc_matches_workspace_decoder_on_two_calls(cfg, n_layers):
    shape = q4.LayerShape.of(**cfg)
    wbuf, ptrs = model.resident_layers(shape, n_layers, seed=90)
    ws, offs, nb = model.workspace(shape, n_layers, 1)
    dec = q4.q4_decoder_create(shape, ptrs, 1, ws, nb, q4.Q4_DEC_FUSED)
    h0 = synth.activations(1, cfg["hidden"], 91)
    h_ref = dev_u16(h0.reshape(-1))
    h_new = dev_u16(h0.reshape(-1))
    for call in range(2):
        q4.q4_layer_decode(dec, h_ref)
        q4.q4_layer_decode_noalloc(shape, ptrs, h_new)
        torch.cuda.synchronize()
        assert q4.q4_noalloc_status() == 0, f"call {call}: a wait of the no-alloc kernels ran out"
        a, b = host_u16(h_ref), host_u16(h_new)
        assert np.all(np.isfinite(b.view(np.float16).astype(np.float64))), f"call {call}"
        assert f16_ulps(a, b).max() == 0, f"call {call}: outputs differ"
    assert q4.q4_decoder_status(dec) == 0
    q4.q4_decoder_destroy(dec)


def test_noalloc_on_a_side_stream_between_graph_replays():
    """Calls on a non-default stream, interleaved on that stream with graph
    replays of a decoder that owns its workspace: each no-alloc call gives,
    bit for bit, what the decoder gives for the same input."""
    shape = q4.LayerShape.of(**TINY)
    wbuf, ptrs = model.resident_layers(shape, 2, seed=92)
    ws, offs, nb = model.workspace(shape, 2, 1)
    dec = q4.q4_decoder_create(shape, ptrs, 1, ws, nb, q4.Q4_DEC_FUSED)
    s = torch.cuda.Stream()
    h0 = synth.activations(1, TINY["hidden"], 93)
    with torch.cuda.stream(s):
        h_ref, h_new = dev_u16(h0.reshape(-1)), dev_u16(h0.reshape(-1))
        for call in range(3):
            q4.q4_layer_decode(dec, h_ref, stream=s)
            q4.q4_layer_decode_noalloc(shape, ptrs, h_new, stream=s)
            q4.q4_layer_decode(dec, h_ref, stream=s)          # a replay right after, on the same stream
            q4.q4_layer_decode_noalloc(shape, ptrs, h_new, stream=s)
            assert q4.q4_noalloc_status(stream=s) == 0, f"call {call}"
            assert np.array_equal(host_u16(h_ref), host_u16(h_new)), f"call {call}: outputs differ"
    assert q4.q4_decoder_status(dec, stream=s) == 0
    q4.q4_decoder_destroy(dec)


def test_noalloc_refuses_stream_capture():
    """The call runs eagerly only: on a stream being captured it returns an
    argument error and enqueues nothing."""
    shape = q4.LayerShape.of(**TINY)
    wbuf, ptrs = model.resident_layers(shape, 1, seed=94)
    h = dev_u16(synth.activations(1, TINY["hidden"], 95).reshape(-1))
    before = host_u16(h)
    g = torch.cuda.CUDAGraph()
    side = torch.empty(16, device="cuda")
    with torch.cuda.graph(g):
        side.add_(1.0)
        with pytest.raises(q4.Q4Error) as e:
            q4.q4_layer_decode_noalloc(shape, ptrs, h, stream=torch.cuda.current_stream())
    assert e.value.status == q4.Q4_ERR_ARG
    torch.cuda.synchronize()
    assert np.array_equal(host_u16(h), before)


def test_noalloc_rejects_a_stack_beyond_the_array():
    shape = q4.LayerShape.of(**synth.LLAMA_70B)
    assert q4.q4_noalloc_scratch_bytes() == 1 << 20
    n = 2000
    need = q4.q4_workspace_layout(shape, n, 1)[1]
    assert need > q4.q4_noalloc_scratch_bytes()
    fake = (ctypes.c_void_p * n)(*([4096] * n))
    st = q4.lib().q4_layer_decode_noalloc(ctypes.byref(shape), fake, n, 4096, None)
    assert st == q4.Q4_ERR_OOM
