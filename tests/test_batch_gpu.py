"""Decoder stack and streamed ring at batch 2..16: the per-product path
(tensor-core products + glue kernels, the default) and the persistent batched
engine (batch 2..8, Q4_DEC_BATCH_ENGINE)."""
import numpy as np
import pytest
import torch

import oracle as ora
import weight_streaming_q4_gb300 as q4
from weight_streaming_q4_gb300 import build, model, synth
from gpu_util import dev_u16, host_u16
from layer_check import check_layer, read_ws, sampled_rows

pytestmark = pytest.mark.gpu

TINY = dict(hidden=256, q_dim=256, kv_dim=128, ffn=1024, head_dim=64)
SMALL = dict(hidden=2048, q_dim=2048, kv_dim=512, ffn=4096, head_dim=128)
MID = dict(hidden=1024, q_dim=1024, kv_dim=256, ffn=14336, head_dim=128)
ODD = dict(hidden=768, q_dim=768, kv_dim=192, ffn=2816, head_dim=64)   # 3 KV heads for 12 query heads


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    ora.build()


class Stack:
    def __init__(self, cfg, n_layers, seed, batch, mode=q4.Q4_DEC_FUSED, ptrs=None):
        self.cfg, self.batch = cfg, batch
        self.shape = q4.LayerShape.of(**cfg)
        if ptrs is None:
            self.wbuf, self.ptrs = model.resident_layers(self.shape, n_layers, seed)
        else:
            self.ptrs = ptrs
        self.ws, self.offs, self.ws_bytes = model.workspace(self.shape, n_layers, batch)
        self.dec = q4.q4_decoder_create(self.shape, self.ptrs, batch, self.ws, self.ws_bytes, mode)

    def run(self, h_np, graph=True, reps=1):
        h = dev_u16(h_np.reshape(-1))
        for _ in range(reps):
            (q4.q4_layer_decode if graph else q4.q4_layer_decode_eager)(self.dec, h)
        torch.cuda.synchronize()
        assert q4.q4_decoder_status(self.dec) == 0
        return host_u16(h).reshape(self.batch, -1)

    def state(self):
        return read_ws(self.ws, self.offs, self.cfg, self.batch)

    def close(self):
        q4.q4_decoder_destroy(self.dec)


BT = q4.Q4_DEC_FUSED | q4.Q4_DEC_BATCH_ENGINE


@pytest.mark.parametrize("batch", [2, 8, 9, 16])
@pytest.mark.parametrize("cfg", [TINY, SMALL, ODD], ids=["tiny", "small", "odd"])
def test_one_layer_step_by_step(cfg, batch):
    st = Stack(cfg, 1, seed=81, batch=batch)
    h0 = synth.activations(batch, cfg["hidden"], 82)
    h1 = st.run(h0)
    check_layer(cfg, 81, 0, st.state(), h1, h_in16=h0)
    st.close()


@pytest.mark.parametrize("batch", [2, 3, 5, 8])
@pytest.mark.parametrize("cfg", [TINY, SMALL, MID], ids=["tiny", "small", "mid"])
def test_batched_engine_one_layer_step_by_step(cfg, batch):
    """The batched engine: every projection against the oracle fed the GPU's
    own input, every glue step (RMSNorms, attention gather, SiLU product,
    residual sums); batch 2, 3, 5, 8 use fragment buffers of 2, 4, 8, 8 columns."""
    st = Stack(cfg, 1, seed=81, batch=batch, mode=BT)
    h0 = synth.activations(batch, cfg["hidden"], 82)
    h1 = st.run(h0)
    check_layer(cfg, 81, 0, st.state(), h1, h_in16=h0)
    st.close()


def test_last_layer_of_a_stack_wide_down():
    cfg, L, B = MID, 3, 8
    h0 = synth.activations(B, cfg["hidden"], 84)
    st = Stack(cfg, L, seed=83, batch=B)
    prev = Stack(cfg, L - 1, seed=83, batch=B, ptrs=st.ptrs[:-1])
    prev.run(h0)
    t_prev = prev.state()["t2"]
    hL = st.run(h0)
    check_layer(cfg, 83, L - 1, st.state(), hL, t_prev=t_prev, rows=sampled_rows(256, 1))
    st.close()
    prev.close()


@pytest.mark.parametrize("engine", ["per_product", "batched"])
def test_rows_do_not_depend_on_the_batch(engine):
    """Each batch row's result is the same whatever the other rows hold and
    whatever the batch size, within one engine (the per-product path: one or
    two n-tiles of the tensor-core product; the batched engine: fragment
    buffers of 2, 4 or 8 columns)."""
    cfg = SMALL
    extra = q4.Q4_DEC_BATCH_ENGINE if engine == "batched" else 0
    full_b = 16 if engine == "per_product" else 8
    h16 = synth.activations(full_b, cfg["hidden"], 90)
    full = Stack(cfg, 2, seed=91, batch=full_b, mode=q4.Q4_DEC_FUSED | extra)
    a = full.run(h16)
    for b in (2, 5, 8):
        if b >= full_b:
            continue
        part = Stack(cfg, 2, seed=91, batch=b, ptrs=full.ptrs, mode=q4.Q4_DEC_FUSED | extra)
        got = part.run(h16[:b])
        assert np.array_equal(got, a[:b]), b
        part.close()
    # change the other rows: row 0 unchanged
    h_mix = h16.copy()
    h_mix[1:] = synth.activations(full_b - 1, cfg["hidden"], 92)
    assert np.array_equal(full.run(h_mix)[0], a[0])
    full.close()


@pytest.mark.parametrize("cfg", [TINY, SMALL], ids=["tiny", "small"])
def test_batched_engine_fused_per_layer_identical(cfg):
    """The batched engine's whole-stack launch and its per-layer launches give
    the same bits (the same units on the same CTAs, sums in the same order)."""
    B, L = 6, 3
    h0 = synth.activations(B, cfg["hidden"], 88)
    fused = Stack(cfg, L, seed=89, batch=B, mode=BT)
    per = Stack(cfg, L, seed=89, batch=B, mode=q4.Q4_DEC_PER_LAYER | q4.Q4_DEC_BATCH_ENGINE, ptrs=fused.ptrs)
    a = fused.run(h0, reps=2)
    b = per.run(h0, reps=2)
    assert np.array_equal(a, b)
    fused.close()
    per.close()


def test_batched_engine_agrees_with_per_product():
    """The batched engine and the per-product path compute the same layer; their
    projections agree within the product error bound, so one layer's output
    (binary16) agrees closely row by row, and each stage of the batched engine
    checks against the oracle."""
    cfg, B = SMALL, 8
    h0 = synth.activations(B, cfg["hidden"], 86)
    a = Stack(cfg, 1, seed=87, batch=B, mode=BT)
    b = Stack(cfg, 1, seed=87, batch=B, ptrs=a.ptrs)
    ha, hb = a.run(h0), b.run(h0)
    sa, sb = a.state(), b.state()
    assert np.array_equal(sa["x"], sb["x"])          # the same input RMSNorm
    check_layer(cfg, 87, 0, sa, ha, h_in16=h0)
    fa, fb = ha.view(np.float16).astype(np.float64), hb.view(np.float16).astype(np.float64)
    for r in range(B):
        assert np.linalg.norm(fa[r] - fb[r]) <= 2e-3 * np.linalg.norm(fb[r]), r
    a.close()
    b.close()


@pytest.mark.parametrize("mode", [q4.Q4_DEC_FUSED, BT], ids=["per_product", "batched"])
def test_graph_eager_and_pointer_change_identical(mode):
    cfg, B = TINY, 4
    h0 = synth.activations(B, cfg["hidden"], 93)
    st = Stack(cfg, 3, seed=94, batch=B, mode=mode)
    a = st.run(h0, graph=True, reps=2)
    b = st.run(h0, graph=False, reps=2)
    c = st.run(h0, graph=True, reps=2)     # a new buffer: captured again
    assert np.array_equal(a, b) and np.array_equal(a, c)
    st.close()


def test_drift_against_oracle_chain():
    cfg, L, B = SMALL, 3, 4
    h0 = synth.activations(B, cfg["hidden"], 95)
    st = Stack(cfg, L, seed=96, batch=B)
    hL = st.run(h0)
    z = ora.rmsnorm(h0, B, cfg["hidden"])
    for l in range(L):
        ws = [synth.q4_matrix(n, k, 96, synth.tensor_id(l, p))
              for p, (n, k) in enumerate(synth.layer_dims(cfg["hidden"], cfg["q_dim"], cfg["kv_dim"], cfg["ffn"]))]
        z, _ = ora.layer(ws, z, B, cfg["hidden"], cfg["q_dim"], cfg["kv_dim"], cfg["ffn"], cfg["head_dim"])
    a = hL.view(np.float16).astype(np.float64)
    b = z.view(np.float16).astype(np.float64)
    for r in range(B):
        assert np.linalg.norm(a[r] - b[r]) / np.linalg.norm(b[r]) < 1e-2, r
    st.close()


@pytest.mark.parametrize("flags", [0, q4.Q4_STREAM_POISON], ids=["plain", "poison"])
def test_streamed_equals_resident(flags):
    cfg, L, B = SMALL, 4, 8
    shape = q4.LayerShape.of(**cfg)
    h0 = synth.activations(B, cfg["hidden"], 97)
    blocks, hptrs = model.host_layers(shape, L, 98)
    stride = model.layer_stride(shape)
    bufs = [torch.empty(stride, dtype=torch.uint8, device="cuda") for _ in range(2)]
    ws, offs, nb = model.workspace(shape, L, B)
    ring = q4.q4_stream_create(shape, hptrs, B, bufs[0], bufs[1], stride, ws, nb, flags)
    h = dev_u16(h0.reshape(-1))
    for _ in range(2):
        q4.q4_stream_layers(ring, h)
    torch.cuda.synchronize()
    assert q4.q4_stream_status(ring) == 0
    got = host_u16(h).reshape(B, -1)
    q4.q4_stream_destroy(ring)
    ref = Stack(cfg, L, seed=98, batch=B)
    want = ref.run(h0, reps=2)
    assert np.array_equal(got, want)
    ref.close()


@pytest.mark.parametrize("mode", [q4.Q4_DEC_FUSED, BT], ids=["per_product", "batched"])
def test_8b_stack_batch8_full_size(mode):
    cfg = dict(synth.LLAMA_8B)
    L = cfg.pop("n_layers")
    B = 8
    st = Stack(cfg, L, seed=0, batch=B, mode=mode)
    prev = Stack(cfg, L - 1, seed=0, batch=B, ptrs=st.ptrs[:-1], mode=mode)
    h0 = synth.activations(B, cfg["hidden"], 1)
    prev.run(h0)
    t_prev = prev.state()["t2"]
    hL = st.run(h0)
    stats = st.state()
    check_layer(cfg, 0, L - 1, stats, hL, t_prev=t_prev, rows=sampled_rows(96, 2))
    assert np.all(np.isfinite(hL.view(np.float16).astype(np.float64)))
    for name in ("qkv", "o", "g", "u", "dn", "t1", "t2"):
        assert np.all(np.isfinite(stats[name])), name
    st.close()
    prev.close()


@pytest.mark.parametrize("mode", [q4.Q4_DEC_FUSED, BT], ids=["per_product", "batched"])
def test_70b_shape_batch8_two_layers(mode):
    """70B-shaped layers (hidden 8192, ffn 28672: 4- and 14-chunk rows) at batch
    8: the second layer checked step by step on sampled rows."""
    cfg = dict(synth.LLAMA_70B)
    cfg.pop("n_layers")
    B, L = 8, 2
    st = Stack(cfg, L, seed=5, batch=B, mode=mode)
    prev = Stack(cfg, L - 1, seed=5, batch=B, ptrs=st.ptrs[:-1], mode=mode)
    h0 = synth.activations(B, cfg["hidden"], 6)
    prev.run(h0)
    t_prev = prev.state()["t2"]
    hL = st.run(h0)
    check_layer(cfg, 5, L - 1, st.state(), hL, t_prev=t_prev, rows=sampled_rows(64, 3))
    st.close()
    prev.close()


def test_batched_engine_wait_runs_out_and_reports():
    """Flags that never carry the awaited tag: every wait of the batched engine
    gives up after its poll limit, the status word reports it (bit 1), and the
    decoder stays usable (the next token equals the first)."""
    st = Stack(TINY, 2, seed=44, batch=4, mode=BT)
    h0 = synth.activations(4, TINY["hidden"], 45)
    a = st.run(h0)
    status = q4.q4_decoder_debug_stall(st.dec, 2000)
    assert status & 1
    b = st.run(h0)
    assert np.array_equal(a, b)
    st.close()


def test_batched_shape_limits():
    shape = q4.LayerShape.of(**TINY)
    wbuf, ptrs = model.resident_layers(shape, 1, 1)
    ws, offs, nb = model.workspace(shape, 1, 16)
    with pytest.raises(q4.Q4Error):
        q4.q4_decoder_create(shape, ptrs, 17, ws, nb)
    bad = q4.LayerShape.of(**dict(TINY, ffn=1056))     # ffn a multiple of 32, not of 256
    with pytest.raises(q4.Q4Error):
        q4.q4_decoder_create(bad, ptrs, 4, ws, nb)
    # the batched engine: batch 2..8 and widths of whole 2048-column chunks
    with pytest.raises(q4.Q4Error):
        q4.q4_decoder_create(shape, ptrs, 9, ws, nb, BT)
    odd = q4.LayerShape.of(**ODD)
    wodd, podd = model.resident_layers(odd, 1, 1)
    wso, _, nbo = model.workspace(odd, 1, 4)
    with pytest.raises(q4.Q4Error):
        q4.q4_decoder_create(odd, podd, 4, wso, nbo, BT)
