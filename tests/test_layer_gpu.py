"""q4_layer_decode (HBM-resident decoder stack under CUDA-graph capture)."""
import numpy as np
import pytest
import torch

import oracle as ora
import weight_streaming_q4_gb300 as q4
from weight_streaming_q4_gb300 import build, model, synth
from gpu_util import dev_u16, f16_ulps, host_u16
from layer_check import check_layer, read_ws, sampled_rows

pytestmark = pytest.mark.gpu

TINY = dict(hidden=256, q_dim=256, kv_dim=128, ffn=1024, head_dim=64)
SMALL = dict(hidden=2048, q_dim=2048, kv_dim=512, ffn=4096, head_dim=128)
MID = dict(hidden=1024, q_dim=1024, kv_dim=256, ffn=14336, head_dim=128)   # down rows 14336 wide
# down rows 20480 wide: the tagged down input is staged in two rounds, the second ragged
WIDE = dict(hidden=1024, q_dim=1024, kv_dim=256, ffn=20480, head_dim=128)


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    ora.build()


class Stack:
    def __init__(self, cfg, n_layers, seed, mode=q4.Q4_DEC_FUSED):
        self.cfg = cfg
        self.shape = q4.LayerShape.of(**cfg)
        self.wbuf, self.ptrs = model.resident_layers(self.shape, n_layers, seed)
        self.ws, self.offs, self.ws_bytes = model.workspace(self.shape, n_layers, 1)
        self.dec = q4.q4_decoder_create(self.shape, self.ptrs, 1, self.ws, self.ws_bytes, mode)

    def run(self, h_np, graph=True, reps=1):
        h = dev_u16(h_np.reshape(-1))
        for _ in range(reps):
            (q4.q4_layer_decode if graph else q4.q4_layer_decode_eager)(self.dec, h)
        torch.cuda.synchronize()
        assert q4.q4_decoder_status(self.dec) == 0
        return host_u16(h).reshape(1, -1)

    def close(self):
        q4.q4_decoder_destroy(self.dec)


# the tensor-core engine (default), the CUDA-core engine with tagged words
# between phases, the CUDA-core engine with a flag barrier after every phase
ENGINES = {"tc": 0, "core": q4.Q4_DEC_CUDA_CORE, "barrier": q4.Q4_DEC_BARRIER}


@pytest.mark.parametrize("engine", list(ENGINES))
@pytest.mark.parametrize("cfg", [TINY, SMALL, MID, WIDE], ids=["tiny", "small", "mid", "wide"])
def test_one_layer_step_by_step(cfg, engine):
    st = Stack(cfg, 1, seed=21, mode=q4.Q4_DEC_FUSED | ENGINES[engine])
    h0 = synth.activations(1, cfg["hidden"], 22)
    h1 = st.run(h0)
    check_layer(cfg, 21, 0, read_ws(st.ws, st.offs, cfg), h1, h_in16=h0)
    st.close()


def test_last_layer_of_a_stack_and_drift():
    cfg, L = SMALL, 4
    h0 = synth.activations(1, cfg["hidden"], 6)
    # the input of the last layer: the residual sum after the first L-1 layers
    st_prev = Stack(cfg, L - 1, seed=5)
    st_prev.run(h0)
    t_prev = read_ws(st_prev.ws, st_prev.offs, cfg)["t2"]
    # GPU: all layers at once; the workspace then holds the last layer's intermediates
    st = Stack(cfg, L, seed=5)
    hL = st.run(h0)
    check_layer(cfg, 5, L - 1, read_ws(st.ws, st.offs, cfg), hL, t_prev=t_prev)
    # end-to-end against the oracle's own layer chain: drift stays small
    z = ora.rmsnorm(h0, 1, cfg["hidden"])
    for l in range(L):
        ws = [synth.q4_matrix(n, k, 5, synth.tensor_id(l, p))
              for p, (n, k) in enumerate(synth.layer_dims(cfg["hidden"], cfg["q_dim"], cfg["kv_dim"], cfg["ffn"]))]
        z, _ = ora.layer(ws, z, 1, cfg["hidden"], cfg["q_dim"], cfg["kv_dim"], cfg["ffn"], cfg["head_dim"])
    a = hL.view(np.float16).astype(np.float64)
    b = z.view(np.float16).astype(np.float64)
    assert np.linalg.norm(a - b) / np.linalg.norm(b) < 1e-2
    st.close()
    st_prev.close()


@pytest.mark.parametrize("engine", list(ENGINES))
def test_graph_eager_modes_identical(engine):
    cfg = TINY
    h0 = synth.activations(1, cfg["hidden"], 30)
    fused = Stack(cfg, 3, seed=31, mode=q4.Q4_DEC_FUSED | ENGINES[engine])
    per = Stack(cfg, 3, seed=31, mode=q4.Q4_DEC_PER_LAYER | ENGINES[engine])
    a = fused.run(h0, graph=True, reps=2)
    b = fused.run(h0, graph=False, reps=2)
    c = per.run(h0, graph=True, reps=2)
    d = per.run(h0, graph=False, reps=2)
    assert np.array_equal(a, b) and np.array_equal(a, c) and np.array_equal(a, d)
    fused.close()
    per.close()


def test_engines_agree_and_tc_head_dims():
    """The two batch-1 engines give the same layer within the products' error
    bound (each is checked against the oracle step by step above); the
    tensor-core engine also takes head dims that are not multiples of 64."""
    cfg = SMALL
    h0 = synth.activations(1, cfg["hidden"], 32)
    a = Stack(cfg, 2, seed=33, mode=q4.Q4_DEC_TENSOR_CORE).run(h0).view(np.float16).astype(np.float64)
    b = Stack(cfg, 2, seed=33, mode=q4.Q4_DEC_CUDA_CORE).run(h0).view(np.float16).astype(np.float64)
    assert np.linalg.norm(a - b) / np.linalg.norm(b) < 2e-3
    odd = dict(hidden=768, q_dim=768, kv_dim=192, ffn=2048, head_dim=48)
    st = Stack(odd, 1, seed=34, mode=q4.Q4_DEC_TENSOR_CORE)
    h0 = synth.activations(1, odd["hidden"], 35)
    h1 = st.run(h0)
    check_layer(odd, 34, 0, read_ws(st.ws, st.offs, odd), h1, h_in16=h0)
    st.close()
    with pytest.raises(q4.Q4Error):
        Stack(odd, 1, seed=34, mode=q4.Q4_DEC_CUDA_CORE)


@pytest.mark.parametrize("cfg", [SMALL, WIDE], ids=["small", "wide"])
def test_tagged_and_barrier_programs_agree(cfg):
    """The tagged program and the flag-barrier program of the CUDA-core engine
    compute the same layers; their RMSNorm sums of squares add up in different
    orders, so they agree within the products' error bound, not bit for bit."""
    h0 = synth.activations(1, cfg["hidden"], 36)
    a = Stack(cfg, 3, seed=37, mode=q4.Q4_DEC_CUDA_CORE).run(h0).view(np.float16).astype(np.float64)
    b = Stack(cfg, 3, seed=37, mode=q4.Q4_DEC_BARRIER).run(h0).view(np.float16).astype(np.float64)
    assert np.linalg.norm(a - b) / np.linalg.norm(b) < 2e-3


def test_protocol_selection():
    """Batch-1 decoders pass tagged words unless asked for the flag barrier
    (which only the CUDA-core engine has); the tensor-core engine always
    passes tagged words."""
    assert Stack(SMALL, 1, seed=38).dec and q4.q4_decoder_tagged(Stack(SMALL, 1, seed=38).dec)
    assert not q4.q4_decoder_tagged(Stack(SMALL, 1, seed=38, mode=q4.Q4_DEC_BARRIER).dec)
    assert q4.q4_decoder_tagged(Stack(SMALL, 1, seed=38, mode=q4.Q4_DEC_TENSOR_CORE).dec)
    assert q4.q4_decoder_tagged(Stack(SMALL, 1, seed=38, mode=q4.Q4_DEC_CUDA_CORE).dec)
    assert q4.q4_decoder_tagged(Stack(WIDE, 1, seed=38).dec)


# hidden above the tagged staging budget (8192 fp32 norm inputs): the decoder
# falls back to the flag-barrier program on its own
BROAD = dict(hidden=10240, q_dim=2048, kv_dim=512, ffn=2048, head_dim=128)


def test_wide_hidden_falls_back_to_flag_program():
    st = Stack(BROAD, 1, seed=39)
    assert not q4.q4_decoder_tagged(st.dec)
    h0 = synth.activations(1, BROAD["hidden"], 40)
    h1 = st.run(h0)
    check_layer(BROAD, 39, 0, read_ws(st.ws, st.offs, BROAD), h1, h_in16=h0)
    st.close()


@pytest.mark.parametrize("engine", ["tc", "core"])
def test_tagged_wait_runs_out_and_reports(engine):
    """A tagged input that never arrives: every wait gives up after its poll
    limit, the status word carries bit 16 (and, on the tensor-core engine, bit
    1 for a phase-flag wait that ran out), and the context and the decoder
    stay usable (the next token is exact)."""
    st = Stack(TINY, 2, seed=42, mode=q4.Q4_DEC_FUSED | ENGINES[engine])
    h0 = synth.activations(1, TINY["hidden"], 43)
    a = st.run(h0)
    status = q4.q4_decoder_debug_stall(st.dec, 2000)
    assert status & 16
    if engine == "tc":
        assert status & 1
    b = st.run(h0)
    assert np.array_equal(a, b)
    st.close()


def test_new_hidden_pointer_rewrites_program():
    cfg = TINY
    st = Stack(cfg, 2, seed=40)
    h0 = synth.activations(1, cfg["hidden"], 41)
    a = st.run(h0)
    b = st.run(h0)     # a new tensor, hence a new pointer
    assert np.array_equal(a, b)
    st.close()


def _full_stack(cfg, n_layers, seed, count):
    st = Stack(cfg, n_layers, seed)
    h0 = synth.activations(1, cfg["hidden"], seed + 1)
    # the last layer's own input: the residual sum after n_layers-1 layers, from a
    # second decoder (own workspace) over the same device weights
    ws2, offs2, nb2 = model.workspace(st.shape, n_layers - 1, 1)
    prev = q4.q4_decoder_create(st.shape, st.ptrs[:-1], 1, ws2, nb2, q4.Q4_DEC_FUSED)
    h = dev_u16(h0.reshape(-1))
    q4.q4_layer_decode(prev, h)
    torch.cuda.synchronize()
    assert q4.q4_decoder_status(prev) == 0
    t_prev = read_ws(ws2, offs2, cfg)["t2"]
    q4.q4_decoder_destroy(prev)
    hL = st.run(h0)
    stats = read_ws(st.ws, st.offs, cfg)
    check_layer(cfg, seed, n_layers - 1, stats, hL, t_prev=t_prev, rows=sampled_rows(count, seed))
    assert np.all(np.isfinite(hL.view(np.float16).astype(np.float64)))
    for name in ("qkv", "o", "g", "u", "dn", "t1", "t2"):
        assert np.all(np.isfinite(stats[name])), name
    st.close()


def test_8b_stack_full_size():
    cfg = dict(synth.LLAMA_8B)
    L = cfg.pop("n_layers")
    _full_stack(cfg, L, seed=0, count=192)


def test_70b_stack_full_size():
    cfg = dict(synth.LLAMA_70B)
    L = cfg.pop("n_layers")
    _full_stack(cfg, L, seed=0, count=96)
