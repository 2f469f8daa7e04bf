"""q4_decoder_create_kv: decoder layers that attend over per-layer KV caches.

Each token runs, per layer, the q|k|v product, the store of the token's k and
v (binary16) in row pos of the layer's caches, decode attention over rows
0..pos and the rest of the layer; the position advances after the last layer.
Checked against the oracle step by step on the GPU's own inputs (products
within the error bound, the cache rows bit for bit, the attention within its
bound), and as a chain of layers and tokens against the oracle's own chain.
"""
import numpy as np
import pytest
import torch

import oracle as ora
import weight_streaming_q4_gb300 as q4
from weight_streaming_q4_gb300 import build, model, synth
from gpu_util import dev_u16, f16_ulps, host_u16
from layer_check import _fp32_sum_ok, _proj, read_ws

pytestmark = pytest.mark.gpu

TINY = dict(hidden=256, q_dim=256, kv_dim=128, ffn=1024, head_dim=64)
SMALL = dict(hidden=2048, q_dim=2048, kv_dim=512, ffn=4096, head_dim=128)


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    ora.build()


class KVStack:
    def __init__(self, cfg, n_layers, seed, capacity):
        self.cfg, self.n_layers, self.capacity = cfg, n_layers, capacity
        self.shape = q4.LayerShape.of(**cfg)
        self.wbuf, self.ptrs = model.resident_layers(self.shape, n_layers, seed)
        self.ws, self.offs, self.ws_bytes = model.workspace(self.shape, n_layers, 1)
        kvd, hd = cfg["kv_dim"], cfg["head_dim"]
        self.kc = [torch.zeros(capacity * kvd, dtype=torch.int16, device="cuda") for _ in range(n_layers)]
        self.vc = [torch.zeros(capacity * kvd, dtype=torch.int16, device="cuda") for _ in range(n_layers)]
        self.pos = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.awb = q4.q4_attn_workspace_bytes(cfg["q_dim"] // hd, kvd // hd, hd, capacity)
        self.aws = torch.empty(self.awb, dtype=torch.uint8, device="cuda")
        self.dec = q4.q4_decoder_create_kv(self.shape, self.ptrs, capacity, self.kc, self.vc, self.pos, self.aws,
                                           self.awb, self.ws, self.ws_bytes)

    def run(self, h_np, graph=True):
        h = dev_u16(h_np.reshape(-1))
        (q4.q4_layer_decode if graph else q4.q4_layer_decode_eager)(self.dec, h)
        torch.cuda.synchronize()
        assert q4.q4_decoder_status(self.dec) == 0
        return host_u16(h).reshape(1, -1)

    def cache(self, layer):
        kvd = self.cfg["kv_dim"]
        return (host_u16(self.kc[layer]).reshape(self.capacity, kvd).copy(),
                host_u16(self.vc[layer]).reshape(self.capacity, kvd).copy())

    def close(self):
        q4.q4_decoder_destroy(self.dec)


def check_kv_layer(cfg, seed, layer, st, kc, vc, kc_before, vc_before, pos, eps=1e-5):
    """The last layer of a KV decoder after the token at `pos`, on the GPU's own inputs."""
    H, Q, KV, hd = cfg["hidden"], cfg["q_dim"], cfg["kv_dim"], cfg["head_dim"]
    qkv = st["qkv"]
    _proj(layer, 0, cfg, seed, st["x"], qkv[:, :Q], None, "q")
    _proj(layer, 1, cfg, seed, st["x"], qkv[:, Q:Q + KV], None, "k")
    _proj(layer, 2, cfg, seed, st["x"], qkv[:, Q + KV:], None, "v")
    # the cache row of this token holds f16 of the GPU's own fp32 k and v; no other row changed
    assert np.array_equal(kc[pos], ora.double_to_half(qkv[0, Q:Q + KV])), "k cache row"
    assert np.array_equal(vc[pos], ora.double_to_half(qkv[0, Q + KV:])), "v cache row"
    others = np.arange(kc.shape[0]) != pos
    assert np.array_equal(kc[others], kc_before[others]) and np.array_equal(vc[others], vc_before[others])
    # attention over rows 0..pos, from the GPU's q and caches
    o_ref, sabs = ora.attn_decode(qkv[0, :Q], kc, vc, pos + 1, Q // hd, KV // hd, hd)
    got = st["attn"][0].view(np.float16).astype(np.float64)
    err = np.abs(got - o_ref)
    tol = 1e-3 * sabs + 1e-6
    assert np.all(err <= tol), f"attention: worst err/tol {float((err / tol).max()):.3g}"
    _proj(layer, 3, cfg, seed, st["attn"], st["o"], None, "o")
    _fp32_sum_ok(st["t1"], st["x"], st["o"], "t1 = z + o")
    assert f16_ulps(st["x2"], ora.rmsnorm_d(st["t1"], 1, H, eps)).max() <= 1, "rmsnorm t1"
    _proj(layer, 4, cfg, seed, st["x2"], st["g"], None, "gate")
    _proj(layer, 5, cfg, seed, st["x2"], st["u"], None, "up")
    assert f16_ulps(st["act"], ora.silu_mul(st["g"], st["u"])).max() <= 1, "silu*up"
    _proj(layer, 6, cfg, seed, st["act"], st["dn"], None, "down")
    _fp32_sum_ok(st["t2"], st["x2"], st["dn"], "t2 = z1 + down")


@pytest.mark.parametrize("cfg", [TINY, SMALL], ids=["tiny", "small"])
def test_position_zero_is_the_context_one_decoder(cfg):
    h0 = synth.activations(1, cfg["hidden"], 100)
    kv = KVStack(cfg, 3, seed=101, capacity=128)
    a = kv.run(h0)
    shape = q4.LayerShape.of(**cfg)
    ws, offs, nb = model.workspace(shape, 3, 1)
    dec = q4.q4_decoder_create(shape, kv.ptrs, 1, ws, nb, q4.Q4_DEC_FUSED)
    h = dev_u16(h0.reshape(-1))
    q4.q4_layer_decode(dec, h)
    torch.cuda.synchronize()
    assert np.array_equal(a, host_u16(h).reshape(1, -1))
    assert int(kv.pos.item()) == 1
    q4.q4_decoder_destroy(dec)
    kv.close()


@pytest.mark.parametrize("cfg,tokens", [(TINY, 6), (SMALL, 4)], ids=["tiny", "small"])
def test_tokens_step_by_step(cfg, tokens):
    L = 2
    kv = KVStack(cfg, L, seed=110, capacity=128)
    for tok in range(tokens):
        kc0, vc0 = kv.cache(L - 1)
        kv.run(synth.activations(1, cfg["hidden"], 111 + tok))
        kc, vc = kv.cache(L - 1)
        check_kv_layer(cfg, 110, L - 1, read_ws(kv.ws, kv.offs, cfg), kc, vc, kc0, vc0, tok)
    assert int(kv.pos.item()) == tokens
    kv.close()


@pytest.mark.parametrize("pos", [200, 1500, 4095])
def test_long_context_positions(pos):
    """A 4096-position bucket (clusters of 16 CTAs, 256 positions each, two
    rounds of 128 at head_dim 128): earlier rows filled with seeded binary16
    values, the token's row in the second round of CTA 0 (200), of CTA 5
    (1500) and of the last CTA (4095); the last layer checked step by step."""
    cfg, L, cap = SMALL, 2, 4096
    kv = KVStack(cfg, L, seed=130, capacity=cap)
    for l in range(L):
        synth.device_fill_normal_f16(kv.kc[l].data_ptr(), cap * cfg["kv_dim"], seed=131, tid=2 * l)
        synth.device_fill_normal_f16(kv.vc[l].data_ptr(), cap * cfg["kv_dim"], seed=131, tid=2 * l + 1)
    kv.pos.fill_(pos)
    torch.cuda.synchronize()
    kc0, vc0 = kv.cache(L - 1)
    kv.run(synth.activations(1, cfg["hidden"], 132))
    kc, vc = kv.cache(L - 1)
    check_kv_layer(cfg, 130, L - 1, read_ws(kv.ws, kv.offs, cfg), kc, vc, kc0, vc0, pos)
    assert int(kv.pos.item()) == pos + 1
    kv.close()


def test_chain_against_the_oracle():
    """Three layers, eight tokens (graph and eager calls alternating): the
    GPU's outputs against the oracle's own chain of KV layers (drift gate)."""
    cfg, L, T, cap, seed = TINY, 3, 8, 128, 120
    kv = KVStack(cfg, L, seed=seed, capacity=cap)
    H, Q, KV, F, hd = cfg["hidden"], cfg["q_dim"], cfg["kv_dim"], cfg["ffn"], cfg["head_dim"]
    wts = [[synth.q4_matrix(n, k, seed, synth.tensor_id(l, p))
            for p, (n, k) in enumerate(synth.layer_dims(H, Q, KV, F))] for l in range(L)]
    kcs = [np.zeros((cap, KV), np.uint16) for _ in range(L)]
    vcs = [np.zeros((cap, KV), np.uint16) for _ in range(L)]
    for tok in range(T):
        h0 = synth.activations(1, H, 121 + tok)
        got = kv.run(h0, graph=tok % 2 == 0).view(np.float16).astype(np.float64)
        z = ora.rmsnorm(h0, 1, H).reshape(-1)
        for l in range(L):
            z, _ = ora.layer_kv(wts[l], z, kcs[l], vcs[l], tok, H, Q, KV, F, hd)
        ref = z.view(np.float16).astype(np.float64)
        assert np.linalg.norm(got - ref) / np.linalg.norm(ref) < 1e-2, f"token {tok}"
    # the caches the GPU built agree with the oracle's (the same drift gate, per cache row)
    f = lambda a: a.view(np.float16).astype(np.float64)
    for l in range(L):
        kc, vc = kv.cache(l)
        for got_c, ref_c in ((kc, kcs[l]), (vc, vcs[l])):
            rel = np.linalg.norm(f(got_c[:T]) - f(ref_c[:T]), axis=1) / np.linalg.norm(f(ref_c[:T]), axis=1)
            assert rel.max() < 1e-2, f"layer {l} cache rows"
        assert not kc[T:].any() and not vc[T:].any()
    kv.close()


def test_bucket_sizes_and_position_counter():
    """A 512-position bucket filled to 300 positions: the counter set by the
    caller is where the next token goes, and the attention covers rows 0..pos."""
    cfg, L = TINY, 1
    kv = KVStack(cfg, L, seed=130, capacity=512)
    rng = np.random.default_rng(131)
    kvd = cfg["kv_dim"]
    pre_k = rng.normal(size=(512, kvd)).astype(np.float16)
    pre_v = rng.normal(size=(512, kvd)).astype(np.float16)
    kv.kc[0].copy_(torch.from_numpy(pre_k.view(np.int16).reshape(-1)).cuda())
    kv.vc[0].copy_(torch.from_numpy(pre_v.view(np.int16).reshape(-1)).cuda())
    kv.pos.fill_(299)
    kc0, vc0 = kv.cache(0)
    kv.run(synth.activations(1, cfg["hidden"], 132))
    kc, vc = kv.cache(0)
    check_kv_layer(cfg, 130, 0, read_ws(kv.ws, kv.offs, cfg), kc, vc, kc0, vc0, 299)
    assert int(kv.pos.item()) == 300
    kv.close()


def test_position_outside_the_bucket_sets_status():
    cfg = TINY
    kv = KVStack(cfg, 1, seed=140, capacity=128)
    kv.pos.fill_(128)
    h = dev_u16(synth.activations(1, cfg["hidden"], 141).reshape(-1))
    q4.q4_layer_decode(kv.dec, h)
    torch.cuda.synchronize()
    assert q4.q4_decoder_status(kv.dec) == 32
    assert not host_u16(kv.kc[0]).any() and not host_u16(kv.vc[0]).any()
    kv.pos.fill_(5)
    kv.run(synth.activations(1, cfg["hidden"], 142))    # status cleared, next call normal
    kv.close()
