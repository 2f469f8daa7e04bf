"""q4_attn_decode / q4_kv_append on the GPU against the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle as ora
import weight_streaming_q4_gb300 as q4
from weight_streaming_q4_gb300 import build
from gpu_util import host_u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    ora.build()


def make_case(n_q, n_kv, hd, capacity, seed, q_scale=1.0):
    rng = np.random.default_rng(seed)
    kv = n_kv * hd
    q = (rng.normal(size=n_q * hd) * q_scale).astype(np.float32)
    kc = rng.normal(size=(capacity, kv)).astype(np.float16).view(np.uint16)
    vc = rng.normal(size=(capacity, kv)).astype(np.float16).view(np.uint16)
    return q, kc, vc


class Attn:
    def __init__(self, q, kc, vc, n_q, n_kv, hd, capacity):
        self.n_q, self.n_kv, self.hd, self.capacity = n_q, n_kv, hd, capacity
        self.q = torch.from_numpy(q).cuda()
        self.kc = torch.from_numpy(kc.view(np.int16).copy()).cuda()
        self.vc = torch.from_numpy(vc.view(np.int16).copy()).cuda()
        self.ctx = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.out = torch.empty(n_q * hd, dtype=torch.int16, device="cuda")
        self.wsb = q4.q4_attn_workspace_bytes(n_q, n_kv, hd, capacity)
        self.ws = torch.zeros(self.wsb, dtype=torch.uint8, device="cuda")

    def run(self, ctx, stream=None):
        self.ctx.fill_(ctx)
        q4.q4_attn_decode(self.q, self.kc, self.vc, self.ctx, self.capacity, self.n_q, self.n_kv, self.hd,
                          self.out, self.ws, self.wsb, stream=stream)
        torch.cuda.synchronize()
        return host_u16(self.out)


def check(got_bits, q, kc, vc, ctx, n_q, n_kv, hd, what=""):
    o_ref, sabs = ora.attn_decode(q.astype(np.float64), kc, vc, ctx, n_q, n_kv, hd)
    got = got_bits.view(np.float16).astype(np.float64)
    err = np.abs(got - o_ref)
    tol = 1e-3 * sabs + 1e-6
    bad = err > tol
    assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} outside, worst err/tol {float((err / tol).max()):.3g}"


SHAPES = [(32, 8, 128), (64, 8, 128), (8, 8, 64), (16, 1, 256), (12, 4, 192)]


@pytest.mark.parametrize("n_q,n_kv,hd", SHAPES, ids=[f"{a}x{b}x{c}" for a, b, c in SHAPES])
@pytest.mark.parametrize("ctx", [1, 5, 127, 128, 129, 1000, 1024])
def test_attention_parity(n_q, n_kv, hd, ctx):
    capacity = 1024
    q, kc, vc = make_case(n_q, n_kv, hd, capacity, seed=ctx * 7 + hd, q_scale=0.25)
    a = Attn(q, kc, vc, n_q, n_kv, hd, capacity)
    check(a.run(ctx), q, kc, vc, ctx, n_q, n_kv, hd, f"ctx {ctx}")


def test_one_position_is_the_value_exactly():
    n_q, n_kv, hd, cap = 32, 8, 128, 512
    q, kc, vc = make_case(n_q, n_kv, hd, cap, seed=3, q_scale=3.0)
    got = Attn(q, kc, vc, n_q, n_kv, hd, cap).run(1)
    v0 = vc[0].reshape(n_kv, hd)
    assert np.array_equal(got.reshape(n_q, hd), np.stack([v0[h // (n_q // n_kv)] for h in range(n_q)]))


def test_sharp_and_flat_softmax():
    n_q, n_kv, hd, cap = 8, 2, 128, 4096
    for q_scale, seed in ((0.0, 4), (4.0, 5)):     # uniform weights; a few dominant positions
        q, kc, vc = make_case(n_q, n_kv, hd, cap, seed=seed, q_scale=q_scale)
        check(Attn(q, kc, vc, n_q, n_kv, hd, cap).run(4096), q, kc, vc, 4096, n_q, n_kv, hd, f"scale {q_scale}")


def test_ctx_beyond_capacity_is_clamped_and_runs_deterministic():
    n_q, n_kv, hd, cap = 32, 8, 128, 512
    q, kc, vc = make_case(n_q, n_kv, hd, cap, seed=6, q_scale=0.5)
    a = Attn(q, kc, vc, n_q, n_kv, hd, cap)
    x = a.run(10 ** 6)
    assert np.array_equal(x, a.run(cap))
    assert np.array_equal(x, a.run(cap))


def test_one_graph_serves_every_length_of_its_bucket():
    n_q, n_kv, hd, cap = 32, 8, 128, 2048
    q, kc, vc = make_case(n_q, n_kv, hd, cap, seed=7, q_scale=0.5)
    a = Attn(q, kc, vc, n_q, n_kv, hd, cap)
    direct = {c: a.run(c) for c in (3, 700, 2048)}
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        q4.q4_attn_decode(a.q, a.kc, a.vc, a.ctx, cap, n_q, n_kv, hd, a.out, a.ws, a.wsb, stream=s)
        s.synchronize()
        with torch.cuda.graph(g, stream=s):
            q4.q4_attn_decode(a.q, a.kc, a.vc, a.ctx, cap, n_q, n_kv, hd, a.out, a.ws, a.wsb, stream=s)
    for c, want in direct.items():
        a.ctx.fill_(c)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(host_u16(a.out), want), c


def test_kv_append_writes_binary16_rows():
    kv, cap = 1024, 64
    kc = torch.zeros(cap * kv, dtype=torch.int16, device="cuda")
    vc = torch.zeros(cap * kv, dtype=torch.int16, device="cuda")
    rng = np.random.default_rng(8)
    k = rng.normal(size=kv).astype(np.float32)
    v = rng.normal(size=kv).astype(np.float32)
    pos = torch.tensor([17], dtype=torch.int32, device="cuda")
    q4.q4_kv_append(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), kc, vc, pos, cap, kv)
    pos.fill_(cap)      # outside the cache: ignored
    q4.q4_kv_append(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), kc, vc, pos, cap, kv)
    torch.cuda.synchronize()
    K = host_u16(kc).reshape(cap, kv)
    V = host_u16(vc).reshape(cap, kv)
    assert np.array_equal(K[17], ora.double_to_half(k.astype(np.float64)))
    assert np.array_equal(V[17], ora.double_to_half(v.astype(np.float64)))
    assert not K[np.arange(cap) != 17].any() and not V[np.arange(cap) != 17].any()


def test_argument_checks():
    t = torch.zeros(1 << 16, dtype=torch.int16, device="cuda")
    ctx = torch.ones(1, dtype=torch.int32, device="cuda")
    for (cap, nq, nkv, hd) in ((500, 32, 8, 128), (512, 30, 8, 128), (512, 32, 8, 96), (512, 34, 2, 128)):
        with pytest.raises(q4.Q4Error) as e:
            q4.q4_attn_decode(t, t, t, ctx, cap, nq, nkv, hd, t, t, 1 << 17)
        assert e.value.status == q4.Q4_ERR_ARG
    with pytest.raises(q4.Q4Error) as e:
        q4.q4_attn_decode(t, t, t, ctx, 512, 32, 8, 128, t, t, q4.q4_attn_workspace_bytes(32, 8, 128, 512) - 1)
    assert e.value.status == q4.Q4_ERR_OOM


@pytest.mark.parametrize("cap,ctx,hd", [(16384, 16384, 128), (16384, 9000, 128), (8192, 8192, 256),
                                        (65536, 40000, 64)])
def test_long_buckets_take_several_rounds(cap, ctx, hd):
    """Spans longer than one round of positions per CTA: the running softmax
    state is rescaled across rounds (and rounds of 128 positions at head_dim
    256)."""
    n_q, n_kv = 8, 2
    q, kc, vc = make_case(n_q, n_kv, hd, cap, seed=ctx % 97 + hd, q_scale=0.5)
    check(Attn(q, kc, vc, n_q, n_kv, hd, cap).run(ctx), q, kc, vc, ctx, n_q, n_kv, hd, f"cap {cap} ctx {ctx}")
