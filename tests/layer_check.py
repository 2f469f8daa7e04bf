"""Step-by-step check of one decoder layer run on the GPU.

Each projection is checked against the oracle fed the GPU's own binary16
input of that projection, with the accepted error bound; each glue step is
checked against the oracle's glue applied to the GPU's own inputs: within one
binary16 ulp where the GPU rounds an fp32 value that the oracle computes in
double, within one fp32 rounding for the fp32 residual sums, and exactly where
both sides round the same fp32 value.  ``rows`` restricts the projection
checks to sampled output rows.
"""
import numpy as np

import oracle as ora
from weight_streaming_q4_gb300 import model, synth
from gpu_util import assert_within_tol, f16_ulps, host_f32, host_u16


def read_ws(ws, offs, cfg, batch=1):
    H, Q, KV, F = cfg["hidden"], cfg["q_dim"], cfg["kv_dim"], cfg["ffn"]
    import torch
    get = lambda name, dt, n: model.ws_view(ws, offs, name, dt, n)
    return dict(
        qkv=host_f32(get("qkv", torch.float32, batch * (Q + 2 * KV))).reshape(batch, -1),
        o=host_f32(get("o", torch.float32, batch * H)).reshape(batch, -1),
        g=host_f32(get("gate", torch.float32, batch * F)).reshape(batch, -1),
        u=host_f32(get("up", torch.float32, batch * F)).reshape(batch, -1),
        dn=host_f32(get("down", torch.float32, batch * H)).reshape(batch, -1),
        act=host_u16(get("act", torch.int16, batch * F)).reshape(batch, -1),
        x=host_u16(get("x", torch.int16, batch * H)).reshape(batch, -1),
        attn=host_u16(get("attn", torch.int16, batch * Q)).reshape(batch, -1),
        x2=host_u16(get("x2", torch.int16, batch * H)).reshape(batch, -1),
        t1=host_f32(get("t1", torch.float32, batch * H)).reshape(batch, -1),
        t2=host_f32(get("t2", torch.float32, batch * H)).reshape(batch, -1),
    )


def _proj(layer, p, cfg, seed, x_bits, y_gpu, rows, what):
    n, k = synth.layer_dims(cfg["hidden"], cfg["q_dim"], cfg["kv_dim"], cfg["ffn"])[p]
    tid = synth.tensor_id(layer, p)
    if rows is None:
        w = synth.q4_matrix(n, k, seed, tid)
        y_ref, s_ref = ora.gemv(w, x_bits, n, k, batch=x_bits.shape[0], threads=8)
        assert_within_tol(y_gpu, y_ref, s_ref, what)
    else:
        r = np.asarray(rows(n))
        w = synth.q4_rows(r, k, seed, tid).reshape(-1)
        y_ref, s_ref = ora.gemv(w, x_bits, len(r), k, batch=x_bits.shape[0])
        assert_within_tol(y_gpu[:, r], y_ref, s_ref, what)


def _fp32_sum_ok(t_gpu, z_bits, o_gpu, what):
    ref = ora.add(z_bits, o_gpu)                 # exact double sum of the GPU's operands
    assert np.all(np.abs(t_gpu - ref) <= 2.0 ** -24 * np.abs(ref) + 1e-45), what


def check_layer(cfg, seed, layer, st, h_out, h_in16=None, t_prev=None, rows=None, eps=1e-5):
    """st = read_ws(...) after the layer ran; h_out = the caller's buffer after it
    (the normalised last residual sum when this is the last layer, else None);
    the layer input is the caller's binary16 h_in16 (first layer) or the previous
    layer's fp32 residual sum t_prev."""
    B = st["x"].shape[0]
    H, Q, KV, F, hd = cfg["hidden"], cfg["q_dim"], cfg["kv_dim"], cfg["ffn"], cfg["head_dim"]
    z_ref = ora.rmsnorm(h_in16, B, H, eps) if h_in16 is not None else ora.rmsnorm_d(t_prev, B, H, eps)
    assert f16_ulps(st["x"], z_ref).max() <= 1, "input rmsnorm"
    qkv = st["qkv"]
    _proj(layer, 0, cfg, seed, st["x"], qkv[:, :Q], rows, "q")
    _proj(layer, 1, cfg, seed, st["x"], qkv[:, Q:Q + KV], rows, "k")
    _proj(layer, 2, cfg, seed, st["x"], qkv[:, Q + KV:], rows, "v")
    assert np.array_equal(st["attn"], ora.attn_ctx1(qkv[:, Q + KV:], B, Q, KV, hd)), "attention"
    _proj(layer, 3, cfg, seed, st["attn"], st["o"], rows, "o")
    _fp32_sum_ok(st["t1"], st["x"], st["o"], "t1 = z + o")
    assert f16_ulps(st["x2"], ora.rmsnorm_d(st["t1"], B, H, eps)).max() <= 1, "rmsnorm t1"
    _proj(layer, 4, cfg, seed, st["x2"], st["g"], rows, "gate")
    _proj(layer, 5, cfg, seed, st["x2"], st["u"], rows, "up")
    assert f16_ulps(st["act"], ora.silu_mul(st["g"], st["u"])).max() <= 1, "silu*up"
    _proj(layer, 6, cfg, seed, st["act"], st["dn"], rows, "down")
    _fp32_sum_ok(st["t2"], st["x2"], st["dn"], "t2 = z1 + down")
    if h_out is not None:
        assert f16_ulps(h_out, ora.rmsnorm_d(st["t2"], B, H, eps)).max() <= 1, "output rmsnorm"


def sampled_rows(count, seed=0):
    rng = np.random.default_rng(seed)
    return lambda n: np.sort(rng.choice(n, min(count, n), replace=False))
