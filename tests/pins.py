"""Pins for the CPU oracle: facts fixed by the format definition or by
mathematics, independent of the oracle's own code.

Each check takes the loaded oracle library, so the same pins can be run
against deliberately broken copies of the oracle (tests/test_oracle_mutants.py).
A check returns None when it holds and raises AssertionError otherwise.
"""
from __future__ import annotations

import os

import numpy as np

import oracle as ora
from weight_streaming_q4_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _block(d_bits: int, codes) -> np.ndarray:
    b = np.zeros(18, dtype=np.uint8)
    b[0] = d_bits & 0xFF
    b[1] = d_bits >> 8
    b[2:] = np.asarray(codes, dtype=np.uint8)
    return b


def _f16(v) -> np.ndarray:
    return np.asarray(v, dtype=np.float16).view(np.uint16)


def golden_blocks():
    """(block bytes, expected weights) pairs from the hand-built fixture."""
    out, blk = [], None
    with open(os.path.join(GOLDEN, "q4_0_hand_blocks.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            tag, rest = line.split(None, 1)
            if tag == "block":
                blk = np.frombuffer(bytes.fromhex(rest), dtype=np.uint8).copy()
            elif tag == "weights":
                out.append((blk, np.array([float(t) for t in rest.split()])))
    return out


def golden_gemv():
    vals = {}
    with open(os.path.join(GOLDEN, "q4_0_hand_gemv.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            tag, rest = line.split(None, 1)
            vals[tag] = rest
    w = np.frombuffer(bytes.fromhex(vals["row"].replace(" ", "")), dtype=np.uint8).copy()
    xs = []
    for tok in vals["x"].split():
        hexv, _, rep = tok.partition("*")
        xs += [int(hexv, 16)] * (int(rep) if rep else 1)
    return w, np.array(xs, dtype=np.uint16), float(vals["y"]), float(vals["s"])


# ------------------------------------------------------------------ binary16

def pin_half_decode_exhaustive(lib):
    bits = np.arange(65536, dtype=np.uint16)
    got = ora.half_to_double(bits, lib=lib)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def pin_half_encode(lib):
    rng = np.random.default_rng(1)
    # every finite binary16 value, the midpoints between neighbours (ties), and
    # random doubles over the whole range, including overflow and subnormals
    fin = np.arange(65536, dtype=np.uint16).view(np.float16)
    fin = fin[np.isfinite(fin)].astype(np.float64)
    fin = np.unique(fin)
    mids = (fin[:-1] + fin[1:]) / 2
    rnd = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-9, 6, 20000),
                          [0.0, -0.0, 65519.99, 65520.0, -65520.0, 1e6, 2.0 ** -25, 2.0 ** -26,
                           3 * 2.0 ** -26, np.inf, -np.inf]])
    v = np.concatenate([fin, mids, rnd])
    got = ora.double_to_half(v, lib=lib)
    with np.errstate(over="ignore"):
        ref = v.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


# ------------------------------------------------------------------ Q4_0 layout

def pin_golden_blocks(lib):
    for blk, expect in golden_blocks():
        got = ora.dequant(blk, 1, 32, lib=lib).ravel()
        assert np.array_equal(got, expect), (got, expect)


def pin_distinct_positions(lib):
    # every element of a block carries a distinct value: element j<16 comes
    # from the low nibble of byte j and element j+16 from its high nibble
    rng = np.random.default_rng(2)
    for _ in range(20):
        codes = rng.integers(0, 256, 16, dtype=np.uint8)
        d = float(rng.uniform(0.01, 2.0))
        dbits = int(_f16(d))
        dd = float(np.uint16(dbits).view(np.float16))
        got = ora.dequant(_block(dbits, codes), 1, 32, lib=lib).ravel()
        lo = (codes & 15).astype(np.float64) - 8
        hi = (codes >> 4).astype(np.float64) - 8
        assert np.array_equal(got, np.concatenate([lo, hi]) * dd)


def pin_block_indexing(lib):
    # block i of row n sits at byte offset (n * K/32 + i) * 18: give every
    # block a distinct scale and all-15 codes, so W[n][k] = 7 * d[n][k // 32]
    n_rows, k_dim = 3, 96
    nb = n_rows * k_dim // 32
    scales = _f16(np.arange(1, nb + 1) / 8.0)
    w = np.concatenate([_block(int(s), [0xFF] * 16) for s in scales])
    got = ora.dequant(w, n_rows, k_dim, lib=lib)
    ds = scales.view(np.float16).astype(np.float64).reshape(n_rows, k_dim // 32)
    assert np.array_equal(got, 7.0 * np.repeat(ds, 32, axis=1))


# ------------------------------------------------------------------ product closed forms

def pin_golden_gemv(lib):
    w, x, y_exp, s_exp = golden_gemv()
    y, s = ora.gemv(w, x, 1, 64, lib=lib)
    assert y[0, 0] == y_exp and s[0, 0] == s_exp, (y, s)


def pin_all_eight_is_zero(lib):
    rng = np.random.default_rng(3)
    n_rows, k_dim = 5, 256
    blocks = [_block(int(_f16(rng.uniform(-3, 3))), [0x88] * 16) for _ in range(n_rows * k_dim // 32)]
    w = np.concatenate(blocks)
    x = _f16(rng.standard_normal((2, k_dim)))
    y, s = ora.gemv(w, x, n_rows, k_dim, batch=2, lib=lib)
    assert np.all(y == 0.0) and np.all(s == 0.0)


def pin_single_nonzero(lib):
    # one code differs from 8 in the whole matrix: y = (q-8) * d * x exactly
    rng = np.random.default_rng(4)
    n_rows, k_dim = 4, 128
    for trial in range(30):
        nb = n_rows * k_dim // 32
        w = np.concatenate([_block(int(_f16(rng.uniform(0.001, 1))), [0x88] * 16) for _ in range(nb)])
        n = int(rng.integers(n_rows))
        k = int(rng.integers(k_dim))
        q = int(rng.choice([c for c in range(16) if c != 8]))
        blk = (n * (k_dim // 32) + k // 32) * 18
        j = k % 32
        byte = blk + 2 + (j % 16)
        if j < 16:
            w[byte] = (w[byte] & 0xF0) | q
        else:
            w[byte] = (w[byte] & 0x0F) | (q << 4)
        x = _f16(rng.standard_normal(k_dim))
        y, _ = ora.gemv(w, x, n_rows, k_dim, lib=lib)
        d = float(w[blk:blk + 2].view(np.uint16).view(np.float16)[0])
        xv = float(x.view(np.float16)[k])
        expect = np.zeros(n_rows)
        expect[n] = (q - 8) * d * xv  # exact in double: <= 4+11+11 significant bits
        assert np.array_equal(y[0], expect), (trial, y, expect)


def pin_constant_codes(lib):
    # all codes 15 (or 0) and x = 1: y = 7*32*d (or -8*32*d) per block
    rng = np.random.default_rng(5)
    for code, fac in ((0xFF, 7), (0x00, -8)):
        ds = rng.uniform(0.01, 1, 6)
        dbits = _f16(ds)
        w = np.concatenate([_block(int(b), [code] * 16) for b in dbits])
        x = _f16(np.ones(32 * 6))
        y, _ = ora.gemv(w, x, 1, 32 * 6, lib=lib)
        exact = sum(fac * 32 * float(b.view(np.float16)) for b in dbits)
        assert abs(y[0, 0] - exact) <= 1e-15 * abs(exact)


def _numpy_dense(w: np.ndarray, n_rows: int, k_dim: int) -> np.ndarray:
    # an independent vectorised dequantiser (numpy's own binary16 decode)
    blk = w.reshape(n_rows * k_dim // 32, 18)
    d = blk[:, :2].copy().view(np.uint16).view(np.float16).astype(np.float64)
    codes = blk[:, 2:]
    q = np.concatenate([codes & 15, codes >> 4], axis=1).astype(np.float64)
    return ((q - 8) * d).reshape(n_rows, k_dim)


def pin_brute_force(lib):
    for (n_rows, k_dim, batch, seed) in ((1, 32, 1, 0), (3, 64, 2, 1), (17, 256, 3, 2), (8, 1024, 1, 3)):
        w = synth.q4_matrix(n_rows, k_dim, seed, 9)
        x = synth.activations(batch, k_dim, seed)
        dense = _numpy_dense(w, n_rows, k_dim)
        xd = x.view(np.float16).astype(np.float64)
        ref = xd @ dense.T
        mag = np.abs(xd) @ np.abs(dense).T
        y, s = ora.gemv(w, x, n_rows, k_dim, batch=batch, lib=lib)
        assert np.all(np.abs(y - ref) <= 1e-12 * mag + 1e-300), (n_rows, k_dim)
        assert np.allclose(s, mag, rtol=1e-12, atol=0)


# ------------------------------------------------------------------ invariants

def pin_invariants(lib):
    n_rows, k_dim, seed = 12, 512, 7
    w = synth.q4_matrix(n_rows, k_dim, seed, 3)
    x = synth.activations(2, k_dim, seed)
    y, s = ora.gemv(w, x, n_rows, k_dim, batch=2, lib=lib)
    # linearity in x for a power-of-two factor: exact
    x2 = _f16(x.view(np.float16).astype(np.float64) * 2.0)
    y2, _ = ora.gemv(w, x2, n_rows, k_dim, batch=2, lib=lib)
    assert np.array_equal(y2, 2.0 * y)
    # row permutation of W permutes y
    perm = np.random.default_rng(0).permutation(n_rows)
    wp = w.reshape(n_rows, -1)[perm].reshape(-1)
    yp, _ = ora.gemv(wp, x, n_rows, k_dim, batch=2, lib=lib)
    assert np.array_equal(yp, y[:, perm])
    # flipping the sign bit of every scale negates y
    wn = w.reshape(-1, 18).copy()
    wn[:, 1] ^= 0x80
    yn, _ = ora.gemv(wn.reshape(-1), x, n_rows, k_dim, batch=2, lib=lib)
    assert np.array_equal(yn, -y)
    # a batch is its rows stacked
    for b in range(2):
        yb, sb = ora.gemv(w, x[b], n_rows, k_dim, batch=1, lib=lib)
        assert np.array_equal(yb[0], y[b]) and np.array_equal(sb[0], s[b])
    # selected rows agree with the full product
    rows = np.array([11, 0, 5])
    yr, sr = ora.gemv_rows(w, x, n_rows, k_dim, rows, batch=2, lib=lib)
    assert np.array_equal(yr, y[:, rows]) and np.array_equal(sr, s[:, rows])


# ------------------------------------------------------------------ glue

def pin_glue(lib):
    # RMSNorm of a constant vector c: c / sqrt(c^2 + eps)
    c = 0.5
    h = _f16(np.full(64, c))
    x = ora.rmsnorm(h, 1, 64, 1e-5, lib=lib)
    assert np.all(x == _f16(c / np.sqrt(c * c + 1e-5)))
    # RMSNorm is invariant to a power-of-two rescale of h (up to the eps term)
    rng = np.random.default_rng(6)
    hv = rng.standard_normal((2, 256))
    a = ora.rmsnorm(_f16(hv), 2, 256, 0.0, lib=lib)
    b = ora.rmsnorm(_f16(hv * 4), 2, 256, 0.0, lib=lib)
    assert np.array_equal(a, b)
    # unit RMS output: mean(x^2) == 1 within binary16 rounding
    xv = a.view(np.float16).astype(np.float64)
    assert np.all(np.abs((xv ** 2).mean(axis=1) - 1) < 2e-3)
    # SiLU gate: silu(0) = 0; silu(g) -> g for large g; silu(-g) = silu(g) - g
    g = np.array([0.0, 30.0, -30.0, 1.0, -1.0])
    u = np.array([5.0, 1.0, 1.0, 1.0, 1.0])
    act = ora.silu_mul(g, u, lib=lib).view(np.float16).astype(np.float64)
    assert act[0] == 0 and act[1] == 30.0 and abs(act[2]) < 1e-9
    assert abs(act[3] - 0.7310585786) < 1e-3 and abs(act[4] + 0.2689414214) < 1e-3
    # residual sum of small integers is exact
    hr = _f16(np.arange(-4, 4, dtype=np.float64))
    r = ora.add(hr, np.full(8, 2.5), lib=lib)
    assert np.array_equal(r, np.arange(-4, 4, dtype=np.float64) + 2.5)
    # RMSNorm of a double vector agrees with the binary16 one on binary16 inputs,
    # and is invariant to a power-of-two scale
    t = hv[0].astype(np.float16).astype(np.float64)
    assert np.array_equal(ora.rmsnorm_d(t, 1, 256, 1e-5, lib=lib), ora.rmsnorm(_f16(t), 1, 256, 1e-5, lib=lib))
    assert np.array_equal(ora.rmsnorm_d(t * 8, 1, 256, 0.0, lib=lib), ora.rmsnorm_d(t, 1, 256, 0.0, lib=lib))
    # a layer of all-8 codes has every projection zero: t1 = z, z1 = norm(z),
    # act = 0, t2 = z1, so the output is norm(norm(z))
    hid, qd, kvd, ffn, hd = 64, 64, 32, 128, 16
    zero_w = []
    for (n, k) in synth.layer_dims(hid, qd, kvd, ffn):
        blk = np.concatenate([[0x00, 0x3C], [0x88] * 16]).astype(np.uint8)
        zero_w.append(np.tile(blk, n * k // 32))
    z = ora.rmsnorm(_f16(rng.standard_normal((1, hid))), 1, hid, 1e-5, lib=lib)
    zo, t2 = ora.layer(zero_w, z, 1, hid, qd, kvd, ffn, hd, lib=lib)
    z1 = ora.rmsnorm(z, 1, hid, 1e-5, lib=lib)
    assert np.array_equal(t2, z1.view(np.float16).astype(np.float64))
    assert np.array_equal(zo, ora.rmsnorm(z1, 1, hid, 1e-5, lib=lib))
    # with random weights the layer output is still unit-RMS (it is a
    # normalised residual sum) and t2 is not
    rnd_w = [synth.q4_matrix(n, k, 4, p) for p, (n, k) in enumerate(synth.layer_dims(hid, qd, kvd, ffn))]
    zo, t2 = ora.layer(rnd_w, z, 1, hid, qd, kvd, ffn, hd, lib=lib)
    zv = zo.view(np.float16).astype(np.float64)
    assert abs((zv ** 2).mean() - 1) < 2e-3 and abs((t2 ** 2).mean() - 1) > 0.1
    # context-1 attention: query head qh reads value head qh // group
    q_dim, kv_dim, hd = 8 * 4, 2 * 4, 4          # 8 query heads, 2 value heads
    v = np.arange(kv_dim, dtype=np.float64)       # value head j holds 4j..4j+3
    att = ora.attn_ctx1(v, 1, q_dim, kv_dim, hd, lib=lib).view(np.float16).astype(np.float64)
    expect = np.concatenate([v[(qh // 4) * hd:(qh // 4) * hd + hd] for qh in range(8)])
    assert np.array_equal(att.ravel(), expect)



def _q4_matrix_of(n: int, k: int, row_fn) -> np.ndarray:
    """A hand-built row-major Q4_0 matrix: row_fn(row) gives (d_bits, codes[k])."""
    rows = []
    for r in range(n):
        d_bits, codes = row_fn(r)
        codes = np.asarray(codes, dtype=np.int64)
        for b in range(k // 32):
            c = codes[32 * b:32 * b + 32]
            rows.append(_block(d_bits, (c[:16] | (c[16:] << 4)).astype(np.uint8)))
    return np.concatenate(rows)


def _codes(k: int, col0: int | None = None, q0: int = 8, fill: int = 8) -> np.ndarray:
    c = np.full(k, fill, dtype=np.int64)
    if col0 is not None:
        c[col0] = q0
    return c


def pin_layer_wiring(lib):
    """Which tensor feeds which step of ora_layer, by closed forms.

    Hand-built weights make every intermediate a known small number (z = 1
    everywhere, d a power of two), so the layer output follows by hand:
      A. v = 2 (Wv rows: one code 10 at column 0, d = 1), o = (a[0], 0, ...)
         (Wo row 0: one code 9 at column 0), Wq and Wk random, Wdown zero:
         the context-1 attention copies v, so t1 = z + o = (3, 1, ..., 1),
         z1 = f16(t1 r) with r = 1/sqrt((9 + 63)/64 + eps), and t2 = z1.
         Reading k or q for the attention, feeding z to Wo, or taking z as
         the feed-forward residual base all change t2.
      B. Wv zero (so t1 = z and z1 = f16(1/sqrt(1 + eps)) = 1), gate rows all
         code 3 with d = 1/16 (g = -5/16 * 64 = -20), up rows all code 9 with
         d = 1/64 (u = 1), Wdown row 0 one code 9 at column 0 (dn = (act[0], 0,
         ...)): act[0] = f16(silu(-20) * 1) = -2^-24 (silu(-20) = -4.12e-8, the
         nearest binary16 is the negative smallest subnormal), so
         t2 = (1 - 2^-24, 1, ..., 1) and every output is binary16 1.0.  With
         gate and up swapped act[0] = f16(silu(1) * -20) = -14.6; with Wdown
         fed z1 instead of act, t2[0] = 2.
    """
    hid, qd, kvd, ffn, hd = 64, 64, 32, 128, 16
    eps = 1e-5
    one = int(_f16(1.0))
    zero = lambda n, k: _q4_matrix_of(n, k, lambda r: (one, _codes(k)))
    rnd = lambda n, k, p: synth.q4_matrix(n, k, 4, p)
    z = np.full((1, hid), one, dtype=np.uint16)
    # A
    wv = _q4_matrix_of(kvd, hid, lambda r: (one, _codes(hid, 0, 10)))
    wo = _q4_matrix_of(hid, qd, lambda r: (one, _codes(qd, 0, 9) if r == 0 else _codes(qd)))
    wts = [rnd(qd, hid, 0), rnd(kvd, hid, 1), wv, wo, rnd(ffn, hid, 4), rnd(ffn, hid, 5), zero(hid, ffn)]
    zo, t2 = ora.layer(wts, z, 1, hid, qd, kvd, ffn, hd, eps, lib=lib)
    r = 1.0 / np.sqrt((9.0 + 63.0) / 64.0 + eps)
    expect = np.concatenate([[3.0 * r], np.full(hid - 1, r)]).astype(np.float16).astype(np.float64)
    assert np.array_equal(t2[0], expect), "A: t2 = f16(norm(z + Wo gather(v)))"
    # B
    d16, d64 = int(_f16(1 / 16)), int(_f16(1 / 64))
    wg = _q4_matrix_of(ffn, hid, lambda r: (d16, _codes(hid, fill=3)))
    wu = _q4_matrix_of(ffn, hid, lambda r: (d64, _codes(hid, fill=9)))
    wd = _q4_matrix_of(hid, ffn, lambda r: (one, _codes(ffn, 0, 9) if r == 0 else _codes(ffn)))
    wts = [rnd(qd, hid, 0), rnd(kvd, hid, 1), zero(kvd, hid), rnd(hid, qd, 3), wg, wu, wd]
    zo, t2 = ora.layer(wts, z, 1, hid, qd, kvd, ffn, hd, eps, lib=lib)
    assert t2[0, 0] == 1.0 - 2.0 ** -24, f"B: t2[0] = 1 + f16(silu(g) u), got {t2[0, 0]!r}"
    assert np.all(t2[0, 1:] == 1.0), "B: rows of Wdown with no code read nothing"
    assert np.all(zo == one), "B: output f16(norm(t2)) is 1.0 everywhere"



def pin_layer_kv(lib):
    """The KV-cache layer: at position 0 the softmax over one key is 1 and the
    layer is the context-1 layer; the cache row of the token is f16(k), f16(v);
    with Wq (or Wk) all code 8 every score is 0, the softmax is uniform and the
    attention output is the mean of the cached values, which hand-built values
    make a closed form: cached value rows all 1 and the token's own v = 4
    (Wv rows one code 12 at column 0, d = 1, z = 1) give a = f16((pos + 4) / (pos + 1))."""
    hid, qd, kvd, ffn, hd = 64, 64, 32, 128, 16
    eps = 1e-5
    one = int(_f16(1.0))
    rnd = lambda n, k, p: synth.q4_matrix(n, k, 4, p)
    zero = lambda n, k: _q4_matrix_of(n, k, lambda r: (one, _codes(k)))
    rng = np.random.default_rng(12)
    z = ora.rmsnorm(_f16(rng.standard_normal((1, hid))), 1, hid, eps, lib=lib)
    wts = [rnd(n, k, p) for p, (n, k) in enumerate(synth.layer_dims(hid, qd, kvd, ffn))]
    cap = 8
    kc = np.zeros((cap, kvd), np.uint16)
    vc = np.zeros((cap, kvd), np.uint16)
    zo, t2 = ora.layer_kv(wts, z, kc, vc, 0, hid, qd, kvd, ffn, hd, eps, lib=lib)
    zr, t2r = ora.layer(wts, z, 1, hid, qd, kvd, ffn, hd, eps, lib=lib)
    assert np.array_equal(zo, zr.reshape(-1)) and np.array_equal(t2, t2r.reshape(-1)), "pos 0 is the context-1 layer"
    kref = ora.double_to_half(ora.gemv(wts[1], z, kvd, hid, lib=lib)[0][0], lib=lib)
    vref = ora.double_to_half(ora.gemv(wts[2], z, kvd, hid, lib=lib)[0][0], lib=lib)
    assert np.array_equal(kc[0], kref) and np.array_equal(vc[0], vref), "cache row 0 = f16(k), f16(v)"
    assert not kc[1:].any() and not vc[1:].any(), "only the token's row is written"
    # uniform scores: Wq all code 8; cached values 1, own value 4 -> attention (pos + 4) / (pos + 1);
    # Wo row 0 one code 9 at column 0 -> o = (a[0], 0, ...); Wdown zero -> t2 = z1 = f16(norm(z + o))
    zc = np.full((1, hid), one, np.uint16)
    wv = _q4_matrix_of(kvd, hid, lambda r: (one, _codes(hid, 0, 12)))
    wo = _q4_matrix_of(hid, qd, lambda r: (one, _codes(qd, 0, 9) if r == 0 else _codes(qd)))
    w2 = [zero(qd, hid), rnd(kvd, hid, 1), wv, wo, rnd(ffn, hid, 4), rnd(ffn, hid, 5), zero(hid, ffn)]
    for pos in (1, 3, 6):
        kc = _f16(rng.standard_normal((cap, kvd)))
        vc = np.full((cap, kvd), one, np.uint16)
        zo, t2 = ora.layer_kv(w2, zc, kc, vc, pos, hid, qd, kvd, ffn, hd, eps, lib=lib)
        a0 = float(np.float16((pos + 4.0) / (pos + 1.0)))
        t1 = np.concatenate([[1.0 + a0], np.ones(hid - 1)])
        r = 1.0 / np.sqrt((t1 ** 2).mean() + eps)
        expect = (t1 * r).astype(np.float16).astype(np.float64)
        assert np.array_equal(t2, expect), f"uniform scores at pos {pos}"
        assert np.all(vc[pos] == int(_f16(4.0))) and np.all(vc[pos + 1:] == one), "v row pos = f16(v) only"


def pin_attn_decode(lib):
    """Decode attention over a KV cache: closed forms of the softmax."""
    rng = np.random.default_rng(11)
    n_q, n_kv, hd = 8, 2, 16
    group = n_q // n_kv
    kv = n_kv * hd
    # one position: the softmax over one key is 1, so head h reads value head h // group
    # (also the context-1 stand-in of the layer, computed by another oracle function)
    v1 = _f16(rng.normal(size=(1, kv)))
    q = rng.normal(size=n_q * hd)
    o, sabs = ora.attn_decode(q, _f16(rng.normal(size=(1, kv))), v1, 1, n_q, n_kv, hd, lib=lib)
    vd = v1.view(np.float16).astype(np.float64).reshape(n_kv, hd)
    expect = np.concatenate([vd[h // group] for h in range(n_q)])
    assert np.array_equal(o, expect), "ctx 1: value head of the group"
    assert np.array_equal(ora.double_to_half(o, lib=lib),
                          ora.attn_ctx1(vd.reshape(1, -1), 1, n_q * hd, kv, hd, lib=lib).reshape(-1))
    # equal keys: uniform weights, o = mean of the values, sabs = mean of |values|
    ctx = 7
    krow = _f16(rng.normal(size=(1, kv)))
    kc = np.repeat(krow, ctx, axis=0)
    vc = _f16(rng.normal(size=(ctx, kv)))
    o, sabs = ora.attn_decode(q, kc, vc, ctx, n_q, n_kv, hd, lib=lib)
    vv = vc.view(np.float16).astype(np.float64).reshape(ctx, n_kv, hd)
    mean = np.concatenate([vv[:, h // group].mean(axis=0) for h in range(n_q)])
    mabs = np.concatenate([np.abs(vv[:, h // group]).mean(axis=0) for h in range(n_q)])
    assert np.allclose(o, mean, rtol=0, atol=1e-12), "equal keys: mean of values"
    assert np.allclose(sabs, mabs, rtol=0, atol=1e-12), "equal keys: mean of |values|"
    # two score levels: key 0 = e0, the others 0; q = a e0 per head:
    # p0 = 1 / (1 + (ctx - 1) exp(-a / sqrt(hd)))
    kc = np.zeros((ctx, kv), dtype=np.uint16)
    kc[0, 0::hd] = _f16(1.0)            # component 0 of every value head's key at position 0
    a = 3.0
    q = np.zeros(n_q * hd)
    q[0::hd] = a
    o, _ = ora.attn_decode(q, kc, vc, ctx, n_q, n_kv, hd, lib=lib)
    p0 = 1.0 / (1.0 + (ctx - 1) * np.exp(-a / np.sqrt(hd)))
    expect = np.concatenate([p0 * vv[0, h // group] + (1 - p0) * vv[1:, h // group].mean(axis=0)
                             for h in range(n_q)])
    assert np.allclose(o, expect, rtol=0, atol=1e-12), "two score levels"
    # a score of 1000 (exp overflows without the max shift): o = the value at that position
    q[0::hd] = 1000.0 * np.sqrt(hd)
    o, _ = ora.attn_decode(q, kc, vc, ctx, n_q, n_kv, hd, lib=lib)
    assert np.all(np.isfinite(o))
    assert np.allclose(o, np.concatenate([vv[0, h // group] for h in range(n_q)]), rtol=0, atol=1e-12)
    # permuting the positions (keys and values together) leaves the result unchanged
    kc = _f16(rng.normal(size=(ctx, kv)))
    q = rng.normal(size=n_q * hd)
    perm = rng.permutation(ctx)
    o1, s1 = ora.attn_decode(q, kc, vc, ctx, n_q, n_kv, hd, lib=lib)
    o2, s2 = ora.attn_decode(q, kc[perm], vc[perm], ctx, n_q, n_kv, hd, lib=lib)
    assert np.allclose(o1, o2, rtol=0, atol=1e-12) and np.allclose(s1, s2, rtol=0, atol=1e-12)
    assert np.all(s1 >= np.abs(o1) - 1e-15)


ALL_PINS = [pin_attn_decode, pin_half_decode_exhaustive, pin_half_encode, pin_golden_blocks, pin_distinct_positions,
            pin_block_indexing, pin_golden_gemv, pin_all_eight_is_zero, pin_single_nonzero,
            pin_constant_codes, pin_brute_force, pin_invariants, pin_glue, pin_layer_wiring, pin_layer_kv]
