"""q4_gemv and q4_dequant_debug on the GPU against the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle as ora
import weight_streaming_q4_gb300 as q4
from weight_streaming_q4_gb300 import build, synth
from gpu_util import assert_within_tol, dev_u8, dev_u16, host_f32
from pins import golden_blocks

pytestmark = pytest.mark.gpu

KERNELS = {"stream": q4.Q4_KERNEL_STREAM, "simple": q4.Q4_KERNEL_SIMPLE, "mma": q4.Q4_KERNEL_MMA,
           "tc": q4.Q4_KERNEL_TC, "oneshot": q4.Q4_KERNEL_ONESHOT}


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    ora.build()


def run(w_np, x_np, n, k, batch, kernel):
    w = dev_u8(w_np)
    x = dev_u16(x_np.reshape(-1))
    y = torch.full((batch * n,), float("nan"), dtype=torch.float32, device="cuda")
    q4.q4_gemv_ex(w, x, y, n, k, batch, kernel)
    torch.cuda.synchronize()
    return host_f32(y).reshape(batch, n)


# ------------------------------------------------------------------ layout, bit for bit

@pytest.mark.parametrize("n,k", [(1, 32), (3, 64), (17, 256), (64, 4096), (5, 14336)])
def test_dequant_bit_exact(n, k):
    w = synth.q4_matrix(n, k, 1, 2)
    out = torch.empty(n * k, dtype=torch.float32, device="cuda")
    q4.q4_dequant_debug(dev_u8(w), out, n, k)
    torch.cuda.synchronize()
    got = out.cpu().numpy().reshape(n, k)
    ref = ora.dequant(w, n, k).astype(np.float32)   # every (q-8)*d is a float: exact
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_dequant_golden_blocks():
    for blk, expect in golden_blocks():
        out = torch.empty(32, dtype=torch.float32, device="cuda")
        q4.q4_dequant_debug(dev_u8(np.concatenate([blk, np.zeros(14, np.uint8)])), out, 1, 32)
        torch.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy().astype(np.float64), expect)


# ------------------------------------------------------------------ closed forms, exact

def _const_matrix(n, k, d, code_byte):
    blk = np.zeros(18, np.uint8)
    blk[0:2] = np.array([d], np.float16).view(np.uint8)
    blk[2:] = code_byte
    return np.tile(blk, n * k // 32)


@pytest.mark.parametrize("kernel", list(KERNELS))
def test_all_eight_is_exactly_zero(kernel):
    n, k = 40, 4096
    w = _const_matrix(n, k, 0.75, 0x88)
    x = synth.activations(1, k, 5)
    y = run(w, x, n, k, 1, KERNELS[kernel])
    assert np.all(y == 0.0)


@pytest.mark.parametrize("kernel", list(KERNELS))
def test_single_nonzero_is_exact(kernel):
    rng = np.random.default_rng(7)
    n, k = 16, 4096
    for _ in range(6):
        w = _const_matrix(n, k, 1.0, 0x88).copy().reshape(-1, 18)
        w[:, 0:2] = np.asarray(rng.uniform(0.001, 0.05, n * k // 32), np.float16).view(np.uint8).reshape(-1, 2)
        row, col = int(rng.integers(n)), int(rng.integers(k))
        code = int(rng.choice([c for c in range(16) if c != 8]))
        b = row * (k // 32) + col // 32
        j = col % 32
        byte = w[b, 2 + (j % 16)]
        w[b, 2 + (j % 16)] = (byte & 0xF0) | code if j < 16 else (byte & 0x0F) | (code << 4)
        x = synth.activations(1, k, int(rng.integers(1000)))
        y = run(w.reshape(-1), x, n, k, 1, KERNELS[kernel])
        d = float(w[b, 0:2].view(np.float16)[0])
        xv = float(x.view(np.float16)[0, col])
        expect = np.zeros(n, np.float32)
        expect[row] = np.float32((code - 8) * d * xv)   # the exact product rounded once to fp32
        assert np.array_equal(y[0].astype(np.float32), expect)


# ------------------------------------------------------------------ parity with the oracle

STREAM_SHAPES = [(1, 256), (7, 256), (33, 512), (100, 1024), (129, 2048), (300, 4096), (61, 14336), (17, 28672),
                 (1000, 8192), (9, 26624), (40, 6144)]


@pytest.mark.parametrize("n,k", STREAM_SHAPES)
def test_stream_kernel_parity(n, k):
    w = synth.q4_matrix(n, k, 3, synth.GEMV_TID)
    x = synth.activations(1, k, 4)
    y = run(w, x, n, k, 1, q4.Q4_KERNEL_STREAM)
    y_ref, s_ref = ora.gemv(w, x, n, k, threads=8)
    assert_within_tol(y, y_ref, s_ref, f"stream {n}x{k}")


# widths of one chunk (up to 2048 columns, unpadded rows) and of whole 64-block
# chunks (padded rows, the last chunk's copy box running past the row end);
# row counts that leave a ragged last tile
TC_SHAPES = [(1, 256), (16, 256), (17, 512), (100, 2048), (129, 4096), (300, 4096), (61, 14336), (33, 28672),
             (1000, 8192), (64, 1024), (5, 30720), (31, 6144), (4096, 4096)]


@pytest.mark.parametrize("n,k", TC_SHAPES)
def test_tc_engine_parity(n, k):
    w = synth.q4_matrix(n, k, 18, synth.GEMV_TID)
    x = synth.activations(1, k, 19)
    y = run(w, x, n, k, 1, q4.Q4_KERNEL_TC)
    y_ref, s_ref = ora.gemv(w, x, n, k, threads=8)
    assert_within_tol(y, y_ref, s_ref, f"tc {n}x{k}")
    assert q4.q4_device_status() == 0


# one-shot kernel: widths from 512 to the shared-memory limit (11 k + 256 <=
# 231424 bytes: k <= 20992), row counts with a ragged last 16-row tile
ONESHOT_SHAPES = [(1, 512), (15, 512), (16, 1024), (17, 4096), (300, 4096), (61, 14336), (33, 20992),
                  (4096, 4096), (1000, 8192), (100, 2560)]


@pytest.mark.parametrize("n,k", ONESHOT_SHAPES)
def test_oneshot_parity(n, k):
    w = synth.q4_matrix(n, k, 20, synth.GEMV_TID)
    x = synth.activations(1, k, 21)
    y = run(w, x, n, k, 1, q4.Q4_KERNEL_ONESHOT)
    y_ref, s_ref = ora.gemv(w, x, n, k, threads=8)
    assert_within_tol(y, y_ref, s_ref, f"oneshot {n}x{k}")
    assert q4.q4_device_status() == 0


CHAIN = q4.Q4_KERNEL_ONESHOT | q4.Q4_GEMV_CHAIN   # chained calls: each may start before the one ahead ends


def test_oneshot_rejects_and_orders_back_to_back_launches():
    w = dev_u8(synth.q4_matrix(64, 4096, 22, synth.GEMV_TID))
    x = dev_u16(synth.activations(1, 21504, 23).reshape(-1))
    y = torch.empty(64, dtype=torch.float32, device="cuda")
    for k, batch in ((256, 1), (4096 + 256, 1), (21504, 1), (4096, 2)):   # width, shared memory, batch
        with pytest.raises(q4.Q4Error):
            q4.q4_gemv_ex(w, x, y, 4, k, batch, q4.Q4_KERNEL_ONESHOT)
    # launches that overlap their setup with the previous one still write y in
    # stream order: alternate two matrices into one y, eagerly and from a graph
    n, k = 1000, 4096
    wa, wb = (synth.q4_matrix(n, k, s, synth.GEMV_TID) for s in (24, 25))
    xs = synth.activations(1, k, 26)
    da, db, dx = dev_u8(wa), dev_u8(wb), dev_u16(xs.reshape(-1))
    y = torch.empty(n, dtype=torch.float32, device="cuda")
    ya, yb = run(wa, xs, n, k, 1, q4.Q4_KERNEL_ONESHOT), run(wb, xs, n, k, 1, q4.Q4_KERNEL_ONESHOT)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for i in range(41):
            q4.q4_gemv_ex(da if i % 2 == 0 else db, dx, y, n, k, 1, CHAIN, stream=s)
        s.synchronize()
        assert np.array_equal(host_f32(y), ya[0])
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for i in range(40):
                q4.q4_gemv_ex(da if i % 2 == 0 else db, dx, y, n, k, 1, CHAIN, stream=s)
        g.replay()
        s.synchronize()
    assert np.array_equal(host_f32(y), yb[0])
    assert q4.q4_device_status() == 0


def test_oneshot_input_from_the_previous_output():
    """x of a product is the memory of the previous one-shot product's y (its
    fp32 bits read as binary16): the launcher must not start the second one
    early, so it sees the whole first output."""
    n1, k1, n2, k2 = 2048, 4096, 512, 4096          # y1: 2048 fp32 = 4096 binary16
    w1 = synth.q4_matrix(n1, k1, 27, synth.GEMV_TID)
    w2 = synth.q4_matrix(n2, k2, 28, synth.GEMV_TID)
    d1, d2 = dev_u8(w1), dev_u8(w2)
    x1 = dev_u16(synth.activations(1, k1, 29).reshape(-1))
    buf = torch.empty(n1, dtype=torch.float32, device="cuda")
    y2 = torch.empty(n2, dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(3):
            buf.fill_(0.0)
            q4.q4_gemv_ex(d1, x1, buf, n1, k1, 1, CHAIN, stream=s)
            q4.q4_gemv_ex(d2, buf, y2, n2, k2, 1, CHAIN, stream=s)
        s.synchronize()
    x2 = buf.detach().cpu().view(torch.int16).numpy().view(np.uint16).copy()
    ref = run(w2, x2, n2, k2, 1, q4.Q4_KERNEL_ONESHOT)
    assert np.array_equal(host_f32(y2), ref[0], equal_nan=True)


def test_chained_product_after_another_kernel_product():
    """A chained one-shot product whose x is the output of the product before
    it, computed by the batched tensor-core kernel: that launch ends the
    stream's list of early starts, so the chained call waits for it."""
    n1, k1, n2, k2 = 2048, 4096, 512, 4096          # y1: 2048 fp32 = 4096 binary16
    w0 = synth.q4_matrix(n1, k1, 33, synth.GEMV_TID)
    w1 = synth.q4_matrix(n1, k1, 34, synth.GEMV_TID)
    w2 = synth.q4_matrix(n2, k2, 35, synth.GEMV_TID)
    d0, d1, d2 = dev_u8(w0), dev_u8(w1), dev_u8(w2)
    x1 = dev_u16(synth.activations(1, k1, 36).reshape(-1))
    y0 = torch.empty(n1, dtype=torch.float32, device="cuda")
    buf = torch.empty(n1, dtype=torch.float32, device="cuda")
    y2 = torch.empty(n2, dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(3):
            buf.fill_(0.0)
            q4.q4_gemv_ex(d0, x1, y0, n1, k1, 1, CHAIN, stream=s)            # the stream is on the list
            q4.q4_gemv_ex(d1, x1, buf, n1, k1, 1, q4.Q4_KERNEL_MMA, stream=s)
            q4.q4_gemv_ex(d2, buf, y2, n2, k2, 1, CHAIN, stream=s)
        s.synchronize()
    x2 = buf.detach().cpu().view(torch.int16).numpy().view(np.uint16).copy()
    ref = run(w2, x2, n2, k2, 1, q4.Q4_KERNEL_ONESHOT)
    assert np.array_equal(host_f32(y2), ref[0], equal_nan=True)
    assert q4.q4_device_status() == 0


def test_oneshot_long_chain_then_a_dependent_product():
    """80 independent one-shot products into distinct slices of one buffer
    (more than the launcher's list of early-started products holds, so the
    list is ended and restarted on the way), then a product whose x is the
    memory of eight late slices: it must wait and see those slices whole."""
    n, k, count, first = 256, 4096, 80, 66           # x of the last product: slices 66..73
    w1 = synth.q4_matrix(n, k, 30, synth.GEMV_TID)
    w2 = synth.q4_matrix(n, k, 32, synth.GEMV_TID)
    xs = synth.activations(1, k, 31)
    d1, d2, dx = dev_u8(w1), dev_u8(w2), dev_u16(xs.reshape(-1))
    ys = torch.empty(count * n, dtype=torch.float32, device="cuda")
    y2 = torch.empty(n, dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(3):
            ys.fill_(0.0)
            for i in range(count):
                q4.q4_gemv_ex(d1, dx, ys[i * n:(i + 1) * n], n, k, 1, CHAIN, stream=s)
            q4.q4_gemv_ex(d2, ys[first * n:(first + 8) * n], y2, n, k, 1, CHAIN, stream=s)
        s.synchronize()
    y1 = run(w1, xs, n, k, 1, q4.Q4_KERNEL_ONESHOT)[0]
    assert np.array_equal(host_f32(ys).reshape(count, n), np.broadcast_to(y1, (count, n)))
    x2 = ys[first * n:(first + 8) * n].detach().cpu().view(torch.int16).numpy().view(np.uint16).copy()
    ref = run(w2, x2, n, k, 1, q4.Q4_KERNEL_ONESHOT)
    assert np.array_equal(host_f32(y2), ref[0], equal_nan=True)
    assert q4.q4_device_status() == 0


def test_tc_engine_rejects_unsupported_widths():
    x = torch.zeros(32768, dtype=torch.int16, device="cuda")
    y = torch.zeros(64, dtype=torch.float32, device="cuda")
    w = torch.zeros(q4.q4_matrix_bytes(4, 32768), dtype=torch.uint8, device="cuda")
    for k in (96, 288, 2304, 3072, 32768):
        with pytest.raises(q4.Q4Error) as e:
            q4.q4_gemv_ex(w, x, y, 4, k, 1, q4.Q4_KERNEL_TC)
        assert e.value.status == q4.Q4_ERR_ARG
    with pytest.raises(q4.Q4Error):
        q4.q4_gemv_ex(w, x, y, 4, 4096, 2, q4.Q4_KERNEL_TC)


MMA_SHAPES = [(1, 256, 1), (16, 256, 2), (17, 512, 3), (100, 2048, 8), (129, 4096, 9), (300, 4096, 16),
              (61, 14336, 4), (33, 28672, 1), (1000, 8192, 7), (64, 2304, 12)]


@pytest.mark.parametrize("n,k,batch", MMA_SHAPES)
def test_mma_kernel_parity(n, k, batch):
    w = synth.q4_matrix(n, k, 12, synth.GEMV_TID)
    x = synth.activations(batch, k, 13)
    y = run(w, x, n, k, batch, q4.Q4_KERNEL_MMA)
    y_ref, s_ref = ora.gemv(w, x, n, k, batch=batch, threads=8)
    assert_within_tol(y, y_ref, s_ref, f"mma {n}x{k}x{batch}")
    assert q4.q4_device_status() == 0


@pytest.mark.parametrize("batch", [2, 8, 16])
def test_mma_batch_rows_are_independent(batch):
    # a batch gives, row for row, what each row gives alone (same kernel)
    n, k = 96, 4096
    w = synth.q4_matrix(n, k, 14, synth.GEMV_TID)
    x = synth.activations(batch, k, 15)
    y = run(w, x, n, k, batch, q4.Q4_KERNEL_MMA)
    for b in (0, batch - 1):
        yb = run(w, x[b:b + 1], n, k, 1, q4.Q4_KERNEL_MMA)
        assert np.array_equal(y[b], yb[0])


def test_auto_picks_mma_for_batches():
    n, k, batch = 64, 4096, 4
    w = synth.q4_matrix(n, k, 16, synth.GEMV_TID)
    x = synth.activations(batch, k, 17)
    assert np.array_equal(run(w, x, n, k, batch, q4.Q4_KERNEL_AUTO), run(w, x, n, k, batch, q4.Q4_KERNEL_MMA))


@pytest.mark.parametrize("n,k,batch", [(1, 32, 1), (9, 96, 2), (40, 800, 5), (65, 4096, 16), (33, 2048, 3)])
def test_simple_kernel_parity(n, k, batch):
    w = synth.q4_matrix(n, k, 8, 9)
    x = synth.activations(batch, k, 10)
    y = run(w, x, n, k, batch, q4.Q4_KERNEL_SIMPLE)
    y_ref, s_ref = ora.gemv(w, x, n, k, batch=batch)
    assert_within_tol(y, y_ref, s_ref, f"simple {n}x{k}x{batch}")


def test_full_size_gemv_all_rows():
    # the single-product workload: N = K = 4096, batch 1, every row against the oracle
    n = k = 4096
    w = synth.q4_matrix(n, k, 0, synth.GEMV_TID)
    x = synth.activations(1, k, 0)
    y = run(w, x, n, k, 1, q4.Q4_KERNEL_AUTO)
    y_ref, s_ref = ora.gemv(w, x, n, k, threads=8)
    assert_within_tol(y, y_ref, s_ref, "gemv 4096x4096")
    assert q4.q4_device_status() == 0


def test_stream_kernel_width_limit():
    # two rows of 30720 columns do not fit a stage: the streaming kernel refuses, auto falls back
    n, k = 4, 30720
    w = torch.zeros(q4.q4_matrix_bytes(n, k), dtype=torch.uint8, device="cuda")
    x = torch.zeros(k, dtype=torch.int16, device="cuda")
    y = torch.zeros(n, dtype=torch.float32, device="cuda")
    with pytest.raises(q4.Q4Error):
        q4.q4_gemv_ex(w, x, y, n, k, 1, q4.Q4_KERNEL_STREAM)
    q4.q4_gemv(w, x, y, n, k, 1)
    torch.cuda.synchronize()
    assert not y.any()


def test_deterministic_and_auto_choice():
    n, k = 512, 4096
    w = synth.q4_matrix(n, k, 1, synth.GEMV_TID)
    x = synth.activations(1, k, 1)
    a = run(w, x, n, k, 1, q4.Q4_KERNEL_AUTO)
    b = run(w, x, n, k, 1, q4.Q4_KERNEL_ONESHOT)
    c = run(w, x, n, k, 1, q4.Q4_KERNEL_ONESHOT)
    assert np.array_equal(a, b) and np.array_equal(b, c)
    t1, t2 = run(w, x, n, k, 1, q4.Q4_KERNEL_TC), run(w, x, n, k, 1, q4.Q4_KERNEL_TC)
    assert np.array_equal(t1, t2)
    # above 64 MB of weights auto takes the persistent engine
    nb, kb = 65536, 2048
    wd = torch.empty(q4.q4_matrix_bytes(nb, kb), dtype=torch.uint8, device="cuda")
    synth.device_fill_q4(wd.data_ptr(), nb * kb // 32, seed=1, tid=synth.GEMV_TID)
    xd = dev_u16(synth.activations(1, kb, 1).reshape(-1))
    ya, yt = (torch.empty(nb, dtype=torch.float32, device="cuda") for _ in range(2))
    q4.q4_gemv_ex(wd, xd, ya, nb, kb, 1, q4.Q4_KERNEL_AUTO)
    q4.q4_gemv_ex(wd, xd, yt, nb, kb, 1, q4.Q4_KERNEL_TC)
    torch.cuda.synchronize()
    assert torch.equal(ya, yt)
    d = run(w, x, n, k, 1, q4.Q4_KERNEL_STREAM)
    e = run(w, x, n, k, 1, q4.Q4_KERNEL_STREAM)
    assert np.array_equal(d, e)
    # widths neither persistent engine takes go to the plain kernel
    n, k = 64, 2304
    w = synth.q4_matrix(n, k, 1, synth.GEMV_TID)
    x = synth.activations(1, k, 1)
    assert np.array_equal(run(w, x, n, k, 1, q4.Q4_KERNEL_AUTO), run(w, x, n, k, 1, q4.Q4_KERNEL_SIMPLE))
    # above the persistent engine's widths auto takes the plain CUDA-core kernel at batch 1
    n, k = 8, 34816
    w = synth.q4_matrix(n, k, 1, synth.GEMV_TID)
    x = synth.activations(1, k, 1)
    assert np.array_equal(run(w, x, n, k, 1, q4.Q4_KERNEL_AUTO), run(w, x, n, k, 1, q4.Q4_KERNEL_SIMPLE))


def test_large_rows_sampled():
    # gate/up-shaped (14336 x 4096) and down-shaped (4096 x 14336) matrices on sampled rows
    for (n, k) in ((14336, 4096), (4096, 14336), (8192, 28672)):
        wd = torch.empty(q4.q4_matrix_bytes(n, k), dtype=torch.uint8, device="cuda")
        synth.device_fill_q4(wd.data_ptr(), n * k // 32, seed=2, tid=synth.GEMV_TID)
        x = synth.activations(1, k, 2)
        y = torch.empty(n, dtype=torch.float32, device="cuda")
        q4.q4_gemv(wd, dev_u16(x.reshape(-1)), y, n, k, 1)
        torch.cuda.synchronize()
        rows = np.sort(np.random.default_rng(n).choice(n, 256, replace=False))
        wr = synth.q4_rows(rows, k, 2, synth.GEMV_TID)
        y_ref, s_ref = ora.gemv(wr.reshape(-1), x, len(rows), k)
        assert_within_tol(host_f32(y)[rows], y_ref[0], s_ref[0], f"{n}x{k} sampled")
