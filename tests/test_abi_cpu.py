"""The C-ABI library on a machine without a GPU: it loads, exports every
function include/q4.h declares, and its host-side checks and layout
arithmetic behave as documented (no kernel is launched here)."""
import ctypes

import numpy as np
import pytest

import weight_streaming_q4_gb300 as q4
from weight_streaming_q4_gb300 import build, synth


@pytest.fixture(scope="module")
def lib():
    build.build()
    return q4.lib()


def test_exports_every_declared_symbol(lib):
    names = q4.header_functions()
    assert len(names) >= 19
    for n in names:
        assert hasattr(lib, n), n
    raw = ctypes.CDLL(build.lib_path("libq4.so"))
    for n in names:
        getattr(raw, n)   # raises AttributeError if not exported


def test_synth_library_exports():
    build.build()
    raw = ctypes.CDLL(build.lib_path("libq4synth.so"))
    for n in ("q4s_fill_q4_0", "q4s_fill_normal_f16", "q4s_philox"):
        getattr(raw, n)


def test_status_strings(lib):
    for st in (0, -1, -2, -3, -4, -5, -6):
        assert q4.status_string(st)
    assert q4.q4_version() >= 100


@pytest.mark.parametrize("n,k", [(1, 32), (4096, 4096), (14336, 4096), (4096, 14336), (8192, 28672)])
def test_matrix_bytes(lib, n, k):
    assert q4.q4_matrix_bytes(n, k) == n * k // 32 * 18
    assert q4.q4_matrix_bytes(n, k + 1) == 0


@pytest.mark.parametrize("cfg", [synth.LLAMA_8B, synth.LLAMA_70B,
                                 dict(hidden=256, q_dim=256, kv_dim=128, ffn=1024, head_dim=64)])
def test_layer_offsets_match_generator(lib, cfg):
    shape = q4.LayerShape.of(**cfg)
    offs, total = q4.q4_layer_offsets(shape)
    g_offs, g_total = synth.layer_offsets(cfg["hidden"], cfg["q_dim"], cfg["kv_dim"], cfg["ffn"])
    assert offs == g_offs and total == g_total


def test_layer_bytes_of_configs(lib):
    # one 8B-shaped layer reads 122 683 392 weight bytes, one 70B-shaped layer 481 296 384
    assert q4.q4_layer_offsets(q4.LayerShape.of(**synth.LLAMA_8B))[1] == 122_683_392
    assert q4.q4_layer_offsets(q4.LayerShape.of(**synth.LLAMA_70B))[1] == 481_296_384


def test_workspace_layout(lib):
    shape = q4.LayerShape.of(**synth.LLAMA_8B)
    offs, total = q4.q4_workspace_layout(shape, 32, 1)
    vals = [offs[n] for n in q4.WS_NAMES]
    assert vals == sorted(vals) and all(v % 256 == 0 for v in vals)
    assert offs["qkv"] - offs["program"] >= 32 * 4 * 64
    assert total - offs["t2"] >= 4 * 4096
    with pytest.raises(q4.Q4Error):
        q4.q4_workspace_layout(shape, 0, 1)
    with pytest.raises(q4.Q4Error):
        q4.q4_workspace_layout(shape, 1, 17)


def test_argument_checks_launch_nothing(lib):
    # every one of these is rejected before any CUDA call
    A = 4096  # a 16-byte aligned fake address; never dereferenced
    assert lib.q4_gemv(None, A, A, 4, 64, 1, None) == q4.Q4_ERR_ARG
    assert lib.q4_gemv(A, A, A, 0, 64, 1, None) == q4.Q4_ERR_ARG
    assert lib.q4_gemv(A, A, A, 4, 48, 1, None) == q4.Q4_ERR_ARG       # k not a multiple of 32
    assert lib.q4_gemv(A, A, A, 4, 64, 0, None) == q4.Q4_ERR_ARG
    assert lib.q4_gemv(A, A, A, 4, 64, 17, None) == q4.Q4_ERR_ARG
    assert lib.q4_gemv(A + 2, A, A, 4, 64, 1, None) == q4.Q4_ERR_ALIGN
    assert lib.q4_gemv(A, A + 8, A, 4, 64, 1, None) == q4.Q4_ERR_ALIGN
    assert lib.q4_gemv_ex(A, A, A, 4, 96, 1, q4.Q4_KERNEL_STREAM, None) == q4.Q4_ERR_ARG  # engine needs k % 256
    assert lib.q4_gemv_ex(A, A, A, 4, 256, 2, q4.Q4_KERNEL_STREAM, None) == q4.Q4_ERR_ARG
    assert lib.q4_gemv_ex(A, A, A, 4, 30720, 1, q4.Q4_KERNEL_STREAM, None) == q4.Q4_ERR_ARG   # 2 rows > a stage
    assert lib.q4_gemv_ex(A, A, A, 4, 256, 1, 99, None) == q4.Q4_ERR_ARG
    assert lib.q4_gemv_ex(A, A, A, 4, 256, 1, 99 | q4.Q4_GEMV_CHAIN, None) == q4.Q4_ERR_ARG   # the flag alone
    assert lib.q4_gemv_ex(A, A, A, 4, 96, 1, q4.Q4_KERNEL_TC | q4.Q4_GEMV_CHAIN, None) == q4.Q4_ERR_ARG
    assert lib.q4_gemv_ex(A, A, A, 4, 96, 1, q4.Q4_KERNEL_TC, None) == q4.Q4_ERR_ARG       # tc needs k % 256
    assert lib.q4_gemv_ex(A, A, A, 4, 32768, 1, q4.Q4_KERNEL_TC, None) == q4.Q4_ERR_ARG    # x buffer limit
    assert lib.q4_gemv_ex(A, A, A, 4, 256, 3, q4.Q4_KERNEL_TC, None) == q4.Q4_ERR_ARG      # batch 1 only
    assert lib.q4_dequant_debug(A, None, 4, 64, None) == q4.Q4_ERR_ARG
    assert lib.q4_dequant_debug(A + 1, A, 4, 64, None) == q4.Q4_ERR_ALIGN


def test_decoder_checks(lib):
    shape = q4.LayerShape.of(hidden=256, q_dim=256, kv_dim=128, ffn=1024, head_dim=64)
    h = ctypes.c_void_p()
    ptrs = (ctypes.c_void_p * 2)(4096, 8192)
    ws_bytes = q4.q4_workspace_layout(shape, 2, 1)[1]
    f = lib.q4_decoder_create
    assert f(ctypes.byref(h), ctypes.byref(shape), ptrs, 0, 1, 4096, ws_bytes, 0, None) == q4.Q4_ERR_ARG
    assert f(ctypes.byref(h), ctypes.byref(shape), ptrs, 2, 1, 4096 + 16, ws_bytes, 0, None) == q4.Q4_ERR_ALIGN
    assert f(ctypes.byref(h), ctypes.byref(shape), ptrs, 2, 1, 4096, ws_bytes - 1, 0, None) == q4.Q4_ERR_OOM
    assert f(ctypes.byref(h), ctypes.byref(shape), ptrs, 2, 1, 4096, ws_bytes, 32, None) == q4.Q4_ERR_ARG  # unknown bit
    both = q4.Q4_DEC_TENSOR_CORE | q4.Q4_DEC_CUDA_CORE
    assert f(ctypes.byref(h), ctypes.byref(shape), ptrs, 2, 1, 4096, ws_bytes, both, None) == q4.Q4_ERR_ARG
    bad = q4.LayerShape.of(hidden=256, q_dim=256, kv_dim=96, ffn=1024, head_dim=64)   # kv not whole heads
    assert f(ctypes.byref(h), ctypes.byref(bad), ptrs, 2, 1, 4096, ws_bytes, 0, None) == q4.Q4_ERR_ARG
    odd = q4.LayerShape.of(hidden=96, q_dim=96, kv_dim=96, ffn=96, head_dim=32)      # rows not 16-byte aligned
    assert f(ctypes.byref(h), ctypes.byref(odd), ptrs, 2, 1, 4096, ws_bytes, 0, None) == q4.Q4_ERR_ARG
    wide = q4.LayerShape.of(hidden=256, q_dim=256, kv_dim=128, ffn=768, head_dim=64)  # 768/64 threads: no team split
    tc = q4.Q4_DEC_FUSED | q4.Q4_DEC_TENSOR_CORE
    core = q4.Q4_DEC_FUSED | q4.Q4_DEC_CUDA_CORE
    assert f(ctypes.byref(h), ctypes.byref(wide), ptrs, 2, 1, 4096, ws_bytes, core, None) == q4.Q4_ERR_ARG
    big = q4.LayerShape.of(hidden=16384, q_dim=256, kv_dim=128, ffn=1024, head_dim=64)  # tc: norm input > 8192
    assert f(ctypes.byref(h), ctypes.byref(big), ptrs, 2, 1, 4096, 1 << 30, tc, None) == q4.Q4_ERR_ARG
    chunked = q4.LayerShape.of(hidden=256, q_dim=256, kv_dim=128, ffn=3072, head_dim=64)  # tc: 3072 % 2048
    assert f(ctypes.byref(h), ctypes.byref(chunked), ptrs, 2, 1, 4096, 1 << 30, tc, None) == q4.Q4_ERR_ARG
    ragged = q4.LayerShape.of(hidden=256, q_dim=256, kv_dim=128, ffn=1056, head_dim=64)  # ffn not 256-aligned
    assert f(ctypes.byref(h), ctypes.byref(ragged), ptrs, 2, 1, 4096, ws_bytes, tc, None) == q4.Q4_ERR_ARG
    heads = q4.LayerShape.of(hidden=256, q_dim=256, kv_dim=128, ffn=1024, head_dim=32)  # CUDA-core: head_dim % 64
    assert f(ctypes.byref(h), ctypes.byref(heads), ptrs, 2, 1, 4096, ws_bytes, core, None) == q4.Q4_ERR_ARG
    # streaming ring
    s = ctypes.c_void_p()
    g = lib.q4_stream_create
    _, lb = q4.q4_layer_offsets(shape)
    assert g(ctypes.byref(s), ctypes.byref(shape), ptrs, 2, 1, 4096, 8192, lb - 1, 4096, ws_bytes, 0) == q4.Q4_ERR_OOM
    assert g(ctypes.byref(s), ctypes.byref(shape), ptrs, 2, 1, 4096, 8192 + 16, lb, 4096, ws_bytes, 0) == q4.Q4_ERR_ALIGN
    assert g(ctypes.byref(s), ctypes.byref(shape), ptrs, 2, 1, 4096, 8192, lb, 4096, ws_bytes, 128) == q4.Q4_ERR_ARG
    # the second staging buffer is required unless the ring runs single-buffered
    assert g(ctypes.byref(s), ctypes.byref(shape), ptrs, 2, 1, 4096, None, lb, 4096, ws_bytes, 0) == q4.Q4_ERR_ARG
    single = q4.Q4_STREAM_SINGLE_BUFFER
    assert g(ctypes.byref(s), ctypes.byref(shape), ptrs, 2, 1, 4096 + 16, None, lb, 4096, ws_bytes,
             single) == q4.Q4_ERR_ALIGN
    # partial residency: a layer needs a host block or a resident block; resident blocks 256-byte aligned
    gx = lib.q4_stream_create_ex
    none = (ctypes.c_void_p * 2)(None, None)
    res_bad = (ctypes.c_void_p * 2)(4096 + 16, None)
    assert gx(ctypes.byref(s), ctypes.byref(shape), none, None, 2, 1, 4096, 8192, lb, 4096, ws_bytes, 0) == q4.Q4_ERR_ARG
    assert gx(ctypes.byref(s), ctypes.byref(shape), ptrs, res_bad, 2, 1, 4096, 8192, lb, 4096, ws_bytes,
              0) == q4.Q4_ERR_ALIGN
    assert gx(ctypes.byref(s), ctypes.byref(shape), none, (ctypes.c_void_p * 2)(4096, None), 2, 1, 4096, 8192, lb,
              4096, ws_bytes, 0) == q4.Q4_ERR_ARG
    assert lib.q4_stream_layers(None, 4096, None, 0) == q4.Q4_ERR_ARG
    assert lib.q4_layer_decode(None, 4096, None) == q4.Q4_ERR_ARG
