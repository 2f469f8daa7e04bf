"""Helpers for the GPU tests: device copies, binary16 ulp distance, tolerance."""
import numpy as np
import torch

import oracle as ora


def dev_u8(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.uint8).reshape(-1).copy()).cuda()


def dev_u16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).astype(np.uint16).view(np.int16).copy()).cuda()


def host_u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def host_f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.float32).numpy().astype(np.float64)


def ordered(bits: np.ndarray) -> np.ndarray:
    """Map binary16 bit patterns to integers in the order of their values."""
    b = bits.astype(np.int64)
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


def f16_ulps(a_bits, b_bits) -> np.ndarray:
    return np.abs(ordered(np.asarray(a_bits)) - ordered(np.asarray(b_bits)))


def assert_within_tol(y_gpu, y_ref, s_ref, what=""):
    err = np.abs(np.asarray(y_gpu, dtype=np.float64) - y_ref)
    tol = ora.tolerance(s_ref)
    bad = err > tol
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} elements outside 1e-3*S+1e-5; "
                           f"worst err/tol {float((err / tol).max()):.3g}")
    return float((err / tol).max())
