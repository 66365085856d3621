"""Helpers for the GPU parity tests: move bf16 bit patterns between NumPy and
CUDA tensors, run the oracle on the same inputs, compare with the acceptance
tolerance max|d| <= 2e-2 * max|ref| per tensor."""

import numpy as np
import torch

from oracle import layer as OL

TOL = 2e-2


def to_dev(bits: np.ndarray) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16).copy()).view(torch.bfloat16)
    return t.cuda()


def from_dev(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


class _DevView:
    """Exposes a raw device range through __cuda_array_interface__ so that
    torch can copy it without owning it."""

    def __init__(self, ptr: int, nbytes: int):
        self.__cuda_array_interface__ = {"shape": (nbytes // 2,), "typestr": "<i2", "data": (int(ptr), False),
                                         "version": 3, "strides": None}


def dev_buffer_bits(ptr: int, nbytes: int) -> np.ndarray:
    """Copy nbytes at a device address into a NumPy uint16 array."""
    t = torch.as_tensor(_DevView(ptr, nbytes), device="cuda")
    return t.cpu().numpy().view(np.uint16).copy()


def rel_err(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    scale = np.max(np.abs(ref))
    return float(np.max(np.abs(got - ref)) / (scale if scale > 0 else 1.0))


def assert_close(name, got, ref, tol=TOL):
    e = rel_err(got, ref)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    assert e <= tol, f"{name}: max|d| / max|ref| = {e:.3e} > {tol}"
    return e


def f64(bits):
    return OL.bf16_bits_to_f64(bits)
