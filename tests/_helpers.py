"""Shared helpers of the GPU parity tests."""

import numpy as np
import torch

import quantized_decode_gguf_gb300 as phb
from quantized_decode_gguf_gb300 import build


def ensure_built():
    build.build()


def to_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def to_host(t: torch.Tensor) -> np.ndarray:
    torch.cuda.synchronize()
    return t.detach().cpu().numpy()


def assert_within(y_gpu: np.ndarray, y_ref: np.ndarray, tol: np.ndarray, what: str = ""):
    """|y_gpu - y_ref| <= tol elementwise, with a readable failure."""
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    err = np.abs(y_gpu - y_ref)
    bad = ~(err <= tol)
    if bad.any():
        i = np.unravel_index(np.argmax(np.where(bad, err / np.maximum(tol, 1e-300), 0)), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; worst at {i}: "
                             f"gpu={y_gpu[i]!r} ref={y_ref[i]!r} err={err[i]:.3e} tol={tol[i]:.3e}")
    assert np.isfinite(y_gpu).all(), what


def check_device_clean():
    assert phb.device_error() == 0
