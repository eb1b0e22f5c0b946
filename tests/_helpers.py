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


def _f32(ws: torch.Tensor, offset: int, count: int) -> np.ndarray:
    torch.cuda.synchronize()
    return ws[offset:offset + 4 * count].cpu().numpy().view(np.float32).astype(np.float64)


def ffn_hidden(ws: torch.Tensor, batch: int, d_ff: int) -> np.ndarray:
    """The SwiGLU activation a phb_ffn_swiglu call left at the start of its workspace."""
    return _f32(ws, 0, batch * d_ff).reshape(batch, d_ff)


def moe_intermediates(ws: torch.Tensor, t: int, top_k: int, d_model: int, d_ff: int):
    """(per-pair activations [t*top_k, d_ff], per-pair expert outputs [t*top_k, d_model])
    that a phb_moe_ffn call left at the start of its workspace."""
    pairs = t * top_k
    yp = _f32(ws, 0, pairs * d_model).reshape(pairs, d_model)
    h_off = (pairs * d_model * 4 + 255) // 256 * 256
    return _f32(ws, h_off, pairs * d_ff).reshape(pairs, d_ff), yp


def assert_stages(stages: dict, dev: dict, what: str):
    """Every stage of a composed step within its one-GEMV-deep bound."""
    for name, (ref, tol) in stages.items():
        assert_within(np.atleast_2d(dev[name]), ref, tol, f"{what}: stage {name}")
