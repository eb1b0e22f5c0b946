"""Seeded synthetic inputs for the GGUF dequantize-and-multiply path.

This module is the one piece shared by the CPU oracle's tests and the CUDA
path's tests and benchmark. It draws random bytes and numbers and nothing
else: it holds none of the method's arithmetic (no unpacking, no
dequantisation, no dot products, no routing).

Distributions follow the workloads of the Phobos README (githubhelp.com,
joa/phobos-lang, section "Inference": Q8_0 and Q4_K_M GGUF models), with the
per-field ranges of the synthetic weights:

* Q8_0 block (34 bytes): an fp16 scale ``d`` drawn from U[1e-3, 1e-2] in
  double and rounded to fp16 (round to nearest even), stored little-endian,
  followed by 32 signed bytes ``q`` drawn uniformly from the integers
  -127..127 (-128 is never drawn).
* Q4_K block (144 bytes): fp16 ``d`` and ``dmin`` drawn like the Q8_0 scale,
  then 140 uniformly random bytes. Those bytes hold sixteen 6-bit fields (the
  eight sub-block scales and mins) and 256 4-bit quants; since the 140 bytes
  pack exactly 12*8 + 128*8 bits of independent fields, uniform bytes are the
  same as independent uniform ``sc``, ``m`` in 0..63 and ``q`` in 0..15 under
  any bijective packing, so the generator needs no knowledge of the layout.
* Activations and router logits: fp32 N(0, 1).

Every tensor is keyed on (seed, tensor id) through numpy's SeedSequence, so
any tensor can be regenerated alone, in any order.
"""

from __future__ import annotations

import numpy as np

Q8_0_BLOCK_WEIGHTS = 32
Q8_0_BLOCK_BYTES = 34
Q4_K_BLOCK_WEIGHTS = 256
Q4_K_BLOCK_BYTES = 144

SCALE_LO = 1e-3
SCALE_HI = 1e-2


def rng(seed: int, tensor_id: int) -> np.random.Generator:
    """Independent generator for one tensor of one workload."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed) & 0xFFFFFFFFFFFF,
                                                                        int(tensor_id)])))


def _fp16_scale_bytes(g: np.random.Generator, count: int) -> np.ndarray:
    """``count`` fp16 values from U[SCALE_LO, SCALE_HI], as little-endian byte pairs."""
    vals = g.uniform(SCALE_LO, SCALE_HI, size=count).astype(np.float16)
    return vals.astype("<f2").view(np.uint8).reshape(count, 2)


def q8_0_blocks(seed: int, tensor_id: int, n_rows: int, k: int) -> np.ndarray:
    """Random Q8_0 matrix: uint8 array of shape [n_rows, k/32*34], rows contiguous."""
    if k % Q8_0_BLOCK_WEIGHTS:
        raise ValueError("k must be a multiple of 32 for Q8_0")
    g = rng(seed, tensor_id)
    nb = n_rows * (k // Q8_0_BLOCK_WEIGHTS)
    out = np.empty((nb, Q8_0_BLOCK_BYTES), dtype=np.uint8)
    out[:, 0:2] = _fp16_scale_bytes(g, nb)
    out[:, 2:] = g.integers(-127, 128, size=(nb, 32), dtype=np.int8).view(np.uint8)
    return out.reshape(n_rows, -1)


def q4_k_blocks(seed: int, tensor_id: int, n_rows: int, k: int) -> np.ndarray:
    """Random Q4_K matrix: uint8 array of shape [n_rows, k/256*144], rows contiguous."""
    if k % Q4_K_BLOCK_WEIGHTS:
        raise ValueError("k must be a multiple of 256 for Q4_K")
    g = rng(seed, tensor_id)
    nb = n_rows * (k // Q4_K_BLOCK_WEIGHTS)
    out = np.frombuffer(g.bytes(nb * Q4_K_BLOCK_BYTES), dtype=np.uint8).reshape(nb, Q4_K_BLOCK_BYTES).copy()
    out[:, 0:2] = _fp16_scale_bytes(g, nb)
    out[:, 2:4] = _fp16_scale_bytes(g, nb)
    return out.reshape(n_rows, -1)


def blocks(qtype: str, seed: int, tensor_id: int, n_rows: int, k: int) -> np.ndarray:
    """Dispatch on the format name ("q8_0" or "q4_k")."""
    if qtype == "q8_0":
        return q8_0_blocks(seed, tensor_id, n_rows, k)
    if qtype == "q4_k":
        return q4_k_blocks(seed, tensor_id, n_rows, k)
    raise ValueError(f"unknown format {qtype!r}")


def row_bytes(qtype: str, k: int) -> int:
    """Bytes of one quantized row of k weights."""
    if qtype == "q8_0":
        return k // Q8_0_BLOCK_WEIGHTS * Q8_0_BLOCK_BYTES
    if qtype == "q4_k":
        return k // Q4_K_BLOCK_WEIGHTS * Q4_K_BLOCK_BYTES
    raise ValueError(f"unknown format {qtype!r}")


def normal_f32(seed: int, tensor_id: int, shape) -> np.ndarray:
    """fp32 N(0, 1) tensor (activations, router logits)."""
    return rng(seed, tensor_id).standard_normal(size=shape, dtype=np.float32)


# Seeds of the five workloads: 0x5EED0000 + workload number.
SEED_BASE = 0x5EED0000


def workload_seed(n: int) -> int:
    return SEED_BASE + int(n)


def normal_f16(seed: int, tensor_id: int, shape) -> np.ndarray:
    """N(0, 1) values rounded to fp16 (round to nearest even), e.g. a KV cache."""
    return normal_f32(seed, tensor_id, shape).astype(np.float16)
