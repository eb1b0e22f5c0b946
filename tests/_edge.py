"""Edge-case quantized matrices for the parity tests.

Each builder starts from a seeded random matrix (synth) and overwrites byte
fields row by row, so that rows of every kind sit side by side in one
matrix at the workload shapes. The kinds are the degenerate cases of the two
block formats: zero quants under a nonzero scale, the int8 value -128,
quants in {-1, 0, 1}, zero scales, Q4_K sub-blocks whose scale term cancels
the min term exactly (d*sc*q == dmin*m, so the weight is exactly zero),
zero 6-bit scales with or without a min, and rows mixing such blocks with
ordinary ones.

The byte positions follow the GGUF layouts (Q8_0: fp16 d in bytes 0-1,
int8 q in 2-33; Q4_K: fp16 d in 0-1, dmin in 2-3, twelve 6-bit scale/min
bytes in 4-15, 4-bit quants in 16-143). Two facts about the Q4_K scale
bytes are used, and the CPU tests check both through the oracle:
  * all twelve bytes equal to 0x11 give sc_j == m_j for every sub-block j
    (17 for j < 4, 1 for j >= 4), so with d == dmin and every quant 1 each
    weight is d*sc - dmin*m = 0 exactly;
  * all twelve bytes zero give sc_j = m_j = 0, so every weight is zero.
"""

from __future__ import annotations

import numpy as np

import synth

Q8_KINDS = ("zero_quants", "unit_quants", "minus_128", "minus_128_mixed", "zero_blocks_mixed",
            "single_nonzero", "ordinary", "zero_scale")
Q4_KINDS = ("cancel_exact", "zero_scale_min", "zero_scale_min_nonzero", "cancel_mixed", "near_cancel",
            "max_fields", "single_nonzero", "ordinary")


def _rows(n: int, kinds, kind: str) -> np.ndarray:
    return np.arange(kinds.index(kind), n, len(kinds))


def q8_0_edge(seed: int, n: int, k: int):
    """Q8_0 [n, k] matrix; row r has kind Q8_KINDS[r % 8]. Returns (blob, kinds per row)."""
    g = synth.rng(seed, 9000)
    nb = k // 32
    b = synth.q8_0_blocks(seed, 9001, n, k).reshape(n, nb, 34).copy()
    q = b[..., 2:]
    q[_rows(n, Q8_KINDS, "zero_quants")] = 0
    r = _rows(n, Q8_KINDS, "unit_quants")
    q[r] = g.integers(-1, 2, size=(len(r), nb, 32)).astype(np.int8).view(np.uint8)
    q[_rows(n, Q8_KINDS, "minus_128")] = 0x80
    q[_rows(n, Q8_KINDS, "minus_128_mixed"), 0::2] = 0x80
    q[_rows(n, Q8_KINDS, "zero_blocks_mixed"), 1::2] = 0
    r = _rows(n, Q8_KINDS, "single_nonzero")
    q[r] = 0
    q[r, g.integers(0, nb, size=len(r)), g.integers(0, 32, size=len(r))] = 1
    b[_rows(n, Q8_KINDS, "zero_scale"), 0::3, 0:2] = 0
    return b.reshape(n, -1), [Q8_KINDS[i % len(Q8_KINDS)] for i in range(n)]


def q4_k_edge(seed: int, n: int, k: int):
    """Q4_K [n, k] matrix; row r has kind Q4_KINDS[r % 8]. Returns (blob, kinds per row)."""
    g = synth.rng(seed, 9100)
    nb = k // 256
    b = synth.q4_k_blocks(seed, 9101, n, k).reshape(n, nb, 144).copy()

    def cancel(rows, blocks):
        b[rows[:, None], blocks, 2:4] = b[rows[:, None], blocks, 0:2]  # dmin = d
        b[rows[:, None], blocks, 4:16] = 0x11                          # sc_j == m_j for every j
        b[rows[:, None], blocks, 16:] = 0x11                           # every quant 1

    every, even = np.arange(nb), np.arange(0, nb, 2)
    cancel(_rows(n, Q4_KINDS, "cancel_exact"), every)
    b[_rows(n, Q4_KINDS, "zero_scale_min"), :, 4:16] = 0
    # sc_j = 0 for every j and m_j random nonzero. sc_0..3 are the low 6 bits of
    # bytes 0-3, sc_4..7 the low nibbles of bytes 8-11 with bits 6-7 of bytes 0-3
    # on top; m_0..3 are the low 6 bits of bytes 4-7, m_4..7 the high nibbles of
    # bytes 8-11 with bits 6-7 of bytes 4-7 on top
    r = _rows(n, Q4_KINDS, "zero_scale_min_nonzero")
    mins = g.integers(1, 64, size=(len(r), nb, 8))
    s = np.zeros((len(r), nb, 12), dtype=np.int64)
    s[..., 4:8] = mins[..., 0:4] | ((mins[..., 4:8] >> 4) << 6)
    s[..., 8:12] = (mins[..., 4:8] & 15) << 4
    b[r, :, 4:16] = s.astype(np.uint8)
    cancel(_rows(n, Q4_KINDS, "cancel_mixed"), even)
    r = _rows(n, Q4_KINDS, "near_cancel")
    cancel(r, every)
    nib = g.integers(0, 3, size=(len(r), nb, 128, 2))
    b[r, :, 16:] = (nib[..., 0] | (nib[..., 1] << 4)).astype(np.uint8)
    r = _rows(n, Q4_KINDS, "max_fields")
    b[r, :, 4:] = 0xFF
    r = _rows(n, Q4_KINDS, "single_nonzero")
    cancel(r, every)
    # low nibble 2: one weight d*sc, every other weight stays zero
    b[r, g.integers(0, nb, size=len(r)), 16 + g.integers(0, 128, size=len(r))] = 0x12
    return b.reshape(n, -1), [Q4_KINDS[i % len(Q4_KINDS)] for i in range(n)]


def edge(qtype: str, seed: int, n: int, k: int):
    if qtype == "q8_0":
        return q8_0_edge(seed, n, k)
    if qtype == "q4_k":
        return q4_k_edge(seed, n, k)
    raise ValueError(qtype)


# Kinds whose rows dequantise to all-zero weights.
ZERO_ROW_KINDS = {"zero_quants", "cancel_exact", "zero_scale_min"}
