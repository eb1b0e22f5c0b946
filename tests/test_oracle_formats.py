"""Pins of the oracle's format code (fp16, bf16, Q8_0, Q4_K) against definitions.

Nothing here calls the CUDA library. Each test checks the oracle against
something other than itself: the IEEE binary16 definition evaluated with
Python integers, exact rational arithmetic, hand-built blocks whose fields
and weights are worked out by hand from the layout, a test-side packer (the
inverse map) over every field value, and torch's own bf16 conversion.
"""

import math
import struct
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth


# ---------------------------------------------------------------- fp16 / bf16

def _fp16_by_definition(bits: int) -> float:
    sign = -1.0 if bits >> 15 else 1.0
    e = (bits >> 10) & 0x1F
    f = bits & 0x3FF
    if e == 0:
        return sign * math.ldexp(f, -24)
    return sign * math.ldexp(1024 + f, e - 25)


def test_fp16_decode_all_finite_patterns():
    bits = np.arange(1 << 16, dtype=np.uint32)
    finite = ((bits >> 10) & 0x1F) != 0x1F
    got = oracle.fp16_bits_to_f64(bits[finite].astype(np.uint16))
    want = np.array([_fp16_by_definition(int(b)) for b in bits[finite]])
    assert np.array_equal(got, want)
    assert np.array_equal(np.signbit(got), np.signbit(want))


def test_bf16_rounding_hand_cases():
    one_ulp = 2.0 ** -7                      # bf16 spacing in [1, 2)
    cases = {
        1.0: 1.0,
        1.0 + 2.0 ** -8: 1.0,                # tie -> even (mantissa 0)
        1.0 + 3 * 2.0 ** -8: 1.0 + 2 * one_ulp,  # tie -> even (mantissa 2)
        1.0 + 2.0 ** -8 + 2.0 ** -20: 1.0 + one_ulp,  # above the tie -> up
        -1.0 - 2.0 ** -8: -1.0,
    }
    for x, want in cases.items():
        got = float(oracle.round_to_bf16(np.float32(x)))
        assert got == want, (x, got, want)
    # overflow to infinity past the largest bf16
    assert np.isinf(oracle.round_to_bf16(np.float32(3.4e38)))
    assert np.isnan(oracle.round_to_bf16(np.float32(np.nan)))


def test_bf16_rounding_matches_torch():
    g = np.random.default_rng(7)
    x = np.concatenate([
        g.standard_normal(20000).astype(np.float32),
        (g.standard_normal(5000) * 1e-38).astype(np.float32),   # subnormals
        np.array([0.0, -0.0, 65504.0, 1e30, -1e-30], dtype=np.float32),
    ])
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.round_to_bf16(x)
    assert np.array_equal(got, want)


# ---------------------------------------------------------------- Q8_0

def _q8_0_block(d_bits: int, q) -> bytes:
    return struct.pack("<H", d_bits) + bytes(int(v) & 0xFF for v in q)


def test_q8_0_every_quant_times_scale_sweep():
    # all 255 generated quant values against fp16 scales incl. subnormals,
    # smallest normal, 1.0, the generator's range and the largest finite value
    d_list = [0x0001, 0x03FF, 0x0400, 0x1419, 0x211F, 0x3C00, 0x7BFF, 0xBC00]
    qs = list(range(-127, 128))
    for d_bits in d_list:
        rows = []
        for start in range(0, 255, 32):
            chunk = qs[start:start + 32]
            chunk = chunk + [0] * (32 - len(chunk))
            rows.append(_q8_0_block(d_bits, chunk))
        blob = np.frombuffer(b"".join(rows), dtype=np.uint8)
        k = 32 * len(rows)
        w = oracle.q8_0_dequant(blob, 1, k)[0]
        d = Fraction(_fp16_by_definition(d_bits))
        for i, qv in enumerate(qs):
            exact = d * qv
            assert Fraction(float(w[i])) == exact, (d_bits, qv)
        assert w.dtype == np.float32


def test_q8_0_unpack_positions():
    # block 0: d=1.0, q = 0..31; block 1: d=0.5, q = -1..-32
    b0 = _q8_0_block(0x3C00, range(32))
    b1 = _q8_0_block(0x3800, [-(i + 1) for i in range(32)])
    blob = np.frombuffer(b0 + b1, dtype=np.uint8)
    d, q = oracle.q8_0_unpack(blob, 1, 64)
    assert d.tolist() == [[1.0, 0.5]]
    assert q[0, 0].tolist() == list(range(32))
    assert q[0, 1].tolist() == [-(i + 1) for i in range(32)]
    w = oracle.q8_0_dequant(blob, 1, 64)[0]
    assert w[:32].tolist() == [float(i) for i in range(32)]
    assert w[32:].tolist() == [-(i + 1) * 0.5 for i in range(32)]


def test_q8_0_rows_are_consecutive_blocks():
    blob = synth.q8_0_blocks(1, 0, 3, 96)
    w = oracle.q8_0_dequant(blob, 3, 96)
    for r in range(3):
        wr = oracle.q8_0_dequant(blob[r], 1, 96)[0]
        assert np.array_equal(w[r], wr)


# ---------------------------------------------------------------- Q4_K

def _pack_q4_k(d_bits, dmin_bits, sc, m, q) -> bytes:
    """Test-side packer: the inverse of the k-quant layout, written from its description."""
    s = [0] * 12
    for j in range(4):
        s[j] = (sc[j] & 63) | ((sc[j + 4] >> 4) << 6)
        s[j + 4] = (m[j] & 63) | ((m[j + 4] >> 4) << 6)
        s[j + 8] = (sc[j + 4] & 15) | ((m[j + 4] & 15) << 4)
    qs = [0] * 128
    for c in range(4):
        for i in range(32):
            qs[32 * c + i] = (q[64 * c + i] & 15) | ((q[64 * c + 32 + i] & 15) << 4)
    return struct.pack("<HH", d_bits, dmin_bits) + bytes(s) + bytes(qs)


def test_q4_k_hand_block_single_fields():
    # d = 1.0, dmin = 0; scale bytes 1,2,3,4 -> sc_0..3 = 1..4, all else 0.
    # qs[0] = 0x21: weight 0 (low nibble, sub-block 0) = 1, weight 32
    # (high nibble, sub-block 1) = 2.
    blk = bytearray(144)
    blk[0:2] = struct.pack("<H", 0x3C00)
    blk[4:8] = bytes([1, 2, 3, 4])
    blk[16] = 0x21
    blob = np.frombuffer(bytes(blk), dtype=np.uint8)
    d, dmin, sc, m, q = oracle.q4_k_unpack(blob, 1, 256)
    assert d.tolist() == [[1.0]] and dmin.tolist() == [[0.0]]
    assert sc[0, 0].tolist() == [1, 2, 3, 4, 0, 0, 0, 0]
    assert m[0, 0].tolist() == [0] * 8
    want = np.zeros(256)
    want[0] = 1.0 * 1 * 1     # sub-block 0, sc 1, q 1
    want[32] = 1.0 * 2 * 2    # sub-block 1, sc 2, q 2
    assert np.array_equal(oracle.q4_k_dequant(blob, 1, 256)[0], want.astype(np.float32))


def test_q4_k_hand_block_high_scale_bits():
    # d = 1.0, dmin = 2.0
    # s[0] = 0xC5: sc_0 = 5, and its top two bits (3) become bits 4-5 of sc_4
    # s[4] = 0x4A: m_0 = 10, and its top two bits (1) become bits 4-5 of m_4
    # s[8] = 0x97: sc_4 low nibble 7, m_4 low nibble 9
    # -> sc_4 = 7 + 48 = 55, m_4 = 9 + 16 = 25
    # qs[64] = 0x0F: weight 128 (chunk 2 low nibble -> sub-block 4) = 15
    blk = bytearray(144)
    blk[0:4] = struct.pack("<HH", 0x3C00, 0x4000)
    blk[4 + 0] = 0xC5
    blk[4 + 4] = 0x4A
    blk[4 + 8] = 0x97
    blk[16 + 64] = 0x0F
    blob = np.frombuffer(bytes(blk), dtype=np.uint8)
    _, _, sc, m, q = oracle.q4_k_unpack(blob, 1, 256)
    assert sc[0, 0].tolist() == [5, 0, 0, 0, 55, 0, 0, 0]
    assert m[0, 0].tolist() == [10, 0, 0, 0, 25, 0, 0, 0]
    assert q[0, 0, 128] == 15 and q[0, 0].sum() == 15
    w = oracle.q4_k_dequant(blob, 1, 256)[0]
    want = np.zeros(256)
    want[0:32] = 1.0 * 5 * 0 - 2.0 * 10          # -20
    want[128:160] = -2.0 * 25                      # -50
    want[128] = 1.0 * 55 * 15 - 2.0 * 25           # 775
    assert np.array_equal(w, want.astype(np.float32))


def test_q4_k_pack_unpack_every_scale_min_in_every_slot():
    # all 64*64 (sc, m) pairs, each placed in every sub-block slot j
    pairs = [(a, b) for a in range(64) for b in range(64)]
    for j in range(8):
        blocks = []
        for (a, b) in pairs:
            sc = [(a + 7 * t) % 64 for t in range(8)]
            m = [(b + 13 * t) % 64 for t in range(8)]
            sc[j], m[j] = a, b
            blocks.append(_pack_q4_k(0x3C00, 0x3C00, sc, m, [0] * 256))
        blob = np.frombuffer(b"".join(blocks), dtype=np.uint8)
        _, _, sc_o, m_o, _ = oracle.q4_k_unpack(blob, 1, 256 * len(pairs))
        assert sc_o[0, :, j].tolist() == [p[0] for p in pairs]
        assert m_o[0, :, j].tolist() == [p[1] for p in pairs]
        for t in range(8):
            assert sc_o[0, :, t].tolist() == [((p[0] + 7 * t) % 64) if t != j else p[0] for p in pairs]
            assert m_o[0, :, t].tolist() == [((p[1] + 13 * t) % 64) if t != j else p[1] for p in pairs]


def test_q4_k_every_nibble_value_in_every_position():
    blocks = []
    for v in range(16):
        blocks.append(_pack_q4_k(0, 0, [0] * 8, [0] * 8, [v] * 256))
        blocks.append(_pack_q4_k(0, 0, [0] * 8, [0] * 8, [(v + i) % 16 for i in range(256)]))
    blob = np.frombuffer(b"".join(blocks), dtype=np.uint8)
    _, _, _, _, q = oracle.q4_k_unpack(blob, 1, 256 * len(blocks))
    for v in range(16):
        assert q[0, 2 * v].tolist() == [v] * 256
        assert q[0, 2 * v + 1].tolist() == [(v + i) % 16 for i in range(256)]


def test_q4_k_unpack_repack_random_bytes():
    blob = synth.q4_k_blocks(11, 0, 4, 512)
    d, dmin, sc, m, q = oracle.q4_k_unpack(blob, 4, 512)
    raw = blob.reshape(8, 144)
    for bi in range(8):
        r, c = divmod(bi, 2)
        again = _pack_q4_k(int(raw[bi, 0]) | int(raw[bi, 1]) << 8, int(raw[bi, 2]) | int(raw[bi, 3]) << 8,
                           sc[r, c].tolist(), m[r, c].tolist(), q[r, c].tolist())
        assert again == raw[bi].tobytes()


def test_q4_k_dequant_exact_rational():
    blob = synth.q4_k_blocks(5, 1, 3, 512)
    d, dmin, sc, m, q = oracle.q4_k_unpack(blob, 3, 512)
    w = oracle.q4_k_dequant(blob, 3, 512)
    for r in range(3):
        for b in range(2):
            for i in range(0, 256, 7):
                j = i // 32
                exact = (Fraction(float(d[r, b])) * int(sc[r, b, j]) * int(q[r, b, i])
                         - Fraction(float(dmin[r, b])) * int(m[r, b, j]))
                # one rounding of the exact value to fp32 (nearest even)
                assert float(w[r, 256 * b + i]) == float(np.float32(float(exact)))
                assert float(exact) == exact  # exact in float64, as the header argues


def test_q4_k_subblock_is_affine_in_q():
    # within a sub-block, w is affine in q with slope d*sc and offset -dmin*m
    blob = synth.q4_k_blocks(9, 2, 2, 256)
    d, dmin, sc, m, q = oracle.q4_k_unpack(blob, 2, 256)
    w = oracle.q4_k_dequant_f64(blob, 2, 256)
    for r in range(2):
        for j in range(8):
            seg = slice(32 * j, 32 * j + 32)
            assert np.allclose(w[r, seg], d[r, 0] * sc[r, 0, j] * q[r, 0, seg] - dmin[r, 0] * m[r, 0, j], rtol=0, atol=0)


# ---------------------------------------------------------------- generator

def test_generator_ranges_and_determinism():
    a = synth.q8_0_blocks(3, 4, 16, 256)
    b = synth.q8_0_blocks(3, 4, 16, 256)
    assert np.array_equal(a, b)
    d, q = oracle.q8_0_unpack(a, 16, 256)
    assert d.min() >= 1e-3 * (1 - 2 ** -10) and d.max() <= 1e-2 * (1 + 2 ** -10)
    assert q.min() >= -127 and q.max() <= 127
    k4 = synth.q4_k_blocks(3, 5, 8, 1024)
    d, dmin, sc, m, q = oracle.q4_k_unpack(k4, 8, 1024)
    assert dmin.min() >= 1e-3 * (1 - 2 ** -10) and dmin.max() <= 1e-2 * (1 + 2 ** -10)
    assert sc.max() <= 63 and m.max() <= 63 and q.max() <= 15
    assert synth.row_bytes("q8_0", 2048) == 2176 and synth.row_bytes("q4_k", 2560) == 1440
