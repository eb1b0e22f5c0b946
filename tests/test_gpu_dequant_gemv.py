"""GPU parity of dequantisation (bit-exact) and GEMV (1e-3 * sum|w x|) against the oracle.

Shapes cover several tiles with ragged tails, the K-split path, the generic
Q8_0 path (K not a multiple of 256), batch 1..8 and the workload sizes of the
Q8_0 decode layer and the Q4_K 4B-class sweep.
"""

import numpy as np
import pytest
import torch

import oracle
import quantized_decode_gguf_gb300 as phb
import synth
from _helpers import assert_within, check_device_clean, ensure_built, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


DEQ_SHAPES = [("q8_0", 1, 32), ("q8_0", 37, 96), ("q8_0", 64, 1024), ("q8_0", 300, 2048 + 32),
              ("q4_k", 1, 256), ("q4_k", 37, 512), ("q4_k", 129, 2560)]


@pytest.mark.parametrize("qtype,n,k", DEQ_SHAPES)
def test_dequant_fp32_bit_exact(qtype, n, k):
    blob = synth.blocks(qtype, 100, n, n, k)
    w = to_host(phb.dequant(qtype, to_dev(blob), n, k))
    want = oracle.dequant(qtype, blob, n, k)
    assert w.dtype == np.float32
    assert np.array_equal(w.view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("qtype,n,k", DEQ_SHAPES)
def test_dequant_bf16_bit_exact(qtype, n, k):
    blob = synth.blocks(qtype, 101, n, n, k)
    w = phb.dequant(qtype, to_dev(blob), n, k, bf16=True)
    got = to_host(w.float()).astype(np.float64)
    want = oracle.round_to_bf16(oracle.dequant(qtype, blob, n, k))
    assert np.array_equal(got, want)


def test_dequant_q4_k_adversarial_fields():
    # extreme fp16 scales (subnormal, max), all-15 quants and mins 63: exercises the single rounding
    blob = synth.q4_k_blocks(102, 0, 16, 512).reshape(-1, 144).copy()
    blob[0::4, 0:2] = [0x01, 0x00]       # d = smallest subnormal
    blob[1::4, 0:2] = [0xFF, 0x7B]       # d = 65504
    blob[2::4, 2:4] = [0xFF, 0x7B]       # dmin = 65504
    blob[3::4, 16:] = 0xFF               # q = 15 everywhere
    blob = blob.reshape(16, -1)
    w = to_host(phb.dequant("q4_k", to_dev(blob), 16, 512))
    want = oracle.dequant("q4_k", blob, 16, 512)
    assert np.array_equal(w.view(np.uint32), want.view(np.uint32))


GEMV_CASES = [
    ("q8_0", 1024, 1024, 1),      # single 1024x1024 GEMV workload
    ("q8_0", 3072, 2048, 1),      # decode layer: QKV
    ("q8_0", 2048, 5632, 1),      # decode layer: down
    ("q8_0", 11264, 2048, 1),     # decode layer: gate and up stacked
    ("q8_0", 37, 96, 3),          # generic path, ragged
    ("q8_0", 301, 2048 + 32, 2),  # generic path, K % 256 != 0
    ("q8_0", 333, 768, 5),
    ("q8_0", 160, 9728, 8),       # K split (8 * 9728 * 4 B > 80 KB)
    ("q4_k", 9728, 2560, 1),      # 4B-class sweep
    ("q4_k", 2560, 9728, 1),
    ("q4_k", 4096, 2560, 1),
    ("q4_k", 9728, 2560, 4),
    ("q4_k", 2560, 9728, 4),      # K split at batch 4
    ("q4_k", 4096, 2560, 4),
    ("q8_0", 1536, 4096, 1),      # batch 1, 32 half units per row, 5 rows per stage: positions fastest
    ("q8_0", 1000, 2560, 1),      # batch 1, 8 rows per stage: threads on row segments fastest, padded
    ("q4_k", 1280, 3072, 1),      # batch 1, 6 rows per stage (16 threads idle per stage)
    ("q4_k", 77, 256, 1),         # one super-block per row
    ("q4_k", 1000, 1280, 7),
    ("q4_k", 3, 512, 8),
]


@pytest.mark.parametrize("qtype,n,k,batch", GEMV_CASES)
def test_gemv_within_contract(qtype, n, k, batch):
    blob = synth.blocks(qtype, 200 + batch, n, n, k)
    x = synth.normal_f32(200 + batch, 10 * n + k, (batch, k))
    y = to_host(phb.gemv(qtype, to_dev(blob), to_dev(x), n, k))
    ref, s = oracle.gemv_quant(qtype, blob, x, n, k)
    assert_within(y, ref, 1e-3 * s, f"gemv {qtype} {n}x{k} b{batch}")
    check_device_clean()


@pytest.mark.parametrize("qtype", ["q8_0", "q4_k"])
def test_gemv_extreme_activation_magnitudes(qtype):
    # per-row power-of-two staging scale at its limits: a row whose largest
    # magnitude is below 2^-129 (scale capped at 2^254), a row near 1e30 and
    # an all-zero row, in one batch
    n, k = 300, 2048
    blob = synth.blocks(qtype, 210, n, n, k)
    x = synth.normal_f32(210, 1, (3, k))
    x[0] *= np.float32(1e-40)
    x[1] *= np.float32(1e30)
    x[2] = 0.0
    y = to_host(phb.gemv(qtype, to_dev(blob), to_dev(x), n, k))
    ref, s = oracle.gemv_quant(qtype, blob, x, n, k)
    assert np.all(np.isfinite(y))
    # Below 2^-126 an fp32 result is a subnormal, spaced 2^-149 apart: scaling a
    # 128-weight partial sum back into fp32 may round it by up to half that
    # spacing, 2^-150, once per partial (k / 128 of them), and so may the
    # result itself; relative error bounds say nothing there.
    quantum = (k // 128 + 1) * 2.0 ** -150
    assert_within(y, ref, 1e-3 * s + quantum, f"gemv {qtype} extreme magnitudes")
    assert np.all(y[2] == 0.0)
    check_device_clean()


@pytest.mark.parametrize("qtype,n,k", [("q8_0", 333, 2048), ("q8_0", 40, 2048 + 32), ("q4_k", 500, 2560),
                                       ("q4_k", 64, 9728)])
def test_gemv_unit_vectors_bit_exact(qtype, n, k):
    # x = e_k returns column k of the dequantised matrix exactly (one product, no rounding)
    blob = synth.blocks(qtype, 300, n, n, k)
    cols = np.array([0, 1, 31, 32, 255, 256, k // 2 + 3, k - 1])
    x = np.zeros((len(cols), k), dtype=np.float32)
    x[np.arange(len(cols)), cols] = 1.0
    y = to_host(phb.gemv(qtype, to_dev(blob), to_dev(x), n, k))
    w = oracle.dequant(qtype, blob, n, k)
    assert np.array_equal(y, w[:, cols].T)


def test_gemv_deterministic_and_batch_consistent():
    n, k = 2560, 9728
    blob = to_dev(synth.q4_k_blocks(301, 0, n, k))
    x = synth.normal_f32(301, 1, (4, k))
    y4a = to_host(phb.gemv("q4_k", blob, to_dev(x), n, k))
    y4b = to_host(phb.gemv("q4_k", blob, to_dev(x), n, k))
    assert np.array_equal(y4a, y4b)
    ref, s = oracle.gemv_quant("q4_k", synth.q4_k_blocks(301, 0, n, k), x, n, k)
    for b in range(4):
        y1 = to_host(phb.gemv("q4_k", blob, to_dev(x[b:b + 1]), n, k))
        assert_within(y1[0], ref[b], 1e-3 * s[b], "batch-1 vs oracle")
        assert np.allclose(y1[0], y4a[b], rtol=0, atol=float(2e-6 * s[b].max()))


def test_gemv_output_canary():
    # nothing is written past the end of y
    n, k = 1000, 2048
    blob = to_dev(synth.q8_0_blocks(302, 0, n, k))
    x = to_dev(synth.normal_f32(302, 1, (1, k)))
    buf = torch.full((n + 64,), 12345.0, device="cuda")
    phb.gemv("q8_0", blob, x, n, k, out=buf[:n].view(1, n))
    tail = to_host(buf[n:])
    assert np.all(tail == 12345.0)
