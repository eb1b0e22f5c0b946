"""GPU parity of the tensor-core prompt-processing GEMM.

Y[t][n] = sum_k bf16(w[n][k]) bf16(x[t][k]) with fp32 accumulation. Checked
against the oracle's bf16-operand product (every shape, bound K * 2^-23 *
sum|w_b x_b|, a twice-the-worst-case fp32 accumulation bound) and, at the
workload shapes, against the exact fp32-operand product under the
1e-3 * sum|w x| contract.
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


CASES = [
    ("q8_0", 64, 128, 256),      # one tile, one K unit
    ("q4_k", 256, 128, 512),     # one tile, K split over a cluster of 2
    ("q4_k", 300, 256, 1024),    # ragged tokens; a cluster of 4 splits per tile
    ("q8_0", 513, 384, 2048),    # ragged tokens past two tiles; clusters of 8
    ("q4_k", 300, 1280, 5120),   # clusters of 7 splits of 3 units (the last split 2)
    ("q8_0", 200, 1280, 4864),   # 10 splits: partials summed by the reduction kernel
    ("q4_k", 128, 768, 8192),    # 16 splits, one token tile of 128
    ("q4_k", 512, 9728, 2560),   # prompt-processing workload: 2560 -> 9728 (one tile per SM)
    ("q8_0", 512, 2560, 9728),   # 9728 -> 2560: clusters of 3 splits
    ("q8_0", 600, 9728, 512),    # 228 tiles: two waves of CTAs, ragged tokens
]


@pytest.mark.parametrize("qtype,m,n,k", CASES)
def test_prefill_gemm(qtype, m, n, k):
    seed = 700 + m + n
    blob = synth.blocks(qtype, seed, 0, n, k)
    x = synth.normal_f32(seed, 1, (m, k))
    y = to_host(phb.gemm_q_prefill(qtype, to_dev(blob), to_dev(x), n, k))
    w = oracle.dequant(qtype, blob, n, k)
    if n * m * k > 2e9:
        # workload shapes: sampled rows keep the float64 oracle fast
        rows = np.random.default_rng(seed).choice(n, size=384, replace=False)
        w, y = w[rows], y[:, rows]
    ye, se, yb, sb = oracle.prefill_gemm(w, x)
    assert_within(y, yb, k * 2.0 ** -23 * sb, f"prefill {qtype} {m}x{n}x{k} vs bf16 operands")
    if k >= 2048:
        assert_within(y, ye, 1e-3 * se, f"prefill {qtype} {m}x{n}x{k} vs fp32 operands")
    check_device_clean()


def test_prefill_identity_like_weights_exact():
    # Q8_0 with d = 1 and q = identity pattern: Y[t][n] = bf16(x[t][n]) exactly
    n = k = 256
    m = 128
    blob = np.zeros((n, k // 32, 34), dtype=np.uint8)
    blob[..., 0:2] = [0x00, 0x3C]                      # d = 1.0
    for r in range(n):
        blob[r, r // 32, 2 + r % 32] = 1
    blob = blob.reshape(n, -1)
    x = synth.normal_f32(710, 1, (m, k))
    y = to_host(phb.gemm_q_prefill("q8_0", to_dev(blob), to_dev(x), n, k))
    assert np.array_equal(y.astype(np.float64), oracle.round_to_bf16(x))


@pytest.mark.parametrize("qtype,m,n,k", [("q4_k", 300, 256, 1024), ("q4_k", 300, 1280, 5120),
                                         ("q8_0", 200, 1280, 4864)])
def test_prefill_deterministic(qtype, m, n, k):
    blob = to_dev(synth.blocks(qtype, 720, 0, n, k))
    x = to_dev(synth.normal_f32(720, 1, (m, k)))
    a = to_host(phb.gemm_q_prefill(qtype, blob, x, n, k))
    b = to_host(phb.gemm_q_prefill(qtype, blob, x, n, k))
    assert np.array_equal(a, b)


def test_prefill_workspace_reused_across_shapes():
    # one workspace serves calls of different grids and split plans; results
    # equal fresh-workspace ones
    shapes = [("q4_k", 300, 1280, 5120), ("q8_0", 512, 2560, 9728), ("q4_k", 64, 128, 256),
              ("q8_0", 512, 9728, 2560), ("q8_0", 200, 1280, 4864), ("q4_k", 600, 9728, 512)]
    size = max(phb.prefill_workspace_size(*shape) for shape in shapes)
    ws = torch.zeros(size, dtype=torch.uint8, device="cuda")
    inputs = []
    for i, (qtype, m, n, k) in enumerate(shapes):
        blob = to_dev(synth.blocks(qtype, 730 + i, 0, n, k))
        x = to_dev(synth.normal_f32(730 + i, 1, (m, k)))
        inputs.append((qtype, m, n, k, blob, x, to_host(phb.gemm_q_prefill(qtype, blob, x, n, k))))
    for _ in range(2):
        for qtype, m, n, k, blob, x, ref in inputs:
            y = to_host(phb.gemm_q_prefill(qtype, blob, x, n, k, ws=ws))
            assert np.array_equal(y, ref), (qtype, m, n, k)
    check_device_clean()
