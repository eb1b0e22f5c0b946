"""GPU parity of decode attention at context depth (phb_attention_decode).

The oracle (oracle.attention_decode) evaluates the softmax in float64 and
returns the fp32 error bound of each output element; the kernel must land
inside it. Cases span one position, ragged tails shorter than a stage (128
positions with the tensor-core score path, 28 with the CUDA-core one), many
chunks, grouped-query heads that are not a power of two, more than 8 query
heads per KV head (two head groups), all three head sizes and the
32k-position workload the bench times.
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


def _inputs(seed, length, n_q, n_kv, hd, q_scale=1.0):
    q = (q_scale * synth.normal_f32(seed, 0, (n_q, hd))).astype(np.float32)
    k = synth.normal_f16(seed, 1, (length, n_kv, hd))
    v = synth.normal_f16(seed, 2, (length, n_kv, hd))
    return q, k, v


def _run(q, k, v, n_ctx, n_q, n_kv, hd, scale):
    out = phb.attention_decode(to_dev(q), to_dev(k), to_dev(v), n_ctx, n_q, n_kv, hd, scale=scale)
    return to_host(out)


def _scale(hd):
    # the fp32 value the kernel uses, handed to the oracle as is
    return float(np.float32(1.0 / np.sqrt(hd)))


CASES = [
    # (n_ctx, n_q, n_kv, head_dim)
    (37, 8, 2, 64),         # one ragged stage
    (1000, 16, 4, 128),     # 31 full stages and a tail of 8
    (4096, 32, 8, 128),     # 8B-class grouped-query heads
    (2049, 28, 4, 128),     # 7 query heads per KV head
    (513, 16, 1, 64),       # 16 query heads on one KV head: two head groups
    (300, 8, 8, 256),       # one query head per KV head
    (5000, 4, 2, 256),
    (32768, 16, 4, 128),    # the depth-32k workload
    (1500, 8, 8, 128),      # one query head per KV head on the tensor-core path
    (700, 4, 2, 64),        # two query heads per KV head, head_dim 64
    (1200, 16, 2, 256),     # eight query heads per KV head, head_dim 256
]


@pytest.mark.parametrize("n_ctx,n_q,n_kv,hd", CASES)
def test_attention_within_bound(n_ctx, n_q, n_kv, hd):
    q, k, v = _inputs(n_ctx + hd, n_ctx, n_q, n_kv, hd)
    sc = _scale(hd)
    y = _run(q, k, v, n_ctx, n_q, n_kv, hd, sc)
    ref, tol = oracle.attention_decode(q, k, v, n_q, n_kv, hd, scale=sc)
    assert_within(y, ref, tol, f"attention L={n_ctx} nq={n_q} nkv={n_kv} hd={hd}")
    check_device_clean()


def test_single_position_returns_v_exactly():
    # one key: weight exactly 1 in every chunk and merge step, so out = V bit for bit
    q, k, v = _inputs(11, 1, 16, 4, 128)
    y = _run(q, k, v, 1, 16, 4, 128, _scale(128))
    for h in range(16):
        assert np.array_equal(y[h], v[0, h // 4].astype(np.float32))


def test_positions_past_n_ctx_are_ignored():
    # a cache with room for more positions; the unused tail holds values that would dominate
    n_ctx, cap, n_q, n_kv, hd = 777, 1024, 16, 4, 128
    q, k, v = _inputs(12, cap, n_q, n_kv, hd)
    k[n_ctx:] = np.float16(60000.0)
    v[n_ctx:] = np.float16(-60000.0)
    sc = _scale(hd)
    y = _run(q, k, v, n_ctx, n_q, n_kv, hd, sc)
    ref, tol = oracle.attention_decode(q, k[:n_ctx], v[:n_ctx], n_q, n_kv, hd, scale=sc)
    assert_within(y, ref, tol, "cache prefix")


def test_wide_score_range_rescales_the_running_state():
    # large query: scores spread over hundreds, so running maxima change many times
    n_ctx, n_q, n_kv, hd = 3000, 8, 2, 128
    q, k, v = _inputs(13, n_ctx, n_q, n_kv, hd, q_scale=30.0)
    y = _run(q, k, v, n_ctx, n_q, n_kv, hd, 1.0)
    ref, tol = oracle.attention_decode(q, k, v, n_q, n_kv, hd, scale=1.0)
    assert_within(y, ref, tol, "wide scores")


def test_dominant_key_selects_its_value():
    n_ctx, n_q, n_kv, hd = 2500, 4, 1, 64
    q, k, v = _inputs(14, n_ctx, n_q, n_kv, hd)
    k[1717, 0] = (4.0 * q[0]).astype(np.float16)
    sc = 1.0
    y = _run(q, k, v, n_ctx, n_q, n_kv, hd, sc)
    ref, tol = oracle.attention_decode(q, k, v, n_q, n_kv, hd, scale=sc)
    assert_within(y, ref, tol, "dominant key")
    assert np.allclose(y[0], v[1717, 0].astype(np.float32), atol=1e-4)


def test_repeatable_and_replays_in_a_cuda_graph():
    n_ctx, n_q, n_kv, hd = 8191, 16, 4, 128
    q, k, v = _inputs(15, n_ctx, n_q, n_kv, hd)
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    ws = phb.workspace(phb.attention_workspace_size(n_ctx, n_q, n_kv, hd))
    out = torch.empty((n_q, hd), dtype=torch.float32, device="cuda")
    phb.attention_decode(qd, kd, vd, n_ctx, n_q, n_kv, hd, out=out, ws=ws)
    first = to_host(out).copy()
    phb.attention_decode(qd, kd, vd, n_ctx, n_q, n_kv, hd, out=out, ws=ws)
    assert np.array_equal(to_host(out), first)
    out.zero_()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            phb.attention_decode(qd, kd, vd, n_ctx, n_q, n_kv, hd, out=out, ws=ws)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        out.zero_()
        g.replay()
        assert np.array_equal(to_host(out), first)
    ref, tol = oracle.attention_decode(q, k, v, n_q, n_kv, hd, scale=_scale(hd))
    assert_within(first, ref, tol, "graph case")
    check_device_clean()
