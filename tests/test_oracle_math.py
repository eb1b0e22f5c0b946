"""Pins of the oracle's arithmetic (GEMV, SwiGLU, MoE, prefill GEMM, decode layer).

Each test checks the oracle against something other than its own code path:
exact rational brute force on tiny inputs, closed forms (unit vectors, zero
inputs, constant vectors), invariants (softmax sums, linearity) and library
routines the special case reduces to (scipy's softmax and expit).
"""

import math
from fractions import Fraction

import numpy as np
import pytest
from scipy.special import expit, softmax

import oracle
import synth


def _frac_matrix(w):
    return [[Fraction(float(v)) for v in row] for row in w]


# ---------------------------------------------------------------- GEMV

@pytest.mark.parametrize("qtype,n,k", [("q8_0", 5, 64), ("q4_k", 3, 256)])
def test_gemv_exact_rational_brute_force(qtype, n, k):
    blob = synth.blocks(qtype, 21, 0, n, k)
    x = synth.normal_f32(21, 1, (2, k))
    y, s = oracle.gemv_quant(qtype, blob, x, n, k)
    w = oracle.dequant(qtype, blob, n, k)
    wf = _frac_matrix(w)
    for b in range(2):
        xf = [Fraction(float(v)) for v in x[b]]
        for r in range(n):
            exact = sum(wr * xr for wr, xr in zip(wf[r], xf))
            sabs = sum(abs(wr * xr) for wr, xr in zip(wf[r], xf))
            assert abs(Fraction(float(y[b, r])) - exact) <= Fraction(1, 10 ** 12) * sabs
            assert abs(Fraction(float(s[b, r])) - sabs) <= Fraction(1, 10 ** 12) * sabs


@pytest.mark.parametrize("qtype,n,k", [("q8_0", 7, 96), ("q4_k", 4, 512)])
def test_gemv_unit_vectors_give_columns_exactly(qtype, n, k):
    blob = synth.blocks(qtype, 22, 0, n, k)
    w = oracle.dequant(qtype, blob, n, k)
    x = np.eye(k, dtype=np.float32)
    y, s = oracle.gemv_quant(qtype, blob, x, n, k)
    assert np.array_equal(y, w.T.astype(np.float64))
    assert np.array_equal(s, np.abs(w.T).astype(np.float64))


def test_gemv_ones_gives_row_sums_and_s_bounds_y():
    blob = synth.q8_0_blocks(23, 0, 9, 128)
    d, q = oracle.q8_0_unpack(blob, 9, 128)
    y, s = oracle.gemv_quant("q8_0", blob, np.ones((1, 128), np.float32), 9, 128)
    row_sums = (d * q.sum(axis=-1)).sum(axis=-1)          # sum_b d_b * sum_i q_bi
    assert np.allclose(y[0], row_sums, rtol=1e-14, atol=0)
    x = synth.normal_f32(23, 1, (3, 128))
    y, s = oracle.gemv_quant("q8_0", blob, x, 9, 128)
    assert np.all(np.abs(y) <= s)


def test_gemv_is_linear_in_x():
    blob = synth.q4_k_blocks(24, 0, 6, 256)
    x1 = synth.normal_f32(24, 1, (1, 256))
    x2 = synth.normal_f32(24, 2, (1, 256))
    y1, _ = oracle.gemv_quant("q4_k", blob, x1, 6, 256)
    y2, _ = oracle.gemv_quant("q4_k", blob, x2, 6, 256)
    y12, s12 = oracle.gemv_quant("q4_k", blob, np.vstack([x1, x2]), 6, 256)
    tight = 1e-13 * float(s12.max())
    assert np.allclose(y12[0], y1[0], rtol=0, atol=tight) and np.allclose(y12[1], y2[0], rtol=0, atol=tight)
    y3, _ = oracle.gemv_quant("q4_k", blob, 2 * x1.astype(np.float64) - x2, 6, 256)
    assert np.allclose(y3, 2 * y1 - y2, rtol=0, atol=1e-12 * float(s12.max()))


# ---------------------------------------------------------------- SwiGLU

def test_silu_closed_forms():
    g = np.array([0.0, 1.0, -1.0, 30.0, -30.0, 1e-8])
    s = oracle.silu(g)
    assert s[0] == 0.0
    assert np.allclose(s, g * expit(g), rtol=1e-15, atol=0)
    assert abs(s[3] - 30.0) < 1e-11 and abs(s[4]) < 1e-11
    # the slope bound used by the tolerance: max silu' on a fine grid
    t = np.linspace(-20, 20, 400001)
    slope = expit(t) * (1 + t * (1 - expit(t)))
    assert slope.max() < oracle.gguf.SILU_SLOPE_MAX and slope.max() > 1.09


def test_swiglu_zero_input_and_zero_gate():
    wg = oracle.q8_0_dequant(synth.q8_0_blocks(25, 0, 8, 32), 8, 32)
    wu = oracle.q8_0_dequant(synth.q8_0_blocks(25, 1, 8, 32), 8, 32)
    wd = oracle.q8_0_dequant(synth.q8_0_blocks(25, 2, 32, 32), 32, 32)[:, :8]
    y, tol, h = oracle.swiglu_ffn(wg, wu, wd, np.zeros((1, 32)))
    assert np.all(y == 0) and np.all(tol == 0) and np.all(h == 0)
    x = synth.normal_f32(25, 3, (1, 32))
    y, tol, h = oracle.swiglu_ffn(np.zeros_like(wg), wu, wd, x)
    assert np.all(h == 0) and np.all(y == 0)


def test_swiglu_brute_force_python():
    d_model, d_ff = 32, 8
    wg = oracle.q8_0_dequant(synth.q8_0_blocks(26, 0, d_ff, d_model), d_ff, d_model)
    wu = oracle.q8_0_dequant(synth.q8_0_blocks(26, 1, d_ff, d_model), d_ff, d_model)
    wd = oracle.q8_0_dequant(synth.q8_0_blocks(26, 2, d_model, 32), d_model, 32)[:, :d_ff]
    x = synth.normal_f32(26, 3, (1, d_model))
    y, tol, h = oracle.swiglu_ffn(wg, wu, wd, x)
    xs = [float(v) for v in x[0]]
    hs = []
    for j in range(d_ff):
        g = math.fsum(float(wg[j, i]) * xs[i] for i in range(d_model))
        u = math.fsum(float(wu[j, i]) * xs[i] for i in range(d_model))
        hs.append(g / (1.0 + math.exp(-g)) * u)
    for i in range(d_model):
        yi = math.fsum(float(wd[i, j]) * hs[j] for j in range(d_ff))
        assert abs(y[0, i] - yi) <= 1e-12 * (1 + abs(yi))
        assert tol[0, i] > 0
    assert np.allclose(h[0], hs, rtol=1e-13, atol=1e-15)


# ---------------------------------------------------------------- MoE routing

def test_route_ties_go_to_lower_index():
    logits = np.array([[1.0, 3.0, 3.0, 2.0, 3.0]])
    idx, p = oracle.moe_route(logits, 2)
    assert idx.tolist() == [[1, 2]]
    assert np.allclose(p, [[0.5, 0.5]], rtol=1e-15)
    idx, p = oracle.moe_route(logits, 4)
    assert idx.tolist() == [[1, 2, 4, 3]]


def test_route_all_equal_and_top1():
    idx, p = oracle.moe_route(np.zeros((2, 128)), 8)
    assert idx.tolist() == [list(range(8))] * 2
    assert np.all(p == 1 / 8)
    lg = synth.normal_f32(27, 0, (16, 128))
    idx, p = oracle.moe_route(lg, 1)
    assert np.all(p == 1.0)
    assert np.array_equal(idx[:, 0], lg.argmax(axis=1))


def test_route_equals_full_softmax_renormalised():
    lg = synth.normal_f32(28, 0, (16, 128)).astype(np.float64)
    idx, p = oracle.moe_route(lg, 8)
    full = softmax(lg, axis=1)
    sel = np.take_along_axis(full, idx, axis=1)
    assert np.allclose(p, sel / sel.sum(axis=1, keepdims=True), rtol=1e-13, atol=0)
    assert np.allclose(p.sum(axis=1), 1.0, rtol=1e-15)
    # selected logits are the 8 largest, in descending order
    srt = -np.sort(-lg, axis=1)[:, :8]
    assert np.array_equal(np.take_along_axis(lg, idx, axis=1), srt)


def _expert_weights(seed, e, d_model, d_ff):
    wg = np.stack([oracle.q4_k_dequant(synth.q4_k_blocks(seed, 3 * i, d_ff, d_model), d_ff, d_model) for i in range(e)])
    wu = np.stack([oracle.q4_k_dequant(synth.q4_k_blocks(seed, 3 * i + 1, d_ff, d_model), d_ff, d_model) for i in range(e)])
    wd = np.stack([oracle.q4_k_dequant(synth.q4_k_blocks(seed, 3 * i + 2, d_model, d_ff), d_model, d_ff) for i in range(e)])
    return wg, wu, wd


def test_moe_one_hot_equals_single_ffn():
    e, d_model, d_ff = 4, 256, 256
    wg, wu, wd = _expert_weights(29, e, d_model, d_ff)
    x = synth.normal_f32(29, 100, (3, d_model))
    logits = np.full((3, e), -5.0)
    chosen = [2, 0, 3]
    for t, c in enumerate(chosen):
        logits[t, c] = 5.0
    y, tol, idx, p = oracle.moe_ffn(wg, wu, wd, x, logits, 1)
    for t, c in enumerate(chosen):
        ye, te, _ = oracle.swiglu_ffn(wg[c], wu[c], wd[c], x[t:t + 1])
        assert np.array_equal(y[t], ye[0])
        assert np.all(tol[t] >= te[0])


def test_moe_identical_experts_equal_one_ffn():
    e, d_model, d_ff = 6, 256, 256
    wg, wu, wd = _expert_weights(30, 1, d_model, d_ff)
    wg, wu, wd = (np.repeat(a, e, axis=0) for a in (wg, wu, wd))
    x = synth.normal_f32(30, 100, (2, d_model))
    logits = synth.normal_f32(30, 101, (2, e))
    y, tol, idx, p = oracle.moe_ffn(wg, wu, wd, x, logits, 3)
    ye, te, _ = oracle.swiglu_ffn(wg[0], wu[0], wd[0], x)
    assert np.allclose(y, ye, rtol=1e-13, atol=1e-13 * np.abs(ye).max())


# ---------------------------------------------------------------- prefill GEMM

def test_prefill_bf16_exact_when_operands_are_bf16():
    # Q8_0 with d = 1.0: w = q, |q| <= 127 has 7 bits, exact in bf16
    n, k = 6, 256
    blob = synth.q8_0_blocks(31, 0, n, k).reshape(n, k // 32, 34).copy()
    blob[..., 0] = 0x00
    blob[..., 1] = 0x3C
    w = oracle.q8_0_dequant(blob.reshape(n, -1), n, k)
    x = oracle.round_to_bf16(synth.normal_f32(31, 1, (4, k))).astype(np.float32)
    y, s, yb, sb = oracle.prefill_gemm(w, x)
    assert np.array_equal(y, yb) and np.array_equal(s, sb)


def test_prefill_bf16_brute_force():
    n, k = 3, 256
    blob = synth.q4_k_blocks(32, 0, n, k)
    w = oracle.q4_k_dequant(blob, n, k)
    x = synth.normal_f32(32, 1, (2, k))
    _, _, yb, _ = oracle.prefill_gemm(w, x)
    for t in range(2):
        for r in range(n):
            exact = sum(Fraction(float(oracle.round_to_bf16(w[r, i]))) * Fraction(float(oracle.round_to_bf16(x[t, i])))
                        for i in range(k))
            assert abs(Fraction(float(yb[t, r])) - exact) <= Fraction(1, 10 ** 12) * (1 + abs(exact))


def test_prefill_bf16_changes_operands():
    # bf16 rounding must actually apply to both operands
    w = np.array([[1.0 + 2.0 ** -10]], dtype=np.float32)
    x = np.array([[1.0 + 2.0 ** -9]], dtype=np.float32)
    y, s, yb, sb = oracle.prefill_gemm(w, x)
    assert y[0, 0] == (1.0 + 2.0 ** -10) * (1.0 + 2.0 ** -9)
    assert yb[0, 0] == 1.0


# ---------------------------------------------------------------- decode layer

def test_rmsnorm_closed_forms():
    c = 3.0
    h = oracle.rmsnorm(np.full((1, 64), c))
    assert np.allclose(h, c / math.sqrt(c * c + oracle.RMS_EPS), rtol=1e-15)
    x = synth.normal_f32(33, 0, (2, 2048)).astype(np.float64)
    h = oracle.rmsnorm(x)
    assert np.allclose(np.mean(h * h, axis=1), 1.0 / (1.0 + oracle.RMS_EPS / np.mean(x * x, axis=1)), rtol=1e-13)
    # scale invariant up to the eps term: relative change <= eps / (2 mean x^2)
    assert np.allclose(oracle.rmsnorm(5.0 * x), oracle.rmsnorm(x), rtol=1e-6, atol=0)


def test_attention_pos0_head_mapping():
    nq, nkv, hd = 16, 4, 128
    qkv = np.zeros((1, (nq + 2 * nkv) * hd))
    v0 = (nq + nkv) * hd
    for g in range(nkv):
        qkv[0, v0 + g * hd:v0 + (g + 1) * hd] = 1000 * (g + 1) + np.arange(hd)
    qkv[0, :v0] = -1.0          # Q and K must not leak into the output
    a = oracle.attention_pos0(qkv, nq, nkv, hd)
    for h in range(nq):
        assert np.array_equal(a[0, h * hd:(h + 1) * hd], 1000 * (h // 4 + 1) + np.arange(hd))


def _tiny_layer_weights(seed, d, nq, nkv, hd, dff):
    wqkv = oracle.q8_0_dequant(synth.q8_0_blocks(seed, 0, (nq + 2 * nkv) * hd, d), (nq + 2 * nkv) * hd, d)
    wo = oracle.q8_0_dequant(synth.q8_0_blocks(seed, 1, d, nq * hd), d, nq * hd)
    wg = oracle.q8_0_dequant(synth.q8_0_blocks(seed, 2, dff, d), dff, d)
    wu = oracle.q8_0_dequant(synth.q8_0_blocks(seed, 3, dff, d), dff, d)
    wd = oracle.q8_0_dequant(synth.q8_0_blocks(seed, 4, d, dff), d, dff)
    return wqkv, wo, wg, wu, wd


def test_decode_layer_zero_weights_is_identity():
    d, nq, nkv, hd, dff = 64, 4, 2, 16, 96
    ws = [np.zeros_like(w) for w in _tiny_layer_weights(34, d, nq, nkv, hd, dff)]
    x = synth.normal_f32(34, 9, (1, d))
    x2, dx2 = oracle.decode_layer(x, np.zeros_like(x, dtype=np.float64), *ws, nq, nkv, hd)
    assert np.array_equal(x2, x.astype(np.float64))


def test_decode_layer_brute_force_python():
    d, nq, nkv, hd, dff = 64, 4, 2, 16, 96
    wqkv, wo, wg, wu, wd = _tiny_layer_weights(35, d, nq, nkv, hd, dff)
    x = synth.normal_f32(35, 9, (1, d))
    x2, dx2 = oracle.decode_layer(x, np.zeros((1, d)), wqkv, wo, wg, wu, wd, nq, nkv, hd)
    xs = [float(v) for v in x[0]]

    def norm(v):
        r = 1.0 / math.sqrt(math.fsum(t * t for t in v) / len(v) + 1e-6)
        return [t * r for t in v]

    def mv(w, v):
        return [math.fsum(float(w[i, j]) * v[j] for j in range(len(v))) for i in range(w.shape[0])]

    h = norm(xs)
    qkv = mv(wqkv, h)
    v_base = (nq + nkv) * hd
    attn = []
    for head in range(nq):
        g = head // (nq // nkv)
        attn += qkv[v_base + g * hd:v_base + (g + 1) * hd]
    x1 = [a + b for a, b in zip(xs, mv(wo, attn))]
    h2 = norm(x1)
    gg, uu = mv(wg, h2), mv(wu, h2)
    act = [gv / (1 + math.exp(-gv)) * uv for gv, uv in zip(gg, uu)]
    want = [a + b for a, b in zip(x1, mv(wd, act))]
    assert np.allclose(x2[0], want, rtol=1e-12, atol=1e-12)
    assert np.all(dx2 > 0)


# ---------------------------------------------------------------- decode attention at context depth

def _attn_inputs(seed, length, n_q, n_kv, hd):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((n_q, hd)).astype(np.float32)
    k = rng.standard_normal((length, n_kv, hd)).astype(np.float16)
    v = rng.standard_normal((length, n_kv, hd)).astype(np.float16)
    return q, k, v


def test_attention_single_position_returns_v_exactly():
    # one key: the softmax weight is exactly 1, so every query head returns its KV head's V
    q, k, v = _attn_inputs(1, 1, 8, 2, 16)
    out, tol = oracle.attention_decode(q, k, v, 8, 2, 16)
    for h in range(8):
        assert np.array_equal(out[h], v[0, h // 4].astype(np.float64))
    assert np.all(tol >= 0)


def test_attention_equal_keys_average_the_values():
    # identical keys (or a zero query): uniform weights, the plain mean of V
    q, k, v = _attn_inputs(2, 37, 4, 4, 8)
    k[:] = k[0]
    out, _ = oracle.attention_decode(q, k, v, 4, 4, 8)
    assert np.allclose(out, v.astype(np.float64).mean(axis=0), rtol=1e-13, atol=1e-15)
    out0, _ = oracle.attention_decode(np.zeros_like(q), *_attn_inputs(3, 37, 4, 4, 8)[1:], 4, 4, 8)
    v3 = _attn_inputs(3, 37, 4, 4, 8)[2].astype(np.float64)
    assert np.allclose(out0, v3.mean(axis=0), rtol=1e-13, atol=1e-15)


def test_attention_dominant_key_selects_its_value():
    q, k, v = _attn_inputs(4, 50, 2, 1, 8)
    k[17, 0] = (40.0 * q[0]).astype(np.float16)  # score ~ 40 * |q|^2 / sqrt(8) dominates for head 0
    out, _ = oracle.attention_decode(q, k, v, 2, 1, 8)
    assert np.allclose(out[0], v[17, 0].astype(np.float64), rtol=0, atol=1e-12)


def test_attention_matches_pure_python_brute_force():
    q, k, v = _attn_inputs(5, 5, 4, 2, 3)
    out, _ = oracle.attention_decode(q, k, v, 4, 2, 3, scale=0.7)
    for h in range(4):
        kv = h // 2
        s = [0.7 * sum(float(q[h, d]) * float(k[j, kv, d]) for d in range(3)) for j in range(5)]
        m = max(s)
        e = [math.exp(x - m) for x in s]
        z = sum(e)
        for d in range(3):
            want = sum(e[j] / z * float(v[j, kv, d]) for j in range(5))
            assert abs(out[h, d] - want) <= 1e-14 * max(1.0, abs(want))


def test_attention_invariances():
    q, k, v = _attn_inputs(6, 33, 4, 2, 8)
    out, _ = oracle.attention_decode(q, k, v, 4, 2, 8)
    # scaling the query and dividing the scale by the same factor changes nothing
    out2, _ = oracle.attention_decode(2.0 * q, k, v, 4, 2, 8, scale=0.5 / math.sqrt(8))
    assert np.allclose(out, out2, rtol=1e-12, atol=1e-14)
    # permuting the cached positions changes nothing
    perm = np.random.default_rng(7).permutation(33)
    out3, _ = oracle.attention_decode(q, k[perm], v[perm], 4, 2, 8)
    assert np.allclose(out, out3, rtol=1e-12, atol=1e-14)
    # grouped heads: changing KV head 1 leaves query heads 0 and 1 alone
    k4, v4 = k.copy(), v.copy()
    k4[:, 1] = 0
    v4[:, 1] = 1
    out4, _ = oracle.attention_decode(q, k4, v4, 4, 2, 8)
    assert np.array_equal(out[:2], out4[:2])
    assert np.allclose(out4[2:], 1.0)
