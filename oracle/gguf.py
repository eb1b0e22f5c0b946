"""CPU oracle: plain, slow, float64 restatement of the GGUF dequant-multiply path.

TEST INFRASTRUCTURE. Only the test suite, the package's smoke check and the
benchmark's CPU-baseline leg may import this module. The product path (the
CUDA library and its binding) never calls it and shares no code with it.

Sources. The Phobos README (githubhelp.com, joa/phobos-lang) names the
formats in its "Inference" section (models at Q8_0 and Q4_K_M), says the
engine's host backend is its verification oracle ("Note" under "Inference":
both backends give the same logits), describes the fused decode path checked
against the launched one (the `fuse_check` row of the examples table), the
prompt-processing path (`phobos-bench`, pp<N>) and mixture-of-experts decode
("Phobos" overview; 35B-A3B). The pages print no bit layout, no formula and no
worked example. The closed forms used here are the problem's own statement:

* Q8_0: ``w = d * q`` (32 int8 per fp16 scale);
* Q4_K: ``w = d * sc_j * q - dmin * m_j`` (256-weight super-block, fp16 d and
  dmin, eight 32-weight sub-blocks with 6-bit scale ``sc_j`` and min ``m_j``,
  4-bit quants);
* GEMV / GEMM: ``y = sum_k w[n, k] * x[k]``;
* SwiGLU: ``h = silu(W_gate x) * (W_up x)``, ``silu(g) = g / (1 + exp(-g))``,
  ``y = W_down h``;
* top-k routed MoE: ``y_t = sum_k p_{t,k} FFN_{e_{t,k}}(x_t)`` with ``p`` the
  softmax over the top-k router logits.

Readings where the pages are silent (each is listed in the design notes):

* Byte layouts follow the public GGUF convention so that files the pages'
  engine loads would interoperate: Q8_0 = {fp16 d; int8 q[32]}; Q4_K = {fp16 d;
  fp16 dmin; u8 scales[12]; u8 qs[128]} with the k-quant 6-bit packing.
* Weight matrices are row-major with N output rows of K/32 (or K/256)
  consecutive blocks; activations are [batch][K].
* Top-k ties go to the lower expert index.
* Prefill: weights and activations are rounded to bf16 (round to nearest
  even) and multiplied exactly, accumulated in fp32.
* Decode layer: RMSNorm without gain, eps = 1e-6; position 0, so attention
  returns V, query head h reads KV head h // (n_q / n_kv); residual adds.
* Decode attention at context depth: fp16 KV cache [L][n_kv][head_dim], fp32
  query and output, scaled dot-product softmax with scale 1/sqrt(head_dim).

Exactness arguments used for bit-exact dequantisation:

* every fp16 value is an integer multiple of 2**-24 with magnitude < 2**16;
* Q8_0: ``d*q`` has at most 11 + 7 significant bits, so it is exact in fp32
  and in float64;
* Q4_K: ``d*sc*q`` and ``dmin*m`` are integer multiples of 2**-24 below 2**26,
  so their difference is an integer multiple of 2**-24 below 2**27 (51 bits):
  exact in float64. Rounding that exact value once to fp32 is the single
  rounding that any fp32 evaluation order ``(d*sc)*q - dmin*m`` performs, since
  ``d*sc``, ``dmin*m`` and ``(d*sc)*q`` are each exact in fp32.
"""

from __future__ import annotations

import numpy as np

QK8_0 = 32
Q8_0_BYTES = 34
QK_K = 256
Q4_K_BYTES = 144
RMS_EPS = 1e-6


# ----------------------------------------------------------------------------
# fp16 / bf16 helpers
# ----------------------------------------------------------------------------

def fp16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """IEEE binary16 bit patterns (uint16) -> exact float64 values."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 with round-to-nearest-even, returned as float64.

    Written from the definition: keep the top 16 bits of the fp32 pattern,
    adding half an ulp of the kept part plus the kept part's lowest bit
    (ties to even). NaN stays NaN.
    """
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16) << 16
    out = r.astype(np.uint32).view(np.float32).astype(np.float64)
    return np.where(np.isnan(f), np.nan, out)


# ----------------------------------------------------------------------------
# Q8_0
# ----------------------------------------------------------------------------

def q8_0_unpack(blocks: np.ndarray, n_rows: int, k: int):
    """Split a Q8_0 matrix into its fields.

    Returns (d [n, k/32] float64, q [n, k/32, 32] int64).
    """
    nb = k // QK8_0
    b = np.asarray(blocks, dtype=np.uint8).reshape(n_rows, nb, Q8_0_BYTES)
    d_bits = b[..., 0].astype(np.uint16) | (b[..., 1].astype(np.uint16) << 8)
    d = fp16_bits_to_f64(d_bits)
    q = b[..., 2:].view(np.int8).astype(np.int64)
    return d, q


def q8_0_dequant_f64(blocks: np.ndarray, n_rows: int, k: int) -> np.ndarray:
    """Exact weights w = d * q, float64 [n_rows, k]."""
    d, q = q8_0_unpack(blocks, n_rows, k)
    return (d[..., None] * q).reshape(n_rows, k)


def q8_0_dequant(blocks: np.ndarray, n_rows: int, k: int) -> np.ndarray:
    """fp32 dequantised weights (exact: 18 significant bits at most)."""
    return q8_0_dequant_f64(blocks, n_rows, k).astype(np.float32)


# ----------------------------------------------------------------------------
# Q4_K
# ----------------------------------------------------------------------------

def q4_k_unpack(blocks: np.ndarray, n_rows: int, k: int):
    """Split a Q4_K matrix into its fields.

    Returns (d [n, nb], dmin [n, nb] float64; sc [n, nb, 8], m [n, nb, 8],
    q [n, nb, 256] int64), nb = k/256, with q indexed by the weight's position
    in the super-block.

    Field layout (GGUF k-quant convention): bytes 0-1 d, 2-3 dmin, 4-15 the
    twelve scale bytes s[0..11], 16-143 the quant bytes qs[0..127].
    Sub-block j < 4: sc = s[j] & 63, m = s[j+4] & 63.
    Sub-block j >= 4: sc = (s[j+4] & 15) | (s[j-4] >> 6) << 4,
                      m  = (s[j+4] >> 4) | (s[j]   >> 6) << 4.
    Quant byte qs[32c + i] (c = 0..3, i = 0..31) holds weight 64c + i in its
    low nibble and weight 64c + 32 + i in its high nibble.
    """
    nb = k // QK_K
    b = np.asarray(blocks, dtype=np.uint8).reshape(n_rows, nb, Q4_K_BYTES).astype(np.int64)
    d = fp16_bits_to_f64((b[..., 0] | (b[..., 1] << 8)).astype(np.uint16))
    dmin = fp16_bits_to_f64((b[..., 2] | (b[..., 3] << 8)).astype(np.uint16))
    s = b[..., 4:16]
    sc = np.empty(s.shape[:-1] + (8,), dtype=np.int64)
    m = np.empty_like(sc)
    for j in range(4):
        sc[..., j] = s[..., j] & 63
        m[..., j] = s[..., j + 4] & 63
    for j in range(4, 8):
        sc[..., j] = (s[..., j + 4] & 15) | ((s[..., j - 4] >> 6) << 4)
        m[..., j] = (s[..., j + 4] >> 4) | ((s[..., j] >> 6) << 4)
    qs = b[..., 16:144]
    q = np.empty(b.shape[:-1] + (QK_K,), dtype=np.int64)
    for c in range(4):
        chunk = qs[..., 32 * c:32 * c + 32]
        q[..., 64 * c:64 * c + 32] = chunk & 15
        q[..., 64 * c + 32:64 * c + 64] = chunk >> 4
    return d, dmin, sc, m, q


def q4_k_dequant_f64(blocks: np.ndarray, n_rows: int, k: int) -> np.ndarray:
    """Exact real value of d*sc*q - dmin*m for every weight, float64 [n, k]."""
    d, dmin, sc, m, q = q4_k_unpack(blocks, n_rows, k)
    nb = k // QK_K
    sub = np.arange(QK_K) // 32                       # sub-block of each weight
    scale = (d[..., None] * sc)[..., sub]             # d*sc_j per weight, exact
    offset = (dmin[..., None] * m)[..., sub]          # dmin*m_j per weight, exact
    return (scale * q - offset).reshape(n_rows, nb * QK_K)


def q4_k_dequant(blocks: np.ndarray, n_rows: int, k: int) -> np.ndarray:
    """fp32 dequantised weights: the exact value rounded once (nearest even)."""
    return q4_k_dequant_f64(blocks, n_rows, k).astype(np.float32)


def dequant(qtype: str, blocks: np.ndarray, n_rows: int, k: int) -> np.ndarray:
    """fp32 dequantised matrix for format "q8_0" or "q4_k"."""
    if qtype == "q8_0":
        return q8_0_dequant(blocks, n_rows, k)
    if qtype == "q4_k":
        return q4_k_dequant(blocks, n_rows, k)
    raise ValueError(qtype)


# ----------------------------------------------------------------------------
# GEMV / GEMM
# ----------------------------------------------------------------------------

def gemv(w: np.ndarray, x: np.ndarray):
    """y[b, n] = sum_k w[n, k] x[b, k] in float64, and S[b, n] = sum_k |w x|.

    ``w`` is the fp32 dequantised matrix [N, K]; ``x`` is [B, K] (or [K]).
    The GPU result must satisfy |y_gpu - y| <= 1e-3 * S elementwise.
    """
    w64 = np.asarray(w, dtype=np.float64)
    x64 = np.atleast_2d(np.asarray(x, dtype=np.float64))
    y = x64 @ w64.T
    s = np.abs(x64) @ np.abs(w64).T
    return y, s


def gemv_quant(qtype: str, blocks: np.ndarray, x: np.ndarray, n_rows: int, k: int):
    """GEMV straight from quantized blocks: dequantise, then :func:`gemv`."""
    return gemv(dequant(qtype, blocks, n_rows, k), x)


def prefill_gemm(w: np.ndarray, x: np.ndarray):
    """Prompt-processing GEMM, Y[t, n] = sum_k w[n, k] x[t, k].

    Returns (y_exact, s_exact, y_bf16, s_bf16): the product of the fp32
    weights with the fp32 activations, and the product after rounding both
    operands to bf16 (nearest even), each with its sum of absolute terms.
    """
    y, s = gemv(w, x)
    wb = round_to_bf16(np.asarray(w, dtype=np.float32))
    xb = round_to_bf16(np.asarray(x, dtype=np.float32))
    yb, sb = gemv(wb, xb)
    return y, s, yb, sb


# ----------------------------------------------------------------------------
# SwiGLU FFN
# ----------------------------------------------------------------------------

def silu(g: np.ndarray) -> np.ndarray:
    """g / (1 + exp(-g)) in float64.

    For g below about -709, exp(-g) overflows to inf and the quotient is the
    correct limit -0.0; numpy's overflow warning for that case is silenced.
    """
    g = np.asarray(g, dtype=np.float64)
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g))


SILU_SLOPE_MAX = 1.1  # max |d silu / dg| = 1.0998..., rounded up


def _swiglu_bound(g, dg, u, du, eps: float):
    """h = silu(g) * u and a bound of |h~ - h|.

    Given |g~ - g| <= dg, |u~ - u| <= du and an fp32 evaluation of silu and
    the product with relative error at most ``eps``: by the mean value
    theorem |silu(g~) - silu(g)| <= 1.1 dg, so
        d1 = 1.1 dg (|u| + du) + |silu(g)| du,   dh = d1 + eps (|h| + d1).
    """
    sg = silu(g)
    h = sg * u
    d1 = SILU_SLOPE_MAX * dg * (np.abs(u) + du) + np.abs(sg) * du
    return h, d1 + eps * (np.abs(h) + d1)


def swiglu_ffn(wg: np.ndarray, wu: np.ndarray, wd: np.ndarray, x: np.ndarray, eps: float = 1e-3):
    """SwiGLU feed-forward block and its error bound.

    ``wg``, ``wu``: fp32 [d_ff, d_model]; ``wd``: fp32 [d_model, d_ff]; ``x``:
    [B, d_model]. Returns (y [B, d_model], tol [B, d_model], h [B, d_ff]).

    ``tol`` propagates the per-GEMV contract |err| <= eps * sum|w x| through
    the block: the gate and up outputs g, u carry at most eps * S_g and
    eps * S_u, the activation h = silu(g) u then at most dh (see
    :func:`_swiglu_bound`), and the down projection, whose contract applies
    to the activation it is actually given, at most
        eps * sum_j |wd_ij h_j| + (1 + eps) * sum_j |wd_ij| dh_j.
    This bound is valid but grows with sum_j |wd_ij| / |y_i|; for checking a
    device against it stage by stage see :func:`swiglu_stages`.
    """
    g, sg = gemv(wg, x)
    u, su = gemv(wu, x)
    h, dh = _swiglu_bound(g, eps * sg, u, eps * su, eps)
    y, tol = _gemv_bound(wd, h, dh, eps)
    return y, tol, h


def swiglu_stages(wg: np.ndarray, wu: np.ndarray, wd: np.ndarray, x: np.ndarray, h_dev: np.ndarray,
                  eps: float = 1e-3):
    """The SwiGLU block checked one stage at a time.

    ``h_dev`` is the activation a device computed ([B, d_ff]). Returns
    ((h, h_tol), (y, y_tol)): the activation and its bound from ``x`` (the
    gate/up contract and the elementwise step, as in :func:`swiglu_ffn`), and
    y = wd h_dev with the GEMV contract eps * sum|wd h_dev| for the input the
    device actually used. Each stage is one GEMV deep, so neither bound
    compounds.
    """
    g, sg = gemv(wg, x)
    u, su = gemv(wu, x)
    h, dh = _swiglu_bound(g, eps * sg, u, eps * su, eps)
    y, s = gemv(wd, h_dev)
    return (h, dh), (y, eps * s)


# ----------------------------------------------------------------------------
# Mixture of experts
# ----------------------------------------------------------------------------

def moe_route(logits: np.ndarray, top_k: int):
    """Top-k routing: per token the top_k largest logits, ties to the lower index.

    Returns (idx [T, top_k] int64, in descending logit order; p [T, top_k]
    float64 = softmax of the selected logits).
    """
    lg = np.atleast_2d(np.asarray(logits, dtype=np.float64))
    order = np.argsort(-lg, axis=1, kind="stable")
    idx = order[:, :top_k]
    sel = np.take_along_axis(lg, idx, axis=1)
    e = np.exp(sel - sel.max(axis=1, keepdims=True))
    p = e / e.sum(axis=1, keepdims=True)
    return idx, p


def moe_ffn(wg, wu, wd, x: np.ndarray, logits: np.ndarray,
            top_k: int, eps: float = 1e-3, p_rel_err: float = 1e-5, sum_rel_err: float = 1e-6):
    """Routed expert FFN: y_t = sum_k p_{t,k} FFN_{e_{t,k}}(x_t).

    ``wg``, ``wu``: fp32 [E, d_ff, d_model]; ``wd``: fp32 [E, d_model, d_ff]
    (or any mapping from expert index to that expert's matrix, so that only
    the routed experts need dequantising); ``x``: [T, d_model]; ``logits``:
    [T, E]. Returns (y, tol, idx, p).

    ``tol`` = sum_k p_k (tol_k + c (|FFN_k(x_t)| + tol_k)), c = a + b + a b,
    covering each expert's FFN bound, a relative error of at most
    a = ``p_rel_err`` in each routing weight (fp32 exp and divide) and
    b = ``sum_rel_err`` for the fp32 weighted sum of at most a few dozen
    terms (each applied to the expert output the device actually has).
    """
    x = np.atleast_2d(np.asarray(x, dtype=np.float64))
    idx, p = moe_route(logits, top_k)
    t_count, d_model = x.shape
    y = np.zeros((t_count, d_model))
    tol = np.zeros((t_count, d_model))
    for t in range(t_count):
        for j in range(top_k):
            e = int(idx[t, j])
            ye, te, _ = swiglu_ffn(wg[e], wu[e], wd[e], x[t:t + 1], eps)
            y[t] += p[t, j] * ye[0]
            c = p_rel_err + sum_rel_err + p_rel_err * sum_rel_err
            tol[t] += p[t, j] * (te[0] + c * (np.abs(ye[0]) + te[0]))
    return y, tol, idx, p


def moe_stages(wg, wu, wd, x: np.ndarray, logits: np.ndarray, top_k: int, h_dev: np.ndarray, y_pair_dev: np.ndarray,
               eps: float = 1e-3, p_rel_err: float = 1e-5, sum_rel_err: float = 1e-6):
    """The routed expert FFN checked one stage at a time.

    ``h_dev`` [T * top_k, d_ff] and ``y_pair_dev`` [T * top_k, d_model] are a
    device's per-(token, slot) activations and expert outputs (pair
    t * top_k + k, slots in descending logit order). Returns
    (idx, p, (h, h_tol), (yp, yp_tol), (y, y_tol)):
      * h, h_tol: each pair's activation and bound from x_t (:func:`swiglu_stages`);
      * yp, yp_tol: each pair's down projection of h_dev and its contract;
      * y, y_tol: the combine sum_k p_k y_pair_dev with the routing-weight and
        weighted-sum errors of :func:`moe_ffn`.
    ``wg``, ``wu``, ``wd`` may be mappings from expert index to matrix.
    """
    x = np.atleast_2d(np.asarray(x, dtype=np.float64))
    idx, p = moe_route(logits, top_k)
    t_count = x.shape[0]
    hs, dhs, yps, dyps = [], [], [], []
    for t in range(t_count):
        for j in range(top_k):
            e = int(idx[t, j])
            pair = t * top_k + j
            (h, dh), (yp, dyp) = swiglu_stages(wg[e], wu[e], wd[e], x[t:t + 1], h_dev[pair:pair + 1], eps)
            hs.append(h[0])
            dhs.append(dh[0])
            yps.append(yp[0])
            dyps.append(dyp[0])
    ypd = np.asarray(y_pair_dev, dtype=np.float64).reshape(t_count, top_k, -1)
    y = np.einsum("tk,tkd->td", p, ypd)
    c = p_rel_err + sum_rel_err + p_rel_err * sum_rel_err
    y_tol = c * np.einsum("tk,tkd->td", p, np.abs(ypd))
    return idx, p, (np.array(hs), np.array(dhs)), (np.array(yps), np.array(dyps)), (y, y_tol)


# ----------------------------------------------------------------------------
# Dense decode layer at position 0
# ----------------------------------------------------------------------------

def rmsnorm(x: np.ndarray, eps: float = RMS_EPS) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps), no gain, float64."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)


def attention_pos0(qkv: np.ndarray, n_q_heads: int, n_kv_heads: int, head_dim: int) -> np.ndarray:
    """Attention over a single cached position: every query head returns its KV head's V.

    ``qkv`` is [B, (n_q + 2 n_kv) * head_dim] laid out as Q | K | V. With one
    key the softmax weight is 1, so the output of query head h is V of KV
    head h // (n_q / n_kv) (grouped-query attention). RoPE at position 0 is
    the identity and does not enter.
    """
    qkv = np.atleast_2d(qkv)
    group = n_q_heads // n_kv_heads
    v0 = (n_q_heads + n_kv_heads) * head_dim
    v = qkv[:, v0:v0 + n_kv_heads * head_dim].reshape(qkv.shape[0], n_kv_heads, head_dim)
    heads = [v[:, h // group, :] for h in range(n_q_heads)]
    return np.concatenate(heads, axis=1)


def attention_decode(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray, n_q_heads: int, n_kv_heads: int,
                     head_dim: int, scale: float | None = None):
    """Attention of one decoding token over ``L`` cached positions.

    Phobos README: ``phobos-bench -d N`` runs generation with N tokens
    already in the context; ``phobos-kbench``'s ``flash_fp16`` kernel keeps
    Q/K/V/O in f16 with an f32 online-softmax state; the ``kv_check``
    example checks one decode step using the KV cache against a full
    recompute. Readings: the cache is fp16 (as ``flash_fp16``), the query
    and the output fp32 (as the rest of the decode path), grouped-query
    heads (query head h reads KV head h // (n_q / n_kv)) and the usual
    scaled dot-product softmax, scale = 1 / sqrt(head_dim) by default:

        s_j = scale * q_h . k_j,   p = softmax(s),   out_h = sum_j p_j v_j

    ``q``: [n_q, head_dim]; ``k_cache``, ``v_cache``: [L, n_kv, head_dim]
    (fp16 values are exact in float64). Returns ``(out, tol)`` in float64:
    ``tol`` bounds an fp32 evaluation (scores, exp and the sums in fp32, in
    any order):

        tol = A * (4 * ds + (L + head_dim + 16) * 2^-22),
        A = sum_j p_j |v_j|,   ds = scale * head_dim * 2^-23 * max_j sum_d |q_d k_jd|

    (a first-order bound: a score error ds moves every p_j by at most
    2 p_j ds; each fp32 sum of n terms is within n * 2^-24 of exact).
    """
    qf = np.asarray(q, dtype=np.float64).reshape(n_q_heads, head_dim)
    k = np.asarray(k_cache, dtype=np.float64).reshape(-1, n_kv_heads, head_dim)
    v = np.asarray(v_cache, dtype=np.float64).reshape(-1, n_kv_heads, head_dim)
    length = k.shape[0]
    if scale is None:
        scale = 1.0 / np.sqrt(head_dim)
    group = n_q_heads // n_kv_heads
    out = np.zeros((n_q_heads, head_dim))
    tol = np.zeros((n_q_heads, head_dim))
    for h in range(n_q_heads):
        kv = h // group
        s = scale * (k[:, kv, :] @ qf[h])
        e = np.exp(s - s.max())
        p = e / e.sum()
        out[h] = p @ v[:, kv, :]
        a = p @ np.abs(v[:, kv, :])
        ds = scale * head_dim * 2.0 ** -23 * np.max(np.abs(k[:, kv, :]) @ np.abs(qf[h]))
        tol[h] = a * (4.0 * ds + (length + head_dim + 16) * 2.0 ** -22)
    return out, tol


def _rmsnorm_bound(x: np.ndarray, dx: np.ndarray, eps_norm: float, eps: float = RMS_EPS):
    """Bound of |h~ - rmsnorm(x)| for h~ = x~ r~ (1 + t2), with |x~ - x| <= dx,
    r~ = r(x~) (1 + t1) and |t1|, |t2| <= eps_norm (the fp32 evaluation).

    With m = mean x^2 and r = (m + eps)^-1/2: |mean x~^2 - m| <= dm =
    (2 sum|x| dx + sum dx^2) / n, and |dr/dm| = r^3 / 2 is largest at the
    smallest m, so |r(x~) - r(x)| <= dr_in = dm / 2 (m + eps - dm)^-3/2
    (infinite when dm >= m + eps). Then dr = dr_in + eps_norm (r + dr_in)
    bounds |r~ - r|, and
        |h~ - h| <= (1 + eps_norm) ((r + dr) dx + |x| dr) + eps_norm |h|.
    """
    x = np.asarray(x, dtype=np.float64)
    dx = np.asarray(dx, dtype=np.float64)
    n = x.shape[-1]
    m = np.mean(x * x, axis=-1, keepdims=True)
    r = 1.0 / np.sqrt(m + eps)
    dm = (2.0 * np.sum(np.abs(x) * dx, axis=-1, keepdims=True) + np.sum(dx * dx, axis=-1, keepdims=True)) / n
    lo = m + eps - dm
    with np.errstate(divide="ignore", invalid="ignore"):
        dr_in = np.where(lo > 0, 0.5 * dm * np.abs(lo) ** -1.5, np.inf)
    dr = dr_in + eps_norm * (r + dr_in)
    with np.errstate(invalid="ignore"):
        dh = (1.0 + eps_norm) * ((r + dr) * dx + np.abs(x) * dr) + eps_norm * np.abs(x * r)
    return np.where(np.isfinite(dr), dh, np.inf)


def _abs_matvec(dx: np.ndarray, aw: np.ndarray) -> np.ndarray:
    """dx @ aw.T for nonnegative dx and aw, where an infinite dx_j makes every
    output with a nonzero weight in column j infinite (never NaN)."""
    fin = np.isfinite(dx)
    out = np.where(fin, dx, 0.0) @ aw.T
    hit = (~fin).astype(np.float64) @ (aw.T > 0).astype(np.float64)
    return np.where(hit > 0, np.inf, out)


def _gemv_bound(w: np.ndarray, x: np.ndarray, dx: np.ndarray, eps: float):
    """y = w x and its bound eps * sum|w x| + (1 + eps) sum|w| dx.

    The contract applies to the input the device actually has, x~ with
    |x~ - x| <= dx: |y~ - y| <= eps sum|w x~| + sum|w| dx, and
    sum|w x~| <= sum|w x| + sum|w| dx.
    """
    y, s = gemv(w, x)
    aw = np.abs(np.asarray(w, dtype=np.float64))
    wdx = _abs_matvec(np.asarray(dx, dtype=np.float64), aw)
    return y, eps * s + (1.0 + eps) * wdx


ADD_REL = 1e-7  # >= 2^-24: one fp32 rounding of a residual add, relative to the rounded sum's magnitude


def decode_layer(x: np.ndarray, dx: np.ndarray, w_qkv, w_o, w_gate, w_up, w_down,
                 n_q_heads: int, n_kv_heads: int, head_dim: int,
                 eps: float = 1e-3, eps_norm: float = 1e-5):
    """One pre-norm decoder layer at position 0, with a propagated error bound.

    x1 = x + W_o attn(W_qkv rmsnorm(x)); x2 = x1 + W_down (silu(W_gate h) * (W_up h)),
    h = rmsnorm(x1). All weights fp32 dequantised [out, in]. ``dx`` bounds
    the error already in ``x`` (zeros for an exact input). Returns (x2, dx2).

    The bound chains the per-GEMV contract through four GEMVs with the
    triangle inequality; it is valid, but each GEMV multiplies the incoming
    allowance by its row sums of |w|, so at model sizes it dwarfs the output.
    A device is checked against :func:`decode_layer_stages` instead.
    """
    x = np.atleast_2d(np.asarray(x, dtype=np.float64))
    dx = np.atleast_2d(np.asarray(dx, dtype=np.float64))
    h = rmsnorm(x)
    dh = _rmsnorm_bound(x, dx, eps_norm)
    qkv, dqkv = _gemv_bound(w_qkv, h, dh, eps)
    a = attention_pos0(qkv, n_q_heads, n_kv_heads, head_dim)
    da = attention_pos0(dqkv, n_q_heads, n_kv_heads, head_dim)
    o, do = _gemv_bound(w_o, a, da, eps)
    x1 = x + o
    dx1 = dx + do + ADD_REL * (np.abs(x1) + dx + do)
    h2 = rmsnorm(x1)
    dh2 = _rmsnorm_bound(x1, dx1, eps_norm)
    g, dg = _gemv_bound(w_gate, h2, dh2, eps)
    u, du = _gemv_bound(w_up, h2, dh2, eps)
    act, dact = _swiglu_bound(g, dg, u, du, eps)
    f, df = _gemv_bound(w_down, act, dact, eps)
    x2 = x1 + f
    dx2 = dx1 + df + ADD_REL * (np.abs(x2) + dx1 + df)
    return x2, dx2


def decode_layer_stages(x: np.ndarray, qkv_dev: np.ndarray, x1_dev: np.ndarray, act_dev: np.ndarray,
                        w_qkv, w_o, w_gate, w_up, w_down, n_q_heads: int, n_kv_heads: int, head_dim: int,
                        eps: float = 1e-3, eps_norm: float = 1e-5):
    """One decoder layer checked one stage at a time, from the intermediate
    vectors a device computed (its QKV vector, its x1 = x + W_o attn, its
    SwiGLU activation; each [1, n]).

    Returns {"qkv": (ref, tol), "x1": ..., "act": ..., "out": ...}, each
    stage's reference and bound computed from the device's own input to
    that stage, one GEMV deep:
      qkv: W_qkv rmsnorm(x), with rmsnorm's evaluation error;
      x1:  x + W_o attn(qkv_dev), the contract plus the residual add's rounding;
      act: silu(W_gate h2) * (W_up h2), h2 = rmsnorm(x1_dev) (:func:`_swiglu_bound`);
      out: x1_dev + W_down act_dev, the contract plus the residual add's rounding.
    """
    x = np.atleast_2d(np.asarray(x, dtype=np.float64))
    qkv_dev, x1_dev, act_dev = (np.atleast_2d(np.asarray(v, dtype=np.float64)) for v in (qkv_dev, x1_dev, act_dev))
    out = {}
    h = rmsnorm(x)
    out["qkv"] = _gemv_bound(w_qkv, h, _rmsnorm_bound(x, np.zeros_like(x), eps_norm), eps)
    o, so = gemv(w_o, attention_pos0(qkv_dev, n_q_heads, n_kv_heads, head_dim))
    x1 = x + o
    out["x1"] = (x1, eps * so + ADD_REL * (np.abs(x1) + eps * so))
    h2 = rmsnorm(x1_dev)
    dh2 = _rmsnorm_bound(x1_dev, np.zeros_like(x1_dev), eps_norm)
    g, dg = _gemv_bound(w_gate, h2, dh2, eps)
    u, du = _gemv_bound(w_up, h2, dh2, eps)
    out["act"] = _swiglu_bound(g, dg, u, du, eps)
    f, sf = gemv(w_down, act_dev)
    x2 = x1_dev + f
    out["out"] = (x2, eps * sf + ADD_REL * (np.abs(x2) + eps * sf))
    return out
