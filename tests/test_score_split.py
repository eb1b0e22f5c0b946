"""The query split of the tensor-core attention score path, checked on the host.

For head_dim 64 and 128 the decode-attention kernel feeds the tensor cores
fp16 keys and the query of each head as two fp16 parts: the head's query is
scaled by the power of two 2^e that puts its largest magnitude in
[2^14, 2^15), then hi = fp16(q 2^e) and lo = fp16(q 2^e - hi). This file
restates that split in numpy (round to nearest even, as the kernel's
conversions) and checks the error claim the kernel relies on: per element
|(hi + lo) 2^-e - q| <= 2^-22 |q| + 2^-39 max|q|, so the score error stays
inside the oracle's bound term ds = scale * head_dim * 2^-23 * sum |q k|.
"""

import math

import numpy as np
import pytest

import oracle


def split(q: np.ndarray):
    mx = float(np.max(np.abs(q)))
    e = 15 - math.frexp(mx)[1] if mx > 0 else 0
    qs = np.ldexp(q.astype(np.float32), e).astype(np.float32)
    hi = qs.astype(np.float16)
    lo = (qs - hi.astype(np.float32)).astype(np.float16)
    return hi, lo, e


def rebuilt(q):
    hi, lo, e = split(q)
    return np.ldexp(hi.astype(np.float64) + lo.astype(np.float64), -e)


@pytest.mark.parametrize("magnitude", [1e-30, 1e-6, 1.0, 3.0e4, 1e30])
def test_split_keeps_22_bits_per_element(magnitude):
    rng = np.random.default_rng(7)
    q = (magnitude * rng.standard_normal(4096)).astype(np.float32)
    err = np.abs(rebuilt(q) - q.astype(np.float64))
    bound = 2.0 ** -22 * np.abs(q.astype(np.float64)) + 2.0 ** -39 * np.max(np.abs(q))
    assert np.all(err <= bound)


def test_scaled_largest_element_lands_in_the_top_fp16_binade():
    rng = np.random.default_rng(8)
    for mag in (1e-20, 0.37, 1.0, 2.0, 65504.0, 1e20):
        q = (mag * rng.standard_normal(128)).astype(np.float32)
        hi, _, e = split(q)
        top = np.max(np.abs(np.ldexp(q.astype(np.float64), e)))
        assert 2.0 ** 14 <= top < 2.0 ** 15
        assert np.all(np.isfinite(hi.astype(np.float32)))


def test_zero_query_splits_to_zero():
    hi, lo, e = split(np.zeros(64, dtype=np.float32))
    assert e == 0 and not hi.any() and not lo.any()


def test_score_error_is_inside_the_oracle_bound_term():
    # scores from the split query against fp16 keys, exact products and float64
    # sums, compared with the exact scores; the difference must sit well under ds
    rng = np.random.default_rng(9)
    hd, length = 128, 300
    for q_scale in (1e-3, 1.0, 50.0):
        q = (q_scale * rng.standard_normal((1, hd))).astype(np.float32)
        k = rng.standard_normal((length, 1, hd)).astype(np.float16)
        v = rng.standard_normal((length, 1, hd)).astype(np.float16)
        scale = 1.0 / math.sqrt(hd)
        exact = scale * (k[:, 0, :].astype(np.float64) @ q[0].astype(np.float64))
        split_s = scale * (k[:, 0, :].astype(np.float64) @ rebuilt(q[0]))
        ds = scale * hd * 2.0 ** -23 * np.max(np.abs(k[:, 0, :].astype(np.float64)) @ np.abs(q[0].astype(np.float64)))
        assert np.max(np.abs(split_s - exact)) <= ds / 8
        # the oracle's bound for the same inputs is positive and finite
        _, tol = oracle.attention_decode(q, k, v, 1, 1, hd)
        assert np.all(np.isfinite(tol)) and np.all(tol > 0)
