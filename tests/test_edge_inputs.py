"""The edge-case matrices are what their names say (checked through the oracle's unpacking)."""

import numpy as np
import pytest

import oracle
from _edge import Q4_KINDS, Q8_KINDS, ZERO_ROW_KINDS, edge, q4_k_edge, q8_0_edge


@pytest.mark.parametrize("qtype,n,k", [("q8_0", 64, 1024), ("q4_k", 64, 1024)])
def test_zero_kinds_dequantise_to_zero_and_others_do_not(qtype, n, k):
    blob, kinds = edge(qtype, 7, n, k)
    w = oracle.dequant(qtype, blob, n, k)
    for r, kind in enumerate(kinds):
        nz = np.count_nonzero(w[r])
        if kind in ZERO_ROW_KINDS:
            assert nz == 0, (kind, nz)
        elif kind == "single_nonzero":
            assert nz == 1, (kind, nz)
        else:
            assert nz > 0, kind


def test_q8_0_quant_fields():
    n, k = 32, 512
    blob, kinds = q8_0_edge(8, n, k)
    d, q = oracle.q8_0_unpack(blob, n, k)
    rows = {kind: [r for r in range(n) if kinds[r] == kind] for kind in Q8_KINDS}
    assert np.all(q[rows["zero_quants"]] == 0) and np.all(d[rows["zero_quants"]] != 0)
    assert np.all(q[rows["minus_128"]] == -128)
    assert np.all(q[rows["minus_128_mixed"]][:, 0::2] == -128)
    assert set(np.unique(q[rows["unit_quants"]])) == {-1, 0, 1}
    assert np.all(q[rows["zero_blocks_mixed"]][:, 1::2] == 0)
    assert np.all(d[rows["zero_scale"]][:, 0::3] == 0)


def test_q4_k_scale_and_min_fields():
    n, k = 32, 512
    blob, kinds = q4_k_edge(9, n, k)
    d, dmin, sc, m, q = oracle.q4_k_unpack(blob, n, k)
    rows = {kind: [r for r in range(n) if kinds[r] == kind] for kind in Q4_KINDS}
    c = rows["cancel_exact"]
    # 0x11 scale bytes: sc_j == m_j (17 for j < 4, 1 for j >= 4); dmin == d; all quants 1
    assert np.all(sc[c] == m[c]) and np.all(sc[c][..., :4] == 17) and np.all(sc[c][..., 4:] == 1)
    assert np.all(d[c] == dmin[c]) and np.all(q[c] == 1)
    z = rows["zero_scale_min_nonzero"]
    assert np.all(sc[z] == 0) and np.all(m[z] >= 1)
    assert np.all(sc[rows["zero_scale_min"]] == 0) and np.all(m[rows["zero_scale_min"]] == 0)
    mx = rows["max_fields"]
    assert np.all(sc[mx] == 63) and np.all(m[mx] == 63) and np.all(q[mx] == 15)
    nc = rows["near_cancel"]
    assert set(np.unique(q[nc])) == {0, 1, 2}
