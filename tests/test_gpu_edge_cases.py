"""GPU parity on the degenerate inputs of the two block formats.

Every matrix mixes, row by row, the edge cases of its format (tests/_edge.py):
zero quants under a nonzero scale, the int8 value -128, quants in {-1, 0, 1},
zero scales, Q4_K sub-blocks whose scale term cancels the min term exactly,
zero 6-bit scales with a nonzero min, and rows that mix such blocks with
ordinary ones. The contract is the unchanged |err| <= 1e-3 * sum|w x| per
output element, which demands y == 0 exactly wherever sum|w x| == 0. The
composed steps are checked stage by stage from the intermediates the GPU
used (the bounds of a stage are zero exactly where every term feeding an
output is zero), and against the end-to-end bounds as well.
"""

import numpy as np
import pytest
import torch

import oracle
import quantized_decode_gguf_gb300 as phb
import synth
from _edge import edge
from _helpers import (assert_stages, assert_within, check_device_clean, ensure_built, ffn_hidden, moe_intermediates,
                      to_dev, to_host)
from test_gpu_ffn_moe_decode import check_decode_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


GEMV_SHAPES = [("q8_0", 2048, 5632), ("q8_0", 3072, 2048), ("q8_0", 1024, 1024), ("q8_0", 40, 2048 + 32),
               ("q4_k", 9728, 2560), ("q4_k", 2560, 9728), ("q4_k", 333, 1280)]


@pytest.mark.parametrize("batch", [1, 2, 4, 8])
@pytest.mark.parametrize("qtype,n,k", GEMV_SHAPES)
def test_gemv_edge_rows(qtype, n, k, batch):
    blob, _ = edge(qtype, 700 + batch, n, k)
    x = synth.normal_f32(700 + batch, 1, (batch, k))
    y = to_host(phb.gemv(qtype, to_dev(blob), to_dev(x), n, k))
    ref, s = oracle.gemv_quant(qtype, blob, x, n, k)
    zero = s == 0
    assert zero.any(), "the edge matrix has rows of zero weights"
    assert np.all(y[zero] == 0.0), "rows whose terms are all zero must give exactly 0"
    assert_within(y, ref, 1e-3 * s, f"edge gemv {qtype} {n}x{k} b{batch}")
    check_device_clean()


@pytest.mark.parametrize("qtype", ["q8_0", "q4_k"])
def test_gemv_single_nonzero_weight_is_exact(qtype):
    # rows with one nonzero weight and x = 1: y is that weight, with no rounding at all
    n, k = 512, 2560 if qtype == "q4_k" else 2048
    blob, kinds = edge(qtype, 710, n, k)
    x = np.ones((1, k), dtype=np.float32)
    y = to_host(phb.gemv(qtype, to_dev(blob), to_dev(x), n, k))[0]
    w = oracle.dequant(qtype, blob, n, k)
    rows = [r for r in range(n) if kinds[r] == "single_nonzero"]
    assert np.array_equal(y[rows], w[rows].sum(axis=1, dtype=np.float64).astype(np.float32))


FFN_SHAPES = [("q8_0", 2048, 5632), ("q4_k", 2048, 768), ("q4_k", 2560, 9728)]


@pytest.mark.parametrize("batch", [1, 4])
@pytest.mark.parametrize("qtype,d_model,d_ff", FFN_SHAPES)
def test_ffn_swiglu_edge_matrices(qtype, d_model, d_ff, batch):
    seed = 720 + batch
    wg, _ = edge(qtype, seed, d_ff, d_model)
    wu, _ = edge(qtype, seed + 10, d_ff, d_model)
    wd, _ = edge(qtype, seed + 20, d_model, d_ff)
    x = synth.normal_f32(seed, 3, (batch, d_model))
    ws = phb.workspace(phb.ffn_workspace_size(qtype, d_model, d_ff, batch))
    y = to_host(phb.ffn_swiglu(qtype, to_dev(wg), to_dev(wu), to_dev(wd), to_dev(x), d_model, d_ff, ws=ws))
    mats = (oracle.dequant(qtype, wg, d_ff, d_model), oracle.dequant(qtype, wu, d_ff, d_model),
            oracle.dequant(qtype, wd, d_model, d_ff))
    h_dev = ffn_hidden(ws, batch, d_ff)
    (h, dh), (yr, dy) = oracle.swiglu_stages(*mats, x, h_dev)
    assert (dh == 0).any() and (dy == 0).any()
    assert_stages({"h": (h, dh), "y": (yr, dy)}, {"h": h_dev, "y": y}, f"edge ffn {qtype} {d_model}->{d_ff} b{batch}")
    ref, tol, _ = oracle.swiglu_ffn(*mats, x)
    assert_within(y, ref, tol, f"edge ffn {qtype} {d_model}->{d_ff} b{batch} end to end")
    check_device_clean()


@pytest.mark.parametrize("t", [1, 16])
def test_moe_edge_experts(t):
    # 128 experts, top-8, d_model 2048, expert FFN 768, Q4_K. Expert e is built
    # from edge seed e % 8 (the kernels do not care that some experts repeat).
    qtype, e, k, d_model, d_ff = "q4_k", 128, 8, 2048, 768
    base = [tuple(edge(qtype, 740 + 3 * i + j, rows, cols)[0] for j, (rows, cols) in
                  enumerate([(d_ff, d_model), (d_ff, d_model), (d_model, d_ff)])) for i in range(8)]
    wg = np.stack([base[i % 8][0] for i in range(e)])
    wu = np.stack([base[i % 8][1] for i in range(e)])
    wd = np.stack([base[i % 8][2] for i in range(e)])
    x = synth.normal_f32(741, t, (t, d_model))
    logits = synth.normal_f32(742, t, (t, e))
    idx = torch.empty((t, k), dtype=torch.int32, device="cuda")
    p = torch.empty((t, k), dtype=torch.float32, device="cuda")
    ws = phb.moe_workspace(qtype, t, d_model, d_ff, e, k)
    y = to_host(phb.moe_ffn(qtype, to_dev(wg), to_dev(wu), to_dev(wd), to_dev(x), to_dev(logits), d_model, d_ff, e,
                            k, out_idx=idx, out_p=p, ws=ws))
    ridx, _ = oracle.moe_route(logits, k)
    assert np.array_equal(to_host(idx), ridx)
    deq = [tuple(oracle.dequant(qtype, m, r, c) for m, (r, c) in
                 zip(base[i], [(d_ff, d_model), (d_ff, d_model), (d_model, d_ff)])) for i in range(8)]
    used = sorted(set(ridx.ravel().tolist()))
    mg, mu, md = ({i: deq[i % 8][j] for i in used} for j in range(3))
    h_dev, yp_dev = moe_intermediates(ws, t, k, d_model, d_ff)
    _, _, hs, yps, comb = oracle.moe_stages(mg, mu, md, x, logits, k, h_dev, yp_dev)
    assert (yps[1] == 0).any()
    assert_stages({"h": hs, "y_pair": yps, "y": comb}, {"h": h_dev, "y_pair": yp_dev, "y": y}, f"edge moe T={t}")
    ref, tol, _, _ = oracle.moe_ffn(mg, mu, md, x, logits, k)
    assert (tol == 0).any()
    assert_within(y, ref, tol, f"edge moe T={t} end to end")
    check_device_clean()


D_MODEL, N_Q, N_KV, HD, D_FF = 2048, 16, 4, 128, 5632
QKV = (N_Q + 2 * N_KV) * HD


@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("qtype", ["q8_0", "q4_k"])
def test_decode_layer_edge_matrices(qtype, fused):
    shapes = [(QKV, D_MODEL), (D_MODEL, N_Q * HD), (D_FF, D_MODEL), (D_FF, D_MODEL), (D_MODEL, D_FF)]
    blobs = [edge(qtype, 760 + i, r, c)[0] for i, (r, c) in enumerate(shapes)]
    table = phb.layer_table([[to_dev(b) for b in blobs]])
    x = synth.normal_f32(760, 99, (D_MODEL,))
    mats = [oracle.dequant(qtype, b, r, c) for b, (r, c) in zip(blobs, shapes)]
    check_decode_layer(qtype, table, mats, x, fused, f"edge decode layer {qtype} fused={fused}")
    check_device_clean()
