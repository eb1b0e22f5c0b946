"""GPU checks of the MoE FFN with tiered experts (phb_moe_ffn_tiered).

Experts live in a device cache or in pinned host memory the GPU reads; the
call must give the same bits as phb_moe_ffn with every expert resident, since
the same kernels run the same arithmetic on the same weights. The
all-resident call is itself checked against the oracle in
test_gpu_ffn_moe_decode.py; here it is checked again, stage by stage, at the
workload shape.
"""

import numpy as np
import pytest
import torch

import oracle
import quantized_decode_gguf_gb300 as phb
import synth
from _helpers import assert_stages, check_device_clean, ensure_built, moe_intermediates, to_dev, to_host

pytestmark = pytest.mark.gpu

E, K, D_MODEL, D_FF = 128, 8, 2048, 768


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


@pytest.fixture(scope="module")
def experts():
    seed = synth.workload_seed(3)
    rb_in, rb_ff = synth.row_bytes("q4_k", D_MODEL), synth.row_bytes("q4_k", D_FF)
    gu = synth.q4_k_blocks(seed, 7000, 2 * E * D_FF, D_MODEL).reshape(2, E, D_FF, rb_in)
    dn = synth.q4_k_blocks(seed, 7001, E * D_MODEL, D_FF).reshape(E, D_MODEL, rb_ff)
    return np.ascontiguousarray(gu[0]), np.ascontiguousarray(gu[1]), dn


def _split(experts, resident):
    """Device cache (slot order), pinned host copy (host order) and the location table."""
    wg, wu, wd = experts
    resident = sorted(resident)
    host = [e for e in range(E) if e not in set(resident)]
    loc = np.empty(E, dtype=np.int32)
    for s, e in enumerate(resident):
        loc[e] = s
    for h, e in enumerate(host):
        loc[e] = -1 - h
    dev = tuple(to_dev(m[resident]) for m in (wg, wu, wd)) if resident else (None, None, None)
    hst = tuple(torch.from_numpy(np.ascontiguousarray(m[host])).pin_memory() for m in (wg, wu, wd)) if host \
        else (None, None, None)
    return dev, hst, to_dev(loc)


def _resident_call(experts, x, logits, t):
    wg, wu, wd = (to_dev(m) for m in experts)
    idx = torch.empty((t, K), dtype=torch.int32, device="cuda")
    p = torch.empty((t, K), dtype=torch.float32, device="cuda")
    ws = phb.moe_workspace("q4_k", t, D_MODEL, D_FF, E, K)
    y = phb.moe_ffn("q4_k", wg, wu, wd, to_dev(x), to_dev(logits), D_MODEL, D_FF, E, K, out_idx=idx, out_p=p, ws=ws)
    return to_host(y), to_host(idx), to_host(p), ws


@pytest.mark.parametrize("t,fraction", [(1, 0.5), (16, 0.5), (5, 0.25), (1, 0.0), (16, 1.0)])
def test_tiered_equals_all_resident(experts, t, fraction):
    rng = np.random.default_rng(int(100 * fraction) + t)
    resident = rng.permutation(E)[:int(round(fraction * E))].tolist()
    x = synth.normal_f32(synth.workload_seed(3), 7100 + t, (t, D_MODEL))
    logits = synth.normal_f32(synth.workload_seed(3), 7200 + t, (t, E))
    y0, idx0, p0, ws0 = _resident_call(experts, x, logits, t)
    dev, hst, loc = _split(experts, resident)
    idx = torch.empty((t, K), dtype=torch.int32, device="cuda")
    p = torch.empty((t, K), dtype=torch.float32, device="cuda")
    ws = phb.moe_tiered_workspace("q4_k", t, D_MODEL, D_FF, E, K)
    for rep in range(2):  # a second call through the same workspace gives the same bits
        y = to_host(phb.moe_ffn_tiered("q4_k", *dev, *hst, loc, to_dev(x), to_dev(logits), D_MODEL, D_FF, E, K,
                                       ws=ws, out_idx=idx, out_p=p))
        assert np.array_equal(to_host(idx), idx0), rep
        assert np.array_equal(to_host(p), p0), rep
        assert np.array_equal(y, y0), rep
    # the documented workspace prefix holds the same per-pair intermediates
    h_t, yp_t = moe_intermediates(ws, t, K, D_MODEL, D_FF)
    h_0, yp_0 = moe_intermediates(ws0, t, K, D_MODEL, D_FF)
    assert np.array_equal(h_t, h_0) and np.array_equal(yp_t, yp_0)
    check_device_clean()


def test_tiered_stages_against_the_oracle(experts):
    # one token, half the experts in host memory: every stage within its bound
    t = 1
    resident = list(range(0, E, 2))
    x = synth.normal_f32(synth.workload_seed(3), 7300, (t, D_MODEL))
    logits = synth.normal_f32(synth.workload_seed(3), 7301, (t, E))
    dev, hst, loc = _split(experts, resident)
    ws = phb.moe_tiered_workspace("q4_k", t, D_MODEL, D_FF, E, K)
    y = to_host(phb.moe_ffn_tiered("q4_k", *dev, *hst, loc, to_dev(x), to_dev(logits), D_MODEL, D_FF, E, K, ws=ws))
    ridx, _ = oracle.moe_route(logits, K)
    used = sorted(set(ridx.ravel().tolist()))
    wg, wu, wd = experts
    mg = {i: oracle.dequant("q4_k", wg[i], D_FF, D_MODEL) for i in used}
    mu = {i: oracle.dequant("q4_k", wu[i], D_FF, D_MODEL) for i in used}
    md = {i: oracle.dequant("q4_k", wd[i], D_MODEL, D_FF) for i in used}
    h_dev, yp_dev = moe_intermediates(ws, t, K, D_MODEL, D_FF)
    _, _, hs, yps, comb = oracle.moe_stages(mg, mu, md, x, logits, K, h_dev, yp_dev)
    assert_stages({"h": hs, "y_pair": yps, "y": comb}, {"h": h_dev, "y_pair": yp_dev, "y": y}, "tiered moe")
    check_device_clean()


def test_tiered_location_outside_both_copies_is_reported(experts):
    # host indices past the end of the host copy: the fetch reads nothing and the device error says so
    t = 1
    wg, wu, wd = experts
    host = tuple(torch.from_numpy(np.ascontiguousarray(m[:4])).pin_memory() for m in (wg, wu, wd))
    loc = to_dev(np.full(E, -1 - 1000, dtype=np.int32))
    x = to_dev(synth.normal_f32(synth.workload_seed(3), 7400, (t, D_MODEL)))
    logits = to_dev(synth.normal_f32(synth.workload_seed(3), 7401, (t, E)))
    phb.moe_ffn_tiered("q4_k", None, None, None, *host, loc, x, logits, D_MODEL, D_FF, E, K)
    assert phb.device_error() == 2  # a location outside both copies
    assert phb.device_error() == 0  # read and cleared
