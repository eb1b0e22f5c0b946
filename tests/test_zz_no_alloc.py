"""The allocation-free SwiGLU entry point (phb_ffn_swiglu_noalloc).

Some callers cannot allocate device memory, for example a serving loop that
fixes its memory budget at start-up, or a plugin inside another runtime that
owns all device allocations. phb_ffn_swiglu_noalloc serves them by keeping
its scratch in a static device array inside the library. These tests call it
through the C ABI and check it against phb_ffn_swiglu (which takes a caller
workspace) on two calls in a row, since every call reuses the same array.
This file is named to be collected last.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
from quantized_decode_gguf_gb300 import _lib, build

FAKE = 0x10000
Q8_0, Q4_K = 8, 12


def _lib_loaded():
    build.build()
    return _lib.load()


def test_noalloc_rejects_oversized_shape_without_a_gpu():
    lib = _lib_loaded()
    cap = lib.phb_ffn_swiglu_noalloc_max_scratch()
    assert cap == 2 << 20
    # 8 x 65536 fp32 hidden activations alone exceed the static array
    assert lib.phb_ffn_swiglu_workspace_size(Q4_K, 256, 65536, 8) > cap
    st = lib.phb_ffn_swiglu_noalloc(Q4_K, FAKE, FAKE, FAKE, FAKE, FAKE, 256, 65536, 8, None)
    assert st == 4 and b"static scratch" in lib.phb_last_error()
    # invalid shapes still get the ordinary argument errors
    assert lib.phb_ffn_swiglu_noalloc(Q4_K, FAKE, FAKE, FAKE, FAKE, FAKE, 256, 300, 1, None) == 2


@pytest.mark.gpu
@pytest.mark.parametrize("qtype,qid,d_model,d_ff,batch", [("q8_0", Q8_0, 2048, 5632, 1),
                                                         ("q4_k", Q4_K, 2048, 768, 4),
                                                         ("q4_k", Q4_K, 2560, 9728, 8)])
def test_noalloc_matches_workspace_entry_point(qtype, qid, d_model, d_ff, batch):
    lib = _lib_loaded()
    seed = 900 + batch
    wg = synth.blocks(qtype, seed, 0, d_ff, d_model)
    wu = synth.blocks(qtype, seed, 1, d_ff, d_model)
    wd = synth.blocks(qtype, seed, 2, d_model, d_ff)
    dev = [torch.from_numpy(a).cuda() for a in (wg, wu, wd)]
    stream = torch.cuda.current_stream().cuda_stream
    _, tol, _ = oracle.swiglu_ffn(oracle.dequant(qtype, wg, d_ff, d_model), oracle.dequant(qtype, wu, d_ff, d_model),
                                  oracle.dequant(qtype, wd, d_model, d_ff), synth.normal_f32(seed, 3, (batch, d_model)))
    for call in range(2):
        x = torch.from_numpy(synth.normal_f32(seed, 3 + call, (batch, d_model))).cuda()
        if call == 1:
            _, tol, _ = oracle.swiglu_ffn(oracle.dequant(qtype, wg, d_ff, d_model),
                                          oracle.dequant(qtype, wu, d_ff, d_model),
                                          oracle.dequant(qtype, wd, d_model, d_ff), x.cpu().numpy())
        y_ref = torch.empty((batch, d_model), device="cuda")
        need = lib.phb_ffn_swiglu_workspace_size(qid, d_model, d_ff, batch)
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        st = lib.phb_ffn_swiglu(qid, *[t.data_ptr() for t in dev], x.data_ptr(), y_ref.data_ptr(), d_model, d_ff,
                                batch, ws.data_ptr(), need, stream)
        assert st == 0, lib.phb_last_error()
        y = torch.full((batch, d_model), float("nan"), device="cuda")
        st = lib.phb_ffn_swiglu_noalloc(qid, *[t.data_ptr() for t in dev], x.data_ptr(), y.data_ptr(), d_model, d_ff,
                                        batch, stream)
        assert st == 0, lib.phb_last_error()
        torch.cuda.synchronize()
        got, want = y.cpu().numpy().astype(np.float64), y_ref.cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(got))
        assert np.all(np.abs(got - want) <= tol), f"call {call}: max diff {np.abs(got - want).max()}"
