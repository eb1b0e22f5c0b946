"""The C ABI without a GPU: the library builds, loads, exports every symbol the
header declares, and rejects bad arguments before touching the device."""

import ctypes
import os
import re

import pytest

from quantized_decode_gguf_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "phb.h")

PHB_OK, INVALID, SHAPE, ALIGN, WORKSPACE = 0, 1, 2, 3, 4


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(phb_\w+)\s*\(", text)))


def test_header_declares_the_expected_calls():
    names = declared_functions()
    for want in ["phb_dequant_q8_0", "phb_dequant_q4_k", "phb_gemv_q8_0", "phb_gemv_q4_k", "phb_ffn_swiglu",
                 "phb_moe_ffn", "phb_gemm_q_prefill", "phb_decode_step", "phb_attention_decode", "phb_last_error"]:
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    assert set(names) == set(_lib.SIGNATURES), set(names) ^ set(_lib.SIGNATURES)


def test_version_and_row_bytes(lib):
    assert lib.phb_version() >= 10000
    assert lib.phb_row_bytes(8, 2048) == 2176
    assert lib.phb_row_bytes(12, 2560) == 1440
    assert lib.phb_row_bytes(12, 100) == 0
    assert lib.phb_row_bytes(99, 256) == 0


FAKE = 0x10000  # 16-byte aligned, never dereferenced: every call below fails validation first


def _err(lib):
    return lib.phb_last_error().decode()


def test_gemv_rejects_bad_arguments(lib):
    g = lib.phb_gemv
    assert g(8, FAKE, FAKE, FAKE, 64, 100, 1, None, 0, None) == SHAPE and "k %" in _err(lib)
    assert g(12, FAKE, FAKE, FAKE, 64, 512 + 32, 1, None, 0, None) == SHAPE
    assert g(8, None, FAKE, FAKE, 64, 64, 1, None, 0, None) == INVALID
    assert g(8, FAKE, FAKE, FAKE, 0, 64, 1, None, 0, None) == INVALID
    assert g(8, FAKE, FAKE, FAKE, 64, 64, 9, None, 0, None) == INVALID
    assert g(8, FAKE, FAKE, FAKE, 64, 64, 0, None, 0, None) == INVALID
    assert g(7, FAKE, FAKE, FAKE, 64, 64, 1, None, 0, None) == INVALID
    assert g(8, FAKE + 2, FAKE, FAKE, 64, 64, 1, None, 0, None) == ALIGN
    assert g(8, FAKE, FAKE + 4, FAKE, 64, 64, 1, None, 0, None) == ALIGN
    need = lib.phb_gemv_workspace_size(12, 2560, 9728, 4)
    assert need > 0
    assert g(12, FAKE, FAKE, FAKE, 2560, 9728, 4, None, 0, None) == WORKSPACE
    assert g(12, FAKE, FAKE, FAKE, 2560, 9728, 4, FAKE, need - 4, None) == WORKSPACE


def test_dequant_rejects_bad_arguments(lib):
    assert lib.phb_dequant_q8_0(FAKE, FAKE, 4, 33, None) == SHAPE
    assert lib.phb_dequant_q4_k(FAKE, FAKE, 4, 128, None) == SHAPE
    assert lib.phb_dequant_q4_k(None, FAKE, 4, 256, None) == INVALID
    assert lib.phb_dequant_q8_0_bf16(FAKE, FAKE + 8, 4, 32, None) == ALIGN
    assert lib.phb_dequant_q4_k_bf16(FAKE, FAKE, -1, 256, None) == INVALID


def test_moe_and_ffn_reject_bad_arguments(lib):
    m = lib.phb_moe_ffn
    args = [12, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE]
    assert m(*args, 1, 2048, 768, 128, 9, None, None, FAKE, 1 << 30, None) == INVALID
    assert m(*args, 1, 2048, 768, 4, 6, None, None, FAKE, 1 << 30, None) == SHAPE
    assert m(*args, 65, 2048, 768, 128, 8, None, None, FAKE, 1 << 30, None) == INVALID
    assert m(*args, 1, 2048 + 32, 768, 128, 8, None, None, FAKE, 1 << 30, None) == SHAPE
    assert m(*args, 1, 2048, 768, 128, 8, None, None, FAKE, 16, None) == WORKSPACE
    f = lib.phb_ffn_swiglu
    assert f(12, FAKE, FAKE, FAKE, FAKE, FAKE, 2048, 768 + 32, 1, FAKE, 1 << 30, None) == SHAPE
    assert f(8, FAKE, None, FAKE, FAKE, FAKE, 2048, 768, 1, FAKE, 1 << 30, None) == INVALID
    assert f(8, FAKE, FAKE, FAKE, FAKE, FAKE, 2048, 768, 1, FAKE, 8, None) == WORKSPACE


def test_prefill_and_decode_reject_bad_arguments(lib):
    p = lib.phb_gemm_q_prefill
    assert p(8, FAKE, FAKE, FAKE, 512, 9728 + 64, 2560, FAKE, 1 << 30, None) == SHAPE
    assert p(8, FAKE, FAKE, FAKE, 0, 9728, 2560, FAKE, 1 << 30, None) == INVALID
    assert p(8, FAKE, FAKE, FAKE, 512, 9728, 2560, FAKE, 16, None) == WORKSPACE
    d = lib.phb_decode_step
    layers = (_lib.DenseLayer * 1)(_lib.DenseLayer(FAKE, FAKE, FAKE, FAKE, FAKE))
    lp = ctypes.cast(layers, ctypes.c_void_p)
    assert d(8, lp, 1, 2048, 16, 3, 128, 5632, FAKE, FAKE + 256, FAKE, 1 << 30, None) == SHAPE
    assert d(8, lp, 1, 2048, 16, 4, 128, 5632, FAKE, FAKE, FAKE, 1 << 30, None) == INVALID
    assert d(8, lp, 0, 2048, 16, 4, 128, 5632, FAKE, FAKE + 256, FAKE, 1 << 30, None) == INVALID
    bad = (_lib.DenseLayer * 1)(_lib.DenseLayer(FAKE, None, FAKE, FAKE, FAKE))
    assert d(8, ctypes.cast(bad, ctypes.c_void_p), 1, 2048, 16, 4, 128, 5632, FAKE, FAKE + 256, FAKE, 1 << 30,
             None) == INVALID
    assert d(8, lp, 1, 2048, 16, 4, 128, 5632, FAKE, FAKE + 256, FAKE, 64, None) == WORKSPACE


def test_attention_rejects_bad_arguments(lib):
    a = lib.phb_attention_decode
    ptrs = [FAKE, FAKE, FAKE, FAKE]
    assert a(*ptrs, 4096, 16, 4, 96, 0.1, FAKE, 1 << 30, None) == SHAPE and "head_dim" in _err(lib)
    assert a(*ptrs, 4096, 6, 4, 128, 0.1, FAKE, 1 << 30, None) == SHAPE
    assert a(*ptrs, 0, 16, 4, 128, 0.1, FAKE, 1 << 30, None) == INVALID
    assert a(*ptrs, (1 << 26) + 1, 16, 4, 128, 0.1, FAKE, 1 << 30, None) == INVALID
    assert a(None, FAKE, FAKE, FAKE, 4096, 16, 4, 128, 0.1, FAKE, 1 << 30, None) == INVALID
    assert a(FAKE, FAKE + 8, FAKE, FAKE, 4096, 16, 4, 128, 0.1, FAKE, 1 << 30, None) == ALIGN
    assert a(*ptrs, 4096, 16, 4, 128, float("inf"), FAKE, 1 << 30, None) == INVALID
    assert a(*ptrs, 4096, 16, 4, 128, 0.1, FAKE, 16, None) == WORKSPACE
    assert lib.phb_attention_decode_workspace_size(4096, 16, 4, 128) > 0
    assert lib.phb_attention_decode_workspace_size(4096, 16, 4, 80) == 0
    assert lib.phb_attention_decode_workspace_size(0, 16, 4, 128) == 0
    assert lib.phb_attention_decode_workspace_size(4096, 16, 5, 128) == 0


def test_attention_binding_rejects_a_non_fp16_cache():
    # the binding checks the cache dtype before it touches the library or a device
    import torch

    import quantized_decode_gguf_gb300 as phb
    q = torch.zeros(8, 64)
    k32 = torch.zeros(16, 2, 64)
    with pytest.raises(TypeError):
        phb.attention_decode(q, k32, k32.half(), 16, 8, 2, 64)
    with pytest.raises(TypeError):
        phb.attention_decode(q, k32.half(), k32, 16, 8, 2, 64)


def test_ffn_noalloc_rejects_bad_arguments_without_a_device(lib):
    # argument errors come back before the device is looked up (no GPU here)
    f = lib.phb_ffn_swiglu_noalloc
    assert f(8, FAKE, None, FAKE, FAKE, FAKE, 2048, 768, 1, None) == INVALID
    assert f(8, FAKE, FAKE + 4, FAKE, FAKE, FAKE, 2048, 768, 1, None) == ALIGN
    assert f(12, FAKE, FAKE, FAKE, FAKE, FAKE, 2048, 768 + 32, 1, None) == SHAPE
    assert f(8, FAKE, FAKE, FAKE, FAKE, FAKE, 2048, 768, 0, None) == INVALID
    assert f(12, FAKE, FAKE, FAKE, FAKE, FAKE, 8192, 28672, 8, None) == WORKSPACE and "scratch" in _err(lib)


def test_moe_tiered_rejects_bad_arguments(lib):
    m = lib.phb_moe_ffn_tiered
    dev = [FAKE, FAKE, FAKE]
    host = [FAKE, FAKE, FAKE]
    tail = [FAKE, FAKE, FAKE, 1, 2048, 768, 128, 8, None, None, FAKE, 1 << 34, None]
    assert m(12, *dev, 0, *host, 0, FAKE, *tail) == INVALID            # no expert copy at all
    assert m(12, *dev, 64, *host, 64, None, *tail) == INVALID          # no location table
    assert m(12, None, FAKE, FAKE, 64, *host, 64, FAKE, *tail) == INVALID
    assert m(12, *dev, 64, None, FAKE, FAKE, 64, FAKE, *tail) == INVALID
    assert m(12, *dev, 64, *host, 64, FAKE + 2, *tail) == ALIGN
    assert m(12, *dev, 64, *host, 64, FAKE, FAKE, FAKE, FAKE, 1, 2048 + 32, 768, 128, 8, None, None, FAKE,
             1 << 34, None) == SHAPE
    assert m(12, *dev, 64, *host, 64, FAKE, *tail[:-3], FAKE, 64, None) == WORKSPACE
    plain = lib.phb_moe_ffn_workspace_size(12, 16, 2048, 768, 128, 8)
    tiered = lib.phb_moe_ffn_tiered_workspace_size(12, 16, 2048, 768, 128, 8)
    # the tiered workspace adds one staging slot per possible active expert (min(E, T*k) = 128)
    assert tiered >= plain + 128 * (2 * 768 * 1152 + 2048 * 432)
