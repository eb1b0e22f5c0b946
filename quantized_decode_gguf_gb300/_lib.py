"""ctypes declarations of libphb.so (the C ABI in include/phb.h).

Loading fails loudly when the library has not been built: there is no
fallback implementation.
"""

from __future__ import annotations

import ctypes
import os
import threading

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libphb.so")

_c_i64 = ctypes.c_int64
_c_vp = ctypes.c_void_p
_c_sz = ctypes.c_size_t
_c_int = ctypes.c_int

# name -> (restype, argtypes); the set of symbols declared in include/phb.h
SIGNATURES = {
    "phb_version": (_c_int, []),
    "phb_last_error": (ctypes.c_char_p, []),
    "phb_row_bytes": (_c_sz, [_c_int, _c_i64]),
    "phb_device_error": (_c_int, [ctypes.POINTER(_c_int)]),
    "phb_dequant_q8_0": (_c_int, [_c_vp, _c_vp, _c_i64, _c_i64, _c_vp]),
    "phb_dequant_q4_k": (_c_int, [_c_vp, _c_vp, _c_i64, _c_i64, _c_vp]),
    "phb_dequant_q8_0_bf16": (_c_int, [_c_vp, _c_vp, _c_i64, _c_i64, _c_vp]),
    "phb_dequant_q4_k_bf16": (_c_int, [_c_vp, _c_vp, _c_i64, _c_i64, _c_vp]),
    "phb_gemv_workspace_size": (_c_sz, [_c_int, _c_i64, _c_i64, _c_int]),
    "phb_gemv": (_c_int, [_c_int, _c_vp, _c_vp, _c_vp, _c_i64, _c_i64, _c_int, _c_vp, _c_sz, _c_vp]),
    "phb_gemv_q8_0": (_c_int, [_c_vp, _c_vp, _c_vp, _c_i64, _c_i64, _c_int, _c_vp, _c_sz, _c_vp]),
    "phb_gemv_q4_k": (_c_int, [_c_vp, _c_vp, _c_vp, _c_i64, _c_i64, _c_int, _c_vp, _c_sz, _c_vp]),
    "phb_ffn_swiglu_workspace_size": (_c_sz, [_c_int, _c_i64, _c_i64, _c_int]),
    "phb_ffn_swiglu": (_c_int, [_c_int, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_i64, _c_i64, _c_int, _c_vp, _c_sz,
                                _c_vp]),
    "phb_moe_ffn_workspace_size": (_c_sz, [_c_int, _c_i64, _c_i64, _c_i64, _c_int, _c_int]),
    "phb_moe_ffn": (_c_int, [_c_int, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_i64, _c_i64, _c_i64, _c_int,
                             _c_int, _c_vp, _c_vp, _c_vp, _c_sz, _c_vp]),
    "phb_moe_ffn_tiered_workspace_size": (_c_sz, [_c_int, _c_i64, _c_i64, _c_i64, _c_int, _c_int]),
    "phb_moe_ffn_tiered": (_c_int, [_c_int, _c_vp, _c_vp, _c_vp, _c_int, _c_vp, _c_vp, _c_vp, _c_int, _c_vp, _c_vp,
                                    _c_vp, _c_vp, _c_i64, _c_i64, _c_i64, _c_int, _c_int, _c_vp, _c_vp, _c_vp, _c_sz,
                                    _c_vp]),
    "phb_gemm_q_prefill_workspace_size": (_c_sz, [_c_int, _c_i64, _c_i64, _c_i64]),
    "phb_gemm_q_prefill": (_c_int, [_c_int, _c_vp, _c_vp, _c_vp, _c_i64, _c_i64, _c_i64, _c_vp, _c_sz, _c_vp]),
    "phb_ffn_swiglu_noalloc_max_scratch": (_c_sz, []),
    "phb_ffn_swiglu_noalloc": (_c_int, [_c_int, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_i64, _c_i64, _c_int, _c_vp]),
    "phb_decode_step_workspace_size": (_c_sz, [_c_int, _c_i64, _c_int, _c_int, _c_int, _c_i64]),
    "phb_decode_step": (_c_int, [_c_int, _c_vp, _c_int, _c_i64, _c_int, _c_int, _c_int, _c_i64, _c_vp, _c_vp, _c_vp,
                                 _c_sz, _c_vp]),
    "phb_decode_step_unfused": (_c_int, [_c_int, _c_vp, _c_int, _c_i64, _c_int, _c_int, _c_int, _c_i64, _c_vp, _c_vp,
                                         _c_vp, _c_sz, _c_vp]),
    "phb_decode_step_probe": (_c_int, [_c_int, _c_i64, _c_int, _c_int, _c_int, _c_i64, _c_vp, _c_vp, _c_vp, _c_vp,
                                       _c_vp]),
    "phb_attention_decode_workspace_size": (_c_sz, [_c_i64, _c_int, _c_int, _c_int]),
    "phb_attention_decode": (_c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_i64, _c_int, _c_int, _c_int, ctypes.c_float,
                                      _c_vp, _c_sz, _c_vp]),
}


class DenseLayer(ctypes.Structure):
    """phb_dense_layer: device pointers of one decoder layer's weights."""
    _fields_ = [("w_qkv", _c_vp), ("w_o", _c_vp), ("w_gate", _c_vp), ("w_up", _c_vp), ("w_down", _c_vp)]


_lock = threading.Lock()
_lib = None


def load() -> ctypes.CDLL:
    """Load libphb.so once; raise if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is not built; run `python -m quantized_decode_gguf_gb300.build`")
            lib = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib
