"""GGUF dequantize-and-multiply on GB300 (sm_103a).

The compute lives in libphb.so (C ABI: include/phb.h), built in-tree by
:mod:`quantized_decode_gguf_gb300.build`. :mod:`quantized_decode_gguf_gb300.api`
is the thin torch binding.
"""

from .api import (Q4_K, Q8_0, PhbError, attention_decode, attention_workspace_size,  # noqa: F401
                  decode_step, decode_step_probe, decode_workspace, decode_workspace_size, dequant, device_error,
                  ffn_swiglu, ffn_workspace_size, gemm_q_prefill, gemv, gemv_workspace_size, layer_table,
                  moe_ffn, moe_ffn_tiered, moe_tiered_workspace, moe_workspace, moe_workspace_size, prefill_workspace_size, row_bytes, workspace)
