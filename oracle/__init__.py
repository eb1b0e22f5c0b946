"""CPU oracle for the GGUF dequantize-and-multiply path (test infrastructure).

Only the tests, the package's smoke check and the benchmark's CPU-baseline
leg may import this package. It shares no code with the CUDA library, and the
library never calls it. Every function and the readings it rests on are
documented in :mod:`oracle.gguf`.

Parity status: every function is pinned by the CPU tests (closed forms,
exhaustive small cases, exact rational brute force, invariants and
hand-built golden blocks); none is "parity unpinned".
"""

from .gguf import *  # noqa: F401,F403
from .gguf import (QK8_0, QK_K, Q4_K_BYTES, Q8_0_BYTES, RMS_EPS, attention_decode, attention_pos0,  # noqa: F401
                   decode_layer, decode_layer_stages,
                   dequant, fp16_bits_to_f64, gemv, gemv_quant, moe_ffn, moe_route, prefill_gemm,
                   q4_k_dequant, q4_k_dequant_f64, q4_k_unpack, q8_0_dequant, q8_0_dequant_f64,
                   q8_0_unpack, rmsnorm, round_to_bf16, silu, swiglu_ffn, swiglu_stages, moe_stages)
