"""Python binding of libphb: torch tensors in, C-ABI calls out.

Every function only marshals arguments (device pointers, sizes and the
current torch CUDA stream) into one call of the C ABI declared in
include/phb.h; all arithmetic runs in the library's CUDA kernels. Tensors
must live on the current CUDA device and be contiguous. Quantized weights
are uint8 tensors holding the GGUF blocks, rows contiguous.
"""

from __future__ import annotations

import ctypes
import math
from typing import Optional, Sequence

import torch

from . import _lib

Q8_0 = 8
Q4_K = 12
_QTYPES = {"q8_0": Q8_0, "q4_k": Q4_K, Q8_0: Q8_0, Q4_K: Q4_K}


class PhbError(RuntimeError):
    """A libphb call returned a non-zero phb_status."""

    def __init__(self, status: int, message: str):
        super().__init__(f"phb status {status}: {message}")
        self.status = status


def qtype_id(qtype) -> int:
    try:
        return _QTYPES[qtype]
    except KeyError:
        raise ValueError(f"unknown qtype {qtype!r}") from None


def _check(status: int) -> None:
    if status != 0:
        raise PhbError(status, _lib.load().phb_last_error().decode())


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _host_ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    """Address of a pinned, contiguous CPU tensor (memory the GPU can read)."""
    if t is None:
        return None
    if t.is_cuda or not t.is_pinned():
        raise ValueError("host tensor must be a pinned CPU tensor")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def row_bytes(qtype, k: int) -> int:
    return int(_lib.load().phb_row_bytes(qtype_id(qtype), k))


def workspace(nbytes: int, device=None) -> torch.Tensor:
    """Caller-owned scratch buffer (uint8) of at least ``nbytes`` bytes."""
    return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=device or "cuda")


def device_error() -> int:
    """Read and clear the kernels' device error word (synchronises): 0, or bit 0
    (a bounded wait ran out) and bit 1 (a device-side input out of range)."""
    code = ctypes.c_int(0)
    st = _lib.load().phb_device_error(ctypes.byref(code))
    if st not in (0, 7, 8):
        _check(st)
    return code.value


# ---------------------------------------------------------------- dequant

def dequant(qtype, blocks: torch.Tensor, n_rows: int, k: int, bf16: bool = False,
            out: Optional[torch.Tensor] = None) -> torch.Tensor:
    qt = qtype_id(qtype)
    if out is None:
        out = torch.empty((n_rows, k), dtype=torch.bfloat16 if bf16 else torch.float32, device=blocks.device)
    L = _lib.load()
    fn = {(Q8_0, False): L.phb_dequant_q8_0, (Q4_K, False): L.phb_dequant_q4_k,
          (Q8_0, True): L.phb_dequant_q8_0_bf16, (Q4_K, True): L.phb_dequant_q4_k_bf16}[(qt, bool(bf16))]
    _check(fn(_ptr(blocks), _ptr(out), n_rows, k, _stream()))
    return out


# ---------------------------------------------------------------- GEMV

def gemv_workspace_size(qtype, n: int, k: int, batch: int) -> int:
    return int(_lib.load().phb_gemv_workspace_size(qtype_id(qtype), n, k, batch))


def gemv(qtype, w: torch.Tensor, x: torch.Tensor, n: int, k: int, out: Optional[torch.Tensor] = None,
         ws: Optional[torch.Tensor] = None) -> torch.Tensor:
    """y[b] = W x[b]; x is [batch][k] (or [k])."""
    qt = qtype_id(qtype)
    x2 = x if x.dim() == 2 else x.view(1, -1)
    batch = x2.shape[0]
    if out is None:
        out = torch.empty((batch, n), dtype=torch.float32, device=x.device)
    need = gemv_workspace_size(qt, n, k, batch)
    if ws is None and need:
        ws = workspace(need, x.device)
    _check(_lib.load().phb_gemv(qt, _ptr(w), _ptr(x2), _ptr(out), n, k, batch, _ptr(ws),
                                0 if ws is None else ws.numel(), _stream()))
    return out


# ---------------------------------------------------------------- SwiGLU FFN

def ffn_workspace_size(qtype, d_model: int, d_ff: int, batch: int) -> int:
    return int(_lib.load().phb_ffn_swiglu_workspace_size(qtype_id(qtype), d_model, d_ff, batch))


def ffn_swiglu(qtype, w_gate, w_up, w_down, x: torch.Tensor, d_model: int, d_ff: int,
               out: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None) -> torch.Tensor:
    qt = qtype_id(qtype)
    x2 = x if x.dim() == 2 else x.view(1, -1)
    batch = x2.shape[0]
    if out is None:
        out = torch.empty((batch, d_model), dtype=torch.float32, device=x.device)
    if ws is None:
        ws = workspace(ffn_workspace_size(qt, d_model, d_ff, batch), x.device)
    _check(_lib.load().phb_ffn_swiglu(qt, _ptr(w_gate), _ptr(w_up), _ptr(w_down), _ptr(x2), _ptr(out), d_model,
                                      d_ff, batch, _ptr(ws), ws.numel(), _stream()))
    return out


# ---------------------------------------------------------------- MoE

def moe_workspace_size(qtype, n_tokens: int, d_model: int, d_ff: int, n_experts: int, top_k: int) -> int:
    return int(_lib.load().phb_moe_ffn_workspace_size(qtype_id(qtype), n_tokens, d_model, d_ff, n_experts, top_k))


def moe_workspace(qtype, n_tokens: int, d_model: int, d_ff: int, n_experts: int, top_k: int, device=None):
    """Workspace for :func:`moe_ffn` (zero-filled), reusable across calls."""
    n = moe_workspace_size(qtype, n_tokens, d_model, d_ff, n_experts, top_k)
    return torch.zeros(max(n, 16), dtype=torch.uint8, device=device or "cuda")


def moe_ffn(qtype, w_gate, w_up, w_down, x: torch.Tensor, logits: torch.Tensor, d_model: int, d_ff: int,
            n_experts: int, top_k: int, out: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
            out_idx: Optional[torch.Tensor] = None, out_p: Optional[torch.Tensor] = None) -> torch.Tensor:
    qt = qtype_id(qtype)
    t = x.shape[0]
    if out is None:
        out = torch.empty((t, d_model), dtype=torch.float32, device=x.device)
    if ws is None:
        ws = moe_workspace(qt, t, d_model, d_ff, n_experts, top_k, x.device)
    _check(_lib.load().phb_moe_ffn(qt, _ptr(w_gate), _ptr(w_up), _ptr(w_down), _ptr(x), _ptr(logits), _ptr(out), t,
                                   d_model, d_ff, n_experts, top_k, _ptr(out_idx), _ptr(out_p), _ptr(ws), ws.numel(),
                                   _stream()))
    return out


# ---------------------------------------------------------------- prefill GEMM

def moe_tiered_workspace(qtype, n_tokens: int, d_model: int, d_ff: int, n_experts: int, top_k: int, device=None):
    """Zeroed workspace for :func:`moe_ffn_tiered` (it carries counters that start at zero)."""
    n = int(_lib.load().phb_moe_ffn_tiered_workspace_size(qtype_id(qtype), n_tokens, d_model, d_ff, n_experts, top_k))
    return torch.zeros(max(n, 16), dtype=torch.uint8, device=device or "cuda")


def moe_ffn_tiered(qtype, w_gate, w_up, w_down, w_gate_host, w_up_host, w_down_host, expert_loc: torch.Tensor,
                   x: torch.Tensor, logits: torch.Tensor, d_model: int, d_ff: int, n_experts: int, top_k: int,
                   out: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
                   out_idx: Optional[torch.Tensor] = None, out_p: Optional[torch.Tensor] = None) -> torch.Tensor:
    """phb_moe_ffn_tiered: ``w_*`` the device expert cache [slots, ...] (or None), ``w_*_host`` the
    host copy [n_host, ...] in pinned CPU memory (or None), ``expert_loc`` int32 [n_experts] on the
    device (slot >= 0, or -1 - host index)."""
    qt = qtype_id(qtype)
    t = x.shape[0] if x.dim() == 2 else 1
    if out is None:
        out = torch.empty((t, d_model), dtype=torch.float32, device=x.device)
    if ws is None:
        ws = moe_tiered_workspace(qt, t, d_model, d_ff, n_experts, top_k, x.device)
    n_dev = 0 if w_gate is None else int(w_gate.shape[0])
    n_host = 0 if w_gate_host is None else int(w_gate_host.shape[0])
    _check(_lib.load().phb_moe_ffn_tiered(qt, _ptr(w_gate), _ptr(w_up), _ptr(w_down), n_dev,
                                          _host_ptr(w_gate_host), _host_ptr(w_up_host), _host_ptr(w_down_host), n_host, _ptr(expert_loc), _ptr(x),
                                          _ptr(logits), _ptr(out), t, d_model, d_ff, n_experts, top_k,
                                          _ptr(out_idx), _ptr(out_p), _ptr(ws), ws.numel(), _stream()))
    return out


def prefill_workspace_size(qtype, m_tokens: int, n: int, k: int) -> int:
    return int(_lib.load().phb_gemm_q_prefill_workspace_size(qtype_id(qtype), m_tokens, n, k))


def gemm_q_prefill(qtype, w, x: torch.Tensor, n: int, k: int, out: Optional[torch.Tensor] = None,
                   ws: Optional[torch.Tensor] = None) -> torch.Tensor:
    qt = qtype_id(qtype)
    m = x.shape[0]
    if out is None:
        out = torch.empty((m, n), dtype=torch.float32, device=x.device)
    if ws is None:
        ws = workspace(prefill_workspace_size(qt, m, n, k), x.device)
    _check(_lib.load().phb_gemm_q_prefill(qt, _ptr(w), _ptr(x), _ptr(out), m, n, k, _ptr(ws), ws.numel(),
                                          _stream()))
    return out


# ---------------------------------------------------------------- decode step

def decode_workspace_size(qtype, d_model: int, n_q: int, n_kv: int, head_dim: int, d_ff: int) -> int:
    return int(_lib.load().phb_decode_step_workspace_size(qtype_id(qtype), d_model, n_q, n_kv, head_dim, d_ff))


def layer_table(layers: Sequence[Sequence[torch.Tensor]]):
    """Host array of phb_dense_layer from [(w_qkv, w_o, w_gate, w_up, w_down), ...].

    The array holds device pointers; it also keeps references to the tensors,
    so that their memory cannot be freed and reused while the table exists."""
    arr = (_lib.DenseLayer * len(layers))()
    for i, ws in enumerate(layers):
        arr[i] = _lib.DenseLayer(*[_ptr(w) for w in ws])
    arr._tensors = [list(ws) for ws in layers]
    return arr


def decode_workspace(qtype, d_model: int, n_q: int, n_kv: int, head_dim: int, d_ff: int, device=None):
    """Zeroed workspace for :func:`decode_step` (the fused step keeps a call counter in it)."""
    n = decode_workspace_size(qtype, d_model, n_q, n_kv, head_dim, d_ff)
    return torch.zeros(max(n, 16), dtype=torch.uint8, device=device or "cuda")


def decode_step(qtype, table, n_layers: int, d_model: int, n_q: int, n_kv: int, head_dim: int, d_ff: int,
                x_in: torch.Tensor, x_out: Optional[torch.Tensor] = None,
                ws: Optional[torch.Tensor] = None, fused: bool = True) -> torch.Tensor:
    """One decode step; ``table`` comes from :func:`layer_table`.

    ``fused`` selects phb_decode_step (one cooperative kernel; ``ws`` from
    :func:`decode_workspace`, reused across calls) or phb_decode_step_unfused.
    """
    qt = qtype_id(qtype)
    if x_out is None:
        x_out = torch.empty_like(x_in)
    if ws is None:
        ws = decode_workspace(qt, d_model, n_q, n_kv, head_dim, d_ff, x_in.device)
    fn = _lib.load().phb_decode_step if fused else _lib.load().phb_decode_step_unfused
    _check(fn(qt, ctypes.cast(table, ctypes.c_void_p), n_layers, d_model, n_q, n_kv, head_dim, d_ff, _ptr(x_in),
              _ptr(x_out), _ptr(ws), ws.numel(), _stream()))
    return x_out


def decode_step_probe(ws: torch.Tensor, d_model: int, n_q: int, n_kv: int, head_dim: int, d_ff: int,
                      fused: bool = True):
    """phb_decode_step_probe: (qkv, x1, act) of the last layer of the latest decode step through ``ws``."""
    qkv = torch.empty((n_q + 2 * n_kv) * head_dim, dtype=torch.float32, device=ws.device)
    x1 = torch.empty(d_model, dtype=torch.float32, device=ws.device)
    act = torch.empty(d_ff, dtype=torch.float32, device=ws.device)
    _check(_lib.load().phb_decode_step_probe(int(bool(fused)), d_model, n_q, n_kv, head_dim, d_ff, _ptr(ws),
                                             _ptr(qkv), _ptr(x1), _ptr(act), _stream()))
    return qkv, x1, act


# ---------------------------------------------------------------- decode attention

def attention_workspace_size(n_ctx: int, n_q: int, n_kv: int, head_dim: int) -> int:
    return int(_lib.load().phb_attention_decode_workspace_size(n_ctx, n_q, n_kv, head_dim))


def attention_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, n_ctx: int, n_q: int, n_kv: int,
                     head_dim: int, scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                     ws: Optional[torch.Tensor] = None) -> torch.Tensor:
    """phb_attention_decode: q [n_q, head_dim] fp32 against the first ``n_ctx``
    positions of an fp16 cache [>= n_ctx, n_kv, head_dim]; returns [n_q, head_dim] fp32."""
    if k_cache.dtype != torch.float16 or v_cache.dtype != torch.float16:
        raise TypeError("the KV cache must be float16")
    if out is None:
        out = torch.empty((n_q, head_dim), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = workspace(attention_workspace_size(n_ctx, n_q, n_kv, head_dim), q.device)
    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)
    _check(_lib.load().phb_attention_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), n_ctx, n_q, n_kv,
                                            head_dim, float(scale), _ptr(ws), ws.numel(), _stream()))
    return out
