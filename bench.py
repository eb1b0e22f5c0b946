"""Benchmark of the GGUF dequantize-and-multiply path on one GB300.

Headline step: one batch-1 decode token through a dense 1B-class decoder
(24 layers, d_model 2048, 16 query / 4 KV heads of 128, SwiGLU FFN 5632, all
weights Q8_0), replayed from a CUDA graph of the library's decode-step call.
The value is the weight-streaming rate: algorithmic bytes (quantized weights
read once plus every GEMV's activation input and output) per second.

Additional rows, timed in the same run, each on seeded synthetic inputs:
  single Q8_0 GEMV 1024x1024; Q4_K GEMV sweep 2560->9728, 9728->2560,
  2560->4096 at batch 1 and 4; Q4_K MoE FFN (48 layers x 128 experts, top-8,
  d_model 2048, expert FFN 768) at 1 and 16 tokens; prompt-processing GEMM
  (512 tokens, Q4_K and Q8_0, 2560->9728 and 9728->2560).

Inputs larger than L2 stay resident in HBM; smaller ones rotate through
copies totalling more than twice the L2 size, so every figure is an HBM
figure. `--impl reference` times the CPU oracle on the machine's host cores.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "Q8_0/Q4_K dequant-GEMV GB/s (% of HBM peak); batch-1 decode tok/s per model"
D_MODEL, N_Q, N_KV, HD, D_FF, N_LAYERS = 2048, 16, 4, 128, 5632, 24
# DRAM bytes (read + write) per launch of the fused decode kernel at 24
# layers: an ncu capture of the 4-layer case (191.75 MB read + 2.95 MB
# written) scaled by 6; the weights are read once per step.
DECODE_TRAFFIC_PER_LAUNCH = 6 * (191.746e6 + 3.146e6)
QKV = (N_Q + 2 * N_KV) * HD
LAYER_SHAPES = [("qkv", QKV, D_MODEL), ("o", D_MODEL, N_Q * HD), ("gate", D_FF, D_MODEL), ("up", D_FF, D_MODEL),
                ("down", D_MODEL, D_FF)]


def row_bytes(qtype, k):
    return synth.row_bytes(qtype, k)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (200 ms) of SM clock and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- helpers

def cuda_time(fn, iters, stream=None):
    """Average ms per call of fn(i), timed with CUDA events on `stream`."""
    import torch
    s = stream or torch.cuda.current_stream()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(s)
    for i in range(iters):
        fn(i)
    stop.record(s)
    torch.cuda.synchronize()
    return start.elapsed_time(stop) / iters


def rotate_copies(t, min_total_bytes):
    """Copies of a device tensor totalling at least min_total_bytes."""
    n = max(2, math.ceil(min_total_bytes / max(1, t.numel() * t.element_size())))
    return [t.clone() for _ in range(n)]


def l2_bytes():
    import torch
    return int(getattr(torch.cuda.get_device_properties(0), "L2_cache_size", 126 * 2 ** 20))


# ----------------------------------------------------------------------------- decode (headline)

def decode_step_bytes():
    """Algorithmic bytes of one decode token: weights once + each GEMV's x and y."""
    w = N_LAYERS * sum(row_bytes("q8_0", k) * n for _, n, k in LAYER_SHAPES)
    act = 0
    for _, n, k in LAYER_SHAPES:
        act += 4 * (n + k)
    act -= 4 * (D_FF + D_MODEL)        # gate and up share x and are stored as one h
    return w, N_LAYERS * act


def build_decode(seed):
    import torch
    import quantized_decode_gguf_gb300 as phb
    layers = []
    for layer in range(N_LAYERS):
        mats = [torch.from_numpy(synth.q8_0_blocks(seed, 5 * layer + i, n, k)).cuda()
                for i, (_, n, k) in enumerate(LAYER_SHAPES)]
        layers.append(mats)
    table = phb.layer_table(layers)
    ws = phb.decode_workspace("q8_0", D_MODEL, N_Q, N_KV, HD, D_FF)
    return layers, table, ws


def bench_decode(steps, warmup, seed):
    import torch
    import quantized_decode_gguf_gb300 as phb
    layers, table, ws = build_decode(seed)
    x = torch.from_numpy(synth.normal_f32(seed, 100_000, (D_MODEL,))).cuda()
    y = torch.empty_like(x)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        phb.decode_step("q8_0", table, N_LAYERS, D_MODEL, N_Q, N_KV, HD, D_FF, x, y, ws)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        phb.decode_step("q8_0", table, N_LAYERS, D_MODEL, N_Q, N_KV, HD, D_FF, x, y, ws)
    torch.cuda.synchronize()
    for _ in range(max(3, warmup)):
        graph.replay()
    torch.cuda.synchronize()
    ms = cuda_time(lambda i: graph.replay(), steps)
    return {"ms": ms, "layers": layers, "table": table, "ws": ws, "x": x, "y": y, "graph": graph}


def bench_decode_e2e(ctx, steps):
    """Per token: pinned host x -> device, graph replay, device y -> pinned host, host reads it."""
    import torch
    x_host = torch.from_numpy(synth.normal_f32(0, 7, (D_MODEL,))).pin_memory()
    y_host = torch.empty(D_MODEL, dtype=torch.float32).pin_memory()
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        ctx["x"].copy_(x_host, non_blocking=True)
        ctx["graph"].replay()
        y_host.copy_(ctx["y"], non_blocking=True)
        stream.synchronize()
        _ = float(y_host[0])
    t1 = time.perf_counter()
    return (t1 - t0) * 1e3 / steps, x_host.numel() * 4, y_host.numel() * 4


def graph_time(fn, reps, iters=5):
    """Average ms per fn() call: fn captured reps times in a CUDA graph, replayed."""
    import torch
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        fn(0)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for i in range(reps):
            fn(i)
    g.replay()
    torch.cuda.synchronize()
    ms = cuda_time(lambda i: g.replay(), iters)
    return ms / reps


def bench_decode_kernels(ctx, seed):
    """The streaming GEMV at each decode-layer shape, 24 launches (one per layer's weights) per graph.

    The gate/up row uses the fused two-matrix kernel (SwiGLU epilogue) the decode step launches.
    """
    import torch
    import quantized_decode_gguf_gb300 as phb
    out = {}
    layers = ctx["layers"]
    xs = torch.randn(D_FF, device="cuda")
    for name, idx, n, k in [("qkv", 0, QKV, D_MODEL), ("o", 1, D_MODEL, N_Q * HD), ("down", 4, D_MODEL, D_FF)]:
        y = torch.empty(1, n, device="cuda")
        ws = phb.workspace(phb.gemv_workspace_size("q8_0", n, k, 1))
        x = xs[:k].contiguous().view(1, k)
        ms = graph_time(lambda i: phb.gemv("q8_0", layers[i % N_LAYERS][idx], x, n, k, out=y, ws=ws), N_LAYERS)
        b = row_bytes("q8_0", k) * n + 4 * (n + k)
        out[name] = {"n": n, "k": k, "us": ms * 1e3, "bytes": b, "gbs": b / (ms * 1e-3) / 1e9}
    # fused gate/up: phb_ffn_swiglu launches gate/up then down; time it whole and subtract the down GEMV
    h = torch.empty(1, D_MODEL, device="cuda")
    x = xs[:D_MODEL].contiguous().view(1, D_MODEL)
    fws = phb.workspace(phb.ffn_workspace_size("q8_0", D_MODEL, D_FF, 1))
    ms_ffn = graph_time(lambda i: phb.ffn_swiglu("q8_0", layers[i % N_LAYERS][2], layers[i % N_LAYERS][3],
                                                 layers[i % N_LAYERS][4], x, D_MODEL, D_FF, out=h, ws=fws), N_LAYERS)
    ms_gu = ms_ffn - out["down"]["us"] * 1e-3
    b = 2 * row_bytes("q8_0", D_MODEL) * D_FF + 4 * (D_MODEL + D_FF)
    out["gate_up"] = {"n": 2 * D_FF, "k": D_MODEL, "us": ms_gu * 1e3, "bytes": b, "gbs": b / (ms_gu * 1e-3) / 1e9,
                      "note": "phb_ffn_swiglu time minus the down GEMV's"}
    return out


# ----------------------------------------------------------------------------- other rows

def bench_gemv_row(qtype, n, k, batch, iters, seed, l2):  # noqa: ARG001
    import torch
    import quantized_decode_gguf_gb300 as phb
    w = torch.from_numpy(synth.blocks(qtype, seed, 0, n, k)).cuda()
    copies = rotate_copies(w, 2 * l2 + 64 * 2 ** 20)
    x = torch.from_numpy(synth.normal_f32(seed, 1, (batch, k))).cuda()
    y = torch.empty((batch, n), device="cuda")
    ws = phb.workspace(phb.gemv_workspace_size(qtype, n, k, batch))
    ms = graph_time(lambda i: phb.gemv(qtype, copies[i % len(copies)], x, n, k, out=y, ws=ws), len(copies))
    b = row_bytes(qtype, k) * n + 4 * batch * (n + k)
    return {"qtype": qtype, "n": n, "k": k, "batch": batch, "us": ms * 1e3, "bytes": b,
            "gbs": b / (ms * 1e-3) / 1e9}


def bench_moe(t_tokens, steps, seed):
    """48 layers x 128 experts (Q4_K), top-8; one step = the MoE FFN of all 48 layers."""
    import torch
    import quantized_decode_gguf_gb300 as phb
    e, k, d_model, d_ff, n_layers = 128, 8, 2048, 768, 48
    rb_in, rb_ff = row_bytes("q4_k", d_model), row_bytes("q4_k", d_ff)
    per_expert = 2 * d_ff * rb_in + d_model * rb_ff
    layers = []
    for layer in range(n_layers):
        # one seeded draw per layer, split into the three expert-major matrices
        gu = synth.q4_k_blocks(seed, 2000 + layer, 2 * e * d_ff, d_model).reshape(2, e, d_ff, rb_in)
        dn = synth.q4_k_blocks(seed, 3000 + layer, e * d_model, d_ff).reshape(e, d_model, rb_ff)
        layers.append((torch.from_numpy(np.ascontiguousarray(gu[0])).cuda(),
                       torch.from_numpy(np.ascontiguousarray(gu[1])).cuda(),
                       torch.from_numpy(dn).cuda()))
    x = torch.from_numpy(synth.normal_f32(seed, 1, (t_tokens, d_model))).cuda()
    logits = [torch.from_numpy(synth.normal_f32(seed, 5000 + l, (t_tokens, e))).cuda() for l in range(n_layers)]
    y = torch.empty_like(x)
    ws = phb.moe_workspace("q4_k", t_tokens, d_model, d_ff, e, k)
    idx = torch.empty((t_tokens, k), dtype=torch.int32, device="cuda")

    def step(_):
        for l in range(n_layers):
            phb.moe_ffn("q4_k", *layers[l], x, logits[l], d_model, d_ff, e, k, out=y, ws=ws, out_idx=idx)

    step(0)
    torch.cuda.synchronize()
    # distinct experts actually read per layer (from the routing the kernels produced)
    distinct = 0
    for l in range(n_layers):
        phb.moe_ffn("q4_k", *layers[l], x, logits[l], d_model, d_ff, e, k, out=y, ws=ws, out_idx=idx)
        distinct += len(set(idx.cpu().numpy().ravel().tolist()))
    ms = graph_time(step, 1, steps)
    b = distinct * per_expert + n_layers * 4 * t_tokens * (2 * d_model + k * (2 * d_ff + d_model))
    return {"tokens": t_tokens, "layers": n_layers, "distinct_experts_per_layer": distinct / n_layers,
            "ms_per_step": ms, "bytes": b, "gbs": b / (ms * 1e-3) / 1e9, "tok_per_s": t_tokens / (ms * 1e-3)}


_HOST_LINK = {}


def host_link_gbs():
    """Measured host->device rate of the copy engines on this machine: 256 MB of pinned host memory as four
    concurrent 64 MB copies on four streams, best of five. Context for the tiered-expert row's host
    traffic, not its bound: the fetch kernel reads host memory with SM loads, which measured faster
    (~520 GB/s for a 10.6 MB fetch alone)."""
    if "gbs" not in _HOST_LINK:
        import torch
        n, parts = 256 << 20, 4
        src = torch.empty(n, dtype=torch.uint8).pin_memory()
        dst = torch.empty(n, dtype=torch.uint8, device="cuda")
        streams = [torch.cuda.Stream() for _ in range(parts)]
        best = float("inf")
        for _ in range(5):
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for i, st in enumerate(streams):
                st.wait_event(a)
                with torch.cuda.stream(st):
                    dst[i * n // parts:(i + 1) * n // parts].copy_(src[i * n // parts:(i + 1) * n // parts],
                                                                   non_blocking=True)
            for st in streams:
                torch.cuda.current_stream().wait_stream(st)
            b.record()
            torch.cuda.synchronize()
            best = min(best, a.elapsed_time(b))
        _HOST_LINK["gbs"] = n / (best * 1e-3) / 1e9
    return _HOST_LINK["gbs"]


def bench_moe_tiered(t_tokens, steps, seed, n_layers=8, resident=0.5):
    """The MoE layer with only part of the experts resident: a device cache of `resident` x 128
    experts per layer, the rest in pinned host memory read by the GPU (phb_moe_ffn_tiered)."""
    import torch
    import quantized_decode_gguf_gb300 as phb
    e, k, d_model, d_ff = 128, 8, 2048, 768
    rb_in, rb_ff = row_bytes("q4_k", d_model), row_bytes("q4_k", d_ff)
    per_expert = 2 * d_ff * rb_in + d_model * rb_ff
    n_res = int(round(resident * e))
    layers = []
    for layer in range(n_layers):
        gu = synth.q4_k_blocks(seed, 2000 + layer, 2 * e * d_ff, d_model).reshape(2, e, d_ff, rb_in)
        dn = synth.q4_k_blocks(seed, 3000 + layer, e * d_model, d_ff).reshape(e, d_model, rb_ff)
        perm = synth.rng(seed, 4000 + layer).permutation(e)
        res, host = np.sort(perm[:n_res]), np.sort(perm[n_res:])
        loc = np.empty(e, dtype=np.int32)
        loc[res] = np.arange(n_res, dtype=np.int32)
        loc[host] = -1 - np.arange(e - n_res, dtype=np.int32)
        dev = tuple(torch.from_numpy(np.ascontiguousarray(m[res])).cuda() for m in (gu[0], gu[1], dn))
        hst = tuple(torch.from_numpy(np.ascontiguousarray(m[host])).pin_memory() for m in (gu[0], gu[1], dn))
        layers.append((dev, hst, torch.from_numpy(loc).cuda(), loc))
    x = torch.from_numpy(synth.normal_f32(seed, 1, (t_tokens, d_model))).cuda()
    logits = [torch.from_numpy(synth.normal_f32(seed, 5000 + l, (t_tokens, e))).cuda() for l in range(n_layers)]
    y = torch.empty_like(x)
    ws = phb.moe_tiered_workspace("q4_k", t_tokens, d_model, d_ff, e, k)
    idx = torch.empty((t_tokens, k), dtype=torch.int32, device="cuda")

    def step(_):
        for l in range(n_layers):
            dev, hst, loc_d, _ = layers[l]
            phb.moe_ffn_tiered("q4_k", *dev, *hst, loc_d, x, logits[l], d_model, d_ff, e, k, out=y, ws=ws,
                               out_idx=idx)

    step(0)
    torch.cuda.synchronize()
    distinct = from_host = 0
    for l in range(n_layers):
        dev, hst, loc_d, loc = layers[l]
        phb.moe_ffn_tiered("q4_k", *dev, *hst, loc_d, x, logits[l], d_model, d_ff, e, k, out=y, ws=ws, out_idx=idx)
        act = set(idx.cpu().numpy().ravel().tolist())
        distinct += len(act)
        from_host += sum(1 for a in act if loc[a] < 0)
    ms = graph_time(step, 1, steps)
    b = distinct * per_expert + n_layers * 4 * t_tokens * (2 * d_model + k * (2 * d_ff + d_model))
    return {"tokens": t_tokens, "layers": n_layers, "resident_fraction": resident,
            "distinct_experts_per_layer": distinct / n_layers, "from_host_per_layer": from_host / n_layers,
            "ms_per_step": ms, "us_per_layer": ms * 1e3 / n_layers, "bytes": b, "gbs": b / (ms * 1e-3) / 1e9,
            "host_bytes": from_host * per_expert, "host_gbs": from_host * per_expert / (ms * 1e-3) / 1e9,
            "host_copy_gbs": host_link_gbs(),
            "note": "experts read from host memory are copied over the host link into staging slots, then "
                    "streamed from HBM like the resident ones; GB/s counts every active expert's bytes once"}


def bench_prefill(qtype, n, k, m, iters, seed, peaks):
    import torch
    import quantized_decode_gguf_gb300 as phb
    w = torch.from_numpy(synth.blocks(qtype, seed, 0, n, k)).cuda()
    x = torch.from_numpy(synth.normal_f32(seed, 1, (m, k))).cuda()
    y = torch.empty((m, n), device="cuda")
    ws = phb.workspace(phb.prefill_workspace_size(qtype, m, n, k))
    try:
        phb.gemm_q_prefill(qtype, w, x, n, k, out=y, ws=ws)
    except phb.PhbError as exc:
        return {"qtype": qtype, "n": n, "k": k, "m": m, "unavailable": str(exc)}
    ms = graph_time(lambda i: phb.gemm_q_prefill(qtype, w, x, n, k, out=y, ws=ws), iters)
    fl = 2.0 * m * n * k
    tf = fl / (ms * 1e-3) / 1e12
    return {"qtype": qtype, "n": n, "k": k, "m": m, "us": ms * 1e3, "tflops": tf,
            "frac_of_bf16_peak": tf / peaks["bf16_tflops"]}


ATTN_SHAPE = (16, 4, 128)  # query heads, KV heads, head size of the dense decode workload


def attention_inputs(n_ctx, seed, hd=ATTN_SHAPE[2]):
    import torch
    n_q, n_kv = ATTN_SHAPE[0], ATTN_SHAPE[1]
    q = torch.from_numpy(synth.normal_f32(seed, 0, (n_q, hd))).cuda()
    k = torch.from_numpy(synth.normal_f16(seed, 1, (n_ctx, n_kv, hd))).cuda()
    v = torch.from_numpy(synth.normal_f16(seed, 2, (n_ctx, n_kv, hd))).cuda()
    return q, k, v


def bench_attention(n_ctx, iters, seed, l2, peaks):
    """Decode attention of one token at context depth n_ctx (fp16 KV cache); GB/s of algorithmic bytes."""
    import torch
    import quantized_decode_gguf_gb300 as phb
    n_q, n_kv, hd = ATTN_SHAPE
    q, k, v = attention_inputs(n_ctx, seed)
    kv = rotate_copies(torch.stack([k, v]), 2 * l2 + 64 * 2 ** 20)
    out = torch.empty((n_q, hd), device="cuda")
    ws = phb.workspace(phb.attention_workspace_size(n_ctx, n_q, n_kv, hd))
    ms = graph_time(lambda i: phb.attention_decode(q, kv[i % len(kv)][0], kv[i % len(kv)][1], n_ctx, n_q, n_kv, hd,
                                                   out=out, ws=ws), len(kv), iters)
    b = 2 * n_ctx * n_kv * hd * 2 + 2 * 4 * n_q * hd
    gbs = b / (ms * 1e-3) / 1e9
    return {"n_ctx": n_ctx, "n_q": n_q, "n_kv": n_kv, "head_dim": hd, "us": ms * 1e3, "bytes": b, "gbs": gbs,
            "frac": gbs / peaks["hbm_gbs"], "launches_per_call": 2,
            "l2": "rotating KV copies larger than L2"}


# ----------------------------------------------------------------------------- CPU oracle baseline

def cpu_baseline(budget_s=12.0):  # about 12 s of oracle work
    """The oracle's dequant + float64 GEMV over row samples of the decode-layer matrices."""
    import oracle
    seed = synth.workload_seed(1)
    done_bytes, t_used, mats = 0, 0.0, 0
    t0 = time.perf_counter()
    while t_used < budget_s and mats < 40 * N_LAYERS:
        layer, i = divmod(mats % (5 * N_LAYERS), 5)
        _, n, k = LAYER_SHAPES[i]
        rows = min(n, 1024)
        blob = synth.q8_0_blocks(seed, 5 * layer + i, n, k)[:rows]
        x = synth.normal_f32(seed, 7, (1, k))
        t1 = time.perf_counter()
        oracle.gemv_quant("q8_0", blob, x, rows, k)
        t_used += time.perf_counter() - t1
        done_bytes += blob.nbytes + 4 * (rows + k)
        mats += 1
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"value": done_bytes / t_used / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{mats} decode-layer matrices, first 1024 rows each, Q8_0 dequant + float64 GEMV "
                      f"({done_bytes / 1e6:.1f} MB in {t_used:.1f} s; numpy BLAS threads = host cores)",
            "wall_s": time.perf_counter() - t0}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    steps, warmup = args.steps, args.warmup
    budget = 90.0
    per_step = budget / max(1, steps + warmup)
    import oracle
    seed = synth.workload_seed(1)
    # one step: oracle dequant + float64 GEMV over a row sample of one decode-layer matrix
    _, n, k = LAYER_SHAPES[2]
    rb = row_bytes("q8_0", k)
    blob_full = synth.q8_0_blocks(seed, 2, n, k)
    x = synth.normal_f32(seed, 7, (1, k))
    t = time.perf_counter()
    oracle.gemv_quant("q8_0", blob_full[:64], x, 64, k)
    per_row = (time.perf_counter() - t) / 64
    rows = int(max(16, min(n, per_step / max(per_row, 1e-7))))
    blob = blob_full[:rows]
    for _ in range(warmup):
        oracle.gemv_quant("q8_0", blob, x, rows, k)
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle.gemv_quant("q8_0", blob, x, rows, k)
    dt = time.perf_counter() - t0
    b = rows * rb + 4 * (rows + k)
    val = b * steps / dt / 1e9
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": steps, "warmup": warmup, "ms_per_step": dt * 1e3 / steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "Q8_0 decode-layer gate matrix 5632x2048, row sample", "rows_per_step": rows},
            "cpu_baseline": {"value": val, "unit": "GB/s", "kind": "oracle", "cores": cores,
                             "sample": f"{rows} rows of the 5632x2048 Q8_0 gate matrix per step"},
            "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


# ----------------------------------------------------------------------------- profiling runs

def run_profile(args):
    """One path only, on a small case, for ncu: --warmup untimed calls then --steps calls."""
    import torch
    import quantized_decode_gguf_gb300 as phb
    seed = synth.workload_seed(1)
    if args.profile in ("decode", "decode-unfused"):
        n_layers = args.layers
        layers = [[torch.from_numpy(synth.q8_0_blocks(seed, 5 * layer + i, n, k)).cuda()
                   for i, (_, n, k) in enumerate(LAYER_SHAPES)] for layer in range(n_layers)]
        table = phb.layer_table(layers)
        ws = phb.decode_workspace("q8_0", D_MODEL, N_Q, N_KV, HD, D_FF)
        x = torch.from_numpy(synth.normal_f32(seed, 100_000, (D_MODEL,))).cuda()
        y = torch.empty_like(x)
        fused = args.profile == "decode"
        call = lambda: phb.decode_step("q8_0", table, n_layers, D_MODEL, N_Q, N_KV, HD, D_FF, x, y, ws,  # noqa: E731
                                       fused=fused)
        what = f"{'fused' if fused else 'launched'} decode step, {n_layers} layers"
    elif args.profile == "gemv":
        qt, n, k, b = args.gemv.split(",")
        n, k, b = int(n), int(k), int(b)
        w = torch.from_numpy(synth.blocks(qt, seed, 0, n, k)).cuda()
        x = torch.from_numpy(synth.normal_f32(seed, 1, (b, k))).cuda()
        y = torch.empty((b, n), device="cuda")
        ws = phb.workspace(phb.gemv_workspace_size(qt, n, k, b))
        call = lambda: phb.gemv(qt, w, x, n, k, out=y, ws=ws)  # noqa: E731
        what = f"GEMV {qt} {n}x{k} batch {b}"
    elif args.profile in ("moe1", "moe16"):
        t_tokens = 1 if args.profile == "moe1" else 16
        e, top_k, d_model, d_ff = 128, 8, 2048, 768
        n_layers = args.layers if args.layers != N_LAYERS else 4
        rb_in = row_bytes("q4_k", d_model)
        mats = []
        for layer in range(n_layers):
            gu = synth.q4_k_blocks(seed, 2000 + layer, 2 * e * d_ff, d_model).reshape(2, e, d_ff, rb_in)
            dn = synth.q4_k_blocks(seed, 3000 + layer, e * d_model, d_ff)
            mats.append((torch.from_numpy(np.ascontiguousarray(gu[0])).cuda(),
                         torch.from_numpy(np.ascontiguousarray(gu[1])).cuda(), torch.from_numpy(dn).cuda()))
        x = torch.from_numpy(synth.normal_f32(seed, 1, (t_tokens, d_model))).cuda()
        logits = [torch.from_numpy(synth.normal_f32(seed, 5000 + l, (t_tokens, e))).cuda() for l in range(n_layers)]
        y = torch.empty_like(x)
        ws = phb.moe_workspace("q4_k", t_tokens, d_model, d_ff, e, top_k)

        def call():
            for l in range(n_layers):
                phb.moe_ffn("q4_k", *mats[l], x, logits[l], d_model, d_ff, e, top_k, out=y, ws=ws)
        what = f"MoE FFN Q4_K, {t_tokens} tokens, {n_layers} layers"
    elif args.profile == "dequant":
        qt, n, k, _ = args.gemv.split(",")
        n, k = int(n), int(k)
        w = torch.from_numpy(synth.blocks(qt, seed, 0, n, k)).cuda()
        out = torch.empty((n, k), device="cuda")
        call = lambda: phb.dequant(qt, w, n, k, out=out)  # noqa: E731
        what = f"dequant {qt} {n}x{k} to fp32"
    elif args.profile == "moe-tiered":
        e, top_k, d_model, d_ff, t_tokens = 128, 8, 2048, 768, 1
        rb_in, rb_ff = row_bytes("q4_k", d_model), row_bytes("q4_k", d_ff)
        gu = synth.q4_k_blocks(seed, 2000, 2 * e * d_ff, d_model).reshape(2, e, d_ff, rb_in)
        dn = synth.q4_k_blocks(seed, 3000, e * d_model, d_ff).reshape(e, d_model, rb_ff)
        res, host = np.arange(0, e, 2), np.arange(1, e, 2)
        loc = np.empty(e, dtype=np.int32)
        loc[res] = np.arange(len(res), dtype=np.int32)
        loc[host] = -1 - np.arange(len(host), dtype=np.int32)
        dev = tuple(torch.from_numpy(np.ascontiguousarray(m[res])).cuda() for m in (gu[0], gu[1], dn))
        hst = tuple(torch.from_numpy(np.ascontiguousarray(m[host])).pin_memory() for m in (gu[0], gu[1], dn))
        loc_d = torch.from_numpy(loc).cuda()
        x = torch.from_numpy(synth.normal_f32(seed, 1, (t_tokens, d_model))).cuda()
        lg = torch.from_numpy(synth.normal_f32(seed, 5000, (t_tokens, e))).cuda()
        y = torch.empty_like(x)
        ws = phb.moe_tiered_workspace("q4_k", t_tokens, d_model, d_ff, e, top_k)
        call = lambda: phb.moe_ffn_tiered("q4_k", *dev, *hst, loc_d, x, lg, d_model, d_ff, e, top_k,  # noqa: E731
                                          out=y, ws=ws)
        what = "MoE FFN Q4_K with tiered experts, half in pinned host memory, one token, one layer"
    elif args.profile == "attention":
        n_q, n_kv, hd = ATTN_SHAPE[0], ATTN_SHAPE[1], args.hd
        q, k, v = attention_inputs(args.ctx, seed, hd)
        out = torch.empty((n_q, hd), device="cuda")
        ws = phb.workspace(phb.attention_workspace_size(args.ctx, n_q, n_kv, hd))
        call = lambda: phb.attention_decode(q, k, v, args.ctx, n_q, n_kv, hd, out=out, ws=ws)  # noqa: E731
        what = f"decode attention, {args.ctx} positions, {n_q}q/{n_kv}kv x {hd}"
    else:
        qt, n, k = args.prefill.split(",")
        n, k, m = int(n), int(k), 512
        w = torch.from_numpy(synth.blocks(qt, seed, 0, n, k)).cuda()
        x = torch.from_numpy(synth.normal_f32(seed, 1, (m, k))).cuda()
        y = torch.empty((m, n), device="cuda")
        ws = phb.workspace(phb.prefill_workspace_size(qt, m, n, k))
        call = lambda: phb.gemm_q_prefill(qt, w, x, n, k, out=y, ws=ws)  # noqa: E731
        what = f"prefill GEMM {qt} {m}x{n}x{k}"
    for _ in range(args.warmup + args.steps):
        call()
    torch.cuda.synchronize()
    err = phb.device_error()
    print(json.dumps({"profile": what, "calls": args.warmup + args.steps, "device_error": err}))
    if err:
        raise SystemExit(1)


# ----------------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="phb", choices=["phb", "reference"])
    ap.add_argument("--headline-only", action="store_true", help="skip the extra rows")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile", choices=["decode", "decode-unfused", "prefill", "moe1", "moe16", "gemv", "attention",
                                          "dequant", "moe-tiered"],
                    help="run only this path --steps times after --warmup calls (a small case for ncu) and print "
                         "one status line instead of the bench line")
    ap.add_argument("--layers", type=int, default=N_LAYERS, help="decode layers in --profile decode modes")
    ap.add_argument("--gemv", default="q4_k,9728,2560,4", help="--profile gemv case: qtype,n,k,batch")
    ap.add_argument("--ctx", type=int, default=32768, help="--profile attention: context positions")
    ap.add_argument("--hd", type=int, default=128, help="--profile attention: head dim")
    ap.add_argument("--prefill", default="q4_k,9728,2560", help="--profile prefill case: qtype,n,k (512 tokens)")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
        return

    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    from quantized_decode_gguf_gb300 import build
    if rank == 0 or world == 1:
        build.build()
    if args.profile:
        run_profile(args)
        return
    if world > 1:
        torch.distributed.barrier()
    import quantized_decode_gguf_gb300 as phb  # noqa: F401

    peaks = load_peaks()
    seed = synth.workload_seed(1)
    warmup = max(3, args.warmup)
    ctx = bench_decode(args.steps, warmup, seed)   # builds weights, graph, warm-up, first timing

    # timed region: K graph replays, barrier + sync on both sides, clocks sampled
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        ms = cuda_time(lambda i: ctx["graph"].replay(), args.steps)
        torch.cuda.synchronize()
        # keep the same work running for a while so the 200 ms clock samples see it under load
        t_soak = time.perf_counter()
        while time.perf_counter() - t_soak < 1.2:
            for _ in range(200):
                ctx["graph"].replay()
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    if world > 1:
        t = torch.tensor([ms], device="cuda")
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        torch.distributed.barrier()
        ms = float(t.item())
    wbytes, abytes = decode_step_bytes()
    step_bytes = wbytes + abytes
    gbs = world * step_bytes / (ms * 1e-3) / 1e9
    tok_s = world / (ms * 1e-3)

    e2e_ms, h2d, d2h = bench_decode_e2e(ctx, max(20, args.steps // 2))
    kernels = bench_decode_kernels(ctx, seed)
    unfused_ms = graph_time(lambda i: phb.decode_step("q8_0", ctx["table"], N_LAYERS, D_MODEL, N_Q, N_KV, HD, D_FF,
                                                      ctx["x"], ctx["y"], ctx["ws"], fused=False), 1, iters=200)
    result = {
        "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": "dense 1B-class decode step, batch 1, 24 layers, d_model 2048, 16q/4kv heads x 128, "
                               "SwiGLU 5632, all weights Q8_0 (1.15 GB per token)",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2 (1.15 GB of weights streamed per step)",
                   "graph": "one CUDA graph replay per step: one cooperative decode_persistent_kernel launch"},
        "tok_per_s": tok_s,
        "pct_of_hbm_peak": 100.0 * gbs / world / peaks["hbm_gbs"],
        "gpu_launches": args.steps,
        "clocks": dict(clk.summary(), window="the timed region and 1.2 s of further replays of the same graph"),
        "e2e": {"value": world * step_bytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s", "tok_per_s": world / (e2e_ms * 1e-3),
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        # the step is one launch of the persistent kernel: its algorithmic bytes (all weights once plus the
        # activation vectors) over the event-timed launch duration
        "roofline": {"bound": "hbm", "kernel": "decode_persistent_kernel (Q8_0, 24 layers, one launch per step)",
                     "achieved": step_bytes / (ms * 1e-3) / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": step_bytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                     "traffic": DECODE_TRAFFIC_PER_LAUNCH if N_LAYERS == 24 else None,
                     "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum of one 4-layer launch "
                                       "of the same kernel, scaled by 6 to 24 layers",
                     "bytes_per_launch": step_bytes, "peak_source": peaks["source"]},
        "decode_launched": {"ms_per_step": unfused_ms, "gbs": step_bytes / (unfused_ms * 1e-3) / 1e9,
                            "note": "phb_decode_step_unfused: 4 launches per layer in one CUDA graph"},
        "decode_kernels": kernels,
    }
    if not args.headline_only and rank == 0:
        l2 = l2_bytes()
        rows = {"gemv_q8_0_1024": bench_gemv_row("q8_0", 1024, 1024, 1, 200, synth.workload_seed(0), l2)}
        sweep = []
        for (n, k) in [(9728, 2560), (2560, 9728), (4096, 2560)]:
            for b in (1, 4):
                sweep.append(bench_gemv_row("q4_k", n, k, b, 100, synth.workload_seed(2), l2))
        rows["gemv_q4_k_sweep"] = sweep
        for r in [rows["gemv_q8_0_1024"]] + sweep:
            r["frac"] = r["gbs"] / peaks["hbm_gbs"]
        del ctx
        torch.cuda.empty_cache()
        moe = [bench_moe(t, 5, synth.workload_seed(3)) for t in (1, 16)]
        for r in moe:
            r["frac"] = r["gbs"] / peaks["hbm_gbs"]
        rows["moe_q4_k"] = moe
        torch.cuda.empty_cache()
        tiered = [bench_moe_tiered(t, 5, synth.workload_seed(3)) for t in (1, 16)]
        for r in tiered:
            r["frac"] = r["gbs"] / peaks["hbm_gbs"]
        rows["moe_q4_k_tiered"] = tiered
        torch.cuda.empty_cache()
        rows["prefill"] = [bench_prefill(q, n, k, 512, 20, synth.workload_seed(4), peaks)
                           for q in ("q4_k", "q8_0") for (n, k) in [(9728, 2560), (2560, 9728)]]
        torch.cuda.empty_cache()
        rows["attention_decode"] = [bench_attention(n, 50, synth.workload_seed(5), l2, peaks) for n in (4096, 32768)]
        result["rows"] = rows
    if rank == 0:
        if not args.no_cpu_baseline:
            result["cpu_baseline"] = cpu_baseline()
        print(json.dumps(result))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
