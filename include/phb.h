/*
 * phb.h - C ABI of the GGUF dequantize-and-multiply library (libphb.so).
 *
 * The operations are the hot path of batch-1 LLM decoding from GGUF
 * block-quantized weights described by the Phobos README
 * (githubhelp.com, joa/phobos-lang): section "Inference" (Q8_0 and Q4_K_M
 * models decoded on the GPU; the host backend as verification oracle), the
 * "Phobos" overview (mixture-of-experts decode; prompt processing), the
 * `phobos-bench` tool (pp<N> prompt processing, tg<N> token generation) and
 * the examples table (`fuse_check`: the fused decode path against the
 * launched one). The pages give no library interface; these calls state the
 * problem those sections describe.
 *
 * Conventions shared by every call
 * --------------------------------
 * - Every tensor pointer is a DEVICE pointer owned by the caller. The library
 *   keeps no reference after the call returns.
 * - Calls are asynchronous on `stream` (the last argument; NULL = legacy
 *   default stream). No call synchronises or allocates memory; scratch space
 *   is the caller's `ws` buffer of `ws_bytes`, sized by the matching
 *   `*_workspace_size` function. A call may overwrite all of `ws`.
 * - Arguments are validated on the host before anything is launched; a call
 *   that returns an error has launched nothing. `phb_last_error()` then gives
 *   a message (per host thread).
 * - Pointers to quantized blocks, activations, outputs and workspaces must be
 *   16-byte aligned (PHB_ERR_ALIGN).
 * - Weight matrices are row-major: N rows (output features), each row K/32
 *   (Q8_0) or K/256 (Q4_K) consecutive blocks, K innermost. Activations are
 *   [batch][K] fp32 and outputs [batch][N] fp32, both dense.
 * - Block formats (GGUF convention; little-endian):
 *     Q8_0 (34 B, 32 weights):   fp16 d; int8 q[32];            w = d*q
 *     Q4_K (144 B, 256 weights): fp16 d; fp16 dmin; u8 scales[12]; u8 qs[128];
 *        sub-block j (weights 32j..32j+31) has 6-bit scale sc_j and min m_j:
 *        j<4: sc=scales[j]&63, m=scales[j+4]&63;
 *        j>=4: sc=(scales[j+4]&15)|(scales[j-4]>>6)<<4,
 *              m =(scales[j+4]>>4)|(scales[j]>>6)<<4;
 *        qs[32c+i] holds weight 64c+i (low nibble) and 64c+32+i (high);
 *        w = d*sc_j*q - dmin*m_j.
 * - Only CUDA devices of compute capability 10.3 (GB300, sm_103a) are
 *   supported (PHB_ERR_UNSUPPORTED_DEVICE).
 */
#ifndef PHB_H
#define PHB_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; declared here so users need no CUDA header. */
struct CUstream_st;
typedef struct CUstream_st* phb_stream_t;

typedef enum phb_status {
    PHB_OK = 0,
    PHB_ERR_INVALID_ARG = 1,        /* null pointer, non-positive size, unknown qtype */
    PHB_ERR_SHAPE = 2,              /* K not a multiple of the block size, top_k > n_experts, ... */
    PHB_ERR_ALIGN = 3,              /* a pointer is not 16-byte aligned */
    PHB_ERR_WORKSPACE = 4,          /* ws too small (or NULL while ws is needed) */
    PHB_ERR_CUDA = 5,               /* a CUDA runtime call failed; see phb_last_error() */
    PHB_ERR_UNSUPPORTED_DEVICE = 6, /* current device is not compute capability 10.3 */
    PHB_ERR_DEVICE_TIMEOUT = 7,     /* a kernel's bounded wait ran out (phb_device_error) */
    PHB_ERR_DEVICE_INPUT = 8        /* a kernel found a device-side input out of range (phb_device_error) */
} phb_status;

/* GGUF tensor type ids of the two formats. */
typedef enum phb_qtype {
    PHB_Q8_0 = 8,
    PHB_Q4_K = 12
} phb_qtype;

/* Library version, major*10000 + minor*100 + patch. */
int phb_version(void);

/* Message of the last failed call on this host thread ("" if none). The
 * string stays valid until the next call on the same thread. */
const char* phb_last_error(void);

/* Bytes of one quantized row of k weights; 0 if k is not a multiple of the
 * block size or qtype is unknown. */
size_t phb_row_bytes(int qtype, int64_t k);

/* Reads and clears the device-side error word that kernels set when a
 * bounded wait runs out (bit 0, PHB_ERR_DEVICE_TIMEOUT) or when a device-side
 * input is out of range (bit 1, PHB_ERR_DEVICE_INPUT: a tiered expert's
 * location outside both copies). Synchronises the current device. *code
 * receives 0 when no kernel reported an error. */
phb_status phb_device_error(int* code);

/* ---------------------------------------------------------------------------
 * Dequantisation (Phobos README, "Inference": the block formats of the
 * Q8_0 / Q4_K_M models). blocks: n_rows*k weights in row-major blocks;
 * w: [n_rows][k] output. fp32 results are bit-exact: Q8_0 d*q is exact in
 * fp32; for Q4_K, d*sc, dmin*m and (d*sc)*q are exact and only the final
 * subtraction rounds (to nearest even). The bf16 variants round that fp32
 * value to bf16 (nearest even); they feed the prompt-processing GEMM.
 * ------------------------------------------------------------------------- */
phb_status phb_dequant_q8_0(const void* blocks, float* w, int64_t n_rows, int64_t k, phb_stream_t stream);
phb_status phb_dequant_q4_k(const void* blocks, float* w, int64_t n_rows, int64_t k, phb_stream_t stream);
/* w: [n_rows][k] bf16 (uint16 bit patterns) */
phb_status phb_dequant_q8_0_bf16(const void* blocks, uint16_t* w, int64_t n_rows, int64_t k, phb_stream_t stream);
phb_status phb_dequant_q4_k_bf16(const void* blocks, uint16_t* w, int64_t n_rows, int64_t k, phb_stream_t stream);

/* ---------------------------------------------------------------------------
 * Quantized GEMV (Phobos README, "Inference" and `phobos-bench` tg<N>: token
 * generation multiplies every weight matrix by one activation vector per
 * sequence). Y[b][n] = sum_k w[n][k] * X[b][k] for b < batch, with w the
 * dequantised weights and fp32 accumulation. Contract: |Y - exact| <=
 * 1e-3 * sum_k |w[n][k] X[b][k]| per element.
 * W: n rows of k weights (qtype format); X: [batch][k]; Y: [batch][n].
 * batch: 1..8. Q4_K needs k % 256 == 0; Q8_0 needs k % 32 == 0.
 * ------------------------------------------------------------------------- */
size_t phb_gemv_workspace_size(int qtype, int64_t n, int64_t k, int batch);
phb_status phb_gemv(int qtype, const void* W, const float* X, float* Y, int64_t n, int64_t k, int batch,
                    void* ws, size_t ws_bytes, phb_stream_t stream);
phb_status phb_gemv_q8_0(const void* W, const float* X, float* Y, int64_t n, int64_t k, int batch,
                         void* ws, size_t ws_bytes, phb_stream_t stream);
phb_status phb_gemv_q4_k(const void* W, const float* X, float* Y, int64_t n, int64_t k, int batch,
                         void* ws, size_t ws_bytes, phb_stream_t stream);

/* ---------------------------------------------------------------------------
 * SwiGLU feed-forward block (Phobos README, "Inference": kernel fusion; the
 * examples table's `fuse_check`). With g = Wgate.x and u = Wup.x computed by
 * one fused pass over both matrices, h = silu(g) * u, silu(g) = g/(1+exp(-g)),
 * then Y = Wdown.h.
 * Wgate, Wup: [d_ff][d_model]; Wdown: [d_model][d_ff] (all qtype);
 * X: [batch][d_model]; Y: [batch][d_model]; batch 1..8. d_model and d_ff must
 * be multiples of the block size (256 for Q4_K, 32 for Q8_0). The hidden
 * activation h lives in ws: once the call has run (stream order), ws
 * begins with h as [batch][d_ff] fp32, so a checker can verify the down
 * projection from the activation the GPU actually used.
 * ------------------------------------------------------------------------- */
size_t phb_ffn_swiglu_workspace_size(int qtype, int64_t d_model, int64_t d_ff, int batch);
phb_status phb_ffn_swiglu(int qtype, const void* Wgate, const void* Wup, const void* Wdown,
                          const float* X, float* Y, int64_t d_model, int64_t d_ff, int batch,
                          void* ws, size_t ws_bytes, phb_stream_t stream);

/* ---------------------------------------------------------------------------
 * Top-k routed mixture-of-experts FFN (Phobos README overview and "Inference":
 * a 35B-A3B MoE; routing picks a few experts per token). Per token t:
 * the top_k largest router logits (ties to the lower expert index) select
 * experts e_{t,k} with weights p_{t,k} = softmax over those top_k logits, and
 * Y[t] = sum_k p_{t,k} * FFN_{e_{t,k}}(X[t]) with FFN the SwiGLU block above.
 * Each active expert's weights are read once per group of up to four
 * tokens routed to it; the weighted sum runs in a fixed order (slot k
 * ascending), so repeated calls are bitwise identical.
 * Wgate, Wup: [n_experts][d_ff][d_model]; Wdown: [n_experts][d_model][d_ff];
 * X: [n_tokens][d_model]; router_logits: [n_tokens][n_experts] fp32;
 * Y: [n_tokens][d_model]. out_idx ([n_tokens][top_k] int32) and out_p
 * ([n_tokens][top_k] fp32) receive the routing in descending logit order
 * when not NULL. n_tokens 1..64, n_experts 1..256, top_k 1..min(8, n_experts).
 * The workspace carries state between calls: per-row-tile counters (two
 * tokens: the last CTA of a tile combines the slots; each call returns them
 * to zero) and, for one token, a call epoch and epoch-tagged copies of the
 * expert activations (one cooperative kernel exchanges them between its
 * CTAs). A workspace belongs to one shape (n_tokens, d_model, d_ff,
 * n_experts, top_k): zero it before its first call and pass it, otherwise
 * untouched, to later calls of that shape; calls sharing a workspace must
 * not overlap on the GPU. After a device error (phb_device_error) zero it
 * again.
 * Once the call has run (stream order), ws begins with the per-pair expert
 * outputs FFN_{e_{t,k}}(X[t]) as [n_tokens * top_k][d_model] fp32 (pair
 * t * top_k + k), followed, at the next multiple of 256 bytes, by their
 * SwiGLU activations [n_tokens * top_k][d_ff], so that each stage can be
 * checked from the values the GPU actually used.
 * ------------------------------------------------------------------------- */
size_t phb_moe_ffn_workspace_size(int qtype, int64_t n_tokens, int64_t d_model, int64_t d_ff,
                                  int n_experts, int top_k);
phb_status phb_moe_ffn(int qtype, const void* Wgate, const void* Wup, const void* Wdown,
                       const float* X, const float* router_logits, float* Y,
                       int64_t n_tokens, int64_t d_model, int64_t d_ff, int n_experts, int top_k,
                       int32_t* out_idx, float* out_p,
                       void* ws, size_t ws_bytes, phb_stream_t stream);

/* ---------------------------------------------------------------------------
 * Routed MoE FFN with tiered experts (Phobos README, intro: MoE decode keeps
 * an expert cache sized by free device memory, and experts that do not fit
 * stay outside it; the author's feed: decode keeps most of its speed with
 * part of the memory taken). Same result as phb_moe_ffn, bit for bit, with
 * each expert's three matrices read from one of two copies:
 *   expert_loc[e] >= 0: slot expert_loc[e] of the device cache
 *       Wgate, Wup [n_dev_slots][d_ff][d_model], Wdown [n_dev_slots][d_model][d_ff];
 *   expert_loc[e] < 0:  entry -1 - expert_loc[e] of the host copy
 *       Wgate_host, Wup_host [n_host][d_ff][d_model], Wdown_host [n_host][d_model][d_ff].
 * expert_loc: DEVICE array [n_experts] int32. The host copy must be memory
 * the GPU can read: pinned (cudaMallocHost / cudaHostAlloc) or registered
 * (cudaHostRegister) host memory, or any host memory on a device that reads
 * pageable memory (a Grace system over NVLink-C2C); otherwise
 * PHB_ERR_INVALID_ARG. Nothing runs on the CPU: after routing, a fetch
 * kernel copies each active expert that lives only in the host copy into a
 * staging slot of the workspace (the GPU reads the host memory directly),
 * and the expert passes read each active expert from the cache or the
 * staging slot. A location outside both copies reads nothing and is
 * reported by phb_device_error (PHB_ERR_DEVICE_INPUT). Other arguments,
 * limits, the workspace rules (zero it before the first call) and the
 * documented workspace prefix are those of phb_moe_ffn; the workspace adds
 * min(n_experts, n_tokens * top_k) staging slots of one expert each.
 * ------------------------------------------------------------------------- */
size_t phb_moe_ffn_tiered_workspace_size(int qtype, int64_t n_tokens, int64_t d_model, int64_t d_ff,
                                         int n_experts, int top_k);
phb_status phb_moe_ffn_tiered(int qtype, const void* Wgate, const void* Wup, const void* Wdown, int n_dev_slots,
                              const void* Wgate_host, const void* Wup_host, const void* Wdown_host, int n_host,
                              const int32_t* expert_loc, const float* X, const float* router_logits, float* Y,
                              int64_t n_tokens, int64_t d_model, int64_t d_ff, int n_experts, int top_k,
                              int32_t* out_idx, float* out_p, void* ws, size_t ws_bytes, phb_stream_t stream);

/* ---------------------------------------------------------------------------
 * Prompt-processing GEMM (Phobos README: `phobos-bench` pp<N>; the
 * `gemm_fp16tc_fp32acc` tensor-core kernel of `phobos-kbench`).
 * Y[t][n] = sum_k bf16(w[n][k]) * bf16(X[t][k]) with fp32 accumulation on
 * the tensor cores, bf16() rounding to nearest even and w the fp32
 * dequantised weight. W: n rows of k weights (qtype); X: [m_tokens][k] fp32
 * (cast to bf16 into ws); Y: [m_tokens][n] fp32.
 * Needs n % 128 == 0, k % 256 == 0 (both formats), 1 <= m_tokens <= 4096.
 * ------------------------------------------------------------------------- */
size_t phb_gemm_q_prefill_workspace_size(int qtype, int64_t m_tokens, int64_t n, int64_t k);
phb_status phb_gemm_q_prefill(int qtype, const void* W, const float* X, float* Y,
                              int64_t m_tokens, int64_t n, int64_t k,
                              void* ws, size_t ws_bytes, phb_stream_t stream);

/* ---------------------------------------------------------------------------
 * One batch-1 decode step through a stack of dense pre-norm decoder layers
 * at position 0 (Phobos README, `phobos-bench` tg<N> and `fuse_check`).
 * Per layer, with x the residual stream [d_model]:
 *   h  = rmsnorm(x)                 (no gain, eps 1e-6)
 *   qkv = Wqkv.h                    [ (n_q + 2 n_kv) * head_dim ], Q | K | V
 *   a  = attention at position 0: query head i returns V of KV head
 *        i / (n_q / n_kv) (one key: softmax weight 1; RoPE is the identity)
 *   x  = x + Wo.a
 *   h  = rmsnorm(x)
 *   x  = x + Wdown.(silu(Wgate.h) * Wup.h)
 * layers: HOST array of n_layers descriptors whose members are DEVICE
 * pointers to qtype matrices: Wqkv [(n_q+2n_kv)*head_dim][d_model],
 * Wo [d_model][n_q*head_dim], Wgate/Wup [d_ff][d_model], Wdown [d_model][d_ff].
 * x_in, x_out: [d_model] fp32 (may not alias).
 *
 * phb_decode_step runs the fused path: one cooperative kernel per 64 layers,
 * one CTA per SM, in which every CTA streams its slice of all the layers'
 * weights through one shared-memory ring while the GEMVs wait on each other
 * through tagged intermediate vectors (with activations held in registers).
 * Its workspace carries a call epoch: zero it before the first call and
 * pass the same, otherwise untouched, workspace to later calls; calls
 * sharing a workspace must not overlap on the GPU. After a device error
 * (phb_device_error) the workspace must be zeroed again. The fused path
 * needs 2*d_model/256 and every K/256 to be at most the stage size (176
 * units), head_dim % 32 == 0 and ceil(d_model/SMs) <= 352; other shapes
 * return PHB_ERR_SHAPE (use phb_decode_step_unfused).
 * phb_decode_step_unfused launches the same arithmetic as 4 kernels per
 * layer (the pages' "launched" path that `fuse_check` compares the fused
 * one against); it needs no zeroing. Both can be captured in a CUDA graph
 * after one uncaptured call.
 * ------------------------------------------------------------------------- */
typedef struct phb_dense_layer {
    const void* w_qkv;
    const void* w_o;
    const void* w_gate;
    const void* w_up;
    const void* w_down;
} phb_dense_layer;

size_t phb_decode_step_workspace_size(int qtype, int64_t d_model, int n_q_heads, int n_kv_heads,
                                      int head_dim, int64_t d_ff);
phb_status phb_decode_step(int qtype, const phb_dense_layer* layers, int n_layers,
                           int64_t d_model, int n_q_heads, int n_kv_heads, int head_dim, int64_t d_ff,
                           const float* x_in, float* x_out,
                           void* ws, size_t ws_bytes, phb_stream_t stream);
phb_status phb_decode_step_unfused(int qtype, const phb_dense_layer* layers, int n_layers,
                                   int64_t d_model, int n_q_heads, int n_kv_heads, int head_dim, int64_t d_ff,
                                   const float* x_in, float* x_out,
                                   void* ws, size_t ws_bytes, phb_stream_t stream);

/* Checking aid for the decode step (the README's examples check the decode
 * path from its intermediate values: `fuse_check` compares the fused and
 * the launched decode, `kv_check` one decode step against a recompute).
 * Copies, in stream order, the intermediate vectors of the LAST layer of
 * the most recent decode-step call that used `ws` (fused != 0: a
 * phb_decode_step call; fused == 0: a phb_decode_step_unfused call) into
 * caller-owned device buffers:
 *   qkv [(n_q_heads + 2*n_kv_heads) * head_dim]  Wqkv . rmsnorm(x)
 *   x1  [d_model]                                 x + Wo . attention
 *   act [d_ff]                                    silu(Wgate.h) * (Wup.h)
 * so that each GEMV of the layer can be checked from the input the GPU
 * actually used. The shape arguments must be those of that call; ws is not
 * modified. Errors: PHB_ERR_INVALID_ARG (null pointer, size <= 0),
 * PHB_ERR_SHAPE (sizes beyond the decode step's limits), PHB_ERR_ALIGN
 * (ws not 16-byte aligned), PHB_ERR_CUDA. */
phb_status phb_decode_step_probe(int fused, int64_t d_model, int n_q_heads, int n_kv_heads, int head_dim,
                                 int64_t d_ff, const void* ws, float* qkv, float* x1, float* act,
                                 phb_stream_t stream);

/* ---------------------------------------------------------------------------
 * Decode attention at context depth (Phobos README: `phobos-bench -d N`,
 * decode with N tokens already in context; `phobos-kbench` `flash_fp16`,
 * f16 K/V with an f32 online-softmax state; the `kv_check` example).
 * One token's n_q_heads query heads against n_ctx cached positions:
 *   s_j = scale * q_h . k_j,   out_h = sum_j softmax(s)_j v_j   (j < n_ctx)
 * with query head h reading KV head h / (n_q_heads / n_kv_heads).
 * q: [n_q_heads][head_dim] fp32; k_cache, v_cache: [n_ctx][n_kv_heads]
 * [head_dim] IEEE fp16 (the first n_ctx positions of a cache in that
 * layout); out: [n_q_heads][head_dim] fp32. scale is usually
 * 1/sqrt(head_dim). Scores are accumulated in fp32 (for head_dim 64 and
 * 128 on the tensor cores, from the fp16 keys and the query split into two
 * fp16 parts after a per-head power-of-two scaling, about 2^-22 relative);
 * exponentials and sums are fp32. The result is within the fp32 error bound
 * of the exact softmax and bitwise identical across calls. K and V are read once (query heads past 8 per KV head
 * re-read them from L2).
 * Needs n_q_heads % n_kv_heads == 0 and head_dim 64, 128 or 256
 * (PHB_ERR_SHAPE), 1 <= n_ctx <= 2^26, positive head counts and a finite
 * scale (PHB_ERR_INVALID_ARG), every pointer 16-byte aligned
 * (PHB_ERR_ALIGN) and ws_bytes >= the workspace size (PHB_ERR_WORKSPACE);
 * a call that fails these launches nothing. The workspace holds
 * one partial result per position chunk; its size depends on the current
 * device's SM count. Nothing in it needs to start at zero.
 * ------------------------------------------------------------------------- */
size_t phb_attention_decode_workspace_size(int64_t n_ctx, int n_q_heads, int n_kv_heads, int head_dim);
phb_status phb_attention_decode(const float* q, const void* k_cache, const void* v_cache, float* out,
                                int64_t n_ctx, int n_q_heads, int n_kv_heads, int head_dim, float scale,
                                void* ws, size_t ws_bytes, phb_stream_t stream);

/* ---------------------------------------------------------------------------
 * SwiGLU feed-forward block that allocates nothing. The paper has no
 * counterpart; this is a convenience for callers that cannot allocate
 * device memory (a serving loop whose memory budget is fixed at start-up,
 * or a plugin running inside another runtime that owns all device memory).
 * Same arguments, result and bounds as phb_ffn_swiglu, minus the workspace:
 * the scratch is a static device array of
 * phb_ffn_swiglu_noalloc_max_scratch() bytes (2 MiB) compiled into the
 * library, which every GPU that loads the library holds until the process
 * exits. A shape whose phb_ffn_swiglu_workspace_size exceeds it returns
 * PHB_ERR_WORKSPACE. The first call on a device looks up the array's
 * device address (cudaGetSymbolAddress); make that first call before any
 * stream capture. Every call on a device uses the same array, which keeps
 * the previous call's contents (nothing in it needs to start at zero):
 * calls whose GPU work overlaps (other streams, other host threads) race.
 * ------------------------------------------------------------------------- */
size_t phb_ffn_swiglu_noalloc_max_scratch(void);
phb_status phb_ffn_swiglu_noalloc(int qtype, const void* Wgate, const void* Wup, const void* Wdown,
                                  const float* X, float* Y, int64_t d_model, int64_t d_ff, int batch,
                                  phb_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PHB_H */
