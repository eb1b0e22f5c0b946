// Host-side interfaces shared by the translation units of libphb.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "phb.h"

namespace phb {

// Record the message of a failed call for phb_last_error() and return `s`.
phb_status set_last_error(phb_status s, const char* fmt, ...);
phb_status validate_ffn(int qtype, const void* Wgate, const void* Wup, const void* Wdown, const float* X,
                        const float* Y, int64_t d_model, int64_t d_ff, int batch);

// ---------------------------------------------------------------- device info
int device_sm_count();         // multiprocessors of the current device (cached)
constexpr size_t kSmemOptin = 232448;  // 227 KB dynamic shared memory per CTA

// Raise a kernel's dynamic shared-memory limit once per device.
template <auto KERN>
inline cudaError_t ensure_smem_attr() {
    static std::atomic<uint32_t> mask{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint32_t bit = 1u << (dev & 31);
    if (mask.load(std::memory_order_acquire) & bit) return cudaSuccess;
    e = cudaFuncSetAttribute(reinterpret_cast<const void*>(KERN), cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemOptin));
    // Every kernel asks for the largest shared-memory carveout, so kernels of
    // a programmatic-dependent chain share one SM configuration and the next
    // kernel's CTAs can be resident beside the current one's.
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(reinterpret_cast<const void*>(KERN), cudaFuncAttributePreferredSharedMemoryCarveout,
                                 static_cast<int>(cudaSharedmemCarveoutMaxShared));
    if (e == cudaSuccess) mask.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

// Launch with the programmatic-stream-serialization attribute (PDL) when
// `pdl` is set: the kernel may begin while its predecessor drains and must
// call griddepcontrol.wait before touching the predecessor's outputs.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                 bool pdl, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = pdl ? attr : nullptr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------- GEMV family
// qt: 0 = Q8_0, 1 = Q4_K.
struct GemvReq {
    int qt = 0;
    int nmat = 1;                 // 2: fused gate/up with SwiGLU epilogue
    const void* w0 = nullptr;
    const void* w1 = nullptr;
    int64_t n = 0, k = 0;
    int batch = 1;
    const float* x = nullptr;
    int64_t ldx = 0;
    float* y = nullptr;
    int64_t ldy = 0;
    const float* r = nullptr;     // residual input (epi == resid)
    int64_t ldr = 0;
    int xmode = 0;                // 0 plain, 1 rmsnorm, 2 gather V heads
    int epi = 0;                  // 0 store, 1 residual add, 2 SwiGLU
    int gather_group = 1, gather_hd = 0;
    int64_t gather_v_off = 0;
    float* ws = nullptr;          // split-K partials
    size_t ws_floats = 0;
    bool pdl = true;
    const void* pf[2] = {nullptr, nullptr};  // weights of later kernels to prefetch into L2
    int64_t pf_bytes[2] = {0, 0};
    int trace_id = -1;            // launch id recorded by debug tracing builds
};

// Workspace floats gemv_run needs for this request (split-K partials).
size_t gemv_ws_floats(const GemvReq& q);
// Plain GEMV (nmat 1, plain x, store) or fused gate/up (nmat 2, SwiGLU), any
// batch 1..8; K % 256 == 0 uses the streaming kernel, other Q8_0 K the
// generic one.
cudaError_t gemv_run(const GemvReq& q, cudaStream_t s);
// Batch-1 plain GEMV or fused gate/up with activations held in registers
// (gemv_xr.cu): whether a request fits it, and the launch.
bool gemv_xr_fits(const GemvReq& q);
cudaError_t gemv_xr_run(const GemvReq& q, cudaStream_t s);
// h[b][j] = silu(g[b][j]) * u[b][j] (unfused SwiGLU for shapes the fused
// kernel does not take).
cudaError_t swiglu_run(const float* g, const float* u, float* h, int64_t count, cudaStream_t s);

// ---------------------------------------------------------------- decode step
cudaError_t decode_gemv_run(const GemvReq& q, cudaStream_t s);  // rmsnorm / gather / residual variants

// Persistent (one cooperative kernel) decode step over at most kPersistMaxLayers
// layers; wl holds 5 weight pointers per layer (qkv, o, gate, up, down); ws
// is decode_persistent_ws_bytes long and zeroed before its first use.
constexpr int kPersistMaxLayers = 64;
size_t decode_persistent_ws_bytes(int64_t d_model, int n_q, int n_kv, int hd, int64_t d_ff);
cudaError_t decode_persistent_run(int qt, const void* const* wl, int n_layers, int64_t d_model, int n_q, int n_kv,
                                  int hd, int64_t d_ff, const float* x_in, float* x_out, void* ws, cudaStream_t s);
// Copies the last layer's qkv, x1 and SwiGLU activation out of a persistent-step workspace.
cudaError_t decode_persistent_probe(const void* ws, int64_t d_model, int n_q, int n_kv, int hd, int64_t d_ff,
                                    float* qkv, float* x1, float* act, cudaStream_t s);

// ---------------------------------------------------------------- dequant
cudaError_t dequant_run(int qt, bool bf16, const void* blocks, void* w, int64_t n, int64_t k, cudaStream_t s);

// ---------------------------------------------------------------- MoE
struct MoeReq {
    int qt = 1;
    const void* wg = nullptr;
    const void* wu = nullptr;
    const void* wd = nullptr;
    const float* x = nullptr;
    const float* logits = nullptr;
    float* y = nullptr;
    int64_t t = 0, d_model = 0, d_ff = 0;
    int e = 0, top_k = 0;
    int32_t* out_idx = nullptr;
    float* out_p = nullptr;
    void* ws = nullptr;
    size_t ws_bytes = 0;
    // tiered experts (nullptr loc: every expert is in wg/wu/wd, indexed by expert):
    // loc[e] >= 0: expert e is slot loc[e] of the device arrays wg/wu/wd (n_dev_slots experts);
    // loc[e] < 0: expert e is entry -1 - loc[e] of the GPU-readable host arrays hg/hu/hd
    const int32_t* loc = nullptr;
    int n_dev_slots = 0, n_host = 0;
    const void* hg = nullptr;
    const void* hu = nullptr;
    const void* hd = nullptr;
};
size_t moe_ws_bytes(const MoeReq& q);
cudaError_t moe_run(const MoeReq& q, cudaStream_t s);
// One-token MoE in one cooperative kernel (moe_token.cu): the workspace
// parts it uses, carved by moe_run.
constexpr int kTokReplicas = 8;  // tagged copies of h (CTA i reads copy i % 8)
struct MoeTokWs {
    float* h;
    float* yp;
    int32_t* idx;
    float* p;
    int32_t* src_sel;
    int32_t* src_z;
    uint8_t* stage[3];
    uint2* hx;        // {value, tag} copies of h: [kTokReplicas][top_k * d_ff]
    unsigned* epoch;  // calls so far (zero in a fresh workspace)
    int trace_id;
};
bool moe_token_fits(const MoeReq& q);
cudaError_t moe_token_run(const MoeReq& q, const MoeTokWs& w, cudaStream_t s);

// ---------------------------------------------------------------- prefill
struct PrefillReq {
    int qt = 0;
    const void* w = nullptr;
    const float* x = nullptr;
    float* y = nullptr;
    int64_t m = 0, n = 0, k = 0;
    void* ws = nullptr;
    size_t ws_bytes = 0;
};
size_t prefill_ws_bytes(const PrefillReq& q);
cudaError_t prefill_run(const PrefillReq& q, cudaStream_t s);

// ---------------------------------------------------------------- device error words
cudaError_t read_dev_err_gemv(int* code);
cudaError_t read_dev_err_decode(int* code);
cudaError_t read_dev_err_moe(int* code);
cudaError_t read_dev_err_prefill(int* code);
cudaError_t read_dev_err_decode_persistent(int* code);
cudaError_t read_dev_err_gemv_rows(int* code);
cudaError_t read_dev_err_attention(int* code);
cudaError_t read_dev_err_gemv_xr(int* code);
cudaError_t read_dev_err_moe_token(int* code);

// Row-resident batched GEMV (gemv_rows.cu): plain store, batch 2..8,
// K % 256 == 0. ksplit_out receives the K splits (> 1: partials in q.ws
// still need splitk reduction).
size_t gemv_rows_ws_floats(int qt, int64_t n, int64_t k, int batch);
cudaError_t gemv_rows_run(const GemvReq& q, cudaStream_t s, int* ksplit_out);

// ---------------------------------------------------------------- decode attention
// Split-KV attention of one token over an fp16 cache (attention.cu).
bool attention_shape_ok(int n_q, int n_kv, int hd);
size_t attention_ws_bytes(int n_q, int n_kv, int hd, int64_t len);
cudaError_t attention_run(const float* q, const void* k, const void* v, float* out, int n_q, int n_kv, int hd,
                          int64_t len, float scale, void* ws, cudaStream_t s);

}  // namespace phb
