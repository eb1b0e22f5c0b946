// C ABI of libphb: argument validation, workspace sizing and dispatch.
// Every check runs on the host before anything is launched, so a call that
// returns an error has launched nothing.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <algorithm>
#include <cstring>
#include <string>

#include "phb.h"
#include "phb_internal.h"

namespace {

thread_local std::string g_last_error;

phb_status fail(phb_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

phb_status ok() {
    g_last_error.clear();
    return PHB_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// 0 = Q8_0, 1 = Q4_K, -1 = unknown
int qt_of(int qtype) { return qtype == PHB_Q8_0 ? 0 : qtype == PHB_Q4_K ? 1 : -1; }
int64_t block_weights(int qt) { return qt == 0 ? 32 : 256; }
const char* qt_name(int qt) { return qt == 0 ? "Q8_0" : "Q4_K"; }

phb_status cuda_fail(cudaError_t e, const char* what) {
    return fail(PHB_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

phb_status check_device() {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    static int cache[64];  // 0 unknown, 1 supported, 2 unsupported
    const int slot = dev & 63;
    if (cache[slot] == 0) {
        int major = 0, minor = 0;
        e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        cache[slot] = (major == 10 && minor == 3) ? 1 : 2;
        if (cache[slot] == 2)
            return fail(PHB_ERR_UNSUPPORTED_DEVICE, "device %d has compute capability %d.%d; libphb needs 10.3",
                        dev, major, minor);
    }
    if (cache[slot] == 2) return fail(PHB_ERR_UNSUPPORTED_DEVICE, "device %d is not compute capability 10.3", dev);
    return PHB_OK;
}

#define PHB_REQUIRE(cond, status, ...) \
    do {                               \
        if (!(cond)) return fail(status, __VA_ARGS__); \
    } while (0)

#define PHB_CUDA(expr, what)                         \
    do {                                             \
        const cudaError_t e_ = (expr);               \
        if (e_ != cudaSuccess) return cuda_fail(e_, what); \
    } while (0)

size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

// ---------------------------------------------------------------- GEMV helpers
phb::GemvReq gemv_req(int qt, const void* W, const float* X, float* Y, int64_t n, int64_t k, int batch) {
    phb::GemvReq q;
    q.qt = qt;
    q.w0 = W;
    q.n = n;
    q.k = k;
    q.batch = batch;
    q.x = X;
    q.ldx = k;
    q.y = Y;
    q.ldy = n;
    return q;
}

phb_status validate_gemv(int qt, const void* W, const float* X, const float* Y, int64_t n, int64_t k, int batch) {
    PHB_REQUIRE(qt >= 0, PHB_ERR_INVALID_ARG, "unknown qtype");
    PHB_REQUIRE(W && X && Y, PHB_ERR_INVALID_ARG, "null tensor pointer");
    PHB_REQUIRE(n > 0 && k > 0, PHB_ERR_INVALID_ARG, "n and k must be positive (n=%lld k=%lld)",
                static_cast<long long>(n), static_cast<long long>(k));
    PHB_REQUIRE(batch >= 1 && batch <= 8, PHB_ERR_INVALID_ARG, "batch must be 1..8 (got %d)", batch);
    PHB_REQUIRE(k % block_weights(qt) == 0, PHB_ERR_SHAPE, "%s needs k %% %lld == 0 (k=%lld)", qt_name(qt),
                static_cast<long long>(block_weights(qt)), static_cast<long long>(k));
    PHB_REQUIRE(n <= (int64_t{1} << 31) && k <= (int64_t{1} << 24), PHB_ERR_SHAPE, "shape too large");
    PHB_REQUIRE(aligned16(W) && aligned16(X) && aligned16(Y), PHB_ERR_ALIGN, "tensors must be 16-byte aligned");
    return PHB_OK;
}

size_t gemv_ws(int qt, int64_t n, int64_t k, int batch) {
    return phb::gemv_ws_floats(gemv_req(qt, nullptr, nullptr, nullptr, n, k, batch)) * sizeof(float);
}

phb_status run_gemv(const phb::GemvReq& q, cudaStream_t s) {
    const cudaError_t e = phb::gemv_run(q, s);
    if (e == cudaErrorInvalidConfiguration) return fail(PHB_ERR_SHAPE, "shape does not fit the GEMV kernel");
    if (e != cudaSuccess) return cuda_fail(e, "gemv launch");
    return PHB_OK;
}

// ---------------------------------------------------------------- FFN layout
struct FfnWs {
    float* g;
    float* u;
    float* h;
    float* split;
    size_t split_bytes;
    size_t bytes;
    bool fused;
};

FfnWs ffn_ws(int qt, int64_t d_model, int64_t d_ff, int batch, void* base) {
    FfnWs w{};
    const size_t hb = align256(static_cast<size_t>(batch) * d_ff * sizeof(float));
    w.fused = (d_model % 256 == 0) && (d_ff % 256 == 0) &&
              static_cast<size_t>(batch) * d_model * sizeof(float) <= 80 * 1024;
    size_t split = gemv_ws(qt, d_model, d_ff, batch);  // down projection
    if (!w.fused) split = std::max(split, gemv_ws(qt, d_ff, d_model, batch));
    w.split_bytes = align256(split);
    auto* b = static_cast<uint8_t*>(base);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        float* p = b ? reinterpret_cast<float*>(b + off) : nullptr;
        off += bytes;
        return p;
    };
    w.h = take(hb);
    if (!w.fused) {
        w.g = take(hb);
        w.u = take(hb);
    }
    w.split = take(w.split_bytes);
    w.bytes = off;
    return w;
}

// ---------------------------------------------------------------- decode layout
struct DecodeWs {
    float* qkv;
    float* x1;
    float* act;
    float* xs[2];
    size_t bytes;
};

DecodeWs decode_ws(int64_t d_model, int n_q, int n_kv, int hd, int64_t d_ff, void* base) {
    DecodeWs w{};
    auto* b = static_cast<uint8_t*>(base);
    size_t off = 0;
    auto take = [&](size_t count) {
        float* p = b ? reinterpret_cast<float*>(b + off) : nullptr;
        off += align256(count * sizeof(float));
        return p;
    };
    w.qkv = take(static_cast<size_t>(n_q + 2 * n_kv) * hd);
    w.x1 = take(d_model);
    w.act = take(d_ff);
    w.xs[0] = take(d_model);
    w.xs[1] = take(d_model);
    w.bytes = off;
    return w;
}

}  // namespace

namespace phb {
phb_status set_last_error(phb_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}
// Host-side argument checks of the SwiGLU block (pointers, alignment,
// shapes); touches no device.
phb_status validate_ffn(int qtype, const void* Wgate, const void* Wup, const void* Wdown, const float* X,
                        const float* Y, int64_t d_model, int64_t d_ff, int batch) {
    const int qt = qt_of(qtype);
    phb_status st = validate_gemv(qt, Wgate, X, Y, d_ff, d_model, batch);
    if (st != PHB_OK) return st;
    PHB_REQUIRE(Wup && Wdown, PHB_ERR_INVALID_ARG, "null weight pointer");
    PHB_REQUIRE(aligned16(Wup) && aligned16(Wdown), PHB_ERR_ALIGN, "pointers must be 16-byte aligned");
    PHB_REQUIRE(d_ff % block_weights(qt) == 0, PHB_ERR_SHAPE, "%s needs d_ff %% %lld == 0", qt_name(qt),
                static_cast<long long>(block_weights(qt)));
    return PHB_OK;
}
}  // namespace phb

extern "C" {

int phb_version(void) { return 10000; }

const char* phb_last_error(void) { return g_last_error.c_str(); }

size_t phb_row_bytes(int qtype, int64_t k) {
    const int qt = qt_of(qtype);
    if (qt < 0 || k <= 0 || k % block_weights(qt)) return 0;
    return qt == 0 ? static_cast<size_t>(k / 32 * 34) : static_cast<size_t>(k / 256 * 144);
}

phb_status phb_device_error(int* code) {
    PHB_REQUIRE(code, PHB_ERR_INVALID_ARG, "null code pointer");
    phb_status st = check_device();
    if (st != PHB_OK) return st;
    PHB_CUDA(cudaDeviceSynchronize(), "cudaDeviceSynchronize");
    int c[9] = {0, 0, 0, 0, 0, 0, 0, 0, 0};
    PHB_CUDA(phb::read_dev_err_gemv(&c[0]), "read device error");
    PHB_CUDA(phb::read_dev_err_decode(&c[1]), "read device error");
    PHB_CUDA(phb::read_dev_err_moe(&c[2]), "read device error");
    PHB_CUDA(phb::read_dev_err_prefill(&c[3]), "read device error");
    PHB_CUDA(phb::read_dev_err_decode_persistent(&c[4]), "read device error");
    PHB_CUDA(phb::read_dev_err_gemv_rows(&c[5]), "read device error");
    PHB_CUDA(phb::read_dev_err_attention(&c[6]), "read device error");
    PHB_CUDA(phb::read_dev_err_gemv_xr(&c[7]), "read device error");
    PHB_CUDA(phb::read_dev_err_moe_token(&c[8]), "read device error");
    *code = 0;
    for (int v : c) *code |= v;
    if (*code & 1) return fail(PHB_ERR_DEVICE_TIMEOUT, "a kernel reported device error %d", *code);
    if (*code) return fail(PHB_ERR_DEVICE_INPUT, "a kernel reported device error %d", *code);
    return ok();
}

// ---------------------------------------------------------------- dequant
static phb_status dequant_common(int qt, bool bf16, const void* blocks, void* w, int64_t n_rows, int64_t k,
                                 phb_stream_t stream) {
    PHB_REQUIRE(blocks && w, PHB_ERR_INVALID_ARG, "null tensor pointer");
    PHB_REQUIRE(n_rows > 0 && k > 0, PHB_ERR_INVALID_ARG, "n_rows and k must be positive");
    PHB_REQUIRE(k % block_weights(qt) == 0, PHB_ERR_SHAPE, "%s needs k %% %lld == 0", qt_name(qt),
                static_cast<long long>(block_weights(qt)));
    PHB_REQUIRE(aligned16(blocks) && aligned16(w), PHB_ERR_ALIGN, "tensors must be 16-byte aligned");
    phb_status st = check_device();
    if (st != PHB_OK) return st;
    PHB_CUDA(phb::dequant_run(qt, bf16, blocks, w, n_rows, k, stream), "dequant launch");
    return ok();
}

phb_status phb_dequant_q8_0(const void* blocks, float* w, int64_t n_rows, int64_t k, phb_stream_t stream) {
    return dequant_common(0, false, blocks, w, n_rows, k, stream);
}
phb_status phb_dequant_q4_k(const void* blocks, float* w, int64_t n_rows, int64_t k, phb_stream_t stream) {
    return dequant_common(1, false, blocks, w, n_rows, k, stream);
}
phb_status phb_dequant_q8_0_bf16(const void* blocks, uint16_t* w, int64_t n_rows, int64_t k,
                                 phb_stream_t stream) {
    return dequant_common(0, true, blocks, w, n_rows, k, stream);
}
phb_status phb_dequant_q4_k_bf16(const void* blocks, uint16_t* w, int64_t n_rows, int64_t k,
                                 phb_stream_t stream) {
    return dequant_common(1, true, blocks, w, n_rows, k, stream);
}

// ---------------------------------------------------------------- GEMV
size_t phb_gemv_workspace_size(int qtype, int64_t n, int64_t k, int batch) {
    const int qt = qt_of(qtype);
    if (qt < 0 || n <= 0 || k <= 0 || batch < 1 || batch > 8 || k % block_weights(qt)) return 0;
    return gemv_ws(qt, n, k, batch);
}

phb_status phb_gemv(int qtype, const void* W, const float* X, float* Y, int64_t n, int64_t k, int batch, void* ws,
                    size_t ws_bytes, phb_stream_t stream) {
    const int qt = qt_of(qtype);
    phb_status st = validate_gemv(qt, W, X, Y, n, k, batch);
    if (st != PHB_OK) return st;
    const size_t need = gemv_ws(qt, n, k, batch);
    PHB_REQUIRE(ws_bytes >= need && (need == 0 || ws), PHB_ERR_WORKSPACE, "workspace needs %zu bytes (got %zu)",
                need, ws_bytes);
    PHB_REQUIRE(aligned16(ws), PHB_ERR_ALIGN, "workspace must be 16-byte aligned");
    st = check_device();
    if (st != PHB_OK) return st;
    phb::GemvReq q = gemv_req(qt, W, X, Y, n, k, batch);
    q.ws = static_cast<float*>(ws);
    q.ws_floats = ws_bytes / sizeof(float);
    st = run_gemv(q, stream);
    return st == PHB_OK ? ok() : st;
}

phb_status phb_gemv_q8_0(const void* W, const float* X, float* Y, int64_t n, int64_t k, int batch, void* ws,
                         size_t ws_bytes, phb_stream_t stream) {
    return phb_gemv(PHB_Q8_0, W, X, Y, n, k, batch, ws, ws_bytes, stream);
}

phb_status phb_gemv_q4_k(const void* W, const float* X, float* Y, int64_t n, int64_t k, int batch, void* ws,
                         size_t ws_bytes, phb_stream_t stream) {
    return phb_gemv(PHB_Q4_K, W, X, Y, n, k, batch, ws, ws_bytes, stream);
}

// ---------------------------------------------------------------- SwiGLU FFN
size_t phb_ffn_swiglu_workspace_size(int qtype, int64_t d_model, int64_t d_ff, int batch) {
    const int qt = qt_of(qtype);
    if (qt < 0 || d_model <= 0 || d_ff <= 0 || batch < 1 || batch > 8) return 0;
    if (d_model % block_weights(qt) || d_ff % block_weights(qt)) return 0;
    return ffn_ws(qt, d_model, d_ff, batch, nullptr).bytes;
}

phb_status phb_ffn_swiglu(int qtype, const void* Wgate, const void* Wup, const void* Wdown, const float* X, float* Y,
                          int64_t d_model, int64_t d_ff, int batch, void* ws, size_t ws_bytes, phb_stream_t stream) {
    const int qt = qt_of(qtype);
    phb_status st = phb::validate_ffn(qtype, Wgate, Wup, Wdown, X, Y, d_model, d_ff, batch);
    if (st != PHB_OK) return st;
    PHB_REQUIRE(aligned16(ws), PHB_ERR_ALIGN, "pointers must be 16-byte aligned");
    const FfnWs need = ffn_ws(qt, d_model, d_ff, batch, nullptr);
    PHB_REQUIRE(ws && ws_bytes >= need.bytes, PHB_ERR_WORKSPACE, "workspace needs %zu bytes (got %zu)", need.bytes,
                ws_bytes);
    st = check_device();
    if (st != PHB_OK) return st;
    const FfnWs w = ffn_ws(qt, d_model, d_ff, batch, ws);
    if (w.fused) {
        phb::GemvReq q = gemv_req(qt, Wgate, X, w.h, d_ff, d_model, batch);
        q.nmat = 2;
        q.w1 = Wup;
        q.epi = 2;
        q.pf[0] = Wdown;  // the down projection streams into L2 while gate/up computes
        q.pf_bytes[0] = d_model * static_cast<int64_t>(phb_row_bytes(qtype, d_ff));
        st = run_gemv(q, stream);
        if (st != PHB_OK) return st;
    } else {
        phb::GemvReq q = gemv_req(qt, Wgate, X, w.g, d_ff, d_model, batch);
        q.ws = w.split;
        q.ws_floats = w.split_bytes / sizeof(float);
        if ((st = run_gemv(q, stream)) != PHB_OK) return st;
        q.w0 = Wup;
        q.y = w.u;
        if ((st = run_gemv(q, stream)) != PHB_OK) return st;
        PHB_CUDA(phb::swiglu_run(w.g, w.u, w.h, static_cast<int64_t>(batch) * d_ff, stream), "swiglu launch");
    }
    phb::GemvReq qd = gemv_req(qt, Wdown, w.h, Y, d_model, d_ff, batch);
    qd.ws = w.split;
    qd.ws_floats = w.split_bytes / sizeof(float);
    st = run_gemv(qd, stream);
    return st == PHB_OK ? ok() : st;
}

// ---------------------------------------------------------------- MoE
size_t phb_moe_ffn_workspace_size(int qtype, int64_t n_tokens, int64_t d_model, int64_t d_ff, int n_experts,
                                  int top_k) {
    const int qt = qt_of(qtype);
    if (qt < 0 || n_tokens < 1 || n_tokens > 64 || n_experts < 1 || n_experts > 256 || top_k < 1 || top_k > 8 ||
        top_k > n_experts || d_model <= 0 || d_ff <= 0)
        return 0;
    phb::MoeReq q;
    q.qt = qt;
    q.t = n_tokens;
    q.d_model = d_model;
    q.d_ff = d_ff;
    q.e = n_experts;
    q.top_k = top_k;
    return phb::moe_ws_bytes(q);
}

phb_status phb_moe_ffn(int qtype, const void* Wgate, const void* Wup, const void* Wdown, const float* X,
                       const float* router_logits, float* Y, int64_t n_tokens, int64_t d_model, int64_t d_ff,
                       int n_experts, int top_k, int32_t* out_idx, float* out_p, void* ws, size_t ws_bytes,
                       phb_stream_t stream) {
    const int qt = qt_of(qtype);
    PHB_REQUIRE(qt >= 0, PHB_ERR_INVALID_ARG, "unknown qtype");
    PHB_REQUIRE(Wgate && Wup && Wdown && X && router_logits && Y, PHB_ERR_INVALID_ARG, "null tensor pointer");
    PHB_REQUIRE(n_tokens >= 1 && n_tokens <= 64, PHB_ERR_INVALID_ARG, "n_tokens must be 1..64");
    PHB_REQUIRE(n_experts >= 1 && n_experts <= 256, PHB_ERR_INVALID_ARG, "n_experts must be 1..256");
    PHB_REQUIRE(top_k >= 1 && top_k <= 8, PHB_ERR_INVALID_ARG, "top_k must be 1..8");
    PHB_REQUIRE(top_k <= n_experts, PHB_ERR_SHAPE, "top_k > n_experts");
    PHB_REQUIRE(d_model > 0 && d_ff > 0, PHB_ERR_INVALID_ARG, "d_model and d_ff must be positive");
    PHB_REQUIRE(d_model % 256 == 0 && d_ff % 256 == 0, PHB_ERR_SHAPE, "MoE needs d_model and d_ff multiples of 256");
    PHB_REQUIRE(d_model <= 4096 && d_ff <= 4096, PHB_ERR_SHAPE, "MoE needs d_model, d_ff <= 4096");
    PHB_REQUIRE(aligned16(Wgate) && aligned16(Wup) && aligned16(Wdown) && aligned16(X) && aligned16(router_logits) &&
                    aligned16(Y) && aligned16(ws),
                PHB_ERR_ALIGN, "tensors must be 16-byte aligned");
    const size_t need = phb_moe_ffn_workspace_size(qtype, n_tokens, d_model, d_ff, n_experts, top_k);
    PHB_REQUIRE(ws && ws_bytes >= need, PHB_ERR_WORKSPACE, "workspace needs %zu bytes (got %zu)", need, ws_bytes);
    phb_status st = check_device();
    if (st != PHB_OK) return st;
    phb::MoeReq q;
    q.qt = qt;
    q.wg = Wgate;
    q.wu = Wup;
    q.wd = Wdown;
    q.x = X;
    q.logits = router_logits;
    q.y = Y;
    q.t = n_tokens;
    q.d_model = d_model;
    q.d_ff = d_ff;
    q.e = n_experts;
    q.top_k = top_k;
    q.out_idx = out_idx;
    q.out_p = out_p;
    q.ws = ws;
    q.ws_bytes = ws_bytes;
    const cudaError_t e = phb::moe_run(q, stream);
    if (e == cudaErrorInvalidConfiguration) return fail(PHB_ERR_SHAPE, "shape does not fit the MoE kernels");
    if (e != cudaSuccess) return cuda_fail(e, "moe launch");
    return ok();
}

// ---------------------------------------------------------------- MoE with tiered experts
size_t phb_moe_ffn_tiered_workspace_size(int qtype, int64_t n_tokens, int64_t d_model, int64_t d_ff, int n_experts,
                                         int top_k) {
    if (phb_moe_ffn_workspace_size(qtype, n_tokens, d_model, d_ff, n_experts, top_k) == 0) return 0;
    phb::MoeReq q;
    q.qt = qt_of(qtype);
    q.t = n_tokens;
    q.d_model = d_model;
    q.d_ff = d_ff;
    q.e = n_experts;
    q.top_k = top_k;
    static const int32_t kAnyLoc = 0;
    q.loc = &kAnyLoc;  // any non-null table: the layout with staging slots
    return phb::moe_ws_bytes(q);
}

// A pointer the GPU can read for the host-resident experts: pinned or
// registered host memory (its device address), device or managed memory, or
// any host address when the device reads pageable memory directly.
static phb_status gpu_readable(const void* p, const void** dev) {
    cudaPointerAttributes a{};
    cudaError_t e = cudaPointerGetAttributes(&a, p);
    if (e != cudaSuccess) return cuda_fail(e, "cudaPointerGetAttributes");
    if (a.type == cudaMemoryTypeHost && a.devicePointer != nullptr) {
        *dev = a.devicePointer;
        return PHB_OK;
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) {
        *dev = p;
        return PHB_OK;
    }
    int devi = 0, pageable = 0;
    if (cudaGetDevice(&devi) == cudaSuccess &&
        cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, devi) == cudaSuccess && pageable) {
        *dev = p;
        return PHB_OK;
    }
    return fail(PHB_ERR_INVALID_ARG, "host experts must be pinned or registered host memory the GPU can read");
}

phb_status phb_moe_ffn_tiered(int qtype, const void* Wgate, const void* Wup, const void* Wdown, int n_dev_slots,
                              const void* Wgate_host, const void* Wup_host, const void* Wdown_host, int n_host,
                              const int32_t* expert_loc, const float* X, const float* router_logits, float* Y,
                              int64_t n_tokens, int64_t d_model, int64_t d_ff, int n_experts, int top_k,
                              int32_t* out_idx, float* out_p, void* ws, size_t ws_bytes, phb_stream_t stream) {
    const int qt = qt_of(qtype);
    PHB_REQUIRE(qt >= 0, PHB_ERR_INVALID_ARG, "unknown qtype");
    PHB_REQUIRE(X && router_logits && Y && expert_loc, PHB_ERR_INVALID_ARG, "null tensor pointer");
    PHB_REQUIRE(n_dev_slots >= 0 && n_host >= 0 && n_dev_slots + n_host >= 1, PHB_ERR_INVALID_ARG,
                "need n_dev_slots >= 0, n_host >= 0 and at least one expert copy");
    PHB_REQUIRE(n_dev_slots == 0 || (Wgate && Wup && Wdown), PHB_ERR_INVALID_ARG, "null device expert pointer");
    PHB_REQUIRE(n_host == 0 || (Wgate_host && Wup_host && Wdown_host), PHB_ERR_INVALID_ARG,
                "null host expert pointer");
    PHB_REQUIRE(n_tokens >= 1 && n_tokens <= 64, PHB_ERR_INVALID_ARG, "n_tokens must be 1..64");
    PHB_REQUIRE(n_experts >= 1 && n_experts <= 256, PHB_ERR_INVALID_ARG, "n_experts must be 1..256");
    PHB_REQUIRE(top_k >= 1 && top_k <= 8, PHB_ERR_INVALID_ARG, "top_k must be 1..8");
    PHB_REQUIRE(top_k <= n_experts, PHB_ERR_SHAPE, "top_k > n_experts");
    PHB_REQUIRE(d_model > 0 && d_ff > 0, PHB_ERR_INVALID_ARG, "d_model and d_ff must be positive");
    PHB_REQUIRE(d_model % 256 == 0 && d_ff % 256 == 0, PHB_ERR_SHAPE, "MoE needs d_model and d_ff multiples of 256");
    PHB_REQUIRE(d_model <= 4096 && d_ff <= 4096, PHB_ERR_SHAPE, "MoE needs d_model, d_ff <= 4096");
    PHB_REQUIRE(aligned16(Wgate) && aligned16(Wup) && aligned16(Wdown) && aligned16(Wgate_host) &&
                    aligned16(Wup_host) && aligned16(Wdown_host) && aligned16(X) && aligned16(router_logits) &&
                    aligned16(Y) && aligned16(ws) && (reinterpret_cast<uintptr_t>(expert_loc) & 3u) == 0,
                PHB_ERR_ALIGN, "tensors must be 16-byte aligned (expert_loc 4-byte)");
    const size_t need = phb_moe_ffn_tiered_workspace_size(qtype, n_tokens, d_model, d_ff, n_experts, top_k);
    PHB_REQUIRE(ws && ws_bytes >= need, PHB_ERR_WORKSPACE, "workspace needs %zu bytes (got %zu)", need, ws_bytes);
    phb_status st = check_device();
    if (st != PHB_OK) return st;
    const void* hg = nullptr;
    const void* hu = nullptr;
    const void* hd = nullptr;
    if (n_host > 0) {
        if ((st = gpu_readable(Wgate_host, &hg)) != PHB_OK || (st = gpu_readable(Wup_host, &hu)) != PHB_OK ||
            (st = gpu_readable(Wdown_host, &hd)) != PHB_OK)
            return st;
    }
    phb::MoeReq q;
    q.qt = qt;
    q.wg = Wgate;
    q.wu = Wup;
    q.wd = Wdown;
    q.x = X;
    q.logits = router_logits;
    q.y = Y;
    q.t = n_tokens;
    q.d_model = d_model;
    q.d_ff = d_ff;
    q.e = n_experts;
    q.top_k = top_k;
    q.out_idx = out_idx;
    q.out_p = out_p;
    q.ws = ws;
    q.ws_bytes = ws_bytes;
    q.loc = expert_loc;
    q.n_dev_slots = n_dev_slots;
    q.n_host = n_host;
    q.hg = hg;
    q.hu = hu;
    q.hd = hd;
    const cudaError_t e = phb::moe_run(q, stream);
    if (e == cudaErrorInvalidConfiguration) return fail(PHB_ERR_SHAPE, "shape does not fit the MoE kernels");
    if (e != cudaSuccess) return cuda_fail(e, "moe launch");
    return ok();
}

// ---------------------------------------------------------------- prefill GEMM
size_t phb_gemm_q_prefill_workspace_size(int qtype, int64_t m_tokens, int64_t n, int64_t k) {
    const int qt = qt_of(qtype);
    if (qt < 0 || m_tokens < 1 || m_tokens > 4096 || n <= 0 || k <= 0 || n % 128 || k % 256) return 0;
    phb::PrefillReq q;
    q.qt = qt;
    q.m = m_tokens;
    q.n = n;
    q.k = k;
    return phb::prefill_ws_bytes(q);
}

phb_status phb_gemm_q_prefill(int qtype, const void* W, const float* X, float* Y, int64_t m_tokens, int64_t n,
                              int64_t k, void* ws, size_t ws_bytes, phb_stream_t stream) {
    const int qt = qt_of(qtype);
    PHB_REQUIRE(qt >= 0, PHB_ERR_INVALID_ARG, "unknown qtype");
    PHB_REQUIRE(W && X && Y, PHB_ERR_INVALID_ARG, "null tensor pointer");
    PHB_REQUIRE(m_tokens >= 1 && m_tokens <= 4096, PHB_ERR_INVALID_ARG, "m_tokens must be 1..4096");
    PHB_REQUIRE(n > 0 && k > 0, PHB_ERR_INVALID_ARG, "n and k must be positive");
    PHB_REQUIRE(n % 128 == 0 && k % 256 == 0, PHB_ERR_SHAPE, "prefill needs n %% 128 == 0 and k %% 256 == 0");
    PHB_REQUIRE(n <= (int64_t{1} << 20) && k <= (int64_t{1} << 20), PHB_ERR_SHAPE, "shape too large");
    PHB_REQUIRE(aligned16(W) && aligned16(X) && aligned16(Y) && aligned16(ws), PHB_ERR_ALIGN,
                "tensors must be 16-byte aligned");
    const size_t need = phb_gemm_q_prefill_workspace_size(qtype, m_tokens, n, k);
    PHB_REQUIRE(ws && ws_bytes >= need, PHB_ERR_WORKSPACE, "workspace needs %zu bytes (got %zu)", need, ws_bytes);
    phb_status st = check_device();
    if (st != PHB_OK) return st;
    phb::PrefillReq q;
    q.qt = qt;
    q.w = W;
    q.x = X;
    q.y = Y;
    q.m = m_tokens;
    q.n = n;
    q.k = k;
    q.ws = ws;
    q.ws_bytes = ws_bytes;
    const cudaError_t e = phb::prefill_run(q, stream);
    if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
    return ok();
}

// ---------------------------------------------------------------- decode step
size_t phb_decode_step_workspace_size(int qtype, int64_t d_model, int n_q_heads, int n_kv_heads, int head_dim,
                                      int64_t d_ff) {
    if (qt_of(qtype) < 0 || d_model <= 0 || n_q_heads <= 0 || n_kv_heads <= 0 || head_dim <= 0 || d_ff <= 0) return 0;
    const size_t unfused = decode_ws(d_model, n_q_heads, n_kv_heads, head_dim, d_ff, nullptr).bytes;
    const size_t fused = phb::decode_persistent_ws_bytes(d_model, n_q_heads, n_kv_heads, head_dim, d_ff) +
                         2 * align256(static_cast<size_t>(d_model) * sizeof(float));
    return std::max(unfused, fused);
}

static phb_status validate_decode(int qt, const phb_dense_layer* layers, int n_layers, int64_t d_model, int n_q_heads,
                                  int n_kv_heads, int head_dim, int64_t d_ff, const float* x_in, float* x_out,
                                  void* ws, size_t ws_bytes) {
    PHB_REQUIRE(qt >= 0, PHB_ERR_INVALID_ARG, "unknown qtype");
    PHB_REQUIRE(layers && x_in && x_out, PHB_ERR_INVALID_ARG, "null pointer");
    PHB_REQUIRE(n_layers >= 1, PHB_ERR_INVALID_ARG, "n_layers must be positive");
    PHB_REQUIRE(d_model > 0 && n_q_heads > 0 && n_kv_heads > 0 && head_dim > 0 && d_ff > 0, PHB_ERR_INVALID_ARG,
                "sizes must be positive");
    PHB_REQUIRE(n_q_heads % n_kv_heads == 0, PHB_ERR_SHAPE, "n_q_heads must be a multiple of n_kv_heads");
    const int64_t q_dim = static_cast<int64_t>(n_q_heads) * head_dim;
    PHB_REQUIRE(d_model % 256 == 0 && q_dim % 256 == 0 && d_ff % 256 == 0, PHB_ERR_SHAPE,
                "decode step needs d_model, n_q_heads*head_dim and d_ff multiples of 256");
    PHB_REQUIRE(d_model <= 16384 && q_dim <= 16384 && d_ff <= 16384, PHB_ERR_SHAPE, "decode step sizes <= 16384");
    PHB_REQUIRE(x_in != x_out, PHB_ERR_INVALID_ARG, "x_in and x_out may not alias");
    PHB_REQUIRE(aligned16(x_in) && aligned16(x_out) && aligned16(ws), PHB_ERR_ALIGN, "pointers must be 16-byte aligned");
    for (int l = 0; l < n_layers; ++l) {
        const phb_dense_layer& L = layers[l];
        PHB_REQUIRE(L.w_qkv && L.w_o && L.w_gate && L.w_up && L.w_down, PHB_ERR_INVALID_ARG, "layer %d: null weight", l);
        PHB_REQUIRE(aligned16(L.w_qkv) && aligned16(L.w_o) && aligned16(L.w_gate) && aligned16(L.w_up) &&
                        aligned16(L.w_down),
                    PHB_ERR_ALIGN, "layer %d: weights must be 16-byte aligned", l);
    }
    const size_t need = phb_decode_step_workspace_size(qt == 0 ? PHB_Q8_0 : PHB_Q4_K, d_model, n_q_heads, n_kv_heads,
                                                       head_dim, d_ff);
    PHB_REQUIRE(ws && ws_bytes >= need, PHB_ERR_WORKSPACE, "workspace needs %zu bytes (got %zu)", need, ws_bytes);
    return PHB_OK;
}

phb_status phb_decode_step(int qtype, const phb_dense_layer* layers, int n_layers, int64_t d_model, int n_q_heads,
                           int n_kv_heads, int head_dim, int64_t d_ff, const float* x_in, float* x_out, void* ws,
                           size_t ws_bytes, phb_stream_t stream) {
    const int qt = qt_of(qtype);
    phb_status st = validate_decode(qt, layers, n_layers, d_model, n_q_heads, n_kv_heads, head_dim, d_ff, x_in, x_out,
                                    ws, ws_bytes);
    if (st != PHB_OK) return st;
    st = check_device();
    if (st != PHB_OK) return st;
    // one cooperative kernel per chunk of at most kPersistMaxLayers layers; the
    // chunks hand the residual stream over through two plain buffers at the
    // end of the workspace
    auto* base = static_cast<uint8_t*>(ws);
    const size_t pbytes = phb::decode_persistent_ws_bytes(d_model, n_q_heads, n_kv_heads, head_dim, d_ff);
    float* hand[2] = {reinterpret_cast<float*>(base + pbytes),
                      reinterpret_cast<float*>(base + pbytes + align256(static_cast<size_t>(d_model) * sizeof(float)))};
    const void* wl[5 * phb::kPersistMaxLayers];
    for (int l0 = 0, chunk = 0; l0 < n_layers; l0 += phb::kPersistMaxLayers, ++chunk) {
        const int nl = std::min(phb::kPersistMaxLayers, n_layers - l0);
        for (int l = 0; l < nl; ++l) {
            const phb_dense_layer& L = layers[l0 + l];
            wl[5 * l] = L.w_qkv;
            wl[5 * l + 1] = L.w_o;
            wl[5 * l + 2] = L.w_gate;
            wl[5 * l + 3] = L.w_up;
            wl[5 * l + 4] = L.w_down;
        }
        const float* in = l0 == 0 ? x_in : hand[(chunk - 1) & 1];
        float* out = l0 + nl == n_layers ? x_out : hand[chunk & 1];
        const cudaError_t e = phb::decode_persistent_run(qt, wl, nl, d_model, n_q_heads, n_kv_heads, head_dim, d_ff,
                                                         in, out, ws, stream);
        if (e == cudaErrorInvalidConfiguration) return fail(PHB_ERR_SHAPE, "shape does not fit the persistent decode kernel");
        if (e != cudaSuccess) return cuda_fail(e, "persistent decode launch");
    }
    return ok();
}

phb_status phb_decode_step_unfused(int qtype, const phb_dense_layer* layers, int n_layers, int64_t d_model,
                                   int n_q_heads, int n_kv_heads, int head_dim, int64_t d_ff, const float* x_in,
                                   float* x_out, void* ws, size_t ws_bytes, phb_stream_t stream) {
    const int qt = qt_of(qtype);
    phb_status st = validate_decode(qt, layers, n_layers, d_model, n_q_heads, n_kv_heads, head_dim, d_ff, x_in, x_out,
                                    ws, ws_bytes);
    if (st != PHB_OK) return st;
    st = check_device();
    if (st != PHB_OK) return st;
    const DecodeWs w = decode_ws(d_model, n_q_heads, n_kv_heads, head_dim, d_ff, ws);
    const int64_t q_dim = static_cast<int64_t>(n_q_heads) * head_dim;
    const int64_t qkv_dim = static_cast<int64_t>(n_q_heads + 2 * n_kv_heads) * head_dim;
    // GEMV launch ids for debug tracing builds. (Prefetching the weights of
    // GEMV i + 2 into L2 from GEMV i measured slightly slower here, so the
    // decode step issues no prefetch.)
    auto set_pf = [&](phb::GemvReq& q, int op) { q.trace_id = op; };
    for (int l = 0; l < n_layers; ++l) {
        const phb_dense_layer& L = layers[l];
        const float* in = l == 0 ? x_in : w.xs[(l - 1) & 1];
        float* out = l == n_layers - 1 ? x_out : w.xs[l & 1];
        // QKV = Wqkv . rmsnorm(x)
        phb::GemvReq q = gemv_req(qt, L.w_qkv, in, w.qkv, qkv_dim, d_model, 1);
        q.xmode = 1;
        set_pf(q, 4 * l);
        PHB_CUDA(phb::decode_gemv_run(q, stream), "decode qkv launch");
        // x1 = x + Wo . attn(qkv)
        q = gemv_req(qt, L.w_o, w.qkv, w.x1, d_model, q_dim, 1);
        q.xmode = 2;
        q.epi = 1;
        q.r = in;
        q.gather_group = n_q_heads / n_kv_heads;
        q.gather_hd = head_dim;
        q.gather_v_off = static_cast<int64_t>(n_q_heads + n_kv_heads) * head_dim;
        set_pf(q, 4 * l + 1);
        PHB_CUDA(phb::decode_gemv_run(q, stream), "decode o launch");
        // act = silu(Wg . rmsnorm(x1)) * (Wu . rmsnorm(x1))
        q = gemv_req(qt, L.w_gate, w.x1, w.act, d_ff, d_model, 1);
        q.nmat = 2;
        q.w1 = L.w_up;
        q.xmode = 1;
        q.epi = 2;
        set_pf(q, 4 * l + 2);
        PHB_CUDA(phb::decode_gemv_run(q, stream), "decode gate/up launch");
        // out = x1 + Wd . act
        q = gemv_req(qt, L.w_down, w.act, out, d_model, d_ff, 1);
        q.epi = 1;
        q.r = w.x1;
        set_pf(q, 4 * l + 3);
        PHB_CUDA(phb::decode_gemv_run(q, stream), "decode down launch");
    }
    return ok();
}

phb_status phb_decode_step_probe(int fused, int64_t d_model, int n_q_heads, int n_kv_heads, int head_dim,
                                 int64_t d_ff, const void* ws, float* qkv, float* x1, float* act,
                                 phb_stream_t stream) {
    PHB_REQUIRE(ws && qkv && x1 && act, PHB_ERR_INVALID_ARG, "null pointer");
    PHB_REQUIRE(d_model > 0 && n_q_heads > 0 && n_kv_heads > 0 && head_dim > 0 && d_ff > 0, PHB_ERR_INVALID_ARG,
                "sizes must be positive");
    PHB_REQUIRE(d_model <= 16384 && d_ff <= 16384 && static_cast<int64_t>(n_q_heads + 2 * n_kv_heads) * head_dim <= 65536,
                PHB_ERR_SHAPE, "decode step sizes out of range");
    PHB_REQUIRE(aligned16(ws), PHB_ERR_ALIGN, "workspace must be 16-byte aligned");
    phb_status st = check_device();
    if (st != PHB_OK) return st;
    if (fused) {
        PHB_CUDA(phb::decode_persistent_probe(ws, d_model, n_q_heads, n_kv_heads, head_dim, d_ff, qkv, x1, act, stream),
                 "probe launch");
        return ok();
    }
    const DecodeWs w = decode_ws(d_model, n_q_heads, n_kv_heads, head_dim, d_ff, const_cast<void*>(ws));
    const size_t nqkv = static_cast<size_t>(n_q_heads + 2 * n_kv_heads) * head_dim;
    PHB_CUDA(cudaMemcpyAsync(qkv, w.qkv, nqkv * sizeof(float), cudaMemcpyDeviceToDevice, stream), "probe copy");
    PHB_CUDA(cudaMemcpyAsync(x1, w.x1, static_cast<size_t>(d_model) * sizeof(float), cudaMemcpyDeviceToDevice, stream),
             "probe copy");
    PHB_CUDA(cudaMemcpyAsync(act, w.act, static_cast<size_t>(d_ff) * sizeof(float), cudaMemcpyDeviceToDevice, stream),
             "probe copy");
    return ok();
}

// ---------------------------------------------------------------- decode attention
static constexpr int64_t kAttnMaxCtx = int64_t{1} << 26;

size_t phb_attention_decode_workspace_size(int64_t n_ctx, int n_q_heads, int n_kv_heads, int head_dim) {
    if (n_ctx < 1 || n_ctx > kAttnMaxCtx || !phb::attention_shape_ok(n_q_heads, n_kv_heads, head_dim)) return 0;
    return phb::attention_ws_bytes(n_q_heads, n_kv_heads, head_dim, n_ctx);
}

phb_status phb_attention_decode(const float* q, const void* k_cache, const void* v_cache, float* out, int64_t n_ctx,
                                int n_q_heads, int n_kv_heads, int head_dim, float scale, void* ws, size_t ws_bytes,
                                phb_stream_t stream) {
    PHB_REQUIRE(q && k_cache && v_cache && out, PHB_ERR_INVALID_ARG, "null tensor pointer");
    PHB_REQUIRE(n_ctx >= 1 && n_ctx <= kAttnMaxCtx, PHB_ERR_INVALID_ARG, "n_ctx must be 1..2^26 (got %lld)",
                static_cast<long long>(n_ctx));
    PHB_REQUIRE(n_q_heads >= 1 && n_kv_heads >= 1, PHB_ERR_INVALID_ARG, "head counts must be positive");
    PHB_REQUIRE(n_q_heads % n_kv_heads == 0, PHB_ERR_SHAPE, "n_q_heads must be a multiple of n_kv_heads");
    PHB_REQUIRE(head_dim == 64 || head_dim == 128 || head_dim == 256, PHB_ERR_SHAPE,
                "head_dim must be 64, 128 or 256 (got %d)", head_dim);
    PHB_REQUIRE(std::isfinite(scale), PHB_ERR_INVALID_ARG, "scale must be finite");
    PHB_REQUIRE(aligned16(q) && aligned16(k_cache) && aligned16(v_cache) && aligned16(out) && aligned16(ws),
                PHB_ERR_ALIGN, "tensors must be 16-byte aligned");
    const size_t need = phb_attention_decode_workspace_size(n_ctx, n_q_heads, n_kv_heads, head_dim);
    PHB_REQUIRE(ws && ws_bytes >= need, PHB_ERR_WORKSPACE, "workspace needs %zu bytes (got %zu)", need, ws_bytes);
    phb_status st = check_device();
    if (st != PHB_OK) return st;
    const cudaError_t e = phb::attention_run(q, k_cache, v_cache, out, n_q_heads, n_kv_heads, head_dim, n_ctx, scale,
                                             ws, stream);
    if (e == cudaErrorInvalidConfiguration) return fail(PHB_ERR_SHAPE, "shape does not fit the attention kernels");
    if (e != cudaSuccess) return cuda_fail(e, "attention launch");
    return ok();
}

}  // extern "C"
