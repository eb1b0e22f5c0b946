// Quantized GEMV entry points: the streaming kernel in its plain and fused
// gate/up (SwiGLU) forms, a generic Q8_0 kernel for K not a multiple of 256,
// the split-K reduction and an elementwise SwiGLU.
#include <atomic>

#include "gemv_plan.cuh"
#include "phb_internal.h"

namespace phb {

int device_sm_count() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    const int slot = dev & 63;
    int v = cache[slot].load(std::memory_order_relaxed);
    if (v > 0) return v;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 1;
    cache[slot].store(v, std::memory_order_relaxed);
    return v;
}

cudaError_t read_dev_err_gemv(int* code) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_dev_err, sizeof(int));
    if (e != cudaSuccess) return e;
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_dev_err, &zero, sizeof(int));
    *code = v;
    return e;
}

// ---------------------------------------------------------------- generic Q8_0 GEMV
// One warp per row, lanes over blocks; 2-byte loads (Q8_0 blocks are only
// 2-byte aligned when K % 256 != 0). Used for shapes the streaming kernel
// does not take.
template <int MAXB>
__global__ void __launch_bounds__(256) gemv_q8_0_generic_kernel(const uint8_t* __restrict__ w, int64_t n, int64_t k,
                                                                int batch, const float* __restrict__ x, int64_t ldx,
                                                                float* __restrict__ y, int64_t ldy) {
    pdl_launch_dependents();
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + warp;
    if (row >= n) return;
    const int64_t nb = k / kQ8Weights;
    const uint8_t* wr = w + row * nb * kQ8Bytes;
    float acc[MAXB];
#pragma unroll
    for (int b = 0; b < MAXB; ++b) acc[b] = 0.f;
    for (int64_t blk = lane; blk < nb; blk += 32) {
        const uint16_t* bp = reinterpret_cast<const uint16_t*>(wr + blk * kQ8Bytes);
        const float d = fp16_bits_to_float(bp[0]);
        float s[MAXB];
#pragma unroll
        for (int b = 0; b < MAXB; ++b) s[b] = 0.f;
#pragma unroll 4
        for (int i = 0; i < 16; ++i) {
            const uint32_t two = bp[1 + i];
            const float q0 = static_cast<float>(static_cast<int8_t>(two & 0xFFu));
            const float q1 = static_cast<float>(static_cast<int8_t>(two >> 8));
#pragma unroll
            for (int b = 0; b < MAXB; ++b) {
                if (b < batch) {
                    const float* xb = x + b * ldx + blk * kQ8Weights + 2 * i;
                    s[b] = fmaf(q0, xb[0], s[b]);
                    s[b] = fmaf(q1, xb[1], s[b]);
                }
            }
        }
#pragma unroll
        for (int b = 0; b < MAXB; ++b) acc[b] = fmaf(d, s[b], acc[b]);
    }
#pragma unroll
    for (int b = 0; b < MAXB; ++b) {
        const float v = warp_sum(acc[b]);
        if (lane == 0 && b < batch) y[b * ldy + row] = v;
    }
}

// y[b][c] = sum over splits, ascending split index.
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float* __restrict__ part, float* __restrict__ y,
                                                            int64_t n, int batch, int ksplit, int64_t ldy) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= static_cast<int64_t>(batch) * n) return;
    const int64_t b = i / n, c = i - b * n;
    float s = 0.f;
    for (int sp = 0; sp < ksplit; ++sp) s += part[(static_cast<int64_t>(sp) * batch + b) * n + c];
    y[b * ldy + c] = s;
}

__global__ void __launch_bounds__(256) swiglu_kernel(const float* __restrict__ g, const float* __restrict__ u,
                                                     float* __restrict__ h, int64_t count) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= count) return;
    const float gv = g[i];
    h[i] = gv / (1.0f + expf(-gv)) * u[i];
}

cudaError_t swiglu_run(const float* g, const float* u, float* h, int64_t count, cudaStream_t s) {
    if (count <= 0) return cudaSuccess;
    return launch_kernel(swiglu_kernel, dim3(static_cast<unsigned>(cdiv(count, 256))), dim3(256), 0, s, true, g, u, h,
                         count);
}

// Batched plain GEMVs take the row-resident kernel (gemv_rows.cu). At batch 1
// the streaming kernel is as fast or faster (no split-K pass for short K).
static bool use_rows_kernel(const GemvReq& q) {
    return q.batch >= 2 && q.nmat == 1 && q.xmode == kXPlain && q.epi == kEpiStore && q.k % kUnitWeights == 0;
}

size_t gemv_ws_floats(const GemvReq& q) {
    if (q.k % kUnitWeights != 0) return 0;
    if (use_rows_kernel(q)) return gemv_rows_ws_floats(q.qt, q.n, q.k, q.batch);
    const int ks = plan_ksplit(q);
    return ks > 1 ? static_cast<size_t>(ks) * q.batch * q.n : 0;
}

template <int QT, int NMAT, int EPI>
static cudaError_t dispatch_maxb(const GemvPlan& pl, int maxb, cudaStream_t s, bool pdl) {
    switch (maxb) {
        case 1: return run_stream<QT, 1, NMAT, kXPlain, EPI>(pl, s, pdl);
        case 2: return run_stream<QT, 2, NMAT, kXPlain, EPI>(pl, s, pdl);
        case 4: return run_stream<QT, 4, NMAT, kXPlain, EPI>(pl, s, pdl);
        default: return run_stream<QT, 8, NMAT, kXPlain, EPI>(pl, s, pdl);
    }
}

template <int QT, int NMAT, int EPI>
static int ctas_per_sm_maxb(int maxb) {
    switch (maxb) {
        case 1: return stream_ctas_per_sm<QT, 1, NMAT, kXPlain, EPI>();
        case 2: return stream_ctas_per_sm<QT, 2, NMAT, kXPlain, EPI>();
        case 4: return stream_ctas_per_sm<QT, 4, NMAT, kXPlain, EPI>();
        default: return stream_ctas_per_sm<QT, 8, NMAT, kXPlain, EPI>();
    }
}

static int ctas_per_sm_for(int qt, int maxb, int nmat) {
    if (nmat == 2)
        return qt == 0 ? ctas_per_sm_maxb<0, 2, kEpiSwiGLU>(maxb) : ctas_per_sm_maxb<1, 2, kEpiSwiGLU>(maxb);
    return qt == 0 ? ctas_per_sm_maxb<0, 1, kEpiStore>(maxb) : ctas_per_sm_maxb<1, 1, kEpiStore>(maxb);
}

cudaError_t gemv_run(const GemvReq& q, cudaStream_t s) {
    const int maxb = maxb_for(q.batch);
    if (q.k % kUnitWeights != 0) {
        if (q.qt != 0 || q.nmat != 1 || q.xmode != kXPlain || q.epi != kEpiStore) return cudaErrorInvalidValue;
        const dim3 grid(static_cast<unsigned>(cdiv(q.n, 8)));
        const auto* w = static_cast<const uint8_t*>(q.w0);
        switch (maxb) {
            case 1: return launch_kernel(gemv_q8_0_generic_kernel<1>, grid, dim3(256), 0, s, q.pdl, w, q.n, q.k,
                                         q.batch, q.x, q.ldx, q.y, q.ldy);
            case 2: return launch_kernel(gemv_q8_0_generic_kernel<2>, grid, dim3(256), 0, s, q.pdl, w, q.n, q.k,
                                         q.batch, q.x, q.ldx, q.y, q.ldy);
            case 4: return launch_kernel(gemv_q8_0_generic_kernel<4>, grid, dim3(256), 0, s, q.pdl, w, q.n, q.k,
                                         q.batch, q.x, q.ldx, q.y, q.ldy);
            default: return launch_kernel(gemv_q8_0_generic_kernel<8>, grid, dim3(256), 0, s, q.pdl, w, q.n, q.k,
                                          q.batch, q.x, q.ldx, q.y, q.ldy);
        }
    }
    if (q.xmode != kXPlain) return cudaErrorInvalidValue;
    if (gemv_xr_fits(q)) return gemv_xr_run(q, s);
    if (use_rows_kernel(q)) {
        int ks = 1;
        cudaError_t e = gemv_rows_run(q, s, &ks);
        if (e != cudaSuccess || ks == 1) return e;
        const int64_t total = static_cast<int64_t>(q.batch) * q.n;
        return launch_kernel(splitk_reduce_kernel, dim3(static_cast<unsigned>(cdiv(total, 256))), dim3(256), 0, s,
                             q.pdl, static_cast<const float*>(q.ws), q.y, q.n, q.batch, ks, q.ldy);
    }
    GemvPlan pl;
    if (!plan_stream(q, &pl, ctas_per_sm_for(q.qt, maxb, q.nmat))) return cudaErrorInvalidConfiguration;
    const int ks = static_cast<int>(pl.grid.y);
    if (ks > 1 && (q.ws == nullptr || q.ws_floats < static_cast<size_t>(ks) * q.batch * q.n))
        return cudaErrorInvalidValue;
    cudaError_t e;
    if (q.nmat == 2) {
        if (ks != 1 || q.epi != kEpiSwiGLU) return cudaErrorInvalidValue;
        e = q.qt == 0 ? dispatch_maxb<0, 2, kEpiSwiGLU>(pl, maxb, s, q.pdl)
                      : dispatch_maxb<1, 2, kEpiSwiGLU>(pl, maxb, s, q.pdl);
    } else {
        if (q.epi != kEpiStore) return cudaErrorInvalidValue;
        e = q.qt == 0 ? dispatch_maxb<0, 1, kEpiStore>(pl, maxb, s, q.pdl)
                      : dispatch_maxb<1, 1, kEpiStore>(pl, maxb, s, q.pdl);
    }
    if (e != cudaSuccess || ks == 1) return e;
    const int64_t total = static_cast<int64_t>(q.batch) * q.n;
    return launch_kernel(splitk_reduce_kernel, dim3(static_cast<unsigned>(cdiv(total, 256))), dim3(256), 0, s, q.pdl,
                         static_cast<const float*>(q.ws), q.y, q.n, q.batch, ks, q.ldy);
}

}  // namespace phb
