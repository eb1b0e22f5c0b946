// Streaming GEMV variants used by the dense decode step: RMSNorm fused into
// the activation staging (QKV and gate/up), the position-0 attention fused
// into the O projection's staging (each query head reads its KV head's V),
// and the residual add fused into the O and down projections' epilogues.
#include "gemv_plan.cuh"
#include "phb_internal.h"

namespace phb {

cudaError_t read_dev_err_decode(int* code) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_dev_err, sizeof(int));
    if (e != cudaSuccess) return e;
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_dev_err, &zero, sizeof(int));
    *code = v;
    return e;
}

PHB_TRACE_READER(phb_trace_read)  // debug builds: the decode kernels' stamps

template <int QT>
static cudaError_t decode_dispatch(const GemvReq& q, const GemvPlan& pl, cudaStream_t s) {
    if (q.nmat == 1 && q.xmode == kXRmsNorm && q.epi == kEpiStore)
        return run_stream<QT, 1, 1, kXRmsNorm, kEpiStore>(pl, s, q.pdl);
    if (q.nmat == 1 && q.xmode == kXGatherV && q.epi == kEpiResid)
        return run_stream<QT, 1, 1, kXGatherV, kEpiResid>(pl, s, q.pdl);
    if (q.nmat == 2 && q.xmode == kXRmsNorm && q.epi == kEpiSwiGLU)
        return run_stream<QT, 1, 2, kXRmsNorm, kEpiSwiGLU>(pl, s, q.pdl);
    if (q.nmat == 1 && q.xmode == kXPlain && q.epi == kEpiResid)
        return run_stream<QT, 1, 1, kXPlain, kEpiResid>(pl, s, q.pdl);
    return cudaErrorInvalidValue;
}

cudaError_t decode_gemv_run(const GemvReq& q, cudaStream_t s) {
    if (q.batch != 1 || q.k % kUnitWeights != 0) return cudaErrorInvalidValue;
    GemvPlan pl;
    if (!plan_stream(q, &pl) || pl.grid.y != 1) return cudaErrorInvalidConfiguration;
    return q.qt == 0 ? decode_dispatch<0>(q, pl, s) : decode_dispatch<1>(q, pl, s);
}

}  // namespace phb
