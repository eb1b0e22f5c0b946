// Prompt-processing GEMM (tcgen05). Placeholder until the tensor-core kernel lands.
#include "phb_internal.h"

namespace phb {

static __device__ int g_dev_err_prefill;

cudaError_t read_dev_err_prefill(int* code) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_dev_err_prefill, sizeof(int));
    *code = v;
    return e;
}

size_t prefill_ws_bytes(const PrefillReq& q) { return static_cast<size_t>(q.m) * q.k * 2 + 256; }

cudaError_t prefill_run(const PrefillReq&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace phb
