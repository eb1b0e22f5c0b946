// SwiGLU feed-forward block without a caller-provided workspace.
//
// Some callers cannot allocate device memory: a serving loop that fixes its
// memory budget at start-up and forbids allocation afterwards, or a plugin
// that runs inside another runtime which owns every device allocation. For
// them this entry point runs the same computation as phb_ffn_swiglu with its
// scratch (the hidden activation and the down projection's split-K partials)
// in a fixed array compiled into the library. Every GPU that loads the
// library holds that array until the process exits.
#include <mutex>

#include "phb.h"
#include "phb_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t{2} << 20;  // 2 MiB

// The scratch. Host code may not use this name as a device address; the
// set-up below asks the runtime for the device address on each device.
static __device__ __align__(256) unsigned char g_ffn_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[64];  // device address of g_ffn_scratch per device ordinal

}  // namespace

extern "C" size_t phb_ffn_swiglu_noalloc_max_scratch(void) { return kNoAllocScratchBytes; }

extern "C" phb_status phb_ffn_swiglu_noalloc(int qtype, const void* Wgate, const void* Wup, const void* Wdown,
                                             const float* X, float* Y, int64_t d_model, int64_t d_ff, int batch,
                                             phb_stream_t stream) {
    // Bad arguments fail here, before anything touches a device.
    const phb_status st = phb::validate_ffn(qtype, Wgate, Wup, Wdown, X, Y, d_model, d_ff, batch);
    if (st != PHB_OK) return st;
    const size_t need = phb_ffn_swiglu_workspace_size(qtype, d_model, d_ff, batch);
    if (need > kNoAllocScratchBytes)
        return phb::set_last_error(PHB_ERR_WORKSPACE,
                                   "phb_ffn_swiglu_noalloc: this shape needs %zu bytes of scratch; the static "
                                   "scratch array holds %zu",
                                   need, kNoAllocScratchBytes);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return phb::set_last_error(PHB_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return phb::set_last_error(PHB_ERR_UNSUPPORTED_DEVICE, "device ordinal %d >= 64", dev);
    void* ptr = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (g_scratch_ptr[dev] == nullptr) {
            // set-up, once per device, with that device current
            void* p = nullptr;
            e = cudaGetSymbolAddress(&p, g_ffn_scratch);
            if (e != cudaSuccess || p == nullptr)
                return phb::set_last_error(PHB_ERR_CUDA, "cudaGetSymbolAddress of the scratch array: %s",
                                           cudaGetErrorString(e));
            g_scratch_ptr[dev] = p;
        }
        ptr = g_scratch_ptr[dev];
    }
    return phb_ffn_swiglu(qtype, Wgate, Wup, Wdown, X, Y, d_model, d_ff, batch, ptr, kNoAllocScratchBytes, stream);
}
