// Debug-only timeline stamps, compiled in with -DPHB_TRACE and out otherwise.
//
//   PHB_TRACE_EV(id, ev)    the executing CTA stores the global timer as event
//                           ev (< 16) of launch id (< 128); CTAs are numbered
//                           linearly over the grid, the first 160 are kept
//   PHB_TRACE_READER(name)  defines extern "C" int name(void* dst, size_t bytes),
//                           which copies this translation unit's stamps out
//
// In normal builds both expand to nothing.
#pragma once

#include <cstdint>

#include "phb_common.cuh"

#ifdef PHB_TRACE
namespace phb {
constexpr int kTraceLaunches = 128, kTraceCtas = 160, kTraceEvents = 16;
static __device__ uint64_t g_trace[kTraceLaunches * kTraceCtas * kTraceEvents];
}  // namespace phb
#define PHB_TRACE_EV(id, ev)                                                                              \
    do {                                                                                                  \
        const unsigned c_ = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);               \
        if ((id) >= 0 && (id) < ::phb::kTraceLaunches && c_ < ::phb::kTraceCtas)                          \
            ::phb::g_trace[((id) * ::phb::kTraceCtas + c_) * ::phb::kTraceEvents + (ev)] =                \
                ::phb::global_timer_ns();                                                                 \
    } while (0)
#define PHB_TRACE_READER(name)                                                                            \
    extern "C" int name(void* dst, size_t bytes) {                                                        \
        if (bytes > sizeof(::phb::g_trace)) bytes = sizeof(::phb::g_trace);                               \
        return static_cast<int>(cudaMemcpyFromSymbol(dst, ::phb::g_trace, bytes));                        \
    }
#else
#define PHB_TRACE_EV(id, ev) \
    do {                     \
    } while (0)
#define PHB_TRACE_READER(name)
#endif
