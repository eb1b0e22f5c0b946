// Device-side helpers shared by the kernels of libphb: block-format
// constants, fp16 decode, exact small-integer -> fp32 conversion, and inline
// PTX for mbarriers, bulk (TMA) copies, L2 prefetch and programmatic
// dependent launch on sm_103a.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace phb {

// ---------------------------------------------------------------- formats
constexpr int kQ8Weights = 32;     // weights per Q8_0 block
constexpr int kQ8Bytes = 34;       // fp16 d + 32 x int8
constexpr int kQ4Weights = 256;    // weights per Q4_K super-block
constexpr int kQ4Bytes = 144;      // d, dmin, scales[12], qs[128]
// A 256-weight "unit" is the smallest 16-byte aligned span of a row in both
// formats: 8 Q8_0 blocks (272 B) or one Q4_K block (144 B).
constexpr int kUnitWeights = 256;
template <int QT> struct Fmt;
template <> struct Fmt<0> { static constexpr int unit_bytes = 272; };  // Q8_0
template <> struct Fmt<1> { static constexpr int unit_bytes = 144; };  // Q4_K

// Device error codes written to a kernel's error word.
constexpr int kDevErrTimeout = 1;   // a bounded wait ran out
constexpr int kDevErrBadIndex = 2;  // an input index (a tiered expert's location) was out of range

// Upper bound on mbarrier polls before a wait is declared stuck (the wall
// clock bound kWaitLimitNs below normally ends a stuck wait first).
constexpr uint32_t kSpinLimit = 1u << 26;

__device__ __forceinline__ float fp16_bits_to_float(uint32_t bits16) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16 & 0xFFFFu)));
}

// Exact fp32 value of a byte 0..255 placed in byte `sel` of `word`:
// the pattern 0x4B0000bb is the float 2^23 + bb, so subtracting 2^23 + bias
// gives bb - bias exactly.
template <int SEL>
__device__ __forceinline__ float byte_to_float(uint32_t word, float magic_plus_bias) {
    const uint32_t bits = __byte_perm(word, 0x4B000000u, 0x7440u | SEL);
    return __uint_as_float(bits) - magic_plus_bias;
}
constexpr float kMagic = 8388608.0f;          // 2^23
constexpr float kMagicS8 = 8388608.0f + 128.f; // 2^23 + 128 (signed bytes stored xor 0x80)

// ---------------------------------------------------------------- PTX: smem / mbarrier
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Make mbarrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// One poll of phase `parity`; a thread whose phase is not yet complete may
// be suspended for up to about kSuspendHintNs before the call returns false.
constexpr uint32_t kSuspendHintNs = 20000;

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "n"(kSuspendHintNs)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wall-clock bound of any single wait.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// Bounded wait on phase `parity` of `bar`. Returns false (and records the
// timeout in *err) when the phase did not complete within kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* err) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 0; i < kSpinLimit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > kWaitLimitNs) break;
    }
    atomicExch(err, kDevErrTimeout);
    return false;
}

// Warp-wide bounded wait: lane 0 polls, the other lanes wait at the warp
// barrier, then every lane acquires the completed phase itself (one poll).
// All 32 lanes must call it.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity, int* err) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, err) ? 1 : 0;
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    if (!ok) return false;
    return mbar_wait(bar, parity, err);
}

// ---------------------------------------------------------------- PTX: bulk copies
// 1-D bulk copy global -> shared, completion counted in bytes on `bar`.
// dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Same, with an L2 eviction-priority hint (weights are read once per call).
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Fire-and-forget prefetch of [src, src+bytes) into L2 (bytes multiple of 16).
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// ---------------------------------------------------------------- PTX: PDL
// Wait until the grids this grid depends on have completed and their memory
// is visible (no-op when launched without programmatic serialization).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Allow the dependent grid to start launching.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

}  // namespace phb
