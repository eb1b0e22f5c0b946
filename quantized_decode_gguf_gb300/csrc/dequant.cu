// Dequantisation kernels: Q8_0 / Q4_K blocks -> fp32 or bf16 weights.
//
// Bit-exact with the closed forms: for Q8_0, d*q is exact in fp32; for Q4_K,
// D = d*sc, M = dmin*m and D*q are exact in fp32, so the explicitly rounded
// product-then-subtract below performs the single rounding the format
// defines. bf16 output rounds that fp32 value to nearest even.
#include <cuda_bf16.h>

#include "gemv_core.cuh"
#include "phb_internal.h"

namespace phb {

namespace {

template <bool BF16>
__device__ __forceinline__ void store8(void* dst, const float (&v)[8]) {
    if constexpr (BF16) {
        uint32_t pk[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 t = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
            pk[i] = *reinterpret_cast<const uint32_t*>(&t);
        }
        *reinterpret_cast<uint4*>(dst) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    } else {
        float4* o = reinterpret_cast<float4*>(dst);
        o[0] = make_float4(v[0], v[1], v[2], v[3]);
        o[1] = make_float4(v[4], v[5], v[6], v[7]);
    }
}

// One thread per 8 weights (a quarter of a 34-byte block).
template <bool BF16>
__global__ void __launch_bounds__(256) dequant_q8_0_kernel(const uint8_t* __restrict__ blocks, void* __restrict__ w,
                                                           int64_t total_quarters) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < total_quarters; t += stride) {
        const int64_t blk = t >> 2;
        const int qtr = static_cast<int>(t & 3);
        const uint16_t* bp = reinterpret_cast<const uint16_t*>(blocks + blk * kQ8Bytes);
        const float d = fp16_bits_to_float(bp[0]);
        float v[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t two = bp[1 + 4 * qtr + i];
            v[2 * i] = d * static_cast<float>(static_cast<int8_t>(two & 0xFFu));
            v[2 * i + 1] = d * static_cast<float>(static_cast<int8_t>(two >> 8));
        }
        const int64_t widx = blk * kQ8Weights + 8 * qtr;
        if constexpr (BF16)
            store8<true>(static_cast<__nv_bfloat16*>(w) + widx, v);
        else
            store8<false>(static_cast<float*>(w) + widx, v);
    }
}

// One thread per 16 weights (half a sub-block) of a 144-byte super-block.
template <bool BF16>
__global__ void __launch_bounds__(256) dequant_q4_k_kernel(const uint8_t* __restrict__ blocks, void* __restrict__ w,
                                                           int64_t total_segs) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < total_segs; t += stride) {
        const int64_t blk = t >> 4;
        const int seg = static_cast<int>(t & 15);
        const int j = seg >> 1;        // sub-block
        const int hh = seg & 1;        // which 16 of its 32 weights
        const uint8_t* bp = blocks + blk * kQ4Bytes;
        const uint4 hdr = *reinterpret_cast<const uint4*>(bp);
        const uint4 qv = *reinterpret_cast<const uint4*>(bp + 16 + 32 * (j >> 1) + 16 * hh);
        const uint32_t sw[3] = {hdr.y, hdr.z, hdr.w};
        uint32_t sc, m;
        q4_k_scale_min(sw, j, sc, m);
        const float dd = __fmul_rn(fp16_bits_to_float(hdr.x), static_cast<float>(sc));
        const float mm = __fmul_rn(fp16_bits_to_float(hdr.x >> 16), static_cast<float>(m));
        const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w};
        const int shift = (j & 1) ? 4 : 0;
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const uint32_t q = (qw[i >> 2] >> (8 * (i & 3) + shift)) & 15u;
            v[i] = __fsub_rn(__fmul_rn(dd, static_cast<float>(q)), mm);
        }
        const int64_t widx = blk * kQ4Weights + 32 * j + 16 * hh;
        float lo[8], hi[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            lo[i] = v[i];
            hi[i] = v[8 + i];
        }
        if constexpr (BF16) {
            store8<true>(static_cast<__nv_bfloat16*>(w) + widx, lo);
            store8<true>(static_cast<__nv_bfloat16*>(w) + widx + 8, hi);
        } else {
            store8<false>(static_cast<float*>(w) + widx, lo);
            store8<false>(static_cast<float*>(w) + widx + 8, hi);
        }
    }
}

}  // namespace

cudaError_t dequant_run(int qt, bool bf16, const void* blocks, void* w, int64_t n, int64_t k, cudaStream_t s) {
    const auto* b = static_cast<const uint8_t*>(blocks);
    const int64_t work = qt == 0 ? n * (k / kQ8Weights) * 4 : n * (k / kQ4Weights) * 16;
    if (work == 0) return cudaSuccess;
    const int64_t cap = static_cast<int64_t>(device_sm_count()) * 16;
    const unsigned grid = static_cast<unsigned>(std::min<int64_t>(cap, (work + 255) / 256));
    if (qt == 0)
        return bf16 ? launch_kernel(dequant_q8_0_kernel<true>, dim3(grid), dim3(256), 0, s, true, b, w, work)
                    : launch_kernel(dequant_q8_0_kernel<false>, dim3(grid), dim3(256), 0, s, true, b, w, work);
    return bf16 ? launch_kernel(dequant_q4_k_kernel<true>, dim3(grid), dim3(256), 0, s, true, b, w, work)
                : launch_kernel(dequant_q4_k_kernel<false>, dim3(grid), dim3(256), 0, s, true, b, w, work);
}

}  // namespace phb
