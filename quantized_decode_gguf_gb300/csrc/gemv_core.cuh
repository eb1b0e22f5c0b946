// Per-thread dequantize-and-dot routines of the streaming GEMV kernels.
//
// A thread owns one "half unit": 128 consecutive weights of one row, i.e.
// four Q8_0 blocks (136 bytes) or half of a Q4_K super-block (its 16-byte
// header plus 64 quant bytes). Quantized bytes sit in shared memory (staged
// by bulk copies); activations sit in shared memory as fp32.
//
// Exact integer -> fp32 conversion for free: an integer u in 0..255 placed
// alone in a 32-bit register is, read as fp32, the subnormal number
// u * 2^-149, exactly. The activations are staged pre-multiplied by 2^s
// (s chosen per activation row from its largest magnitude so nothing
// overflows), so one fma of the raw register with x * 2^s accumulates
// u * x * 2^(s-149) with ordinary fp32 rounding, and the block sum is
// scaled back by the exact power of two 2^(149-s). Per block:
//   Q8_0 (u = q + 128, the quant byte xor 0x80):
//        sum_i w_i x_i = d * (sum_i u_i x_i - 128 * sum_i x_i)
//   Q4_K (u = q):
//        sum_i w_i x_i = (d*sc_j) * sum_i q_i x_i - (dmin*m_j) * sum_i x_i
// with sum_i x_i of every 32-weight block precomputed once per call.
// Products are issued two at a time with the packed fp32 FMA of sm_100+.
#pragma once

#include "phb_common.cuh"

namespace phb {

// Byte SEL of w, zero-extended: read as fp32 it is the subnormal u * 2^-149.
template <int SEL>
__device__ __forceinline__ float byte_subnormal(uint32_t w) {
    return __uint_as_float(__byte_perm(w, 0u, 0x4440u | SEL));
}

__device__ __forceinline__ float byte_subnormal_rt(uint32_t w, int sel) {
    return __uint_as_float(__byte_perm(w, 0u, 0x4440u | static_cast<uint32_t>(sel)));
}

__device__ __forceinline__ float2 ffma2(float a0, float a1, float b0, float b1, float2 c) {
    return __ffma2_rn(make_float2(a0, a1), make_float2(b0, b1), c);
}

// Rows b >= batch of the staged activations are zero, so the loops below run
// over all MAXB rows without guards.
// Activation layout in shared memory: a pad of 4 floats after every 128, so
// consecutive half units start in different bank groups.
constexpr int kXPadEvery = 128;
constexpr int kXPad = 4;
__host__ __device__ constexpr int xpad_len(int k) { return k + (k / kXPadEvery) * kXPad; }
__device__ __forceinline__ int xpad_idx(int k) { return k + (k / kXPadEvery) * kXPad; }

// Dot of one Q8_0 half unit (4 blocks) with MAXB activation rows.
//   wsrc: 136 quantized bytes (8-byte aligned)
//   xs:   scaled activations of this half unit for row 0; row stride xstride
//   xsum: unscaled 32-sums of this half unit's 4 blocks for row 0; stride sstride
//   xfac: per-row 2^(149 - s)
template <int MAXB>
__device__ __forceinline__ void dot_q8_0_half(const uint8_t* wsrc, const float* xs, int xstride, const float* xsum,
                                              int sstride, const float* xfac, float (&acc)[MAXB]) {
    uint32_t wd[34];
#pragma unroll
    for (int i = 0; i < 17; ++i) {
        const uint2 v = *reinterpret_cast<const uint2*>(wsrc + 8 * i);
        wd[2 * i] = v.x;
        wd[2 * i + 1] = v.y;
    }
    uint32_t wx[34];
#pragma unroll
    for (int i = 0; i < 34; ++i) wx[i] = wd[i] ^ 0x80808080u;
#pragma unroll
    for (int bb = 0; bb < 4; ++bb) {
        const int ob = 34 * bb;  // compile-time after unrolling
        const float d = fp16_bits_to_float((ob % 4) ? (wd[ob / 4] >> 16) : wd[ob / 4]);
        float2 s2[MAXB];
#pragma unroll
        for (int b = 0; b < MAXB; ++b) s2[b] = make_float2(0.f, 0.f);
#pragma unroll
        for (int i4 = 0; i4 < 8; ++i4) {
            float q[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int p = ob + 2 + 4 * i4 + t;
                q[t] = byte_subnormal_rt(wx[p / 4], p % 4);
            }
#pragma unroll
            for (int b = 0; b < MAXB; ++b) {
                const float4 xv = *reinterpret_cast<const float4*>(xs + b * xstride + 32 * bb + 4 * i4);
                s2[b] = ffma2(q[0], q[1], xv.x, xv.y, s2[b]);
                s2[b] = ffma2(q[2], q[3], xv.z, xv.w, s2[b]);
            }
        }
#pragma unroll
        for (int b = 0; b < MAXB; ++b) {
            const float su = s2[b].x + s2[b].y;
            const float blk = fmaf(su, xfac[b], -128.f * xsum[b * sstride + bb]);
            acc[b] = fmaf(d, blk, acc[b]);
        }
    }
}

// dot_q8_0_half for one activation row held in registers: xr the half
// unit's 128 scaled activations, xsr its four unscaled 32-sums. A thread that
// keeps xr across many rows reads only weights from shared memory. Same
// arithmetic, in the same order, as dot_q8_0_half with MAXB = 1.
__device__ __forceinline__ float dot_q8_0_half_xr(const uint8_t* wsrc, const float (&xr)[128], const float (&xsr)[4],
                                                  float xfac) {
    uint32_t wd[34];
#pragma unroll
    for (int i = 0; i < 17; ++i) {
        const uint2 v = *reinterpret_cast<const uint2*>(wsrc + 8 * i);
        wd[2 * i] = v.x;
        wd[2 * i + 1] = v.y;
    }
    float acc = 0.f;
#pragma unroll
    for (int bb = 0; bb < 4; ++bb) {
        const int ob = 34 * bb;
        const float d = fp16_bits_to_float((ob % 4) ? (wd[ob / 4] >> 16) : wd[ob / 4]);
        float2 s2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int i4 = 0; i4 < 8; ++i4) {
            float q[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int p = ob + 2 + 4 * i4 + t;
                q[t] = byte_subnormal_rt(wd[p / 4] ^ 0x80808080u, p % 4);
            }
            const int k = 32 * bb + 4 * i4;
            s2 = ffma2(q[0], q[1], xr[k], xr[k + 1], s2);
            s2 = ffma2(q[2], q[3], xr[k + 2], xr[k + 3], s2);
        }
        const float su = s2.x + s2.y;
        const float blk = fmaf(su, xfac, -128.f * xsr[bb]);
        acc = fmaf(d, blk, acc);
    }
    return acc;
}

// 6-bit scale and min of sub-block 4h + jj from the 12 scale bytes (packed
// little-endian in sw[0..2]); branch-free in h.
__device__ __forceinline__ void q4_k_scale_min_half(const uint32_t (&sw)[3], int h, int jj, uint32_t& sc, uint32_t& m) {
    auto sb = [&](int i) -> uint32_t { return (sw[i >> 2] >> (8 * (i & 3))) & 0xFFu; };
    const uint32_t a = sb(jj), b4 = sb(jj + 4), c8 = sb(jj + 8);
    const uint32_t sc0 = a & 63u, m0 = b4 & 63u;
    const uint32_t sc1 = (c8 & 15u) | ((a >> 6) << 4), m1 = (c8 >> 4) | ((b4 >> 6) << 4);
    sc = h ? sc1 : sc0;
    m = h ? m1 : m0;
}

// General form used by the dequantisation kernel: sub-block j of 0..7.
__device__ __forceinline__ void q4_k_scale_min(const uint32_t (&sw)[3], int j, uint32_t& sc, uint32_t& m) {
    q4_k_scale_min_half(sw, j >> 2, j & 3, sc, m);
}

// Dot of one Q4_K half super-block (sub-blocks 4h..4h+3) with MAXB rows.
//   blk:  the 144-byte block (16-byte aligned)
//   xs, xsum, xfac: as for Q8_0 (xsum points at sub-block 4h of the block)
template <int MAXB>
__device__ __forceinline__ void dot_q4_k_half(const uint8_t* blk, int h, const float* xs, int xstride,
                                              const float* xsum, int sstride, const float* xfac, float (&acc)[MAXB]) {
    const uint4 hdr = *reinterpret_cast<const uint4*>(blk);
    const float d = fp16_bits_to_float(hdr.x);
    const float dmin = fp16_bits_to_float(hdr.x >> 16);
    const uint32_t sw[3] = {hdr.y, hdr.z, hdr.w};
    uint32_t qw[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint4 v = *reinterpret_cast<const uint4*>(blk + 16 + 64 * h + 16 * i);
        qw[4 * i] = v.x;
        qw[4 * i + 1] = v.y;
        qw[4 * i + 2] = v.z;
        qw[4 * i + 3] = v.w;
    }
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
        float2 slo[MAXB], shi[MAXB];
#pragma unroll
        for (int b = 0; b < MAXB; ++b) slo[b] = shi[b] = make_float2(0.f, 0.f);
#pragma unroll
        for (int wi = 0; wi < 8; ++wi) {
            const uint32_t w = qw[8 * cc + wi];
            const uint32_t lo = w & 0x0F0F0F0Fu;
            const uint32_t hi = (w >> 4) & 0x0F0F0F0Fu;
            const float l0 = byte_subnormal<0>(lo), l1 = byte_subnormal<1>(lo);
            const float l2 = byte_subnormal<2>(lo), l3 = byte_subnormal<3>(lo);
            const float h0 = byte_subnormal<0>(hi), h1 = byte_subnormal<1>(hi);
            const float h2 = byte_subnormal<2>(hi), h3 = byte_subnormal<3>(hi);
#pragma unroll
            for (int b = 0; b < MAXB; ++b) {
                const float4 xl = *reinterpret_cast<const float4*>(xs + b * xstride + 64 * cc + 4 * wi);
                const float4 xh = *reinterpret_cast<const float4*>(xs + b * xstride + 64 * cc + 32 + 4 * wi);
                slo[b] = ffma2(l0, l1, xl.x, xl.y, slo[b]);
                slo[b] = ffma2(l2, l3, xl.z, xl.w, slo[b]);
                shi[b] = ffma2(h0, h1, xh.x, xh.y, shi[b]);
                shi[b] = ffma2(h2, h3, xh.z, xh.w, shi[b]);
            }
        }
        uint32_t sc_l, m_l, sc_h, m_h;
        q4_k_scale_min_half(sw, h, 2 * cc, sc_l, m_l);
        q4_k_scale_min_half(sw, h, 2 * cc + 1, sc_h, m_h);
        const float dl = d * static_cast<float>(sc_l), ml = dmin * static_cast<float>(m_l);
        const float dh = d * static_cast<float>(sc_h), mh = dmin * static_cast<float>(m_h);
#pragma unroll
        for (int b = 0; b < MAXB; ++b) {
            const float ql = (slo[b].x + slo[b].y) * xfac[b];
            const float qh = (shi[b].x + shi[b].y) * xfac[b];
            acc[b] = fmaf(dl, ql, acc[b]);
            acc[b] = fmaf(-ml, xsum[b * sstride + 2 * cc], acc[b]);
            acc[b] = fmaf(dh, qh, acc[b]);
            acc[b] = fmaf(-mh, xsum[b * sstride + 2 * cc + 1], acc[b]);
        }
    }
}

// dot_q4_k_half for one activation row held in registers (see
// dot_q8_0_half_xr); same arithmetic, in the same order, as MAXB = 1.
__device__ __forceinline__ float dot_q4_k_half_xr(const uint8_t* blk, int h, const float (&xr)[128],
                                                  const float (&xsr)[4], float xfac) {
    const uint4 hdr = *reinterpret_cast<const uint4*>(blk);
    const float d = fp16_bits_to_float(hdr.x);
    const float dmin = fp16_bits_to_float(hdr.x >> 16);
    const uint32_t sw[3] = {hdr.y, hdr.z, hdr.w};
    uint32_t qw[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint4 v = *reinterpret_cast<const uint4*>(blk + 16 + 64 * h + 16 * i);
        qw[4 * i] = v.x;
        qw[4 * i + 1] = v.y;
        qw[4 * i + 2] = v.z;
        qw[4 * i + 3] = v.w;
    }
    float acc = 0.f;
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
        float2 slo = make_float2(0.f, 0.f), shi = make_float2(0.f, 0.f);
#pragma unroll
        for (int wi = 0; wi < 8; ++wi) {
            const uint32_t w = qw[8 * cc + wi];
            const uint32_t lo = w & 0x0F0F0F0Fu;
            const uint32_t hi = (w >> 4) & 0x0F0F0F0Fu;
            const int kl = 64 * cc + 4 * wi, kh = kl + 32;
            slo = ffma2(byte_subnormal<0>(lo), byte_subnormal<1>(lo), xr[kl], xr[kl + 1], slo);
            slo = ffma2(byte_subnormal<2>(lo), byte_subnormal<3>(lo), xr[kl + 2], xr[kl + 3], slo);
            shi = ffma2(byte_subnormal<0>(hi), byte_subnormal<1>(hi), xr[kh], xr[kh + 1], shi);
            shi = ffma2(byte_subnormal<2>(hi), byte_subnormal<3>(hi), xr[kh + 2], xr[kh + 3], shi);
        }
        uint32_t sc_l, m_l, sc_h, m_h;
        q4_k_scale_min_half(sw, h, 2 * cc, sc_l, m_l);
        q4_k_scale_min_half(sw, h, 2 * cc + 1, sc_h, m_h);
        const float dl = d * static_cast<float>(sc_l), ml = dmin * static_cast<float>(m_l);
        const float dh = d * static_cast<float>(sc_h), mh = dmin * static_cast<float>(m_h);
        const float ql = (slo.x + slo.y) * xfac;
        const float qh = (shi.x + shi.y) * xfac;
        acc = fmaf(dl, ql, acc);
        acc = fmaf(-ml, xsr[2 * cc], acc);
        acc = fmaf(dh, qh, acc);
        acc = fmaf(-mh, xsr[2 * cc + 1], acc);
    }
    return acc;
}

}  // namespace phb
