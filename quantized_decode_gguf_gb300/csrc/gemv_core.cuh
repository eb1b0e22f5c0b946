// Per-thread dequantize-and-dot routines of the streaming GEMV kernels.
//
// A thread owns one "half unit": 128 consecutive weights of one row, i.e.
// four Q8_0 blocks (136 bytes) or half of a Q4_K super-block (its 16-byte
// header plus 64 quant bytes). Quantized bytes sit in shared memory (staged
// by bulk copies); activations sit in shared memory or registers as fp32.
//
// Every weight enters the dot exactly as the dequantiser forms it, times the
// constant 2^-85, so the result is an ordinary fp32 dot product of the exact
// dequantised weights with the activations:
//  - an integer u in 0..255 placed alone in a 32-bit register is, read as
//    fp32, the subnormal u * 2^-149, exactly (one byte permute, no convert);
//  - one fused multiply-add per weight then forms the scaled weight:
//      Q8_0 (u = q + 128, the quant byte xor 0x80):
//        fma(d * 2^64, u * 2^-149, -d * 2^-78) = d * q * 2^-85
//      Q4_K (u = q):
//        fma(d*sc_j * 2^64, u * 2^-149, -(dmin*m_j) * 2^-85) = (d*sc_j*q - dmin*m_j) * 2^-85
//    The product is exact inside the fma and the sum is rounded once: for
//    Q8_0 d*q has at most 18 significant bits, so nothing rounds; for Q4_K
//    the single rounding is the one the dequantiser performs, so the scaled
//    weight is the dequantised fp32 weight times 2^-85, bit for bit. Every
//    nonzero weight is a multiple of 2^-24 below 2^27, so its scaled copy
//    is a normal number (no underflow), and a zero weight is exactly zero;
//  - a second packed fma per weight pair accumulates w * 2^-85 * x * 2^s,
//    with the activations staged pre-multiplied by a power of two 2^s chosen
//    from their largest magnitude (no overflow, no early underflow); the
//    half-unit sum is scaled back by the exact power of two 2^(85 - s).
// Hence each output obeys the textbook bound of an fp32 sum of products,
// |err| <= ~(n_terms) * 2^-24 * sum|w x| (n_terms the longest chain of
// roundings a term goes through), and a row whose terms are all zero gives
// exactly zero. Products are issued two at a time with the packed fp32 FMA
// of sm_100+.
#pragma once

#include "phb_common.cuh"

namespace phb {

// Scaled weights are w * 2^-kWShift; staged activations carry 2^s; the
// half-unit sums are scaled back by xfac = 2^(kWShift - s).
constexpr int kWShift = 85;

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

// Two scaled weights fma(a, u, c) at once.
__device__ __forceinline__ float2 wpair(float a, float u0, float u1, float c) {
    return __ffma2_rn(make_float2(a, a), make_float2(u0, u1), make_float2(c, c));
}

// Multipliers of one Q8_0 block with scale d: a = d * 2^64 and c = -d * 2^-78
// (= -128 * a * 2^-149). Both are exact: fp16 values lie in [2^-24, 2^16).
__device__ __forceinline__ void q8_0_mult(float d, float& a, float& c) {
    a = d * 0x1p64f;
    c = d * -0x1p-78f;
}

// Rows b >= batch of the staged activations are zero, so the loops below run
// over all MAXB rows without guards.
// Activation layout in shared memory: a pad of 4 floats after every 128, so
// consecutive half units start in different bank groups.
constexpr int kXPadEvery = 128;
constexpr int kXPad = 4;
__host__ __device__ constexpr int xpad_len(int k) { return k + (k / kXPadEvery) * kXPad; }
__device__ __forceinline__ int xpad_idx(int k) { return k + (k / kXPadEvery) * kXPad; }

// Dot of one Q8_0 half unit (4 blocks) with MAXB activation rows, added to
// acc[b] after scaling by xfac[b].
//   wsrc: 136 quantized bytes (8-byte aligned)
//   xs:   scaled activations of this half unit for row 0; row stride xstride
//   xfac: per-row 2^(kWShift - s)
template <int MAXB>
__device__ __forceinline__ void dot_q8_0_half(const uint8_t* wsrc, const float* xs, int xstride, const float* xfac,
                                              float (&acc)[MAXB]) {
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
    float2 s2[MAXB];
#pragma unroll
    for (int b = 0; b < MAXB; ++b) s2[b] = make_float2(0.f, 0.f);
#pragma unroll
    for (int bb = 0; bb < 4; ++bb) {
        const int ob = 34 * bb;  // compile-time after unrolling
        float a, c;
        q8_0_mult(fp16_bits_to_float((ob % 4) ? (wd[ob / 4] >> 16) : wd[ob / 4]), a, c);
#pragma unroll
        for (int i4 = 0; i4 < 8; ++i4) {
            float u[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int p = ob + 2 + 4 * i4 + t;
                u[t] = byte_subnormal_rt(wx[p / 4], p % 4);
            }
            const float2 w01 = wpair(a, u[0], u[1], c);
            const float2 w23 = wpair(a, u[2], u[3], c);
#pragma unroll
            for (int b = 0; b < MAXB; ++b) {
                const float4 xv = *reinterpret_cast<const float4*>(xs + b * xstride + 32 * bb + 4 * i4);
                s2[b] = __ffma2_rn(w01, make_float2(xv.x, xv.y), s2[b]);
                s2[b] = __ffma2_rn(w23, make_float2(xv.z, xv.w), s2[b]);
            }
        }
    }
#pragma unroll
    for (int b = 0; b < MAXB; ++b) acc[b] = fmaf(s2[b].x + s2[b].y, xfac[b], acc[b]);
}

// dot_q8_0_half for one activation row held in registers: xr the half
// unit's 128 scaled activations. A thread that keeps xr across many rows
// reads only weights from shared memory. The same exact scaled weights as
// dot_q8_0_half, summed in two interleaved accumulators (weights 4i, 4i+1
// and 4i+2, 4i+3) so that consecutive fused multiply-adds do not wait on
// each other; returns the scaled-back sum.
__device__ __forceinline__ float dot_q8_0_half_xr(const uint8_t* wsrc, const float (&xr)[128], float xfac) {
    uint32_t wd[34];
#pragma unroll
    for (int i = 0; i < 17; ++i) {
        const uint2 v = *reinterpret_cast<const uint2*>(wsrc + 8 * i);
        wd[2 * i] = v.x;
        wd[2 * i + 1] = v.y;
    }
    float2 s2 = make_float2(0.f, 0.f), t2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int bb = 0; bb < 4; ++bb) {
        const int ob = 34 * bb;
        float a, c;
        q8_0_mult(fp16_bits_to_float((ob % 4) ? (wd[ob / 4] >> 16) : wd[ob / 4]), a, c);
#pragma unroll
        for (int i4 = 0; i4 < 8; ++i4) {
            float u[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int p = ob + 2 + 4 * i4 + t;
                u[t] = byte_subnormal_rt(wd[p / 4] ^ 0x80808080u, p % 4);
            }
            const int k = 32 * bb + 4 * i4;
            s2 = __ffma2_rn(wpair(a, u[0], u[1], c), make_float2(xr[k], xr[k + 1]), s2);
            t2 = __ffma2_rn(wpair(a, u[2], u[3], c), make_float2(xr[k + 2], xr[k + 3]), t2);
        }
    }
    return ((s2.x + s2.y) + (t2.x + t2.y)) * xfac;
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

// Multipliers of the four sub-blocks 4h..4h+3 of a Q4_K block header, with
// the scale and min bytes extracted word-wide: for h = 0 the low 6 bits of
// scale bytes 0-3 (scales) and 4-7 (mins); for h = 1 the low (scales) or high
// (mins) nibbles of bytes 8-11 with bits 6-7 of bytes 0-3 (scales) or 4-7
// (mins) on top. A 6-bit value v in byte jj of a word becomes the float v
// exactly as (2^23 + v) - 2^23.
__device__ __forceinline__ void q4_k_half_mults(const uint4& hdr, int h, float (&a)[4], float (&c)[4]) {
    const float d = fp16_bits_to_float(hdr.x);
    const float dmin = fp16_bits_to_float(hdr.x >> 16);
    const uint32_t sc0 = hdr.y & 0x3F3F3F3Fu, m0 = hdr.z & 0x3F3F3F3Fu;
    const uint32_t sc1 = (hdr.w & 0x0F0F0F0Fu) | ((hdr.y >> 2) & 0x30303030u);
    const uint32_t m1 = ((hdr.w >> 4) & 0x0F0F0F0Fu) | ((hdr.z >> 2) & 0x30303030u);
    const uint32_t scb = h ? sc1 : sc0, mb = h ? m1 : m0;
    const float ds = d * 0x1p64f, dm = dmin * -0x1p-85f;
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
        const float scf = __uint_as_float(__byte_perm(scb, 0x4B000000u, 0x7440u | jj)) - 8388608.0f;
        const float mf = __uint_as_float(__byte_perm(mb, 0x4B000000u, 0x7440u | jj)) - 8388608.0f;
        a[jj] = ds * scf;  // d * sc * 2^64, exact
        c[jj] = dm * mf;   // -dmin * m * 2^-85, exact
    }
}

// Dot of one Q4_K half super-block (sub-blocks 4h..4h+3) with MAXB rows.
//   blk:  the 144-byte block (16-byte aligned)
//   xs, xfac: as for Q8_0
// Quant byte i of 64-weight chunk cc holds weight i of sub-block 2cc in its
// low nibble and weight i of sub-block 2cc + 1 in its high nibble. The high
// nibbles are masked in place (the byte is then 16 q) and the factor 1/16
// goes into that sub-block's multiplier, which stays exact.
template <int MAXB>
__device__ __forceinline__ void dot_q4_k_half(const uint8_t* blk, int h, const float* xs, int xstride,
                                              const float* xfac, float (&acc)[MAXB]) {
    const uint4 hdr = *reinterpret_cast<const uint4*>(blk);
    float a[4], c[4];
    q4_k_half_mults(hdr, h, a, c);
    uint32_t qw[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint4 v = *reinterpret_cast<const uint4*>(blk + 16 + 64 * h + 16 * i);
        qw[4 * i] = v.x;
        qw[4 * i + 1] = v.y;
        qw[4 * i + 2] = v.z;
        qw[4 * i + 3] = v.w;
    }
    float2 s2[MAXB];
#pragma unroll
    for (int b = 0; b < MAXB; ++b) s2[b] = make_float2(0.f, 0.f);
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
        const float al = a[2 * cc], cl = c[2 * cc], ah = a[2 * cc + 1] * 0.0625f, ch = c[2 * cc + 1];
#pragma unroll
        for (int wi = 0; wi < 8; ++wi) {
            const uint32_t w = qw[8 * cc + wi];
            const uint32_t lo = w & 0x0F0F0F0Fu;
            const uint32_t hi = w & 0xF0F0F0F0u;
            const float2 l01 = wpair(al, byte_subnormal<0>(lo), byte_subnormal<1>(lo), cl);
            const float2 l23 = wpair(al, byte_subnormal<2>(lo), byte_subnormal<3>(lo), cl);
            const float2 h01 = wpair(ah, byte_subnormal<0>(hi), byte_subnormal<1>(hi), ch);
            const float2 h23 = wpair(ah, byte_subnormal<2>(hi), byte_subnormal<3>(hi), ch);
#pragma unroll
            for (int b = 0; b < MAXB; ++b) {
                const float4 xl = *reinterpret_cast<const float4*>(xs + b * xstride + 64 * cc + 4 * wi);
                const float4 xh = *reinterpret_cast<const float4*>(xs + b * xstride + 64 * cc + 32 + 4 * wi);
                s2[b] = __ffma2_rn(l01, make_float2(xl.x, xl.y), s2[b]);
                s2[b] = __ffma2_rn(l23, make_float2(xl.z, xl.w), s2[b]);
                s2[b] = __ffma2_rn(h01, make_float2(xh.x, xh.y), s2[b]);
                s2[b] = __ffma2_rn(h23, make_float2(xh.z, xh.w), s2[b]);
            }
        }
    }
#pragma unroll
    for (int b = 0; b < MAXB; ++b) acc[b] = fmaf(s2[b].x + s2[b].y, xfac[b], acc[b]);
}

// dot_q4_k_half for one activation row held in registers (see
// dot_q8_0_half_xr): the same exact scaled weights, the low-nibble and the
// high-nibble terms summed in two accumulators.
__device__ __forceinline__ float dot_q4_k_half_xr(const uint8_t* blk, int h, const float (&xr)[128], float xfac) {
    const uint4 hdr = *reinterpret_cast<const uint4*>(blk);
    float a[4], c[4];
    q4_k_half_mults(hdr, h, a, c);
    uint32_t qw[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint4 v = *reinterpret_cast<const uint4*>(blk + 16 + 64 * h + 16 * i);
        qw[4 * i] = v.x;
        qw[4 * i + 1] = v.y;
        qw[4 * i + 2] = v.z;
        qw[4 * i + 3] = v.w;
    }
    float2 s2 = make_float2(0.f, 0.f), t2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
        const float al = a[2 * cc], cl = c[2 * cc], ah = a[2 * cc + 1] * 0.0625f, ch = c[2 * cc + 1];
#pragma unroll
        for (int wi = 0; wi < 8; ++wi) {
            const uint32_t w = qw[8 * cc + wi];
            const uint32_t lo = w & 0x0F0F0F0Fu;
            const uint32_t hi = w & 0xF0F0F0F0u;
            const int kl = 64 * cc + 4 * wi, kh = kl + 32;
            s2 = __ffma2_rn(wpair(al, byte_subnormal<0>(lo), byte_subnormal<1>(lo), cl), make_float2(xr[kl], xr[kl + 1]), s2);
            s2 = __ffma2_rn(wpair(al, byte_subnormal<2>(lo), byte_subnormal<3>(lo), cl), make_float2(xr[kl + 2], xr[kl + 3]), s2);
            t2 = __ffma2_rn(wpair(ah, byte_subnormal<0>(hi), byte_subnormal<1>(hi), ch), make_float2(xr[kh], xr[kh + 1]), t2);
            t2 = __ffma2_rn(wpair(ah, byte_subnormal<2>(hi), byte_subnormal<3>(hi), ch), make_float2(xr[kh + 2], xr[kh + 3]), t2);
        }
    }
    return ((s2.x + s2.y) + (t2.x + t2.y)) * xfac;
}

// Sum of a row's n half-unit partials in a fixed order. With n a multiple of
// four and p 16-byte aligned: four interleaved sums over 16-byte loads
// (partials i, i + 4, ... in sum i % 4), combined as (s0 + s1) + (s2 + s3);
// otherwise one sum in index order. Either way the order depends only on n,
// so results are reproducible.
__device__ __forceinline__ float row_sum(const float* p, int n) {
    if ((n & 3) == 0 && (reinterpret_cast<uintptr_t>(p) & 15) == 0) {
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int i = 0; i < n; i += 4) {
            const float4 v = *reinterpret_cast<const float4*>(p + i);
            a.x += v.x;
            a.y += v.y;
            a.z += v.z;
            a.w += v.w;
        }
        return (a.x + a.y) + (a.z + a.w);
    }
    float v = 0.f;
    for (int i = 0; i < n; ++i) v += p[i];
    return v;
}

}  // namespace phb
