// Streaming dequantize-GEMV building blocks for sm_103a.
//
// A CTA owns a tile: rows [row0, row0 + rows_here) of each of its NMAT
// matrices (NMAT = 2 for the fused gate/up pair), restricted to the K slice
// of units [u0, u0 + useg). The tile's weight bytes are a list of 256-weight
// units (272 B of Q8_0, 144 B of Q4_K) ordered by row, then matrix, then
// unit, so row r of the gate matrix is followed by row r of the up matrix.
// One producer thread streams the list into a ring of shared-memory stages
// with 1-D bulk copies (the TMA engine) that complete on mbarriers; it also
// prefetches into L2 a share of the weights the next kernels will read, so
// HBM keeps streaming across kernel boundaries. CW consumer warps dequantise
// one half unit (128 weights) per thread per stage in registers and dot it
// with activations staged in shared memory (gemv_core.cuh). Thread t owns
// half unit t of a stage, so a warp holds 32 consecutive half units.
//
// Row sums, three ways, all in a fixed order (bitwise reproducible):
//  - warp rows: when a row segment (a gate/up pair counting as one) is a
//    power of two of at most 32 half units, every warp holds whole rows,
//    reduced by a butterfly of warp shuffles; the lane that owns a row runs
//    the epilogue at once and no block barrier is needed;
//  - tile partials: otherwise, when the tile's half-unit sums fit, they stay
//    in shared memory and after the last stage one warp per row reduces
//    them (lanes strided over the row, then a butterfly);
//  - stage fold: otherwise each stage's sums are added, in unit order, to
//    per-row accumulators after the stage.
//
// Every mbarrier wait is bounded (kSpinLimit); one that runs out sets the
// translation unit's device error word and the kernel returns.
#pragma once

#include "gemv_core.cuh"
#include "phb_common.cuh"
#include "trace.cuh"

namespace phb {

// Device error word of the translation unit that includes this header.
static __device__ int g_dev_err;

enum XMode : int { kXPlain = 0, kXRmsNorm = 1, kXGatherV = 2, kXRowList = 3 };
enum Epi : int { kEpiStore = 0, kEpiResid = 1, kEpiSwiGLU = 2 };
enum RowSum : int { kSumWarp = 0, kSumTile = 1, kSumFold = 2 };

constexpr int kAccStride = 8;      // floats per row accumulator slot (max batch)
constexpr float kRmsEps = 1e-6f;
constexpr int kMaxConsumerWarps = 16;

// Per-configuration constants: QT format, CW consumer warps.
template <int QT, int CW, int NS = (QT == 0 ? 2 : 3)>
struct KCfg {
    static constexpr int consumers = 32 * CW;
    static constexpr int threads = consumers + 32;    // + one producer warp
    static constexpr int stage_units = consumers / 2; // one half unit per consumer thread
    static constexpr int ub = Fmt<QT>::unit_bytes;
    static constexpr int stage_bytes = stage_units * ub;
    // ring depth; the default (70 KB of Q8_0 or 55 KB of Q4_K at 8 warps)
    // lets two CTAs (this kernel's and the next one's) share an SM
    static constexpr int ns = NS;
};

// Floats after the mbarriers: xfac [kAccStride], reduction scratch
// [(2 * kMaxConsumerWarps + 3) * kAccStride], row list [kAccStride] (ints).
constexpr int kTailFloats = kAccStride * (1 + 2 * kMaxConsumerWarps + 3 + 1);

template <int N>
__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(N) : "memory");
}

// Geometry of one CTA tile.
struct Tile {
    const uint8_t* w[2];   // first byte of row row0, unit u0, in each matrix
    int64_t row_bytes;     // stride between rows
    int rows_here;         // rows per matrix in this tile
    int useg;              // units per row in this tile
    bool contiguous;       // useg covers whole rows (consecutive rows adjacent)
};

// True when rows reduce inside a warp (see the header comment).
__host__ __device__ __forceinline__ bool warp_rows(int useg, int nmat) {
    const int seg = 2 * useg * nmat;
    return seg <= 32 && (seg & (seg - 1)) == 0;
}

// Prefetch this CTA's share of [p, p + bytes) into L2 (fire and forget).
__device__ __forceinline__ void prefetch_share(const uint8_t* p, int64_t bytes) {
    if (p == nullptr || bytes <= 0) return;
    const int64_t chunk = ((bytes + gridDim.x * gridDim.y - 1) / (gridDim.x * gridDim.y) + 15) & ~int64_t{15};
    const int64_t cta = static_cast<int64_t>(blockIdx.y) * gridDim.x + blockIdx.x;
    int64_t lo = cta * chunk;
    const int64_t hi = min(bytes, lo + chunk) & ~int64_t{15};
    lo &= ~int64_t{15};
    constexpr int64_t kPiece = 32768;
    for (; lo < hi; lo += kPiece) prefetch_l2(p + lo, static_cast<uint32_t>(min(kPiece, hi - lo)));
}

// Producer: stream the tile's unit list through the stage ring, continuing
// the ring position `s` (a stage counter shared with the consumers).
// Returns false on a wait timeout.
template <int QT, int CW, int NS = KCfg<QT, CW>::ns>
__device__ __forceinline__ bool produce_tile(const Tile& t, int nmat, uint8_t* stages, uint64_t* full,
                                             uint64_t* empty, int& s, uint64_t pol,
                                             int stage_units = KCfg<QT, CW, NS>::stage_units) {
    using C = KCfg<QT, CW, NS>;
    const int units = nmat * t.rows_here * t.useg;
    // with one matrix and whole rows the list is one contiguous byte range
    const bool flat = (nmat == 1) && t.contiguous;
    for (int g0 = 0; g0 < units; g0 += stage_units, ++s) {
        const int slot = s % C::ns;
        if (s >= C::ns && !mbar_wait(&empty[slot], ((s / C::ns) - 1) & 1, &g_dev_err)) return false;
        const int g1 = min(units, g0 + stage_units);
        mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>((g1 - g0) * C::ub));
        uint8_t* dst = stages + slot * C::stage_bytes;
        if (flat) {
            bulk_g2s_hint(dst, t.w[0] + static_cast<int64_t>(g0) * C::ub, static_cast<uint32_t>((g1 - g0) * C::ub),
                          &full[slot], pol);
            continue;
        }
        int g = g0;
        while (g < g1) {
            const int seg = g / t.useg;       // row * nmat + mat
            const int u = g - seg * t.useg;
            const int r = seg / nmat;
            const int mat = seg - r * nmat;
            const int end = min(g1, g + (t.useg - u));
            const uint8_t* src = (mat == 0 ? t.w[0] : t.w[1]) + r * t.row_bytes + static_cast<int64_t>(u) * C::ub;
            bulk_g2s_hint(dst + (g - g0) * C::ub, src, static_cast<uint32_t>((end - g) * C::ub), &full[slot], pol);
            g = end;
        }
    }
    return true;
}

// Segment-major stages (the register-resident kernels): a stage holds whole
// row segments (one row of one matrix each; gate and up rows alternate when
// nmat == 2) ss bytes apart. With consecutive threads on consecutive
// segments at one half-unit position, every segment gets a 16-byte pad, so
// that those threads' weight reads spread over the shared-memory banks
// (measured better than padding only segments of a multiple of 64 bytes:
// Q4_K 9728x2560 batch-1 GEMV 7.17 -> 6.68 us, fused decode step
// 0.528 -> 0.525 ms).
__host__ __device__ constexpr int seg_stride_bytes(int useg, int ub) { return useg * ub + 16; }

// Producer of segment-major stages: the tile's segments in order, segs per
// stage, each at its place; one copy per stage when the rows are unpadded.
template <class C>
__device__ __forceinline__ bool produce_segs(const Tile& t, int nmat, int segs, int ss, uint8_t* stages,
                                             uint32_t stage_stride, uint64_t* full, uint64_t* empty, int& s,
                                             uint64_t pol) {
    const int nseg = nmat * t.rows_here;
    const int seg_bytes = t.useg * C::ub;
    for (int seg0 = 0; seg0 < nseg; seg0 += segs, ++s) {
        const int slot = s % C::ns;
        if (s >= C::ns && !mbar_wait(&empty[slot], ((s / C::ns) - 1) & 1, &g_dev_err)) return false;
        const int n = min(segs, nseg - seg0);
        mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(n * seg_bytes));
        uint8_t* dst = stages + static_cast<size_t>(slot) * stage_stride;
        if (nmat == 1 && ss == seg_bytes) {
            bulk_g2s_hint(dst, t.w[0] + static_cast<int64_t>(seg0) * t.row_bytes, static_cast<uint32_t>(n * seg_bytes),
                          &full[slot], pol);
            continue;
        }
        for (int j = 0; j < n; ++j) {
            const int seg = seg0 + j, r = seg / nmat, mat = seg - r * nmat;
            bulk_g2s_hint(dst + j * ss, (mat == 0 ? t.w[0] : t.w[1]) + static_cast<int64_t>(r) * t.row_bytes,
                          static_cast<uint32_t>(seg_bytes), &full[slot], pol);
        }
    }
    return true;
}

// Consumers: dot every staged half unit with the activations and hand each
// finished row to epi(r, b, a0, a1) for b < batch, with a0 the row's sum
// (the gate row's for NMAT == 2) and a1 the up row's sum. `mode` is the
// row-sum method (kSumWarp needs warp_rows). `part` holds
// 2 * units * MAXB floats for kSumTile, MAXB * consumers for kSumFold;
// `row_acc` NMAT * rows_here * kAccStride floats (kSumFold; zeroed by the
// caller before its last consumer barrier). Returns false on a wait timeout.
template <int QT, int CW, int MAXB, int NMAT, int NS = KCfg<QT, CW>::ns, class EpiF>
__device__ __forceinline__ bool consume_tile(const Tile& t, int mode, const uint8_t* stages, uint64_t* full,
                                             uint64_t* empty, int& s, const float* xs, int xstride,
                                             const float* xfac, int batch, float* part, float* row_acc, EpiF epi) {
    using C = KCfg<QT, CW, NS>;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int hsel = tid & 1;
    const int ulocal = tid >> 1;
    const int units = NMAT * t.rows_here * t.useg;
    const int seg_half = 2 * t.useg;  // half units per row segment
    for (int g0 = 0; g0 < units; g0 += C::stage_units, ++s) {
        const int slot = s % C::ns;
        if (!mbar_wait_warp(&full[slot], (s / C::ns) & 1, &g_dev_err)) {
            mbar_wait(&full[slot], (s / C::ns) & 1, &g_dev_err);  // second bounded wait for the copy in flight
            return false;
        }
        const int g = g0 + ulocal;
        const int segi = g / t.useg;
        const int u = g - segi * t.useg;
        float acc[MAXB];
#pragma unroll
        for (int b = 0; b < MAXB; ++b) acc[b] = 0.f;
        if (g < units) {
            const int hu = 2 * u + hsel;  // half unit within the row segment
            const uint8_t* ub = stages + slot * C::stage_bytes + ulocal * C::ub;
            const float* xsp = xs + hu * (kXPadEvery + kXPad);
            if constexpr (QT == 0)
                dot_q8_0_half<MAXB>(ub + 136 * hsel, xsp, xstride, xfac, acc);
            else
                dot_q4_k_half<MAXB>(ub, hsel, xsp, xstride, xfac, acc);
        }
        if (mode == kSumWarp) {
            float other[MAXB];
#pragma unroll
            for (int b = 0; b < MAXB; ++b) {
                float v = acc[b];
                for (int o = 1; o < seg_half; o <<= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
                acc[b] = v;
                other[b] = NMAT == 2 ? __shfl_xor_sync(0xFFFFFFFFu, v, seg_half) : 0.f;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
            if ((lane & (NMAT * seg_half - 1)) == 0 && g < units) {
                const int r = segi / NMAT;
#pragma unroll
                for (int b = 0; b < MAXB; ++b)
                    if (b < batch) epi(r, b, acc[b], other[b]);
            }
            continue;
        }
        if (mode == kSumTile) {
            if (g < units) {
#pragma unroll
                for (int b = 0; b < MAXB; ++b) part[(2 * g + hsel) * MAXB + b] = acc[b];
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
            continue;
        }
#pragma unroll
        for (int b = 0; b < MAXB; ++b) part[b * C::consumers + tid] = acc[b];
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
        consumer_sync<C::consumers>();
        // fold this stage into the row segments it touched, half units in order
        const int g1 = min(units, g0 + C::stage_units);
        const int r_first = g0 / t.useg, r_last = (g1 - 1) / t.useg;
        const int items = (r_last - r_first + 1) * batch;
        for (int it = tid; it < items; it += C::consumers) {
            const int rr = r_first + it / batch;
            const int b = it - (it / batch) * batch;
            const int ha = 2 * (max(g0, rr * t.useg) - g0), hb = 2 * (min(g1, (rr + 1) * t.useg) - g0);
            const float* q = part + b * C::consumers;
            float sum = row_acc[rr * kAccStride + b];
            for (int hh = ha; hh < hb; ++hh) sum += q[hh];
            row_acc[rr * kAccStride + b] = sum;
        }
        consumer_sync<C::consumers>();
    }
    if (mode == kSumTile) {
        consumer_sync<C::consumers>();
        // one warp per row: lanes strided over the row's half units, then a butterfly
        for (int r = warp; r < t.rows_here; r += CW) {
            float a[NMAT][MAXB];
#pragma unroll
            for (int m = 0; m < NMAT; ++m) {
                const float* base = part + static_cast<size_t>(r * NMAT + m) * seg_half * MAXB;
#pragma unroll
                for (int b = 0; b < MAXB; ++b) {
                    float v = 0.f;
                    for (int j = lane; j < seg_half; j += 32) v += base[j * MAXB + b];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
                    a[m][b] = v;
                }
            }
            if (lane == 0) {
#pragma unroll
                for (int b = 0; b < MAXB; ++b)
                    if (b < batch) epi(r, b, a[0][b], a[NMAT - 1][b]);
            }
        }
    } else if (mode == kSumFold) {
        for (int it = tid; it < t.rows_here * batch; it += C::consumers) {
            const int r = it / batch;
            const int b = it - r * batch;
            const float a0 = row_acc[(r * NMAT) * kAccStride + b];
            const float a1 = NMAT == 2 ? row_acc[(r * NMAT + 1) * kAccStride + b] : 0.f;
            epi(r, b, a0, a1);
        }
    }
    return true;
}

// Stage activations a[b][0 .. kseg) for b < batch into shared memory:
//   xs   [MAXB][xpad_len(kseg)]: a * 2^s_b in the padded layout (xpad_idx)
//   xfac [MAXB]:                 2^(kWShift - s_b)
// Rows batch..MAXB-1 are zero (xfac 1). a is x[b][kbase + k] (kXPlain),
// x[rowidx[b]][k] (kXRowList), the V head of the query head that owns k
// (kXGatherV), or x[b][k] * r_b with r_b = (mean_k x^2 + eps)^-1/2
// (kXRmsNorm; rows are whole). s_b is chosen from max|a| so that
// |a| * 2^s_b < 2^125: the scaled weights are below 2^-58, so no product
// or sum of up to 2^20 products can overflow, and no product of a weight
// with an activation of more than 2^-140 times the row's largest magnitude
// can underflow. One global read pass, three consumer barriers.
// `red` needs (2 * CW + 3) * kAccStride floats.
// Capped at kWShift + 126 so that 2^(kWShift - s) stays a normal number
// (vectors whose largest magnitude is below 2^-86 are scaled by 2^211,
// still below 2^125); s >= -3 for every finite vector.
__device__ __forceinline__ int pick_scale_exp(float amax) {
    if (!(amax > 0.f) || !isfinite(amax)) return 125;
    const int e = ilogbf(amax) + 1;  // amax < 2^e
    return min(kWShift + 126, 125 - e);
}

// Register-resident activations: copy the 128 values of one half unit from
// shared memory (padded layout, 16-byte aligned) into xr, scaled by 2^s with
// s picked from their own largest magnitude, and return the factor
// 2^(kWShift - s) that takes a half-unit dot back to the true scale.
__device__ __forceinline__ float load_xr_scaled(const float* xp, float (&xr)[128]) {
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const float4 v = *reinterpret_cast<const float4*>(xp + 4 * i);
        xr[4 * i] = v.x;
        xr[4 * i + 1] = v.y;
        xr[4 * i + 2] = v.z;
        xr[4 * i + 3] = v.w;
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
    const int se = pick_scale_exp(amax);
    const int e1 = min(se, 127);
    const float f1 = __int_as_float((e1 + 127) << 23);
#pragma unroll
    for (int i = 0; i < 128; ++i) xr[i] *= f1;
    if (se > 127) {  // largest magnitude below 2^-3: the rest of the power of two
        const float f2 = __int_as_float((se - e1 + 127) << 23);
#pragma unroll
        for (int i = 0; i < 128; ++i) xr[i] *= f2;
    }
    return __int_as_float((kWShift - se + 127) << 23);
}

template <int CW, int MAXB, int XMODE>
__device__ __forceinline__ void stage_x(const float* x, int64_t ldx, int64_t kbase, int kseg, int batch, float* xs,
                                       float* xfac, float* red, int gather_group, int gather_hd,
                                       int64_t gather_v_off, const int* rowidx = nullptr) {
    constexpr int NC = 32 * CW;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int xstride = xpad_len(kseg);
    const int nch = kseg / 8;  // 8-float chunks per row
    float ssq[MAXB], mx[MAXB];
#pragma unroll
    for (int b = 0; b < MAXB; ++b) ssq[b] = mx[b] = 0.f;
    for (int i = tid; i < MAXB * nch; i += NC) {
        const int b = i / nch;
        const int c = i - b * nch;
        float v[8];
        if (b < batch) {
            if constexpr (XMODE == kXGatherV) {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int k = 8 * c + e;
                    const int hh = k / gather_hd;
                    v[e] = x[b * ldx + gather_v_off + static_cast<int64_t>(hh / gather_group) * gather_hd +
                             (k - hh * gather_hd)];
                }
            } else {
                const float* src = XMODE == kXRowList ? x + static_cast<int64_t>(rowidx[b]) * ldx + 8 * c
                                                      : x + b * ldx + kbase + 8 * c;
                const float4 p0 = *reinterpret_cast<const float4*>(src);
                const float4 p1 = *reinterpret_cast<const float4*>(src + 4);
                v[0] = p0.x;
                v[1] = p0.y;
                v[2] = p0.z;
                v[3] = p0.w;
                v[4] = p1.x;
                v[5] = p1.y;
                v[6] = p1.z;
                v[7] = p1.w;
            }
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = 0.f;
        }
        float* dst = xs + b * xstride + xpad_idx(8 * c);
        *reinterpret_cast<float4*>(dst) = make_float4(v[0], v[1], v[2], v[3]);
        *reinterpret_cast<float4*>(dst + 4) = make_float4(v[4], v[5], v[6], v[7]);
        const float cm = fmaxf(fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3]))),
                               fmaxf(fmaxf(fabsf(v[4]), fabsf(v[5])), fmaxf(fabsf(v[6]), fabsf(v[7]))));
        float cq = 0.f;
        if constexpr (XMODE == kXRmsNorm) {
#pragma unroll
            for (int e = 0; e < 8; ++e) cq = fmaf(v[e], v[e], cq);
        }
#pragma unroll
        for (int bb = 0; bb < MAXB; ++bb) {
            if (bb == b) {
                mx[bb] = fmaxf(mx[bb], cm);
                ssq[bb] += cq;
            }
        }
    }
#pragma unroll
    for (int b = 0; b < MAXB; ++b) {
        float m = mx[b], q = ssq[b];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
            q += __shfl_xor_sync(0xFFFFFFFFu, q, o);
        }
        if (lane == 0) {
            red[warp * kAccStride + b] = m;
            red[(CW + warp) * kAccStride + b] = q;
        }
    }
    consumer_sync<NC>();
    // per row: rms factor r (1 unless kXRmsNorm) and the two power-of-two multipliers
    float* rfac = red + 2 * CW * kAccStride;  // [MAXB]
    float* f1 = rfac + kAccStride;             // [MAXB]
    float* f2 = f1 + kAccStride;               // [MAXB]
    if (tid < MAXB) {
        float m = 0.f, q = 0.f;
        for (int w = 0; w < CW; ++w) {
            m = fmaxf(m, red[w * kAccStride + tid]);
            q += red[(CW + w) * kAccStride + tid];
        }
        float r = 1.f;
        if constexpr (XMODE == kXRmsNorm) r = rsqrtf(q / static_cast<float>(kseg) + kRmsEps);
        const int se = tid < batch ? pick_scale_exp(m * r) : 0;
        const int e1 = min(se, 127);
        rfac[tid] = r;
        f1[tid] = ldexpf(1.0f, e1);
        f2[tid] = ldexpf(1.0f, se - e1);
        xfac[tid] = tid < batch ? ldexpf(1.0f, kWShift - se) : 1.0f;
    }
    consumer_sync<NC>();
    const int per_row4 = kseg / 4;
    for (int i = tid; i < batch * per_row4; i += NC) {
        const int b = i / per_row4;
        const int k4 = i - b * per_row4;
        const float r = rfac[b], a = f1[b], c = f2[b];
        float4* p = reinterpret_cast<float4*>(xs + b * xstride + xpad_idx(4 * k4));
        float4 v = *p;
        if constexpr (XMODE == kXRmsNorm) {
            v.x *= r;
            v.y *= r;
            v.z *= r;
            v.w *= r;
        }
        v.x = v.x * a * c;
        v.y = v.y * a * c;
        v.z = v.z * a * c;
        v.w = v.w * a * c;
        *p = v;
    }
    consumer_sync<NC>();
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

// ----------------------------------------------------------------------------
// Dense kernel
// ----------------------------------------------------------------------------
struct GemvParams {
    const uint8_t* w[2];
    int64_t row_bytes;     // bytes of one full row
    int64_t n;             // rows of each matrix
    int units_row;         // K / 256
    int units_seg;         // units per K split (last split may hold fewer)
    int rows_per_cta;
    int batch;
    int sum_mode;          // RowSum
    const float* x;
    int64_t ldx;
    float* y;
    int64_t ldy;
    const float* r;        // residual (kEpiResid)
    int64_t ldr;
    float* part;           // split-K partials [gridDim.y][batch][n]
    int gather_group;      // kXGatherV: query heads per KV head
    int gather_hd;         // kXGatherV: head dim
    int64_t gather_v_off;  // kXGatherV: offset of V in the qkv vector
    const uint8_t* pf[2];  // weights of later kernels to prefetch into L2 (optional)
    int64_t pf_bytes[2];
    uint32_t xs_off, part_off, acc_off, bar_off;  // dynamic shared memory layout
    int trace_id;          // launch id for debug tracing builds (-1: none)
};

template <int QT, int CW, int MAXB, int NMAT, int XMODE, int EPI>
// Batch 1 and 2: registers capped so that two CTAs share an SM; larger
// batches hold more accumulators and run one wider CTA per SM.
__global__ void __launch_bounds__(KCfg<QT, CW>::threads, MAXB <= 2 ? 2 : 1)
    gemv_stream_kernel(const __grid_constant__ GemvParams p) {
    using C = KCfg<QT, CW>;
    extern __shared__ __align__(1024) uint8_t smem[];
    float* xs = reinterpret_cast<float*>(smem + p.xs_off);
    float* part = reinterpret_cast<float*>(smem + p.part_off);
    float* row_acc = reinterpret_cast<float*>(smem + p.acc_off);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.bar_off);
    uint64_t* empty = full + C::ns;
    float* xfac = reinterpret_cast<float*>(empty + C::ns);
    float* red = xfac + kAccStride;

    const int tid = threadIdx.x;
    if (tid == 0) PHB_TRACE_EV(p.trace_id, 0);
    const int64_t row0 = static_cast<int64_t>(blockIdx.x) * p.rows_per_cta;
    const int split = blockIdx.y;
    const int u0 = split * p.units_seg;
    Tile t;
    t.rows_here = static_cast<int>(min(static_cast<int64_t>(p.rows_per_cta), p.n - row0));
    t.useg = min(p.units_seg, p.units_row - u0);
    t.row_bytes = p.row_bytes;
    t.contiguous = (t.useg == p.units_row);
    t.w[0] = p.w[0] + row0 * p.row_bytes + static_cast<int64_t>(u0) * C::ub;
    t.w[1] = p.w[NMAT - 1] + row0 * p.row_bytes + static_cast<int64_t>(u0) * C::ub;
    pdl_launch_dependents();
    if (t.rows_here <= 0 || t.useg <= 0) {
        pdl_wait();
        return;
    }
    const int kseg = t.useg * kUnitWeights;
    const int batch = p.batch;

    if (tid == 0) {
        for (int s = 0; s < C::ns; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], CW);
        }
        fence_barrier_init();
    }
    if (p.sum_mode == kSumFold)
        for (int i = tid; i < NMAT * t.rows_here * kAccStride; i += C::threads) row_acc[i] = 0.f;
    __syncthreads();

    if (tid >= C::consumers) {
        if (tid == C::consumers) {
            int s = 0;
            const uint64_t pol = policy_evict_first();
            produce_tile<QT, CW>(t, NMAT, smem, full, empty, s, pol);
        } else if (tid == C::consumers + 1) {
            prefetch_share(p.pf[0], p.pf_bytes[0]);
            prefetch_share(p.pf[1], p.pf_bytes[1]);
        }
        return;
    }

    pdl_wait();
    if (tid == 0) PHB_TRACE_EV(p.trace_id, 1);
    stage_x<CW, MAXB, XMODE>(p.x, p.ldx, static_cast<int64_t>(u0) * kUnitWeights, kseg, batch, xs, xfac, red,
                             p.gather_group, p.gather_hd, p.gather_v_off);
    if (tid == 0) PHB_TRACE_EV(p.trace_id, 2);
    const bool split_out = gridDim.y > 1;
    auto epi = [&](int r, int b, float a0, float a1) {
        const int64_t n = row0 + r;
        if (split_out) {
            p.part[(static_cast<int64_t>(split) * batch + b) * p.n + n] = a0;
        } else if constexpr (EPI == kEpiStore) {
            p.y[b * p.ldy + n] = a0;
        } else if constexpr (EPI == kEpiResid) {
            p.y[b * p.ldy + n] = p.r[b * p.ldr + n] + a0;
        } else {
            p.y[b * p.ldy + n] = silu_mul(a0, a1);
        }
    };
    int s = 0;
    consume_tile<QT, CW, MAXB, NMAT>(t, p.sum_mode, smem, full, empty, s, xs, xpad_len(kseg), xfac, batch, part,
                                     row_acc, epi);
    if (tid == 0) PHB_TRACE_EV(p.trace_id, 4);
}

// Host-side plan of one streaming GEMV launch.
struct GemvPlan {
    dim3 grid;
    size_t smem;
    int cw;                // consumer warps of the chosen instantiation
    GemvParams p;
};

}  // namespace phb
