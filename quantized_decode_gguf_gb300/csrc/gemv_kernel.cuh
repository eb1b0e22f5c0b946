// Streaming dequantize-GEMV building blocks for sm_103a.
//
// A CTA owns a tile: rows [row0, row0 + rows_here) of each of its NMAT
// matrices, restricted to the K slice of units [u0, u0 + useg). The tile's
// weight bytes are a list of 256-weight units (272 B of Q8_0, 144 B of Q4_K),
// ordered matrix-major, then row, then unit. One producer thread streams the
// list into a ring of shared-memory stages with 1-D bulk copies (the TMA
// engine) that complete on mbarriers. Eight consumer warps dequantise one
// half unit per thread per stage in registers and dot it with activations
// staged in shared memory (gemv_core.cuh). After each stage the half-unit
// sums of every row the stage touched are added, in unit order, to that
// row's accumulator; accumulation order is therefore fixed and results are
// bitwise reproducible.
//
// The dense kernel (gemv_stream_kernel) issues its weight copies before the
// programmatic-dependent-launch wait, so they overlap the previous kernel.
// Every mbarrier wait is bounded (kSpinLimit); one that runs out sets the
// translation unit's device error word and the kernel returns.
#pragma once

#include "gemv_core.cuh"
#include "phb_common.cuh"

namespace phb {

// Device error word of the translation unit that includes this header.
static __device__ int g_dev_err;

enum XMode : int { kXPlain = 0, kXRmsNorm = 1, kXGatherV = 2, kXRowList = 3 };
enum Epi : int { kEpiStore = 0, kEpiResid = 1, kEpiSwiGLU = 2 };

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = 32 * kConsumerWarps;
constexpr int kGemvThreads = kConsumers + 32;
constexpr int kStageUnits = 128;   // 256 half units: one per consumer thread
constexpr int kAccStride = 8;      // floats per (half unit | row) accumulator slot
constexpr float kRmsEps = 1e-6f;

template <int QT> struct StageCfg;
template <> struct StageCfg<0> { static constexpr int ns = 2; };  // 2 x 34816 B
template <> struct StageCfg<1> { static constexpr int ns = 4; };  // 4 x 18432 B

__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
}

// Geometry of one CTA tile.
struct Tile {
    const uint8_t* w[2];   // first byte of row row0, unit u0, in each matrix
    int64_t row_bytes;     // stride between rows
    int rows_here;         // rows per matrix in this tile
    int useg;              // units per row in this tile
    bool contiguous;       // useg covers whole rows (consecutive rows adjacent)
};

__device__ __forceinline__ int tile_units(const Tile& t, int nmat) { return nmat * t.rows_here * t.useg; }

// Producer: stream `nst` stages of the tile's unit list, continuing the ring
// position `s` (stage counter shared with the consumers). Returns false on a
// wait timeout.
template <int QT>
__device__ __forceinline__ bool produce_tile(const Tile& t, int nmat, uint8_t* stages, uint64_t* full,
                                             uint64_t* empty, int& s, uint64_t pol) {
    constexpr int UB = Fmt<QT>::unit_bytes;
    constexpr int NS = StageCfg<QT>::ns;
    constexpr int SB = kStageUnits * UB;
    const int units_mat = t.rows_here * t.useg;
    const int units = nmat * units_mat;
    for (int g0 = 0; g0 < units; g0 += kStageUnits, ++s) {
        const int slot = s % NS;
        if (s >= NS && !mbar_wait(&empty[slot], ((s / NS) - 1) & 1, &g_dev_err)) return false;
        const int g1 = min(units, g0 + kStageUnits);
        mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>((g1 - g0) * UB));
        uint8_t* dst = stages + slot * SB;
        int g = g0;
        while (g < g1) {
            const int mat = g / units_mat;
            const int rem = g - mat * units_mat;
            const int r = rem / t.useg;
            const int u = rem - r * t.useg;
            const int end = t.contiguous ? min(g1, (mat + 1) * units_mat) : min(g1, g + (t.useg - u));
            const uint8_t* src = (mat == 0 ? t.w[0] : t.w[1]) + r * t.row_bytes + static_cast<int64_t>(u) * UB;
            bulk_g2s_hint(dst + (g - g0) * UB, src, static_cast<uint32_t>((end - g) * UB), &full[slot], pol);
            g = end;
        }
    }
    return true;
}

// Consumers: dot every staged half unit with the activations and fold the
// sums into row_acc[(mat * rows_here + r) * kAccStride + b]. row_acc must be
// zeroed by the caller. Consumer thread t owns half unit t of each stage
// (unit t/2, half t%2), so a warp reads 32 consecutive half units: bank
// conflict free for the weights, and (with the padded activation layout)
// for the activations. Returns false on a wait timeout.
//   xs, xsum, xfac: staged activations (see stage_x)
template <int QT, int MAXB>
__device__ __forceinline__ bool consume_tile(const Tile& t, int nmat, const uint8_t* stages, uint64_t* full,
                                             uint64_t* empty, int& s, const float* xs, int xstride,
                                             const float* xsum, int sstride, const float* xfac, int batch,
                                             float* part, float* row_acc) {
    constexpr int UB = Fmt<QT>::unit_bytes;
    constexpr int NS = StageCfg<QT>::ns;
    constexpr int SB = kStageUnits * UB;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int hsel = tid & 1;
    const int ulocal = tid >> 1;
    const int units = nmat * t.rows_here * t.useg;
    for (int g0 = 0; g0 < units; g0 += kStageUnits, ++s) {
        const int slot = s % NS;
        if (!mbar_wait(&full[slot], (s / NS) & 1, &g_dev_err)) {
            mbar_wait(&full[slot], (s / NS) & 1, &g_dev_err);  // second bounded wait for the copy in flight
            return false;
        }
        const int g = g0 + ulocal;
        float acc[MAXB];
#pragma unroll
        for (int b = 0; b < MAXB; ++b) acc[b] = 0.f;
        if (g < units) {
            const int hu = 2 * (g % t.useg) + hsel;  // half unit within the row segment
            const uint8_t* ub = stages + slot * SB + ulocal * UB;
            const float* xsp = xs + hu * (kXPadEvery + kXPad);
            const float* xsm = xsum + hu * 4;
            if constexpr (QT == 0)
                dot_q8_0_half<MAXB>(ub + 136 * hsel, xsp, xstride, xsm, sstride, xfac, batch, acc);
            else
                dot_q4_k_half<MAXB>(ub, hsel, xsp, xstride, xsm, sstride, xfac, batch, acc);
        }
#pragma unroll
        for (int b = 0; b < MAXB; ++b) part[b * 2 * kStageUnits + tid] = acc[b];
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
        consumer_sync();
        // fold this stage into the rows it touched, half units in order
        const int g1 = min(units, g0 + kStageUnits);
        const int r_first = g0 / t.useg, r_last = (g1 - 1) / t.useg;
        const int items = (r_last - r_first + 1) * batch;
        for (int it = tid; it < items; it += kConsumers) {
            const int rr = r_first + it / batch;
            const int b = it - (it / batch) * batch;
            const int ha = 2 * (max(g0, rr * t.useg) - g0), hb = 2 * (min(g1, (rr + 1) * t.useg) - g0);
            const float* q = part + b * 2 * kStageUnits;
            float sum = row_acc[rr * kAccStride + b];
            for (int hh = ha; hh < hb; ++hh) sum += q[hh];
            row_acc[rr * kAccStride + b] = sum;
        }
        consumer_sync();
    }
    return true;
}

// Stage activations a[b][0 .. kseg) for b < batch into shared memory:
//   xs   [b][xpad_len(kseg)]: a * 2^s_b in the padded layout (xpad_idx)
//   xsum [b][kseg/32]:        unscaled sums of every 32 consecutive a
//   xfac [b]:                 2^(149 - s_b)
// a is x[b][kbase + k] (kXPlain), x[rowidx[b]][k] (kXRowList), rmsnorm of
// the whole row (kXRmsNorm), or the V head of the query head that owns k
// (kXGatherV). s_b is chosen from
// max|a| so that |a| * 2^s_b < 2^125. `red` needs (kConsumerWarps+1) *
// kAccStride floats. Ends with a consumer barrier.
__device__ __forceinline__ int pick_scale_exp(float amax) {
    if (!(amax > 0.f) || !isfinite(amax)) return 125;
    const int e = ilogbf(amax) + 1;  // amax < 2^e
    return min(270, max(22, 125 - e));
}

template <int QT, int MAXB, int XMODE>
__device__ __forceinline__ void stage_x(const float* x, int64_t ldx, int64_t kbase, int kseg, int batch, float* xs,
                                       float* xsum, float* xfac, float* red, int gather_group, int gather_hd,
                                       int64_t gather_v_off, const int* rowidx = nullptr) {
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int xstride = xpad_len(kseg);
    const int per_row4 = kseg / 4;
    if constexpr (XMODE == kXGatherV) {
        for (int i = tid; i < batch * kseg; i += kConsumers) {
            const int b = i / kseg;
            const int k = i - b * kseg;
            const int hh = k / gather_hd;
            const int e = k - hh * gather_hd;
            xs[b * xstride + xpad_idx(k)] =
                x[b * ldx + gather_v_off + static_cast<int64_t>(hh / gather_group) * gather_hd + e];
        }
    } else {
        float ss[MAXB];
#pragma unroll
        for (int b = 0; b < MAXB; ++b) ss[b] = 0.f;
        for (int i = tid; i < batch * per_row4; i += kConsumers) {
            const int b = i / per_row4;
            const int k4 = i - b * per_row4;
            const float* src = XMODE == kXRowList ? x + static_cast<int64_t>(rowidx[b]) * ldx : x + b * ldx + kbase;
            const float4 v = *reinterpret_cast<const float4*>(src + 4 * k4);
            *reinterpret_cast<float4*>(xs + b * xstride + xpad_idx(4 * k4)) = v;
            if constexpr (XMODE == kXRmsNorm) {
#pragma unroll
                for (int bb = 0; bb < MAXB; ++bb) {
                    if (bb == b) {
                        ss[bb] = fmaf(v.x, v.x, ss[bb]);
                        ss[bb] = fmaf(v.y, v.y, ss[bb]);
                        ss[bb] = fmaf(v.z, v.z, ss[bb]);
                        ss[bb] = fmaf(v.w, v.w, ss[bb]);
                    }
                }
            }
        }
        if constexpr (XMODE == kXRmsNorm) {
#pragma unroll
            for (int b = 0; b < MAXB; ++b) {
                const float w = warp_sum(ss[b]);
                if (lane == 0) red[warp * kAccStride + b] = w;
            }
            consumer_sync();
            if (tid < batch) {
                float tsum = 0.f;
                for (int w = 0; w < kConsumerWarps; ++w) tsum += red[w * kAccStride + tid];
                red[kConsumerWarps * kAccStride + tid] = rsqrtf(tsum / static_cast<float>(kseg) + kRmsEps);
            }
            consumer_sync();
            for (int i = tid; i < batch * per_row4; i += kConsumers) {
                const int b = i / per_row4;
                const int k4 = i - b * per_row4;
                const float sc = red[kConsumerWarps * kAccStride + b];
                float4* p = reinterpret_cast<float4*>(xs + b * xstride + xpad_idx(4 * k4));
                float4 v = *p;
                v.x *= sc;
                v.y *= sc;
                v.z *= sc;
                v.w *= sc;
                *p = v;
            }
        }
    }
    consumer_sync();
    // 32-sums and per-row max |a|
    const int nsub = kseg / 32;
    float mx[MAXB];
#pragma unroll
    for (int b = 0; b < MAXB; ++b) mx[b] = 0.f;
    for (int i = tid; i < batch * nsub; i += kConsumers) {
        const int b = i / nsub;
        const int j = i - b * nsub;
        const float* src = xs + b * xstride + xpad_idx(32 * j);
        float tsum = 0.f, tmax = 0.f;
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            tsum += src[e];
            tmax = fmaxf(tmax, fabsf(src[e]));
        }
        xsum[i] = tsum;
#pragma unroll
        for (int bb = 0; bb < MAXB; ++bb)
            if (bb == b) mx[bb] = fmaxf(mx[bb], tmax);
    }
#pragma unroll
    for (int b = 0; b < MAXB; ++b) {
        float v = mx[b];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
        if (lane == 0) red[warp * kAccStride + b] = v;
    }
    consumer_sync();
    if (tid < batch) {
        float v = 0.f;
        for (int w = 0; w < kConsumerWarps; ++w) v = fmaxf(v, red[w * kAccStride + tid]);
        const int se = pick_scale_exp(v);
        red[kConsumerWarps * kAccStride + tid] = static_cast<float>(se);
        xfac[tid] = ldexpf(1.0f, 149 - se);
    }
    consumer_sync();
    for (int i = tid; i < batch * per_row4; i += kConsumers) {
        const int b = i / per_row4;
        const int k4 = i - b * per_row4;
        const int se = static_cast<int>(red[kConsumerWarps * kAccStride + b]);
        float4* p = reinterpret_cast<float4*>(xs + b * xstride + xpad_idx(4 * k4));
        float4 v = *p;
        v.x = ldexpf(v.x, se);
        v.y = ldexpf(v.y, se);
        v.z = ldexpf(v.z, se);
        v.w = ldexpf(v.w, se);
        *p = v;
    }
    consumer_sync();
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
    uint32_t xs_off, xsum_off, part_off, acc_off, bar_off;  // dynamic shared memory layout
};

template <int QT, int MAXB, int NMAT, int XMODE, int EPI>
__global__ void __launch_bounds__(kGemvThreads, 1) gemv_stream_kernel(const __grid_constant__ GemvParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    constexpr int NS = StageCfg<QT>::ns;
    float* xs = reinterpret_cast<float*>(smem + p.xs_off);
    float* xsum = reinterpret_cast<float*>(smem + p.xsum_off);
    float* part = reinterpret_cast<float*>(smem + p.part_off);
    float* row_acc = reinterpret_cast<float*>(smem + p.acc_off);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.bar_off);
    uint64_t* empty = full + NS;
    float* red = reinterpret_cast<float*>(empty + NS);
    float* xfac = red + (kConsumerWarps + 1) * kAccStride;

    const int tid = threadIdx.x;
    const int64_t row0 = static_cast<int64_t>(blockIdx.x) * p.rows_per_cta;
    const int split = blockIdx.y;
    const int u0 = split * p.units_seg;
    Tile t;
    t.rows_here = static_cast<int>(min(static_cast<int64_t>(p.rows_per_cta), p.n - row0));
    t.useg = min(p.units_seg, p.units_row - u0);
    t.row_bytes = p.row_bytes;
    t.contiguous = (t.useg == p.units_row);
    constexpr int UB = Fmt<QT>::unit_bytes;
    t.w[0] = p.w[0] + row0 * p.row_bytes + static_cast<int64_t>(u0) * UB;
    t.w[1] = p.w[NMAT - 1] + row0 * p.row_bytes + static_cast<int64_t>(u0) * UB;
    pdl_launch_dependents();
    if (t.rows_here <= 0 || t.useg <= 0) {
        pdl_wait();
        return;
    }
    const int kseg = t.useg * kUnitWeights;
    const int batch = p.batch;

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        fence_barrier_init();
    }
    for (int i = tid; i < NMAT * t.rows_here * kAccStride; i += kGemvThreads) row_acc[i] = 0.f;
    __syncthreads();

    if (tid >= kConsumers) {
        if (tid == kConsumers) {
            int s = 0;
            produce_tile<QT>(t, NMAT, smem, full, empty, s, policy_evict_first());
        }
        return;
    }

    pdl_wait();
    stage_x<QT, MAXB, XMODE>(p.x, p.ldx, static_cast<int64_t>(u0) * kUnitWeights, kseg, batch, xs, xsum, xfac, red,
                             p.gather_group, p.gather_hd, p.gather_v_off);
    int s = 0;
    if (!consume_tile<QT, MAXB>(t, NMAT, smem, full, empty, s, xs, xpad_len(kseg), xsum, kseg / 32, xfac, batch, part,
                                row_acc))
        return;

    for (int it = tid; it < t.rows_here * batch; it += kConsumers) {
        const int rr = it / batch;
        const int b = it - rr * batch;
        const int64_t n = row0 + rr;
        const float a0 = row_acc[rr * kAccStride + b];
        if (gridDim.y > 1) {
            p.part[(static_cast<int64_t>(split) * batch + b) * p.n + n] = a0;
        } else if constexpr (EPI == kEpiStore) {
            p.y[b * p.ldy + n] = a0;
        } else if constexpr (EPI == kEpiResid) {
            p.y[b * p.ldy + n] = p.r[b * p.ldr + n] + a0;
        } else {
            const float a1 = row_acc[(t.rows_here + rr) * kAccStride + b];
            p.y[b * p.ldy + n] = silu_mul(a0, a1);
        }
    }
}

// Host-side plan of one streaming GEMV launch.
struct GemvPlan {
    dim3 grid;
    size_t smem;
    GemvParams p;
};

}  // namespace phb
