// Building blocks of the persistent cooperative kernels (one CTA per SM,
// a producer warp streaming weight stages through a ring, consumer threads
// holding their activations in registers, tagged vectors exchanged through
// the workspace). Included by one translation unit per kernel, after
// gemv_plan.cuh; every name lives in that unit's anonymous namespace.
#pragma once

#include <cstdint>

#include "gemv_plan.cuh"

namespace phb {
namespace {

// 11 consumer warps + the producer warp: 12 warps, three per scheduler, at
// the 168 registers the 128 resident activations need (65,536 / 384 threads).
constexpr int kCW = 11;            // consumer warps per CTA
constexpr int kNC = 32 * kCW;      // consumer threads
constexpr int kHalfK = 128;        // activations a consumer thread keeps in registers
// Every intermediate vector is stored kRep times (replicas one stride apart)
// and CTA i reads replica i % kRep, so the 152 readers of a vector spread
// over kRep sets of L2 lines instead of queueing on one.
constexpr int kRep = 8;
constexpr uint64_t kOpWaitNs = 2000000000ull;
// state words of a persistent kernel's workspace: [0] finish counter,
// [1] abort, [2] epoch, [kCtrBase + op] CTAs done with op
constexpr int kCtrBase = 64;

__device__ __forceinline__ unsigned ld_relaxed(const unsigned* p) {
    unsigned v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Tagged pairs are moved as single 64-bit accesses ({value, tag} in the low
// and high word), which the memory model makes single-copy atomic: a reader
// never sees the tag of one store with the value of another.
__device__ __forceinline__ void ld_l2_pairs2(const uint2* p, uint2& a, uint2& b) {
    unsigned long long u, v;
    asm volatile("ld.global.cg.v2.u64 {%0, %1}, [%2];" : "=l"(u), "=l"(v) : "l"(p) : "memory");
    a = make_uint2(static_cast<unsigned>(u), static_cast<unsigned>(u >> 32));
    b = make_uint2(static_cast<unsigned>(v), static_cast<unsigned>(v >> 32));
}

__device__ __forceinline__ uint2 ld_l2_pair(const uint2* p) {
    unsigned long long u;
    asm volatile("ld.global.cg.u64 %0, [%1];" : "=l"(u) : "l"(p) : "memory");
    return make_uint2(static_cast<unsigned>(u), static_cast<unsigned>(u >> 32));
}

__device__ __forceinline__ float4 ld_l2_f4(const float* p) {
    float4 v;
    asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p)
                 : "memory");
    return v;
}

__device__ __forceinline__ void st_pair(uint2* p, float v, unsigned tag) {
    const unsigned long long u = static_cast<unsigned long long>(tag) << 32 | __float_as_uint(v);
    asm volatile("st.global.u64 [%0], %1;" ::"l"(p), "l"(u) : "memory");
}

// Four consecutive tagged values starting at pair e; true when all carry tag.
__device__ __forceinline__ bool ld_tagged4(const uint2* src, int e, unsigned tag, float4& v) {
    uint2 a, b, c, d;
    ld_l2_pairs2(src + e, a, b);
    ld_l2_pairs2(src + e + 2, c, d);
    v = make_float4(__uint_as_float(a.x), __uint_as_float(b.x), __uint_as_float(c.x), __uint_as_float(d.x));
    return a.y == tag && b.y == tag && c.y == tag && d.y == tag;
}

__device__ __forceinline__ void set_abort(unsigned* state) {
    atomicExch(&g_dev_err, kDevErrTimeout);
    atomicExch(state + 1, 1u);
}

// Bounded-wait bookkeeping shared by the polling loops: false once the
// call is aborted (by this wait running out or by another CTA).
struct WaitClock {
    uint64_t t0 = 0;
    __device__ __forceinline__ bool tick(unsigned* state) {
        if (t0 == 0) t0 = global_timer_ns();
        if (*reinterpret_cast<volatile unsigned*>(state + 1)) {
            atomicExch(&g_dev_err, kDevErrTimeout);
            return false;
        }
        if (global_timer_ns() - t0 > kOpWaitNs) {
            set_abort(state);
            return false;
        }
        return true;
    }
};

// One thread per CTA waits (bounded) until all `target` CTAs have counted
// their arrival at op `op`. Returns false on timeout or abort.
__device__ __forceinline__ bool wait_op_arrivals(unsigned* state, int op, unsigned target) {
    const unsigned* c = state + kCtrBase + op;
    WaitClock clk;
    while (ld_relaxed(c) < target) {
        if (!clk.tick(state)) return false;
        __nanosleep(20);
    }
    return true;
}

// Stage one activation vector of kseg floats for the register-resident
// dot: one coalesced read pass (four values per lane and load group, up to 8
// groups in flight per thread), raw values into xs (padded layout), then
// scaled in place exactly as the launched GEMV's staging does:
// x * r (RMSNorm) * 2^s. The source is a tagged vector (pairs carrying
// `tag`; pairs that are not yet current are re-read, bounded) or, for the
// first layer, the caller's plain vector. XMODE: 0 plain, 1 RMSNorm, 2 gather
// of the V heads. In the same pass threads t < nres read the next
// epilogue's residual, res_t[t] (tagged, `res_tag`) or res_p[t] (plain), into
// res_dst[t]. Returns false on timeout or abort (all threads agree).
// What stage_vec needs besides the source: the workspace state (for the
// bounded waits) and the head layout (XMODE 2).
struct StageCtx {
    unsigned* state;
    int n_q, n_kv, head_dim;
};

template <int XMODE>
__device__ __forceinline__ bool stage_vec(const StageCtx& p, const uint2* src_t, const float* src_p, unsigned tag,
                                          int kseg, float* xs, float* xfac, float* red, int* flag,
                                          const uint2* res_t, const float* res_p, unsigned res_tag, float* res_dst,
                                          int nres, int trace_op) {
    (void)trace_op;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n4 = kseg / 4;  // a multiple of 64
    bool ok = true;
    // residual: issued first, checked after the vector's loads
    uint2 ra = make_uint2(0u, res_tag);
    if (tid < nres) {
        if (res_p != nullptr)
            ra.x = __float_as_uint(res_p[tid]);
        else
            ra = ld_l2_pair(res_t + tid);
    }
    float ssq = 0.f, mx = 0.f;
    // XMODE 2 reads only the n_kv V heads (group query heads share each) and
    // writes every value to the group positions that use it
    const int group = XMODE == 2 ? p.n_q / p.n_kv : 1;
    const int nsrc4 = XMODE == 2 ? (p.n_kv * p.head_dim) / 4 : n4;
    const int src_off = XMODE == 2 ? (p.n_q + p.n_kv) * p.head_dim : 0;
    for (int base = 0; base < nsrc4; base += 8 * kNC) {
        float4 v[8];
        unsigned miss = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int c = base + i * kNC + tid;
            v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (c < nsrc4) {
                if (src_p != nullptr)
                    v[i] = ld_l2_f4(src_p + 4 * c);
                else if (!ld_tagged4(src_t, src_off + 4 * c, tag, v[i]))
                    miss |= 1u << i;
            }
        }
        if (miss != 0) {
            // some pairs were not yet current: re-read those (bounded)
            WaitClock clk;
            while (miss != 0 && ok) {
                if (!clk.tick(p.state)) {
                    ok = false;
                    break;
                }
                __nanosleep(32);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if ((miss & (1u << i)) && ld_tagged4(src_t, src_off + 4 * (base + i * kNC + tid), tag, v[i]))
                        miss &= ~(1u << i);
            }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int c = base + i * kNC + tid;
            if (base + i * kNC >= nsrc4) break;  // uniform over the CTA
            if (c < nsrc4) {
                if constexpr (XMODE == 2) {
                    const int e = 4 * c, g = e / p.head_dim, o = e - g * p.head_dim;
                    for (int m = 0; m < group; ++m) {
                        const int k = (g * group + m) * p.head_dim + o;
                        *reinterpret_cast<float4*>(xs + xpad_idx(k)) = v[i];
                    }
                } else {
                    *reinterpret_cast<float4*>(xs + xpad_idx(4 * c)) = v[i];
                }
                mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)), fmaxf(fabsf(v[i].z), fabsf(v[i].w))));
                if constexpr (XMODE == 1) {
                    ssq = fmaf(v[i].x, v[i].x, ssq);
                    ssq = fmaf(v[i].y, v[i].y, ssq);
                    ssq = fmaf(v[i].z, v[i].z, ssq);
                    ssq = fmaf(v[i].w, v[i].w, ssq);
                }
            }
        }
    }
    if (tid < nres) {
        WaitClock clk;
        while (ra.y != res_tag && ok) {
            if (!clk.tick(p.state)) {
                ok = false;
                break;
            }
            __nanosleep(32);
            ra = ld_l2_pair(res_t + tid);
        }
        res_dst[tid] = __uint_as_float(ra.x);
    }
    if (!ok) *flag = 1;
    if (tid == 0) PHB_TRACE_EV(trace_op, 4);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
        ssq += __shfl_xor_sync(0xFFFFFFFFu, ssq, o);
    }
    if (lane == 0) {
        red[warp] = mx;
        red[kCW + warp] = ssq;
    }
    consumer_sync<kNC>();
    if (tid == 0) PHB_TRACE_EV(trace_op, 5);
    // every thread derives the same scale from the per-warp partials
    float m = 0.f, sq = 0.f;
    for (int w = 0; w < kCW; ++w) {
        m = fmaxf(m, red[w]);
        sq += red[kCW + w];
    }
    const float r = XMODE == 1 ? rsqrtf(sq / static_cast<float>(kseg) + kRmsEps) : 1.f;
    const int se = pick_scale_exp(m * r);
    const int e1 = min(se, 127);
    const float f1 = __int_as_float((e1 + 127) << 23), f2 = __int_as_float((se - e1 + 127) << 23);
    if (tid == 0) xfac[0] = __int_as_float((kWShift - se + 127) << 23);
    const bool all_ok = *flag == 0;
    for (int k4 = tid; k4 < n4; k4 += kNC) {
        float4* q = reinterpret_cast<float4*>(xs + xpad_idx(4 * k4));
        float4 v = *q;
        if constexpr (XMODE == 1) {
            v.x *= r;
            v.y *= r;
            v.z *= r;
            v.w *= r;
        }
        v.x = v.x * f1 * f2;
        v.y = v.y * f1 * f2;
        v.z = v.z * f1 * f2;
        v.w = v.w * f1 * f2;
        *q = v;
    }
    consumer_sync<kNC>();
    return all_ok;
}

// Segments (row, matrix) per stage for a tile of useg units per segment.
__host__ __device__ __forceinline__ int segs_per_stage(int stage_units, int useg, int nmat) {
    return (stage_units / (nmat * useg)) * nmat;
}

// Warp-wide bounded wait on a stage: lane 0 polls, the warp barrier orders
// the other lanes' reads of the stage after lane 0's completed wait.
__device__ __forceinline__ bool stage_wait(uint64_t* bar, uint32_t parity) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, &g_dev_err) ? 1 : 0;
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    __syncwarp();
    return ok != 0;
}

// This thread's half-unit position within a row segment: consecutive threads
// take consecutive segments at one position (segments fastest), so a warp's
// threads share few positions and the register fill of their activations is
// mostly broadcasts. Threads past segs * 2 useg get the last position (their
// fill stays in range; they compute nothing).
__device__ __forceinline__ int xr_pos(int segs, int useg) { return min(static_cast<int>(threadIdx.x) / segs, 2 * useg - 1); }

// Consumers, activations in registers: dot every staged half unit of the
// tile, park the half-unit sums in `part` (NMAT * rows_here * 2 useg
// floats) and, once the tile is done, sum each row (one thread per row and
// matrix, in row_sum's fixed order) and hand it to epi(r, a0, a1) (a1 the up
// row's sum for NMAT == 2; `rsum` holds NMAT * rows_here floats). Thread t
// works on segment t % segs at position xr_pos(segs, useg) of every stage.
// Returns false on a wait timeout.
template <int QT, int NMAT, int NS, class EpiF>
__device__ __forceinline__ bool consume_xr(const Tile& t, int segs, const uint8_t* stages, uint32_t stage_stride,
                                           uint64_t* full, uint64_t* empty, int& s, const float (&xr)[kHalfK],
                                           float xfac, float* part, float* rsum, bool compute, int trace_op, EpiF epi) {
    (void)trace_op;
    using C = KCfg<QT, kCW, NS>;
    const int tid = threadIdx.x, lane = tid & 31;
    const int seg_half = 2 * t.useg;
    const int j = tid % segs, pos = tid / segs;
    const int ss = seg_stride_bytes(t.useg, C::ub);
    const int nseg = NMAT * t.rows_here;
    for (int seg0 = 0; seg0 < nseg; seg0 += segs, ++s) {
        const int slot = s % C::ns;
        if (!stage_wait(&full[slot], (s / C::ns) & 1)) {
            if (lane == 0) mbar_wait(&full[slot], (s / C::ns) & 1, &g_dev_err);  // second bounded wait for the copy
            return false;
        }
        const int seg = seg0 + j;
        if (compute && pos < seg_half && seg < nseg) {
            const uint8_t* ub = stages + static_cast<size_t>(slot) * stage_stride + j * ss + (pos >> 1) * C::ub;
            float acc;
            if constexpr (QT == 0)
                acc = dot_q8_0_half_xr(ub + 136 * (pos & 1), xr, xfac);
            else
                acc = dot_q4_k_half_xr(ub, pos & 1, xr, xfac);
            part[seg * seg_half + pos] = acc;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
    }
    if (!compute) return true;
    if (threadIdx.x == 0) PHB_TRACE_EV(trace_op, 7);
    consumer_sync<kNC>();
    // one thread per (row, matrix) sum, in row_sum's fixed order; the gate/up
    // pair meets in rsum
    for (int it = tid; it < nseg; it += kNC) {
        const float v = row_sum(part + static_cast<size_t>(it) * seg_half, seg_half);
        if constexpr (NMAT == 1)
            epi(it, v, 0.f);
        else
            rsum[it] = v;
    }
    if constexpr (NMAT == 2) {
        consumer_sync<kNC>();
        for (int r = tid; r < t.rows_here; r += kNC) epi(r, rsum[2 * r], rsum[2 * r + 1]);
    }
    return true;
}


}  // namespace
}  // namespace phb
