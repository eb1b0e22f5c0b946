// Persistent decode step: the whole stack of dense decoder layers as one
// cooperative kernel, one CTA per SM.
//
// The 4 GEMVs of a layer (QKV, O, gate/up, down) form a chain where every
// GEMV needs the whole output vector of the one before. Launching one kernel
// per GEMV restarts the weight stream of every CTA at every boundary. Here
// each CTA keeps one deep ring of shared-memory stages for the whole step:
// its producer warp streams the CTA's row slice of every GEMV in chain order,
// running ahead across GEMV boundaries, so the next GEMVs' weights are
// already resident while the previous output vector is exchanged.
//
// Activations stay in registers. A consumer thread owns one fixed half-unit
// position (128 consecutive k) of the GEMV's rows and keeps those 128 scaled
// activations (and their four 32-sums) in registers for the whole GEMV, so
// per weight only the quantized bytes come from shared memory. A stage holds
// whole row segments: with useg units per row segment, a stage carries
// floor(128 / (nmat * useg)) * nmat segments and thread t works on segment
// t / (2 * useg), half unit t % (2 * useg).
//
// Readiness travels with the data. Every intermediate vector (qkv, x1, the
// SwiGLU activation, each layer's output) is stored as 64-bit pairs
// {fp32 value, tag} written by one 8-byte store, tag = epoch * n_ops + op + 1
// naming the GEMV and the call that wrote it, so no fence is needed on the
// writer's side. After its slice of a GEMV is stored each CTA adds one to the
// GEMV's arrival counter (relaxed); a CTA that needs the output polls that
// counter with one thread until every CTA has arrived, then reads the vector
// once, re-reading (bounded) only pairs whose tag is not yet the expected one.
// The counter only saves polling traffic; the tags decide. The last CTA to
// finish zeroes the counters and advances the epoch, so consecutive calls and
// graph replays never mistake an older value for a current one. The
// workspace must be zeroed before its first use.
//
// Every wait is bounded by wall clock; a wait that runs out sets the
// workspace's abort word (all CTAs then drain their rings without computing)
// and this translation unit's device error word. A workspace left aborted
// reports the error again on every later call until it is zeroed.
#include <algorithm>
#include <cstdint>

#ifdef PHB_TRACE
// Debug builds only: per-stage times of the first CTAs [cta][stage][issued, ready, wait start].
constexpr int kStTraceCtas = 4, kStTraceStages = 512;
static __device__ unsigned long long g_stage_trace[kStTraceCtas * kStTraceStages * 3];
#define PHB_STAGE_HOOK(kind, s)                                                                       \
    do {                                                                                              \
        if (blockIdx.x < kStTraceCtas && (s) < kStTraceStages) {                                      \
            unsigned long long t_;                                                                    \
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_));                                    \
            g_stage_trace[(blockIdx.x * kStTraceStages + (s)) * 3 + (kind)] = t_;                      \
        }                                                                                             \
    } while (0)
#endif

#include "gemv_plan.cuh"
#include "phb_internal.h"

namespace phb {

cudaError_t read_dev_err_decode_persistent(int* code) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_dev_err, sizeof(int));
    if (e != cudaSuccess) return e;
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_dev_err, &zero, sizeof(int));
    *code = v;
    return e;
}

#ifdef PHB_TRACE
extern "C" int phb_trace_read_persistent(void* dst, size_t bytes) {
    if (bytes > sizeof(g_trace)) bytes = sizeof(g_trace);
    return static_cast<int>(cudaMemcpyFromSymbol(dst, g_trace, bytes));
}
extern "C" int phb_trace_read_stages(void* dst, size_t bytes) {
    if (bytes > sizeof(g_stage_trace)) bytes = sizeof(g_stage_trace);
    return static_cast<int>(cudaMemcpyFromSymbol(dst, g_stage_trace, bytes));
}
#endif

namespace {

// 11 consumer warps + the producer warp: 12 warps, three per scheduler, at
// the 168 registers the 128 resident activations need (65,536 / 384 threads).
constexpr int kCW = 11;            // consumer warps per CTA
constexpr int kNC = 32 * kCW;      // consumer threads
constexpr int kMaxLayers = 64;
constexpr int kHalfK = 128;        // activations a consumer thread keeps in registers
// Every intermediate vector is stored kRep times (replicas one stride apart)
// and CTA i reads replica i % kRep, so the 152 readers of a vector spread
// over kRep sets of L2 lines instead of queueing on one.
constexpr int kRep = 8;
constexpr uint64_t kOpWaitNs = 2000000000ull;
// state words: [0] finish counter, [1] abort, [2] epoch, [kCtrBase + op] CTAs done with op
constexpr int kCtrBase = 64;
constexpr int kStateWords = kCtrBase + 4 * kMaxLayers;

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

struct LayerW {
    const uint8_t* w[5];  // qkv, o, gate, up, down
};

struct PersistParams {
    LayerW layers[kMaxLayers];
    int n_layers;
    int d_model, q_dim, qkv_dim, d_ff;
    int n_q, n_kv, head_dim;
    int64_t rb_dm, rb_q, rb_ff;    // row bytes of rows with K = d_model, q_dim, d_ff
    const float* x_in;
    float* x_out;
    uint2* qkv;                    // tagged intermediate vectors in the workspace
    uint2* x1;
    uint2* act;
    uint2* xl[2];
    int64_t rs_qkv, rs_dm, rs_ff;  // replica strides (pairs) of qkv, the d_model vectors, act
    unsigned* state;
    uint32_t xs_off, xsum_off, part_off, res_off, bar_off;
};

// Stage one activation vector of kseg floats for the register-resident
// dot: one coalesced read pass (four values per lane and load group, up to 8
// groups in flight per thread), raw values into xs (padded layout), 32-sums
// into xsum, then scaled in place exactly as the launched GEMV's staging
// does: x * r (RMSNorm) * 2^s. The source is a tagged vector (pairs carrying
// `tag`; pairs that are not yet current are re-read, bounded) or, for the
// first layer, the caller's plain vector. XMODE: 0 plain, 1 RMSNorm, 2 gather
// of the V heads. In the same pass threads t < nres read the next
// epilogue's residual, res_t[t] (tagged, `res_tag`) or res_p[t] (plain), into
// res_dst[t]. Returns false on timeout or abort (all threads agree).
template <int XMODE>
__device__ __forceinline__ bool stage_vec(const PersistParams& p, const uint2* src_t, const float* src_p, unsigned tag,
                                          int kseg, float* xs, float* xsum, float* xfac, float* red, int* flag,
                                          const uint2* res_t, const float* res_p, unsigned res_tag, float* res_dst,
                                          int nres, int* retries, int trace_op) {
    (void)trace_op;
    (void)retries;
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
#ifdef PHB_TRACE
        if (tid == 0 && base == 0) {
            float chk = v[0].x;  // wait for the first pass's data
            asm volatile("" ::"f"(chk));
            if (miss == 0) PHB_TRACE_EV(trace_op, 8);
        }
        if (miss != 0 && retries != nullptr) atomicAdd(retries, 1);
#endif
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
            float cs = (v[i].x + v[i].y) + (v[i].z + v[i].w);
            cs += __shfl_xor_sync(0xFFFFFFFFu, cs, 1);
            cs += __shfl_xor_sync(0xFFFFFFFFu, cs, 2);
            cs += __shfl_xor_sync(0xFFFFFFFFu, cs, 4);
            if (c < nsrc4) {
                if constexpr (XMODE == 2) {
                    const int e = 4 * c, g = e / p.head_dim, o = e - g * p.head_dim;
                    for (int m = 0; m < group; ++m) {
                        const int k = (g * group + m) * p.head_dim + o;
                        *reinterpret_cast<float4*>(xs + xpad_idx(k)) = v[i];
                        if ((lane & 7) == 0) xsum[k >> 5] = cs;
                    }
                } else {
                    *reinterpret_cast<float4*>(xs + xpad_idx(4 * c)) = v[i];
                    if ((lane & 7) == 0) xsum[c >> 3] = cs;
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
#ifdef PHB_TRACE
    if (tid == 0) {
        if (trace_op < kTraceLaunches && blockIdx.x < kTraceCtas)
            g_trace[(trace_op * kTraceCtas + blockIdx.x) * kTraceEvents + 9] = static_cast<uint64_t>(*retries);
        *retries = 0;
    }
#endif
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
    if (tid == 0) xfac[0] = __int_as_float((149 - se + 127) << 23);
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
    if constexpr (XMODE == 1) {
        for (int i = tid; i < kseg / 32; i += kNC) xsum[i] *= r;
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

// Consumers, activations in registers: dot every staged half unit of the
// tile, park the half-unit sums in `part` (2 * NMAT * rows_here * useg
// floats) and, once the tile is done, sum each row (one thread per row and
// matrix, half units in order) and hand it to epi(r, a0, a1) (a1 the up
// row's sum for NMAT == 2; `rsum` holds NMAT * rows_here floats). Returns
// false on a wait timeout.
template <int QT, int NMAT, int NS, class EpiF>
__device__ __forceinline__ bool consume_xr(const Tile& t, int segs, const uint8_t* stages, uint64_t* full,
                                           uint64_t* empty, int& s, const float (&xr)[kHalfK], const float (&xsr)[4],
                                           float xfac, float* part, float* rsum, bool compute, int trace_op,
                                           EpiF epi) {
    (void)trace_op;
    using C = KCfg<QT, kCW, NS>;
    const int tid = threadIdx.x, lane = tid & 31;
    const int seg_half = 2 * t.useg;
    const int j = tid / seg_half, pos = tid - j * seg_half;
    const int nseg = NMAT * t.rows_here;
    for (int seg0 = 0; seg0 < nseg; seg0 += segs, ++s) {
        const int slot = s % C::ns;
        if (threadIdx.x == 0) PHB_STAGE_HOOK(2, s);
        if (!stage_wait(&full[slot], (s / C::ns) & 1)) {
            if (lane == 0) mbar_wait(&full[slot], (s / C::ns) & 1, &g_dev_err);  // second bounded wait for the copy
            return false;
        }
        if (threadIdx.x == 0) PHB_STAGE_HOOK(1, s);
        const int seg = seg0 + j;
        if (compute && j < segs && seg < nseg) {
            const uint8_t* ub = stages + slot * C::stage_bytes + (j * t.useg + (pos >> 1)) * C::ub;
            float acc;
            if constexpr (QT == 0)
                acc = dot_q8_0_half_xr(ub + 136 * (pos & 1), xr, xsr, xfac);
            else
                acc = dot_q4_k_half_xr(ub, pos & 1, xr, xsr, xfac);
            part[seg * seg_half + pos] = acc;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
    }
    if (!compute) return true;
    if (threadIdx.x == 0) PHB_TRACE_EV(trace_op, 7);
    consumer_sync<kNC>();
    // one thread per (row, matrix) sum, half units in order; the gate/up
    // pair meets in rsum
    for (int it = tid; it < nseg; it += kNC) {
        const float* q = part + static_cast<size_t>(it) * seg_half;
        float v = 0.f;
        for (int h = 0; h < seg_half; ++h) v += q[h];
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

template <int QT, int NS>
__global__ void __launch_bounds__(KCfg<QT, kCW>::threads, 1) decode_persistent_kernel(const __grid_constant__ PersistParams p) {
    using C = KCfg<QT, kCW, NS>;
    extern __shared__ __align__(1024) uint8_t smem[];
    float* xs = reinterpret_cast<float*>(smem + p.xs_off);
    float* xsum = reinterpret_cast<float*>(smem + p.xsum_off);
    float* part = reinterpret_cast<float*>(smem + p.part_off);
    float* res = reinterpret_cast<float*>(smem + p.res_off);
    float* rsum = res + kNC;  // NMAT * rows_here row sums
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.bar_off);
    uint64_t* empty = full + C::ns;
    float* xfac = reinterpret_cast<float*>(empty + C::ns);
    float* red = xfac + kAccStride;
    int* flag = reinterpret_cast<int*>(red + (2 * kMaxConsumerWarps + 3) * kAccStride);
#ifdef PHB_TRACE
    int* retries = flag + 1;  // debug builds: re-read rounds of the staging pass
#else
    int* retries = nullptr;
#endif

    const int tid = threadIdx.x;
    const int nctas = gridDim.x;
    const int n_ops = 4 * p.n_layers;
    if (tid == 0) {
        for (int s = 0; s < C::ns; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kCW);
        }
        fence_barrier_init();
        *flag = 0;
        if (retries != nullptr) *retries = 0;
    }
    __syncthreads();
    const unsigned epoch = ld_relaxed(p.state + 2);
    pdl_launch_dependents();

    // the tile of op `op` owned by this CTA, and its segments per stage
    auto op_tile = [&](int op, Tile& t, int& nmat, int64_t& row0, int& segs) -> bool {
        const LayerW& L = p.layers[op >> 2];
        int n, useg;
        int64_t rb;
        const uint8_t *w0, *w1;
        switch (op & 3) {
            case 0: n = p.qkv_dim; useg = p.d_model / kUnitWeights; rb = p.rb_dm; w0 = w1 = L.w[0]; nmat = 1; break;
            case 1: n = p.d_model; useg = p.q_dim / kUnitWeights; rb = p.rb_q; w0 = w1 = L.w[1]; nmat = 1; break;
            case 2: n = p.d_ff; useg = p.d_model / kUnitWeights; rb = p.rb_dm; w0 = L.w[2]; w1 = L.w[3]; nmat = 2; break;
            default: n = p.d_model; useg = p.d_ff / kUnitWeights; rb = p.rb_ff; w0 = w1 = L.w[4]; nmat = 1; break;
        }
        const int rpc = (n + nctas - 1) / nctas;
        row0 = static_cast<int64_t>(blockIdx.x) * rpc;
        t.rows_here = static_cast<int>(min(static_cast<int64_t>(rpc), n - row0));
        t.useg = useg;
        t.row_bytes = rb;
        t.contiguous = true;
        t.w[0] = w0 + row0 * rb;
        t.w[1] = w1 + row0 * rb;
        segs = segs_per_stage(C::stage_units, useg, nmat);
        return t.rows_here > 0;
    };

    if (tid >= C::consumers) {
        // ---------------- producer: every op's slice, in chain order, through one ring
        if (tid == C::consumers) {
            const uint64_t pol = policy_evict_first();
            int s = 0;
            for (int op = 0; op < n_ops; ++op) {
                Tile t;
                int nmat, segs;
                int64_t row0;
                if (!op_tile(op, t, nmat, row0, segs)) continue;
                if (!produce_tile<QT, kCW, NS>(t, nmat, smem, full, empty, s, pol, segs * t.useg)) break;
            }
        }
        return;
    }

    int s = 0;
    bool alive = true;
    for (int op = 0; op < n_ops; ++op) {
        Tile t;
        int nmat, segs;
        int64_t row0;
        const bool mine = op_tile(op, t, nmat, row0, segs);
        const int l = op >> 2, j = op & 3;
        const unsigned tag_prev = epoch * n_ops + op;  // tag of op - 1
        const unsigned tag_me = tag_prev + 1;
        const unsigned tag_lin = epoch * n_ops + 4 * l;  // tag of the op that wrote this layer's input
        if (!mine) {
            if (tid == 0) atomicAdd(p.state + kCtrBase + op, 1u);  // nothing to write for this op
            continue;
        }
        const int kseg = t.useg * kUnitWeights;
        if (tid == 0) PHB_TRACE_EV(op, 0);
        // wait until every CTA has counted its arrival at the op this one reads
        if (alive && op > 0) {
            if (tid == 0 && !wait_op_arrivals(p.state, op - 1, static_cast<unsigned>(nctas))) *flag = 1;
            consumer_sync<kNC>();
            if (*flag) alive = false;
        }
        if (tid == 0) PHB_TRACE_EV(op, 1);
        // this layer's input: the caller's vector or the previous layer's output
        const int rep = blockIdx.x % kRep;
        const uint2* lin_t = l == 0 ? nullptr : p.xl[(l - 1) & 1] + rep * p.rs_dm;
        const float* lin_p = l == 0 ? p.x_in : nullptr;
        if (alive) {
            bool ok;
            switch (j) {
                case 0:
                    ok = stage_vec<1>(p, lin_t, lin_p, tag_lin, kseg, xs, xsum, xfac, red, flag, nullptr, nullptr, 0,
                                      res, 0, retries, op);
                    break;
                case 1:
                    ok = stage_vec<2>(p, p.qkv + rep * p.rs_qkv, nullptr, tag_prev, kseg, xs, xsum, xfac, red, flag,
                                      lin_t ? lin_t + row0 : nullptr, lin_p ? lin_p + row0 : nullptr, tag_lin, res,
                                      t.rows_here, retries, op);
                    break;
                case 2:
                    ok = stage_vec<1>(p, p.x1 + rep * p.rs_dm, nullptr, tag_prev, kseg, xs, xsum, xfac, red, flag, nullptr, nullptr, 0,
                                      res, 0, retries, op);
                    break;
                default:
                    ok = stage_vec<0>(p, p.act + rep * p.rs_ff, nullptr, tag_prev, kseg, xs, xsum, xfac, red, flag,
                                      p.x1 + rep * p.rs_dm + row0,
                                      nullptr, tag_me - 2, res, t.rows_here, retries, op);
                    break;
            }
            alive = ok;
        }
        if (tid == 0) PHB_TRACE_EV(op, 2);
        // this thread's half-unit position: activations and 32-sums into registers
        float xr[kHalfK], xsr[4];
        {
            const int pos = tid % (2 * t.useg);
            const float* xp = xs + pos * (kXPadEvery + kXPad);
#pragma unroll
            for (int i = 0; i < kHalfK; i += 4) {
                const float4 v = *reinterpret_cast<const float4*>(xp + i);
                xr[i] = v.x;
                xr[i + 1] = v.y;
                xr[i + 2] = v.z;
                xr[i + 3] = v.w;
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) xsr[i] = xsum[4 * pos + i];
        }
        const float xf = xfac[0];
        const bool last = (l == p.n_layers - 1);
        auto store_all = [&](uint2* buf, int64_t rs, int64_t n, float v) {
#pragma unroll
            for (int q = 0; q < kRep; ++q) st_pair(buf + q * rs + n, v, tag_me);
        };
        auto epi = [&](int r, float a0, float a1) {
            const int64_t n = row0 + r;
            switch (j) {
                case 0: store_all(p.qkv, p.rs_qkv, n, a0); break;
                case 1: store_all(p.x1, p.rs_dm, n, res[r] + a0); break;
                case 2: store_all(p.act, p.rs_ff, n, silu_mul(a0, a1)); break;
                default:
                    if (last)
                        p.x_out[n] = res[r] + a0;
                    else
                        store_all(p.xl[l & 1], p.rs_dm, n, res[r] + a0);
                    break;
            }
        };
        // on abort the stages are still drained (no copy may be left in flight)
        bool ok;
        if (nmat == 2)
            ok = consume_xr<QT, 2, NS>(t, segs, smem, full, empty, s, xr, xsr, xf, part, rsum, alive, op, epi);
        else
            ok = consume_xr<QT, 1, NS>(t, segs, smem, full, empty, s, xr, xsr, xf, part, rsum, alive, op, epi);
        alive = alive && ok;
        consumer_sync<kNC>();
        if (tid == 0) {
            PHB_TRACE_EV(op, 3);
            atomicAdd(p.state + kCtrBase + op, 1u);  // this CTA's outputs of op are stored (readers check tags)
            PHB_TRACE_EV(op, 6);
        }
    }
    // the last CTA to finish resets the counters and advances the epoch
    if (tid == 0) {
        __threadfence();
        const unsigned prev = atomicAdd(p.state, 1u);
        if (prev == static_cast<unsigned>(nctas) - 1) {
            for (int op = 0; op < n_ops; ++op) p.state[kCtrBase + op] = 0;
            p.state[0] = 0;
            p.state[2] = epoch + 1;
        }
    }
}

// Every CTA must be resident at once (they wait on each other's outputs): one
// CTA per SM, which the cooperative launch guarantees or refuses.
template <int QT, int NS>
cudaError_t launch_persistent(cudaLaunchConfig_t cfg, const PersistParams& p) {
    constexpr auto kern = decode_persistent_kernel<QT, NS>;
    cudaError_t e = ensure_smem_attr<kern>();
    if (e != cudaSuccess) return e;
    cfg.blockDim = dim3(KCfg<QT, kCW>::threads);
    return cudaLaunchKernelEx(&cfg, kern, p);
}

// Ring depths: the deep ring keeps ~180 KB of weights in flight per SM so
// that the copies of the next GEMVs run while a dependent activation vector
// is exchanged; the shallow one is for shapes whose activations leave less
// room.
template <int QT>
struct Rings {
    static constexpr int deep = QT == 0 ? 4 : 7;
    static constexpr int shallow = QT == 0 ? 2 : 3;
};

}  // namespace

// Workspace of the persistent step: tagged intermediate vectors and the state words.
size_t decode_persistent_ws_bytes(int64_t d_model, int n_q, int n_kv, int hd, int64_t d_ff) {
    auto al = [](size_t v) { return (v + 255) & ~size_t{255}; };
    size_t b = al(kStateWords * 4);
    b += kRep * al(static_cast<size_t>(n_q + 2 * n_kv) * hd * 8);
    b += kRep * al(static_cast<size_t>(d_model) * 8) * 3;
    b += kRep * al(static_cast<size_t>(d_ff) * 8);
    return b;
}

cudaError_t decode_persistent_run(int qt, const void* const* wl, int n_layers, int64_t d_model, int n_q, int n_kv,
                                  int hd, int64_t d_ff, const float* x_in, float* x_out, void* ws, cudaStream_t s) {
    if (n_layers > kMaxLayers) return cudaErrorInvalidValue;
    auto al = [](size_t v) { return (v + 255) & ~size_t{255}; };
    PersistParams p{};
    for (int l = 0; l < n_layers; ++l)
        for (int i = 0; i < 5; ++i) p.layers[l].w[i] = static_cast<const uint8_t*>(wl[5 * l + i]);
    p.n_layers = n_layers;
    p.d_model = static_cast<int>(d_model);
    p.q_dim = n_q * hd;
    p.qkv_dim = (n_q + 2 * n_kv) * hd;
    p.d_ff = static_cast<int>(d_ff);
    p.n_q = n_q;
    p.n_kv = n_kv;
    p.head_dim = hd;
    const int ub = qt == 0 ? Fmt<0>::unit_bytes : Fmt<1>::unit_bytes;
    p.rb_dm = d_model / kUnitWeights * ub;
    p.rb_q = static_cast<int64_t>(p.q_dim) / kUnitWeights * ub;
    p.rb_ff = d_ff / kUnitWeights * ub;
    p.x_in = x_in;
    p.x_out = x_out;
    auto* b = static_cast<uint8_t*>(ws);
    size_t off = 0;
    p.state = reinterpret_cast<unsigned*>(b);
    off += al(kStateWords * 4);
    p.rs_qkv = static_cast<int64_t>(al(static_cast<size_t>(p.qkv_dim) * 8) / 8);
    p.rs_dm = static_cast<int64_t>(al(static_cast<size_t>(d_model) * 8) / 8);
    p.rs_ff = static_cast<int64_t>(al(static_cast<size_t>(d_ff) * 8) / 8);
    p.qkv = reinterpret_cast<uint2*>(b + off);
    off += kRep * p.rs_qkv * 8;
    p.x1 = reinterpret_cast<uint2*>(b + off);
    off += kRep * p.rs_dm * 8;
    p.xl[0] = reinterpret_cast<uint2*>(b + off);
    off += kRep * p.rs_dm * 8;
    p.xl[1] = reinterpret_cast<uint2*>(b + off);
    off += kRep * p.rs_dm * 8;
    p.act = reinterpret_cast<uint2*>(b + off);

    const int grid = device_sm_count();
    constexpr int kStageUnits = KCfg<0, kCW>::stage_units;
    // every GEMV's row segment must fit one stage (with the gate/up pair) and
    // the residual rows one pass of the consumer threads
    static_assert(KCfg<0, kCW>::stage_units == KCfg<1, kCW>::stage_units, "one stage size");
    const int64_t kmax = std::max<int64_t>({d_model, static_cast<int64_t>(p.q_dim), d_ff});
    if (2 * (d_model / kUnitWeights) > kStageUnits || kmax / kUnitWeights > kStageUnits)
        return cudaErrorInvalidConfiguration;
    const int64_t max_rows = std::max<int64_t>({(p.qkv_dim + grid - 1) / grid, (d_model + grid - 1) / grid,
                                               (d_ff + grid - 1) / grid});
    if ((d_model + grid - 1) / grid > kNC) return cudaErrorInvalidConfiguration;
    if (hd % 32 != 0 || n_q % n_kv != 0) return cudaErrorInvalidConfiguration;  // gather by whole 32-blocks
    const int max_useg = static_cast<int>(kmax / kUnitWeights);
    const int deep = qt == 0 ? Rings<0>::deep : Rings<1>::deep;
    const int shallow = qt == 0 ? Rings<0>::shallow : Rings<1>::shallow;
    // every op may need tile partials (2 * nmat * rows * useg floats)
    const size_t tile_part = 2 * 2 * static_cast<size_t>(max_rows) * max_useg * sizeof(float);
    int ns = 0;
    size_t smem = 0;
    for (int cand : {deep, shallow}) {
        const SmemLayout lay = stream_smem_layout(qt, kCW, 2, 1, static_cast<int>(max_rows), max_useg, cand);
        const size_t res_off = lay.part + tile_part;
        // residuals (kNC floats) then row sums (2 * max_rows floats)
        const size_t bar_off = (res_off + (kNC + 2 * static_cast<size_t>(max_rows)) * sizeof(float) + 15) & ~size_t{15};
        const size_t total = bar_off + 2 * cand * sizeof(uint64_t) + kTailFloats * sizeof(float);
        if (total > kSmemOptin) continue;
        ns = cand;
        smem = total;
        p.xs_off = lay.xs;
        p.xsum_off = lay.xsum;
        p.part_off = lay.part;
        p.res_off = static_cast<uint32_t>(res_off);
        p.bar_off = static_cast<uint32_t>(bar_off);
        break;
    }
    if (ns == 0) return cudaErrorInvalidConfiguration;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.dynamicSmemBytes = smem;
    if (qt == 0)
        return ns == deep ? launch_persistent<0, Rings<0>::deep>(cfg, p) : launch_persistent<0, Rings<0>::shallow>(cfg, p);
    return ns == deep ? launch_persistent<1, Rings<1>::deep>(cfg, p) : launch_persistent<1, Rings<1>::shallow>(cfg, p);
}

}  // namespace phb
