// Top-k routed mixture-of-experts FFN.
//
// 1. moe_route_kernel (one CTA): per token the top_k largest router logits
//    (ties to the lower expert index) and their softmax; then a counting sort
//    of the (token, slot) pairs by expert, ascending pair id within an
//    expert, giving the active-expert list.
// 2. moe_stream_kernel<NMAT=2>: grid (CTAs per expert, expert slot). Each CTA
//    streams a row range of its expert's gate and up matrices once and
//    applies it to every token routed to that expert (groups of up to 8),
//    writing h[pair] = silu(gate.x) * (up.x).
// 3. moe_stream_kernel<NMAT=1>: the same over the down matrices, x = h[pair],
//    writing y_pair[pair].
// 4. moe_combine_kernel: y[t] = sum over slots (ascending) of p[t][slot] *
//    y_pair[t*top_k + slot].
// All orders are fixed, so repeated calls give identical bits.
#include <algorithm>
#include <cfloat>
#include <cmath>

#include "gemv_plan.cuh"
#include "phb_internal.h"

namespace phb {

cudaError_t read_dev_err_moe(int* code) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_dev_err, sizeof(int));
    if (e != cudaSuccess) return e;
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_dev_err, &zero, sizeof(int));
    *code = v;
    return e;
}

#ifdef PHB_TRACE
extern "C" int phb_trace_read_moe(void* dst, size_t bytes) {
    if (bytes > sizeof(g_trace)) bytes = sizeof(g_trace);
    return static_cast<int>(cudaMemcpyFromSymbol(dst, g_trace, bytes));
}
#endif

namespace {

constexpr int kMaxExperts = 256;
constexpr int kMaxTopK = 8;
constexpr int kMaxTokens = 64;
// Tokens per pass over a staged weight tile. Four keeps the staged
// activations small enough for two CTAs per SM; an expert chosen by more
// tokens streams its tile once per group of four.
constexpr int kMoeGroup = 4;
constexpr int kMoeCW = 8;     // consumer warps of the grouped kernels

struct RouteOut {
    int32_t* idx;        // [T][k]
    float* p;            // [T][k]
    int32_t* n_active;   // [1]
    int32_t* act_expert; // [slots]
    int32_t* act_off;    // [slots]
    int32_t* act_cnt;    // [slots]
    int32_t* pair_list;  // [T*k]
};

// Order-preserving map of a finite float to an unsigned key (larger float,
// larger key).
__device__ __forceinline__ uint32_t float_key(float v) {
    const uint32_t u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_float(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Routing. Warps take tokens; per token, K rounds of a warp-wide arg-max
// (largest logit, then lowest expert index) over the logits held in
// registers give the top_k in slot order, and lane 0 takes their softmax.
// Then warp 0 sorts the (token, slot) pairs by expert with a stable
// counting sort (match groups per 32 pairs, a warp scan over the experts)
// and lists the active experts in ascending order.
__global__ void __launch_bounds__(256) moe_route_kernel(const float* __restrict__ logits, int T, int E, int K,
                                                        RouteOut o, int32_t* out_idx, float* out_p, int trace_id) {
    (void)trace_id;
    if (threadIdx.x == 0) PHB_TRACE_EV(trace_id, 0);
    pdl_launch_dependents();
    pdl_wait();
    if (threadIdx.x == 0) PHB_TRACE_EV(trace_id, 1);
    __shared__ int32_t sidx[kMaxTokens * kMaxTopK];
    __shared__ int32_t rank[kMaxTokens * kMaxTopK];
    __shared__ int32_t cnt[kMaxExperts];
    __shared__ int32_t off[kMaxExperts];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nwarps = blockDim.x >> 5;
    for (int e = tid; e < kMaxExperts; e += blockDim.x) cnt[e] = 0;
    for (int t = warp; t < T; t += nwarps) {
        uint32_t key[kMaxExperts / 32];
#pragma unroll
        for (int j = 0; j < kMaxExperts / 32; ++j) {
            const int e = lane + 32 * j;
            key[j] = e < E ? float_key(logits[static_cast<int64_t>(t) * E + e]) : 0u;
        }
        uint32_t taken = 0;
        float sel_v[kMaxTopK];
        int sel_e[kMaxTopK];
#pragma unroll
        for (int r = 0; r < kMaxTopK; ++r) {
            if (r >= K) break;
            // this lane's best untaken expert: largest key, then lowest index (ascending j)
            uint32_t bk = 0;
            int be = 0x7FFFFFFF;
#pragma unroll
            for (int j = 0; j < kMaxExperts / 32; ++j) {
                const int e = lane + 32 * j;
                if (e < E && !((taken >> j) & 1u) && (be == 0x7FFFFFFF || key[j] > bk)) {
                    bk = key[j];
                    be = e;
                }
            }
            const uint32_t kmax = __reduce_max_sync(0xFFFFFFFFu, bk);
            const uint32_t emin = __reduce_min_sync(0xFFFFFFFFu, (be != 0x7FFFFFFF && bk == kmax)
                                                                     ? static_cast<uint32_t>(be) : 0xFFFFFFFFu);
            if (static_cast<int>(emin & 31u) == lane) taken |= 1u << (emin >> 5);
            sel_v[r] = key_float(kmax);
            sel_e[r] = static_cast<int>(emin);
        }
        if (lane == 0) {
            float ex[kMaxTopK];
            float sum = 0.f;
#pragma unroll
            for (int r = 0; r < kMaxTopK; ++r) {
                if (r >= K) break;
                ex[r] = expf(sel_v[r] - sel_v[0]);
                sum += ex[r];
            }
#pragma unroll
            for (int r = 0; r < kMaxTopK; ++r) {
                if (r >= K) break;
                const float pr = ex[r] / sum;
                const int q = t * K + r;
                sidx[q] = sel_e[r];
                o.idx[q] = sel_e[r];
                o.p[q] = pr;
                if (out_idx) out_idx[q] = sel_e[r];
                if (out_p) out_p[q] = pr;
            }
        }
    }
    __syncthreads();
    const int pairs = T * K;
    if (warp == 0) {
        // stable rank of every pair within its expert, 32 pairs at a time
        for (int q0 = 0; q0 < pairs; q0 += 32) {
            const int q = q0 + lane;
            const bool valid = q < pairs;
            const int e = valid ? sidx[q] : -1 - lane;  // invalid lanes match nobody
            const unsigned grp = __match_any_sync(0xFFFFFFFFu, e);
            const int base = valid ? cnt[e] : 0;
            __syncwarp();
            if (valid) {
                rank[q] = base + __popc(grp & ((1u << lane) - 1u));
                if ((__ffs(grp) - 1) == lane) cnt[e] = base + __popc(grp);
            }
            __syncwarp();
        }
        // exclusive scan over experts (8 consecutive experts per lane) and the active list
        constexpr int kPer = kMaxExperts / 32;
        int c[kPer], lc = 0, la = 0;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int e = kPer * lane + i;
            c[i] = e < E ? cnt[e] : 0;
            lc += c[i];
            la += c[i] > 0;
        }
        int sc = lc, sa = la;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int vc = __shfl_up_sync(0xFFFFFFFFu, sc, d), va = __shfl_up_sync(0xFFFFFFFFu, sa, d);
            if (lane >= d) {
                sc += vc;
                sa += va;
            }
        }
        int acc = sc - lc, a = sa - la;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int e = kPer * lane + i;
            if (e < E) {
                off[e] = acc;
                if (c[i] > 0) {
                    o.act_expert[a] = e;
                    o.act_off[a] = acc;
                    o.act_cnt[a] = c[i];
                    ++a;
                }
                acc += c[i];
            }
        }
        if (lane == 31) *o.n_active = sa;
    }
    __syncthreads();
    for (int q = tid; q < pairs; q += blockDim.x) o.pair_list[off[sidx[q]] + rank[q]] = q;
    if (threadIdx.x == 0) PHB_TRACE_EV(trace_id, 3);
}

struct MoeParams {
    const uint8_t* w[2];      // expert 0 of each matrix
    int64_t expert_stride;    // bytes per expert matrix
    int64_t row_bytes;
    int64_t n;                // rows per expert matrix
    int units_row;
    int rows_per_cta;
    const float* x;           // gate/up: X [T][K]; down: h [pairs][K]
    int64_t ldx;
    int x_by_pair;            // 0: x row = pair / top_k; 1: x row = pair
    int top_k;
    float* y;                 // [pairs][n]
    int64_t ldy;
    RouteOut r;
    int sum_mode;
    const uint8_t* pf;        // per-expert matrix to prefetch into L2 (the down matrix), or null
    int64_t pf_stride;        // its bytes per expert
    uint32_t xs_off, xsum_off, part_off, acc_off, bar_off;
    int trace_id;
};

template <int QT, int NMAT, int MAXB>
__device__ __forceinline__ bool moe_group(const MoeParams& p, const Tile& t, int row0, int first_pair_idx, int nb,
                                          uint8_t* smem, uint64_t* full, uint64_t* empty, int& s) {
    float* xs = reinterpret_cast<float*>(smem + p.xs_off);
    float* xsum = reinterpret_cast<float*>(smem + p.xsum_off);
    float* part = reinterpret_cast<float*>(smem + p.part_off);
    float* row_acc = reinterpret_cast<float*>(smem + p.acc_off);
    float* xfac = reinterpret_cast<float*>(full + 2 * KCfg<QT, kMoeCW>::ns);
    float* red = xfac + kAccStride;
    int* rowidx = reinterpret_cast<int*>(red + (2 * kMaxConsumerWarps + 3) * kAccStride);
    const int tid = threadIdx.x;
    const int kseg = t.useg * kUnitWeights;
    if (tid < nb) {
        const int pair = p.r.pair_list[first_pair_idx + tid];
        rowidx[tid] = p.x_by_pair ? pair : pair / p.top_k;
    }
    if (p.sum_mode == kSumFold)
        for (int i = tid; i < NMAT * t.rows_here * kAccStride; i += KCfg<QT, kMoeCW>::consumers) row_acc[i] = 0.f;
    consumer_sync<KCfg<QT, kMoeCW>::consumers>();
    stage_x<kMoeCW, MAXB, kXRowList>(p.x, p.ldx, 0, kseg, nb, xs, xsum, xfac, red, 1, 1, 0, rowidx);
    if (tid == 0) PHB_TRACE_EV(p.trace_id, 2);
    const int* pairs = p.r.pair_list + first_pair_idx;
    auto epi = [&](int r, int b, float a0, float a1) {
        const float out = NMAT == 2 ? silu_mul(a0, a1) : a0;
        p.y[static_cast<int64_t>(pairs[b]) * p.ldy + row0 + r] = out;
    };
    if (!consume_tile<QT, kMoeCW, MAXB, NMAT>(t, p.sum_mode, smem, full, empty, s, xs, xpad_len(kseg), xsum,
                                              kseg / 32, xfac, nb, part, row_acc, epi))
        return false;
    consumer_sync<KCfg<QT, kMoeCW>::consumers>();  // the next group overwrites xs, xsum and row_acc
    return true;
}

template <int QT, int NMAT>
__global__ void __launch_bounds__(KCfg<QT, kMoeCW>::threads, 2) moe_stream_kernel(const __grid_constant__ MoeParams p) {
    using C = KCfg<QT, kMoeCW>;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.bar_off);
    uint64_t* empty = full + C::ns;
    if (threadIdx.x == 0) PHB_TRACE_EV(p.trace_id, 0);
    pdl_launch_dependents();
    pdl_wait();  // routing results (and, for the down pass, h) come from the previous kernels
    if (threadIdx.x == 0) PHB_TRACE_EV(p.trace_id, 1);
    const int slot = blockIdx.y;
    if (slot >= *p.r.n_active) return;
    const int e = p.r.act_expert[slot];
    const int first = p.r.act_off[slot];
    const int cnt = p.r.act_cnt[slot];
    const int row0 = blockIdx.x * p.rows_per_cta;
    Tile t;
    t.rows_here = static_cast<int>(min(static_cast<int64_t>(p.rows_per_cta), p.n - row0));
    if (t.rows_here <= 0) return;
    t.useg = p.units_row;
    t.row_bytes = p.row_bytes;
    t.contiguous = true;
    t.w[0] = p.w[0] + e * p.expert_stride + static_cast<int64_t>(row0) * p.row_bytes;
    t.w[1] = p.w[NMAT - 1] + e * p.expert_stride + static_cast<int64_t>(row0) * p.row_bytes;
    const int tid = threadIdx.x;
    if (tid == 0) {
        for (int s = 0; s < C::ns; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kMoeCW);
        }
        fence_barrier_init();
    }
    __syncthreads();
    const int ngroups = (cnt + kMoeGroup - 1) / kMoeGroup;
    if (tid >= C::consumers) {
        if (tid == C::consumers) {
            const uint64_t pol = policy_evict_first();
            int s = 0;
            for (int gi = 0; gi < ngroups; ++gi)
                if (!produce_tile<QT, kMoeCW>(t, NMAT, smem, full, empty, s, pol)) break;
        } else if (tid == C::consumers + 1 && p.pf != nullptr && blockIdx.x == 0) {
            // the expert's down matrix, needed by the next kernel
            const uint8_t* base = p.pf + e * p.pf_stride;
            for (int64_t off = 0; off < p.pf_stride; off += 32768)
                prefetch_l2(base + off, static_cast<uint32_t>(p.pf_stride - off < 32768 ? p.pf_stride - off : 32768));
        }
        return;
    }
    int s = 0;
    for (int gi = 0; gi < ngroups; ++gi) {
        const int nb = min(kMoeGroup, cnt - gi * kMoeGroup);
        const int fp = first + gi * kMoeGroup;
        bool ok;
        if (nb == 1)
            ok = moe_group<QT, NMAT, 1>(p, t, row0, fp, nb, smem, full, empty, s);
        else if (nb == 2)
            ok = moe_group<QT, NMAT, 2>(p, t, row0, fp, nb, smem, full, empty, s);
        else
            ok = moe_group<QT, NMAT, 4>(p, t, row0, fp, nb, smem, full, empty, s);
        if (!ok) return;
    }
    consumer_sync<C::consumers>();
    if (tid == 0) PHB_TRACE_EV(p.trace_id, 3);
}

__global__ void __launch_bounds__(256) moe_combine_kernel(const float* __restrict__ yp, const float* __restrict__ p,
                                                          float* __restrict__ y, int T, int K, int64_t D,
                                                          int trace_id) {
    (void)trace_id;
    if (threadIdx.x == 0) PHB_TRACE_EV(trace_id, 0);
    pdl_launch_dependents();
    pdl_wait();
    if (threadIdx.x == 0) PHB_TRACE_EV(trace_id, 1);
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= static_cast<int64_t>(T) * D) return;
    const int64_t t = i / D, d = i - t * D;
    float acc = 0.f;
    for (int s = 0; s < K; ++s) acc = fmaf(p[t * K + s], yp[(t * K + s) * D + d], acc);
    y[i] = acc;
    if (threadIdx.x == 0) PHB_TRACE_EV(trace_id, 3);
}

struct MoeWs {
    RouteOut r;
    float* h;
    float* yp;
    size_t bytes;
};

inline size_t align_up(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

MoeWs moe_ws_layout(const MoeReq& q, void* base) {
    const size_t pairs = static_cast<size_t>(q.t) * q.top_k;
    const size_t slots = static_cast<size_t>(std::min<int64_t>(q.e, static_cast<int64_t>(pairs)));
    auto* b = static_cast<uint8_t*>(base);
    size_t off = 0;
    MoeWs w{};
    auto take = [&](size_t bytes) {
        uint8_t* ptr = b ? b + off : nullptr;
        off = align_up(off + bytes);
        return ptr;
    };
    w.r.idx = reinterpret_cast<int32_t*>(take(pairs * 4));
    w.r.p = reinterpret_cast<float*>(take(pairs * 4));
    w.r.n_active = reinterpret_cast<int32_t*>(take(16));
    w.r.act_expert = reinterpret_cast<int32_t*>(take(slots * 4));
    w.r.act_off = reinterpret_cast<int32_t*>(take(slots * 4));
    w.r.act_cnt = reinterpret_cast<int32_t*>(take(slots * 4));
    w.r.pair_list = reinterpret_cast<int32_t*>(take(pairs * 4));
    w.h = reinterpret_cast<float*>(take(pairs * q.d_ff * 4));
    w.yp = reinterpret_cast<float*>(take(pairs * q.d_model * 4));
    w.bytes = off;
    return w;
}

template <int QT, int NMAT>
cudaError_t launch_moe_stream(const MoeParams& p, dim3 grid, size_t smem, cudaStream_t s) {
    constexpr auto kern = moe_stream_kernel<QT, NMAT>;
    cudaError_t e = ensure_smem_attr<kern>();
    if (e != cudaSuccess) return e;
    return launch_kernel(kern, grid, dim3(KCfg<QT, kMoeCW>::threads), smem, s, true, p);
}

// Rows per CTA and shared-memory layout of one grouped pass. `maxb` is the
// largest token group (at most the token count). A CTA gets at most about 8
// stages of weights per token group, and few enough rows that its row sums fit
// the tile partials (the fold mode synchronises the CTA at every stage).
bool plan_moe(int qt, int nmat, int64_t n, int64_t k, int cpe, int maxb, MoeParams* p, unsigned* gx,
              size_t* smem) {
    const int units_row = static_cast<int>(k / kUnitWeights);
    int rows_per_cta = static_cast<int>(cdiv(n, cpe));
    rows_per_cta = std::min(rows_per_cta, std::max(1, 8 * KCfg<0, kMoeCW>::stage_units / (nmat * units_row)));
    SmemLayout lay{};
    for (;;) {
        lay = stream_smem_layout(qt, kMoeCW, nmat, maxb, rows_per_cta, units_row);
        if (lay.total <= kSmemOptin && lay.sum_mode != kSumFold) break;
        if (rows_per_cta == 1) {
            if (lay.total <= kSmemOptin) break;
            return false;
        }
        rows_per_cta = (rows_per_cta + 1) / 2;
    }
    p->units_row = units_row;
    p->rows_per_cta = rows_per_cta;
    p->row_bytes = static_cast<int64_t>(units_row) * (qt == 0 ? Fmt<0>::unit_bytes : Fmt<1>::unit_bytes);
    p->n = n;
    p->expert_stride = n * p->row_bytes;
    p->sum_mode = lay.sum_mode;
    p->xs_off = lay.xs;
    p->xsum_off = lay.xsum;
    p->part_off = lay.part;
    p->acc_off = lay.acc;
    p->bar_off = lay.bar;
    *gx = static_cast<unsigned>(cdiv(n, rows_per_cta));
    *smem = lay.total;
    return true;
}

}  // namespace

size_t moe_ws_bytes(const MoeReq& q) { return moe_ws_layout(q, nullptr).bytes; }

cudaError_t moe_run(const MoeReq& q, cudaStream_t s) {
    const MoeWs w = moe_ws_layout(q, q.ws);
#ifdef PHB_TRACE
    static int trace_call = 0;  // debug builds: 4 trace slots per call, 32 calls
    const int tb = 4 * (trace_call++ % 32);
#else
    const int tb = -1000;
#endif
    const int pairs = static_cast<int>(q.t * q.top_k);
    const int slots = std::min(q.e, pairs);
    cudaError_t e = launch_kernel(moe_route_kernel, dim3(1), dim3(256), 0, s, true, q.logits, static_cast<int>(q.t),
                                  q.e, q.top_k, w.r, q.out_idx, q.out_p, tb);
    if (e != cudaSuccess) return e;
    // CTAs per expert: enough to cover the GPU twice for the expected number
    // of distinct experts, E * (1 - (1 - k/E)^T).
    double expected = q.e * (1.0 - std::pow(1.0 - static_cast<double>(q.top_k) / q.e, static_cast<double>(q.t)));
    expected = std::min<double>(slots, std::max(1.0, expected));
    const int cpe = std::max(1, static_cast<int>(std::ceil(2.0 * device_sm_count() / expected)));

    MoeParams pg{};
    unsigned gx = 0;
    size_t smem = 0;
    // tokens per expert never exceed the token count: size the staged activations for that
    const int maxb = maxb_for(static_cast<int>(std::min<int64_t>(kMoeGroup, q.t)));
    if (!plan_moe(q.qt, 2, q.d_ff, q.d_model, cpe, maxb, &pg, &gx, &smem)) return cudaErrorInvalidConfiguration;
    pg.w[0] = static_cast<const uint8_t*>(q.wg);
    pg.w[1] = static_cast<const uint8_t*>(q.wu);
    pg.x = q.x;
    pg.ldx = q.d_model;
    pg.x_by_pair = 0;
    pg.top_k = q.top_k;
    pg.y = w.h;
    pg.ldy = q.d_ff;
    pg.r = w.r;
    pg.pf = static_cast<const uint8_t*>(q.wd);
    pg.trace_id = tb + 1;
    pg.pf_stride = q.d_model * static_cast<int64_t>(q.qt == 0 ? q.d_ff / 32 * 34 : q.d_ff / 256 * 144);
    e = q.qt == 0 ? launch_moe_stream<0, 2>(pg, dim3(gx, slots), smem, s)
                  : launch_moe_stream<1, 2>(pg, dim3(gx, slots), smem, s);
    if (e != cudaSuccess) return e;

    MoeParams pd{};
    if (!plan_moe(q.qt, 1, q.d_model, q.d_ff, cpe, maxb, &pd, &gx, &smem)) return cudaErrorInvalidConfiguration;
    pd.w[0] = pd.w[1] = static_cast<const uint8_t*>(q.wd);
    pd.x = w.h;
    pd.ldx = q.d_ff;
    pd.x_by_pair = 1;
    pd.top_k = q.top_k;
    pd.y = w.yp;
    pd.ldy = q.d_model;
    pd.r = w.r;
    pd.trace_id = tb + 2;
    e = q.qt == 0 ? launch_moe_stream<0, 1>(pd, dim3(gx, slots), smem, s)
                  : launch_moe_stream<1, 1>(pd, dim3(gx, slots), smem, s);
    if (e != cudaSuccess) return e;

    const int64_t total = q.t * q.d_model;
    return launch_kernel(moe_combine_kernel, dim3(static_cast<unsigned>(cdiv(total, 256))), dim3(256), 0, s, true,
                         static_cast<const float*>(w.yp), static_cast<const float*>(w.r.p), q.y,
                         static_cast<int>(q.t), q.top_k, q.d_model, tb + 3);
}

}  // namespace phb
