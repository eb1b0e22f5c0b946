// Top-k routed mixture-of-experts FFN.
//
// 1. Routing (for one or two tokens in every CTA of the gate/up pass, CTA
//    (0, 0) publishing it; for more tokens in a one-CTA kernel):
//    per token the top_k largest router logits (ties to the lower expert
//    index) and their softmax; then a counting sort of the (token, slot)
//    pairs by expert, ascending pair id within an expert, giving the
//    active-expert list.
// 2. moe_rows_kernel<NMAT=2>: grid (row tiles of 64, expert slot). Each CTA
//    streams 64 rows of its expert's gate and up matrices (one 3-D TMA copy
//    per matrix and 256-weight unit) once per group of up to four tokens
//    routed to that expert, keeps every row's per-token sums in registers
//    and writes h[pair] = silu(gate.x) * (up.x).
// 3. moe_rows_kernel<NMAT=1>: the same over 128 rows of the down matrices,
//    x = h[pair], writing y_pair[pair].
// 4. The ordered combine y[t] = sum over slots (ascending) of p[t][slot] *
//    y_pair[t*top_k + slot]: for one or two tokens the last down-pass CTA of
//    each 128-row tile does it (a per-tile counter in the workspace, back to
//    zero after each call); for more tokens moe_combine_kernel.
// All orders are fixed, so repeated calls give identical bits.
//
// Tiered experts (the expert cache of the README's MoE decode): when only
// some experts fit in device memory, the caller keeps the rest in host
// memory the GPU can read and passes a location table. After routing, a
// fetch kernel copies every active expert that lives only in host memory
// (read by the GPU over the host link; no CPU compute) into a device staging
// slot and records per active slot which copy to read; the two passes then
// take each active expert's tiles from the cache or the staging area. The
// arithmetic is the same, so results equal the all-resident call's bit for bit.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cfloat>
#include <cmath>
#include <mutex>

#include "gemv_plan.cuh"
#include "moe_route.cuh"
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

PHB_TRACE_READER(phb_trace_read_moe)

namespace {

constexpr int kMaxTokens = 64;
// Tokens per pass over a staged weight tile. Four keeps the staged
// activations small enough for two CTAs per SM; an expert chosen by more
// tokens streams its tile once per group of four.
constexpr int kMoeGroup = 4;


struct RouteOut {
    int32_t* idx;        // [T][k]
    float* p;            // [T][k]
    int32_t* n_active;   // [1]
    int32_t* act_expert; // [slots]
    int32_t* act_off;    // [slots]
    int32_t* act_cnt;    // [slots]
    int32_t* pair_list;  // [T*k]
};


// Routing state in shared memory.
struct RouteSm {
    int32_t sidx[kMaxTokens * kMaxTopK];
    int32_t rank[kMaxTokens * kMaxTopK];
    int32_t cnt[kMaxExperts];
    int32_t off[kMaxExperts];
    int32_t act_expert[kMaxExperts];
    int32_t act_off[kMaxExperts];
    int32_t act_cnt[kMaxExperts];
    int32_t pair_list[kMaxTokens * kMaxTopK];
    int32_t n_active;
};


// Routing by 256 threads (the CTA's consumers; named barrier 1). Warps take
// tokens; per token, K rounds of a warp-wide arg-max (largest logit, then
// lowest expert index) over the logits held in registers give the top_k in
// slot order, and lane 0 takes their softmax. Then warp 0 sorts the
// (token, slot) pairs by expert with a stable counting sort (match groups
// per 32 pairs, a warp scan over the experts) and lists the active experts
// in ascending order. Everything lands in `sm`; with `go` non-null the
// lists, indices and weights are also written to global memory.
__device__ __forceinline__ void route_block(const float* __restrict__ logits, int T, int E, int K, RouteSm* sm,
                                            const RouteOut* go, int32_t* out_idx, float* out_p) {
    constexpr int NT = 256;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int e = tid; e < kMaxExperts; e += NT) sm->cnt[e] = 0;
    for (int t = warp; t < T; t += NT / 32) {
        int sel_e[kMaxTopK];
        float pr[kMaxTopK];
        route_token_warp(logits + static_cast<int64_t>(t) * E, E, K, lane, sel_e, pr);
        if (lane == 0) {
#pragma unroll
            for (int r = 0; r < kMaxTopK; ++r) {
                if (r >= K) break;
                const int q = t * K + r;
                sm->sidx[q] = sel_e[r];
                if (go) {
                    go->idx[q] = sel_e[r];
                    go->p[q] = pr[r];
                    if (out_idx) out_idx[q] = sel_e[r];
                    if (out_p) out_p[q] = pr[r];
                }
            }
        }
    }
    consumer_sync<NT>();
    const int pairs = T * K;
    if (warp == 0) {
        // stable rank of every pair within its expert, 32 pairs at a time
        for (int q0 = 0; q0 < pairs; q0 += 32) {
            const int q = q0 + lane;
            const bool valid = q < pairs;
            const int e = valid ? sm->sidx[q] : -1 - lane;  // invalid lanes match nobody
            const unsigned grp = __match_any_sync(0xFFFFFFFFu, e);
            const int base = valid ? sm->cnt[e] : 0;
            __syncwarp();
            if (valid) {
                sm->rank[q] = base + __popc(grp & ((1u << lane) - 1u));
                if ((__ffs(grp) - 1) == lane) sm->cnt[e] = base + __popc(grp);
            }
            __syncwarp();
        }
        // exclusive scan over experts (8 consecutive experts per lane) and the active list
        constexpr int kPer = kMaxExperts / 32;
        int c[kPer], lc = 0, la = 0;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int e = kPer * lane + i;
            c[i] = e < E ? sm->cnt[e] : 0;
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
                sm->off[e] = acc;
                if (c[i] > 0) {
                    sm->act_expert[a] = e;
                    sm->act_off[a] = acc;
                    sm->act_cnt[a] = c[i];
                    if (go) {
                        go->act_expert[a] = e;
                        go->act_off[a] = acc;
                        go->act_cnt[a] = c[i];
                    }
                    ++a;
                }
                acc += c[i];
            }
        }
        if (lane == 31) {
            sm->n_active = sa;
            if (go) *go->n_active = sa;
        }
    }
    consumer_sync<NT>();
    for (int q = tid; q < pairs; q += NT) {
        const int w = sm->off[sm->sidx[q]] + sm->rank[q];
        sm->pair_list[w] = q;
        if (go) go->pair_list[w] = q;
    }
    consumer_sync<NT>();
}

// Routing as its own one-CTA kernel (used when many tokens would make every
// gate/up CTA sort all pairs itself).
__global__ void __launch_bounds__(256) moe_route_kernel(const float* __restrict__ logits, int T, int E, int K,
                                                        RouteOut o, int32_t* out_idx, float* out_p) {
    __shared__ RouteSm sm;
    pdl_launch_dependents();
    pdl_wait();
    route_block(logits, T, E, K, &sm, &o, out_idx, out_p);
}

// Token counts up to which every gate/up CTA routes the tokens itself.
constexpr int kMoeInlineRouteTokens = 2;

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

// ---------------------------------------------------------------- row-resident grouped kernel
// The expert-grouped pass with the row-resident mapping of gemv_rows.cu: a
// CTA owns 128 rows of one active expert (for gate/up: 64 gate rows and the
// same 64 up rows), each stage is one 256-weight unit of those rows brought
// by one 3-D TMA copy per matrix ([expert][rows][row bytes]), thread t keeps
// row t % 128's sums for up to four tokens in registers over half unit
// t / 128, and the activations are shared-memory broadcasts.
constexpr int kMrRows = 128;
constexpr int kMrCW = 8;
constexpr int kMrNC = 32 * kMrCW;
constexpr int kMrThreads = kMrNC + 32;

template <int QT>
struct MrCfg {
    static constexpr int ub = Fmt<QT>::unit_bytes;
    static constexpr int stage_bytes = kMrRows * ub;
    static constexpr int ns = 3;
    static constexpr int ctas_per_sm = QT == 0 ? 1 : 2;  // Q4_K: two CTAs per SM overlap one's staging with the other's dots
};

struct MoeRowsParams {
    const float* x;        // gate/up: X [T][K]; down: h [pairs][K]
    int64_t ldx;
    int x_by_pair;         // 0: x row = pair / top_k; 1: x row = pair
    int top_k;
    float* y;              // [pairs][n]
    int64_t ldy;
    RouteOut r;
    int64_t n;             // rows per expert matrix
    int units_row;
    int row_tile;          // rows of each matrix per CTA: 64 (gate/up) or 128 (down)
    uint32_t xs_off, comb_off, bar_off, route_off;
    int trace_id;
    // gate/up pass: the routing is computed in the kernel from the logits
    const float* logits;
    int n_tokens, n_experts;
    int32_t* out_idx;
    float* out_p;
    int route_inline;  // gate/up pass: 1 = route in the kernel, 0 = read the routing kernel's lists
    // down pass: 1 = the last CTA of a row tile combines the slots into y_out
    int combine;
    // tiered experts: per active slot, 1 = read the staging copy (second maps),
    // and the expert index within the copy read (nullptr: the cache, index = expert)
    const int32_t* src_sel;
    const int32_t* src_z;
    int* tile_ctr;     // [row tiles], zero between calls
    float* y_out;      // Y [n_tokens][n]
};

__device__ __forceinline__ void tma_load_3d_hint(void* dst, const CUtensorMap* map, int x, int y, int z,
                                                 uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
        "%3, %4}], [%5], %6;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// One token group (nb <= MAXB tokens) over the CTA's rows: stage the tokens'
// activations, stream every unit, write silu(gate) * up (NMAT 2) or the row
// sums (NMAT 1) for each token.
template <int QT, int NMAT, int MAXB>
__device__ __forceinline__ bool moe_rows_group(const MoeRowsParams& p, const int32_t* plist, int64_t row0, int first,
                                               int nb, uint8_t* smem, uint64_t* full, uint64_t* empty, int& s) {
    using R = MrCfg<QT>;
    float* xs = reinterpret_cast<float*>(smem + p.xs_off);
    float* comb = reinterpret_cast<float*>(smem + p.comb_off);  // [2][MAXB][128]
    float* xfac = reinterpret_cast<float*>(full + 2 * R::ns);
    float* red = xfac + kAccStride;
    int* rowidx = reinterpret_cast<int*>(red + (2 * kMaxConsumerWarps + 3) * kAccStride);
    const int tid = threadIdx.x, lane = tid & 31;
    const int kseg = p.units_row * kUnitWeights;
    if (tid < nb) {
        const int pair = plist[first + tid];
        rowidx[tid] = p.x_by_pair ? pair : pair / p.top_k;
    }
    consumer_sync<kMrNC>();
    stage_x<kMrCW, MAXB, kXRowList>(p.x, p.ldx, 0, kseg, nb, xs, xfac, red, 1, 1, 0, rowidx);
    const int row = tid & (kMrRows - 1);
    const int h = tid >> 7;
    const int xstride = xpad_len(kseg);
    float acc[MAXB];
#pragma unroll
    for (int b = 0; b < MAXB; ++b) acc[b] = 0.f;
    for (int u = 0; u < p.units_row; ++u, ++s) {
        const int slot = s % R::ns;
        int good = 1;
        if (lane == 0) good = mbar_wait(&full[slot], (s / R::ns) & 1, &g_dev_err) ? 1 : 0;
        good = __shfl_sync(0xFFFFFFFFu, good, 0);
        __syncwarp();
        if (!good) return false;
        const uint8_t* ub = smem + slot * R::stage_bytes + row * R::ub;
        const int hu = 2 * u + h;
        if constexpr (QT == 0)
            dot_q8_0_half<MAXB>(ub + 136 * h, xs + hu * (kXPadEvery + kXPad), xstride, xfac, acc);
        else
            dot_q4_k_half<MAXB>(ub, h, xs + hu * (kXPadEvery + kXPad), xstride, xfac, acc);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
    }
    // halves of a row meet, then (NMAT 2) gate row r and up row r
    if (h == 1) {
#pragma unroll
        for (int b = 0; b < MAXB; ++b) comb[b * kMrRows + row] = acc[b];
    }
    consumer_sync<kMrNC>();
    if (h == 0) {
#pragma unroll
        for (int b = 0; b < MAXB; ++b) comb[(MAXB + b) * kMrRows + row] = acc[b] + comb[b * kMrRows + row];
    }
    consumer_sync<kMrNC>();
    const int* pairs = plist + first;
    const int outs = NMAT == 2 ? p.row_tile : kMrRows;
    for (int i = tid; i < outs * nb; i += kMrNC) {
        const int r = i % outs, b = i / outs;
        const int64_t n = row0 + r;
        if (n >= p.n) continue;
        const float a0 = comb[(MAXB + b) * kMrRows + r];
        const float out = NMAT == 2 ? silu_mul(a0, comb[(MAXB + b) * kMrRows + p.row_tile + r]) : a0;
        p.y[static_cast<int64_t>(pairs[b]) * p.ldy + n] = out;
    }
    consumer_sync<kMrNC>();  // the next group overwrites xs and comb
    return true;
}

template <int QT, int NMAT>
__global__ void __launch_bounds__(kMrThreads, MrCfg<QT>::ctas_per_sm)
    moe_rows_kernel(const __grid_constant__ CUtensorMap tm0, const __grid_constant__ CUtensorMap tm1,
                    const __grid_constant__ CUtensorMap tm0b, const __grid_constant__ CUtensorMap tm1b,
                    const __grid_constant__ MoeRowsParams p) {
    using R = MrCfg<QT>;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.bar_off);
    uint64_t* empty = full + R::ns;
    if (threadIdx.x == 0) PHB_TRACE_EV(p.trace_id, 0);
    pdl_launch_dependents();
    pdl_wait();  // x and the logits (gate/up), or the routing and h (down), come from earlier kernels
    if (threadIdx.x == 0) PHB_TRACE_EV(p.trace_id, 1);
    const int32_t* act_expert = p.r.act_expert;
    const int32_t* act_off = p.r.act_off;
    const int32_t* act_cnt = p.r.act_cnt;
    const int32_t* plist = p.r.pair_list;
    int n_active;
    if (NMAT == 2 && p.route_inline) {
        // every CTA routes the tokens itself; CTA (0, 0) publishes the result for the later passes
        RouteSm* rs = reinterpret_cast<RouteSm*>(smem + p.route_off);
        if (threadIdx.x < kMrNC)
            route_block(p.logits, p.n_tokens, p.n_experts, p.top_k, rs,
                        (blockIdx.x == 0 && blockIdx.y == 0) ? &p.r : nullptr, p.out_idx, p.out_p);
        __syncthreads();
        act_expert = rs->act_expert;
        act_off = rs->act_off;
        act_cnt = rs->act_cnt;
        plist = rs->pair_list;
        n_active = rs->n_active;
    } else {
        n_active = *p.r.n_active;
    }
    const int slot = blockIdx.y;
    if (slot >= n_active) return;
    const int e = act_expert[slot];
    const bool alt = p.src_sel != nullptr && p.src_sel[slot] != 0;
    const int z = p.src_z != nullptr ? p.src_z[slot] : e;  // expert index within the copy read
    const CUtensorMap* m0 = alt ? &tm0b : &tm0;
    const CUtensorMap* m1 = alt ? &tm1b : &tm1;
    const int first = act_off[slot];
    const int cnt = act_cnt[slot];
    const int64_t row0 = static_cast<int64_t>(blockIdx.x) * p.row_tile;
    if (row0 >= p.n) return;
    const int tid = threadIdx.x;
    if (tid == 0) {
        for (int s = 0; s < R::ns; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kMrCW);
        }
        fence_barrier_init();
    }
    __syncthreads();
    const int ngroups = (cnt + kMoeGroup - 1) / kMoeGroup;
    if (tid >= kMrNC) {
        if (tid == kMrNC) {
            const uint64_t pol = policy_evict_first();
            constexpr int kElems = QT == 0 ? R::ub / 2 : R::ub;
            int s = 0, issued = 0;
            bool ok = true;
            for (int gi = 0; gi < ngroups && ok; ++gi)
                for (int u = 0; u < p.units_row; ++u, ++s) {
                    const int sl = s % R::ns;
                    if (s >= R::ns && !mbar_wait(&empty[sl], ((s / R::ns) - 1) & 1, &g_dev_err)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[sl], static_cast<uint32_t>(R::stage_bytes));
                    uint8_t* dst = smem + sl * R::stage_bytes;
                    tma_load_3d_hint(dst, m0, u * kElems, static_cast<int>(row0), z, &full[sl], pol);
                    if (NMAT == 2)
                        tma_load_3d_hint(dst + p.row_tile * R::ub, m1, u * kElems, static_cast<int>(row0), z,
                                         &full[sl], pol);
                    ++issued;
                }
            for (int i = max(0, issued - R::ns); i < issued; ++i) mbar_wait(&full[i % R::ns], (i / R::ns) & 1, &g_dev_err);
        }
        return;
    }
    int s = 0;
    for (int gi = 0; gi < ngroups; ++gi) {
        const int nb = min(kMoeGroup, cnt - gi * kMoeGroup);
        const int fp = first + gi * kMoeGroup;
        bool ok;
        if (nb == 1)
            ok = moe_rows_group<QT, NMAT, 1>(p, plist, row0, fp, nb, smem, full, empty, s);
        else if (nb == 2)
            ok = moe_rows_group<QT, NMAT, 2>(p, plist, row0, fp, nb, smem, full, empty, s);
        else
            ok = moe_rows_group<QT, NMAT, 4>(p, plist, row0, fp, nb, smem, full, empty, s);
        if (!ok) return;
    }
    if constexpr (NMAT == 1) {
        if (p.combine) {
            // the last CTA of this row tile to publish its pairs sums the slots in ascending order
            int* flag = reinterpret_cast<int*>(smem + p.route_off);  // the routing area is unused here
            __threadfence();
            consumer_sync<kMrNC>();
            if (tid == 0) *flag = atomicAdd(p.tile_ctr + blockIdx.x, 1) == n_active - 1 ? 1 : 0;
            consumer_sync<kMrNC>();
            if (*flag) {
                __threadfence();
                for (int i = tid; i < p.n_tokens * kMrRows; i += kMrNC) {
                    const int t = i / kMrRows, r = i - t * kMrRows;
                    const int64_t n = row0 + r;
                    if (n >= p.n) continue;
                    float acc = 0.f;
                    for (int k = 0; k < p.top_k; ++k)
                        acc = fmaf(__ldcg(p.r.p + t * p.top_k + k),
                                   __ldcg(p.y + static_cast<int64_t>(t * p.top_k + k) * p.ldy + n), acc);
                    p.y_out[static_cast<int64_t>(t) * p.n + n] = acc;
                }
                if (tid == 0) p.tile_ctr[blockIdx.x] = 0;
            }
        }
    }
    if (tid == 0) PHB_TRACE_EV(p.trace_id, 3);
}

PFN_cuTensorMapEncodeTiled_v12000 moe_encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// [E][rows][row bytes] expert-major matrix as a 3-D tensor; one box = one unit of `box_rows` rows of one expert.
bool encode_expert_map(CUtensorMap* m, int qt, const void* w, int e, int64_t rows, int64_t k, int box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 encode = moe_encode_fn();
    if (encode == nullptr) return false;
    const int ub = qt == 0 ? Fmt<0>::unit_bytes : Fmt<1>::unit_bytes;
    const int64_t row_bytes = k / kUnitWeights * ub;
    const int esz = qt == 0 ? 2 : 1;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(row_bytes / esz), static_cast<cuuint64_t>(rows),
                                static_cast<cuuint64_t>(e)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(rows * row_bytes)};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(ub / esz), static_cast<cuuint32_t>(box_rows), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return encode(m, qt == 0 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(w),
                  dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Shared-memory layout of the row-resident pass for K and the token group size.
size_t moe_rows_layout(int qt, int64_t k, MoeRowsParams* p) {
    const int ns = qt == 0 ? MrCfg<0>::ns : MrCfg<1>::ns;
    const size_t stage = static_cast<size_t>(kMrRows) * (qt == 0 ? Fmt<0>::unit_bytes : Fmt<1>::unit_bytes);
    const int kseg = static_cast<int>(k);
    size_t off = ns * stage;
    p->xs_off = static_cast<uint32_t>(off);
    off += static_cast<size_t>(kMoeGroup) * xpad_len(kseg) * 4;
    p->comb_off = static_cast<uint32_t>(off);
    off += 2 * static_cast<size_t>(kMoeGroup) * kMrRows * 4;
    off = (off + 15) & ~size_t{15};
    p->route_off = static_cast<uint32_t>(off);
    off += sizeof(RouteSm);
    off = (off + 15) & ~size_t{15};
    p->bar_off = static_cast<uint32_t>(off);
    off += 2 * ns * sizeof(uint64_t) + kTailFloats * sizeof(float);
    return off;
}

template <int QT, int NMAT>
cudaError_t launch_moe_rows(const CUtensorMap& t0, const CUtensorMap& t1, const CUtensorMap& t0b,
                            const CUtensorMap& t1b, const MoeRowsParams& p, dim3 grid, size_t smem, cudaStream_t s) {
    constexpr auto kern = moe_rows_kernel<QT, NMAT>;
    cudaError_t e = ensure_smem_attr<kern>();
    if (e != cudaSuccess) return e;
    return launch_kernel(kern, grid, dim3(kMrThreads), smem, s, true, t0, t1, t0b, t1b, p);
}

constexpr int kFetchCtas = 96;  // CTAs per active slot of the fetch kernel

// Tiered experts: for every active slot whose expert lives only in host
// memory, copy its gate, up and down matrices into staging slot `slot`
// (grid: CTAs per slot x slots; each CTA a contiguous share, 16-byte
// accesses), and record which copy the passes read.
__global__ void __launch_bounds__(256) moe_fetch_kernel(const int32_t* __restrict__ n_active,
                                                        const int32_t* __restrict__ act_expert,
                                                        const int32_t* __restrict__ loc, int n_dev, int n_host,
                                                        const uint8_t* hg,
                                                        const uint8_t* hu, const uint8_t* hd, uint8_t* sg, uint8_t* su,
                                                        uint8_t* sd, int64_t bytes_gu, int64_t bytes_d,
                                                        int32_t* src_sel, int32_t* src_z) {
    pdl_launch_dependents();
    pdl_wait();  // the routing comes from the previous kernel
    const int slot = blockIdx.y;
    if (slot >= *n_active) return;
    const int v = loc[act_expert[slot]];
    const int64_t h = -1 - static_cast<int64_t>(v);
    const bool bad = v >= n_dev || (v < 0 && h >= n_host);  // neither copy exists: record it, read nothing
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        src_sel[slot] = v < 0 ? 1 : 0;
        src_z[slot] = v < 0 ? slot : v;
        if (bad) atomicExch(&g_dev_err, kDevErrBadIndex);
    }
    if (v >= 0 || bad) return;
    auto copy = [&](const uint8_t* src, uint8_t* dst, int64_t bytes) {
        const int64_t n16 = bytes / 16;
        const int64_t share = (n16 + gridDim.x - 1) / gridDim.x;
        const int64_t lo = blockIdx.x * share, hi = min(n16, lo + share);
        const uint4* s4 = reinterpret_cast<const uint4*>(src);
        uint4* d4 = reinterpret_cast<uint4*>(dst);
        constexpr int kInFlight = 8;  // 16-byte reads in flight per thread: the host link's latency is long
        int64_t i = lo + threadIdx.x;
        for (; i + (kInFlight - 1) * blockDim.x < hi; i += kInFlight * blockDim.x) {
            uint4 v[kInFlight];
#pragma unroll
            for (int u = 0; u < kInFlight; ++u) v[u] = s4[i + u * blockDim.x];
#pragma unroll
            for (int u = 0; u < kInFlight; ++u) d4[i + u * blockDim.x] = v[u];
        }
        for (; i < hi; i += blockDim.x) d4[i] = s4[i];
    };
    copy(hg + h * bytes_gu, sg + slot * bytes_gu, bytes_gu);
    copy(hu + h * bytes_gu, su + slot * bytes_gu, bytes_gu);
    copy(hd + h * bytes_d, sd + slot * bytes_d, bytes_d);
}

struct MoeWs {
    RouteOut r;
    float* h;
    float* yp;
    int* tile_ctr;  // down-pass row tiles: combine counters
    // one token: the one-token kernel's tagged h replicas and its call epoch
    uint2* tok_hx;
    unsigned* tok_epoch;
    // tiered experts only: staging copies [slots][rows][row bytes] and the per-slot source tables
    uint8_t* stage[3];
    int32_t* src_sel;
    int32_t* src_z;
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
    // the per-pair outputs and activations lead (a documented part of the ABI)
    w.yp = reinterpret_cast<float*>(take(pairs * q.d_model * 4));
    w.h = reinterpret_cast<float*>(take(pairs * q.d_ff * 4));
    w.r.idx = reinterpret_cast<int32_t*>(take(pairs * 4));
    w.r.p = reinterpret_cast<float*>(take(pairs * 4));
    w.r.n_active = reinterpret_cast<int32_t*>(take(16));
    w.r.act_expert = reinterpret_cast<int32_t*>(take(slots * 4));
    w.r.act_off = reinterpret_cast<int32_t*>(take(slots * 4));
    w.r.act_cnt = reinterpret_cast<int32_t*>(take(slots * 4));
    w.r.pair_list = reinterpret_cast<int32_t*>(take(pairs * 4));
    w.tile_ctr = reinterpret_cast<int*>(take(static_cast<size_t>((q.d_model + kMrRows - 1) / kMrRows) * 4));
    if (q.t == 1) {
        w.tok_epoch = reinterpret_cast<unsigned*>(take(16));
        w.tok_hx = reinterpret_cast<uint2*>(take(static_cast<size_t>(kTokReplicas) * q.top_k * q.d_ff * 8));
    }
    if (q.loc != nullptr) {
        const int ub = q.qt == 0 ? Fmt<0>::unit_bytes : Fmt<1>::unit_bytes;
        const size_t gu = static_cast<size_t>(q.d_ff) * (q.d_model / kUnitWeights) * ub;
        const size_t dn = static_cast<size_t>(q.d_model) * (q.d_ff / kUnitWeights) * ub;
        w.src_sel = reinterpret_cast<int32_t*>(take(slots * 4));
        w.src_z = reinterpret_cast<int32_t*>(take(slots * 4));
        w.stage[0] = take(slots * gu);
        w.stage[1] = take(slots * gu);
        w.stage[2] = take(slots * dn);
    }
    w.bytes = off;
    return w;
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
    cudaError_t e;
    const bool tiered = q.loc != nullptr;
    // one token: one cooperative kernel over all SMs (moe_token.cu) where the shape fits
    const bool token = q.t == 1 && moe_token_fits(q);
    // tiered experts route in their own kernel: the fetch kernel needs the list first
    const bool inline_route = q.t <= kMoeInlineRouteTokens && !tiered;
    if (!inline_route) {
        e = launch_kernel(moe_route_kernel, dim3(1), dim3(256), 0, s, true, q.logits, static_cast<int>(q.t), q.e,
                          q.top_k, w.r, q.out_idx, q.out_p);
        if (e != cudaSuccess) return e;
    }
    if (tiered) {
        const int ub = q.qt == 0 ? Fmt<0>::unit_bytes : Fmt<1>::unit_bytes;
        const int64_t gu = q.d_ff * (q.d_model / kUnitWeights) * ub;
        const int64_t dn = q.d_model * (q.d_ff / kUnitWeights) * ub;
        // enough CTAs per active expert to keep many host reads in flight
        e = launch_kernel(moe_fetch_kernel, dim3(kFetchCtas, static_cast<unsigned>(slots)), dim3(256), 0, s, true,
                          static_cast<const int32_t*>(w.r.n_active), static_cast<const int32_t*>(w.r.act_expert),
                          q.loc, q.n_dev_slots, q.n_host, static_cast<const uint8_t*>(q.hg),
                          static_cast<const uint8_t*>(q.hu), static_cast<const uint8_t*>(q.hd), w.stage[0],
                          w.stage[1], w.stage[2], gu, dn, w.src_sel, w.src_z);
        if (e != cudaSuccess) return e;
    }
    if (token) {
        MoeTokWs tw{};
        tw.h = w.h;
        tw.yp = w.yp;
        tw.idx = w.r.idx;
        tw.p = w.r.p;
        tw.src_sel = w.src_sel;
        tw.src_z = w.src_z;
        for (int i = 0; i < 3; ++i) tw.stage[i] = w.stage[i];
        tw.hx = w.tok_hx;
        tw.epoch = w.tok_epoch;
        tw.trace_id = tb + 1;
        return moe_token_run(q, tw, s);
    }
    // row-resident grouped passes (3-D TMA unit stages)
    {
        // experts in the arrays wg, wu, wd (a tiered call without a device cache maps the staging area there)
        const bool no_cache = tiered && q.n_dev_slots == 0;
        const int n_cache = no_cache ? slots : tiered ? q.n_dev_slots : q.e;
        const void* cg = no_cache ? w.stage[0] : q.wg;
        const void* cu = no_cache ? w.stage[1] : q.wu;
        const void* cd = no_cache ? w.stage[2] : q.wd;
        CUtensorMap tg, tu, td, sg, su, sd;
        if (!encode_expert_map(&tg, q.qt, cg, n_cache, q.d_ff, q.d_model, 64) ||
            !encode_expert_map(&tu, q.qt, cu, n_cache, q.d_ff, q.d_model, 64) ||
            !encode_expert_map(&td, q.qt, cd, n_cache, q.d_model, q.d_ff, kMrRows))
            return cudaErrorInvalidValue;
        sg = tg;
        su = tu;
        sd = td;
        if (tiered) {
            if (!encode_expert_map(&sg, q.qt, w.stage[0], slots, q.d_ff, q.d_model, 64) ||
                !encode_expert_map(&su, q.qt, w.stage[1], slots, q.d_ff, q.d_model, 64) ||
                !encode_expert_map(&sd, q.qt, w.stage[2], slots, q.d_model, q.d_ff, kMrRows))
                return cudaErrorInvalidValue;
        }
        MoeRowsParams pg{};
        const size_t smem_g = moe_rows_layout(q.qt, q.d_model, &pg);
        pg.x = q.x;
        pg.ldx = q.d_model;
        pg.x_by_pair = 0;
        pg.top_k = q.top_k;
        pg.y = w.h;
        pg.ldy = q.d_ff;
        pg.r = w.r;
        pg.n = q.d_ff;
        pg.units_row = static_cast<int>(q.d_model / kUnitWeights);
        pg.row_tile = 64;
        pg.trace_id = tb + 1;
        pg.logits = q.logits;
        pg.n_tokens = static_cast<int>(q.t);
        pg.n_experts = q.e;
        pg.out_idx = q.out_idx;
        pg.out_p = q.out_p;
        pg.route_inline = inline_route ? 1 : 0;
        pg.src_sel = tiered ? w.src_sel : nullptr;
        pg.src_z = tiered ? w.src_z : nullptr;
        if (smem_g > kSmemOptin) return cudaErrorInvalidConfiguration;
        const dim3 gg(static_cast<unsigned>(cdiv(q.d_ff, 64)), static_cast<unsigned>(slots));
        e = q.qt == 0 ? launch_moe_rows<0, 2>(tg, tu, sg, su, pg, gg, smem_g, s)
                      : launch_moe_rows<1, 2>(tg, tu, sg, su, pg, gg, smem_g, s);
        if (e != cudaSuccess) return e;
        MoeRowsParams pd{};
        const size_t smem_d = moe_rows_layout(q.qt, q.d_ff, &pd);
        pd.x = w.h;
        pd.ldx = q.d_ff;
        pd.x_by_pair = 1;
        pd.top_k = q.top_k;
        pd.y = w.yp;
        pd.ldy = q.d_model;
        pd.r = w.r;
        pd.n = q.d_model;
        pd.units_row = static_cast<int>(q.d_ff / kUnitWeights);
        pd.row_tile = kMrRows;
        pd.trace_id = tb + 2;
        // one or two tokens: the combine is a few loads per output, done by the down pass
        pd.combine = q.t <= kMoeInlineRouteTokens ? 1 : 0;
        pd.src_sel = tiered ? w.src_sel : nullptr;
        pd.src_z = tiered ? w.src_z : nullptr;
        pd.tile_ctr = w.tile_ctr;
        pd.y_out = q.y;
        pd.n_tokens = static_cast<int>(q.t);
        if (smem_d > kSmemOptin) return cudaErrorInvalidConfiguration;
        const dim3 gd(static_cast<unsigned>(cdiv(q.d_model, kMrRows)), static_cast<unsigned>(slots));
        e = q.qt == 0 ? launch_moe_rows<0, 1>(td, td, sd, sd, pd, gd, smem_d, s)
                      : launch_moe_rows<1, 1>(td, td, sd, sd, pd, gd, smem_d, s);
        if (e != cudaSuccess || pd.combine) return e;
        const int64_t total = q.t * q.d_model;
        return launch_kernel(moe_combine_kernel, dim3(static_cast<unsigned>(cdiv(total, 256))), dim3(256), 0, s, true,
                             static_cast<const float*>(w.yp), static_cast<const float*>(w.r.p), q.y,
                             static_cast<int>(q.t), q.top_k, q.d_model, tb + 3);
    }
}

}  // namespace phb
