// Routed MoE FFN of one token in one cooperative kernel (one CTA per SM).
//
// At one token the expert-grouped passes of moe.cu leave most SMs idle: eight
// active experts give a grid of row tiles x 8 CTAs, and every CTA stages the
// activations and waits on barriers between its token groups. Here the top_k
// active experts' matrices are spread evenly over all SMs, and each CTA's
// whole share is requested from HBM at once:
//
// 1. Every CTA routes the token itself (the producer warp: one expert per
//    round of a warp-wide arg-max, largest logit then lowest index; softmax
//    over the top_k); CTA 0 publishes the routing. The copies of a chunk are
//    issued as soon as the rounds that name its experts are done. A tiered
//    call reads the routing kernel's result instead and takes each active
//    expert from the device cache or its staging slot.
// 2. Gate/up: the K * d_ff (slot, row) pairs, slot-major, are cut into equal
//    ranges, one per CTA. The producer warp issues one bulk copy per matrix
//    and run of rows of one expert into shared memory, in chunks of `pp` row
//    pairs with one mbarrier each, then the CTA's down rows of all K
//    experts. Consumer thread t holds 128 activations of half unit t % (2U)
//    in registers (U units per row), scaled by a power of two, and dots them
//    with the same half unit of one gate or up row per chunk; half-unit sums
//    go to shared memory and one warp per row pair adds them in a fixed tree
//    order and stores h[slot][row] = silu(gate) * up.
// 3. Exchange: every h value is also stored as a {value, tag} pair in kRep
//    replicas (CTA i reads replica i % kRep, so the readers of a line are
//    spread over eight copies); the tag is the call's epoch + 1, the epoch a
//    workspace word advanced by CTA 0 at the end of each call, so nothing
//    needs clearing. A reader issues the strong loads of all its pairs at
//    once and re-reads only those whose tag is not yet current (bounded):
//    the data is its own ready signal, one round trip once it is there.
// 4. Down + combine: each consumer thread holds the 128 values of one
//    (slot, half unit) of h and dots them with that half unit of the CTA's
//    down rows of that slot's expert (already in shared memory). Row sums in
//    position order give y_pair[slot][n]; then y[n] = sum over slots
//    ascending of p_slot * y_pair[slot][n] (fma chain from zero), the same
//    combine as the grouped path.
//
// Every order is fixed, so repeated calls give identical bits, and a tiered
// call gives the same bits as the all-resident one.
#include "gemv_plan.cuh"
#include "moe_route.cuh"
#include "persist_common.cuh"
#include "phb_internal.h"

namespace phb {

cudaError_t read_dev_err_moe_token(int* code) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_dev_err, sizeof(int));
    if (e != cudaSuccess) return e;
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_dev_err, &zero, sizeof(int));
    *code = v;
    return e;
}

PHB_TRACE_READER(phb_trace_read_moe_token)

namespace {

constexpr int kTokCW = 11;               // consumer warps: 12 warps at the 168 registers of 128 activations
constexpr int kTokNC = 32 * kTokCW;
constexpr int kTokThreads = kTokNC + 32;
constexpr int kTokMaxChunks = 16;        // gate/up mbarriers per CTA
constexpr uint32_t kTokMaxTx = (1u << 20) - 1;  // bytes one mbarrier phase can count
static_assert(kRep == kTokReplicas, "the workspace holds one tagged copy of h per replica");
constexpr uint64_t kTokWaitNs = 2000000000ull;  // wall-clock bound of the exchange wait

struct TokParams {
    const uint8_t* wg;  // device cache: [n_dev][d_ff][rb_in], [n_dev][d_ff][rb_in], [n_dev][d_model][rb_ff]
    const uint8_t* wu;
    const uint8_t* wd;
    int n_dev;          // experts in the cache arrays (a larger index is not read)
    const uint8_t* sg;  // tiered: staging slots, same layouts
    const uint8_t* su;
    const uint8_t* sd;
    const int32_t* src_sel;  // tiered: per active slot (experts ascending), 1 = staging copy
    const int32_t* src_z;    //         and the expert's index within the copy read
    const int32_t* r_idx;    // tiered: routing written by the routing kernel (nullptr: route here)
    const float* r_p;
    const float* x;
    const float* logits;
    int E, K;
    int d_model, d_ff;
    int rb_in, rb_ff;   // bytes of a gate/up row and of a down row
    int rg, rd;         // gate/up row pairs and down rows per CTA
    int pp;             // gate/up row pairs per chunk
    float* h;           // [K][d_ff]
    float* yp;          // [K][d_model]
    float* y;           // [d_model]
    int32_t* ws_idx;    // CTA 0 publishes the routing (routed here only)
    float* ws_p;
    int32_t* out_idx;
    float* out_p;
    uint2* hx;          // [kRep][K * d_ff] {value, tag} copies of h
    unsigned* epoch;    // calls so far (zero in a fresh workspace)
    uint32_t wgu_off, wd_off, xs_off, part_off, bar_off;
    int trace_id;
};

// Four consecutive tagged pairs starting at pair e, read with strong
// (relaxed, gpu-scope) loads: a weak load of a line that another SM is
// rewriting may keep returning an old copy, a strong one sees the newest
// store in bounded time. True when all four carry `tag`.
__device__ __forceinline__ bool ld_tagged4_gpu(const uint2* src, int e, unsigned tag, float4& v) {
    unsigned long long a, b, c, d;
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(src + e) : "memory");
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(c), "=l"(d) : "l"(src + e + 2) : "memory");
    v = make_float4(__uint_as_float(static_cast<unsigned>(a)), __uint_as_float(static_cast<unsigned>(b)),
                    __uint_as_float(static_cast<unsigned>(c)), __uint_as_float(static_cast<unsigned>(d)));
    return static_cast<unsigned>(a >> 32) == tag && static_cast<unsigned>(b >> 32) == tag &&
           static_cast<unsigned>(c >> 32) == tag && static_cast<unsigned>(d >> 32) == tag;
}

constexpr int kTokXB = 8;  // groups of four pairs a consumer thread reads per pass of the exchange

template <int QT>
__device__ __forceinline__ float half_dot(const uint8_t* unit, int h, const float (&xr)[128], float xf) {
    if constexpr (QT == 0)
        return dot_q8_0_half_xr(unit + 136 * h, xr, xf);
    else
        return dot_q4_k_half_xr(unit, h, xr, xf);
}

template <int QT>
__global__ void __launch_bounds__(kTokThreads, 1) moe_token_kernel(const __grid_constant__ TokParams p) {
    constexpr int kUB = Fmt<QT>::unit_bytes;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.bar_off);  // [kTokMaxChunks] gate/up, then down
    uint64_t* full_d = full + kTokMaxChunks;
    float* sp = reinterpret_cast<float*>(full + kTokMaxChunks + 1);  // routing weights [kMaxTopK]
    float* sv = sp + kMaxTopK;                                        // selected logits [kMaxTopK]
    int* ssrc = reinterpret_cast<int*>(sv + kMaxTopK);                // per slot: 0 cache, 1 staging, -1 unreadable
    int* sz = ssrc + kMaxTopK;                                        // per slot: expert index within the copy

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = p.K * p.d_ff;
    const int g0 = blockIdx.x * p.rg;
    const int rows_g = max(0, min(p.rg, G - g0));
    const int n0 = blockIdx.x * p.rd;
    const int rows_d = max(0, min(p.rd, p.d_model - n0));
    const int nchunks = (rows_g + p.pp - 1) / p.pp;
    if (tid == 0) PHB_TRACE_EV(p.trace_id, 0);
    pdl_launch_dependents();
    if (tid == 0) {
        for (int c = 0; c <= kTokMaxChunks; ++c) mbar_init(&full[c], 1);
        fence_barrier_init();
    }
    __syncthreads();

    if (tid >= kTokNC) {
        // ---- producer warp: routing, then every copy of this CTA's share
        pdl_wait();  // the logits (or the routing and staged experts) come from earlier kernels
        const bool route_here = p.r_idx == nullptr;
        TopKWarp tk;
        int rounds = 0;
        if (route_here) {
            tk.load(p.logits, p.E, lane);
        } else if (lane == 0) {
            for (int r = 0; r < p.K; ++r) {
                const int e = __ldcg(p.r_idx + r);
                int a = 0;  // active slot of e: the active list is in ascending expert order
                for (int r2 = 0; r2 < p.K; ++r2) a += __ldcg(p.r_idx + r2) < e;
                const int sel = __ldcg(p.src_sel + a), z = __ldcg(p.src_z + a);
                sp[r] = __ldcg(p.r_p + r);
                ssrc[r] = (sel == 0 && (z < 0 || z >= p.n_dev)) ? -1 : sel;  // an unreadable slot copies nothing
                sz[r] = z;
            }
        }
        // routing rounds up to slot `slot` (warp-collective; lane 0 records the experts)
        auto route_to = [&](int slot) {
            if (!route_here) return;
            for (; rounds <= slot; ++rounds) {
                float v;
                const int e = tk.next(p.E, lane, &v);
                if (lane == 0) {
                    sv[rounds] = v;
                    ssrc[rounds] = 0;
                    sz[rounds] = e;
                }
            }
        };
        const uint64_t pol = policy_evict_first();
        const int64_t gu_bytes = static_cast<int64_t>(p.d_ff) * p.rb_in;
        const int64_t dn_bytes = static_cast<int64_t>(p.d_model) * p.rb_ff;
        auto base = [&](int slot, const uint8_t* cache, const uint8_t* stage, int64_t mbytes) {
            return (ssrc[slot] == 1 ? stage : cache) + sz[slot] * mbytes;
        };
        for (int c = 0; c < nchunks; ++c) {
            const int q0 = c * p.pp, q1 = min(rows_g, q0 + p.pp);
            route_to((g0 + q1 - 1) / p.d_ff);
            if (lane == 0) {
                uint32_t tx = 0;
                for (int q = q0; q < q1;) {
                    const int g = g0 + q, slot = g / p.d_ff, row = g - slot * p.d_ff;
                    const int n = min(q1 - q, p.d_ff - row);
                    if (ssrc[slot] >= 0) tx += 2u * n * p.rb_in;
                    q += n;
                }
                mbar_arrive_expect_tx(&full[c], tx);
                uint8_t* dst = smem + p.wgu_off + static_cast<size_t>(c) * p.pp * 2 * p.rb_in;
                for (int q = q0; q < q1;) {
                    const int g = g0 + q, slot = g / p.d_ff, row = g - slot * p.d_ff;
                    const int n = min(q1 - q, p.d_ff - row);
                    if (ssrc[slot] >= 0) {
                        const uint32_t bytes = static_cast<uint32_t>(n) * p.rb_in;
                        const int64_t off = static_cast<int64_t>(row) * p.rb_in;
                        bulk_g2s_hint(dst + static_cast<size_t>(q - q0) * p.rb_in,
                                      base(slot, p.wg, p.sg, gu_bytes) + off, bytes, &full[c], pol);
                        bulk_g2s_hint(dst + static_cast<size_t>(p.pp + q - q0) * p.rb_in,
                                      base(slot, p.wu, p.su, gu_bytes) + off, bytes, &full[c], pol);
                    }
                    q += n;
                }
            }
            __syncwarp();
        }
        route_to(p.K - 1);
        if (lane == 0) {
            if (route_here) {
                topk_softmax(sv, p.K, sp);
                if (blockIdx.x == 0)
                    for (int r = 0; r < p.K; ++r) {
                        p.ws_idx[r] = sz[r];
                        p.ws_p[r] = sp[r];
                        if (p.out_idx) p.out_idx[r] = sz[r];
                        if (p.out_p) p.out_p[r] = sp[r];
                    }
            }
            uint32_t txd = 0;
            for (int r = 0; r < p.K; ++r)
                if (ssrc[r] >= 0) txd += static_cast<uint32_t>(rows_d) * p.rb_ff;
            mbar_arrive_expect_tx(full_d, txd);  // also publishes sp to the consumers
            if (rows_d > 0)
                for (int r = 0; r < p.K; ++r)
                    if (ssrc[r] >= 0)
                        bulk_g2s_hint(smem + p.wd_off + static_cast<size_t>(r) * p.rd * p.rb_ff,
                                      base(r, p.wd, p.sd, dn_bytes) + static_cast<int64_t>(n0) * p.rb_ff,
                                      static_cast<uint32_t>(rows_d) * p.rb_ff, full_d, pol);
            // stay until every copy into this CTA's shared memory has landed (bounded)
            for (int c = 0; c < nchunks; ++c) mbar_wait(&full[c], 0, &g_dev_err);
            mbar_wait(full_d, 0, &g_dev_err);
        }
        return;
    }

    // ---- consumers: gate/up
    pdl_wait();  // x and the epoch come from earlier kernels
    const unsigned tag = __ldcg(p.epoch) + 1u;
    float* xs = reinterpret_cast<float*>(smem + p.xs_off);
    {
        const float4* xg = reinterpret_cast<const float4*>(p.x);
        for (int i = tid; i < p.d_model / 4; i += kTokNC)
            *reinterpret_cast<float4*>(xs + xpad_idx(4 * i)) = __ldcg(xg + i);
    }
    consumer_sync<kTokNC>();
    const int sh_in = 2 * (p.d_model / kUnitWeights);  // half units per gate/up row
    const int jp = tid / (2 * sh_in), rem = tid - jp * 2 * sh_in;
    const int mat = rem / sh_in, pos = rem - mat * sh_in;
    const bool act = jp < p.pp;
    float* part = reinterpret_cast<float*>(smem + p.part_off);
    auto publish = [&](int q, float hv, int r0, int nl) {  // lanes r0, r0 + nl, ... store the replicas
        for (int rep = r0; rep < kRep; rep += nl) st_pair(p.hx + static_cast<int64_t>(rep) * G + g0 + q, hv, tag);
        if (r0 == 0) p.h[g0 + q] = hv;
    };
    {
        float xr[128];  // this phase's activations (a second array serves the down phase)
        float xf = 1.f;
        if (act) xf = load_xr_scaled(xs + pos * (kXPadEvery + kXPad), xr);
        for (int c = 0; c < nchunks; ++c) {
            if (!mbar_wait_warp(&full[c], 0, &g_dev_err)) break;
            const int q = c * p.pp + jp;
            if (act && q < rows_g) {
                const uint8_t* unit = smem + p.wgu_off + (static_cast<size_t>(c) * p.pp * 2 + mat * p.pp + jp) * p.rb_in +
                                      (pos >> 1) * kUB;
                part[(q * 2 + mat) * sh_in + pos] = half_dot<QT>(unit, pos & 1, xr, xf);
            }
        }
    }
    consumer_sync<kTokNC>();  // every dot is done: the gate/up weights' shared memory is free
    {
        // eight lanes per row pair, four row pairs per warp: lanes 0-3 of a
        // group add the gate row's half-unit sums, lanes 4-7 the up row's
        // (strided, then a fixed xor tree); lane k of the group stores replica k
        const int grp = lane >> 3, gl = lane & 7;
        for (int q0 = 4 * warp; q0 < rows_g; q0 += 4 * kTokCW) {
            const int q = q0 + grp;
            float v = 0.f;
            if (q < rows_g) {
                const float* pr = part + (q * 2 + (gl >> 2)) * sh_in;
                for (int i = gl & 3; i < sh_in; i += 4) v += pr[i];
            }
            v += __shfl_xor_sync(0xFFFFFFFFu, v, 2);
            v += __shfl_xor_sync(0xFFFFFFFFu, v, 1);
            const float gate = __shfl_sync(0xFFFFFFFFu, v, lane & ~7), up = __shfl_sync(0xFFFFFFFFu, v, (lane & ~7) | 4);
            if (q < rows_g) publish(q, silu_mul(gate, up), gl, 8);
        }
    }
    if (tid == 0) PHB_TRACE_EV(p.trace_id, 2);

    // ---- exchange: all of h from this CTA's replica, tags checked
    float* hs = reinterpret_cast<float*>(smem + p.wgu_off);  // the gate/up weights are consumed
    {
        const uint2* src = p.hx + static_cast<int64_t>(blockIdx.x % kRep) * G;
        const int n4 = G / 4;
        uint64_t t0 = 0;
        bool late = false;
        for (int b0 = 0; b0 < n4; b0 += kTokNC * kTokXB) {
            uint32_t pending = 0;  // bit u: group b0 + tid + u * kTokNC still to read
#pragma unroll
            for (int u = 0; u < kTokXB; ++u)
                if (b0 + tid + u * kTokNC < n4) pending |= 1u << u;
            while (pending != 0) {
                float4 v[kTokXB];
                bool ok[kTokXB];
#pragma unroll
                for (int u = 0; u < kTokXB; ++u)  // every load of the pass is in flight before the first check
                    ok[u] = ((pending >> u) & 1u) && ld_tagged4_gpu(src, 4 * (b0 + tid + u * kTokNC), tag, v[u]);
#pragma unroll
                for (int u = 0; u < kTokXB; ++u)
                    if (ok[u]) {
                        *reinterpret_cast<float4*>(hs + xpad_idx(4 * (b0 + tid + u * kTokNC))) = v[u];
                        pending &= ~(1u << u);
                    }
                if (pending == 0) break;
                const uint64_t t = global_timer_ns();
                if (t0 == 0) t0 = t;
                if (late || t - t0 > kTokWaitNs) {  // give up: the error word says the result is not valid
                    if (!late) atomicOr(&g_dev_err, kDevErrTimeout);
                    late = true;
                    break;
                }
                __nanosleep(64);
            }
        }
    }
    consumer_sync<kTokNC>();
    if (tid == 0) PHB_TRACE_EV(p.trace_id, 3);

    // ---- down + combine
    const int sh_ff = 2 * (p.d_ff / kUnitWeights);
    // position (slot r, half unit hh) = tid / rpass, row group jr = tid % rpass:
    // the rpass threads that hold the same activations sit side by side, so
    // a warp's register fill reads few distinct addresses (broadcasts)
    const int p2 = p.K * sh_ff;  // (slot, half unit) positions of a down row
    const int rpass = kTokNC / p2;
    const int pos2 = tid / rpass, jr = tid - pos2 * rpass;
    const int r = pos2 / sh_ff, hh = pos2 - r * sh_ff;
    const bool act2 = pos2 < p2;
    // the activations into registers first: they do not wait for the down weights
    float xr[128];
    float xf = 1.f;
    if (act2) xf = load_xr_scaled(hs + (r * sh_ff + hh) * (kXPadEvery + kXPad), xr);
    const bool okd = mbar_wait_warp(full_d, 0, &g_dev_err);
    if (okd && act2) {
        for (int nl = jr; nl < rows_d; nl += rpass) {
            const uint8_t* unit = smem + p.wd_off + (static_cast<size_t>(r) * p.rd + nl) * p.rb_ff + (hh >> 1) * kUB;
            part[(nl * p.K + r) * sh_ff + hh] = half_dot<QT>(unit, hh & 1, xr, xf);
        }
    }
    consumer_sync<kTokNC>();
    // one warp per output row: lane r adds slot r's half-unit sums in order
    // (y_pair), then the slots are combined in ascending order
    for (int nl = warp; nl < rows_d; nl += kTokCW) {
        float v = 0.f;
        if (lane < p.K) {
            const float* pr = part + (nl * p.K + lane) * sh_ff;
            for (int j = 0; j < sh_ff; ++j) v += pr[j];
            p.yp[static_cast<int64_t>(lane) * p.d_model + n0 + nl] = v;
        }
        float acc = 0.f;
        for (int rr = 0; rr < p.K; ++rr) acc = fmaf(sp[rr], __shfl_sync(0xFFFFFFFFu, v, rr), acc);
        if (lane == 0) p.y[n0 + nl] = acc;
    }
    // CTA 0 has read every CTA's h, so every CTA has read the epoch: advance it
    if (blockIdx.x == 0 && tid == 0) *p.epoch = tag;
    if (tid == 0) PHB_TRACE_EV(p.trace_id, 4);
}

// Shared-memory layout and work split; false when the shape does not fit.
bool tok_plan(const MoeReq& q, TokParams* p, size_t* smem, int* grid) {
    if (q.t != 1 || q.top_k > kMaxTopK || q.d_model % kUnitWeights != 0 || q.d_ff % kUnitWeights != 0) return false;
    if (q.d_model > (1 << 20) || q.d_ff > (1 << 20)) return false;
    const int ub = q.qt == 0 ? Fmt<0>::unit_bytes : Fmt<1>::unit_bytes;
    const int sh_in = static_cast<int>(2 * (q.d_model / kUnitWeights));
    const int sh_ff = static_cast<int>(2 * (q.d_ff / kUnitWeights));
    const int pp = kTokNC / (2 * sh_in);
    if (pp < 1 || q.top_k * sh_ff > kTokNC) return false;
    const int sms = device_sm_count();
    const int64_t G = q.top_k * q.d_ff;
    const int rg = static_cast<int>(cdiv(G, sms));
    const int rd = static_cast<int>(cdiv(q.d_model, sms));
    const int nchunks = static_cast<int>(cdiv(rg, pp));
    if (nchunks > kTokMaxChunks) return false;
    const int64_t rb_in = q.d_model / kUnitWeights * ub, rb_ff = q.d_ff / kUnitWeights * ub;
    if (2 * pp * rb_in > kTokMaxTx || static_cast<int64_t>(q.top_k) * rd * rb_ff > kTokMaxTx) return false;
    auto al = [](size_t v) { return (v + 127) & ~size_t{127}; };
    size_t off = 0;
    p->wgu_off = 0;
    off += al(std::max<size_t>(static_cast<size_t>(nchunks) * pp * 2 * rb_in,
                               static_cast<size_t>(xpad_len(static_cast<int>(G))) * sizeof(float)));
    p->wd_off = static_cast<uint32_t>(off);
    off += al(static_cast<size_t>(q.top_k) * rd * rb_ff);
    p->xs_off = static_cast<uint32_t>(off);
    off += al(static_cast<size_t>(xpad_len(static_cast<int>(q.d_model))) * sizeof(float));
    p->part_off = static_cast<uint32_t>(off);
    off += al(std::max<size_t>(static_cast<size_t>(rg) * 2 * sh_in, static_cast<size_t>(rd) * q.top_k * (sh_ff + 1)) *
              sizeof(float));
    p->bar_off = static_cast<uint32_t>(off);
    off += (kTokMaxChunks + 1) * sizeof(uint64_t) + 4 * kMaxTopK * sizeof(int);
    if (off > kSmemOptin) return false;
    p->E = q.e;
    p->K = q.top_k;
    p->d_model = static_cast<int>(q.d_model);
    p->d_ff = static_cast<int>(q.d_ff);
    p->rb_in = static_cast<int>(rb_in);
    p->rb_ff = static_cast<int>(rb_ff);
    p->rg = rg;
    p->rd = rd;
    p->pp = pp;
    *smem = off;
    *grid = sms;
    return true;
}

}  // namespace

bool moe_token_fits(const MoeReq& q) {
    TokParams p{};
    size_t smem = 0;
    int grid = 0;
    return tok_plan(q, &p, &smem, &grid);
}

cudaError_t moe_token_run(const MoeReq& q, const MoeTokWs& w, cudaStream_t s) {
    TokParams p{};
    size_t smem = 0;
    int grid = 0;
    if (!tok_plan(q, &p, &smem, &grid)) return cudaErrorInvalidValue;
    const bool tiered = q.loc != nullptr;
    const bool no_cache = tiered && q.n_dev_slots == 0;
    p.wg = static_cast<const uint8_t*>(no_cache ? w.stage[0] : q.wg);
    p.wu = static_cast<const uint8_t*>(no_cache ? w.stage[1] : q.wu);
    p.wd = static_cast<const uint8_t*>(no_cache ? w.stage[2] : q.wd);
    p.n_dev = no_cache ? 0 : tiered ? q.n_dev_slots : q.e;
    if (tiered) {
        p.sg = w.stage[0];
        p.su = w.stage[1];
        p.sd = w.stage[2];
        p.src_sel = w.src_sel;
        p.src_z = w.src_z;
        p.r_idx = w.idx;
        p.r_p = w.p;
    }
    p.x = q.x;
    p.logits = q.logits;
    p.h = w.h;
    p.yp = w.yp;
    p.y = q.y;
    p.ws_idx = w.idx;
    p.ws_p = w.p;
    p.out_idx = q.out_idx;
    p.out_p = q.out_p;
    p.hx = w.hx;
    p.epoch = w.epoch;
    p.trace_id = w.trace_id;
    constexpr auto k0 = moe_token_kernel<0>;
    constexpr auto k1 = moe_token_kernel<1>;
    cudaError_t e = q.qt == 0 ? ensure_smem_attr<k0>() : ensure_smem_attr<k1>();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kTokThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    // every CTA waits for every other CTA's h: the cooperative launch guarantees they are resident together
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return q.qt == 0 ? cudaLaunchKernelEx(&cfg, k0, p) : cudaLaunchKernelEx(&cfg, k1, p);
}

}  // namespace phb
