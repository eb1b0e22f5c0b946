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
// activations in registers for the whole GEMV, so per weight only the
// quantized bytes come from shared memory. A stage holds whole row segments:
// with useg units per row segment, a stage carries
// floor(176 / (nmat * useg)) * nmat segments (176 = half the consumer
// threads) and thread t works on segment t % segs at half unit t / segs, so a
// warp's threads share a few positions and fill their registers mostly by
// broadcasts. Segments are padded by 16 bytes in the stage, so that the
// threads' weight reads at one position spread over the shared-memory banks.
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

#include "gemv_plan.cuh"
#include "persist_common.cuh"
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

PHB_TRACE_READER(phb_trace_read_persistent)

namespace {

constexpr int kMaxLayers = 64;
constexpr int kStateWords = kCtrBase + 4 * kMaxLayers;

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
    uint32_t stage_stride;         // bytes per ring stage (row segments at padded places)
    uint32_t xs_off, part_off, res_off, bar_off;
};

template <int QT, int NS>
__global__ void __launch_bounds__(KCfg<QT, kCW>::threads, 1) decode_persistent_kernel(const __grid_constant__ PersistParams p) {
    using C = KCfg<QT, kCW, NS>;
    extern __shared__ __align__(1024) uint8_t smem[];
    float* xs = reinterpret_cast<float*>(smem + p.xs_off);
    float* part = reinterpret_cast<float*>(smem + p.part_off);
    float* res = reinterpret_cast<float*>(smem + p.res_off);
    float* rsum = res + kNC;  // NMAT * rows_here row sums
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.bar_off);
    uint64_t* empty = full + C::ns;
    float* xfac = reinterpret_cast<float*>(empty + C::ns);
    float* red = xfac + kAccStride;
    int* flag = reinterpret_cast<int*>(red + (2 * kMaxConsumerWarps + 3) * kAccStride);

    const int tid = threadIdx.x;
    const int nctas = gridDim.x;
    const int n_ops = 4 * p.n_layers;
    const StageCtx sctx{p.state, p.n_q, p.n_kv, p.head_dim};
    if (tid == 0) {
        for (int s = 0; s < C::ns; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kCW);
        }
        fence_barrier_init();
        *flag = 0;
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
                if (!produce_segs<KCfg<QT, kCW, NS>>(t, nmat, segs, seg_stride_bytes(t.useg, KCfg<QT, kCW, NS>::ub),
                                                     smem, p.stage_stride, full, empty, s, pol))
                    break;
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
                    ok = stage_vec<1>(sctx, lin_t, lin_p, tag_lin, kseg, xs, xfac, red, flag, nullptr, nullptr, 0,
                                      res, 0, op);
                    break;
                case 1:
                    ok = stage_vec<2>(sctx, p.qkv + rep * p.rs_qkv, nullptr, tag_prev, kseg, xs, xfac, red, flag,
                                      lin_t ? lin_t + row0 : nullptr, lin_p ? lin_p + row0 : nullptr, tag_lin, res,
                                      t.rows_here, op);
                    break;
                case 2:
                    ok = stage_vec<1>(sctx, p.x1 + rep * p.rs_dm, nullptr, tag_prev, kseg, xs, xfac, red, flag, nullptr, nullptr, 0,
                                      res, 0, op);
                    break;
                default:
                    ok = stage_vec<0>(sctx, p.act + rep * p.rs_ff, nullptr, tag_prev, kseg, xs, xfac, red, flag,
                                      p.x1 + rep * p.rs_dm + row0,
                                      nullptr, tag_me - 2, res, t.rows_here, op);
                    break;
            }
            alive = ok;
        }
        if (tid == 0) PHB_TRACE_EV(op, 2);
        // this thread's half-unit position: activations into registers
        float xr[kHalfK];
        {
            const int pos = xr_pos(segs, t.useg);
            const float* xp = xs + pos * (kXPadEvery + kXPad);
#pragma unroll
            for (int i = 0; i < kHalfK; i += 4) {
                const float4 v = *reinterpret_cast<const float4*>(xp + i);
                xr[i] = v.x;
                xr[i + 1] = v.y;
                xr[i + 2] = v.z;
                xr[i + 3] = v.w;
            }
        }
        const float xf = xfac[0];
        if (tid == 0) PHB_TRACE_EV(op, 9);
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
            ok = consume_xr<QT, 2, NS>(t, segs, smem, p.stage_stride, full, empty, s, xr, xf, part, rsum, alive, op, epi);
        else
            ok = consume_xr<QT, 1, NS>(t, segs, smem, p.stage_stride, full, empty, s, xr, xf, part, rsum, alive, op, epi);
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

// Copies the values (low words) of replica 0 of three tagged vectors.
__global__ void probe_pairs_kernel(const uint2* qkv, int n_qkv, const uint2* x1, int n_dm, const uint2* act, int n_ff,
                                   float* qkv_out, float* x1_out, float* act_out) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n_qkv) qkv_out[i] = __uint_as_float(qkv[i].x);
    if (i < n_dm) x1_out[i] = __uint_as_float(x1[i].x);
    if (i < n_ff) act_out[i] = __uint_as_float(act[i].x);
}

// Workspace of the persistent step: tagged intermediate vectors and the state words.
size_t decode_persistent_ws_bytes(int64_t d_model, int n_q, int n_kv, int hd, int64_t d_ff) {
    auto al = [](size_t v) { return (v + 255) & ~size_t{255}; };
    size_t b = al(kStateWords * 4);
    b += kRep * al(static_cast<size_t>(n_q + 2 * n_kv) * hd * 8);
    b += kRep * al(static_cast<size_t>(d_model) * 8) * 3;
    b += kRep * al(static_cast<size_t>(d_ff) * 8);
    return b;
}

cudaError_t decode_persistent_probe(const void* ws, int64_t d_model, int n_q, int n_kv, int hd, int64_t d_ff,
                                    float* qkv, float* x1, float* act, cudaStream_t s) {
    auto al = [](size_t v) { return (v + 255) & ~size_t{255}; };
    const int qkv_dim = (n_q + 2 * n_kv) * hd;
    const auto* b = static_cast<const uint8_t*>(ws);
    const size_t rs_qkv = al(static_cast<size_t>(qkv_dim) * 8), rs_dm = al(static_cast<size_t>(d_model) * 8);
    size_t off = al(kStateWords * 4);
    const auto* pq = reinterpret_cast<const uint2*>(b + off);
    off += kRep * rs_qkv;
    const auto* px1 = reinterpret_cast<const uint2*>(b + off);
    off += 3 * kRep * rs_dm;  // x1, then the two layer-output vectors
    const auto* pact = reinterpret_cast<const uint2*>(b + off);
    const int n = static_cast<int>(std::max<int64_t>({static_cast<int64_t>(qkv_dim), d_model, d_ff}));
    probe_pairs_kernel<<<(n + 255) / 256, 256, 0, s>>>(pq, qkv_dim, px1, static_cast<int>(d_model), pact,
                                                       static_cast<int>(d_ff), qkv, x1, act);
    return cudaGetLastError();
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
    // a stage holds the widest op's row segments at their padded places;
    // `part` the largest op's half-unit sums (nmat * rows * 2 useg floats)
    const int64_t op_n[4] = {p.qkv_dim, d_model, d_ff, d_model};
    const int64_t op_k[4] = {d_model, p.q_dim, d_model, d_ff};
    const int op_nmat[4] = {1, 1, 2, 1};
    size_t stage_stride = 0, part_floats = 0;
    for (int o = 0; o < 4; ++o) {
        const int useg = static_cast<int>(op_k[o] / kUnitWeights);
        const int segs = segs_per_stage(kStageUnits, useg, op_nmat[o]);
        stage_stride = std::max(stage_stride, static_cast<size_t>(segs) * seg_stride_bytes(useg, ub));
        const size_t rows = static_cast<size_t>((op_n[o] + grid - 1) / grid);
        part_floats = std::max(part_floats, static_cast<size_t>(op_nmat[o]) * rows * 2 * useg);
    }
    stage_stride = (stage_stride + 127) & ~size_t{127};
    p.stage_stride = static_cast<uint32_t>(stage_stride);
    int ns = 0;
    size_t smem = 0;
    for (int cand : {deep, shallow}) {
        size_t off = static_cast<size_t>(cand) * stage_stride;
        const size_t xs_off = off;
        off += static_cast<size_t>(xpad_len(static_cast<int>(kmax))) * sizeof(float);
        const size_t part_off = off;
        const size_t res_off = part_off + part_floats * sizeof(float);
        // residuals (kNC floats) then row sums (2 * max_rows floats)
        const size_t bar_off = (res_off + (kNC + 2 * static_cast<size_t>(max_rows)) * sizeof(float) + 15) & ~size_t{15};
        const size_t total = bar_off + 2 * cand * sizeof(uint64_t) + kTailFloats * sizeof(float);
        if (total > kSmemOptin) continue;
        ns = cand;
        smem = total;
        p.xs_off = static_cast<uint32_t>(xs_off);
        p.part_off = static_cast<uint32_t>(part_off);
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
