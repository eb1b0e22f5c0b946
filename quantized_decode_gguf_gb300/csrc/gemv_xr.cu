// Batch-1 streaming GEMV with register-resident activations.
//
// The streaming kernel of gemv_kernel.cuh reads one activation from shared
// memory per weight and stages the activation vector with a CTA-wide scale
// reduction. At batch 1 both show: the dot runs at about half the rate of a
// dot whose activations sit in registers, and staging costs two barriers.
// Here every stage holds whole row segments (a gate/up pair counting as
// two), so a consumer thread works on the same half-unit position of every
// stage: for rows of more than 16 half units, when a stage holds at least 8
// row segments, thread t takes segment t % segs at position t / segs (a
// warp's threads share few positions, so their register fills are mostly
// broadcasts; segments are padded in the stage as seg_stride_bytes says),
// otherwise segment t / (2 useg) at position t % (2 useg) (measured faster
// for short rows and for stages of few long rows). The CTA reads x once
// (coalesced, each element once) into shared memory; after one barrier every
// thread copies its 128 activations x[128 pos .. 128 pos + 127] into
// registers, scaled by a power of two 2^s chosen from their own largest
// magnitude, and undoes the scale per half-unit sum (xfac = 2^(85 - s)) before
// anything is added across threads. No CTA-wide reduction stands between the
// previous kernel's end and the first dot. (Every thread reading its slice
// from global memory itself funnels the whole grid onto the few L2 lines
// that hold x: measured several times slower.)
//
// Half-unit sums go to shared memory; after the last stage one thread per row
// adds them in row_sum's fixed order (deterministic) and runs the epilogue:
// store, or silu(gate) * up for the fused pair. Rows of more than 16 half
// units run one CTA of ten consumer warps per SM, shorter rows two CTAs of
// five (both measured faster that way). A producer warp streams the CTA's
// row slice through a ring of stages with bulk copies (before the
// programmatic-dependent-launch wait: weights never depend on the previous
// kernel) and optionally prefetches later kernels' weights into L2.
#include "gemv_plan.cuh"
#include "phb_internal.h"

namespace phb {

cudaError_t read_dev_err_gemv_xr(int* code) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_dev_err, sizeof(int));
    if (e != cudaSuccess) return e;
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_dev_err, &zero, sizeof(int));
    *code = v;
    return e;
}

PHB_TRACE_READER(phb_trace_read_gemv_xr)

namespace {

constexpr int kXrNS = 4;  // ring stages

struct XrParams {
    const uint8_t* w[2];
    int64_t row_bytes;
    int64_t n;
    int useg;          // units per row (K / 256)
    int rows_per_cta;
    int segs;          // segments per stage
    int segfast;       // 1: thread t on segment t % segs, position t / segs; 0: the reverse
    int ss;            // bytes between a stage's segments
    uint32_t stage_stride;
    const float* x;
    float* y;
    const uint8_t* pf[2];
    int64_t pf_bytes[2];
    uint32_t xs_off, part_off, bar_off;
    int trace_id;      // launch id for debug tracing builds (-1: none)
};

template <int QT, int NMAT, int CW>
__global__ void __launch_bounds__(32 * CW + 32, CW <= 6 ? 2 : 1) gemv_xr_kernel(const __grid_constant__ XrParams p) {
    using C = KCfg<QT, CW, kXrNS>;
    extern __shared__ __align__(1024) uint8_t smem[];
    float* xs = reinterpret_cast<float*>(smem + p.xs_off);  // x in the padded layout (xpad_idx)
    float* part = reinterpret_cast<float*>(smem + p.part_off);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.bar_off);
    uint64_t* empty = full + kXrNS;

    const int tid = threadIdx.x, lane = tid & 31;
    if (tid == 0) PHB_TRACE_EV(p.trace_id, 0);
    const int64_t row0 = static_cast<int64_t>(blockIdx.x) * p.rows_per_cta;
    Tile t;
    t.rows_here = static_cast<int>(min(static_cast<int64_t>(p.rows_per_cta), p.n - row0));
    t.useg = p.useg;
    t.row_bytes = p.row_bytes;
    t.contiguous = true;
    t.w[0] = p.w[0] + row0 * p.row_bytes;
    t.w[1] = p.w[NMAT - 1] + row0 * p.row_bytes;
    pdl_launch_dependents();
    if (t.rows_here <= 0) return;

    if (tid == 0) {
        for (int s = 0; s < kXrNS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], CW);
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (tid >= C::consumers) {
        if (tid == C::consumers) {
            int s = 0;
            produce_segs<C>(t, NMAT, p.segs, p.ss, smem, p.stage_stride, full, empty, s, policy_evict_first());
        } else if (tid == C::consumers + 1) {
            prefetch_share(p.pf[0], p.pf_bytes[0]);
            prefetch_share(p.pf[1], p.pf_bytes[1]);
        }
        return;
    }

    const int seg_half = 2 * t.useg;
    const int j = p.segfast ? tid % p.segs : tid / seg_half;
    const int pos = p.segfast ? tid / p.segs : tid % seg_half;
    const bool active = j < p.segs && pos < seg_half;
    pdl_wait();  // x may come from the previous kernel
    if (tid == 0) PHB_TRACE_EV(p.trace_id, 1);
    {
        const int n4 = t.useg * (kUnitWeights / 4);
        const float4* xg = reinterpret_cast<const float4*>(p.x);
        for (int i = tid; i < n4; i += C::consumers)
            *reinterpret_cast<float4*>(xs + xpad_idx(4 * i)) = __ldcg(xg + i);  // written by the previous kernel
    }
    consumer_sync<C::consumers>();
    float xr[128];
    float xf = 1.f;
    if (active) xf = load_xr_scaled(xs + pos * (kXPadEvery + kXPad), xr);
    if (tid == 0) PHB_TRACE_EV(p.trace_id, 2);

    const int nseg = NMAT * t.rows_here;
    int s = 0;
    bool ok = true;
    for (int seg0 = 0; seg0 < nseg; seg0 += p.segs, ++s) {
        const int slot = s % kXrNS;
        if (!mbar_wait_warp(&full[slot], (s / kXrNS) & 1, &g_dev_err)) {
            mbar_wait(&full[slot], (s / kXrNS) & 1, &g_dev_err);  // second bounded wait for the copy in flight
            ok = false;
            break;
        }
        const int seg = seg0 + j;
        if (active && seg < nseg) {
            const uint8_t* ub = smem + static_cast<size_t>(slot) * p.stage_stride + j * p.ss + (pos >> 1) * C::ub;
            float acc;
            if constexpr (QT == 0)
                acc = dot_q8_0_half_xr(ub + 136 * (pos & 1), xr, xf);
            else
                acc = dot_q4_k_half_xr(ub, pos & 1, xr, xf);
            part[seg * seg_half + pos] = acc;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
    }
    if (tid == 0) PHB_TRACE_EV(p.trace_id, 3);
    consumer_sync<C::consumers>();
    if (!ok) return;
    for (int r = tid; r < t.rows_here; r += C::consumers) {
        float a[NMAT];
#pragma unroll
        for (int m = 0; m < NMAT; ++m) {
            a[m] = row_sum(part + static_cast<size_t>(r * NMAT + m) * seg_half, seg_half);
        }
        p.y[row0 + r] = NMAT == 2 ? silu_mul(a[0], a[NMAT - 1]) : a[0];
    }
    if (tid == 0) PHB_TRACE_EV(p.trace_id, 4);
}

template <int QT, int NMAT, int CW>
cudaError_t launch_xr(const XrParams& p, dim3 grid, size_t smem, cudaStream_t s, bool pdl) {
    constexpr auto kern = gemv_xr_kernel<QT, NMAT, CW>;
    cudaError_t e = ensure_smem_attr<kern>();
    if (e != cudaSuccess) return e;
    return launch_kernel(kern, grid, dim3(32 * CW + 32), smem, s, pdl, p);
}

// Consumer warps per CTA of the register-resident kernel: five (two CTAs per
// SM), or ten (one CTA per SM) for rows of more than 16 half units.
constexpr int kXrCW = 5;
constexpr int kXrCWLong = 10;

}  // namespace

bool gemv_xr_fits(const GemvReq& q) {
    if (q.batch != 1 || q.xmode != kXPlain || q.k % kUnitWeights != 0) return false;
    if (!((q.nmat == 1 && q.epi == kEpiStore) || (q.nmat == 2 && q.epi == kEpiSwiGLU))) return false;
    const int seg_half = static_cast<int>(2 * (q.k / kUnitWeights));
    return q.nmat * seg_half <= 32 * kXrCW;  // a stage holds at least one row (pair) segment
}

cudaError_t gemv_xr_run(const GemvReq& q, cudaStream_t s) {
    if (!gemv_xr_fits(q)) return cudaErrorInvalidValue;
    const int useg = static_cast<int>(q.k / kUnitWeights);
    const int seg_half = 2 * useg;
    const int ub = q.qt == 0 ? Fmt<0>::unit_bytes : Fmt<1>::unit_bytes;
    // The launch for cw consumer warps per CTA (two CTAs per SM at 5, one at
    // 10); false if its shared memory does not fit.
    auto plan = [&](int cw, XrParams& p, size_t& off) {
        const int consumers = 32 * cw;
        p = XrParams{};
        p.w[0] = static_cast<const uint8_t*>(q.w0);
        p.w[1] = static_cast<const uint8_t*>(q.nmat == 2 ? q.w1 : q.w0);
        p.row_bytes = static_cast<int64_t>(useg) * ub;
        p.n = q.n;
        p.useg = useg;
        p.segs = (consumers / (q.nmat * seg_half)) * q.nmat;
        // measured: segments fastest pays when a stage holds 8 segments or more
        // (Q8_0 9728x2560 8.4 -> 7.8 us) and costs with fewer (Q8_0 2048x5632
        // 6.0 -> 6.5 us); at 16 half units or less positions fastest is cheaper
        p.segfast = (seg_half > 16 && p.segs >= 8) ? 1 : 0;
        p.ss = p.segfast ? seg_stride_bytes(useg, ub) : useg * ub;
        p.stage_stride = static_cast<uint32_t>((static_cast<size_t>(p.segs) * p.ss + 127) & ~size_t{127});
        const int ctas_per_sm = cw <= 6 ? 2 : 1;
        const int64_t ctas = std::min<int64_t>(q.n, static_cast<int64_t>(device_sm_count()) * ctas_per_sm);
        p.rows_per_cta = static_cast<int>(cdiv(q.n, ctas));
        p.x = q.x;
        p.y = q.y;
        p.trace_id = q.trace_id;
        for (int i = 0; i < 2; ++i) {
            p.pf[i] = static_cast<const uint8_t*>(q.pf[i]);
            p.pf_bytes[i] = q.pf_bytes[i];
        }
        off = kXrNS * static_cast<size_t>(p.stage_stride);
        p.xs_off = static_cast<uint32_t>(off);
        off += static_cast<size_t>(xpad_len(static_cast<int>(q.k))) * sizeof(float);
        p.part_off = static_cast<uint32_t>(off);
        off += static_cast<size_t>(q.nmat) * p.rows_per_cta * seg_half * sizeof(float);
        off = (off + 15) & ~size_t{15};
        p.bar_off = static_cast<uint32_t>(off);
        off += 2 * kXrNS * sizeof(uint64_t);
        return off <= kSmemOptin;
    };
    // measured: rows of more than 16 half units run faster as one CTA of ten
    // consumer warps per SM (Q4_K 9728x2560 6.62 -> 6.41 us, Q8_0 2048x5632
    // 6.15 -> 5.76 us), shorter ones as two CTAs of five (Q8_0 3072x2048
    // 4.20 against 4.35 us)
    XrParams p;
    size_t off = 0;
    int cw = kXrCW;
    if (seg_half > 16 && plan(kXrCWLong, p, off))
        cw = kXrCWLong;
    else if (!plan(kXrCW, p, off))
        return cudaErrorInvalidConfiguration;
    const dim3 grid(static_cast<unsigned>(cdiv(q.n, p.rows_per_cta)));
    if (cw == kXrCWLong) {
        if (q.qt == 0)
            return q.nmat == 2 ? launch_xr<0, 2, kXrCWLong>(p, grid, off, s, q.pdl)
                               : launch_xr<0, 1, kXrCWLong>(p, grid, off, s, q.pdl);
        return q.nmat == 2 ? launch_xr<1, 2, kXrCWLong>(p, grid, off, s, q.pdl)
                           : launch_xr<1, 1, kXrCWLong>(p, grid, off, s, q.pdl);
    }
    if (q.qt == 0)
        return q.nmat == 2 ? launch_xr<0, 2, kXrCW>(p, grid, off, s, q.pdl) : launch_xr<0, 1, kXrCW>(p, grid, off, s, q.pdl);
    return q.nmat == 2 ? launch_xr<1, 2, kXrCW>(p, grid, off, s, q.pdl) : launch_xr<1, 1, kXrCW>(p, grid, off, s, q.pdl);
}

}  // namespace phb
