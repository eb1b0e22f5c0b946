// Host-side planning of streaming GEMV launches: K split, rows per CTA,
// grid and the dynamic shared-memory layout.
#pragma once

#include <algorithm>

#include "gemv_kernel.cuh"
#include "phb_internal.h"

namespace phb {

inline int maxb_for(int batch) { return batch <= 1 ? 1 : batch <= 2 ? 2 : batch <= 4 ? 4 : 8; }

constexpr size_t kXSmemBudget = 80 * 1024;  // activations staged per CTA before K is split

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Number of K splits for a request (1 unless the staged activations would
// not fit the per-CTA budget).
inline int plan_ksplit(const GemvReq& q) {
    const int units_row = static_cast<int>(q.k / kUnitWeights);
    if (q.nmat != 1 || q.xmode != kXPlain || q.epi != kEpiStore) return 1;
    const size_t xbytes = static_cast<size_t>(q.batch) * q.k * sizeof(float);
    int ks = static_cast<int>(cdiv(static_cast<int64_t>(xbytes), kXSmemBudget));
    ks = std::max(1, std::min(ks, units_row));
    const int seg = static_cast<int>(cdiv(units_row, ks));
    return static_cast<int>(cdiv(units_row, seg));
}

// Consumer warps per CTA. Batch 1 and 2: eight, a CTA takes about half an
// SM, so the next kernel in a programmatic-dependent chain can be resident
// and stream its weights while this one finishes. Batch 3..8 needs more
// registers per thread (128 to 168) and fills one SM with as many warps as
// the register file then holds: 12 + 1 at <= 128, 11 + 1 at <= 168.
constexpr int cw_for(int maxb) { return maxb <= 2 ? 8 : maxb <= 4 ? 12 : 11; }

// Dynamic shared memory of a streaming-GEMV CTA:
//   stages | xs [maxb][xpad_len(kseg)] |
//   part (row-sum mode dependent) | row_acc [nmat*rows][kAccStride] (fold) |
//   mbarriers | xfac, reduction scratch, row list
struct SmemLayout {
    uint32_t xs, part, acc, bar;
    size_t total;
    int sum_mode;
};

constexpr size_t kTilePartBudget = 48 * 1024;

// CTAs of one GEMV per SM. Two half-SM CTAs measured fastest for the chained
// decode GEMVs (a 24-layer Q8_0 step: 550 us with 2, 775 us with 1).
constexpr int kCtasPerSm = 2;

inline SmemLayout stream_smem_layout(int qt, int cw, int nmat, int maxb, int rows_per_cta, int units_seg,
                                     int ring_stages = 0) {
    const int ub = qt == 0 ? Fmt<0>::unit_bytes : Fmt<1>::unit_bytes;
    const int consumers = 32 * cw;
    const int stage_units = consumers / 2;
    const int ns = ring_stages > 0 ? ring_stages : (qt == 0 ? KCfg<0, 8>::ns : KCfg<1, 8>::ns);
    SmemLayout l{};
    size_t off = static_cast<size_t>(ns) * stage_units * ub;
    const size_t kseg = static_cast<size_t>(units_seg) * kUnitWeights;
    l.xs = static_cast<uint32_t>(off);
    off += static_cast<size_t>(maxb) * xpad_len(static_cast<int>(kseg)) * sizeof(float);
    l.part = static_cast<uint32_t>(off);
    const size_t tile_part = 2 * static_cast<size_t>(nmat) * rows_per_cta * units_seg * maxb * sizeof(float);
    if (warp_rows(units_seg, nmat)) {
        l.sum_mode = kSumWarp;
    } else if (tile_part <= kTilePartBudget) {
        l.sum_mode = kSumTile;
        off += tile_part;
    } else {
        l.sum_mode = kSumFold;
        off += static_cast<size_t>(maxb) * consumers * sizeof(float);
    }
    l.acc = static_cast<uint32_t>(off);
    if (l.sum_mode == kSumFold) off += static_cast<size_t>(nmat) * rows_per_cta * kAccStride * sizeof(float);
    off = (off + 15) & ~static_cast<size_t>(15);
    l.bar = static_cast<uint32_t>(off);
    off += 2 * ns * sizeof(uint64_t);
    off += kTailFloats * sizeof(float);  // xfac, reduction scratch, row list
    l.total = off;
    return l;
}

// Fill a launch plan (one CTA per SM per K split). Returns false if no
// layout fits shared memory.
inline bool plan_stream(const GemvReq& q, GemvPlan* pl, int ctas_per_sm = kCtasPerSm) {
    const int units_row = static_cast<int>(q.k / kUnitWeights);
    const int ksplit0 = plan_ksplit(q);
    const int units_seg = static_cast<int>(cdiv(units_row, ksplit0));
    const int ksplit = static_cast<int>(cdiv(units_row, units_seg));
    const int maxb = maxb_for(q.batch);
    const int cw = cw_for(maxb);
    const int sms = device_sm_count();
    const int64_t target = std::max<int64_t>(1, cdiv(static_cast<int64_t>(sms) * ctas_per_sm, ksplit));
    int64_t nrow_ctas = std::min<int64_t>(q.n, target);
    int rows_per_cta = static_cast<int>(cdiv(q.n, nrow_ctas));
    SmemLayout lay{};
    for (;;) {
        lay = stream_smem_layout(q.qt, cw, q.nmat, maxb, rows_per_cta, units_seg);
        if (lay.total <= kSmemOptin) break;
        if (rows_per_cta == 1) return false;
        rows_per_cta = (rows_per_cta + 1) / 2;
    }
    nrow_ctas = cdiv(q.n, rows_per_cta);
    GemvParams& p = pl->p;
    p = GemvParams{};
    p.w[0] = static_cast<const uint8_t*>(q.w0);
    p.w[1] = static_cast<const uint8_t*>(q.nmat == 2 ? q.w1 : q.w0);
    p.row_bytes = static_cast<int64_t>(units_row) * (q.qt == 0 ? Fmt<0>::unit_bytes : Fmt<1>::unit_bytes);
    p.n = q.n;
    p.units_row = units_row;
    p.units_seg = units_seg;
    p.rows_per_cta = rows_per_cta;
    p.batch = q.batch;
    p.sum_mode = lay.sum_mode;
    p.x = q.x;
    p.ldx = q.ldx;
    p.y = q.y;
    p.ldy = q.ldy;
    p.r = q.r;
    p.ldr = q.ldr;
    p.part = q.ws;
    p.gather_group = q.gather_group;
    p.gather_hd = q.gather_hd;
    p.gather_v_off = q.gather_v_off;
    for (int i = 0; i < 2; ++i) {
        p.pf[i] = static_cast<const uint8_t*>(q.pf[i]);
        p.pf_bytes[i] = q.pf_bytes[i];
    }
    p.xs_off = lay.xs;
    p.part_off = lay.part;
    p.acc_off = lay.acc;
    p.bar_off = lay.bar;
    p.trace_id = q.trace_id;
    pl->grid = dim3(static_cast<unsigned>(nrow_ctas), static_cast<unsigned>(ksplit), 1);
    pl->smem = lay.total;
    pl->cw = cw;
    return true;
}

// CTAs of one streaming-GEMV instantiation that fit an SM (its registers
// decide), at most kCtasPerSm; queried once per instantiation.
template <int QT, int MAXB, int NMAT, int XMODE, int EPI>
inline int stream_ctas_per_sm() {
    static int cached = 0;
    if (cached == 0) {
        constexpr int CW = cw_for(MAXB);
        constexpr auto kern = gemv_stream_kernel<QT, CW, MAXB, NMAT, XMODE, EPI>;
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, KCfg<QT, CW>::threads, 0) != cudaSuccess || n < 1)
            n = 1;
        cached = std::min(n, kCtasPerSm);
    }
    return cached;
}

template <int QT, int MAXB, int NMAT, int XMODE, int EPI>
inline cudaError_t run_stream(const GemvPlan& pl, cudaStream_t s, bool pdl) {
    constexpr int CW = cw_for(MAXB);
    constexpr auto kern = gemv_stream_kernel<QT, CW, MAXB, NMAT, XMODE, EPI>;
    cudaError_t e = ensure_smem_attr<kern>();
    if (e != cudaSuccess) return e;
    return launch_kernel(kern, pl.grid, dim3(KCfg<QT, CW>::threads), pl.smem, s, pdl, pl.p);
}

}  // namespace phb
