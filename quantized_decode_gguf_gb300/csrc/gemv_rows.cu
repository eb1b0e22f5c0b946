// Row-resident streaming GEMV for batched activations (batch 2..8).
//
// The kernel of gemv_kernel.cuh maps threads to half units along K; every
// thread reads its own activations from shared memory, batch rows times
// per weight, and rows are reduced across threads. With several activation
// rows that shared-memory traffic bounds it. Here the mapping is transposed.
//
// A CTA owns 128 weight rows and a K range. Each stage is one 256-weight unit
// of all 128 rows, moved by one 2-D TMA copy ([128 rows][one unit], rows
// `row_bytes` apart in HBM, packed in shared memory). Thread t works on row
// t % 128 and half unit t / 128 of every stage. It keeps the row's batch
// partial sums in registers across the whole K range. All threads of a warp
// read the same activations (a shared-memory broadcast), so activation
// traffic no longer scales with the rows, and no cross-thread row reduction
// is needed; the two halves of a row meet once at the end.
//
// The dequantize-and-dot arithmetic (exact scaled weights, power-of-two
// activation scaling, packed FMAs) is gemv_core.cuh's.
// K splits write partials reduced in split order by splitk_reduce_kernel,
// so results are deterministic.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "gemv_plan.cuh"
#include "phb_internal.h"

namespace phb {

cudaError_t read_dev_err_gemv_rows(int* code) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_dev_err, sizeof(int));
    if (e != cudaSuccess) return e;
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_dev_err, &zero, sizeof(int));
    *code = v;
    return e;
}

namespace {

constexpr int kRows = 128;            // weight rows per CTA (one per thread pair)
constexpr int kRowsCW = 8;            // consumer warps
constexpr int kRowsNC = 32 * kRowsCW;
constexpr int kRowsThreads = kRowsNC + 32;
constexpr size_t kRowsXBudget = 96 * 1024;  // staged activations per CTA

template <int QT>
struct RowsCfg {
    static constexpr int ub = Fmt<QT>::unit_bytes;
    static constexpr int stage_bytes = kRows * ub;  // 18 KB (Q4_K) or 34 KB (Q8_0)
    static constexpr int ns = QT == 0 ? 3 : 6;
};

struct RowsParams {
    const float* x;
    int64_t ldx;
    float* y;
    int64_t ldy;
    float* part;              // split-K partials [split][batch][n]
    int64_t n;
    int units_row, units_per_split;
    int batch;
    uint32_t xs_off, comb_off, bar_off;
};

__device__ __forceinline__ void tma_load_2d_hint(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                                 uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
        "%3}], [%4], %5;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

template <int QT, int MAXB>
__global__ void __launch_bounds__(kRowsThreads, 1)
    gemv_rows_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ RowsParams p) {
    using R = RowsCfg<QT>;
    extern __shared__ __align__(1024) uint8_t smem[];
    float* xs = reinterpret_cast<float*>(smem + p.xs_off);
    float* comb = reinterpret_cast<float*>(smem + p.comb_off);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.bar_off);
    uint64_t* empty = full + R::ns;
    float* xfac = reinterpret_cast<float*>(empty + R::ns);
    float* red = xfac + kAccStride;

    const int tid = threadIdx.x, lane = tid & 31;
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kRows;
    const int split = blockIdx.y;
    const int u0 = split * p.units_per_split;
    const int nst = min(p.units_per_split, p.units_row - u0);  // stages = units of this split
    if (tid == 0) {
        for (int s = 0; s < R::ns; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kRowsCW);
        }
        fence_barrier_init();
    }
    __syncthreads();
    pdl_launch_dependents();

    if (tid >= kRowsNC) {
        // ---------------- producer: one 2-D copy per stage (weights do not depend on earlier kernels)
        if (tid == kRowsNC) {
            const uint64_t pol = policy_evict_first();
            constexpr int kElems = QT == 0 ? R::ub / 2 : R::ub;  // Q8_0 rows are mapped as 16-bit elements
            int issued = 0;
            for (int st = 0; st < nst; ++st, ++issued) {
                const int slot = st % R::ns;
                if (st >= R::ns && !mbar_wait(&empty[slot], ((st / R::ns) - 1) & 1, &g_dev_err)) break;
                mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(R::stage_bytes));
                tma_load_2d_hint(smem + slot * R::stage_bytes, &tmap_w, (u0 + st) * kElems, static_cast<int>(n0),
                                 &full[slot], pol);
            }
            // every copy issued must land before the CTA exits (bounded waits; long done on the normal path)
            for (int st = max(0, issued - R::ns); st < issued; ++st)
                mbar_wait(&full[st % R::ns], (st / R::ns) & 1, &g_dev_err);
        }
        return;
    }

    // ---------------- consumers
    pdl_wait();  // x may come from the previous kernel
    const int kseg = nst * kUnitWeights;
    stage_x<kRowsCW, MAXB, kXPlain>(p.x, p.ldx, static_cast<int64_t>(u0) * kUnitWeights, kseg, p.batch, xs, xfac,
                                    red, 1, 1, 0);
    const int row = tid & (kRows - 1);
    const int h = tid >> 7;  // half unit; uniform per warp, so activation loads are broadcasts
    const int xstride = xpad_len(kseg);
    float acc[MAXB];
#pragma unroll
    for (int b = 0; b < MAXB; ++b) acc[b] = 0.f;
    bool ok = true;
    for (int st = 0; st < nst; ++st) {
        const int slot = st % R::ns;
        int good = 1;
        if (lane == 0) good = mbar_wait(&full[slot], (st / R::ns) & 1, &g_dev_err) ? 1 : 0;
        good = __shfl_sync(0xFFFFFFFFu, good, 0);
        __syncwarp();
        if (!good) {
            ok = false;
            break;
        }
        const uint8_t* ub = smem + slot * R::stage_bytes + row * R::ub;
        const int hu = 2 * st + h;
        const float* xsp = xs + hu * (kXPadEvery + kXPad);
        if constexpr (QT == 0)
            dot_q8_0_half<MAXB>(ub + 136 * h, xsp, xstride, xfac, acc);
        else
            dot_q4_k_half<MAXB>(ub, h, xsp, xstride, xfac, acc);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
    }
    // the two halves of a row meet: second half through shared memory, first half adds and stores
    if (h == 1) {
#pragma unroll
        for (int b = 0; b < MAXB; ++b) comb[b * kRows + row] = acc[b];
    }
    consumer_sync<kRowsNC>();
    if (h == 0 && ok) {
        const int64_t n = n0 + row;
        if (n < p.n) {
            const bool split_out = gridDim.y > 1;
#pragma unroll
            for (int b = 0; b < MAXB; ++b) {
                if (b < p.batch) {
                    const float v = acc[b] + comb[b * kRows + row];
                    if (split_out)
                        p.part[(static_cast<int64_t>(split) * p.batch + b) * p.n + n] = v;
                    else
                        p.y[b * p.ldy + n] = v;
                }
            }
        }
    }
}

PFN_cuTensorMapEncodeTiled_v12000 rows_encode_fn() {
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

struct RowsPlan {
    int ksplit = 1, units_per_split = 0;
    size_t smem = 0;
    uint32_t xs_off = 0, comb_off = 0, bar_off = 0;
};

// Splits of K: enough CTAs to cover the SMs once (the kernel fills an SM),
// and each split's staged activations within kRowsXBudget.
RowsPlan plan_rows(int qt, int64_t n, int64_t k, int batch) {
    const int maxb = maxb_for(batch);
    const int units_row = static_cast<int>(k / kUnitWeights);
    const int64_t tiles = cdiv(n, kRows);
    const int sms = device_sm_count();
    int ksplit = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(units_row, sms / std::max<int64_t>(1, tiles))));
    const size_t x_per_unit = static_cast<size_t>(maxb) * xpad_len(kUnitWeights) * 4;
    const int max_units = std::max(1, static_cast<int>(kRowsXBudget / x_per_unit));
    ksplit = std::max(ksplit, static_cast<int>(cdiv(units_row, max_units)));
    RowsPlan pl;
    pl.units_per_split = static_cast<int>(cdiv(units_row, ksplit));
    pl.ksplit = static_cast<int>(cdiv(units_row, pl.units_per_split));
    const int kseg = pl.units_per_split * kUnitWeights;
    const int ns = qt == 0 ? RowsCfg<0>::ns : RowsCfg<1>::ns;
    const size_t stage = static_cast<size_t>(kRows) * (qt == 0 ? Fmt<0>::unit_bytes : Fmt<1>::unit_bytes);
    size_t off = ns * stage;
    pl.xs_off = static_cast<uint32_t>(off);
    off += static_cast<size_t>(maxb) * xpad_len(kseg) * 4;
    pl.comb_off = static_cast<uint32_t>(off);
    off += static_cast<size_t>(maxb) * kRows * 4;
    off = (off + 15) & ~size_t{15};
    pl.bar_off = static_cast<uint32_t>(off);
    off += 2 * ns * sizeof(uint64_t) + kTailFloats * sizeof(float);
    pl.smem = off;
    return pl;
}

template <int QT, int MAXB>
cudaError_t launch_rows(const CUtensorMap& tmap, const RowsParams& p, dim3 grid, size_t smem, cudaStream_t s,
                        bool pdl) {
    constexpr auto kern = gemv_rows_kernel<QT, MAXB>;
    cudaError_t e = ensure_smem_attr<kern>();
    if (e != cudaSuccess) return e;
    return launch_kernel(kern, grid, dim3(kRowsThreads), smem, s, pdl, tmap, p);
}

}  // namespace

size_t gemv_rows_ws_floats(int qt, int64_t n, int64_t k, int batch) {
    const RowsPlan pl = plan_rows(qt, n, k, batch);
    return pl.ksplit > 1 ? static_cast<size_t>(pl.ksplit) * batch * n : 0;
}

cudaError_t gemv_rows_run(const GemvReq& q, cudaStream_t s, int* ksplit_out) {
    PFN_cuTensorMapEncodeTiled_v12000 encode = rows_encode_fn();
    if (encode == nullptr) return cudaErrorNotSupported;
    const RowsPlan pl = plan_rows(q.qt, q.n, q.k, q.batch);
    if (pl.smem > kSmemOptin) return cudaErrorInvalidConfiguration;
    if (pl.ksplit > 1 && (q.ws == nullptr || q.ws_floats < static_cast<size_t>(pl.ksplit) * q.batch * q.n))
        return cudaErrorInvalidValue;
    // the weight matrix as a 2-D tensor [n rows][row bytes]; one box = one unit of 128 rows
    const int ub = q.qt == 0 ? Fmt<0>::unit_bytes : Fmt<1>::unit_bytes;
    const int64_t row_bytes = q.k / kUnitWeights * ub;
    const int esz = q.qt == 0 ? 2 : 1;
    CUtensorMap tmap;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes / esz), static_cast<cuuint64_t>(q.n)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(ub / esz), static_cast<cuuint32_t>(kRows)};
    const cuuint32_t estr[2] = {1, 1};
    if (encode(&tmap, q.qt == 0 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
               const_cast<void*>(q.w0), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    RowsParams p{};
    p.x = q.x;
    p.ldx = q.ldx;
    p.y = q.y;
    p.ldy = q.ldy;
    p.part = q.ws;
    p.n = q.n;
    p.units_row = static_cast<int>(q.k / kUnitWeights);
    p.units_per_split = pl.units_per_split;
    p.batch = q.batch;
    p.xs_off = pl.xs_off;
    p.comb_off = pl.comb_off;
    p.bar_off = pl.bar_off;
    const dim3 grid(static_cast<unsigned>(cdiv(q.n, kRows)), static_cast<unsigned>(pl.ksplit));
    *ksplit_out = pl.ksplit;
    const int maxb = maxb_for(q.batch);
    if (q.qt == 0) {
        switch (maxb) {
            case 1: return launch_rows<0, 1>(tmap, p, grid, pl.smem, s, q.pdl);
            case 2: return launch_rows<0, 2>(tmap, p, grid, pl.smem, s, q.pdl);
            case 4: return launch_rows<0, 4>(tmap, p, grid, pl.smem, s, q.pdl);
            default: return launch_rows<0, 8>(tmap, p, grid, pl.smem, s, q.pdl);
        }
    }
    switch (maxb) {
        case 1: return launch_rows<1, 1>(tmap, p, grid, pl.smem, s, q.pdl);
        case 2: return launch_rows<1, 2>(tmap, p, grid, pl.smem, s, q.pdl);
        case 4: return launch_rows<1, 4>(tmap, p, grid, pl.smem, s, q.pdl);
        default: return launch_rows<1, 8>(tmap, p, grid, pl.smem, s, q.pdl);
    }
}

}  // namespace phb
