// Prompt-processing GEMM on the 5th-generation tensor cores (tcgen05).
//
//   Y[t][n] = sum_k bf16(w[n][k]) * bf16(X[t][k]),  fp32 accumulation.
//
// The weights are the MMA's M operand: a CTA owns 128 weight rows and 256
// tokens (D = 128 x 256 fp32 in TMEM, columns 0-255). Per 64-wide K block:
//  - eight producer warps, in two groups taking alternate K blocks,
//    dequantise their rows (one row per thread) to bf16 and write them
//    straight into TMEM with tcgen05.st (lane = weight row,
//    32 columns of bf16 pairs per K block, one slot per stage after the
//    accumulator): the MMA reads its A operand from TMEM, so the weight tile
//    never passes through shared memory and needs no proxy fence. Raw units
//    come from global memory into a register double buffer (Q4_K) or are
//    staged in shared memory by a 2-D TMA copy per 256-weight unit of the
//    CTA's 128 rows (Q8_0);
//  - one thread loads the token tile (bf16, 256 x 64) with a 2-D TMA copy
//    into the 128-byte-swizzled K-major layout the MMA reads;
//  - one thread issues four tcgen05.mma (M128 N256 K16, A in TMEM, B in
//    shared memory) and commits them to the stage's "empty" barrier;
// after the last K block the four producer warps drain the accumulator
// (tcgen05.ld, one TMEM lane per weight row) and write Y. With K split
// over several CTAs (fewer tiles than SMs), the splits of a tile form one
// thread-block cluster: each drains its partial tile into its own shared
// memory and, after a cluster barrier, sums a share of the tile's tokens
// over the splits' shared memory (in split order) and writes Y. Splits
// beyond a portable cluster write partials that a second kernel reduces in
// split order. X is cast to bf16 (round to nearest even) by a first kernel
// into the caller's workspace.
//
// Every wait is bounded; a wait that runs out sets this translation unit's
// device error word, the kernel drains and frees its TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "gemv_core.cuh"
#include "phb_common.cuh"
#include "phb_internal.h"
#include "trace.cuh"

namespace phb {

static __device__ int g_dev_err_prefill;

// debug builds: stamps of the last GEMM launch per CTA (entry, TMEM allocated, first
// weight tile stored, X ready, first MMA, last MMA issued, accumulator complete, outputs written)
PHB_TRACE_READER(phb_trace_read_prefill)

cudaError_t read_dev_err_prefill(int* code) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_dev_err_prefill, sizeof(int));
    if (e != cudaSuccess) return e;
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_dev_err_prefill, &zero, sizeof(int));
    *code = v;
    return e;
}

namespace {

constexpr int kBM = 128;                   // weight rows per CTA (MMA M)
constexpr int kBN = 256;                   // tokens per CTA (MMA N)
constexpr int kBK = 64;                    // K per stage: one 128-byte bf16 row
constexpr int kBTile = kBN * kBK * 2;      // 32 KB
constexpr int kProducerWarps = 4;          // warps per K block, one weight row per thread; warps 0-3 drain TMEM
constexpr int kProducerGroups = 2;         // groups of producer warps, taking alternate K blocks
constexpr int kTmaWarp = kProducerWarps * kProducerGroups;  // token tiles
constexpr int kMmaWarp = kTmaWarp + 1;
constexpr int kRawWarp = kTmaWarp + 2;     // raw weight units
constexpr int kThreads = 32 * (kRawWarp + 1);
// TMEM: the fp32 accumulator in columns 0-255, then one 32-column slot per
// stage for the bf16 weight tile (the MMA's A operand, read from TMEM: lane
// = weight row, column c = the bf16 pair k = 2c, 2c + 1 of the K block).
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAcol0 = 256;

// Per format: Q8_0 stages its raw 256-weight units (128 rows x 272 bytes) in
// shared memory by TMA, beside four token-tile stages; Q4_K double-buffers
// its raw units (144 bytes a row) in registers, read by each producer thread
// from global memory, and keeps six stages. (TMEM holds the accumulator and
// one 32-column weight slot per stage: at most 8 stages.)
template <int QT>
struct PCfg {
    static constexpr bool staged = QT == 0;
    static constexpr int stages = staged ? 4 : 6;
    static constexpr int raw_stages = staged ? 2 : 0;
    static constexpr int raw_bytes = kBM * 272;  // one raw slot
    static_assert(kAcol0 + 32 * stages <= kTmemCols, "a weight slot per stage after the accumulator");
    static constexpr size_t smem =
        stages * kBTile + raw_stages * raw_bytes + 1024 /* align */ + 256 /* barriers */;
};
constexpr int kKbPerUnit = 4;              // a 256-weight unit spans four K blocks

struct PrefillParams {
    const uint8_t* w;
    int64_t row_bytes;
    int64_t n, m, k;
    int units_per_split;  // 256-weight units of K per split
    int n_units;          // K / 256
    float* y;             // [m][n]
    float* part;          // [splits][m][n] when gridDim.z > 1 and the splits are not a cluster
    int cluster;          // 1: the gridDim.z splits of a tile are one cluster (sum over shared memory)
};

// ---------------------------------------------------------------- tcgen05 / TMA PTX
__device__ __forceinline__ uint64_t smem_desc_sw128(const void* p) {
    // K-major operand in the 128-byte swizzle layout: 8-row groups of
    // 128-byte rows, 1024 bytes apart (stride byte offset); version 1.
    const uint64_t addr = smem_addr(p);
    return ((addr & 0x3FFFFull) >> 4) | (1ull << 16) | ((1024ull >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

// kind::f16, D fp32, A and B bf16, both K-major, M = 128, N = 256.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(kBN >> 3) << 17) | (uint32_t(kBM >> 4) << 24);

// One MMA with A read from TMEM (128 lanes x 8 columns of bf16 pairs per K = 16), B from shared memory.
__device__ __forceinline__ void mma_bf16_ta(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
        "r"(tmem_a), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

// ---------------------------------------------------------------- cluster / distributed shared memory
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of every CTA of the cluster: release this CTA's shared-memory
// writes, then acquire the others'.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// 16 bytes at shared address `addr` of the cluster's CTA `rank`.
__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t addr, uint32_t rank) {
    uint32_t ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(addr), "r"(rank));
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(ra)
                 : "memory");
    return v;
}

// 32 consecutive TMEM columns of this warp's 32 lanes, one lane per thread.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 consecutive TMEM columns of this warp's 32 lanes from 32 registers a thread, then
// wait until the stores are done.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
        "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
        "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- dequant to bf16 pairs
__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    const __nv_bfloat162 t = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&t);
}

// Byte SEL of w as the float 2^23 + byte (exact).
template <int SEL>
__device__ __forceinline__ float byte_magic(uint32_t w) {
    return __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7440u | SEL));
}

__device__ __forceinline__ float byte_magic_rt(uint32_t w, int sel) {
    return __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7440u | static_cast<uint32_t>(sel)));
}

// One K block (64 weights) of a Q8_0 unit held in registers (68 words).
// Two weights per packed operation: (2^23 + u) - (2^23 + 128) = q and d q,
// both exact, then one rounding to bf16.
template <int J>
__device__ __forceinline__ void dequant_q8_0_kb(const uint32_t (&u)[68], uint32_t (&out)[32]) {
    const float2 bias = make_float2(-8388736.0f, -8388736.0f);
#pragma unroll
    for (int hb = 0; hb < 2; ++hb) {
        const int ob = 68 * J + 34 * hb;  // byte offset of the block in the unit
        const uint32_t dw = u[ob / 4];
        const float d = fp16_bits_to_float((ob % 4) ? (dw >> 16) : dw);
        const float2 d2 = make_float2(d, d);
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
            const int p0 = ob + 2 + i, p1 = p0 + 1;
            const float2 m = make_float2(byte_magic_rt(u[p0 / 4] ^ 0x80808080u, p0 % 4),
                                         byte_magic_rt(u[p1 / 4] ^ 0x80808080u, p1 % 4));
            const float2 w = __fmul2_rn(d2, __fadd2_rn(m, bias));  // exact
            out[16 * hb + i / 2] = pack_bf16(w.x, w.y);
        }
    }
}

// One K block (64 weights: sub-blocks 2J and 2J+1) of a Q4_K block in
// registers (36 words). Two weights per packed operation: the nibble as
// (2^23 + q) - 2^23 = q exactly, then one rounding of D q - M (fma), then bf16.
template <int J>
__device__ __forceinline__ void dequant_q4_k_kb(const uint32_t (&u)[36], uint32_t (&out)[32]) {
    const float d = fp16_bits_to_float(u[0]);
    const float dmin = fp16_bits_to_float(u[0] >> 16);
    const uint32_t sw[3] = {u[1], u[2], u[3]};
    const float2 magic = make_float2(-8388608.0f, -8388608.0f);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        uint32_t sc, m;
        q4_k_scale_min(sw, 2 * J + half, sc, m);
        const float D = d * static_cast<float>(sc);     // exact
        const float M = dmin * static_cast<float>(m);   // exact
        const float2 D2 = make_float2(D, D), nM2 = make_float2(-M, -M);
#pragma unroll
        for (int i4 = 0; i4 < 8; ++i4) {
            const uint32_t word = u[4 + 8 * J + i4];
            const uint32_t nib = (half ? (word >> 4) : word) & 0x0F0F0F0Fu;
            const float2 q01 = __fadd2_rn(make_float2(byte_magic<0>(nib), byte_magic<1>(nib)), magic);
            const float2 q23 = __fadd2_rn(make_float2(byte_magic<2>(nib), byte_magic<3>(nib)), magic);
            const float2 w01 = __ffma2_rn(D2, q01, nM2);  // one rounding of the exact D q - M
            const float2 w23 = __ffma2_rn(D2, q23, nM2);
            out[16 * half + 2 * i4] = pack_bf16(w01.x, w01.y);
            out[16 * half + 2 * i4 + 1] = pack_bf16(w23.x, w23.y);
        }
    }
}

template <int NW>
__device__ __forceinline__ void load_unit(const uint8_t* src, uint32_t (&u)[NW]) {
#pragma unroll
    for (int i = 0; i < NW / 4; ++i) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(src) + i);
        u[4 * i] = v.x;
        u[4 * i + 1] = v.y;
        u[4 * i + 2] = v.z;
        u[4 * i + 3] = v.w;
    }
}

// ---------------------------------------------------------------- the GEMM kernel
template <int QT>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_gemm_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_w,
                        const __grid_constant__ PrefillParams p) {
    constexpr int kStages = PCfg<QT>::stages;
    constexpr int kRawStages = PCfg<QT>::raw_stages > 0 ? PCfg<QT>::raw_stages : 1;
    constexpr int kRawBytesMax = PCfg<QT>::raw_stages * PCfg<QT>::raw_bytes;
    constexpr int UB = QT == 0 ? 272 : 144;      // bytes of one 256-weight unit of a row
    constexpr int kUnitElems = QT == 0 ? 136 : 144;  // the same in tensor-map elements (u16 / u8)
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t{1023});
    uint8_t* sB = smem;
    uint8_t* sR = sB + kStages * kBTile;  // staged raw units: [raw stages][128 rows][UB]
    uint64_t* full = reinterpret_cast<uint64_t*>(sR + kRawBytesMax);
    uint64_t* empty = full + kStages;
    uint64_t* accb = empty + kStages;
    uint64_t* rfull = accb + 1;
    uint64_t* rempty = rfull + kRawStages;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(rempty + kRawStages);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) PHB_TRACE_EV(0, 0);
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kBM;
    const int t0 = blockIdx.y * kBN;
    const int split = blockIdx.z;
    const int u0 = split * p.units_per_split;
    const int nu = min(p.units_per_split, p.n_units - u0);
    const int nkb = nu * kKbPerUnit;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], kProducerWarps + 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(accb, 1);
        for (int s = 0; s < PCfg<QT>::raw_stages; ++s) {
            mbar_init(&rfull[s], 1);
            mbar_init(&rempty[s], kProducerWarps * kProducerGroups);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (tid == 0) PHB_TRACE_EV(0, 1);
    pdl_launch_dependents();

    if (warp < kProducerWarps * kProducerGroups) {
        // ---------------- dequant producers: thread tid owns weight row n0 + tid % 128 and,
        // in group g = tid / 128, the K blocks j = g, g + groups, ... of every unit
        const int row = tid & (kBM - 1);
        const int grp = tid / kBM;
        constexpr int NW = UB / 4;
        uint32_t cur[NW];
        [[maybe_unused]] uint32_t nxt[PCfg<QT>::staged ? 1 : NW];
        const uint8_t* wr = p.w + (n0 + row) * p.row_bytes;
        if constexpr (!PCfg<QT>::staged)
            if (nu > 0) load_unit<NW>(wr + static_cast<int64_t>(u0) * UB, cur);
        for (int uu = 0; uu < nu; ++uu) {
            if constexpr (PCfg<QT>::staged) {
                // this row's raw unit from the staged copy of the CTA's 128 rows
                const int rs = uu % kRawStages;
                if (!mbar_wait_warp(&rfull[rs], (uu / kRawStages) & 1, &g_dev_err_prefill)) {
                    *abort_flag = 1;
                    break;
                }
                const uint8_t* src = sR + rs * PCfg<QT>::raw_bytes + row * UB;
#pragma unroll
                for (int i = 0; i < NW / 4; ++i) {
                    const uint4 v = *reinterpret_cast<const uint4*>(src + 16 * i);
                    cur[4 * i] = v.x;
                    cur[4 * i + 1] = v.y;
                    cur[4 * i + 2] = v.z;
                    cur[4 * i + 3] = v.w;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&rempty[rs]);  // the slot may be refilled
            } else {
                if (uu + 1 < nu) load_unit<NW>(wr + static_cast<int64_t>(u0 + uu + 1) * UB, nxt);
            }
#pragma unroll
            for (int j = 0; j < kKbPerUnit; ++j) {
                if (j % kProducerGroups != grp) continue;
                const int i = uu * kKbPerUnit + j;
                const int s = i % kStages;
                if (i >= kStages && !mbar_wait_warp(&empty[s], ((i / kStages) - 1) & 1, &g_dev_err_prefill)) {
                    *abort_flag = 1;
                    break;
                }
                tc_fence_after();  // the MMAs that read this slot have completed (empty barrier)
                uint32_t pk[32];
                if constexpr (QT == 0) {
                    if (j == 0) dequant_q8_0_kb<0>(cur, pk);
                    else if (j == 1) dequant_q8_0_kb<1>(cur, pk);
                    else if (j == 2) dequant_q8_0_kb<2>(cur, pk);
                    else dequant_q8_0_kb<3>(cur, pk);
                } else {
                    if (j == 0) dequant_q4_k_kb<0>(cur, pk);
                    else if (j == 1) dequant_q4_k_kb<1>(cur, pk);
                    else if (j == 2) dequant_q4_k_kb<2>(cur, pk);
                    else dequant_q4_k_kb<3>(cur, pk);
                }
                tmem_st32(tmem + (static_cast<uint32_t>(32 * (warp % kProducerWarps)) << 16) + kAcol0 + 32 * s, pk);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&full[s]);
                if (tid == 0 && i == 0) PHB_TRACE_EV(0, 2);
            }
            if (*abort_flag) break;
            if constexpr (!PCfg<QT>::staged) {
#pragma unroll
                for (int i = 0; i < NW; ++i) cur[i] = nxt[i];
            }
        }
    } else if (warp == kTmaWarp) {
        // ---------------- token tiles by TMA
        if (lane == 0) {
            pdl_wait();  // the bf16 copy of X comes from the previous kernel
            PHB_TRACE_EV(0, 3);
            for (int i = 0; i < nkb; ++i) {
                const int s = i % kStages;
                if (i >= kStages && !mbar_wait(&empty[s], ((i / kStages) - 1) & 1, &g_dev_err_prefill)) {
                    *abort_flag = 1;
                    break;
                }
                mbar_arrive_expect_tx(&full[s], kBTile);
                tma_load_2d(sB + s * kBTile, &tmap_x, (u0 * kKbPerUnit + i) * kBK, t0, &full[s]);
            }
            // Before the CTA can exit, every copy issued into shared memory must
            // have landed: wait (bounded) on the last phase of each slot. On the
            // normal path these phases completed long ago.
            for (int i = max(0, nkb - kStages); i < nkb; ++i)
                mbar_wait(&full[i % kStages], (i / kStages) & 1, &g_dev_err_prefill);
        }
    } else if (PCfg<QT>::staged && warp == kRawWarp) {
        // ---------------- raw weight units by TMA (weights never depend on the previous kernel)
        if (lane == 0) {
            for (int uu = 0; uu < nu; ++uu) {
                const int rs = uu % kRawStages;
                if (uu >= kRawStages && !mbar_wait(&rempty[rs], ((uu / kRawStages) - 1) & 1, &g_dev_err_prefill)) {
                    *abort_flag = 1;
                    break;
                }
                mbar_arrive_expect_tx(&rfull[rs], static_cast<uint32_t>(kBM * UB));
                tma_load_2d(sR + rs * PCfg<QT>::raw_bytes, &tmap_w, (u0 + uu) * kUnitElems, static_cast<int>(n0), &rfull[rs]);
            }
            // every copy into shared memory must land before the CTA exits (bounded waits)
            for (int uu = max(0, nu - kRawStages); uu < nu; ++uu)
                mbar_wait(&rfull[uu % kRawStages], (uu / kRawStages) & 1, &g_dev_err_prefill);
        }
    } else if (warp == kMmaWarp) {
        // ---------------- one thread issues the MMAs
        if (lane == 0) {
            bool ok = true;
            for (int i = 0; i < nkb; ++i) {
                const int s = i % kStages;
                if (!mbar_wait(&full[s], (i / kStages) & 1, &g_dev_err_prefill)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (i == 0) PHB_TRACE_EV(0, 4);
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk) {
                    const uint64_t bd = smem_desc_sw128(sB + s * kBTile + kk * 32);
                    mma_bf16_ta(tmem, tmem + kAcol0 + 32 * s + 8 * kk, bd, (i > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(&empty[s]);
            }
            if (!ok) *abort_flag = 1;
            PHB_TRACE_EV(0, 5);
            mma_commit(accb);  // arrives once every MMA issued above has completed
        }
    }

    // ---------------- epilogue: warps 0-3 drain TMEM lanes 0..127 (one weight row each)
    if (p.cluster) {
        // this split's partial tile into shared memory as [256 tokens][128 rows]
        // fp32 (the token-tile stages are idle once every MMA has completed)
        float* sAcc = reinterpret_cast<float*>(sB);
        if (warp < kProducerWarps) {
            const bool ready = mbar_wait_warp(accb, 0, &g_dev_err_prefill);
            if (tid == 0) PHB_TRACE_EV(0, 6);
            tc_fence_after();
            if (ready && !*abort_flag) {
                const int r = 32 * warp + lane;
#pragma unroll 1
                for (int c0 = 0; c0 < kBN; c0 += 32) {
                    float v[32];
                    tmem_ld32(tmem + (static_cast<uint32_t>(32 * warp) << 16) + c0, v);
#pragma unroll
                    for (int j = 0; j < 32; ++j) sAcc[(c0 + j) * kBM + r] = v[j];
                }
            }
        }
        tc_fence_before();
        cluster_sync_all();
        // this CTA's share of the tile's tokens: the splits' partials summed in
        // split order, 4 rows a thread, one token per warp pass
        pdl_wait();  // outputs may still be read by the previous kernel
        const int nsplit = static_cast<int>(gridDim.z);
        const int per = (kBN + nsplit - 1) / nsplit;
        const int rank = static_cast<int>(cluster_rank());
        const int ta = rank * per, tb = min(kBN, min(ta + per, static_cast<int>(p.m - t0)));
        const uint32_t base = smem_addr(sAcc);
        for (int it = ta * (kBM / 4) + tid; it < tb * (kBM / 4); it += kThreads) {
            const int t = it / (kBM / 4), r4 = 4 * (it % (kBM / 4));
            const uint32_t off = base + static_cast<uint32_t>((t * kBM + r4) * sizeof(float));
            float4 acc = ld_dsmem_f4(off, 0);
            for (int q = 1; q < nsplit; ++q) {
                const float4 v = ld_dsmem_f4(off, static_cast<uint32_t>(q));
                acc.x += v.x;
                acc.y += v.y;
                acc.z += v.z;
                acc.w += v.w;
            }
            *reinterpret_cast<float4*>(p.y + static_cast<int64_t>(t0 + t) * p.n + n0 + r4) = acc;
        }
        // no CTA may leave while another still reads its shared memory
        cluster_sync_all();
        if (tid == 0) PHB_TRACE_EV(0, 7);
    } else if (warp < kProducerWarps) {
        pdl_wait();  // outputs may still be read by the previous kernel
        const bool ready = mbar_wait_warp(accb, 0, &g_dev_err_prefill);
        if (tid == 0) PHB_TRACE_EV(0, 6);
        tc_fence_after();
        if (ready && !*abort_flag && nkb > 0) {
            const int64_t n = n0 + 32 * warp + lane;
            float* out = gridDim.z > 1 ? p.part + static_cast<int64_t>(split) * p.m * p.n : p.y;
#pragma unroll 1
            for (int c0 = 0; c0 < kBN; c0 += 32) {
                float v[32];
                tmem_ld32(tmem + (static_cast<uint32_t>(32 * warp) << 16) + c0, v);
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int t = t0 + c0 + j;
                    if (t < p.m) out[static_cast<int64_t>(t) * p.n + n] = v[j];
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && !p.cluster) PHB_TRACE_EV(0, 7);
    if (warp == kMmaWarp) {
        // every MMA issued has completed once accb has arrived (bounded wait)
        mbar_wait_warp(accb, 0, &g_dev_err_prefill);
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

// X fp32 [m][k] -> bf16 (round to nearest even), 8 values per thread.
__global__ void __launch_bounds__(256) cast_bf16_kernel(const float* __restrict__ x, uint32_t* __restrict__ xb,
                                                        int64_t count8) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < count8; i += stride) {
        const float4 a = reinterpret_cast<const float4*>(x)[2 * i];
        const float4 b = reinterpret_cast<const float4*>(x)[2 * i + 1];
        reinterpret_cast<uint4*>(xb)[i] =
            make_uint4(pack_bf16(a.x, a.y), pack_bf16(a.z, a.w), pack_bf16(b.x, b.y), pack_bf16(b.z, b.w));
    }
}

// Y = sum over splits in split order.
__global__ void __launch_bounds__(256) prefill_reduce_kernel(const float4* __restrict__ part, float4* __restrict__ y,
                                                             int64_t count4, int splits) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < count4; i += stride) {
        float4 acc = part[i];
        for (int s = 1; s < splits; ++s) {
            const float4 v = part[static_cast<int64_t>(s) * count4 + i];
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        y[i] = acc;
    }
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
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

struct SplitPlan {
    int splits;
    int units_per_split;
    bool cluster;  // the splits of a tile run as one cluster and sum in shared memory
};

constexpr int kMaxClusterSplits = 8;  // portable cluster size

// Whether clusters of `splits` CTAs of this kernel can be resident (queried once per size).
template <int QT>
bool cluster_fits(int splits) {
    static std::atomic<int> known[kMaxClusterSplits + 1] = {};
    int v = known[splits].load(std::memory_order_acquire);
    if (v != 0) return v > 0;
    constexpr auto kern = prefill_gemm_kernel<QT>;
    int n = 0;
    if (ensure_smem_attr<kern>() == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(1, 1, static_cast<unsigned>(splits));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = PCfg<QT>::smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 1;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = static_cast<unsigned>(splits);
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
            (void)cudaGetLastError();
            n = 0;
        }
    }
    known[splits].store(n > 0 ? 1 : -1, std::memory_order_release);
    return n > 0;
}

SplitPlan plan_splits(int qt, int64_t m, int64_t n, int64_t k) {
    const int n_units = static_cast<int>(k / kUnitWeights);
    const int64_t tiles = (n / kBM) * ((m + kBN - 1) / kBN);
    const int sms = device_sm_count();
    int splits = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(sms / std::max<int64_t>(1, tiles), n_units)));
    const int ups = (n_units + splits - 1) / splits;
    splits = (n_units + ups - 1) / ups;
    const bool cluster = splits > 1 && splits <= kMaxClusterSplits &&
                         (qt == 0 ? cluster_fits<0>(splits) : cluster_fits<1>(splits));
    return {splits, ups, cluster};
}

inline size_t align_up(size_t v) { return (v + 255) & ~size_t{255}; }

}  // namespace

size_t prefill_ws_bytes(const PrefillReq& q) {
    const SplitPlan sp = plan_splits(q.qt, q.m, q.n, q.k);
    size_t b = align_up(static_cast<size_t>(q.m) * q.k * 2);
    if (sp.splits > 1 && !sp.cluster) b += static_cast<size_t>(sp.splits) * q.m * q.n * sizeof(float);
    return b;
}

cudaError_t prefill_run(const PrefillReq& q, cudaStream_t s) {
    PFN_cuTensorMapEncodeTiled_v12000 encode = get_encode_fn();
    if (encode == nullptr) return cudaErrorNotSupported;
    const SplitPlan sp = plan_splits(q.qt, q.m, q.n, q.k);
    auto* ws = static_cast<uint8_t*>(q.ws);
    uint32_t* xb = reinterpret_cast<uint32_t*>(ws);
    float* part = reinterpret_cast<float*>(ws + align_up(static_cast<size_t>(q.m) * q.k * 2));

    // token matrix (bf16 [m][k]) as a 2-D tensor: 64 x 256 boxes, 128-byte swizzle
    CUtensorMap tmap;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(q.k), static_cast<cuuint64_t>(q.m)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(q.k) * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(kBN)};
    const cuuint32_t estr[2] = {1, 1};
    if (encode(&tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, xb, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;

    // weights [n][row bytes] as a 2-D tensor: one box = one 256-weight unit of 128 rows
    // (u16 elements for Q8_0 so the 272-byte unit stays within the 256-element box limit)
    CUtensorMap tmap_w;
    {
        const int64_t row_bytes = q.qt == 0 ? q.k / 32 * 34 : q.k / 256 * 144;
        const int esz = q.qt == 0 ? 2 : 1;
        const cuuint64_t wd[2] = {static_cast<cuuint64_t>(row_bytes / esz), static_cast<cuuint64_t>(q.n)};
        const cuuint64_t ws_[1] = {static_cast<cuuint64_t>(row_bytes)};
        const cuuint32_t wb[2] = {static_cast<cuuint32_t>((q.qt == 0 ? 272 : 144) / esz), static_cast<cuuint32_t>(kBM)};
        if (encode(&tmap_w, q.qt == 0 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                   const_cast<void*>(q.w), wd, ws_, wb, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }

    const int64_t count8 = q.m * q.k / 8;
    cudaError_t e = launch_kernel(cast_bf16_kernel, dim3(static_cast<unsigned>(std::min<int64_t>(
                                                          (count8 + 255) / 256, int64_t{device_sm_count()} * 8))),
                                  dim3(256), 0, s, true, q.x, xb, count8);
    if (e != cudaSuccess) return e;

    PrefillParams p{};
    p.w = static_cast<const uint8_t*>(q.w);
    p.row_bytes = q.qt == 0 ? q.k / 32 * 34 : q.k / 256 * 144;
    p.n = q.n;
    p.m = q.m;
    p.k = q.k;
    p.units_per_split = sp.units_per_split;
    p.n_units = static_cast<int>(q.k / kUnitWeights);
    p.y = q.y;
    p.part = part;
    p.cluster = sp.cluster ? 1 : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(q.n / kBM), static_cast<unsigned>((q.m + kBN - 1) / kBN),
                       static_cast<unsigned>(sp.splits));
    cfg.blockDim = dim3(kThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 1;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = static_cast<unsigned>(sp.splits);
    cfg.attrs = attr;
    cfg.numAttrs = sp.cluster ? 2 : 1;
    if (q.qt == 0) {
        constexpr auto kern = prefill_gemm_kernel<0>;
        if ((e = ensure_smem_attr<kern>()) != cudaSuccess) return e;
        cfg.dynamicSmemBytes = PCfg<0>::smem;
        e = cudaLaunchKernelEx(&cfg, kern, tmap, tmap_w, p);
    } else {
        constexpr auto kern = prefill_gemm_kernel<1>;
        if ((e = ensure_smem_attr<kern>()) != cudaSuccess) return e;
        cfg.dynamicSmemBytes = PCfg<1>::smem;
        e = cudaLaunchKernelEx(&cfg, kern, tmap, tmap_w, p);
    }
    if (e != cudaSuccess || sp.splits == 1 || sp.cluster) return e;
    const int64_t count4 = q.m * q.n / 4;
    return launch_kernel(prefill_reduce_kernel,
                         dim3(static_cast<unsigned>(std::min<int64_t>((count4 + 255) / 256,
                                                                      int64_t{device_sm_count()} * 8))),
                         dim3(256), 0, s, true, reinterpret_cast<const float4*>(part), reinterpret_cast<float4*>(q.y),
                         count4, sp.splits);
}

}  // namespace phb
