// Decode attention at context depth: one token's query heads against an
// fp16 KV cache of L positions (Phobos README: `phobos-bench -d N`, decode
// with N tokens already in context; `phobos-kbench` `flash_fp16`, f16 K/V
// with an f32 online-softmax state; the `kv_check` example).
//
//   s_j = scale * q_h . k_j,   out_h = sum_j softmax(s)_j v_j
//
// with query head h reading KV head h / (n_q / n_kv). Split-KV ("flash
// decode") in two kernels:
//  1. Split pass, grid (KV head x group of at most 8 query heads, position
//     chunk). A producer thread streams the chunk's K and V rows through a
//     shared-memory ring with 3-D tensor copies (TMA) of one KV head's rows
//     (they are strided in the cache; small per-row copies measured far
//     below HBM speed). Consumer warps keep per-warp online-softmax states
//     (running maximum m, exp-sum l and o = sum_j e^(s_j - m) v_j per query
//     head), combined in warp order into the chunk's (m, l, o). Two score
//     paths:
//     - attn_tc_kernel (head_dim 64, 128): the scores of a 128-position
//       stage are a tcgen05 MMA (see the section below);
//     - attn_split_kernel (head_dim 256): 28-position stages, 8 lanes per
//       position, each lane a fixed set of 16-byte chunks of the key for
//       every query head of the CTA, on the CUDA cores.
//     The CTA's head count is a template argument, so the head loops unroll.
//  2. attn_merge_kernel, one CTA per query head: out = sum_c e^(m_c - M) o_c /
//     sum_c e^(m_c - M) l_c over the chunks c in order (M their maximum).
// Scores and maxima are held in base 2 (scale folded with log2 e), so every
// exponential is one exp2f.
// Every order is fixed, so repeated calls give identical bits. K and V are
// each read once from HBM (query-head groups beyond 8 re-read them from L2).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>

#include "phb_common.cuh"
#include "phb_internal.h"

namespace phb {

static __device__ int g_attn_err;

cudaError_t read_dev_err_attention(int* code) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_attn_err, sizeof(int));
    if (e != cudaSuccess) return e;
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_attn_err, &zero, sizeof(int));
    *code = v;
    return e;
}

namespace {

// CUDA-core score path (head_dim 256). 7 consumer warps + 1 producer warp:
// two CTAs (16 warps) per SM leave 128 registers a thread (register files
// are split between an SM's 4 schedulers), enough to keep the query values
// in registers.
constexpr int kCW = 7;                // consumer warps, 4 positions of each stage apiece
constexpr int kTileRows = 4 * kCW;    // positions per ring stage
constexpr int kNC = 32 * kCW;
constexpr int kThreads = kNC + 32;    // + one producer warp
constexpr int kMaxHeads = 8;          // query heads per CTA
constexpr int kMaxStages = 8;
constexpr int kWarpFloats = 80;       // per consumer warp: (p, p) pairs [4][8], alpha [8], spare [8]

struct AttnParams {
    const float* q;
    float* o_part;   // [nsplit][n_q][hd]: chunk outputs, unnormalised, relative to the chunk maximum
    float* ml_part;  // [nsplit][n_q][2]: chunk maximum and exp-sum
    int64_t len;
    int n_q, n_kv, group, hgroups, chunk, ns;
    float scale;     // the caller's scale times log2(e)
    uint32_t stage_bytes, q_off, warp_off, bar_off;
};

// One box of the [n_ctx][n_kv][head_dim] cache at (element x, KV head y,
// position z): the map's box width x 1 KV head x its positions, landing as
// packed rows (swizzled when the map says so).
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
        "%3, %4}], [%5], %6;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

template <int N>
__device__ __forceinline__ void named_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ float2 h2f(uint32_t w) {
    __half2 h;
    memcpy(&h, &w, 4);
    return __half22float2(h);
}

// Sum of the GP per-head partials over the 8 lanes of a position (lane
// bits 2, 1, 0) as a reduce-scatter: each step hands half the heads to the
// partner lane, so a lane ends with the full sum of head `head` (held by
// 8 / GP lanes).
template <int N, int B>
__device__ __forceinline__ float head_reduce(float* w, int lane, int& head) {
    if constexpr (N > 1) {
        const bool up = (lane & B) != 0;
#pragma unroll
        for (int k = 0; k < N / 2; ++k) {
            const float send = up ? w[k] : w[k + N / 2];
            const float keep = up ? w[k + N / 2] : w[k];
            w[k] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, B);
        }
        if (up) head += N / 2;
        if constexpr (B > 1) return head_reduce<N / 2, B / 2>(w, lane, head);
        return w[0];
    } else {
        w[0] += __shfl_xor_sync(0xFFFFFFFFu, w[0], B);
        if constexpr (B > 1) return head_reduce<1, B / 2>(w, lane, head);
        return w[0];
    }
}

// Shared memory: ring [ns][K rows kTileRows | V rows kTileRows][head_dim] | q | per-warp
// p/alpha | per-warp (m, l) | mbarriers.
// GP: query heads per CTA rounded up to a power of two (heads past the CTA's
// count are idle); E = head_dim / 32.
template <int GP, int E>
__global__ void __launch_bounds__(kThreads, 2)
    attn_split_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                      const __grid_constant__ AttnParams p) {
    constexpr int HD = 32 * E;
    constexpr int NCH = HD / 8;                // 16-byte chunks of a K row
    constexpr int CPL = NCH / 8;               // chunks per lane in the score pass
    constexpr bool kQReg = GP * E <= 16;       // query values in registers (else shared memory): <= 64 a thread
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int kv = blockIdx.x / p.hgroups, hg = blockIdx.x - kv * p.hgroups;
    const int h0 = kv * p.group + hg * kMaxHeads;              // first query head of this CTA
    const int gh = min(kMaxHeads, p.group - hg * kMaxHeads);   // its query heads (<= GP)
    const int split = blockIdx.y;
    const int64_t pos0 = static_cast<int64_t>(split) * p.chunk;
    const int np = static_cast<int>(min(static_cast<int64_t>(p.chunk), p.len - pos0));
    const int ntiles = (np + kTileRows - 1) / kTileRows;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.bar_off);
    uint64_t* empty = full + kMaxStages;
    if (tid == 0) {
        for (int s = 0; s < p.ns; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kCW);
        }
        fence_barrier_init();
    }
    __syncthreads();
    pdl_launch_dependents();
    pdl_wait();  // the query and the cache may come from the kernels before this one

    if (warp == kCW) {
        // ---------------- producer: one tensor copy for K and one for V per stage
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            constexpr uint32_t kRowBytes = 2 * HD;
            int issued = 0;
            for (int t = 0, slot = 0, phase = 0; t < ntiles; ++t) {
                if (t >= p.ns && !mbar_wait(&empty[slot], phase ^ 1, &g_attn_err)) break;
                // a box past n_ctx is zero-filled and still counts its full size
                mbar_arrive_expect_tx(&full[slot], 2 * kTileRows * kRowBytes);
                uint8_t* st = smem + static_cast<size_t>(slot) * p.stage_bytes;
                const int y0 = static_cast<int>(pos0) + t * kTileRows;
                tma_load_3d(st, &tmap_k, 0, kv, y0, &full[slot], pol);
                tma_load_3d(st + kTileRows * kRowBytes, &tmap_v, 0, kv, y0, &full[slot], pol);
                ++issued;
                if (++slot == p.ns) {
                    slot = 0;
                    phase ^= 1;
                }
            }
            // copies still in flight land before the CTA may exit (bounded; long done on the normal path)
            for (int t = max(0, issued - p.ns); t < issued; ++t)
                mbar_wait(&full[t % p.ns], (t / p.ns) & 1, &g_attn_err);
        }
        return;
    }

    // ---------------- consumers
    // Score pass: 8 lanes per position, 4 positions per warp. Lane u = lane & 7
    // takes the 16-byte chunks u, u + 8, ... of the key row for every query
    // head, so a quarter-warp reads 128 contiguous bytes and each K element is
    // converted once.
    const int jl = lane >> 3, u = lane & 7;
    float2 qr[kQReg ? GP : 1][kQReg ? CPL : 1][4];  // pairs, as the packed FMA takes them
    float* qsm = reinterpret_cast<float*>(smem + p.q_off);  // [GP][2][NCH][4]: chunk halves, chunk-major
    if constexpr (kQReg) {
#pragma unroll
        for (int h = 0; h < GP; ++h)
#pragma unroll
            for (int i = 0; i < CPL; ++i)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float* src = p.q + static_cast<int64_t>(h0 + h) * HD + (u + 8 * i) * 8 + 2 * e;
                    qr[h][i][e] = h < gh ? make_float2(src[0], src[1]) : make_float2(0.f, 0.f);
                }
    } else {
        for (int i = tid; i < GP * HD; i += kNC) {
            const int h = i / HD, d = i - h * HD, c = d >> 3, e = d & 7;
            qsm[((h * 2 + (e >> 2)) * NCH + c) * 4 + (e & 3)] = h < gh ? p.q[static_cast<int64_t>(h0 + h) * HD + d] : 0.f;
        }
        named_sync<kNC>();
    }

    float2* pw = reinterpret_cast<float2*>(smem + p.warp_off) + warp * (kWarpFloats / 2);  // (p, p) [4 pos][8 heads]
    float* aw = reinterpret_cast<float*>(pw + 32);                                         // alpha [8 heads]
    float m_run = -INFINITY, l_run = 0.f;  // of head hl, below
    int hl = 0;
    float2 acc[GP][E / 2];
#pragma unroll
    for (int h = 0; h < GP; ++h)
#pragma unroll
        for (int e = 0; e < E / 2; ++e) acc[h][e] = make_float2(0.f, 0.f);

    for (int t = 0, slot = 0, phase = 0; t < ntiles; ++t) {
        if (!mbar_wait_warp(&full[slot], phase, &g_attn_err)) break;
        const uint8_t* st = smem + static_cast<size_t>(slot) * p.stage_bytes;
        const int rows = min(kTileRows, np - t * kTileRows);

        // scores of this warp's 4 positions
        const int j = warp * 4 + jl;
        float2 a2[GP];
#pragma unroll
        for (int h = 0; h < GP; ++h) a2[h] = make_float2(0.f, 0.f);
        if (j < rows) {
            const uint8_t* kr = st + j * (2 * HD) + u * 16;
#pragma unroll
            for (int i = 0; i < CPL; ++i) {
                const uint4 raw = *reinterpret_cast<const uint4*>(kr + i * 128);
                const float2 k0 = h2f(raw.x), k1 = h2f(raw.y), k2 = h2f(raw.z), k3 = h2f(raw.w);
#pragma unroll
                for (int h = 0; h < GP; ++h) {
                    float2 q0, q1, q2, q3;
                    if constexpr (kQReg) {
                        q0 = qr[h][i][0];
                        q1 = qr[h][i][1];
                        q2 = qr[h][i][2];
                        q3 = qr[h][i][3];
                    } else {
                        const float4 qa = *reinterpret_cast<const float4*>(qsm + ((h * 2) * NCH + u + 8 * i) * 4);
                        const float4 qb = *reinterpret_cast<const float4*>(qsm + ((h * 2 + 1) * NCH + u + 8 * i) * 4);
                        q0 = make_float2(qa.x, qa.y);
                        q1 = make_float2(qa.z, qa.w);
                        q2 = make_float2(qb.x, qb.y);
                        q3 = make_float2(qb.z, qb.w);
                    }
                    a2[h] = __ffma2_rn(q0, k0, a2[h]);
                    a2[h] = __ffma2_rn(q1, k1, a2[h]);
                    a2[h] = __ffma2_rn(q2, k2, a2[h]);
                    a2[h] = __ffma2_rn(q3, k3, a2[h]);
                }
            }
        }
        float d[GP];
#pragma unroll
        for (int h = 0; h < GP; ++h) d[h] = a2[h].x + a2[h].y;
        hl = 0;
        const float dot = head_reduce<GP, 4>(d, lane, hl);
        const float s = (j < rows && hl < gh) ? p.scale * dot : -INFINITY;

        // online softmax of head hl over the warp's positions (lane bits 3 and 4)
        float mt = fmaxf(s, __shfl_xor_sync(0xFFFFFFFFu, s, 8));
        mt = fmaxf(mt, __shfl_xor_sync(0xFFFFFFFFu, mt, 16));
        const float m_new = fmaxf(m_run, mt);
        const float alpha = m_new == -INFINITY ? 1.f : exp2f(m_run - m_new);
        const float pj = s == -INFINITY ? 0.f : exp2f(s - m_new);
        float ls = pj + __shfl_xor_sync(0xFFFFFFFFu, pj, 8);
        ls += __shfl_xor_sync(0xFFFFFFFFu, ls, 16);
        l_run = fmaf(l_run, alpha, ls);
        m_run = m_new;
        pw[jl * 8 + hl] = make_float2(pj, pj);
        if (jl == 0) aw[hl] = alpha;
        const bool rescale = __any_sync(0xFFFFFFFFu, alpha != 1.f);
        __syncwarp();

        // values: lane owns elements [E*lane, E*lane + E) of every row; the
        // accumulators move only when some head's maximum moved
        if (rescale) {
#pragma unroll
            for (int h = 0; h < GP; ++h) {
                const float a = aw[h];
#pragma unroll
                for (int e = 0; e < E / 2; ++e) acc[h][e] = make_float2(acc[h][e].x * a, acc[h][e].y * a);
            }
        }
        const uint8_t* vbase = st + kTileRows * (2 * HD) + lane * (2 * E);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            if (warp * 4 + r < rows) {
                const uint8_t* vr = vbase + (warp * 4 + r) * (2 * HD);
                float2 vv[E / 2];
                if constexpr (E == 2) {
                    vv[0] = h2f(*reinterpret_cast<const uint32_t*>(vr));
                } else if constexpr (E == 4) {
                    const uint2 w = *reinterpret_cast<const uint2*>(vr);
                    vv[0] = h2f(w.x);
                    vv[1] = h2f(w.y);
                } else {
                    const uint4 w = *reinterpret_cast<const uint4*>(vr);
                    vv[0] = h2f(w.x);
                    vv[1] = h2f(w.y);
                    vv[2] = h2f(w.z);
                    vv[3] = h2f(w.w);
                }
                float2 ph[GP];
                if constexpr (GP >= 2) {
#pragma unroll
                    for (int h = 0; h < GP; h += 2) {
                        const float4 p4 = *reinterpret_cast<const float4*>(pw + r * 8 + h);
                        ph[h] = make_float2(p4.x, p4.y);
                        ph[h + 1] = make_float2(p4.z, p4.w);
                    }
                } else {
                    ph[0] = pw[r * 8];
                }
#pragma unroll
                for (int h = 0; h < GP; ++h)
#pragma unroll
                    for (int e = 0; e < E / 2; ++e) acc[h][e] = __ffma2_rn(ph[h], vv[e], acc[h][e]);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
        if (++slot == p.ns) {
            slot = 0;
            phase ^= 1;
        }
    }

    // ---------------- combine the warps' states, in warp order
    named_sync<kNC>();  // every warp is done with the ring; it now holds the warps' scaled outputs
    float* wml = reinterpret_cast<float*>(smem + p.warp_off) + kCW * kWarpFloats;  // [warp][8 heads][m, l]
    if (jl == 0) {
        wml[(warp * kMaxHeads + hl) * 2] = m_run;
        wml[(warp * kMaxHeads + hl) * 2 + 1] = l_run;
    }
    named_sync<kNC>();
    float* red = reinterpret_cast<float*>(smem);  // [warp][gh][HD]
#pragma unroll
    for (int h = 0; h < GP; ++h) {
        if (h < gh) {
            float mx = -INFINITY;
            for (int w = 0; w < kCW; ++w) mx = fmaxf(mx, wml[(w * kMaxHeads + h) * 2]);
            const float mw = wml[(warp * kMaxHeads + h) * 2];
            const float f = mw == -INFINITY ? 0.f : exp2f(mw - mx);
            float* dst = red + (warp * gh + h) * HD + lane * E;
#pragma unroll
            for (int e = 0; e < E / 2; ++e) {
                dst[2 * e] = f * acc[h][e].x;
                dst[2 * e + 1] = f * acc[h][e].y;
            }
        }
    }
    named_sync<kNC>();
    const int64_t obase = (static_cast<int64_t>(split) * p.n_q + h0) * HD;
    for (int i = tid; i < gh * HD; i += kNC) {
        float sum = 0.f;
        for (int w = 0; w < kCW; ++w) sum += red[w * gh * HD + i];
        p.o_part[obase + i] = sum;
    }
    if (tid < gh) {
        float mx = -INFINITY;
        for (int w = 0; w < kCW; ++w) mx = fmaxf(mx, wml[(w * kMaxHeads + tid) * 2]);
        float l = 0.f;
        for (int w = 0; w < kCW; ++w) {
            const float mw = wml[(w * kMaxHeads + tid) * 2];
            const float f = mw == -INFINITY ? 0.f : exp2f(mw - mx);
            l = fmaf(f, wml[(w * kMaxHeads + tid) * 2 + 1], l);
        }
        float* ml = p.ml_part + (static_cast<int64_t>(split) * p.n_q + h0 + tid) * 2;
        ml[0] = mx;
        ml[1] = l;
    }
}

// One CTA of 256 threads per query head. The chunk weights w_c = 2^(m_c - M)
// and the exp-sums l_c go to shared memory in parallel; thread (d, part)
// sums w_c o_c[d] over the chunks c = part, part + parts, ... (loads unrolled,
// so they overlap), and the parts and l are added in a fixed order.
constexpr int kMergeThreads = 256;

__global__ void __launch_bounds__(kMergeThreads) attn_merge_kernel(const float* __restrict__ o_part,
                                                                   const float* __restrict__ ml_part,
                                                                   float* __restrict__ out, int n_q, int hd,
                                                                   int nsplit) {
    extern __shared__ float msm[];  // w [nsplit] | l [nsplit] | partial sums [256] | warp maxima [8]
    float* w = msm;
    float* lc = w + nsplit;
    float* part_sum = lc + nsplit;
    float* wmax = part_sum + kMergeThreads;
    pdl_launch_dependents();
    pdl_wait();
    const int h = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    float mx = -INFINITY;
    for (int c = tid; c < nsplit; c += kMergeThreads) {
        const float2 ml = *reinterpret_cast<const float2*>(ml_part + (static_cast<int64_t>(c) * n_q + h) * 2);
        w[c] = ml.x;
        lc[c] = ml.y;
        mx = fmaxf(mx, ml.x);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
    if (lane == 0) wmax[warp] = mx;
    __syncthreads();
    mx = wmax[0];
#pragma unroll
    for (int i = 1; i < kMergeThreads / 32; ++i) mx = fmaxf(mx, wmax[i]);
    for (int c = tid; c < nsplit; c += kMergeThreads) w[c] = exp2f(w[c] - mx);
    __syncthreads();
    const int parts = kMergeThreads / hd;  // hd divides 256
    const int d = tid % hd, pt = tid / hd;
    const float* src = o_part + static_cast<int64_t>(h) * hd + d;
    const int64_t cstride = static_cast<int64_t>(n_q) * hd;
    float acc = 0.f;
    int c = pt;
    for (; c + 7 * parts < nsplit; c += 8 * parts) {
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = src[(c + u * parts) * cstride];
#pragma unroll
        for (int u = 0; u < 8; ++u) acc = fmaf(w[c + u * parts], v[u], acc);
    }
    for (; c < nsplit; c += parts) acc = fmaf(w[c], src[c * cstride], acc);
    part_sum[tid] = acc;
    __syncthreads();
    if (pt == 0) {
        float sum = part_sum[d];
        for (int q = 1; q < parts; ++q) sum += part_sum[q * hd + d];
        float l = 0.f;
        for (int k = 0; k < nsplit; ++k) l = fmaf(w[k], lc[k], l);
        out[static_cast<int64_t>(h) * hd + d] = sum / l;
    }
}

// ---------------------------------------------------------------- tensor-core score path (head_dim 64, 128)
// The scores of a 128-position stage are one tcgen05 MMA chain:
//   S^T [128 positions][16] = K [128][head_dim] . B^T,
// with B's 16 rows the CTA's (up to) 8 query heads split into fp16 high and
// low parts (rows h and 8 + h). Each head's query is first scaled by a power
// of two 2^e_h that brings its largest magnitude into [2^14, 2^15), so
// q 2^e_h = hi + lo to about 2^-22 relative (the scaling is exact and is
// undone with the score scale). K is fp16 and enters the MMA unconverted;
// products are exact and summed in fp32. Two warpgroups of 4 consumer warps
// take alternate stages: each warp reads its 32 positions' scores from TMEM
// (one thread per position, all heads in registers), keeps a per-warp
// online softmax, and accumulates the value rows on the CUDA cores as the
// other kernel does. The accumulator has two 16-column TMEM buffers, so the
// MMA of stage t + 1 runs while stage t is consumed.
constexpr int kTcRows = 128;                   // positions per stage (MMA M)
constexpr int kTcCW = 8;                       // consumer warps
constexpr int kTcTmaWarp = kTcCW;
constexpr int kTcMmaWarp = kTcCW + 1;
constexpr int kTcThreads = 32 * (kTcCW + 2);
constexpr uint32_t kTcTmemCols = 32;           // two 16-column score buffers
constexpr int kTcMaxStages = 6;
constexpr uint32_t kTcKBlock = kTcRows * 128;  // one 64-dim block of a K stage, 128-byte swizzled rows
constexpr uint32_t kTcQBlock = 16 * 128;       // one 64-dim block of the 16 query rows
// kind::f16: D fp32, A and B fp16, both K-major, N = 16, M = 128
constexpr uint32_t kTcIdesc = (1u << 4) | (uint32_t(16 >> 3) << 17) | (uint32_t(kTcRows >> 4) << 24);

struct TcParams {
    const float* q;
    float* o_part;
    float* ml_part;
    int64_t len;
    int n_q, n_kv, group, hgroups, chunk, ns;
    float scale;  // the caller's scale times log2(e)
    uint32_t stage_bytes, qb_off, pbuf_off, warp_off, bar_off;
};

__device__ __forceinline__ uint64_t desc_sw128(const void* ptr) {
    // K-major operand in the 128-byte swizzle layout: 8-row groups of
    // 128-byte rows, 1024 bytes apart (stride byte offset); version 1.
    const uint64_t addr = smem_addr(ptr);
    return ((addr & 0x3FFFFull) >> 4) | (1ull << 16) | ((1024ull >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

__device__ __forceinline__ void tc_mma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(kTcIdesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

// 16 consecutive TMEM columns of this warp's 32 lanes, one lane per thread.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ uint32_t pack_half2(__half a, __half b) {
    return static_cast<uint32_t>(__half_as_ushort(a)) | (static_cast<uint32_t>(__half_as_ushort(b)) << 16);
}

// Shared memory (1024-byte aligned base): ring [ns][K blocks | V rows] |
// query operand [HD/64][16 rows][128 B] | per-warp (p, p) [8][32 pos][8 heads]
// | per-warp (m, l) [8][8][2], head scales [8] | mbarriers, TMEM address.
template <int GP, int HD>
__global__ void __launch_bounds__(kTcThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                   const __grid_constant__ TcParams p) {
    constexpr int E = HD / 32;
    constexpr int KB = HD / 64;
    constexpr uint32_t kVOff = KB * kTcKBlock;
    extern __shared__ uint8_t tc_smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~uintptr_t{1023});
    uint8_t* qb = smem + p.qb_off;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.bar_off);
    uint64_t* empty = full + kTcMaxStages;
    uint64_t* sfull = empty + kTcMaxStages;
    uint64_t* sfree = sfull + 2;
    uint64_t* qready = sfree + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(qready + 1);
    float* wml = reinterpret_cast<float*>(smem + p.warp_off);  // [warp][8 heads][m, l]
    float* hscale = wml + kTcCW * kMaxHeads * 2;              // [8]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int kv = blockIdx.x / p.hgroups, hg = blockIdx.x - kv * p.hgroups;
    const int h0 = kv * p.group + hg * kMaxHeads;
    const int gh = min(kMaxHeads, p.group - hg * kMaxHeads);
    const int split = blockIdx.y;
    const int64_t pos0 = static_cast<int64_t>(split) * p.chunk;
    const int np = static_cast<int>(min(static_cast<int64_t>(p.chunk), p.len - pos0));
    const int ntiles = (np + kTcRows - 1) / kTcRows;

    if (tid == 0) {
        for (int s = 0; s < p.ns; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 4);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sfull[b], 1);
            mbar_init(&sfree[b], 4);
        }
        mbar_init(qready, kTcCW);
        fence_barrier_init();
    }
    if (warp == kTcMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(kTcTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_before();
    __syncthreads();
    tc_after();
    const uint32_t tmem = *tmem_slot;
    pdl_launch_dependents();
    pdl_wait();  // the query and the cache may come from the kernels before this one

    if (warp == kTcTmaWarp) {
        // ---------------- producer: per stage hd/64 swizzled K boxes and one V box
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            int issued = 0;
            for (int t = 0, slot = 0, phase = 0; t < ntiles; ++t) {
                if (t >= p.ns && !mbar_wait(&empty[slot], phase ^ 1, &g_attn_err)) break;
                // boxes past n_ctx are zero-filled and still count their full size
                mbar_arrive_expect_tx(&full[slot], kVOff + kTcRows * HD * 2);
                uint8_t* st = smem + static_cast<size_t>(slot) * p.stage_bytes;
                const int y0 = static_cast<int>(pos0) + t * kTcRows;
#pragma unroll
                for (int c = 0; c < KB; ++c) tma_load_3d(st + c * kTcKBlock, &tmap_k, 64 * c, kv, y0, &full[slot], pol);
                tma_load_3d(st + kVOff, &tmap_v, 0, kv, y0, &full[slot], pol);
                ++issued;
                if (++slot == p.ns) {
                    slot = 0;
                    phase ^= 1;
                }
            }
            for (int t = max(0, issued - p.ns); t < issued; ++t)
                mbar_wait(&full[t % p.ns], (t / p.ns) & 1, &g_attn_err);
        }
    } else if (warp == kTcMmaWarp) {
        // ---------------- one thread issues the score MMAs
        if (lane == 0) {
            int issued = 0;
            if (mbar_wait(qready, 0, &g_attn_err)) {
                for (int t = 0, slot = 0, phase = 0; t < ntiles; ++t) {
                    const int b = t & 1;
                    if (!mbar_wait(&full[slot], phase, &g_attn_err)) break;
                    if (t >= 2 && !mbar_wait(&sfree[b], ((t >> 1) - 1) & 1, &g_attn_err)) break;
                    tc_after();
                    const uint8_t* st = smem + static_cast<size_t>(slot) * p.stage_bytes;
#pragma unroll
                    for (int c = 0; c < KB; ++c)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            tc_mma_f16(tmem + 16 * b, desc_sw128(st + c * kTcKBlock + kk * 32),
                                       desc_sw128(qb + c * kTcQBlock + kk * 32), (c | kk) ? 1u : 0u);
                    tc_commit(&sfull[b]);
                    ++issued;
                    if (++slot == p.ns) {
                        slot = 0;
                        phase ^= 1;
                    }
                }
            }
            // every MMA issued has completed before TMEM is released (bounded; long done on the normal path)
            for (int t = max(0, issued - 2); t < issued; ++t) mbar_wait(&sfull[t & 1], (t >> 1) & 1, &g_attn_err);
        }
    } else {
        // ---------------- consumers
        // query operand: warp w writes rows w (high part) and 8 + w (low part)
        {
            const int h = warp;
            float qv[E];
            float mx = 0.f;
#pragma unroll
            for (int i = 0; i < E; ++i) {
                qv[i] = h < gh ? p.q[static_cast<int64_t>(h0 + h) * HD + E * lane + i] : 0.f;
                mx = fmaxf(mx, fabsf(qv[i]));
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
            int ex = 0;
            frexpf(mx, &ex);
            const int e = mx > 0.f ? 15 - ex : 0;
            if (lane == 0) hscale[h] = ldexpf(p.scale, -e);
            __half hi[E], lo[E];
#pragma unroll
            for (int i = 0; i < E; ++i) {
                const float qs = ldexpf(qv[i], e);
                hi[i] = __float2half_rn(qs);
                lo[i] = __float2half_rn(qs - __half2float(hi[i]));
            }
            const int d0 = E * lane, blk = d0 >> 6, ch = (d0 & 63) >> 3, byte = (d0 & 7) * 2;
#pragma unroll
            for (int part = 0; part < 2; ++part) {
                const int r = h + 8 * part;
                uint8_t* dst = qb + blk * kTcQBlock + r * 128 + ((ch ^ (r & 7)) << 4) + byte;
                const __half* src = part == 0 ? hi : lo;
                if constexpr (E == 2) {
                    *reinterpret_cast<uint32_t*>(dst) = pack_half2(src[0], src[1]);
                } else {
                    *reinterpret_cast<uint2*>(dst) = make_uint2(pack_half2(src[0], src[1]), pack_half2(src[2], src[3]));
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(qready);
        }
        named_sync<32 * kTcCW>();  // head scales visible to every consumer

        const int g = warp >> 2, wq = warp & 3;
        float2* pb = reinterpret_cast<float2*>(smem + p.pbuf_off) + warp * (32 * kMaxHeads);  // (p, p) [32][8]
        float hs[GP];
#pragma unroll
        for (int h = 0; h < GP; ++h) hs[h] = hscale[h];
        float m_run[GP], l_lane[GP];
        float2 acc[GP][E / 2];
#pragma unroll
        for (int h = 0; h < GP; ++h) {
            m_run[h] = -INFINITY;
            l_lane[h] = 0.f;
#pragma unroll
            for (int e = 0; e < E / 2; ++e) acc[h][e] = make_float2(0.f, 0.f);
        }
        for (int t = g; t < ntiles; t += 2) {
            const int slot = t % p.ns, b = t & 1;
            if (!mbar_wait_warp(&sfull[b], (t >> 1) & 1, &g_attn_err)) break;
            tc_after();
            __syncwarp();  // the TMEM load is warp-collective
            float sv[16];
            tmem_ld16(tmem + (static_cast<uint32_t>(32 * wq) << 16) + 16 * b, sv);
            tc_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sfree[b]);
            const int rows = min(kTcRows, np - t * kTcRows);
            const bool valid = 32 * wq + lane < rows;
            bool moved = false;
            float alpha[GP];
#pragma unroll
            for (int h = 0; h < GP; ++h) {
                const float s = (valid && h < gh) ? (sv[h] + sv[8 + h]) * hs[h] : -INFINITY;
                float mt = s;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xFFFFFFFFu, mt, o));
                const float m_new = fmaxf(m_run[h], mt);
                alpha[h] = m_new == -INFINITY ? 1.f : exp2f(m_run[h] - m_new);
                const float pj = s == -INFINITY ? 0.f : exp2f(s - m_new);
                l_lane[h] = fmaf(l_lane[h], alpha[h], pj);
                m_run[h] = m_new;
                moved |= alpha[h] != 1.f;
                pb[lane * kMaxHeads + h] = make_float2(pj, pj);
            }
            __syncwarp();
            if (moved) {  // uniform over the warp: the maxima are
#pragma unroll
                for (int h = 0; h < GP; ++h)
#pragma unroll
                    for (int e = 0; e < E / 2; ++e)
                        acc[h][e] = make_float2(acc[h][e].x * alpha[h], acc[h][e].y * alpha[h]);
            }
            // value rows of this warp's 32 positions (the stage's copies have landed: observe it)
            if (!mbar_wait_warp(&full[slot], (t / p.ns) & 1, &g_attn_err)) break;
            const uint8_t* vb = smem + static_cast<size_t>(slot) * p.stage_bytes + kVOff +
                                static_cast<size_t>(32 * wq) * (2 * HD) + lane * (2 * E);
            auto value_row = [&](int r) {
                const uint8_t* vr = vb + r * (2 * HD);
                float2 vv[E / 2];
                if constexpr (E == 2) {
                    vv[0] = h2f(*reinterpret_cast<const uint32_t*>(vr));
                } else {
                    const uint2 w = *reinterpret_cast<const uint2*>(vr);
                    vv[0] = h2f(w.x);
                    vv[1] = h2f(w.y);
                }
                float2 ph[GP];
                if constexpr (GP >= 2) {
#pragma unroll
                    for (int h = 0; h < GP; h += 2) {
                        const float4 p4 = *reinterpret_cast<const float4*>(pb + r * kMaxHeads + h);
                        ph[h] = make_float2(p4.x, p4.y);
                        ph[h + 1] = make_float2(p4.z, p4.w);
                    }
                } else {
                    ph[0] = pb[r * kMaxHeads];
                }
#pragma unroll
                for (int h = 0; h < GP; ++h)
#pragma unroll
                    for (int e = 0; e < E / 2; ++e) acc[h][e] = __ffma2_rn(ph[h], vv[e], acc[h][e]);
            };
            const int nrow = min(32, rows - 32 * wq);
            if (nrow == 32) {
                // a full stage: unrolled, so several rows' loads are in flight at once
#pragma unroll 8
                for (int r = 0; r < 32; ++r) value_row(r);
            } else {
                for (int r = 0; r < nrow; ++r) value_row(r);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
        }

        // ---------------- combine the 8 warps' states, in warp order
#pragma unroll
        for (int h = 0; h < GP; ++h)
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) l_lane[h] += __shfl_xor_sync(0xFFFFFFFFu, l_lane[h], o);
        if (lane == 0) {
#pragma unroll
            for (int h = 0; h < GP; ++h) {
                wml[(warp * kMaxHeads + h) * 2] = m_run[h];
                wml[(warp * kMaxHeads + h) * 2 + 1] = l_lane[h];
            }
        }
        named_sync<32 * kTcCW>();  // every stage consumed: the ring now holds the warps' scaled outputs
        float* red = reinterpret_cast<float*>(smem);  // [warp][gh][HD]
#pragma unroll
        for (int h = 0; h < GP; ++h) {
            if (h < gh) {
                float mx = -INFINITY;
                for (int w = 0; w < kTcCW; ++w) mx = fmaxf(mx, wml[(w * kMaxHeads + h) * 2]);
                const float mw = wml[(warp * kMaxHeads + h) * 2];
                const float f = mw == -INFINITY ? 0.f : exp2f(mw - mx);
                float* dst = red + (warp * gh + h) * HD + lane * E;
#pragma unroll
                for (int e = 0; e < E / 2; ++e) {
                    dst[2 * e] = f * acc[h][e].x;
                    dst[2 * e + 1] = f * acc[h][e].y;
                }
            }
        }
        named_sync<32 * kTcCW>();
        const int64_t obase = (static_cast<int64_t>(split) * p.n_q + h0) * HD;
        for (int i = tid; i < gh * HD; i += 32 * kTcCW) {
            float sum = 0.f;
            for (int w = 0; w < kTcCW; ++w) sum += red[w * gh * HD + i];
            p.o_part[obase + i] = sum;
        }
        if (tid < gh) {
            float mx = -INFINITY;
            for (int w = 0; w < kTcCW; ++w) mx = fmaxf(mx, wml[(w * kMaxHeads + tid) * 2]);
            float l = 0.f;
            for (int w = 0; w < kTcCW; ++w) {
                const float mw = wml[(w * kMaxHeads + tid) * 2];
                const float f = mw == -INFINITY ? 0.f : exp2f(mw - mx);
                l = fmaf(f, wml[(w * kMaxHeads + tid) * 2 + 1], l);
            }
            float* ml = p.ml_part + (static_cast<int64_t>(split) * p.n_q + h0 + tid) * 2;
            ml[0] = mx;
            ml[1] = l;
        }
    }
    tc_before();
    __syncthreads();
    if (warp == kTcMmaWarp) {
        __syncwarp();
        tc_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTcTmemCols) : "memory");
    }
}

struct AttnPlan {
    bool tc = false;  // tensor-core score kernel (head_dim 64, 128) or the CUDA-core one (256)
    int hgroups = 1, chunk = 0, nsplit = 0, ns = 0;
    uint32_t stage_bytes = 0, q_off = 0, warp_off = 0, bar_off = 0, pbuf_off = 0;
    size_t smem = 0;
};

AttnPlan plan_attn(int n_q, int n_kv, int hd, int64_t len) {
    AttnPlan pl;
    pl.tc = hd <= 128;
    const int group = n_q / n_kv;
    pl.hgroups = (group + kMaxHeads - 1) / kMaxHeads;
    const int ctas = pl.tc ? 1 : 2;  // CTAs per SM
    const int rows = pl.tc ? kTcRows : kTileRows;
    const int64_t items = static_cast<int64_t>(n_kv) * pl.hgroups;
    const int64_t want = std::max<int64_t>(1, (static_cast<int64_t>(ctas) * device_sm_count() + items - 1) / items);
    int64_t chunk = (len + want - 1) / want;
    chunk = (chunk + rows - 1) / rows * rows;
    pl.chunk = static_cast<int>(chunk);
    pl.nsplit = static_cast<int>((len + chunk - 1) / chunk);
    if (pl.tc) {
        // ring of 128-position stages | query operand | (p, p) buffers | warp states | barriers
        pl.stage_bytes = static_cast<uint32_t>((hd / 64) * kTcKBlock + kTcRows * hd * 2);
        const size_t qb_bytes = static_cast<size_t>(hd / 64) * kTcQBlock;
        const size_t pbuf_bytes = static_cast<size_t>(kTcCW) * 32 * kMaxHeads * sizeof(float2);
        const size_t warp_bytes = 1024;  // (m, l) [8][8][2] and head scales [8]
        const size_t bar_bytes = 256;
        const size_t fixed = qb_bytes + pbuf_bytes + warp_bytes + bar_bytes;
        pl.ns = static_cast<int>(std::min<size_t>(kTcMaxStages, (kSmemOptin - 1024 - fixed) / pl.stage_bytes));
        pl.q_off = static_cast<uint32_t>(static_cast<size_t>(pl.ns) * pl.stage_bytes);
        pl.pbuf_off = static_cast<uint32_t>(pl.q_off + qb_bytes);
        pl.warp_off = static_cast<uint32_t>(pl.pbuf_off + pbuf_bytes);
        pl.bar_off = static_cast<uint32_t>(pl.warp_off + warp_bytes);
        pl.smem = pl.bar_off + bar_bytes + 1024;  // + alignment of the base to 1024 bytes
        return pl;
    }
    // shared memory: as many ring stages as fit two CTAs per SM (at most kMaxStages)
    pl.stage_bytes = static_cast<uint32_t>(4 * kTileRows * hd);  // K and V rows, packed (multiple of 128 bytes)
    const size_t q_bytes = static_cast<size_t>(kMaxHeads) * (hd + 4) * sizeof(float);
    const size_t warp_bytes = static_cast<size_t>(kCW) * (kWarpFloats + 2 * kMaxHeads) * sizeof(float);
    const size_t fixed = q_bytes + warp_bytes + 2 * kMaxStages * sizeof(uint64_t);
    const size_t budget = size_t{112} * 1024;
    pl.ns = static_cast<int>(std::min<size_t>(kMaxStages, (budget - fixed) / pl.stage_bytes));
    pl.q_off = static_cast<uint32_t>(static_cast<size_t>(pl.ns) * pl.stage_bytes);
    pl.warp_off = static_cast<uint32_t>(pl.q_off + q_bytes);
    pl.bar_off = static_cast<uint32_t>(pl.warp_off + warp_bytes);
    pl.smem = pl.bar_off + 2 * kMaxStages * sizeof(uint64_t);
    return pl;
}

struct AttnMaps {
    CUtensorMap k, v;
};

template <int GP, int E>
cudaError_t launch_split(const AttnPlan& pl, dim3 grid, const AttnMaps& m, const AttnParams& p, cudaStream_t s) {
    cudaError_t e = ensure_smem_attr<attn_split_kernel<GP, E>>();
    if (e != cudaSuccess) return e;
    return launch_kernel(attn_split_kernel<GP, E>, grid, dim3(kThreads), pl.smem, s, true, m.k, m.v, p);
}

template <int E>
cudaError_t launch_split_e(int gp, const AttnPlan& pl, dim3 grid, const AttnMaps& m, const AttnParams& p,
                           cudaStream_t s) {
    switch (gp) {
        case 1: return launch_split<1, E>(pl, grid, m, p, s);
        case 2: return launch_split<2, E>(pl, grid, m, p, s);
        case 4: return launch_split<4, E>(pl, grid, m, p, s);
        default: return launch_split<8, E>(pl, grid, m, p, s);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 attn_encode_fn() {
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

// The cache [n_ctx][n_kv][hd] fp16 as a 3-D tensor (hd innermost); a box is
// one KV head's hd values at kTileRows consecutive positions.
// `box_x` head_dim values (64 with the 128-byte swizzle the MMA operand
// layout needs, else head_dim) of `rows` positions.
bool encode_cache_map(CUtensorMap* map, const void* base, int n_kv, int hd, int64_t len, int box_x, int rows,
                      bool swizzle) {
    PFN_cuTensorMapEncodeTiled_v12000 encode = attn_encode_fn();
    if (encode == nullptr) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(hd), static_cast<cuuint64_t>(n_kv),
                                static_cast<cuuint64_t>(len)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(hd) * 2, static_cast<cuuint64_t>(n_kv) * hd * 2};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(box_x), 1, static_cast<cuuint32_t>(rows)};
    const cuuint32_t estr[3] = {1, 1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int GP, int HD>
cudaError_t launch_tc(const AttnPlan& pl, dim3 grid, const AttnMaps& m, const TcParams& p, cudaStream_t s) {
    cudaError_t e = ensure_smem_attr<attn_tc_kernel<GP, HD>>();
    if (e != cudaSuccess) return e;
    return launch_kernel(attn_tc_kernel<GP, HD>, grid, dim3(kTcThreads), pl.smem, s, true, m.k, m.v, p);
}

template <int HD>
cudaError_t launch_tc_hd(int gp, const AttnPlan& pl, dim3 grid, const AttnMaps& m, const TcParams& p,
                         cudaStream_t s) {
    switch (gp) {
        case 1: return launch_tc<1, HD>(pl, grid, m, p, s);
        case 2: return launch_tc<2, HD>(pl, grid, m, p, s);
        case 4: return launch_tc<4, HD>(pl, grid, m, p, s);
        default: return launch_tc<8, HD>(pl, grid, m, p, s);
    }
}

}  // namespace

bool attention_shape_ok(int n_q, int n_kv, int hd) {
    return n_q >= 1 && n_kv >= 1 && n_q % n_kv == 0 && (hd == 64 || hd == 128 || hd == 256);
}

size_t attention_ws_bytes(int n_q, int n_kv, int hd, int64_t len) {
    const AttnPlan pl = plan_attn(n_q, n_kv, hd, len);
    return static_cast<size_t>(pl.nsplit) * n_q * (hd + 2) * sizeof(float);
}

cudaError_t attention_run(const float* q, const void* k, const void* v, float* out, int n_q, int n_kv, int hd,
                          int64_t len, float scale, void* ws, cudaStream_t s) {
    const AttnPlan pl = plan_attn(n_q, n_kv, hd, len);
    // the ring doubles as the buffer of the warps' outputs at the end
    const int cw = pl.tc ? kTcCW : kCW;
    if (pl.ns < 2 || pl.smem > kSmemOptin ||
        static_cast<size_t>(pl.ns) * pl.stage_bytes < static_cast<size_t>(cw) * kMaxHeads * hd * 4)
        return cudaErrorInvalidConfiguration;
    AttnMaps maps;
    const int box_x = pl.tc ? 64 : hd, rows = pl.tc ? kTcRows : kTileRows;
    if (!encode_cache_map(&maps.k, k, n_kv, hd, len, box_x, rows, pl.tc) ||
        !encode_cache_map(&maps.v, v, n_kv, hd, len, hd, rows, false))
        return cudaErrorInvalidValue;
    float* o_part = static_cast<float*>(ws);
    float* ml_part = o_part + static_cast<size_t>(pl.nsplit) * n_q * hd;
    const int group = n_q / n_kv;
    // scores are kept in base 2: s2 = scale * log2(e) * q.k, so exp(s - m) = 2^(s2 - m2)
    const float scale2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    const dim3 grid(static_cast<unsigned>(n_kv * pl.hgroups), static_cast<unsigned>(pl.nsplit));
    const int g = std::min(group, kMaxHeads);
    const int gp = g <= 1 ? 1 : g <= 2 ? 2 : g <= 4 ? 4 : 8;
    cudaError_t e;
    if (pl.tc) {
        TcParams p;
        p.q = q;
        p.o_part = o_part;
        p.ml_part = ml_part;
        p.len = len;
        p.n_q = n_q;
        p.n_kv = n_kv;
        p.group = group;
        p.hgroups = pl.hgroups;
        p.chunk = pl.chunk;
        p.ns = pl.ns;
        p.scale = scale2;
        p.stage_bytes = pl.stage_bytes;
        p.qb_off = pl.q_off;
        p.pbuf_off = pl.pbuf_off;
        p.warp_off = pl.warp_off;
        p.bar_off = pl.bar_off;
        e = hd == 64 ? launch_tc_hd<64>(gp, pl, grid, maps, p, s) : launch_tc_hd<128>(gp, pl, grid, maps, p, s);
    } else {
        AttnParams p;
        p.q = q;
        p.o_part = o_part;
        p.ml_part = ml_part;
        p.len = len;
        p.n_q = n_q;
        p.n_kv = n_kv;
        p.group = group;
        p.hgroups = pl.hgroups;
        p.chunk = pl.chunk;
        p.ns = pl.ns;
        p.scale = scale2;
        p.stage_bytes = pl.stage_bytes;
        p.q_off = pl.q_off;
        p.warp_off = pl.warp_off;
        p.bar_off = pl.bar_off;
        e = launch_split_e<8>(gp, pl, grid, maps, p, s);
    }
    if (e != cudaSuccess) return e;
    const size_t msmem = (2 * static_cast<size_t>(pl.nsplit) + kMergeThreads + 8) * sizeof(float);
    return launch_kernel(attn_merge_kernel, dim3(static_cast<unsigned>(n_q)), dim3(kMergeThreads), msmem, s, true,
                         static_cast<const float*>(o_part), static_cast<const float*>(ml_part), out, n_q, hd,
                         pl.nsplit);
}

}  // namespace phb
