// Decode attention at context depth: one token's query heads against an
// fp16 KV cache of L positions (Phobos README: `phobos-bench -d N`, decode
// with N tokens already in context; `phobos-kbench` `flash_fp16`, f16 K/V
// with an f32 online-softmax state; the `kv_check` example).
//
//   s_j = scale * q_h . k_j,   out_h = sum_j softmax(s)_j v_j
//
// with query head h reading KV head h / (n_q / n_kv). Split-KV ("flash
// decode") in two kernels:
//  1. attn_split_kernel, grid (KV head x group of at most 8 query heads,
//     position chunk). A producer thread streams the chunk's K and V rows
//     through a ring of 28-position stages, one 3-D tensor copy (TMA) per
//     stage for K and one for V (the rows of one KV head are strided in the
//     cache; small per-row copies measured far below HBM speed);
//     each of 7 consumer warps owns 4 positions of every stage and keeps its
//     own online-softmax state (running maximum m, exp-sum l and
//     o = sum_j e^(s_j - m) v_j per query head). At the end the warps' states
//     are combined in warp order into the chunk's (m, l, o). Scores take 8
//     lanes per position, each lane a fixed set of 16-byte chunks of the key
//     for every query head of the CTA (the CTA's head count is a template
//     argument, so these loops unroll).
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

// 7 consumer warps + 1 producer warp: two CTAs (16 warps) per SM leave 128
// registers a thread (register files are split between an SM's 4
// schedulers), enough to keep the query values in registers.
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

// One box of the [n_ctx][n_kv][head_dim] cache: head_dim x 1 KV head x
// kTileRows positions, landing as kTileRows packed rows.
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

struct AttnPlan {
    int hgroups = 1, chunk = 0, nsplit = 0, ns = 0;
    uint32_t stage_bytes = 0, q_off = 0, warp_off = 0, bar_off = 0;
    size_t smem = 0;
};


AttnPlan plan_attn(int n_q, int n_kv, int hd, int64_t len) {
    AttnPlan pl;
    const int group = n_q / n_kv;
    pl.hgroups = (group + kMaxHeads - 1) / kMaxHeads;
    const int ctas = 2;  // CTAs per SM
    const int64_t items = static_cast<int64_t>(n_kv) * pl.hgroups;
    const int64_t want = std::max<int64_t>(1, (static_cast<int64_t>(ctas) * device_sm_count() + items - 1) / items);
    int64_t chunk = (len + want - 1) / want;
    chunk = (chunk + kTileRows - 1) / kTileRows * kTileRows;
    pl.chunk = static_cast<int>(chunk);
    pl.nsplit = static_cast<int>((len + chunk - 1) / chunk);
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
bool encode_cache_map(CUtensorMap* map, const void* base, int n_kv, int hd, int64_t len) {
    PFN_cuTensorMapEncodeTiled_v12000 encode = attn_encode_fn();
    if (encode == nullptr) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(hd), static_cast<cuuint64_t>(n_kv),
                                static_cast<cuuint64_t>(len)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(hd) * 2, static_cast<cuuint64_t>(n_kv) * hd * 2};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(hd), 1, static_cast<cuuint32_t>(kTileRows)};
    const cuuint32_t estr[3] = {1, 1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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
    if (pl.ns < 2 || static_cast<size_t>(pl.ns) * pl.stage_bytes < static_cast<size_t>(kCW) * kMaxHeads * hd * 4)
        return cudaErrorInvalidConfiguration;
    AttnMaps maps;
    if (!encode_cache_map(&maps.k, k, n_kv, hd, len) || !encode_cache_map(&maps.v, v, n_kv, hd, len))
        return cudaErrorInvalidValue;
    AttnParams p;
    p.q = q;
    p.o_part = static_cast<float*>(ws);
    p.ml_part = p.o_part + static_cast<size_t>(pl.nsplit) * n_q * hd;
    p.len = len;
    p.n_q = n_q;
    p.n_kv = n_kv;
    p.group = n_q / n_kv;
    p.hgroups = pl.hgroups;
    p.chunk = pl.chunk;
    p.ns = pl.ns;
    // scores are kept in base 2: s2 = scale * log2(e) * q.k, so exp(s - m) = 2^(s2 - m2)
    p.scale = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    p.stage_bytes = pl.stage_bytes;
    p.q_off = pl.q_off;
    p.warp_off = pl.warp_off;
    p.bar_off = pl.bar_off;
    const dim3 grid(static_cast<unsigned>(n_kv * pl.hgroups), static_cast<unsigned>(pl.nsplit));
    const int g = std::min(p.group, kMaxHeads);
    const int gp = g <= 1 ? 1 : g <= 2 ? 2 : g <= 4 ? 4 : 8;
    cudaError_t e = hd == 64    ? launch_split_e<2>(gp, pl, grid, maps, p, s)
                    : hd == 128 ? launch_split_e<4>(gp, pl, grid, maps, p, s)
                                : launch_split_e<8>(gp, pl, grid, maps, p, s);
    if (e != cudaSuccess) return e;
    const size_t msmem = (2 * static_cast<size_t>(pl.nsplit) + kMergeThreads + 8) * sizeof(float);
    return launch_kernel(attn_merge_kernel, dim3(static_cast<unsigned>(n_q)), dim3(kMergeThreads), msmem, s, true,
                         static_cast<const float*>(p.o_part), static_cast<const float*>(p.ml_part), out, n_q, hd,
                         pl.nsplit);
}

}  // namespace phb
