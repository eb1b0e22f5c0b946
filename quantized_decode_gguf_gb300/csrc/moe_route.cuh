// Router of the top-k MoE FFN, shared by the expert-grouped passes and the
// one-token kernel: per token the top_k largest router logits (ties to the
// lower expert index) in descending order and their softmax.
#pragma once

#include <cstdint>

namespace phb {
namespace {

constexpr int kMaxExperts = 256;
constexpr int kMaxTopK = 8;

// Order-preserving map of a finite float to an unsigned key (larger float,
// larger key).
__device__ __forceinline__ uint32_t float_key(float v) {
    const uint32_t u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_float(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Top-k selection for one token by one warp, one expert per round: the
// logits are held as order-preserving keys, eight per lane (expert
// lane + 32 j); a round takes the largest untaken key, the lowest expert
// index among equal keys, by two warp reductions. All 32 lanes call every
// member and get the same results.
struct TopKWarp {
    uint32_t key[kMaxExperts / 32];
    uint32_t taken;

    __device__ __forceinline__ void load(const float* __restrict__ row, int E, int lane) {
#pragma unroll
        for (int j = 0; j < kMaxExperts / 32; ++j) {
            const int e = lane + 32 * j;
            key[j] = e < E ? float_key(row[e]) : 0u;
        }
        taken = 0;
    }

    // Next expert in descending logit order; its logit in *v.
    __device__ __forceinline__ int next(int E, int lane, float* v) {
        uint32_t bk = 0;
        int be = 0x7FFFFFFF;
#pragma unroll
        for (int j = 0; j < kMaxExperts / 32; ++j) {  // this lane's best untaken expert (ascending j)
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
        *v = key_float(kmax);
        return static_cast<int>(emin);
    }
};

// Softmax over the K selected logits v[0] >= v[1] >= ...: exp(v_r - v_0),
// summed in slot order, each divided by the sum.
__device__ __forceinline__ void topk_softmax(const float* v, int K, float* p) {
    float ex[kMaxTopK];
    float sum = 0.f;
#pragma unroll
    for (int r = 0; r < kMaxTopK; ++r) {
        if (r >= K) break;
        ex[r] = expf(v[r] - v[0]);
        sum += ex[r];
    }
#pragma unroll
    for (int r = 0; r < kMaxTopK; ++r) {
        if (r >= K) break;
        p[r] = ex[r] / sum;
    }
}

// Routing of one token by one warp (all 32 lanes call it): the top K in
// slot order in sel_e (every lane) and their softmax weights in p (lane 0).
__device__ __forceinline__ void route_token_warp(const float* __restrict__ row, int E, int K, int lane,
                                                 int (&sel_e)[kMaxTopK], float (&p)[kMaxTopK]) {
    TopKWarp tk;
    tk.load(row, E, lane);
    float sel_v[kMaxTopK];
#pragma unroll
    for (int r = 0; r < kMaxTopK; ++r) {
        if (r >= K) break;
        sel_e[r] = tk.next(E, lane, &sel_v[r]);
    }
    if (lane == 0) topk_softmax(sel_v, K, p);
}

}  // namespace
}  // namespace phb
