// router_common.cuh -- the sigmoid top-k selection of one token, shared by the
// router kernel and the fused layer kernel.
//
// "Day-0 Support for Flint on vLLM", section "Model architecture": sigmoid
// scores over the routed experts, top-k selection, weights renormalised over
// the selected k.
#pragma once

#include "flint_device.cuh"

namespace flint {
namespace {

// Sigmoid scores of T tokens x E experts (logits [T][E], plus bias[e] when
// given) into shared memory as their bit patterns, one score per thread at a
// time: sigmoid scores are positive floats, so the bits order like the
// values. Logits come from global memory (written by other CTAs: read past
// L1). Every thread of the CTA calls this; a __syncthreads must follow.
__device__ __forceinline__ uint32_t sigmoid_score(float z, const float* bias, int e) {
    if (bias) z = z + bias[e];
    return __float_as_uint(1.f / (1.f + expf(-z)));
}

__device__ __forceinline__ void sigmoid_scores(const float* logits, const float* bias, int T, int E,
                                               uint32_t* scores) {
    for (int i = threadIdx.x; i < T * E; i += blockDim.x) scores[i] = sigmoid_score(ld_cg(logits + i), bias, i % E);
}

// Top-k of one token's scores (shared memory; global memory written by other
// CTAs when L2 is set: read past L1), one warp: lane holds experts
// lane + 32 i. Each lane keeps its best untaken score; a round takes the warp
// maximum, breaks ties toward the lowest expert index with a warp minimum,
// and only the owning lane rescans its scores. Weights are the selected
// scores over their sum.
template <int SLOTS, bool L2 = false>
__device__ __forceinline__ void topk_warp(const uint32_t* sc, int E, int k, int lane, int32_t* ids,
                                          float* weights) {
    uint32_t s[SLOTS];
#pragma unroll
    for (int i = 0; i < SLOTS; ++i) {
        const int e = lane + 32 * i;
        s[i] = e >= E ? 0u : L2 ? (uint32_t)ld_cg(reinterpret_cast<const int32_t*>(sc) + e) : sc[e];
    }
    uint32_t valid = 0;  // bit i: slot i holds an untaken expert
#pragma unroll
    for (int i = 0; i < SLOTS; ++i)
        if (lane + 32 * i < E) valid |= 1u << i;
    auto head = [&](uint32_t& hv, int& hi) {  // best untaken slot, lowest index on ties
        hv = 0u;
        hi = SLOTS;
#pragma unroll
        for (int i = 0; i < SLOTS; ++i)
            if (((valid >> i) & 1u) && (hi == SLOTS || s[i] > hv)) {
                hv = s[i];
                hi = i;
            }
    };
    uint32_t hv;
    int hi;
    head(hv, hi);
    float sel_s = 0.f, sum = 0.f;
    int sel_e = 0;
    for (int j = 0; j < k; ++j) {
        const uint32_t best = __reduce_max_sync(0xffffffffu, hi < SLOTS ? hv : 0u);
        const uint32_t cand = (hi < SLOTS && hv == best) ? (uint32_t)(lane + 32 * hi) : 0xFFFFFFFFu;
        const uint32_t e = __reduce_min_sync(0xffffffffu, cand);
        if ((int)(e & 31u) == lane) {
            valid &= ~(1u << (e >> 5));
            head(hv, hi);
        }
        const float sv = __uint_as_float(best);
        sum += sv;
        if (lane == j) {
            sel_e = (int)e;
            sel_s = sv;
        }
    }
    if (lane < k) {
        ids[lane] = sel_e;
        weights[lane] = sel_s / sum;
    }
}

}  // namespace
}  // namespace flint
