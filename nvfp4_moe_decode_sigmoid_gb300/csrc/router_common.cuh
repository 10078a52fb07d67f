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

// Top-k of one token's scores, one warp: lane holds the scores of experts
// lane + 32 i in s[i] (0 past E). Weights are the selected scores over their sum. Each round
// takes the warp maximum of the lanes' best untaken scores and breaks ties
// toward the lowest expert index with a warp minimum.
//   SLOTS == 8 (E <= 256): each lane first sorts its keys (score bits above,
//   255 - slot below, so that equal scores keep the lower expert first; 0 for
//   no expert) with Batcher's 19-comparator network, so that its best
//   untaken key is always key[0] and the owning lane of a round just shifts.
//   Otherwise the owning lane rescans its slots.
template <int SLOTS>
__device__ __forceinline__ void topk_warp_regs(const uint32_t (&s)[SLOTS], int E, int k, int lane, int32_t* ids,
                                               float* weights) {
    const uint32_t full = 0xffffffffu;
    float sel_s = 0.f, sum = 0.f;
    int sel_e = 0;
    if constexpr (SLOTS == 8) {
        unsigned long long key[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            key[i] = lane + 32 * i < E ? ((unsigned long long)s[i] << 32) | (unsigned long long)(255 - i) : 0ull;
        auto cx = [&](int i, int j) {  // key[i] >= key[j] afterwards
            const unsigned long long a = key[i], b = key[j];
            key[i] = a > b ? a : b;
            key[j] = a > b ? b : a;
        };
        cx(0, 1); cx(2, 3); cx(4, 5); cx(6, 7);
        cx(0, 2); cx(1, 3); cx(4, 6); cx(5, 7);
        cx(1, 2); cx(5, 6);
        cx(0, 4); cx(1, 5); cx(2, 6); cx(3, 7);
        cx(2, 4); cx(3, 5);
        cx(1, 2); cx(3, 4); cx(5, 6);
        for (int j = 0; j < k; ++j) {
            const bool has = key[0] != 0ull;
            const uint32_t hs = (uint32_t)(key[0] >> 32);
            const uint32_t best = __reduce_max_sync(full, has ? hs : 0u);
            const uint32_t cand = has && hs == best ? (uint32_t)lane + 32u * (255u - (uint32_t)(key[0] & 0xFFu))
                                                    : 0xFFFFFFFFu;
            const uint32_t e = __reduce_min_sync(full, cand);
            if ((int)(e & 31u) == lane) {
#pragma unroll
                for (int i = 0; i < 7; ++i) key[i] = key[i + 1];
                key[7] = 0ull;
            }
            const float sv = __uint_as_float(best);
            sum += sv;
            if (lane == j) {
                sel_e = (int)e;
                sel_s = sv;
            }
        }
    } else {
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
        for (int j = 0; j < k; ++j) {
            const uint32_t best = __reduce_max_sync(full, hi < SLOTS ? hv : 0u);
            const uint32_t cand = (hi < SLOTS && hv == best) ? (uint32_t)(lane + 32 * hi) : 0xFFFFFFFFu;
            const uint32_t e = __reduce_min_sync(full, cand);
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
    }
    if (lane < k) {
        ids[lane] = sel_e;
        weights[lane] = sel_s / sum;
    }
}

// The same over scores in memory (lane l: experts l + 32 i).
template <int SLOTS, bool L2 = false>
__device__ __forceinline__ void topk_warp(const uint32_t* sc, int E, int k, int lane, int32_t* ids,
                                          float* weights) {
    uint32_t s[SLOTS];
#pragma unroll
    for (int i = 0; i < SLOTS; ++i) {
        const int e = lane + 32 * i;
        s[i] = e >= E ? 0u : L2 ? (uint32_t)ld_cg(reinterpret_cast<const int32_t*>(sc) + e) : sc[e];
    }
    topk_warp_regs<SLOTS>(s, E, k, lane, ids, weights);
}

// The same from one token's FP32 logits in global memory (written by other
// CTAs: read past L1), the sigmoid (and bias) applied on load.
template <int SLOTS>
__device__ __forceinline__ void topk_warp_logits(const float* logits, const float* bias, int E, int k, int lane,
                                                 int32_t* ids, float* weights) {
    uint32_t s[SLOTS];
#pragma unroll
    for (int i = 0; i < SLOTS; ++i) {
        const int e = lane + 32 * i;
        s[i] = e >= E ? 0u : sigmoid_score(ld_cg(logits + e), bias, e);
    }
    topk_warp_regs<SLOTS>(s, E, k, lane, ids, weights);
}

}  // namespace
}  // namespace flint
