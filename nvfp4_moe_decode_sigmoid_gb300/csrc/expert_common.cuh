// expert_common.cuh -- device code shared by the expert GEMV kernels and the
// fused layer kernel: the per-CTA routing view, activation staging (bf16 ->
// chunk-scaled f16 in shared memory), the gate/up and down warp passes and
// the warp reduce-scatter. Included by one translation unit each; everything
// here is internal to that unit.
#pragma once

#include "flint_device.cuh"

namespace flint {
namespace {

constexpr int kMaxDistinct = FLINT_MAX_TOKENS * FLINT_MAX_TOPK;

// Per-CTA view of the routing: the distinct selected experts in ascending id
// order and, for each, which ranks of which tokens chose it.
struct RouteInfo {
    uint32_t bitmap[FLINT_MAX_EXPERTS / 32];
    uint32_t base[FLINT_MAX_EXPERTS / 32];
    int32_t dlist[kMaxDistinct];
    unsigned long long dmask[kMaxDistinct];  // byte t: ranks j with ids[t][j] == dlist[d]
    uint32_t tmask[kMaxDistinct];            // bit t: token t chose dlist[d]
    int32_t ids[kMaxDistinct];               // ids[t*k+j], -1 if out of range
    int D;
};

// ids: global memory (written by an earlier kernel; IDS_SMEM false) or this
// CTA's shared memory (IDS_SMEM true).
template <bool IDS_SMEM = false>
__device__ void build_route_info(RouteInfo& ri, const int32_t* ids, int T, int k, int E, uint32_t* status) {
    const int tid = threadIdx.x, nt = blockDim.x;
    for (int i = tid; i < FLINT_MAX_EXPERTS / 32; i += nt) ri.bitmap[i] = 0;
    for (int i = tid; i < kMaxDistinct; i += nt) {
        ri.dmask[i] = 0ull;
        ri.tmask[i] = 0u;
    }
    __syncthreads();
    int e = -1;
    if (tid < T * k) {
        e = IDS_SMEM ? ids[tid] : ld_cg(ids + tid);
        if (e >= 0 && e < E) {
            atomicOr(&ri.bitmap[e >> 5], 1u << (e & 31));
        } else {
            if (status) atomicOr(status, kStatusBadExpertId);
            e = -1;
        }
        ri.ids[tid] = e;
    }
    __syncthreads();
    if (tid < 32) {  // exclusive prefix sum of popcounts over the bitmap words
        const int nb = (E + 31) / 32;
        const uint32_t cnt = tid < nb ? __popc(ri.bitmap[tid]) : 0u;
        uint32_t incl = cnt;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const uint32_t v = __shfl_up_sync(0xffffffffu, incl, off);
            if (tid >= off) incl += v;
        }
        ri.base[tid] = incl - cnt;
        if (tid == 31) ri.D = (int)incl;
    }
    __syncthreads();
    if (e >= 0) {
        const int d = (int)(ri.base[e >> 5] + __popc(ri.bitmap[e >> 5] & ((1u << (e & 31)) - 1u)));
        const int t = tid / k, j = tid % k;
        ri.dlist[d] = e;
        atomicOr(&ri.dmask[d], 1ull << (8 * t + j));
        atomicOr(&ri.tmask[d], 1u << t);
    }
    __syncthreads();
}

__device__ __forceinline__ uint32_t rank_bits(unsigned long long dm, int t) {
    return (uint32_t)((dm >> (8 * t)) & 0xFFull);
}

__device__ __forceinline__ float silu_f32(float g) { return g / (1.f + expf(-g)); }

// acc0/acc1 += the 8 products of one code word (4 f16x2) with its 8
// activations (one 16-byte word of 4 f16x2).
__device__ __forceinline__ void fma8(const uint32_t (&c)[4], const uint4 xv, float& acc0, float& acc1) {
    const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        acc0 = fma_lo_f16(c[q], xw[q], acc0);
        acc1 = fma_hi_f16(c[q], xw[q], acc1);
    }
}

// Sums each of M values (M a power of two, at most 32) over the warp's lanes.
// Halving steps: at offset 16 >> s the lanes with that bit set keep the upper
// half of their remaining values and hand the lower half to their partner
// (one shuffle per value kept), so M sums cost about M shuffles instead of
// 5 M. Lane l ends up with the sum of value rs_index<M>(l); 32 / M lanes hold
// each value.
template <int M>
__device__ __forceinline__ float reduce_scatter(float (&v)[M], int lane) {
#pragma unroll
    for (int s = 0; (M >> s) > 1; ++s) {
        const int w = M >> s, off = 16 >> s;
        const bool up = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < w / 2; ++i) {
            const float keep = up ? v[i + w / 2] : v[i];
            const float send = up ? v[i] : v[i + w / 2];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
    float r = v[0];
#pragma unroll
    for (int off = 16 / M; off > 0; off >>= 1) r += __shfl_xor_sync(0xffffffffu, r, off);
    return r;
}

template <int M>
__device__ __forceinline__ int rs_index(int lane) {
    int idx = 0;
#pragma unroll
    for (int s = 0; (M >> s) > 1; ++s)
        if (lane & (16 >> s)) idx += M >> (s + 1);
    return idx;
}

// ===========================================================================
// Activation staging: bf16 vectors in global memory -> chunk-scaled f16 in
// shared memory. One thread moves one 32-value chunk (its four 16-byte loads
// issued together). csc[v * (K / 32) + c] = 2^s multiplies chunk c's partial
// dot product back.
//   GATE order (K % 1024 == 0): word w (0..3, 8 values each) of chunk c at
//     16-byte index (c / 32) * 128 + w * 32 + c % 32 of the vector: lane l
//     reads chunk l + 32 m's words at (m * 4 + w) * 32 + l.
//   DOWN order (K % 32 == 0): the two words of 16-value block b at indices b
//     and nb + b (nb = K / 16): lane l reads block l + 32 m at l + 32 m and
//     nb + l + 32 m.
// ===========================================================================
// One staging source: nvec bf16 vectors of K values.
struct StageSrc {
    const uint16_t* src;
    uint4* dst;
    float* csc;
    int nvec, K;
};

// Chunk q of the concatenated sources: its source (copied out field by field
// with constant indices, so that the sources stay in registers) and offset;
// false past the end.
template <int NS>
__device__ __forceinline__ bool stage_locate(const StageSrc (&ss)[NS], int q, StageSrc& src, int& v, int& c) {
    bool found = false;
#pragma unroll
    for (int i = 0; i < NS; ++i) {
        const int cpv = ss[i].K / 32, n = ss[i].nvec * cpv;
        if (!found && q < n) {
            src = ss[i];
            v = q / cpv;
            c = q - v * cpv;
            found = true;
        }
        q -= n;
    }
    return found;
}

__device__ __forceinline__ void stage_load(const StageSrc& ss, int v, int c, uint4 (&w)[4]) {
    const uint4* s4 = reinterpret_cast<const uint4*>(ss.src + (size_t)v * ss.K + 32 * c);
#pragma unroll
    for (int i = 0; i < 4; ++i) w[i] = ld_cg(s4 + i);
}

template <bool DOWN_ORDER>
__device__ __forceinline__ void stage_store(const StageSrc& ss, int v, int c, const uint4 (&w)[4]) {
    uint32_t m2 = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        m2 = __vmaxu2(m2, w[i].x & 0x7FFF7FFFu);
        m2 = __vmaxu2(m2, w[i].y & 0x7FFF7FFFu);
        m2 = __vmaxu2(m2, w[i].z & 0x7FFF7FFFu);
        m2 = __vmaxu2(m2, w[i].w & 0x7FFF7FFFu);
    }
    // bf16 exponent field of the largest magnitude -> s with max * 2^-s in [2^14, 2^15)
    const uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
    const int sh = min(126, max(-126, (int)(m >> 7) - 141));
    const float down = __int_as_float((127 - sh) << 23);
    const int K = ss.K;
    ss.csc[v * (K / 32) + c] = __int_as_float((127 + sh) << 23);
    uint4* d = ss.dst + (size_t)v * (K / 8);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        int idx;
        if (DOWN_ORDER) {
            idx = (i & 1) * (K / 16) + 2 * c + (i >> 1);
        } else {
            idx = (c / 32) * 128 + i * 32 + c % 32;
        }
        d[idx] = make_uint4(f32x2_to_f16x2(bf16_lo(w[i].x) * down, bf16_hi(w[i].x) * down),
                            f32x2_to_f16x2(bf16_lo(w[i].y) * down, bf16_hi(w[i].y) * down),
                            f32x2_to_f16x2(bf16_lo(w[i].z) * down, bf16_hi(w[i].z) * down),
                            f32x2_to_f16x2(bf16_lo(w[i].w) * down, bf16_hi(w[i].w) * down));
    }
}

// Stages the sources; every thread first issues the loads of its first chunk
// (first two in DOWN order: h of 8 tokens is more than one chunk per thread),
// then runs `between` (the callers issue their weight copies there, so that
// these small loads are not queued behind the weight stream), then converts.
// Further chunks are loaded and converted after.
template <bool DOWN_ORDER, int NS, typename F>
__device__ __forceinline__ void stage_f16(const StageSrc (&ss)[NS], F&& between) {
    constexpr int AHEAD = DOWN_ORDER ? 2 : 1;  // chunks loaded ahead of `between` (h: up to two per thread)
    const int nt = (int)blockDim.x;
    StageSrc s0 = ss[0], s1 = ss[0];
    int v0 = 0, c0 = 0, v1 = 0, c1 = 0;
    uint4 w[4], w1[4];
    bool have = stage_locate(ss, threadIdx.x, s0, v0, c0);
    bool have1 = AHEAD > 1 && stage_locate(ss, threadIdx.x + nt, s1, v1, c1);
    if (have) stage_load(s0, v0, c0, w);
    if (have1) stage_load(s1, v1, c1, w1);
    between();
    // one conversion site; the next chunk is loaded while the current one is
    // converted
    for (int q = threadIdx.x + AHEAD * nt; have; q += nt) {
        stage_store<DOWN_ORDER>(s0, v0, c0, w);
        if (AHEAD > 1) {
            have = have1;
            s0 = s1;
            v0 = v1;
            c0 = c1;
#pragma unroll
            for (int i = 0; i < 4; ++i) w[i] = w1[i];
            have1 = stage_locate(ss, q, s1, v1, c1);
            if (have1) stage_load(s1, v1, c1, w1);
        } else {
            have = stage_locate(ss, q, s0, v0, c0);
            if (have) stage_load(s0, v0, c0, w);
        }
    }
}

// One 16-byte word (8 values) of a chunk, staged by the thread that holds it
// when the four words of every chunk are held by four consecutive lanes (word
// i = lane % 4): the chunk's largest magnitude comes from two shuffles, then
// each value is converted on its own. The same bits as stage_store, with a
// quarter of the dependent steps per thread. Every lane of the warp calls it.
template <bool DOWN_ORDER>
__device__ __forceinline__ void stage_store_word(const StageSrc& ss, int v, int c, int i, const uint4 w) {
    uint32_t m2 = __vmaxu2(__vmaxu2(w.x & 0x7FFF7FFFu, w.y & 0x7FFF7FFFu),
                           __vmaxu2(w.z & 0x7FFF7FFFu, w.w & 0x7FFF7FFFu));
    m2 = __vmaxu2(m2, __shfl_xor_sync(0xffffffffu, m2, 1));
    m2 = __vmaxu2(m2, __shfl_xor_sync(0xffffffffu, m2, 2));
    // bf16 exponent field of the largest magnitude -> s with max * 2^-s in [2^14, 2^15)
    const uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
    const int sh = min(126, max(-126, (int)(m >> 7) - 141));
    const float down = __int_as_float((127 - sh) << 23);
    const int K = ss.K;
    if (i == 0) ss.csc[v * (K / 32) + c] = __int_as_float((127 + sh) << 23);
    const int idx = DOWN_ORDER ? (i & 1) * (K / 16) + 2 * c + (i >> 1) : (c / 32) * 128 + i * 32 + c % 32;
    ss.dst[(size_t)v * (K / 8) + idx] = make_uint4(f32x2_to_f16x2(bf16_lo(w.x) * down, bf16_hi(w.x) * down),
                                                   f32x2_to_f16x2(bf16_lo(w.y) * down, bf16_hi(w.y) * down),
                                                   f32x2_to_f16x2(bf16_lo(w.z) * down, bf16_hi(w.z) * down),
                                                   f32x2_to_f16x2(bf16_lo(w.w) * down, bf16_hi(w.w) * down));
}

// stage_f16 with four threads per 32-value chunk (thread q of the sources'
// 16-byte words takes word q % 4 of chunk q / 4), every thread's words loaded
// at once (up to four per thread per round). The same bits as stage_f16. It
// pays where the chunks are few against the threads (all of h at one token:
// the 49-block stack 907 -> 892 us per token step) and measured slower where
// every thread already has a chunk (eight tokens). Every source holds a
// multiple of 32 words (K % 256 == 0), so whole warps take part.
template <bool DOWN_ORDER, int NS>
__device__ __forceinline__ void stage_f16_quarters(const StageSrc (&ss)[NS]) {
    constexpr int MW = 4;  // words per thread per round
    const int nt = (int)blockDim.x;
    int total = 0;
#pragma unroll
    for (int i = 0; i < NS; ++i) total += ss[i].nvec * (ss[i].K / 8);
    for (int base = 0; base < total; base += MW * nt) {
        uint4 w[MW];
        StageSrc sw[MW];
        int vw[MW], cw[MW];
#pragma unroll
        for (int r = 0; r < MW; ++r) {
            const int q = base + (int)threadIdx.x + r * nt;
            if (q < total && stage_locate(ss, q >> 2, sw[r], vw[r], cw[r]))
                w[r] = ld_cg(reinterpret_cast<const uint4*>(sw[r].src + (size_t)vw[r] * sw[r].K + 32 * cw[r]) + (q & 3));
        }
#pragma unroll
        for (int r = 0; r < MW; ++r) {
            const int q = base + (int)threadIdx.x + r * nt;  // q < total is the same in all lanes of a warp
            if (q < total) stage_store_word<DOWN_ORDER>(sw[r], vw[r], cw[r], q & 3, w[r]);
        }
    }
}

// ===========================================================================
// Residual add + RMSNorm ahead of a block, fused into the activation staging
// ("Flint 是什么": pre-norm blocks; "Optimizations": norm kernels that follow
// the reference's rounding). Per token: r' = bf16(r + y), x =
// bf16(r' / sqrt(mean(r'^2) + eps) * gamma), in FP32. Every CTA normalises the
// whole [T, H] input itself (its sums run in one fixed order, so all CTAs get
// the same x); the CTA `cta` of G writes the chunks q with q % G == cta of r'
// (and of x) out.
// ===========================================================================
// bf16(a + b) of the two bf16 pairs of a word (FP32 add, round to nearest even).
__device__ __forceinline__ uint32_t bf16x2_add_round(uint32_t a, uint32_t b) {
    return (uint32_t)f32_to_bf16_bits(bf16_lo(a) + bf16_lo(b)) |
           ((uint32_t)f32_to_bf16_bits(bf16_hi(a) + bf16_hi(b)) << 16);
}
// bf16(a * inv * g) of the two bf16 pairs of a word.
__device__ __forceinline__ uint32_t bf16x2_scale_round(uint32_t a, float inv, uint32_t g) {
    return (uint32_t)f32_to_bf16_bits(bf16_lo(a) * inv * bf16_lo(g)) |
           ((uint32_t)f32_to_bf16_bits(bf16_hi(a) * inv * bf16_hi(g)) << 16);
}
__device__ __forceinline__ float bf16x2_sumsq(uint32_t a, float ss) {
    ss = fmaf(bf16_lo(a), bf16_lo(a), ss);
    return fmaf(bf16_hi(a), bf16_hi(a), ss);
}

// r' of the 32 values at `off` into w (bf16 words) and their sum of squares.
__device__ __forceinline__ float norm_residual_chunk(const NormArgs& n, size_t off, uint4 (&w)[4]) {
    const uint4* r4 = reinterpret_cast<const uint4*>(n.r + off);
#pragma unroll
    for (int i = 0; i < 4; ++i) w[i] = ld_cg(r4 + i);
    if (n.y) {
        const uint4* y4 = reinterpret_cast<const uint4*>(n.y + off);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 yv = ld_cg(y4 + i);
            w[i] = make_uint4(bf16x2_add_round(w[i].x, yv.x), bf16x2_add_round(w[i].y, yv.y),
                              bf16x2_add_round(w[i].z, yv.z), bf16x2_add_round(w[i].w, yv.w));
        }
    }
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        ss = bf16x2_sumsq(w[i].x, ss);
        ss = bf16x2_sumsq(w[i].y, ss);
        ss = bf16x2_sumsq(w[i].z, ss);
        ss = bf16x2_sumsq(w[i].w, ss);
    }
    return ss;
}

// w (r' words of the 32 values at column `col`) := bf16(r' * inv * gamma).
__device__ __forceinline__ void norm_scale_chunk(const NormArgs& n, int col, float inv, uint4 (&w)[4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint4 g = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);  // bf16 1.0 pairs
        if (n.gamma) g = ld_cg(reinterpret_cast<const uint4*>(n.gamma + col) + i);
        w[i] = make_uint4(bf16x2_scale_round(w[i].x, inv, g.x), bf16x2_scale_round(w[i].y, inv, g.y),
                          bf16x2_scale_round(w[i].z, inv, g.z), bf16x2_scale_round(w[i].w, inv, g.w));
    }
}

// Stages x = norm(r (+ y)) of all ss.nvec tokens as chunk-scaled f16 (GATE
// order). red: shared memory for ss.nvec * ss.K / 32 floats; inv: for
// ss.nvec floats.
// FEW (the one-token instantiations): with few chunks against the threads, the
// second pass runs four threads per chunk. A compile-time choice: with the
// branch compiled in, the eight-token block measured 1.1 us slower.
template <bool FEW>
__device__ void stage_norm_f16(const NormArgs& n, const StageSrc& ss, float* red, float* inv, int cta, int G) {
    const int cpv = ss.K / 32, nq = ss.nvec * cpv;
    const int q0 = threadIdx.x, nt = blockDim.x;
    uint4 w0[4] = {};
    for (int q = q0; q < nq; q += nt) {
        uint4 w[4];
        const int t = q / cpv, c = q - t * cpv;
        const size_t off = (size_t)t * ss.K + 32 * c;
        red[q] = norm_residual_chunk(n, off, w);
        if (n.r_out && q % G == cta) {
#pragma unroll
            for (int i = 0; i < 4; ++i) reinterpret_cast<uint4*>(n.r_out + off)[i] = w[i];
        }
        if (q == q0) {
#pragma unroll
            for (int i = 0; i < 4; ++i) w0[i] = w[i];
        }
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int t = warp; t < ss.nvec; t += nt >> 5) {
        float s = 0.f;
        for (int c = lane; c < cpv; c += 32) s += red[t * cpv + c];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        if (lane == 0) inv[t] = 1.f / sqrtf(s / (float)ss.K + n.eps);
    }
    __syncthreads();
    if (FEW && 4 * nq <= nt) {
        // Few chunks (one token): the chunk threads park r' in the staging area
        // in natural order, then four threads per chunk scale a 16-byte word
        // each and stage it (stage_store_word; the same bits as below, fewer
        // dependent steps per thread). 4 nq = nvec K / 8 is a multiple of 32:
        // whole warps.
        if (q0 < nq) {
#pragma unroll
            for (int i = 0; i < 4; ++i) ss.dst[4 * q0 + i] = w0[i];
        }
        __syncthreads();
        uint4 w = make_uint4(0u, 0u, 0u, 0u);
        if (q0 < 4 * nq) w = ss.dst[q0];
        __syncthreads();  // every parked word read before the staged words land
        if (q0 < 4 * nq) {
            const int q = q0 >> 2, i = q0 & 3, t = q / cpv, c = q - t * cpv;
            uint4 g = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);  // bf16 1.0 pairs
            if (n.gamma) g = ld_cg(reinterpret_cast<const uint4*>(n.gamma + 32 * c) + i);
            const float iv = inv[t];
            w = make_uint4(bf16x2_scale_round(w.x, iv, g.x), bf16x2_scale_round(w.y, iv, g.y),
                           bf16x2_scale_round(w.z, iv, g.z), bf16x2_scale_round(w.w, iv, g.w));
            if (n.x_out && q % G == cta) reinterpret_cast<uint4*>(n.x_out + (size_t)t * ss.K + 32 * c)[i] = w;
            stage_store_word<false>(ss, t, c, i, w);
        }
        return;
    }
    for (int q = q0; q < nq; q += nt) {
        uint4 w[4];
        const int t = q / cpv, c = q - t * cpv;
        const size_t off = (size_t)t * ss.K + 32 * c;
        if (q == q0) {
#pragma unroll
            for (int i = 0; i < 4; ++i) w[i] = w0[i];
        } else {
            norm_residual_chunk(n, off, w);
        }
        norm_scale_chunk(n, 32 * c, inv[t], w);
        if (n.x_out && q % G == cta) {
#pragma unroll
            for (int i = 0; i < 4; ++i) reinterpret_cast<uint4*>(n.x_out + off)[i] = w[i];
        }
        stage_store<false>(ss, t, c, w);
    }
}

// One pass of a warp over gate row `grow` (and up row `urow`) against the NT
// (1 or 2) tokens tk[]: the lanes split the row into 32-value chunks
// (lane l: chunks l, l + 32, ...); the per-lane sums are reduce-scattered and
// the lanes holding them store the raw sums (before the tensor scale) at
// resg[t] / resu[t].
template <bool PAIR, int NT>
__device__ __forceinline__ void gate_up_pass(const uint8_t* grow, const uint8_t* urow, int H, const uint4* xh,
                                             const float* csc, const int (&tk)[NT], int lane, float* resg,
                                             float* resu) {
    constexpr int M = PAIR ? 2 * NT : NT;
    const uint4* xb[NT];
    const float* cb[NT];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        xb[j] = xh + (size_t)tk[j] * (H / 8) + lane;
        cb[j] = csc + (size_t)tk[j] * (H / 32) + lane;
    }
    const uint4* g4 = reinterpret_cast<const uint4*>(grow) + lane;
    const uint4* u4 = reinterpret_cast<const uint4*>(urow) + lane;
    const uint16_t* gsc = reinterpret_cast<const uint16_t*>(grow + H / 2) + lane;
    const uint16_t* usc = reinterpret_cast<const uint16_t*>(urow + H / 2) + lane;
    float acc[M];
#pragma unroll
    for (int i = 0; i < M; ++i) acc[i] = 0.f;
    const int nch = H >> 10;
#pragma unroll 1
    for (int ch = 0; ch < nch; ++ch) {
        const uint4 gq = g4[32 * ch];
        const float2 gs = ue4m3x2_to_float2(gsc[32 * ch]);
        uint4 uq = make_uint4(0u, 0u, 0u, 0u);
        float2 us = make_float2(0.f, 0.f);
        if (PAIR) {
            uq = u4[32 * ch];
            us = ue4m3x2_to_float2(usc[32 * ch]);
        }
        const uint32_t gw[4] = {gq.x, gq.y, gq.z, gq.w}, uw[4] = {uq.x, uq.y, uq.z, uq.w};
        float cg[NT], cu[NT];
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {  // one scale block: code words 2 hf, 2 hf + 1
            float g0[NT], g1[NT], u0[NT], u1[NT];
#pragma unroll
            for (int j = 0; j < NT; ++j) g0[j] = g1[j] = u0[j] = u1[j] = 0.f;
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const int w = 2 * hf + h2;
                uint32_t hg[4], hu[4];
                decode_word_h2(gw[w], hg);
                if (PAIR) decode_word_h2(uw[w], hu);
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    const uint4 xv = xb[j][(ch * 4 + w) * 32];
                    fma8(hg, xv, g0[j], g1[j]);
                    if (PAIR) fma8(hu, xv, u0[j], u1[j]);
                }
            }
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                if (hf == 0) {
                    cg[j] = gs.x * (g0[j] + g1[j]);
                    if (PAIR) cu[j] = us.x * (u0[j] + u1[j]);
                } else {
                    cg[j] = fmaf(gs.y, g0[j] + g1[j], cg[j]);
                    if (PAIR) cu[j] = fmaf(us.y, u0[j] + u1[j], cu[j]);
                }
            }
        }
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            const float xs = cb[j][32 * ch];
            acc[j] = fmaf(xs, cg[j], acc[j]);
            if (PAIR) acc[NT + j] = fmaf(xs, cu[j], acc[NT + j]);
        }
    }
    const float r = reduce_scatter<M>(acc, lane);
    if (lane % (32 / M) == 0) {
        const int idx = rs_index<M>(lane);  // [gate of tk[0..NT), up of tk[0..NT)]
        const int j = idx % NT;
        int t = tk[0];
#pragma unroll
        for (int jj = 1; jj < NT; ++jj)
            if (j == jj) t = tk[jj];
        (idx < NT ? resg : resu)[t] = r;
    }
}

// All tokens of `tmask` against one item, two per pass.
template <bool PAIR>
__device__ __forceinline__ void gate_up_item(const uint8_t* grow, const uint8_t* urow, int H, const uint4* xh,
                                             const float* csc, uint32_t tmask, int lane, float* resg,
                                             float* resu) {
    while (tmask) {
        const int t0 = __ffs(tmask) - 1;
        tmask &= tmask - 1u;
        if (tmask) {
            const int tk[2] = {t0, __ffs(tmask) - 1};
            tmask &= tmask - 1u;
            gate_up_pass<PAIR, 2>(grow, urow, H, xh, csc, tk, lane, resg, resu);
        } else {
            const int tk[1] = {t0};
            gate_up_pass<PAIR, 1>(grow, urow, H, xh, csc, tk, lane, resg, resu);
        }
    }
}

// One pass of a warp over RP rows (row r at rows + r RS, r < nr valid) of K
// columns against NT tokens whose staged h vectors are hv[] (DOWN order) with
// chunk scales cv[]: lane l takes the 16-value blocks l, l + 32, ...
// acc[j * RP + r] gets the lane's part of row r . h_j.
template <int RP, int NT>
__device__ __forceinline__ void down_pass(const uint8_t* rows, int RS, int nr, int K, const uint4* const (&hv)[NT],
                                          const float* const (&cv)[NT], int lane, float (&acc)[RP * NT]) {
#pragma unroll
    for (int i = 0; i < RP * NT; ++i) acc[i] = 0.f;
    const int nb = K / 16;
    for (int b = lane; b < nb; b += 32) {
        uint4 x0[NT], x1[NT];
        float xs[NT];
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            x0[j] = hv[j][b];
            x1[j] = hv[j][nb + b];
            xs[j] = cv[j][b >> 1];
        }
#pragma unroll
        for (int r = 0; r < RP; ++r) {
            if (r < nr) {
                const uint8_t* row = rows + (size_t)r * RS;
                const uint2 q = *reinterpret_cast<const uint2*>(row + 8 * b);
                const float s = ue4m3_to_float(row[K / 2 + b]);
                uint32_t c0[4], c1[4];
                decode_word_h2(q.x, c0);
                decode_word_h2(q.y, c1);
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    float p0 = 0.f, p1 = 0.f;
                    fma8(c0, x0[j], p0, p1);
                    fma8(c1, x1[j], p0, p1);
                    acc[j * RP + r] = fmaf(s * xs[j], p0 + p1, acc[j * RP + r]);
                }
            }
        }
    }
}


}  // namespace
}  // namespace flint
