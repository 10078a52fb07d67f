// gemv.cu -- the expert GEMVs of the MoE decode step (and the dense GEMV).
//
// "Day-0 Support for Flint on vLLM", section "Optimizations": small-batch MoE
// kernels whose expert GEMVs read only the selected experts' weights; routing
// and the expert combine fused into the neighbouring GEMV kernels; each kernel
// launched with programmatic dependent launch so it loads its weights while
// the previous kernel still runs; norm and SiLU following the reference's
// rounding. Section "Model architecture": weight-only NVFP4 (W4A16) with bf16
// activations; every kernel follows the reference's rounding points.
//
// gate_up_kernel: per (selected expert, h index i) "pair" a warp dots gate row
//   i and up row i with every token that selected the expert (FP32), then
//   g = bf16(ts_g * acc_g), u = bf16(ts_u * acc_u), h = bf16(silu(g) * u).
//   The pair space (shared expert first, then the distinct selected experts in
//   ascending id order) is split evenly over one CTA per SM; each CTA streams
//   its rows through a ring of shared-memory stages filled by 1-D bulk (TMA)
//   copies. The shared expert's rows are requested before the PDL wait.
// down_kernel: each CTA owns a slice of output rows of every selected expert's
//   down matrix (and the shared one), computes d = bf16(ts_d * Wd h) for all
//   of them, then the combine y = bf16(sum_j w_j d_j + d_shared) in rank order.
//   No atomics: the result is deterministic. Its weight rows are requested
//   before the PDL wait (the routing is final by then).
#include "flint_device.cuh"

namespace flint {
namespace {

constexpr int kItemsPerStage = kWarps;  // one gate/up pair per warp per stage
constexpr int kMaxDistinct = FLINT_MAX_TOKENS * FLINT_MAX_TOPK;

// 128-byte XOR swizzle of 16-byte granules: granule G of a buffer lives at
// G ^ ((G >> 3) & 7). Lanes that read granule i of consecutive 64/128-byte
// chunks then hit distinct bank groups.
__device__ __forceinline__ int swz(int G) { return G ^ ((G >> 3) & 7); }

// Per-CTA view of the routing: the distinct selected experts in ascending id
// order and, for each, which ranks of which tokens chose it.
struct RouteInfo {
    uint32_t bitmap[FLINT_MAX_EXPERTS / 32];
    uint32_t base[FLINT_MAX_EXPERTS / 32];
    int32_t dlist[kMaxDistinct];
    unsigned long long dmask[kMaxDistinct];  // byte t: ranks j with ids[t][j] == dlist[d]
    int32_t ids[kMaxDistinct];               // ids[t*k+j], -1 if out of range
    int D;
};

__device__ void build_route_info(RouteInfo& ri, const int32_t* ids, int T, int k, int E, uint32_t* status) {
    const int tid = threadIdx.x;
    for (int i = tid; i < FLINT_MAX_EXPERTS / 32; i += kThreads) ri.bitmap[i] = 0;
    for (int i = tid; i < kMaxDistinct; i += kThreads) ri.dmask[i] = 0ull;
    __syncthreads();
    int e = -1;
    if (tid < T * k) {
        e = ld_cg(ids + tid);
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
    }
    __syncthreads();
}

__device__ __forceinline__ uint32_t token_mask(unsigned long long dm) {
    uint32_t m = 0;
#pragma unroll
    for (int t = 0; t < FLINT_MAX_TOKENS; ++t) m |= ((dm >> (8 * t)) & 0xFFull) ? (1u << t) : 0u;
    return m;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

__device__ __forceinline__ float silu_f32(float g) { return g / (1.f + expf(-g)); }

// dot of 32 decoded codes with 32 swizzled f32 activations of chunk `c`
__device__ __forceinline__ void dot32_f32(const float (&w)[32], const float* xt, int c, float& lo, float& hi) {
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float4 x4 = reinterpret_cast<const float4*>(xt)[swz(8 * c + i)];
        float& s = i < 4 ? s0 : s1;
        s = fmaf(w[4 * i + 0], x4.x, s);
        s = fmaf(w[4 * i + 1], x4.y, s);
        s = fmaf(w[4 * i + 2], x4.z, s);
        s = fmaf(w[4 * i + 3], x4.w, s);
    }
    lo = s0;
    hi = s1;
}

// dot of 32 decoded codes with 32 swizzled bf16 activations of chunk `c`
__device__ __forceinline__ void dot32_bf16(const float (&w)[32], const uint16_t* ht, int c, float& lo, float& hi) {
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint4 v = reinterpret_cast<const uint4*>(ht)[swz(4 * c + i)];
        const uint32_t vv[4] = {v.x, v.y, v.z, v.w};
        float& s = i < 2 ? s0 : s1;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            s = fmaf(w[8 * i + 2 * q], bf16_lo(vv[q]), s);
            s = fmaf(w[8 * i + 2 * q + 1], bf16_hi(vv[q]), s);
        }
    }
    lo = s0;
    hi = s1;
}

// ===========================================================================
// gate/up + SiLU
// ===========================================================================
struct GateUpSmem {
    size_t route, xs, ring, total;
};
__host__ __device__ inline GateUpSmem gate_up_layout(int T, int H, int nstages) {
    GateUpSmem L;
    L.route = 128;
    L.xs = align_up(L.route + sizeof(RouteInfo), 128);
    L.ring = align_up(L.xs + sizeof(float) * (size_t)T * H, 128);
    L.total = L.ring + (size_t)nstages * 2 * kItemsPerStage * nvfp4_row_stride(H);
    return L;
}

__global__ void __launch_bounds__(kThreads, 1) gate_up_kernel(const GateUpArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int NS = a.nstages, H = a.H, T = a.T, I = a.I, Is = a.Is;
    const GateUpSmem L = gate_up_layout(T, H, NS);
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
    RouteInfo& ri = *reinterpret_cast<RouteInfo*>(smem + L.route);
    float* xs = reinterpret_cast<float*>(smem + L.xs);
    uint8_t* ring = smem + L.ring;
    const int RS = (int)nvfp4_row_stride(H);
    const int half = kItemsPerStage * RS;  // gate rows of one stage; up rows follow

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = blockIdx.x, G = gridDim.x;
    const int sp0 = (int)((long long)c * Is / G), sp1 = (int)((long long)(c + 1) * Is / G);
    const int n_sh = a.s_gu ? sp1 - sp0 : 0;

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) mbar_init(&bar[s], 1);
        fence_mbar_init();
    }
    __syncthreads();
    // Before the wait: the shared expert's rows do not depend on the routing.
    if (tid == 0) {
        for (int st = 0; st < NS && st * kItemsPerStage < n_sh; ++st) {
            const int i0 = st * kItemsPerStage, n = min(n_sh - i0, kItemsPerStage);
            const uint32_t bytes = (uint32_t)(n * RS);
            uint8_t* g = ring + (size_t)st * 2 * half;
            mbar_expect_tx(&bar[st], 2 * bytes);
            bulk_g2s(g, a.s_gu + (size_t)(sp0 + i0) * RS, bytes, &bar[st]);
            bulk_g2s(g + half, a.s_gu + (size_t)(Is + sp0 + i0) * RS, bytes, &bar[st]);
        }
    }
    pdl_wait();  // ids and x are written by earlier kernels
    if (a.gu) {
        build_route_info(ri, a.ids, T, a.k, a.E, a.status);
    } else {
        if (tid == 0) ri.D = 0;
        __syncthreads();
    }
    pdl_launch_dependents();

    const int D = ri.D;
    const long long RP = (long long)D * I;
    const long long rp0 = (long long)c * RP / G, rp1 = (long long)(c + 1) * RP / G;
    const int n_items = n_sh + (int)(rp1 - rp0);
    const int n_stages = (n_items + kItemsPerStage - 1) / kItemsPerStage;

    // Thread 0: request the rows of stage `st` (routed ones; shared ones too
    // unless they were requested before the wait).
    auto issue = [&](int st, bool with_shared) {
        const int b = st % NS;
        uint8_t* g = ring + (size_t)b * 2 * half;
        const int i0 = st * kItemsPerStage, i1 = min(n_items, i0 + kItemsPerStage);
        for (int pass = 0; pass < 2; ++pass) {  // pass 0 counts bytes, pass 1 copies
            uint32_t bytes = 0;
            if (with_shared && i0 < n_sh) {
                const int n = min(i1, n_sh) - i0;
                if (pass) {
                    bulk_g2s(g, a.s_gu + (size_t)(sp0 + i0) * RS, n * RS, &bar[b]);
                    bulk_g2s(g + half, a.s_gu + (size_t)(Is + sp0 + i0) * RS, n * RS, &bar[b]);
                }
                bytes += 2u * n * RS;
            }
            const int ir = max(i0, n_sh);
            long long q0 = rp0 + (ir - n_sh);
            const long long q1 = rp0 + (i1 - n_sh);
            int slot = ir - i0;
            while (q0 < q1) {
                const int d = (int)(q0 / I), p0 = (int)(q0 % I);
                const int n = (int)min((long long)(I - p0), q1 - q0);
                if (pass) {
                    const uint8_t* base = a.gu + (size_t)ri.dlist[d] * 2 * I * RS;
                    bulk_g2s(g + slot * RS, base + (size_t)p0 * RS, n * RS, &bar[b]);
                    bulk_g2s(g + half + slot * RS, base + (size_t)(I + p0) * RS, n * RS, &bar[b]);
                }
                bytes += 2u * n * RS;
                slot += n;
                q0 += n;
            }
            if (!pass) mbar_arrive_expect_tx(&bar[b], bytes);
        }
    };
    if (tid == 0)
        for (int st = 0; st < min(NS, n_stages); ++st) issue(st, false);

    // x -> shared memory as f32, swizzled per 128-byte line
    for (int i = tid; i < T * H / 4; i += kThreads) {
        const int t = i / (H / 4), gi = i % (H / 4);  // granule of 4 floats
        const uint2 v = ld_cg(reinterpret_cast<const uint2*>(a.x + (size_t)t * H) + gi);
        reinterpret_cast<float4*>(xs + (size_t)t * H)[swz(gi)] =
            make_float4(bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y));
    }
    __syncthreads();

    const int nch = H / 1024;  // 16-byte chunks per lane per row
    bool ok = true;
    for (int st = 0; st < n_stages; ++st) {
        const int b = st % NS;
        ok = ok && mbar_wait_bounded(&bar[b], (uint32_t)((st / NS) & 1), lane == 0 ? a.status : nullptr,
                                     kStatusTimeoutGateUp);
        ok = __all_sync(0xffffffffu, ok);  // warp-uniform before any shuffle
        const int item = st * kItemsPerStage + warp;
        if (ok && item < n_items) {
            const uint8_t* grow = ring + (size_t)b * 2 * half + warp * RS;
            const uint8_t* urow = grow + half;
            bool shared_item = item < n_sh;
            int p, e = -1;
            unsigned long long dm = 0;
            uint32_t tmask;
            float tsg, tsu;
            if (shared_item) {
                p = sp0 + item;
                tmask = (1u << T) - 1u;
                tsg = a.s_ts[0];
                tsu = a.s_ts[1];
            } else {
                const long long q = rp0 + (item - n_sh);
                const int d = (int)(q / I);
                p = (int)(q % I);
                e = ri.dlist[d];
                dm = ri.dmask[d];
                tmask = token_mask(dm);
                tsg = a.ts[3 * e + 0];
                tsu = a.ts[3 * e + 1];
            }
            float ga[FLINT_MAX_TOKENS], ua[FLINT_MAX_TOKENS];
#pragma unroll
            for (int t = 0; t < FLINT_MAX_TOKENS; ++t) ga[t] = ua[t] = 0.f;
            for (int ch = 0; ch < nch; ++ch) {
                const int cidx = lane + 32 * ch;
                const uint4 gq = reinterpret_cast<const uint4*>(grow)[cidx];
                const uint4 uq = reinterpret_cast<const uint4*>(urow)[cidx];
                const float2 gs = ue4m3x2_to_float2(*reinterpret_cast<const uint16_t*>(grow + H / 2 + 2 * cidx));
                const float2 us = ue4m3x2_to_float2(*reinterpret_cast<const uint16_t*>(urow + H / 2 + 2 * cidx));
                float wg[32], wu[32];
                decode_chunk(gq, wg);
                decode_chunk(uq, wu);
#pragma unroll
                for (int t = 0; t < FLINT_MAX_TOKENS; ++t) {
                    if ((tmask >> t) & 1u) {
                        const float* xt = xs + (size_t)t * H;
                        float lo, hi;
                        dot32_f32(wg, xt, cidx, lo, hi);
                        ga[t] = fmaf(gs.x, lo, fmaf(gs.y, hi, ga[t]));
                        dot32_f32(wu, xt, cidx, lo, hi);
                        ua[t] = fmaf(us.x, lo, fmaf(us.y, hi, ua[t]));
                    }
                }
            }
#pragma unroll
            for (int t = 0; t < FLINT_MAX_TOKENS; ++t) {
                if ((tmask >> t) & 1u) {  // uniform across the warp
                    const float gsum = warp_sum(ga[t]), usum = warp_sum(ua[t]);
                    if (lane == t) {
                        const float g = bf16_round_f32(tsg * gsum);
                        const float u = bf16_round_f32(tsu * usum);
                        const uint16_t h = f32_to_bf16_bits(silu_f32(g) * u);
                        if (shared_item) {
                            a.h_shared[(size_t)t * Is + p] = h;
                        } else {
                            const uint32_t ranks = (uint32_t)((dm >> (8 * t)) & 0xFFull);
                            for (int j = 0; j < a.k; ++j)
                                if ((ranks >> j) & 1u) a.h_routed[((size_t)t * a.k + j) * I + p] = h;
                        }
                    }
                }
            }
        }
        if (!__syncthreads_and(ok)) return;
        if (tid == 0 && st + NS < n_stages) issue(st + NS, true);
    }
}

// ===========================================================================
// down + combine
// ===========================================================================
struct DownSmem {
    size_t route, w, dval, hr, hs, ring, total;
};
__host__ __device__ inline DownSmem down_layout(const DownArgs& a) {
    DownSmem L;
    L.route = 128;
    L.w = align_up(L.route + sizeof(RouteInfo), 128);
    L.dval = align_up(L.w + sizeof(float) * kMaxDistinct, 128);
    L.hr = align_up(L.dval + sizeof(float) * FLINT_MAX_TOKENS * (FLINT_MAX_TOPK + 1) * (size_t)a.rows_max, 128);
    L.hs = align_up(L.hr + 2 * (size_t)a.T * a.k * a.I, 128);
    L.ring = align_up(L.hs + 2 * (size_t)a.T * a.Is, 128);
    L.total = L.ring + (size_t)a.nstages * a.units_per_stage * a.slot_bytes;
    return L;
}

__global__ void __launch_bounds__(kThreads, 1) down_kernel(const DownArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const DownSmem L = down_layout(a);
    const int NS = a.nstages, UPS = a.units_per_stage, LPR = a.lpr;
    const int T = a.T, k = a.k, H = a.H, I = a.I, Is = a.Is, RM = a.rows_max;
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
    RouteInfo& ri = *reinterpret_cast<RouteInfo*>(smem + L.route);
    float* wsm = reinterpret_cast<float*>(smem + L.w);
    float* dval = reinterpret_cast<float*>(smem + L.dval);  // [t][j (k = shared)][row]
    uint16_t* hr = reinterpret_cast<uint16_t*>(smem + L.hr);
    uint16_t* hs = reinterpret_cast<uint16_t*>(smem + L.hs);
    uint8_t* ring = smem + L.ring;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = blockIdx.x, G = gridDim.x;
    const int n0 = (int)((long long)c * H / G), n1 = (int)((long long)(c + 1) * H / G), nr = n1 - n0;
    const int RSr = (int)nvfp4_row_stride(I), RSs = Is ? (int)nvfp4_row_stride(Is) : 0;
    if (nr == 0) return;  // more CTAs than output rows: nothing to copy or compute

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) mbar_init(&bar[s], 1);
        fence_mbar_init();
    }
    __syncthreads();
    // The routing is final before this kernel can start: the gate/up kernel
    // triggers its dependents only after its own wait on the router.
    if (a.down) {
        build_route_info(ri, a.ids, T, k, a.E, a.status);
    } else {
        if (tid == 0) ri.D = 0;
        __syncthreads();
    }
    const int D = ri.D;
    const bool has_sh = a.s_down != nullptr;
    const int n_units = D + (has_sh ? 1 : 0);
    const int n_stages = (n_units + UPS - 1) / UPS;

    auto issue = [&](int st) {  // thread 0
        const int b = st % NS;
        const int u0 = st * UPS, u1 = min(n_units, u0 + UPS);
        uint32_t bytes = 0;
        for (int u = u0; u < u1; ++u) bytes += (uint32_t)(nr * (u < D ? RSr : RSs));
        mbar_arrive_expect_tx(&bar[b], bytes);
        for (int u = u0; u < u1; ++u) {
            uint8_t* dst = ring + ((size_t)b * UPS + (u - u0)) * a.slot_bytes;
            if (u < D)
                bulk_g2s(dst, a.down + ((size_t)ri.dlist[u] * H + n0) * RSr, (uint32_t)(nr * RSr), &bar[b]);
            else
                bulk_g2s(dst, a.s_down + (size_t)n0 * RSs, (uint32_t)(nr * RSs), &bar[b]);
        }
    };
    if (tid == 0)
        for (int st = 0; st < min(NS, n_stages); ++st) issue(st);

    pdl_wait();  // h comes from the gate/up kernel
    pdl_launch_dependents();

    // h -> shared memory (bf16, swizzled), routing weights -> shared memory
    if (a.down) {
        const int gpr = I / 8;  // 16-byte granules per (t, j) vector
        for (int i = tid; i < T * k * gpr; i += kThreads) {
            const int v = i / gpr, gi = i % gpr;
            reinterpret_cast<uint4*>(hr + (size_t)v * I)[swz(gi)] =
                ld_cg(reinterpret_cast<const uint4*>(a.h_routed + (size_t)v * I) + gi);
        }
        for (int i = tid; i < T * k; i += kThreads) wsm[i] = ld_cg(a.w + i);
    }
    if (has_sh) {
        const int gpr = Is / 8;
        for (int i = tid; i < T * gpr; i += kThreads) {
            const int v = i / gpr, gi = i % gpr;
            reinterpret_cast<uint4*>(hs + (size_t)v * Is)[swz(gi)] =
                ld_cg(reinterpret_cast<const uint4*>(a.h_shared + (size_t)v * Is) + gi);
        }
    }
    __syncthreads();

    const int groups = kThreads / LPR, gpw = 32 / LPR;  // row groups per CTA / per warp
    const int gl = lane % LPR;
    bool ok = true;
    for (int st = 0; st < n_stages; ++st) {
        const int b = st % NS;
        ok = ok && mbar_wait_bounded(&bar[b], (uint32_t)((st / NS) & 1), lane == 0 ? a.status : nullptr,
                                     kStatusTimeoutDown);
        ok = __all_sync(0xffffffffu, ok);  // warp-uniform before any shuffle
        const int u0 = st * UPS, nu = min(n_units - u0, UPS);
        const int ntask = nu * nr;
        // warp-uniform trip count: every lane takes part in the shuffles
        for (int qb = warp * gpw; ok && qb < ntask; qb += groups) {
            const int q = qb + lane / LPR;
            const bool active = q < ntask;
            const int s = active ? q / nr : 0, r = active ? q % nr : 0;
            const int u = u0 + s;
            const bool sh = u >= D;
            const int K = sh ? Is : I;
            const uint8_t* row = ring + ((size_t)b * UPS + s) * a.slot_bytes + (size_t)r * (sh ? RSs : RSr);
            unsigned long long dm = 0;
            uint32_t tmask = 0;
            float tsd = 0.f;
            if (active) {
                if (sh) {
                    tmask = (1u << T) - 1u;
                    tsd = a.s_ts[a.s_ts_idx];
                } else {
                    dm = ri.dmask[u];
                    tmask = token_mask(dm);
                    tsd = a.ts[3 * ri.dlist[u] + 2];
                }
            }
            float acc[FLINT_MAX_TOKENS];
#pragma unroll
            for (int t = 0; t < FLINT_MAX_TOKENS; ++t) acc[t] = 0.f;
            if (active) {
                const int nch = K / 32 / LPR;
                for (int m = 0; m < nch; ++m) {
                    const int cidx = gl + LPR * m;
                    const uint4 q4 = reinterpret_cast<const uint4*>(row)[cidx];
                    const float2 sc = ue4m3x2_to_float2(*reinterpret_cast<const uint16_t*>(row + K / 2 + 2 * cidx));
                    float w[32];
                    decode_chunk(q4, w);
#pragma unroll
                    for (int t = 0; t < FLINT_MAX_TOKENS; ++t) {
                        if ((tmask >> t) & 1u) {
                            const uint16_t* ht;
                            if (sh) {
                                ht = hs + (size_t)t * Is;
                            } else {
                                const uint32_t ranks = (uint32_t)((dm >> (8 * t)) & 0xFFull);
                                ht = hr + ((size_t)t * k + (__ffs(ranks) - 1)) * I;
                            }
                            float lo, hi;
                            dot32_bf16(w, ht, cidx, lo, hi);
                            acc[t] = fmaf(sc.x, lo, fmaf(sc.y, hi, acc[t]));
                        }
                    }
                }
            }
#pragma unroll
            for (int t = 0; t < FLINT_MAX_TOKENS; ++t) {
                if (t >= T) break;  // T is uniform over the CTA
                float v = acc[t];
                for (int off = LPR / 2; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
                if (active && gl == 0 && ((tmask >> t) & 1u)) {
                    const float dv = bf16_round_f32(tsd * v);
                    if (sh) {
                        dval[((size_t)t * (k + 1) + k) * RM + r] = dv;
                    } else {
                        const uint32_t ranks = (uint32_t)((dm >> (8 * t)) & 0xFFull);
                        for (int j = 0; j < k; ++j)
                            if ((ranks >> j) & 1u) dval[((size_t)t * (k + 1) + j) * RM + r] = dv;
                    }
                }
            }
        }
        if (!__syncthreads_and(ok)) return;
        if (tid == 0 && st + NS < n_stages) issue(st + NS);
    }
    // combine, in rank order then the shared expert
    for (int i = tid; i < T * nr; i += kThreads) {
        const int t = i / nr, r = i % nr;
        float acc = 0.f;
        if (a.down) {
            for (int j = 0; j < k; ++j)
                if (ri.ids[t * k + j] >= 0) acc = fmaf(wsm[t * k + j], dval[((size_t)t * (k + 1) + j) * RM + r], acc);
        }
        if (has_sh) acc += dval[((size_t)t * (k + 1) + k) * RM + r];
        a.y[(size_t)t * H + n0 + r] = f32_to_bf16_bits(acc);
    }
}

template <typename K, typename A>
cudaError_t launch_ex(K kernel, const A& args, unsigned grid, size_t smem, bool pdl, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args);
}

}  // namespace

size_t gate_up_smem_bytes(const GateUpArgs& a) { return gate_up_layout(a.T, a.H, a.nstages).total; }
size_t down_smem_bytes(const DownArgs& a) { return down_layout(a).total; }

cudaError_t launch_gate_up(const GateUpArgs& a, const DevInfo& d, bool pdl, cudaStream_t s) {
    static int configured_for = -1;
    cudaError_t e = configure_smem(gate_up_kernel, d, configured_for);
    if (e != cudaSuccess) return e;
    return launch_ex(gate_up_kernel, a, (unsigned)d.sm_count, gate_up_smem_bytes(a), pdl, s);
}

cudaError_t launch_down(const DownArgs& a, const DevInfo& d, bool pdl, cudaStream_t s) {
    static int configured_for = -1;
    cudaError_t e = configure_smem(down_kernel, d, configured_for);
    if (e != cudaSuccess) return e;
    return launch_ex(down_kernel, a, (unsigned)d.sm_count, down_smem_bytes(a), pdl, s);
}

}  // namespace flint
