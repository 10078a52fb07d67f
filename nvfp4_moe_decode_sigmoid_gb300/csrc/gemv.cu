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
// Both kernels are warp-specialised: one producer warp streams weight rows
// from HBM into a ring of shared-memory stages with 1-D bulk (TMA) copies
// (full/empty mbarriers), and 15 consumer warps dequantise in registers
// (cvt e2m1x2 -> f16x2 -> f32 pairs, UE4M3 block scale once per 16 values)
// and accumulate exact products in FP32 with packed f32x2 FMAs. Activations
// are staged in shared memory as FP32 in a lane-interleaved order, so lane l
// reads consecutive 16-byte words (no bank conflicts, no address math).
//
// gate_up_kernel<PAIR=true>: per (selected expert, h index i) "pair" one warp
//   dots gate row i and up row i with every token that selected the expert,
//   then g = bf16(ts_g acc_g), u = bf16(ts_u acc_u), h = bf16(silu(g) u).
//   The pair space (shared expert first, then the distinct selected experts in
//   ascending id order) is split evenly over one CTA per SM. The shared
//   expert's rows are requested before the PDL wait.
// gate_up_kernel<PAIR=false>: the same machinery over plain rows: the dense
//   GEMV y = bf16(ts W x).
// down_kernel: each CTA owns a slice of output rows of every selected expert's
//   down matrix (and the shared one), computes d = bf16(ts_d Wd h) for all of
//   them, then the combine y = bf16(sum_j w_j d_j + d_shared) in rank order.
//   No atomics: the result is deterministic. Its weight rows are requested
//   before the PDL wait (the routing is final by then).
#include "flint_device.cuh"

namespace flint {
namespace {

constexpr int kCW = kConsumerWarps;
constexpr int kMaxDistinct = FLINT_MAX_TOKENS * FLINT_MAX_TOPK;

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
    const int tid = threadIdx.x, nt = blockDim.x;
    for (int i = tid; i < FLINT_MAX_EXPERTS / 32; i += nt) ri.bitmap[i] = 0;
    for (int i = tid; i < kMaxDistinct; i += nt) ri.dmask[i] = 0ull;
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

__device__ __forceinline__ uint32_t rank_bits(unsigned long long dm, int t) {
    return (uint32_t)((dm >> (8 * t)) & 0xFFull);
}

template <int W>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
    for (int off = W / 2; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

__device__ __forceinline__ float silu_f32(float g) { return g / (1.f + expf(-g)); }

// Token list of a bitmask, in ascending order, into compile-time slots.
template <int NT>
__device__ __forceinline__ void token_list(uint32_t mask, int (&tok)[NT]) {
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        tok[j] = mask ? __ffs(mask) - 1 : 0;
        mask &= mask - 1u;
    }
}

// FP32 activations of one token, lane-interleaved for `lanes` lanes per row:
// 16-byte word i (0..7) of the 32-value chunk cidx = gl + lanes * m sits at
// word index (m * 8 + i) * lanes + gl.
__device__ __forceinline__ int interleaved_word(int g, int lanes) {
    const int cidx = g >> 3, i = g & 7;
    return ((cidx / lanes) * 8 + i) * lanes + (cidx % lanes);
}

// Dot products of 8 decoded code pairs (16 values, one scale block) with 16
// activations (4 float4 words, stride `ws` float4 between words).
__device__ __forceinline__ float dot16(const float2* w, const float4* x, int ws) {
    float2 a = make_float2(0.f, 0.f), b = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float4 x4 = x[i * ws];
        a = __ffma2_rn(w[2 * i], make_float2(x4.x, x4.y), a);
        b = __ffma2_rn(w[2 * i + 1], make_float2(x4.z, x4.w), b);
    }
    const float2 s = __fadd2_rn(a, b);
    return s.x + s.y;
}

// ===========================================================================
// gate/up + SiLU (PAIR) or plain rows
// ===========================================================================
struct GateUpSmem {
    size_t route, xs, ring, stage, total;
};
template <bool PAIR>
__host__ __device__ inline GateUpSmem gate_up_layout(int T, int H, int nstages) {
    GateUpSmem L;
    L.route = 128;
    L.xs = align_up(L.route + sizeof(RouteInfo), 128);
    L.ring = align_up(L.xs + sizeof(float) * (size_t)T * H, 128);
    L.stage = (size_t)(PAIR ? 2 : 1) * kCW * nvfp4_row_stride(H);
    L.total = L.ring + (size_t)nstages * L.stage;
    return L;
}

// One item: rows grow (and urow) against the NT tokens of `mask`; lane t < n
// ends up holding the warp-reduced sums of token tok[t].
template <bool PAIR, int NT>
__device__ __forceinline__ void gate_up_item(const uint8_t* grow, const uint8_t* urow, int H, const float* xs,
                                             uint32_t mask, int lane, int (&tok)[8], float& gout, float& uout) {
    int tk[NT];
    token_list<NT>(mask, tk);
    const int n = __popc(mask);
    float ga[NT], ua[NT];
#pragma unroll
    for (int j = 0; j < NT; ++j) ga[j] = ua[j] = 0.f;
    const int nch = H >> 10;
    const float4* xs4 = reinterpret_cast<const float4*>(xs);
    for (int ch = 0; ch < nch; ++ch) {
        const int c = lane + 32 * ch;
        const uint4 gq = reinterpret_cast<const uint4*>(grow)[c];
        const float2 gs = ue4m3x2_to_float2(*reinterpret_cast<const uint16_t*>(grow + H / 2 + 2 * c));
        uint4 uq = make_uint4(0, 0, 0, 0);
        float2 us = make_float2(0.f, 0.f);
        if (PAIR) {
            uq = reinterpret_cast<const uint4*>(urow)[c];
            us = ue4m3x2_to_float2(*reinterpret_cast<const uint16_t*>(urow + H / 2 + 2 * c));
        }
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            float2 wg[8], wu[8];
            decode_word(hf ? gq.z : gq.x, wg);
            decode_word(hf ? gq.w : gq.y, wg + 4);
            if (PAIR) {
                decode_word(hf ? uq.z : uq.x, wu);
                decode_word(hf ? uq.w : uq.y, wu + 4);
            }
            const float sg = hf ? gs.y : gs.x, su = hf ? us.y : us.x;
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                if (j < n) {
                    const float4* xp = xs4 + (size_t)tk[j] * (H / 4) + (ch * 8 + hf * 4) * 32 + lane;
                    ga[j] = fmaf(sg, dot16(wg, xp, 32), ga[j]);
                    if (PAIR) ua[j] = fmaf(su, dot16(wu, xp, 32), ua[j]);
                }
            }
        }
    }
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        if (j < n) {
            const float gsum = group_sum<32>(ga[j]);
            const float usum = PAIR ? group_sum<32>(ua[j]) : 0.f;
            if (lane == j) {
                gout = gsum;
                uout = usum;
            }
            tok[j] = tk[j];
        }
    }
}

template <bool PAIR>
__global__ void __launch_bounds__(kGemvThreads, 1) gate_up_kernel(const GateUpArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int NS = a.nstages, H = a.H, T = a.T, I = a.I, Is = a.Is;
    const GateUpSmem L = gate_up_layout<PAIR>(T, H, NS);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + 4;
    RouteInfo& ri = *reinterpret_cast<RouteInfo*>(smem + L.route);
    float* xs = reinterpret_cast<float*>(smem + L.xs);
    uint8_t* ring = smem + L.ring;
    const int RS = (int)nvfp4_row_stride(H);
    const int half = kCW * RS;  // gate rows of one stage; up rows follow (PAIR)

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = blockIdx.x, G = gridDim.x;
    const int sp0 = (int)((long long)c * Is / G), sp1 = (int)((long long)(c + 1) * Is / G);
    const int n_sh = a.s_gu ? sp1 - sp0 : 0;

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kCW);
        }
        fence_mbar_init();
    }
    __syncthreads();
    // Before the wait: the shared expert's (or dense matrix's) rows do not
    // depend on the routing or on any earlier kernel.
    if (warp == kCW && lane == 0) {
        for (int st = 0; st < NS && st * kCW < n_sh; ++st) {
            const int i0 = st * kCW, n = min(n_sh - i0, kCW);
            const uint32_t bytes = (uint32_t)(n * RS);
            uint8_t* g = ring + (size_t)st * L.stage;
            mbar_expect_tx(&full[st], PAIR ? 2 * bytes : bytes);
            bulk_g2s(g, a.s_gu + (size_t)(sp0 + i0) * RS, bytes, &full[st]);
            if (PAIR) bulk_g2s(g + half, a.s_gu + (size_t)(Is + sp0 + i0) * RS, bytes, &full[st]);
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
    const int n_stages = (n_items + kCW - 1) / kCW;

    if (warp == kCW) {
        // ---------------- producer ----------------
        if (lane == 0) {
            for (int st = 0; st < n_stages; ++st) {
                const int b = st % NS;
                if (st >= NS &&
                    !mbar_wait_bounded(&empty[b], (uint32_t)(((st / NS) - 1) & 1), a.status, kStatusTimeoutGateUp))
                    break;
                uint8_t* g = ring + (size_t)b * L.stage;
                const int i0 = st * kCW, i1 = min(n_items, i0 + kCW);
                const bool with_shared = st >= NS;  // the first NS stages' shared rows are in flight
                for (int pass = 0; pass < 2; ++pass) {  // pass 0 counts bytes, pass 1 copies
                    uint32_t bytes = 0;
                    if (with_shared && i0 < n_sh) {
                        const int n = min(i1, n_sh) - i0;
                        if (pass) {
                            bulk_g2s(g, a.s_gu + (size_t)(sp0 + i0) * RS, n * RS, &full[b]);
                            if (PAIR) bulk_g2s(g + half, a.s_gu + (size_t)(Is + sp0 + i0) * RS, n * RS, &full[b]);
                        }
                        bytes += (PAIR ? 2u : 1u) * n * RS;
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
                            bulk_g2s(g + slot * RS, base + (size_t)p0 * RS, n * RS, &full[b]);
                            bulk_g2s(g + half + slot * RS, base + (size_t)(I + p0) * RS, n * RS, &full[b]);
                        }
                        bytes += 2u * n * RS;
                        slot += n;
                        q0 += n;
                    }
                    if (!pass) mbar_arrive_expect_tx(&full[b], bytes);
                }
            }
        }
        return;
    }

    // ---------------- consumers ----------------
    for (int i = tid; i < T * H / 4; i += kCW * 32) {  // x -> FP32, lane-interleaved
        const int t = i / (H / 4), g = i % (H / 4);
        const uint2 v = ld_cg(reinterpret_cast<const uint2*>(a.x + (size_t)t * H) + g);
        reinterpret_cast<float4*>(xs + (size_t)t * H)[interleaved_word(g, 32)] =
            make_float4(bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y));
    }
    named_sync(1, kCW * 32);

    for (int st = 0; st < n_stages; ++st) {
        const int b = st % NS;
        bool ok = mbar_wait_bounded(&full[b], (uint32_t)((st / NS) & 1), lane == 0 ? a.status : nullptr,
                                    kStatusTimeoutGateUp);
        if (!__all_sync(0xffffffffu, ok)) break;
        const int item = st * kCW + warp;
        if (item < n_items) {
            const uint8_t* grow = ring + (size_t)b * L.stage + warp * RS;
            const uint8_t* urow = grow + half;
            const bool shared_item = item < n_sh;
            int p, e = -1;
            unsigned long long dm = 0;
            uint32_t tmask;
            float tsg, tsu;
            if (shared_item) {
                p = sp0 + item;
                tmask = (1u << T) - 1u;
                tsg = a.s_ts[0];
                tsu = PAIR ? a.s_ts[1] : 0.f;
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
            const int n = __popc(tmask);
            int tok[8];
            float gsum = 0.f, usum = 0.f;
            if (n == 1)
                gate_up_item<PAIR, 1>(grow, urow, H, xs, tmask, lane, tok, gsum, usum);
            else if (n == 2)
                gate_up_item<PAIR, 2>(grow, urow, H, xs, tmask, lane, tok, gsum, usum);
            else if (n <= 4)
                gate_up_item<PAIR, 4>(grow, urow, H, xs, tmask, lane, tok, gsum, usum);
            else
                gate_up_item<PAIR, 8>(grow, urow, H, xs, tmask, lane, tok, gsum, usum);
            if (lane < n) {
                int t = tok[0];
#pragma unroll
                for (int j = 1; j < 8; ++j)
                    if (lane == j) t = tok[j];
                const float g = bf16_round_f32(tsg * gsum);
                if (!PAIR) {
                    a.h_shared[(size_t)t * Is + p] = f32_to_bf16_bits(g);
                } else {
                    const float u = bf16_round_f32(tsu * usum);
                    const uint16_t h = f32_to_bf16_bits(silu_f32(g) * u);
                    if (shared_item) {
                        a.h_shared[(size_t)t * Is + p] = h;
                    } else {
                        const uint32_t ranks = rank_bits(dm, t);
                        for (int j = 0; j < a.k; ++j)
                            if ((ranks >> j) & 1u) a.h_routed[((size_t)t * a.k + j) * I + p] = h;
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[b]);
    }
}

// ===========================================================================
// down + combine
// ===========================================================================
struct DownSmem {
    size_t route, w, dval, hr, hs, ring, stage, total;
};
__host__ __device__ inline DownSmem down_layout(const DownArgs& a) {
    DownSmem L;
    L.route = 128;
    L.w = align_up(L.route + sizeof(RouteInfo), 128);
    L.dval = align_up(L.w + sizeof(float) * kMaxDistinct, 128);
    L.hr = align_up(L.dval + sizeof(float) * FLINT_MAX_TOKENS * (FLINT_MAX_TOPK + 1) * (size_t)a.rows_max, 128);
    L.hs = align_up(L.hr + sizeof(float) * (size_t)a.T * a.k * a.I, 128);
    L.ring = align_up(L.hs + sizeof(float) * (size_t)a.T * a.Is, 128);
    L.stage = (size_t)kCW * a.slot_bytes;
    L.total = L.ring + (size_t)a.nstages * L.stage;
    return L;
}

// One task: rows ra (and rb = ra + 1) of a unit's slice against NT tokens.
// Lanes of one LPR-group split the row's chunks; every lane does two rows.
template <int LPR, int NT>
__device__ __forceinline__ void down_task(const uint8_t* row_a, const uint8_t* row_b, bool has_b, int K,
                                          const float* const (&hv)[NT], int n, int gl, float (&out_a)[8],
                                          float (&out_b)[8]) {
    float aa[NT], ab[NT];
#pragma unroll
    for (int j = 0; j < NT; ++j) aa[j] = ab[j] = 0.f;
    const int cpl = K / 32 / LPR;
    for (int m = 0; m < cpl; ++m) {
        const int cidx = gl + LPR * m;
        const uint4 qa = reinterpret_cast<const uint4*>(row_a)[cidx];
        const uint4 qb = has_b ? reinterpret_cast<const uint4*>(row_b)[cidx] : make_uint4(0, 0, 0, 0);
        const float2 sa = ue4m3x2_to_float2(*reinterpret_cast<const uint16_t*>(row_a + K / 2 + 2 * cidx));
        const float2 sb =
            has_b ? ue4m3x2_to_float2(*reinterpret_cast<const uint16_t*>(row_b + K / 2 + 2 * cidx)) : make_float2(0, 0);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            float2 wa[8], wb[8];
            decode_word(hf ? qa.z : qa.x, wa);
            decode_word(hf ? qa.w : qa.y, wa + 4);
            decode_word(hf ? qb.z : qb.x, wb);
            decode_word(hf ? qb.w : qb.y, wb + 4);
            const float s_a = hf ? sa.y : sa.x, s_b = hf ? sb.y : sb.x;
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                if (j < n) {
                    const float4* xp = reinterpret_cast<const float4*>(hv[j]) + (m * 8 + hf * 4) * LPR + gl;
                    aa[j] = fmaf(s_a, dot16(wa, xp, LPR), aa[j]);
                    ab[j] = fmaf(s_b, dot16(wb, xp, LPR), ab[j]);
                }
            }
        }
    }
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        if (j < n) {
            out_a[j] = group_sum<LPR>(aa[j]);
            out_b[j] = group_sum<LPR>(ab[j]);
        }
    }
}

template <int LPR>
__global__ void __launch_bounds__(kGemvThreads, 1) down_kernel(const DownArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const DownSmem L = down_layout(a);
    const int NS = a.nstages;
    const int T = a.T, k = a.k, H = a.H, I = a.I, Is = a.Is, RM = a.rows_max;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + 4;
    RouteInfo& ri = *reinterpret_cast<RouteInfo*>(smem + L.route);
    float* wsm = reinterpret_cast<float*>(smem + L.w);
    float* dval = reinterpret_cast<float*>(smem + L.dval);  // [t][j (k = shared)][row]
    float* hr = reinterpret_cast<float*>(smem + L.hr);      // [t*k + j][I], lane-interleaved
    float* hs = reinterpret_cast<float*>(smem + L.hs);      // [t][Is], lane-interleaved
    uint8_t* ring = smem + L.ring;
    constexpr int kRowsPerTask = 2 * (32 / LPR);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = blockIdx.x, G = gridDim.x;
    const int n0 = (int)((long long)c * H / G), n1 = (int)((long long)(c + 1) * H / G), nr = n1 - n0;
    const int RSr = (int)nvfp4_row_stride(I), RSs = Is ? (int)nvfp4_row_stride(Is) : 0;
    if (nr == 0) return;  // more CTAs than output rows: nothing to copy or compute

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kCW);
        }
        fence_mbar_init();
    }
    // The routing is final before this kernel can start: the gate/up kernel
    // triggers its dependents only after its own wait on the router.
    build_route_info(ri, a.ids, T, k, a.E, a.status);  // (contains __syncthreads)
    const int D = ri.D;
    const bool has_sh = a.s_down != nullptr;
    const int n_units = D + (has_sh ? 1 : 0);
    const int tpu = (nr + kRowsPerTask - 1) / kRowsPerTask;  // tasks per unit
    const int n_tasks = n_units * tpu;
    const int n_stages = (n_tasks + kCW - 1) / kCW;

    if (warp == kCW) {
        // ---------------- producer: weights do not depend on h ----------------
        if (lane == 0) {
            for (int st = 0; st < n_stages; ++st) {
                const int b = st % NS;
                if (st >= NS &&
                    !mbar_wait_bounded(&empty[b], (uint32_t)(((st / NS) - 1) & 1), a.status, kStatusTimeoutDown))
                    break;
                const int q0 = st * kCW, q1 = min(n_tasks, q0 + kCW);
                uint32_t bytes = 0;
                for (int q = q0; q < q1; ++q) {
                    const int u = q / tpu, r0 = (q % tpu) * kRowsPerTask, r1 = min(nr, r0 + kRowsPerTask);
                    bytes += (uint32_t)((r1 - r0) * (u < D ? RSr : RSs));
                }
                mbar_arrive_expect_tx(&full[b], bytes);
                for (int q = q0; q < q1; ++q) {
                    const int u = q / tpu, r0 = (q % tpu) * kRowsPerTask, r1 = min(nr, r0 + kRowsPerTask);
                    uint8_t* dst = ring + (size_t)b * L.stage + (size_t)(q - q0) * a.slot_bytes;
                    if (u < D)
                        bulk_g2s(dst, a.down + ((size_t)ri.dlist[u] * H + n0 + r0) * RSr, (uint32_t)((r1 - r0) * RSr),
                                 &full[b]);
                    else
                        bulk_g2s(dst, a.s_down + (size_t)(n0 + r0) * RSs, (uint32_t)((r1 - r0) * RSs), &full[b]);
                }
            }
        }
        pdl_wait();
        pdl_launch_dependents();
        return;
    }

    // ---------------- consumers ----------------
    pdl_wait();  // h comes from the gate/up kernel
    pdl_launch_dependents();
    {  // h -> FP32 in shared memory, lane-interleaved for LPR lanes per row
        const int gr = I / 4, gsh = Is / 4;
        for (int i = tid; i < T * k * gr; i += kCW * 32) {
            const int v = i / gr, g = i % gr;
            const uint2 hv = ld_cg(reinterpret_cast<const uint2*>(a.h_routed + (size_t)v * I) + g);
            reinterpret_cast<float4*>(hr + (size_t)v * I)[interleaved_word(g, LPR)] =
                make_float4(bf16_lo(hv.x), bf16_hi(hv.x), bf16_lo(hv.y), bf16_hi(hv.y));
        }
        if (has_sh) {
            for (int i = tid; i < T * gsh; i += kCW * 32) {
                const int v = i / gsh, g = i % gsh;
                const uint2 hv = ld_cg(reinterpret_cast<const uint2*>(a.h_shared + (size_t)v * Is) + g);
                reinterpret_cast<float4*>(hs + (size_t)v * Is)[interleaved_word(g, LPR)] =
                    make_float4(bf16_lo(hv.x), bf16_hi(hv.x), bf16_lo(hv.y), bf16_hi(hv.y));
            }
        }
        for (int i = tid; i < T * k; i += kCW * 32) wsm[i] = ld_cg(a.w + i);
    }
    named_sync(1, kCW * 32);

    const int grp = lane / LPR, gl = lane % LPR;
    for (int st = 0; st < n_stages; ++st) {
        const int b = st % NS;
        bool ok = mbar_wait_bounded(&full[b], (uint32_t)((st / NS) & 1), lane == 0 ? a.status : nullptr,
                                    kStatusTimeoutDown);
        if (!__all_sync(0xffffffffu, ok)) break;
        const int q = st * kCW + warp;
        if (q < n_tasks) {
            const int u = q / tpu, r0 = (q % tpu) * kRowsPerTask, r1 = min(nr, r0 + kRowsPerTask);
            const bool sh = u >= D;
            const int K = sh ? Is : I, RS = sh ? RSs : RSr;
            const uint8_t* slot = ring + (size_t)b * L.stage + (size_t)warp * a.slot_bytes;
            const int ra = r0 + 2 * grp;  // this group's two rows
            const bool has_a = ra < r1, has_b = ra + 1 < r1;
            const uint8_t* row_a = slot + (size_t)(has_a ? ra - r0 : 0) * RS;
            const uint8_t* row_b = slot + (size_t)(has_b ? ra + 1 - r0 : 0) * RS;
            unsigned long long dm = 0;
            uint32_t tmask;
            float tsd;
            if (sh) {
                tmask = (1u << T) - 1u;
                tsd = a.s_ts[2];
            } else {
                dm = ri.dmask[u];
                tmask = token_mask(dm);
                tsd = a.ts[3 * ri.dlist[u] + 2];
            }
            const int n = __popc(tmask);
            int tok[8];
            token_list<8>(tmask, tok);
            float oa[8], ob[8];
#define FLINT_DOWN_CALL(NTV)                                                                                   \
    {                                                                                                          \
        const float* hv[NTV];                                                                                  \
        _Pragma("unroll") for (int j = 0; j < NTV; ++j) {                                                      \
            const int t = tok[j];                                                                              \
            hv[j] = sh ? hs + (size_t)t * Is : hr + ((size_t)t * k + (__ffs(rank_bits(dm, t) | 0x100u) - 1)) * I; \
        }                                                                                                      \
        down_task<LPR, NTV>(row_a, row_b, has_b, K, hv, n, gl, oa, ob);                                       \
    }
            if (n == 1) FLINT_DOWN_CALL(1)
            else if (n == 2) FLINT_DOWN_CALL(2)
            else if (n <= 4) FLINT_DOWN_CALL(4)
            else FLINT_DOWN_CALL(8)
#undef FLINT_DOWN_CALL
            if (gl == 0 && has_a) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (j < n) {
                        const int t = tok[j];
                        const float da = bf16_round_f32(tsd * oa[j]);
                        const float db = bf16_round_f32(tsd * ob[j]);
                        if (sh) {
                            dval[((size_t)t * (k + 1) + k) * RM + ra] = da;
                            if (has_b) dval[((size_t)t * (k + 1) + k) * RM + ra + 1] = db;
                        } else {
                            const uint32_t ranks = rank_bits(dm, t);
                            for (int jj = 0; jj < k; ++jj) {
                                if ((ranks >> jj) & 1u) {
                                    dval[((size_t)t * (k + 1) + jj) * RM + ra] = da;
                                    if (has_b) dval[((size_t)t * (k + 1) + jj) * RM + ra + 1] = db;
                                }
                            }
                        }
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[b]);
    }
    named_sync(1, kCW * 32);
    // combine, in rank order then the shared expert
    for (int i = tid; i < T * nr; i += kCW * 32) {
        const int t = i / nr, r = i % nr;
        float acc = 0.f;
        for (int j = 0; j < k; ++j)
            if (ri.ids[t * k + j] >= 0) acc = fmaf(wsm[t * k + j], dval[((size_t)t * (k + 1) + j) * RM + r], acc);
        if (has_sh) acc += dval[((size_t)t * (k + 1) + k) * RM + r];
        a.y[(size_t)t * H + n0 + r] = f32_to_bf16_bits(acc);
    }
}

template <typename K, typename A>
cudaError_t launch_ex(K kernel, const A& args, unsigned grid, size_t smem, bool pdl, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kGemvThreads);
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

size_t gate_up_smem_bytes(const GateUpArgs& a, bool pair) {
    return pair ? gate_up_layout<true>(a.T, a.H, a.nstages).total : gate_up_layout<false>(a.T, a.H, a.nstages).total;
}
size_t gate_up_stage_bytes(int H, bool pair) { return (size_t)(pair ? 2 : 1) * kCW * nvfp4_row_stride(H); }
size_t down_smem_bytes(const DownArgs& a) { return down_layout(a).total; }
size_t down_stage_bytes(const DownArgs& a) { return (size_t)kCW * a.slot_bytes; }

cudaError_t launch_gate_up(const GateUpArgs& a, bool pair, const DevInfo& d, bool pdl, cudaStream_t s) {
    static int cfg_pair = -1, cfg_rows = -1;
    cudaError_t e = pair ? configure_smem(gate_up_kernel<true>, d, cfg_pair)
                         : configure_smem(gate_up_kernel<false>, d, cfg_rows);
    if (e != cudaSuccess) return e;
    const size_t smem = gate_up_smem_bytes(a, pair);
    return pair ? launch_ex(gate_up_kernel<true>, a, (unsigned)d.sm_count, smem, pdl, s)
                : launch_ex(gate_up_kernel<false>, a, (unsigned)d.sm_count, smem, pdl, s);
}

cudaError_t launch_down(const DownArgs& a, const DevInfo& d, bool pdl, cudaStream_t s) {
    static int cfg8 = -1, cfg16 = -1, cfg32 = -1;
    const size_t smem = down_smem_bytes(a);
    cudaError_t e;
    switch (a.lpr) {
        case 8:
            if ((e = configure_smem(down_kernel<8>, d, cfg8)) != cudaSuccess) return e;
            return launch_ex(down_kernel<8>, a, (unsigned)d.sm_count, smem, pdl, s);
        case 16:
            if ((e = configure_smem(down_kernel<16>, d, cfg16)) != cudaSuccess) return e;
            return launch_ex(down_kernel<16>, a, (unsigned)d.sm_count, smem, pdl, s);
        default:
            if ((e = configure_smem(down_kernel<32>, d, cfg32)) != cudaSuccess) return e;
            return launch_ex(down_kernel<32>, a, (unsigned)d.sm_count, smem, pdl, s);
    }
}

}  // namespace flint
