// layer.cu -- the whole decode step of one MoE layer in one cooperative
// kernel: router GEMV + sigmoid top-k, gate/up + SiLU, down + weighted
// combine with the shared expert.
//
// "Day-0 Support for Flint on vLLM", section "Optimizations": the small-batch
// MoE path is a short chain of kernels whose expert GEMVs read only the
// selected experts' weights, with routing and the combine fused into the
// neighbouring GEMVs. Here the chain is one launch: at batch 1 to 8 the
// layer moves 13-80 MB, a few microseconds of HBM time, so the fixed cost of
// each kernel boundary (launch, prologue, drain) is a large share; inside one
// kernel the three steps meet at two grid-wide barriers instead.
//
// One CTA per SM, all resident (cooperative launch):
//   0. Before the PDL wait: this CTA's router rows, its slice of the shared
//      expert's gate/up pairs and its slice of the shared expert's down rows
//      are copied into shared memory (static weights).
//   1. x is staged (chunk-scaled f16, for gate/up); for a pre-norm block
//      every CTA first computes x = rmsnorm(r + y_prev) itself from the
//      residual stream and writes its share of the new residual out. The
//      CTA's router logits are computed in FP32 from the staged x and bf16
//      router rows; their sigmoid scores go to the workspace. Grid barrier.
//   2. Every CTA reads all scores and selects the top-k of every token itself
//      (one warp per token, straight from L2), so no second barrier is needed
//      to share the routing; CTA 0 also writes ids and weights out.
//   3. gate/up + SiLU as in gate_up_kernel: the CTA's share of the routed
//      pairs through per-warp cp.async rings, its shared-expert pairs from
//      shared memory; h goes to the workspace. Grid barrier.
//   4. down + combine as in down_kernel: h is staged, the CTA's output rows of
//      every selected expert stream through per-warp rings (the shared
//      expert's rows are already resident), then y = bf16(sum_j w_j d_j +
//      d_shared) in rank order.
#include "expert_common.cuh"
#include "router_common.cuh"

namespace flint {
namespace {

constexpr int kLW = kLayerWarps;
constexpr int kLT = kLayerThreads;

// Small per-CTA arrays: tensor scales (gate, up) of the distinct experts then
// of the shared expert; down scales of the units; combine weights; ids.
struct LayerSmall {
    uint64_t dbar;  // completion of the prefetched down rows
    uint64_t rbar[kLayerWarps * 4];  // the gate/up ring slots of each warp (up to 4)
    float tss[2 * kMaxDistinct + 2];
    float tsd[kMaxDistinct + 1];
    float w[kMaxDistinct];
    int32_t ids[kMaxDistinct];
    float ninv[FLINT_MAX_TOKENS];  // per-token 1 / rms of the normalised input
};

// Shared memory, by lifetime:
//   persistent: routing view, small arrays, the shared expert's down rows;
//   phases 0-3 (region U1): staged x and its chunk scales (and the norm's
//     per-chunk sums of squares when the input is normalised here), the shared
//     expert's gate/up pairs, then one of: router rows (phases 0-1), raw
//     gate/up sums + the gate/up rings (phase 3);
//   phase 4 (region U4, over U1): staged h and its chunk scales, d values,
//     the down rings;
//   the prefetched down rows (a.dpre), beside both.
struct LayerSmem {
    size_t ri, small, shdn, U;
    size_t xs, csc, nred, shgu, V;
    size_t wrows;
    size_t resg, resu, ring3;
    size_t hr, hs, csr, css, dval, ring4;
    size_t dpre;
    size_t total;
};

__host__ __device__ inline LayerSmem layer_layout(const LayerArgs& a) {
    LayerSmem L;
    const size_t RS = (size_t)nvfp4_row_stride(a.H), RSs = a.Is ? (size_t)nvfp4_row_stride(a.Is) : 0;
    const size_t T = a.T, H = a.H;
    L.ri = 0;
    L.small = align_up(sizeof(RouteInfo), 128);
    L.shdn = align_up(L.small + sizeof(LayerSmall), 128);
    L.U = align_up(L.shdn + (size_t)a.rows_max * RSs, 128);
    // U1
    L.xs = L.U;
    L.csc = align_up(L.xs + 2 * T * H, 128);
    L.nred = align_up(L.csc + sizeof(float) * T * (H / 32), 128);
    L.shgu = align_up(L.nred + (a.norm.r ? sizeof(float) * T * (H / 32) : 0), 128);
    L.V = align_up(L.shgu + 2 * (size_t)a.shp * RS, 128);
    L.wrows = L.V;
    L.resg = L.V;
    L.resu = align_up(L.resg + sizeof(float) * (size_t)a.res_items * T, 128);
    L.ring3 = align_up(L.resu + sizeof(float) * (size_t)a.res_items * T, 128);
    size_t end1 = L.ring3 + (size_t)kLW * a.ns3 * 2 * RS;
    const size_t e_rows = L.wrows + 2 * (size_t)a.rpc * H;
    if (end1 < e_rows) end1 = e_rows;
    // U4
    L.hr = L.U;
    L.hs = align_up(L.hr + 2 * T * a.k * a.I, 128);
    L.csr = align_up(L.hs + 2 * T * a.Is, 128);
    L.css = align_up(L.csr + sizeof(float) * T * a.k * (a.I / 32), 128);
    L.dval = align_up(L.css + sizeof(float) * T * (a.Is / 32), 128);
    L.ring4 = align_up(L.dval + sizeof(float) * T * (a.k + 1) * a.rows_max, 128);
    const size_t end4 = L.ring4 + (size_t)kLW * a.ns4 * a.slot4;
    L.total = end1 > end4 ? end1 : end4;
    L.dpre = align_up(L.total, 128);
    if (a.dpre) {
        const size_t units = (size_t)(a.T * a.k < a.E ? a.T * a.k : a.E);
        L.total = L.dpre + units * a.rows_max * (size_t)nvfp4_row_stride(a.I);
    }
    return L;
}

// All threads of the CTA copy `bytes` (a multiple of 16) from src to dst with
// 16-byte cp.async (no commit).
__device__ __forceinline__ void block_copy_async(void* dst, const void* src, size_t bytes) {
    uint8_t* d = static_cast<uint8_t*>(dst);
    const uint8_t* s = static_cast<const uint8_t*>(src);
    for (size_t o = 16 * (size_t)threadIdx.x; o < bytes; o += 16 * (size_t)kLT) cp_async16(d + o, s + o);
}

// NORM: the input is rmsnorm(r + y_prev) of the residual stream (a.norm), not
// a.x. Two instantiations, so that the plain layer carries none of the norm's
// code (measured: the never-taken branch alone cost 3-4 us at T = 8).
template <bool NORM>
__global__ void __launch_bounds__(kLT, 1) layer_kernel(const LayerArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const LayerSmem L = layer_layout(a);
    const int T = a.T, H = a.H, E = a.E, k = a.k, I = a.I, Is = a.Is, RM = a.rows_max;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = blockIdx.x, G = gridDim.x;
    RouteInfo& ri = *reinterpret_cast<RouteInfo*>(smem + L.ri);
    LayerSmall& sm = *reinterpret_cast<LayerSmall*>(smem + L.small);
    uint4* xh = reinterpret_cast<uint4*>(smem + L.xs);
    float* csc = reinterpret_cast<float*>(smem + L.csc);
    const uint16_t* wrows = reinterpret_cast<const uint16_t*>(smem + L.wrows);
    uint8_t* shgu = smem + L.shgu;
    uint8_t* shdn = smem + L.shdn;
    const int RS = (int)nvfp4_row_stride(H), RSr = (int)nvfp4_row_stride(I);
    const int RSs = Is ? (int)nvfp4_row_stride(Is) : 0;
    const bool has_sh = a.s_gu != nullptr;

    // This CTA's router rows, shared-expert pairs and output rows.
    const int r0 = c * a.rpc, nrr = max(0, min(a.rpc, E - r0));
    const int sp0 = (int)((unsigned)c * (unsigned)Is / (unsigned)G);
    const int n_sh = has_sh ? (int)((unsigned)(c + 1) * (unsigned)Is / (unsigned)G) - sp0 : 0;
    const int n0 = (int)((unsigned)c * (unsigned)H / (unsigned)G);
    const int nr = (int)((unsigned)(c + 1) * (unsigned)H / (unsigned)G) - n0;

    // ---- 0: static weights, before the PDL wait ------------------------------------
    block_copy_async(smem + L.wrows, a.wr + (size_t)r0 * H, (size_t)nrr * H * 2);
    if (n_sh > 0) {
        block_copy_async(shgu, a.s_gu + (size_t)sp0 * RS, (size_t)n_sh * RS);
        block_copy_async(shgu + (size_t)a.shp * RS, a.s_gu + (size_t)(Is + sp0) * RS, (size_t)n_sh * RS);
        block_copy_async(shdn, a.s_down + (size_t)n0 * RSs, (size_t)nr * RSs);
    }
    cp_async_commit();
    if (tid < 2 * kMaxDistinct + 2) sm.tss[tid] = 0.f;
    if (tid == 0) mbar_init(&sm.dbar, 1);
    if (tid < kLW * 4) mbar_init(&sm.rbar[tid], 1);
    if (tid <= kLW * 4) fence_mbar_init();

    pdl_wait();  // x comes from the previous kernel

    // ---- 1: stage x (or the norm of the residual stream); this CTA's router scores --
    const StageSrc xsrc[1] = {{a.x, xh, csc, T, H}};
    if constexpr (NORM)
        stage_norm_f16(a.norm, xsrc[0], reinterpret_cast<float*>(smem + L.nred), sm.ninv, c, G);
    else
        stage_f16<false>(xsrc, [] {});
    cp_async_wait<0>();
    __syncthreads();
    // logits from the staged (exact, chunk-scaled f16) x: lane l takes the
    // 32-value chunks l, l + 32, ...; each chunk's FP32 partial sum is
    // multiplied back by its power-of-two scale
    for (int q = warp; q < nrr * T; q += kLW) {
        const int r = q / T, t = q - r * T;
        const uint4* xb = xh + (size_t)t * (H / 8) + lane;
        const float* cb = csc + (size_t)t * (H / 32) + lane;
        const uint4* wv = reinterpret_cast<const uint4*>(wrows + (size_t)r * H);
        float v = 0.f;
        for (int m = 0; m < H / 1024; ++m) {
            const int ch = lane + 32 * m;
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const uint4 xv = xb[(m * 4 + w) * 32], wq = wv[4 * ch + w];
                const uint32_t xa[4] = {xv.x, xv.y, xv.z, xv.w}, wa[4] = {wq.x, wq.y, wq.z, wq.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 xf = __half22float2(*reinterpret_cast<const __half2*>(&xa[i]));
                    s0 = fmaf(bf16_lo(wa[i]), xf.x, s0);
                    s1 = fmaf(bf16_hi(wa[i]), xf.y, s1);
                }
            }
            v = fmaf(cb[32 * m], s0 + s1, v);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        // the sigmoid score (its bits), once per logit in the grid
        if (lane == 0) reinterpret_cast<uint32_t*>(a.logits)[(size_t)t * E + r0 + r] = sigmoid_score(v, a.bias, r0 + r);
    }
    if (!grid_sync(a.bar_ticket, a.status, kStatusTimeoutLayer)) return;

    // ---- 2: top-k of every token, in every CTA ------------------------------------
    float* wsel = sm.w;
    {
        if (warp < T) {
            const uint32_t* sc = reinterpret_cast<const uint32_t*>(a.logits) + (size_t)warp * E;
            if (E <= 256)
                topk_warp<8, true>(sc, E, k, lane, sm.ids + warp * k, wsel + warp * k);
            else
                topk_warp<FLINT_MAX_EXPERTS / 32, true>(sc, E, k, lane, sm.ids + warp * k, wsel + warp * k);
        }
        __syncthreads();
    }
    if (c == 0 && tid < T * k) {
        a.ids[tid] = sm.ids[tid];
        a.weights[tid] = wsel[tid];
    }
    build_route_info<true>(ri, sm.ids, T, k, E, a.status);
    const int D = ri.D;
    // The routing is known: this CTA's down rows of every selected expert can
    // stream in now, behind gate/up, when they fit (one bulk copy per expert).
    uint8_t* dpre = smem + L.dpre;
    if (a.dpre && nr > 0 && warp == 0) {
        if (lane == 0) mbar_arrive_expect_tx(&sm.dbar, (uint32_t)(D * nr * RSr));
        __syncwarp();
        for (int u = lane; u < D; u += 32)
            bulk_g2s(dpre + (size_t)u * nr * RSr, a.down + ((size_t)ri.dlist[u] * H + n0) * RSr,
                     (uint32_t)(nr * RSr), &sm.dbar);
    }

    // ---- 3: gate/up + SiLU ---------------------------------------------------------
    {
        float* resg = reinterpret_cast<float*>(smem + L.resg);
        float* resu = reinterpret_cast<float*>(smem + L.resu);
        const int NSW = a.ns3;
        uint8_t* ring = smem + L.ring3 + (size_t)warp * NSW * 2 * RS;
        // The routed pairs in list order (pair q = d I + p: row p of expert
        // dlist[d]) are dealt out round-robin: CTA c takes pairs c, c + G, ...
        // (its local items 0, 1, ...) and its warp w the local items w, w + kLW,
        // .... An expert that several tokens chose costs more per pair, and
        // dealing spreads its rows evenly over the CTAs and warps; contiguous
        // ranges left a few CTAs ~1.5x the mean work at T = 8, and the grid
        // barrier after this phase waits for the slowest.
        const int RP = D * I;
        const int nl = c < RP ? (RP - c + G - 1) / G : 0;
        const int n_items_w = nl > warp ? (nl - warp + kLW - 1) / kLW : 0;
        // The ring is fed by bulk copies (the copy engine, one lane per warp):
        // the gate and up rows of an item land in its slot and complete on the
        // slot's mbarrier. Against all 32 lanes issuing 16-byte cp.async this
        // frees issue slots in a phase bound by instruction latency and issue.
        uint64_t* rbar = sm.rbar + warp * 4;
        auto issue = [&](int m) {  // local item warp + m kLW into slot m % NSW
            if (lane == 0) {
                const int q = c + (warp + m * kLW) * G, d = q / I, p = q - d * I;
                const uint8_t* g = a.gu + ((size_t)ri.dlist[d] * 2 * I + p) * RS;
                uint8_t* slot = ring + (size_t)(m % NSW) * 2 * RS;
                uint64_t* bar = rbar + m % NSW;
                fence_proxy_async_smem();  // the slot's earlier reads come first
                mbar_arrive_expect_tx(bar, 2u * (uint32_t)RS);
                bulk_g2s(slot, g, (uint32_t)RS, bar);
                bulk_g2s(slot + RS, g + (size_t)I * RS, (uint32_t)RS, bar);
            }
        };
        // scales first, then this warp's first copies
        float tsv = 0.f;
        if (tid < 2 * D) tsv = ld_cg(a.ts + 3 * ri.dlist[tid >> 1] + (tid & 1));
        else if (tid < 2 * D + 2 && has_sh) tsv = ld_cg(a.s_ts + tid - 2 * D);
        float tdv = 0.f;
        if (tid >= 256 && tid < 256 + D) tdv = ld_cg(a.ts + 3 * ri.dlist[tid - 256] + 2);
        else if (tid == 256 + D && has_sh) tdv = ld_cg(a.s_ts + 2);
        for (int m = 0; m < NSW && m < n_items_w; ++m) issue(m);
        if (tid < 2 * D + 2) sm.tss[tid] = tsv;
        if (tid >= 256 && tid <= 256 + D) sm.tsd[tid - 256] = tdv;
        // The warp's work, in one loop so that the pass code is inlined once:
        // first its shared-expert units (resident; one per (pair, two tokens),
        // spread over the warps from the last one: every token reads every
        // shared row, so at T = 8 a shared pair is four units), then its routed
        // items from the ring.
        const int ntp = (T + 1) >> 1, su0 = kLW - 1 - warp;
        const int n_su_w = su0 < n_sh * ntp ? (n_sh * ntp - su0 + kLW - 1) / kLW : 0;
        int m_fail = -1;  // the item whose copy never landed
        for (int it = 0; it < n_su_w + n_items_w; ++it) {
            const int m = it - n_su_w;
            const uint8_t *grow, *urow;
            uint32_t tm;
            int slot;  // row of resg / resu
            if (m < 0) {
                const int q = su0 + it * kLW, i = q / ntp, t0 = 2 * (q - i * ntp);
                grow = shgu + (size_t)i * RS;
                urow = grow + (size_t)a.shp * RS;
                tm = (t0 + 1 < T ? 3u : 1u) << t0;  // t0 alone at an odd T
                slot = i;
            } else {
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(rbar + m % NSW, (uint32_t)(m / NSW) & 1u, a.status,
                                                               kStatusTimeoutLayer))) {
                    m_fail = m;
                    break;
                }
                grow = ring + (size_t)(m % NSW) * 2 * RS;
                urow = grow + RS;
                const int li = warp + m * kLW;
                tm = ri.tmask[(c + li * G) / I];
                slot = n_sh + li;
            }
            gate_up_item<true>(grow, urow, H, xh, csc, tm, lane, resg + slot * T, resu + slot * T);
            if (m >= 0 && m + NSW < n_items_w) {
                __syncwarp();
                issue(m + NSW);
            }
        }
        if (__syncthreads_or(m_fail >= 0)) {
            // a copy timed out: let this warp's copies still in flight land
            // (bounded), then stop
            for (int mm = max(m_fail, 0); m_fail >= 0 && mm < min(n_items_w, m_fail + NSW); ++mm)
                mbar_wait_bounded(rbar + mm % NSW, (uint32_t)(mm / NSW) & 1u, nullptr, 0);
            return;
        }
        const int n_items = n_sh + nl;
        for (int e = tid; e < n_items * T; e += kLT) {
            const int t = e / n_items, i = e - t * n_items;
            float tsg, tsu;
            int pp;
            uint32_t ranks = 0;
            if (i < n_sh) {
                pp = sp0 + i;
                tsg = sm.tss[2 * D];
                tsu = sm.tss[2 * D + 1];
            } else {
                const int q = c + (i - n_sh) * G, dd = q / I;
                pp = q - dd * I;
                ranks = rank_bits(ri.dmask[dd], t);
                if (!ranks) continue;
                tsg = sm.tss[2 * dd];
                tsu = sm.tss[2 * dd + 1];
            }
            const float g = bf16_round_f32(tsg * resg[i * T + t]);
            const float u = bf16_round_f32(tsu * resu[i * T + t]);
            const uint16_t out = f32_to_bf16_bits(silu_f32(g) * u);
            if (i < n_sh) {
                a.h_shared[(size_t)t * Is + pp] = out;
            } else {
                for (int j = 0; j < k; ++j)
                    if ((ranks >> j) & 1u) a.h_routed[((size_t)t * k + j) * I + pp] = out;
            }
        }
    }
    // ---- 4: down + combine ---------------------------------------------------------
    // The down rows depend on the routing only. This CTA's first ring copies
    // are issued between its arrival at the grid barrier and its wait (the
    // regions of phases 0-3 are dead once the epilogue is done), so that their
    // latency overlaps the barrier.
    const int NSW = a.ns4, RG = a.rg;
    uint8_t* ring = smem + L.ring4 + (size_t)warp * NSW * a.slot4;
    const int ngr = (nr + RG - 1) / RG;
    const int n_tasks = D * ngr;  // routed; the shared expert's groups are resident
    const int my_tasks = a.dpre ? 0 : (n_tasks > warp ? (n_tasks - warp + kLW - 1) / kLW : 0);
    auto issue = [&](int kk) {
        const int q = warp + kk * kLW, u = q / ngr, r0g = (q - u * ngr) * RG, r1g = min(nr, r0g + RG);
        uint8_t* dst = ring + (size_t)(kk % NSW) * a.slot4;
        warp_copy_async(dst, a.down + ((size_t)ri.dlist[u] * H + n0 + r0g) * RSr, (r1g - r0g) * RSr, lane);
        cp_async_commit();
    };
    const unsigned long long target = grid_arrive(a.bar_ticket);
    for (int kk = 0; kk < NSW; ++kk) {
        if (kk < my_tasks)
            issue(kk);
        else
            cp_async_commit();
    }
    if (!grid_wait(a.bar_ticket, target, a.status, kStatusTimeoutLayer)) {
        cp_async_wait<0>();
        return;
    }
    pdl_launch_dependents();
    if (nr == 0) return;
    {
        uint4* hr = reinterpret_cast<uint4*>(smem + L.hr);
        uint4* hs = reinterpret_cast<uint4*>(smem + L.hs);
        float* csr = reinterpret_cast<float*>(smem + L.csr);
        float* css = reinterpret_cast<float*>(smem + L.css);
        float* dval = reinterpret_cast<float*>(smem + L.dval);
        const StageSrc hsrc[2] = {{a.h_routed, hr, csr, T * k, I}, {a.h_shared, hs, css, has_sh ? T : 0, Is ? Is : 32}};
        stage_f16<true>(hsrc, [] {});
        __syncthreads();
        // One task: rows [r0g, r1g) of unit u (u < D routed, from `rows`; u == D shared).
        auto task = [&](int u, int r0g, int r1g, const uint8_t* rows, uint32_t rest) {
            const bool sh = u >= D;
            const int K = sh ? Is : I, RSu = sh ? RSs : RSr;
            const unsigned long long dm = sh ? 0ull : ri.dmask[u];
            const float tsd = sm.tsd[u];
            auto vec = [&](int t, const uint4*& h, const float*& cs) {
                if (sh) {
                    h = hs + (size_t)t * (Is / 8);
                    cs = css + (size_t)t * (Is / 32);
                } else {
                    const int j = __ffs(rank_bits(dm, t)) - 1;
                    h = hr + ((size_t)t * k + j) * (I / 8);
                    cs = csr + ((size_t)t * k + j) * (I / 32);
                }
            };
            auto put = [&](float v, int r, int t) {
                const float dv = bf16_round_f32(tsd * v);
                if (sh) {
                    dval[((size_t)t * (k + 1) + k) * RM + r] = dv;
                } else {
                    const uint32_t ranks = rank_bits(dm, t);
                    for (int jj = 0; jj < k; ++jj)
                        if ((ranks >> jj) & 1u) dval[((size_t)t * (k + 1) + jj) * RM + r] = dv;
                }
            };
            while (rest) {
                const int t0 = __ffs(rest) - 1;
                rest &= rest - 1u;
                if (rest) {  // two tokens, rows in groups of 8
                    const int t1 = __ffs(rest) - 1;
                    rest &= rest - 1u;
                    const uint4* hv[2];
                    const float* cv[2];
                    vec(t0, hv[0], cv[0]);
                    vec(t1, hv[1], cv[1]);
                    for (int hb = 0; hb < RG && r0g + hb < r1g; hb += 8) {
                        float acc[16];
                        down_pass<8, 2>(rows + (size_t)hb * RSu, RSu, r1g - r0g - hb, K, hv, cv, lane, acc);
                        const float v = reduce_scatter<16>(acc, lane);
                        const int idx = rs_index<16>(lane), r = r0g + hb + (idx & 7);
                        if ((lane & 1) == 0 && r < r1g) put(v, r, (idx >> 3) ? t1 : t0);
                    }
                } else {
                    const uint4* hv[1];
                    const float* cv[1];
                    vec(t0, hv[0], cv[0]);
                    for (int hb = 0; hb < RG && r0g + hb < r1g; hb += 8) {
                        float acc[8];
                        down_pass<8, 1>(rows + (size_t)hb * RSu, RSu, r1g - r0g - hb, K, hv, cv, lane, acc);
                        const float v = reduce_scatter<8>(acc, lane);
                        const int r = r0g + hb + rs_index<8>(lane);
                        if ((lane & 3) == 0 && r < r1g) put(v, r, t0);
                    }
                }
            }
        };
        if (a.dpre) {  // every routed group is resident once the prefetch lands
            const bool ok = mbar_wait_bounded(&sm.dbar, 0, tid == 0 ? a.status : nullptr, kStatusTimeoutLayer);
            if (!__syncthreads_and(ok)) return;
        }
        // The warp's work, in one loop so that the task's code is inlined once:
        // first its units of the shared expert's rows (resident; one per (8
        // rows, two tokens), spread over the warps from the last one), then its
        // routed tasks warp, warp + kLW, ... (rows from the prefetch, else from
        // the ring).
        const int ng8 = has_sh ? (nr + 7) >> 3 : 0, ntp = (T + 1) >> 1, su0 = kLW - 1 - warp;
        const int n_su_w = su0 < ng8 * ntp ? (ng8 * ntp - su0 + kLW - 1) / kLW : 0;
        const int n_mine = n_tasks > warp ? (n_tasks - warp + kLW - 1) / kLW : 0;
        for (int it = 0; it < n_su_w + n_mine; ++it) {
            const int kk = it - n_su_w;
            int u, r0g, r1g;
            const uint8_t* rows;
            uint32_t tm;
            if (kk < 0) {
                const int q = su0 + it * kLW, g = q / ntp, t0 = 2 * (q - g * ntp);
                u = D;
                r0g = 8 * g;
                r1g = min(nr, r0g + 8);
                rows = shdn + (size_t)r0g * RSs;
                tm = (t0 + 1 < T ? 3u : 1u) << t0;
            } else {
                const int q = warp + kk * kLW;
                u = q / ngr;
                r0g = (q - u * ngr) * RG;
                r1g = min(nr, r0g + RG);
                if (a.dpre) {
                    rows = dpre + ((size_t)u * nr + (size_t)r0g) * RSr;
                } else {
                    cp_async_wait_n(NSW - 1);
                    __syncwarp();
                    rows = ring + (size_t)(kk % NSW) * a.slot4;
                }
                tm = ri.tmask[u];
            }
            task(u, r0g, r1g, rows, tm);
            if (kk >= 0 && !a.dpre) {
                __syncwarp();
                if (kk + NSW < n_mine)
                    issue(kk + NSW);
                else
                    cp_async_commit();
            }
        }
        cp_async_wait<0>();
        __syncthreads();
        // combine, in rank order then the shared expert
        for (int i = tid; i < T * nr; i += kLT) {
            const int t = i / nr, r = i - t * nr;
            float acc = 0.f;
            for (int j = 0; j < k; ++j)
                if (ri.ids[t * k + j] >= 0) acc = fmaf(wsel[t * k + j], dval[((size_t)t * (k + 1) + j) * RM + r], acc);
            if (has_sh) acc += dval[((size_t)t * (k + 1) + k) * RM + r];
            a.y[(size_t)t * H + n0 + r] = f32_to_bf16_bits(acc);
        }
    }
}

}  // namespace

size_t layer_smem_bytes(const LayerArgs& a) { return layer_layout(a).total; }

namespace {
template <bool NORM>
cudaError_t launch_layer_t(const LayerArgs& a, const DevInfo& d, bool pdl, cudaStream_t s) {
    static int configured_for = -1;
    cudaError_t e = configure_smem(layer_kernel<NORM>, d, configured_for);
    if (e != cudaSuccess) return e;
    const size_t smem = layer_smem_bytes(a);
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, layer_kernel<NORM>, kLT, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)d.sm_count);
    cfg.blockDim = dim3(kLT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, layer_kernel<NORM>, a);
}
}  // namespace

cudaError_t launch_layer(const LayerArgs& a, const DevInfo& d, bool pdl, cudaStream_t s) {
    return a.norm.r ? launch_layer_t<true>(a, d, pdl, s) : launch_layer_t<false>(a, d, pdl, s);
}

}  // namespace flint
