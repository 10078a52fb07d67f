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
// Both kernels run one CTA of 24 warps per SM. Each warp streams its own work
// items (weight rows) through a private ring of shared-memory slots, copied
// by all its lanes with 16-byte cp.async (one commit group per item).
// 1-D bulk copies were tried first: one item's rows are only 1-4 KB, and at
// that size the bulk-copy path delivered well under half of the HBM
// bandwidth, while per-lane 16-byte copies saturate it. Dequantisation happens
// in registers: cvt e2m1x2 gives exact f16 code values, which multiply f16
// activations in mixed-precision FMAs accumulating in FP32 (an f16 x f16
// product is exact in FP32, so every step rounds once, as an FP32 FMA of the
// same values would). The UE4M3 block scale is applied once per 16 values.
//
// Activations (x for gate/up, h for down) are staged in shared memory as f16:
// every 32-value chunk is multiplied by the power of two that puts its largest
// magnitude in [2^14, 2^15), which keeps every bf16 value of the chunk down to
// 2^-31 of that maximum exact (smaller ones are off by at most 2^-39 of it),
// and the chunk's partial dot product is multiplied back by the inverse power
// of two (exact). The staging order puts each lane's 16-byte words side by
// side, so the warp's shared-memory loads are conflict-free.
//
// gate_up_kernel<PAIR=true>: per (selected expert, h index p) "pair" one warp
//   dots gate row p and up row p with every token that selected the expert
//   (two tokens per pass), the lanes splitting the columns. The pairs of the
//   distinct selected experts (ascending id) are split evenly over the CTAs
//   and then over the warps; the CTA's slice of the shared expert is
//   requested before the PDL wait. The raw sums go to shared memory; once the
//   CTA is done, all its threads apply g = bf16(ts_g acc_g),
//   u = bf16(ts_u acc_u), h = bf16(silu(g) u) and write h.
// gate_up_kernel<PAIR=false>: the same machinery over plain rows: the dense
//   GEMV y = bf16(ts W x).
// down_kernel: each CTA owns a slice of output rows of every selected
//   expert's down matrix (and the shared one). A task is (expert, group of up
//   to 16 of those rows); one warp computes d = bf16(ts_d Wd h) for the group,
//   the lanes splitting the 16-value blocks of the row, and a reduce-scatter
//   of the per-row sums over the lanes. Then the CTA combines
//   y = bf16(sum_j w_j d_j + d_shared) in rank order. No atomics: the result is
//   deterministic. Weight rows are requested right after the PDL wait, behind
//   the small loads of h and the scales.
#include "expert_common.cuh"

namespace flint {
namespace {

constexpr int kW = kGemvWarps;

// ===========================================================================
// gate/up + SiLU (PAIR) or plain rows
// ===========================================================================
// Shared memory: routing view, chunk scales, f16 activations, raw sums
// [item][T] (gate, then up), the warps' slot rings (one item per slot: its
// gate row, then its up row).
struct GateUpSmem {
    size_t route, tss, csc, xs, resg, resu, ring, slot, total;
};
template <bool PAIR>
__host__ __device__ inline GateUpSmem gate_up_layout(int T, int H, int items, int nslots) {
    GateUpSmem L;
    L.route = 0;
    L.tss = align_up(L.route + sizeof(RouteInfo), 128);
    L.csc = align_up(L.tss + sizeof(float) * (2 * kMaxDistinct + 2), 128);
    L.xs = align_up(L.csc + sizeof(float) * (size_t)T * (H / 32), 128);
    L.resg = align_up(L.xs + 2 * (size_t)T * H, 128);
    L.resu = align_up(L.resg + sizeof(float) * (size_t)items * T, 128);
    L.ring = align_up(L.resu + (PAIR ? sizeof(float) * (size_t)items * T : 0), 128);
    L.slot = (size_t)(PAIR ? 2 : 1) * nvfp4_row_stride(H);
    L.total = L.ring + (size_t)kW * nslots * L.slot;
    return L;
}

// Work items of a CTA: its slice [sp0, sp1) of the shared expert's pairs (or
// of the dense matrix's rows / pairs), then (MoE) its share of the routed
// pairs of the distinct selected experts. Warp w's list: shared items
// kW-1-w, 2 kW-1-w, ... (known before the PDL wait, so requested then), then
// the routed list items [lw0, lw1) once the routing is read. Dense: rows
// [lw0, lw1) of the CTA's slice, requested before the wait. Each item goes
// through the warp's ring of nslots slots with 16-byte cp.async copies by
// all its lanes (one commit group per item). Item i of the CTA (shared pair /
// dense row i < n_sh, then routed pair n_sh + j) keeps its raw sums at
// res[i * T + t].
template <bool PAIR>
__global__ void __launch_bounds__(kGemvThreads, 1) gate_up_kernel(const GateUpArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int NSW = a.nslots, H = a.H, T = a.T, I = a.I, Is = a.Is;
    const bool moe = a.gu != nullptr;
    const int c = blockIdx.x, G = gridDim.x;
    const int sp0 = (int)((long long)c * Is / G), sp1 = (int)((long long)(c + 1) * Is / G);
    const int n_sh = a.s_gu ? sp1 - sp0 : 0;
    const GateUpSmem L = gate_up_layout<PAIR>(T, H, a.res_items, NSW);
    RouteInfo& ri = *reinterpret_cast<RouteInfo*>(smem + L.route);
    float* csc = reinterpret_cast<float*>(smem + L.csc);
    uint4* xh = reinterpret_cast<uint4*>(smem + L.xs);
    float* resg = reinterpret_cast<float*>(smem + L.resg);
    float* resu = reinterpret_cast<float*>(smem + L.resu);
    float* tss = reinterpret_cast<float*>(smem + L.tss);  // [d][2] routed, then the shared pair
    const int RS = (int)nvfp4_row_stride(H);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint8_t* ring = smem + L.ring + (size_t)warp * NSW * L.slot;

    // This warp's list: n_sw shared items, then routed list items [lw0, lw1)
    // (MoE); or dense rows [lw0, lw1).
    const int n_sw = moe && n_sh > kW - 1 - warp ? (n_sh - (kW - 1 - warp) + kW - 1) / kW : 0;
    int rp0 = 0, lw0 = 0, lw1 = 0, nl = 0;
    if (!moe) {
        lw0 = (int)((long long)warp * n_sh / kW);
        lw1 = (int)((long long)(warp + 1) * n_sh / kW);
    }
    // Requests item m of the list into slot m % NSW (one commit group).
    auto issue = [&](int m) {
        const uint8_t *g, *u;
        if (m < n_sw) {
            const int i = kW - 1 - warp + kW * m;
            g = a.s_gu + (size_t)(sp0 + i) * RS;
            u = a.s_gu + (size_t)(Is + sp0 + i) * RS;
        } else if (moe) {
            const int q = rp0 + lw0 + m - n_sw, d = q / I, p = q - d * I;
            g = a.gu + ((size_t)ri.dlist[d] * 2 * I + p) * RS;
            u = g + (size_t)I * RS;
        } else {
            const int j = lw0 + m;
            g = a.s_gu + (size_t)(sp0 + j) * RS;
            u = a.s_gu + (size_t)(Is + sp0 + j) * RS;
        }
        uint8_t* slot = ring + (size_t)(m % NSW) * L.slot;
        warp_copy_async(slot, g, RS, lane);
        if (PAIR) warp_copy_async(slot + RS, u, RS, lane);
        cp_async_commit();
    };

    if (tid == kGemvThreads - 1) {
        prefetch_range(a.x, 2 * (size_t)T * H);
        prefetch_range(a.s_ts, 8);
        prefetch_range(a.h_shared, 2 * (size_t)T * Is);
        if (moe) {
            prefetch_range(a.ids, 4 * (size_t)T * a.k);
            prefetch_range(a.ts, 12 * (size_t)a.E);
            prefetch_range(a.h_routed, 2 * (size_t)T * a.k * I);
        }
    }
    // Before the wait: weights that depend on no earlier kernel.
    const int n_pre = moe ? n_sw : lw1 - lw0;
    int issued = 0;
    for (; issued < NSW && issued < n_pre; ++issued) issue(issued);
    const StageSrc xsrc[1] = {{a.x, xh, csc, T, H}};
    if (a.x_early) stage_f16<false>(xsrc, [] {});
    pdl_wait();  // ids (and x, unless staged already) are written by earlier kernels
    if (moe) {
        build_route_info(ri, a.ids, T, a.k, a.E, a.status);
        const int RP = ri.D * I;
        rp0 = (int)((long long)c * RP / G);
        nl = (int)((long long)(c + 1) * RP / G) - rp0;
        lw0 = (int)((long long)warp * nl / kW);
        lw1 = (int)((long long)(warp + 1) * nl / kW);
    }
    pdl_launch_dependents();
    // The small loads first (tensor scales, activations): behind the routed
    // weight copies they would wait for the whole stream ahead of them.
    const int D = moe ? ri.D : 0;
    float tsv = 0.f;
    if (tid < 2 * D) tsv = ld_cg(a.ts + 3 * ri.dlist[tid >> 1] + (tid & 1));
    else if (tid < 2 * D + 2 && a.s_ts) tsv = ld_cg(a.s_ts + (PAIR ? tid - 2 * D : 0));
    const int n_items_w = moe ? n_sw + lw1 - lw0 : lw1 - lw0;
    auto burst = [&] {
        for (; issued < NSW; ++issued) {
            if (issued < n_items_w)
                issue(issued);
            else
                cp_async_commit();  // empty group: NSW groups ahead of the first wait
        }
    };
    if (a.x_early)
        burst();
    else
        stage_f16<false>(xsrc, burst);
    if (tid < 2 * D + 2) tss[tid] = tsv;
    __syncthreads();  // activations, scales and the routing view visible to all warps

    const uint32_t all_tokens = (1u << T) - 1u;
    int d = 0, p = 0;  // expert index and pair index of the next routed item (MoE)
    if (moe && lw1 > lw0) {
        d = (rp0 + lw0) / I;
        p = rp0 + lw0 - d * I;
    }
    for (int m = 0; m < n_items_w; ++m) {
        cp_async_wait_n(NSW - 1);
        __syncwarp();
        const uint8_t* grow = ring + (size_t)(m % NSW) * L.slot;
        if (m < n_sw) {
            const int i = kW - 1 - warp + kW * m;
            gate_up_item<PAIR>(grow, grow + RS, H, xh, csc, all_tokens, lane, resg + i * T, resu + i * T);
        } else {
            const int item = moe ? n_sh + lw0 + m - n_sw : lw0 + m;
            gate_up_item<PAIR>(grow, grow + RS, H, xh, csc, moe ? ri.tmask[d] : all_tokens, lane,
                               resg + item * T, resu + item * T);
            if (++p == I) {
                p = 0;
                ++d;
            }
        }
        __syncwarp();
        if (m + NSW < n_items_w)
            issue(m + NSW);
        else
            cp_async_commit();
    }
    cp_async_wait<0>();  // retire the trailing empty groups before warps exit
    __syncthreads();
    // Epilogue over (token, item): tensor scales, bf16 rounding points, SiLU.
    const int n_items = n_sh + nl;
    for (int e = tid; e < n_items * T; e += kGemvThreads) {
        const int t = e / n_items, i = e - t * n_items;
        float tsg, tsu;
        int pp;
        uint32_t ranks = 0;
        if (i < n_sh) {
            pp = sp0 + i;
            tsg = tss[2 * D];
            tsu = tss[2 * D + 1];
        } else {
            const int q = rp0 + i - n_sh, dd = q / I;
            pp = q - dd * I;
            ranks = rank_bits(ri.dmask[dd], t);
            if (!ranks) continue;
            tsg = tss[2 * dd];
            tsu = tss[2 * dd + 1];
        }
        const float g = bf16_round_f32(tsg * resg[i * T + t]);
        uint16_t out;
        if (PAIR) {
            const float u = bf16_round_f32(tsu * resu[i * T + t]);
            out = f32_to_bf16_bits(silu_f32(g) * u);
        } else {
            out = f32_to_bf16_bits(g);
        }
        if (i < n_sh) {
            a.h_shared[(size_t)t * Is + pp] = out;
        } else {
            for (int j = 0; j < a.k; ++j)
                if ((ranks >> j) & 1u) a.h_routed[((size_t)t * a.k + j) * I + pp] = out;
        }
    }
}

// ===========================================================================
// down + combine
// ===========================================================================
struct DownSmem {
    size_t route, w, csr, css, dval, hr, hs, ring, total;
};
__host__ __device__ inline DownSmem down_layout(const DownArgs& a) {
    DownSmem L;
    L.route = 0;
    L.w = align_up(L.route + sizeof(RouteInfo), 128);
    L.csr = align_up(L.w + sizeof(float) * (2 * kMaxDistinct + 1), 128);
    L.css = align_up(L.csr + sizeof(float) * (size_t)a.T * a.k * (a.I / 32), 128);
    L.dval = align_up(L.css + sizeof(float) * (size_t)a.T * (a.Is / 32), 128);
    L.hr = align_up(L.dval + sizeof(float) * (size_t)a.T * (a.k + 1) * a.rows_max, 128);
    L.hs = align_up(L.hr + 2 * (size_t)a.T * a.k * a.I, 128);
    L.ring = align_up(L.hs + 2 * (size_t)a.T * a.Is, 128);
    L.total = L.ring + (size_t)kW * a.nslots * a.slot_bytes;
    return L;
}

// Each CTA owns output rows [n0, n1). Units are the distinct selected experts
// (ascending id) and the shared expert; a task is a group of up to RG of the
// CTA's rows of one unit. Warp w takes tasks w, w + kW, ... through its own
// ring (16-byte cp.async copies by all its lanes, one commit group per
// task); the routing is final before this kernel starts (the gate/up kernel
// triggers it only after its own wait), so the first slots are requested
// before the PDL wait.
template <int RG>
__global__ void __launch_bounds__(kGemvThreads, 1) down_kernel(const DownArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const DownSmem L = down_layout(a);
    const int NSW = a.nslots;
    const int T = a.T, k = a.k, H = a.H, I = a.I, Is = a.Is, RM = a.rows_max;
    RouteInfo& ri = *reinterpret_cast<RouteInfo*>(smem + L.route);
    float* wsm = reinterpret_cast<float*>(smem + L.w);            // [t*k + j]
    float* tsd_s = reinterpret_cast<float*>(smem + L.w) + kMaxDistinct;  // down scale of unit u
    float* csr = reinterpret_cast<float*>(smem + L.csr);    // chunk scales of h_routed [t*k + j][I / 32]
    float* css = reinterpret_cast<float*>(smem + L.css);    // chunk scales of h_shared [t][Is / 32]
    float* dval = reinterpret_cast<float*>(smem + L.dval);  // [t][j (k = shared)][row]
    uint4* hr = reinterpret_cast<uint4*>(smem + L.hr);      // [t*k + j][I] f16, DOWN order
    uint4* hs = reinterpret_cast<uint4*>(smem + L.hs);      // [t][Is] f16, DOWN order

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint8_t* ring = smem + L.ring + (size_t)warp * NSW * a.slot_bytes;
    const int c = blockIdx.x, G = gridDim.x;
    const int n0 = (int)((long long)c * H / G), n1 = (int)((long long)(c + 1) * H / G), nr = n1 - n0;
    const int RSr = (int)nvfp4_row_stride(I), RSs = Is ? (int)nvfp4_row_stride(Is) : 0;
    if (nr == 0) return;  // more CTAs than output rows: nothing to copy or compute

    if (tid == kGemvThreads - 1) {
        prefetch_range(a.ids, 4 * (size_t)T * k);
        prefetch_range(a.w, 4 * (size_t)T * k);
        prefetch_range(a.ts, 12 * (size_t)a.E);
        prefetch_range(a.s_ts, 12);
        prefetch_range(a.h_routed, 2 * (size_t)T * k * I);
        prefetch_range(a.h_shared, 2 * (size_t)T * Is);
        prefetch_range(a.y + (size_t)n0, 2 * ((size_t)(T - 1) * H + nr));
    }
    build_route_info(ri, a.ids, T, k, a.E, a.status);
    const int D = ri.D;
    const bool has_sh = a.s_down != nullptr;
    const int n_units = D + (has_sh ? 1 : 0);
    const int ngr = (nr + RG - 1) / RG;  // row groups per unit
    const int n_tasks = n_units * ngr;
    const int my_tasks = n_tasks > warp ? (n_tasks - warp + kW - 1) / kW : 0;

    auto issue = [&](int kk) {  // this warp's kk-th task (one commit group)
        const int q = warp + kk * kW, u = q / ngr, r0 = (q - u * ngr) * RG, r1 = min(nr, r0 + RG);
        uint8_t* dst = ring + (size_t)(kk % NSW) * a.slot_bytes;
        if (u < D)
            warp_copy_async(dst, a.down + ((size_t)ri.dlist[u] * H + n0 + r0) * RSr, (r1 - r0) * RSr, lane);
        else
            warp_copy_async(dst, a.s_down + (size_t)(n0 + r0) * RSs, (r1 - r0) * RSs, lane);
        cp_async_commit();
    };
    pdl_wait();  // h comes from the gate/up kernel
    pdl_launch_dependents();
    // The small loads first (combine weights, tensor scales, h); then this
    // warp's first weight copies; then h is converted. (Requesting the weights
    // before the wait gains nothing here: this kernel's CTAs do not fit on an
    // SM beside the gate/up kernel's, and h queued behind the whole weight
    // stream would arrive last.)
    float wv = 0.f;
    if (tid < T * k) wv = ld_cg(a.w + tid);
    else if (tid >= 64 && tid < 64 + n_units) wv = tid - 64 < D ? ld_cg(a.ts + 3 * ri.dlist[tid - 64] + 2) : ld_cg(a.s_ts + 2);
    const StageSrc hsrc[2] = {{a.h_routed, hr, csr, T * k, I}, {a.h_shared, hs, css, has_sh ? T : 0, Is ? Is : 32}};
    stage_f16<true>(hsrc, [&] {
        for (int kk = 0; kk < NSW; ++kk) {
            if (kk < my_tasks)
                issue(kk);
            else
                cp_async_commit();  // empty group: NSW groups ahead of the first wait
        }
    });
    if (tid < T * k) wsm[tid] = wv;
    else if (tid >= 64 && tid < 64 + n_units) tsd_s[tid - 64] = wv;
    __syncthreads();

    for (int kk = 0; kk < my_tasks; ++kk) {
        cp_async_wait_n(NSW - 1);
        __syncwarp();
        const int q = warp + kk * kW, u = q / ngr, r0 = (q - u * ngr) * RG, r1 = min(nr, r0 + RG);
        const bool sh = u >= D;
        const int K = sh ? Is : I, RS = sh ? RSs : RSr;
        const uint8_t* slot = ring + (size_t)(kk % NSW) * a.slot_bytes;
        const unsigned long long dm = sh ? 0ull : ri.dmask[u];
        uint32_t rest = sh ? (1u << T) - 1u : ri.tmask[u];
        const float tsd = tsd_s[u];
        // Token t's staged h vector (and chunk scales) for this unit.
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
        // d value of row r (of the CTA's rows) for token t, for every rank of t.
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
                for (int hb = 0; hb < RG && r0 + hb < r1; hb += 8) {
                    float acc[16];
                    down_pass<8, 2>(slot + (size_t)hb * RS, RS, r1 - r0 - hb, K, hv, cv, lane, acc);
                    const float v = reduce_scatter<16>(acc, lane);
                    const int idx = rs_index<16>(lane), r = r0 + hb + (idx & 7);
                    if ((lane & 1) == 0 && r < r1) put(v, r, (idx >> 3) ? t1 : t0);
                }
            } else {
                const uint4* hv[1];
                const float* cv[1];
                vec(t0, hv[0], cv[0]);
                float acc[RG];
                down_pass<RG, 1>(slot, RS, r1 - r0, K, hv, cv, lane, acc);
                const float v = reduce_scatter<RG>(acc, lane);
                const int r = r0 + rs_index<RG>(lane);
                if (lane % (32 / RG) == 0 && r < r1) put(v, r, t0);
            }
        }
        __syncwarp();
        if (kk + NSW < my_tasks)
            issue(kk + NSW);
        else
            cp_async_commit();
    }
    cp_async_wait<0>();  // retire the trailing empty groups before warps exit
    __syncthreads();
    // combine, in rank order then the shared expert
    for (int i = tid; i < T * nr; i += kGemvThreads) {
        const int t = i / nr, r = i - t * nr;
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
    return pair ? gate_up_layout<true>(a.T, a.H, a.res_items, a.nslots).total
                : gate_up_layout<false>(a.T, a.H, a.res_items, a.nslots).total;
}
size_t down_smem_bytes(const DownArgs& a) { return down_layout(a).total; }

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
    static int cfg8 = -1, cfg16 = -1;
    const size_t smem = down_smem_bytes(a);
    cudaError_t e;
    if (a.rg == 8) {
        if ((e = configure_smem(down_kernel<8>, d, cfg8)) != cudaSuccess) return e;
        return launch_ex(down_kernel<8>, a, (unsigned)d.sm_count, smem, pdl, s);
    }
    if ((e = configure_smem(down_kernel<16>, d, cfg16)) != cudaSuccess) return e;
    return launch_ex(down_kernel<16>, a, (unsigned)d.sm_count, smem, pdl, s);
}

}  // namespace flint
