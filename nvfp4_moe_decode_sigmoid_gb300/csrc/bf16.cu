// bf16.cu -- the expert GEMVs of the MoE decode step with BF16 expert weights.
//
// "Day-0 Support for Flint on vLLM", section "Optimizations" (Figure 2 and the
// totals after it): the same small-batch MoE decode path also runs the BF16
// checkpoint, whose experts are plain bf16 matrices (4x the bytes of NVFP4).
// The arithmetic is the NVFP4 path's with w = the bf16 value: g and u are
// FP32 dot products with the bf16 activations, scaled by the per-matrix
// tensor scale (1 when none is given), rounded to bf16; h = bf16(silu(g) u);
// d = bf16(ts_d Wd h); y = bf16(sum_j w_j d_j + d_shared).
//
// Every product is a bf16 x bf16 mixed-precision FMA accumulating in FP32
// (the product of two bf16 values is exact in FP32), so the activations are
// staged in shared memory as they are, without the chunk scaling of the NVFP4
// kernels. Both kernels run one CTA of 16 warps per SM; each warp streams its
// weight rows through a private ring of shared-memory slots filled with
// 16-byte cp.async (one commit group per item), as the NVFP4 kernels do.
//
// gate_up_bf16_kernel: the CTA owns a slice of the shared expert's (gate row
//   p, up row p) pairs and of the routed pairs of the distinct selected
//   experts (the same split as the NVFP4 kernel); every pair is two items
//   (its gate row, its up row), dealt to the warps round-robin. Lane l takes
//   the 16-byte words l, l + 32, ... of the row against up to four tokens per
//   pass. The raw sums stay in shared memory until the CTA's epilogue writes h.
// down_bf16_kernel: the CTA owns output rows [n0, n1) of every selected
//   expert's down matrix and the shared one; a task is a group of RG of those
//   rows of one unit, against up to two tokens per pass; then the combine in
//   rank order, as the NVFP4 down kernel.
#include "expert_common.cuh"

namespace flint {
namespace {

constexpr int kBW = kBf16Warps;
constexpr int kBT = kBf16Threads;

// acc + a.lo * b.lo and acc + a.hi * b.hi for bf16x2 operands, FP32 accumulate.
__device__ __forceinline__ float fma_lo_bf16(uint32_t a, uint32_t b, float acc) {
    float d;
    asm("{\n .reg .b16 a0, a1, b0, b1;\n mov.b32 {a0, a1}, %1;\n mov.b32 {b0, b1}, %2;\n"
        " fma.rn.f32.bf16 %0, a0, b0, %3;\n}"
        : "=f"(d)
        : "r"(a), "r"(b), "f"(acc));
    return d;
}
__device__ __forceinline__ float fma_hi_bf16(uint32_t a, uint32_t b, float acc) {
    float d;
    asm("{\n .reg .b16 a0, a1, b0, b1;\n mov.b32 {a0, a1}, %1;\n mov.b32 {b0, b1}, %2;\n"
        " fma.rn.f32.bf16 %0, a1, b1, %3;\n}"
        : "=f"(d)
        : "r"(a), "r"(b), "f"(acc));
    return d;
}

// acc0/acc1 += the 8 products of one 16-byte weight word with one 16-byte
// activation word.
__device__ __forceinline__ void fma8_bf16(const uint4 w, const uint4 x, float& acc0, float& acc1) {
    acc0 = fma_lo_bf16(w.x, x.x, acc0);
    acc1 = fma_hi_bf16(w.x, x.x, acc1);
    acc0 = fma_lo_bf16(w.y, x.y, acc0);
    acc1 = fma_hi_bf16(w.y, x.y, acc1);
    acc0 = fma_lo_bf16(w.z, x.z, acc0);
    acc1 = fma_hi_bf16(w.z, x.z, acc1);
    acc0 = fma_lo_bf16(w.w, x.w, acc0);
    acc1 = fma_hi_bf16(w.w, x.w, acc1);
}

// The warp asks L2 for the bytes [p, p + n) (one 128-byte line per lane and step).
__device__ __forceinline__ void warp_prefetch_l2(const void* p, size_t n, int lane) {
    const char* c = static_cast<const char*>(p);
    for (size_t o = 128 * (size_t)lane; o < n; o += 32 * 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(c + o));
}

// All threads of the CTA copy `bytes` (a multiple of 16) with 16-byte cp.async (no commit).
__device__ __forceinline__ void cta_copy_async(void* dst, const void* src, size_t bytes) {
    uint8_t* d = static_cast<uint8_t*>(dst);
    const uint8_t* s = static_cast<const uint8_t*>(src);
    for (size_t o = 16 * (size_t)threadIdx.x; o < bytes; o += 16 * (size_t)kBT) cp_async16(d + o, s + o);
}

// ===========================================================================
// gate/up + SiLU
// ===========================================================================
// Shared memory: routing view, tensor scales, bf16 activations [T][H], raw
// sums [pair][T] (gate, then up), the warps' rings (one row per slot).
struct Bf16GuSmem {
    size_t route, tss, xs, resg, resu, ring, slot, total;
};
__host__ __device__ inline Bf16GuSmem bf16_gu_layout(int T, int H, int items, int nslots) {
    Bf16GuSmem L;
    L.route = 0;
    L.tss = align_up(sizeof(RouteInfo), 128);
    L.xs = align_up(L.tss + sizeof(float) * (2 * kMaxDistinct + 2), 128);
    L.resg = align_up(L.xs + 2 * (size_t)T * H, 128);
    L.resu = align_up(L.resg + sizeof(float) * (size_t)items * T, 128);
    L.ring = align_up(L.resu + sizeof(float) * (size_t)items * T, 128);
    L.slot = 2 * (size_t)H;
    L.total = L.ring + (size_t)kBW * nslots * L.slot;
    return L;
}

// One pass of a warp over a bf16 row against NT tokens tk[]; the sums (before
// the tensor scale) land at res[tk[j]].
template <int NT>
__device__ __forceinline__ void bf16_row_pass(const uint4* w4, const uint4* xs, int H, const int (&tk)[NT], int lane,
                                              float* res) {
    float a0[NT], a1[NT];
#pragma unroll
    for (int j = 0; j < NT; ++j) a0[j] = a1[j] = 0.f;
    const int nw = H >> 8;  // 16-byte words per lane
#pragma unroll 4
    for (int m = 0; m < nw; ++m) {
        const uint4 wq = w4[lane + 32 * m];
#pragma unroll
        for (int j = 0; j < NT; ++j) fma8_bf16(wq, xs[(size_t)tk[j] * (H / 8) + lane + 32 * m], a0[j], a1[j]);
    }
    float v[NT];
#pragma unroll
    for (int j = 0; j < NT; ++j) v[j] = a0[j] + a1[j];
    const float s = reduce_scatter<NT>(v, lane);
    const int idx = rs_index<NT>(lane);
    int t = tk[0];
#pragma unroll
    for (int j = 1; j < NT; ++j)
        if (idx == j) t = tk[j];
    if (lane % (32 / NT) == 0) res[t] = s;
}

// All tokens of `mask` against one row, four (else two, else one) at a time.
__device__ __forceinline__ void bf16_row(const uint4* w4, const uint4* xs, int H, uint32_t mask, int lane, float* res) {
    while (mask) {
        const int cnt = __popc(mask);
        const int t0 = __ffs(mask) - 1;
        mask &= mask - 1u;
        if (cnt == 1) {
            const int tk[1] = {t0};
            bf16_row_pass<1>(w4, xs, H, tk, lane, res);
            continue;
        }
        const int t1 = __ffs(mask) - 1;
        mask &= mask - 1u;
        if (cnt < 4) {
            const int tk[2] = {t0, t1};
            bf16_row_pass<2>(w4, xs, H, tk, lane, res);
            continue;
        }
        const int t2 = __ffs(mask) - 1;
        mask &= mask - 1u;
        const int t3 = __ffs(mask) - 1;
        mask &= mask - 1u;
        const int tk[4] = {t0, t1, t2, t3};
        bf16_row_pass<4>(w4, xs, H, tk, lane, res);
    }
}

// Item q of the CTA is row (q & 1 ? up : gate) of pair q >> 1; pairs [0, n_sh)
// are the CTA's shared-expert pairs sp0 + i, the rest its routed pairs
// rp0 + i - n_sh of the distinct selected experts. Warp w takes items w,
// w + kBW, ...
__global__ void __launch_bounds__(kBT, 1) gate_up_bf16_kernel(const GateUpArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int NSW = a.nslots, H = a.H, T = a.T, I = a.I, Is = a.Is;
    const int c = blockIdx.x, G = gridDim.x;
    const int sp0 = (int)((long long)c * Is / G), sp1 = (int)((long long)(c + 1) * Is / G);
    const int n_sh = a.s_gu ? sp1 - sp0 : 0;
    const Bf16GuSmem L = bf16_gu_layout(T, H, a.res_items, NSW);
    RouteInfo& ri = *reinterpret_cast<RouteInfo*>(smem + L.route);
    float* tss = reinterpret_cast<float*>(smem + L.tss);
    uint4* xs = reinterpret_cast<uint4*>(smem + L.xs);
    float* resg = reinterpret_cast<float*>(smem + L.resg);
    float* resu = reinterpret_cast<float*>(smem + L.resu);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint8_t* ring = smem + L.ring + (size_t)warp * NSW * L.slot;
    const uint16_t* gu = reinterpret_cast<const uint16_t*>(a.gu);
    const uint16_t* sgu = reinterpret_cast<const uint16_t*>(a.s_gu);

    // Before the wait: the shared expert's rows of this warp into L2 (static
    // weights), and the small buffers' translations.
    for (int q = warp; q < 2 * n_sh; q += kBW)
        warp_prefetch_l2(sgu + ((size_t)(q & 1) * Is + sp0 + (q >> 1)) * H, 2 * (size_t)H, lane);
    if (tid == kBT - 1) {
        prefetch_range(a.x, 2 * (size_t)T * H);
        prefetch_range(a.ids, 4 * (size_t)T * a.k);
        prefetch_range(a.h_routed, 2 * (size_t)T * a.k * I);
        prefetch_range(a.h_shared, 2 * (size_t)T * Is);
    }
    pdl_wait();  // ids (and x) come from earlier kernels
    build_route_info(ri, a.ids, T, a.k, a.E, a.status);
    const int D = ri.D;
    const int RP = D * I;
    const int rp0 = (int)((long long)c * RP / G);
    const int nl = (int)((long long)(c + 1) * RP / G) - rp0;
    const int n_items = 2 * (n_sh + nl);
    const int my_items = n_items > warp ? (n_items - warp + kBW - 1) / kBW : 0;
    pdl_launch_dependents();

    auto row_ptr = [&](int q) -> const uint16_t* {
        const int i = q >> 1, up = q & 1;
        if (i < n_sh) return sgu + ((size_t)up * Is + sp0 + i) * H;
        const int j = rp0 + i - n_sh, d = j / I, p = j - d * I;
        return gu + ((size_t)ri.dlist[d] * 2 * I + (size_t)up * I + p) * H;
    };
    auto issue = [&](int m) {
        warp_copy_async(ring + (size_t)(m % NSW) * L.slot, row_ptr(warp + m * kBW), 2 * H, lane);
        cp_async_commit();
    };
    // x first (one commit group per thread), then the scales, then the rows.
    cta_copy_async(xs, a.x, 2 * (size_t)T * H);
    cp_async_commit();
    float tsv = 1.f;
    if (tid < 2 * D) {
        if (a.ts) tsv = ld_cg(a.ts + 3 * ri.dlist[tid >> 1] + (tid & 1));
    } else if (tid < 2 * D + 2 && a.s_ts) {
        tsv = ld_cg(a.s_ts + tid - 2 * D);
    }
    for (int m = 0; m < NSW; ++m) {
        if (m < my_items)
            issue(m);
        else
            cp_async_commit();
    }
    if (tid < 2 * D + 2) tss[tid] = tsv;
    cp_async_wait_n(NSW);  // this thread's part of x
    __syncthreads();       // x, the scales and the routing view visible to all warps

    const uint32_t all_tokens = (1u << T) - 1u;
    for (int m = 0; m < my_items; ++m) {
        cp_async_wait_n(NSW - 1);
        __syncwarp();
        const int q = warp + m * kBW, i = q >> 1;
        uint32_t mask = all_tokens;
        if (i >= n_sh) mask = ri.tmask[(rp0 + i - n_sh) / I];
        const uint4* w4 = reinterpret_cast<const uint4*>(ring + (size_t)(m % NSW) * L.slot);
        bf16_row(w4, xs, H, mask, lane, ((q & 1) ? resu : resg) + (size_t)i * T);
        __syncwarp();
        if (m + NSW < my_items)
            issue(m + NSW);
        else
            cp_async_commit();
    }
    cp_async_wait<0>();
    __syncthreads();
    // Epilogue over (token, pair): tensor scales, bf16 rounding points, SiLU.
    const int n_pairs = n_sh + nl;
    for (int e = tid; e < n_pairs * T; e += kBT) {
        const int t = e / n_pairs, i = e - t * n_pairs;
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
        const float u = bf16_round_f32(tsu * resu[i * T + t]);
        const uint16_t out = f32_to_bf16_bits(silu_f32(g) * u);
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
struct Bf16DnSmem {
    size_t route, w, dval, hr, hs, ring, total;
};
__host__ __device__ inline Bf16DnSmem bf16_dn_layout(const DownArgs& a) {
    Bf16DnSmem L;
    L.route = 0;
    L.w = align_up(sizeof(RouteInfo), 128);
    L.dval = align_up(L.w + sizeof(float) * (2 * kMaxDistinct + 1), 128);
    L.hr = align_up(L.dval + sizeof(float) * (size_t)a.T * (a.k + 1) * a.rows_max, 128);
    L.hs = align_up(L.hr + 2 * (size_t)a.T * a.k * a.I, 128);
    L.ring = align_up(L.hs + 2 * (size_t)a.T * a.Is, 128);
    L.total = L.ring + (size_t)kBW * a.nslots * a.slot_bytes;
    return L;
}

// RG rows of K values (row stride K) against NT tokens' vectors hv[]:
// acc[r * NT + j] = lane's part of row r . hv[j].
template <int RG, int NT>
__device__ __forceinline__ void bf16_down_pass(const uint4* rows, int nrows, int K, const uint4* const (&hv)[NT],
                                               int lane, float (&acc)[RG * NT]) {
    float a1[RG * NT];
#pragma unroll
    for (int i = 0; i < RG * NT; ++i) acc[i] = a1[i] = 0.f;
    const int wpr = K >> 3;  // 16-byte words per row
    for (int m = 0; m < (K >> 8); ++m) {
        uint4 hq[NT];
#pragma unroll
        for (int j = 0; j < NT; ++j) hq[j] = hv[j][lane + 32 * m];
#pragma unroll
        for (int r = 0; r < RG; ++r) {
            if (r < nrows) {
                const uint4 wq = rows[(size_t)r * wpr + lane + 32 * m];
#pragma unroll
                for (int j = 0; j < NT; ++j) fma8_bf16(wq, hq[j], acc[r * NT + j], a1[r * NT + j]);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < RG * NT; ++i) acc[i] += a1[i];
}

// Each CTA owns output rows [n0, n1); units are the distinct selected experts
// (ascending id) and the shared expert; task q = (unit q / ngr, row group
// q % ngr); warp w takes tasks w, w + kBW, ...
template <int RG>
__global__ void __launch_bounds__(kBT, 1) down_bf16_kernel(const DownArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const Bf16DnSmem L = bf16_dn_layout(a);
    const int NSW = a.nslots;
    const int T = a.T, k = a.k, H = a.H, I = a.I, Is = a.Is, RM = a.rows_max;
    RouteInfo& ri = *reinterpret_cast<RouteInfo*>(smem + L.route);
    float* wsm = reinterpret_cast<float*>(smem + L.w);
    float* tsd_s = wsm + kMaxDistinct;
    float* dval = reinterpret_cast<float*>(smem + L.dval);  // [t][j (k = shared)][row]
    const uint4* hr = reinterpret_cast<const uint4*>(smem + L.hr);  // [t*k + j][I] bf16
    const uint4* hs = reinterpret_cast<const uint4*>(smem + L.hs);  // [t][Is] bf16
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint8_t* ring = smem + L.ring + (size_t)warp * NSW * a.slot_bytes;
    const int c = blockIdx.x, G = gridDim.x;
    const int n0 = (int)((long long)c * H / G), n1 = (int)((long long)(c + 1) * H / G), nr = n1 - n0;
    if (nr == 0) return;
    const uint16_t* dn = reinterpret_cast<const uint16_t*>(a.down);
    const uint16_t* sdn = reinterpret_cast<const uint16_t*>(a.s_down);
    const bool has_sh = sdn != nullptr;

    if (has_sh && warp == kBW - 1) warp_prefetch_l2(sdn + (size_t)n0 * Is, 2 * (size_t)nr * Is, lane);
    if (tid == kBT - 1) {
        prefetch_range(a.ids, 4 * (size_t)T * k);
        prefetch_range(a.w, 4 * (size_t)T * k);
        prefetch_range(a.h_routed, 2 * (size_t)T * k * I);
        prefetch_range(a.h_shared, 2 * (size_t)T * Is);
        prefetch_range(a.y + (size_t)n0, 2 * ((size_t)(T - 1) * H + nr));
    }
    build_route_info(ri, a.ids, T, k, a.E, a.status);  // final before the gate/up kernel triggers this one
    const int D = ri.D;
    const int n_units = D + (has_sh ? 1 : 0);
    const int ngr = (nr + RG - 1) / RG;
    const int n_tasks = n_units * ngr;
    const int my_tasks = n_tasks > warp ? (n_tasks - warp + kBW - 1) / kBW : 0;
    auto issue = [&](int kk) {
        const int q = warp + kk * kBW, u = q / ngr, r0 = (q - u * ngr) * RG, r1 = min(nr, r0 + RG);
        uint8_t* dst = ring + (size_t)(kk % NSW) * a.slot_bytes;
        if (u < D)
            warp_copy_async(dst, dn + ((size_t)ri.dlist[u] * H + n0 + r0) * I, 2 * (r1 - r0) * I, lane);
        else
            warp_copy_async(dst, sdn + (size_t)(n0 + r0) * Is, 2 * (r1 - r0) * Is, lane);
        cp_async_commit();
    };
    pdl_wait();  // h comes from the gate/up kernel
    pdl_launch_dependents();
    // h first (one commit group per thread), then the small loads, then the rows.
    cta_copy_async(smem + L.hr, a.h_routed, 2 * (size_t)T * k * I);
    if (has_sh) cta_copy_async(smem + L.hs, a.h_shared, 2 * (size_t)T * Is);
    cp_async_commit();
    float wv = 0.f;
    if (tid < T * k) wv = ld_cg(a.w + tid);
    else if (tid >= 64 && tid < 64 + n_units) {
        const int u = tid - 64;
        wv = 1.f;
        if (u < D) {
            if (a.ts) wv = ld_cg(a.ts + 3 * ri.dlist[u] + 2);
        } else if (a.s_ts) {
            wv = ld_cg(a.s_ts + 2);
        }
    }
    for (int kk = 0; kk < NSW; ++kk) {
        if (kk < my_tasks)
            issue(kk);
        else
            cp_async_commit();
    }
    if (tid < T * k) wsm[tid] = wv;
    else if (tid >= 64 && tid < 64 + n_units) tsd_s[tid - 64] = wv;
    cp_async_wait_n(NSW);
    __syncthreads();

    for (int kk = 0; kk < my_tasks; ++kk) {
        cp_async_wait_n(NSW - 1);
        __syncwarp();
        const int q = warp + kk * kBW, u = q / ngr, r0 = (q - u * ngr) * RG, r1 = min(nr, r0 + RG);
        const bool sh = u >= D;
        const int K = sh ? Is : I;
        const uint4* rows = reinterpret_cast<const uint4*>(ring + (size_t)(kk % NSW) * a.slot_bytes);
        const unsigned long long dm = sh ? 0ull : ri.dmask[u];
        uint32_t rest = sh ? (1u << T) - 1u : ri.tmask[u];
        const float tsd = tsd_s[u];
        auto vec = [&](int t) -> const uint4* {
            if (sh) return hs + (size_t)t * (Is / 8);
            const int j = __ffs(rank_bits(dm, t)) - 1;
            return hr + ((size_t)t * k + j) * (I / 8);
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
            if (rest) {
                const int t1 = __ffs(rest) - 1;
                rest &= rest - 1u;
                const uint4* const hv[2] = {vec(t0), vec(t1)};
                float acc[RG * 2];
                bf16_down_pass<RG, 2>(rows, r1 - r0, K, hv, lane, acc);
                const float v = reduce_scatter<RG * 2>(acc, lane);
                const int idx = rs_index<RG * 2>(lane), r = r0 + idx / 2;
                if (lane % (32 / (RG * 2)) == 0 && r < r1) put(v, r, (idx & 1) ? t1 : t0);
            } else {
                const uint4* const hv[1] = {vec(t0)};
                float acc[RG];
                bf16_down_pass<RG, 1>(rows, r1 - r0, K, hv, lane, acc);
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
    cp_async_wait<0>();
    __syncthreads();
    for (int i = tid; i < T * nr; i += kBT) {
        const int t = i / nr, r = i - t * nr;
        float acc = 0.f;
        for (int j = 0; j < k; ++j)
            if (ri.ids[t * k + j] >= 0) acc = fmaf(wsm[t * k + j], dval[((size_t)t * (k + 1) + j) * RM + r], acc);
        if (has_sh) acc += dval[((size_t)t * (k + 1) + k) * RM + r];
        a.y[(size_t)t * H + n0 + r] = f32_to_bf16_bits(acc);
    }
}

template <typename K, typename A>
cudaError_t launch_bf16(K kernel, const A& args, unsigned grid, size_t smem, bool pdl, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kBT);
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

size_t gate_up_bf16_smem_bytes(const GateUpArgs& a) { return bf16_gu_layout(a.T, a.H, a.res_items, a.nslots).total; }
size_t down_bf16_smem_bytes(const DownArgs& a) { return bf16_dn_layout(a).total; }

cudaError_t launch_gate_up_bf16(const GateUpArgs& a, const DevInfo& d, bool pdl, cudaStream_t s) {
    static int cfg = -1;
    cudaError_t e = configure_smem(gate_up_bf16_kernel, d, cfg);
    if (e != cudaSuccess) return e;
    return launch_bf16(gate_up_bf16_kernel, a, (unsigned)d.sm_count, gate_up_bf16_smem_bytes(a), pdl, s);
}

cudaError_t launch_down_bf16(const DownArgs& a, const DevInfo& d, bool pdl, cudaStream_t s) {
    static int cfg4 = -1, cfg8 = -1;
    const size_t smem = down_bf16_smem_bytes(a);
    cudaError_t e;
    if (a.rg == 8) {
        if ((e = configure_smem(down_bf16_kernel<8>, d, cfg8)) != cudaSuccess) return e;
        return launch_bf16(down_bf16_kernel<8>, a, (unsigned)d.sm_count, smem, pdl, s);
    }
    if ((e = configure_smem(down_bf16_kernel<4>, d, cfg4)) != cudaSuccess) return e;
    return launch_bf16(down_bf16_kernel<4>, a, (unsigned)d.sm_count, smem, pdl, s);
}

}  // namespace flint
