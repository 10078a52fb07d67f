// layer.cu -- the whole decode step of one MoE layer in one cooperative
// kernel: router GEMV + sigmoid top-k, gate/up + SiLU, down + weighted
// combine with the shared expert.
//
// "Day-0 Support for Flint on vLLM", section "Optimizations": the small-batch
// MoE path is a short chain of kernels whose expert GEMVs read only the
// selected experts' weights, with routing and the combine fused into the
// neighbouring GEMVs, each kernel launched with programmatic dependent launch
// so that it loads its weights while the previous kernel still runs. Here the
// chain is one launch, one CTA per SM, all CTAs resident (cooperative launch),
// and no CTA waits for the whole grid to reach a point:
//
//   * The CTAs are split by expert. CTAs [0, Gs) run the shared expert (it
//     needs no routing); CTAs [Gs, G) run the routed experts the tokens
//     selected. Each CTA owns one contiguous, cost-balanced range of gate/up
//     pairs and one of down-row blocks in the concatenation of its group's
//     experts (an expert's row costs ~ 4 + 3 x the tokens that chose it: its
//     decode once, a multiply-add per token), so a CTA touches one or two
//     experts.
//   * The CTA's items (a gate/up pair; a group of up to 8 down rows) are dealt
//     to its warps round-robin; each warp streams its own items through a
//     private ring of shared-memory slots fed by bulk copies (TMA) that its
//     lane 0 issues, so a slot is refilled as soon as its warp is done with it.
//   * Before the PDL wait each CTA starts the copies of its static weights:
//     in the routed group its router rows and the routed experts' tensor
//     scales, in the shared group the first items of every warp's ring.
//   * Exchanges go through the workspace with release / acquire counters,
//     each polled by one thread per CTA: the router rows published (every CTA
//     then reads all scores and selects the top-k itself), and per expert the
//     gate/up pairs whose h is written (a CTA waits only for the experts whose
//     down rows it computes).
//   * The combine y = bf16(sum_j w_j d_j + d_shared) runs per 16-row block:
//     each expert's down CTA writes its d rows and counts its arrival on the
//     block's counter; the CTA that arrives last (all experts' d present)
//     combines the block in rank order and resets the counter. Nothing waits.
//   * One token (the ROWS instantiation): the combine's last arrivers make the
//     call's tail, so down and the combine are split by output rows instead.
//     CTA c owns rows [c H / G, (c + 1) H / G) of y, computes them for every
//     selected expert and the shared one from all of h (once every pair is
//     published: one count) and sums them in rank order in shared memory; no
//     d leaves the CTA. (From two tokens on this measured slower: every CTA
//     then walks the rows of every selected expert.)
//   * The last CTA to finish resets the exchange counters for the next call.
//   * Given routing (the GIVEN instantiation, behind flint_moe_decode): the
//     router rows, the score exchange and the top-k are left out; every CTA
//     reads the caller's ids and weights after its PDL wait. Those may repeat
//     an expert within a token (its h and d are computed once and d is written
//     for each of its ranks) or hold an id outside [0, E) (reported in the
//     status word; the rank adds nothing to y).
//
// After a timed-out wait (or any other failure that stops a CTA) the counters
// are left mid-call and the workspace must be re-initialised
// (flint_workspace_check does it); until then every call returns at once,
// leaving its outputs unwritten, and the status stays set.
#include <climits>
#include <type_traits>

#include "expert_common.cuh"
#include "router_common.cuh"

namespace flint {
namespace {

// Phase trace (a separate build of the library, with FLINT_PHASE_TRACE
// defined, for the phase_trace tool): thread 0 of every CTA stamps %clock64 at
// the phase boundaries into shared memory and, at the end of the call, copies
// the stamps to a ring of the last kTraceCalls calls, indexed by the
// workspace's call count. The plain build has none of this code.
#ifdef FLINT_PHASE_TRACE
constexpr int kTraceStamps = 48, kTraceCalls = 64, kTraceCtas = 256;
__device__ unsigned long long g_phase_trace[kTraceCalls][kTraceCtas][kTraceStamps];
#define FLINT_PHASE(i)                                     \
    do {                                                   \
        if (threadIdx.x == 0) sm.trace[(i)] = clock64();   \
    } while (0)
#else
#define FLINT_PHASE(i) \
    do {               \
    } while (0)
#endif

constexpr int kLW = kLayerWarps;
constexpr int kLT = kLayerThreads;
constexpr int kMaxSegs = 4;
constexpr int kEpiBatch = 4;  // gate/up items per epilogue pass of a warp (8 measured slower)
constexpr int kMaxDownUnits = 4;
constexpr int kMaxVec = kMaxDownUnits * FLINT_MAX_TOKENS;
constexpr int kRowBlock = 16;                 // output rows per combine block
constexpr int kSharedUnit = -1;
constexpr int kShIdx = kMaxDistinct;          // index of the shared expert in the per-expert arrays
// Status bits after which a call must not run (the exchange counters may
// have been left mid-call).
constexpr uint32_t kStatusPoisonMask = kStatusTimeoutRoute | kStatusTimeoutGateUp | kStatusTimeoutDown |
                                       kStatusTimeoutSelftest | kStatusTimeoutLayer | kStatusTimeoutPrefill |
                                       kStatusLayerPlan;

// A run of a CTA's items from one expert: gate/up pairs [start, start +
// count) (one item each), or down rows [start, start + count) in items of rg
// rows.
struct Seg {
    int16_t unit;   // index into the distinct-expert list, or kSharedUnit
    int8_t q;       // down runs: index of the expert among the CTA's down experts
    int8_t rg;      // down runs: rows per item
    int32_t item0;  // the run's first item (CTA-local index)
    int32_t start, count;
};

struct LayerSmall {
    uint64_t wbar[kLW][kLayerSlots];  // warp w's ring slot s holds its item's bytes
    uint64_t rbar;                   // the router rows (and tensor scales) are in
    int32_t issued[kLW];             // items a warp has issued (for the drain on failure)
    uint32_t hdr[8];                 // workspace header at the start of the call
    int fail, n_last, ok;
    int n_gseg, n_dseg, n_gi, n_di;  // runs and items of this CTA
    int b0, b1;                      // this CTA's down range, in (expert, row block) items
    Seg gseg[kMaxSegs], dseg[kMaxDownUnits];
    int16_t vec[kMaxDownUnits][FLINT_MAX_TOKENS];  // staged h vector of (down expert, token), or -1
    int n_vec;
    int32_t v_item0[kMaxVec + 1];    // first 32-value staging item of each vector
    int32_t v_off[kMaxVec];          // byte offset of its f16 values in the staging region
    int32_t v_coff[kMaxVec];         // byte offset of its chunk scales
    int16_t v_q[kMaxVec], v_t[kMaxVec];
    float w[kMaxDistinct];
    int32_t ids[kMaxDistinct];
    // a warp's raw gate / up sums of its last items (per token), and per item
    // its pair (below 2^16: a slot holds a down row of I values, so I < 2 H <=
    // 16384), unit (kShIdx: the shared expert) and token mask
    float gres[kLW][kEpiBatch][2][FLINT_MAX_TOKENS];
    uint32_t gkey[kLW][kEpiBatch];
    float ninv[FLINT_MAX_TOKENS];
    int16_t last[kLayerMaxHidden / kRowBlock];  // row blocks this CTA combines
#ifdef FLINT_PHASE_TRACE
    unsigned long long trace[kTraceStamps];
    unsigned long long wend[kLW];  // when each warp left its gate/up loop
#endif
};

// Shared memory: small arrays, the routing view, the tensor scales of all
// routed experts, the staging region (x, then h of the CTA's down experts)
// and its chunk scales, the norm's partial sums, the router rows, the warps'
// rings.
struct LayerSmem {
    size_t small, ri, tsall, xs, csc, nred, rows, dres, ring, total;
};

__host__ __device__ inline LayerSmem layer_layout(const LayerArgs& a) {
    LayerSmem L;
    const size_t T = a.T, H = a.H;
    L.small = 0;
    L.ri = align_up(sizeof(LayerSmall), 128);
    L.tsall = align_up(L.ri + sizeof(RouteInfo), 128);
    L.xs = align_up(L.tsall + 12 * (size_t)a.E, 128);
    L.csc = align_up(L.xs + (size_t)a.stage_vals, 128);
    L.nred = align_up(L.csc + (size_t)a.stage_scales, 128);
    L.rows = align_up(L.nred + (a.norm.r ? sizeof(float) * T * (H / 32) : 0), 128);
    // ROWS: the CTA's expert outputs d[t][rank, or k: shared][row] (FP32
    // holding the bf16 values)
    L.dres = align_up(L.rows + 2 * (size_t)a.rpc * H, 128);
    L.ring = align_up(L.dres + (a.rows ? sizeof(float) * T * (a.k + 1) * (size_t)a.rows_max : 0), 128);
    L.total = L.ring + (size_t)kLW * a.ns * a.slot;
    return L;
}

__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t* p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}
// Publishes the CTA's earlier writes (ordered before this thread by a
// __syncthreads) and adds v to a counter at GPU scope: the fence, then the
// relaxed add (several adds may follow one fence).
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
__device__ __forceinline__ void red_add_relaxed_gpu(uint32_t* p, uint32_t v) {
    asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void release_add_gpu(uint32_t* p, uint32_t v) {
    fence_acq_rel_gpu();
    red_add_relaxed_gpu(p, v);
}
// Thread 0 waits until *p >= target (acquire), for at most budget_ns; the
// result reaches every thread of the CTA. `code` goes to *status on expiry.
__device__ __forceinline__ bool cta_wait_count(const uint32_t* p, uint32_t target, uint32_t* status, uint32_t code,
                                               uint64_t budget_ns, int* s_ok) {
    if (threadIdx.x == 0) {
        int ok = 1;
        if (ld_acquire_gpu(p) < target) {
            const uint64_t t0 = globaltimer_ns();
            while (ld_acquire_gpu(p) < target) {
                if (globaltimer_ns() - t0 > budget_ns) {
                    atomicOr(status, code);
                    ok = 0;
                    break;
                }
            }
        }
        *s_ok = ok;
    }
    __syncthreads();
    return *s_ok != 0;
}

// The routing view (the distinct selected experts in ascending id order, and
// per expert which ranks of which tokens chose it) built by one warp from the
// T x k ids in shared memory (every id valid, distinct within a token, E <=
// 1024, T k <= 64): lane l holds ids l and l + 32 and marks them in a bitmap
// of 32 words (word w: experts 32 w .. 32 w + 31); the prefix popcounts of the
// words give each selected expert its dense index.
__device__ void route_view_warp(RouteInfo& ri, const int32_t* ids, int T, int k, int lane) {
    const uint32_t full = 0xffffffffu;
    const int n = T * k;
    const int e0 = lane < n ? ids[lane] : -1, e1 = lane + 32 < n ? ids[lane + 32] : -1;
    ri.bitmap[lane] = 0u;
    __syncwarp();
    if (e0 >= 0) atomicOr(&ri.bitmap[e0 >> 5], 1u << (e0 & 31));
    if (e1 >= 0) atomicOr(&ri.bitmap[e1 >> 5], 1u << (e1 & 31));
    __syncwarp();
    const uint32_t word = ri.bitmap[lane], cnt = __popc(word);
    uint32_t incl = cnt;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t v = __shfl_up_sync(full, incl, off);
        if (lane >= off) incl += v;
    }
    const uint32_t base = incl - cnt;
    const int D = (int)__shfl_sync(full, incl, 31);
    auto dense = [&](int e) {  // every lane calls it (shuffles)
        const int src = e >= 0 ? e >> 5 : 0;
        const uint32_t bw = __shfl_sync(full, word, src), bb = __shfl_sync(full, base, src);
        return e >= 0 ? (int)(bb + __popc(bw & ((1u << (e & 31)) - 1u))) : -1;
    };
    const int d0 = dense(e0), d1 = dense(e1);
    if (lane < D) {
        ri.dmask[lane] = 0ull;
        ri.tmask[lane] = 0u;
    }
    if (lane + 32 < D) {
        ri.dmask[lane + 32] = 0ull;
        ri.tmask[lane + 32] = 0u;
    }
    __syncwarp();
    auto mark = [&](int i, int e, int d) {
        ri.ids[i] = e;  // -1: no expert (past T k, or an invalid given id)
        if (e < 0) return;
        const int t = i / k, j = i - t * k;
        ri.dlist[d] = e;  // (every lane holding e writes the same value)
        atomicOr(&ri.dmask[d], 1ull << (8 * t + j));
        atomicOr(&ri.tmask[d], 1u << t);
    };
    mark(lane, e0, d0);
    mark(lane + 32, e1, d1);
    if (lane == 0) ri.D = D;
    __syncwarp();
}

// This routed CTA's share of the D selected experts (one warp, after
// route_view_warp): the concatenation of the experts' items (per of each) is
// cut where the cumulative cost reaches the CTA's equal shares, an item of
// expert u costing w_u = 4 + 3 x its tokens (its decode once, a multiply-add
// per token). pos(tau) is the number of items whose cost starts below tau:
// the experts u with per cum[u] <= tau (cum: inclusive prefix of w) and the
// first ceil((tau - per cum[u - 1]) / w_u) items of the next one. Monotone in
// tau, pos(0) = 0, pos(per cum[D - 1]) = D per, so the CTAs' ranges tile the
// items exactly. Lane u holds cum[u] and cum[u + 32]; the search is two
// ballots. Returns (lo, hi) of share `cr` of `Gr` in lanes 0 and 1.
// (32-bit arithmetic: per cum[D - 1] (Gr + 1) < 2^32 for the shapes the host
// accepts.)
__device__ __forceinline__ void cost_split_warp(const RouteInfo& ri, int per_a, int per_b, uint32_t cr, uint32_t Gr,
                                                int lane, int& a0, int& a1, int& b0, int& b1, int& ua0, int& ub0) {
    const uint32_t full = 0xffffffffu;
    const int D = ri.D;
    uint32_t ca = lane < D ? 4u + 3u * __popc(ri.tmask[lane]) : 0u;
    uint32_t cb = lane + 32 < D ? 4u + 3u * __popc(ri.tmask[lane + 32]) : 0u;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t va = __shfl_up_sync(full, ca, off), vb = __shfl_up_sync(full, cb, off);
        if (lane >= off) {
            ca += va;
            cb += vb;
        }
    }
    cb += __shfl_sync(full, ca, 31);
    const uint32_t Wt = __shfl_sync(full, cb, 31);
    // lane q < 4 takes cut q: gate/up lo, hi; down lo, hi (the divisions in
    // parallel, the searches one after the other)
    const int q = lane & 3;
    const uint32_t per = (uint32_t)(q < 2 ? per_a : per_b);
    const uint32_t tau = (cr + (uint32_t)(q & 1)) * (Wt * per) / Gr;
    int lo = D;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t ti = __shfl_sync(full, tau, i), pi = (uint32_t)(i < 2 ? per_a : per_b);
        const uint32_t ma = __ballot_sync(full, lane < D && pi * ca > ti);
        const uint32_t mb = __ballot_sync(full, lane + 32 < D && pi * cb > ti);
        if (q == i) lo = ma ? __ffs(ma) - 1 : (mb ? 31 + __ffs(mb) : D);
    }
    // cum[lo] and cum[lo - 1] (each lane its own source)
    const int s1 = lo < D ? lo : 0, s0 = lo > 0 && lo < D ? lo - 1 : 0;
    const uint32_t x1 = __shfl_sync(full, ca, s1 & 31), y1 = __shfl_sync(full, cb, s1 & 31);
    const uint32_t x0 = __shfl_sync(full, ca, s0 & 31), y0 = __shfl_sync(full, cb, s0 & 31);
    int r = D * (int)per, u = D;  // the cut, and the expert it falls in
    if (lo < D) {
        const uint32_t cl = s1 < 32 ? x1 : y1, cp = lo ? (s0 < 32 ? x0 : y0) : 0u;
        const uint32_t wu = cl - cp, n = (tau - per * cp + wu - 1u) / wu;
        r = lo * (int)per + (int)(n < per ? n : per);
        u = n < per ? lo : lo + 1;
    }
    ua0 = __shfl_sync(full, u, 0);
    ub0 = __shfl_sync(full, u, 2);
    a0 = __shfl_sync(full, r, 0);
    a1 = __shfl_sync(full, r, 1);
    b0 = __shfl_sync(full, r, 2);
    b1 = __shfl_sync(full, r, 3);
}

// The runs of the pair range [p0, p1) and of the down block range [b0, b1)
// (items of a concatenation of experts of per_gu pairs / NB blocks: the
// routed experts in list order, or the shared expert alone); a down item
// takes rg rows. One thread.
__device__ void build_segs(LayerSmall& sm, int p0, int up0, int p1, int per_gu, int b0, int ub0, int b1, int NB,
                           uint32_t* status, bool shared, int rg) {
    // up0, ub0: the experts that p0 and b0 fall in (p0 / per_gu, b0 / NB)
    int n = 0;
    for (int P = p0, u = up0, p = p0 - u * per_gu; P < p1; ++u, p = 0) {
        const int m = min(p1 - P, per_gu - p);
        if (n == kMaxSegs) {
            sm.fail = 1;  // the host sizes the grid so that this cannot happen
            atomicOr(status, kStatusLayerPlan);
            break;
        }
        sm.gseg[n++] = Seg{(int16_t)(shared ? kSharedUnit : u), 0, 0, P - p0, p, m};
        P += m;
    }
    sm.n_gseg = n;
    sm.n_gi = p1 > p0 ? p1 - p0 : 0;
    int nd = 0, items = 0;
    const int rg_log2 = __ffs(rg) - 1;  // rg is a power of two
    for (int B = b0, u = ub0, b = b0 - u * NB; B < b1; ++u, b = 0) {
        const int take = min(b1 - B, NB - b);
        if (nd == kMaxDownUnits) {
            sm.fail = 1;
            atomicOr(status, kStatusLayerPlan);
            break;
        }
        const int rows = take * kRowBlock;
        sm.dseg[nd] = Seg{(int16_t)(shared ? kSharedUnit : u), (int8_t)nd, (int8_t)rg, items, b * kRowBlock, rows};
        items += (rows + rg - 1) >> rg_log2;
        ++nd;
        B += take;
    }
    sm.n_dseg = nd;
    sm.n_di = items;
    sm.b0 = b0;
    sm.b1 = b1;
}

// NORM: the input is rmsnorm(r + y_prev) of the residual stream (a.norm), not
// a.x. Two instantiations, so that the plain layer carries none of the norm's
// code (measured: a never-taken norm branch cost 3-4 us at T = 8).
template <bool NORM, bool ROWS, bool GIVEN>
__global__ void __launch_bounds__(kLT, 1) layer_kernel(const LayerArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const LayerSmem L = layer_layout(a);
    const int T = a.T, H = a.H, E = a.E, k = a.k, I = a.I, Is = a.Is;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = blockIdx.x, G = gridDim.x, Gs = a.Gs;
    constexpr int NSW = kLayerSlots;
    const bool sh_cta = c < Gs;
    const bool has_sh = a.s_gu != nullptr;
    LayerSmall& sm = *reinterpret_cast<LayerSmall*>(smem + L.small);
    RouteInfo& ri = *reinterpret_cast<RouteInfo*>(smem + L.ri);
    uint4* xh = reinterpret_cast<uint4*>(smem + L.xs);
    float* csc = reinterpret_cast<float*>(smem + L.csc);
    uint8_t* wring = smem + L.ring + (size_t)warp * NSW * a.slot;  // this warp's ring
    uint64_t* wbar = sm.wbar[warp];
    const int RS = (int)nvfp4_row_stride(H), RSr = (int)nvfp4_row_stride(I);
    const int RSs = Is ? (int)nvfp4_row_stride(Is) : 0;
    const int NB = H / kRowBlock;
    // ROWS: this CTA's output rows [R0, R1), in down items of rg rows (ng per
    // expert)
    const int R0 = c * H / G, R1 = (c + 1) * H / G, nrows = R1 - R0;
    const int ng = (nrows + a.rg - 1) / a.rg;
    // router rows: rpc each on the routed CTAs (the shared CTAs queue their
    // expert's copies before the PDL wait and would publish late)
    const int r0 = (c - Gs) * a.rpc, nrr = (GIVEN || sh_cta) ? 0 : max(0, min(a.rpc, E - r0));
    const uint32_t full_mask = 0xffffffffu;
    // The routed group copies the tensor scales of all routed experts before
    // the PDL wait (static; one bulk copy when their bytes allow it).
    const bool ts_bulk = !sh_cta && (reinterpret_cast<uintptr_t>(a.ts) % 16 == 0) && ((12 * E) % 16 == 0);
    const uint32_t rbar_bytes = (uint32_t)(nrr * H * 2) + (ts_bulk ? 12u * (uint32_t)E : 0u);
    const float* tsall = reinterpret_cast<const float*>(smem + L.tsall);
    // tensor scale j (gate, up, down) of unit u: the shared expert, or routed
    // expert ri.dlist[u] (from the copy of all of them when there is one)
    auto tscale = [&](bool sh, int u, int j) -> float {
        if (sh) return __ldg(a.s_ts + j);
        const int e = ri.dlist[u];
        return ts_bulk ? tsall[3 * e + j] : __ldg(a.ts + 3 * e + j);
    };
    // rows per down item: up to 8 (4 when the CTA has at most 4 per warp), as
    // many as one slot holds
    auto rows_per_item = [&](int RSu, int rows) {
        int rg = rows <= 4 * kLW ? 4 : 8;
        while (rg > 1 && rg * RSu > a.slot) rg >>= 1;
        return rg;
    };

    // This warp's items: the CTA's gate/up items warp, warp + kLW, ... then
    // its down items warp, warp + kLW, ... (sequence index it).
    int my_g = 0, my_d = 0;
    auto count_mine = [&]() {
        my_g = sm.n_gi > warp ? (sm.n_gi - warp + kLW - 1) / kLW : 0;
        my_d = sm.n_di > warp ? (sm.n_di - warp + kLW - 1) / kLW : 0;
    };
    // Issues item `it` of this warp's sequence into its slot (lane 0).
    auto issue = [&](int it) {
        const int slot = it % NSW;
        uint8_t* dst = wring + (size_t)slot * a.slot;
        uint64_t* bar = wbar + slot;
        fence_proxy_async_smem();  // the slot's earlier reads come first
        if (it < my_g) {
            const int m = warp + it * kLW;
            int s = 0;
            while (s + 1 < sm.n_gseg && sm.gseg[s + 1].item0 <= m) ++s;
            const Seg sg = sm.gseg[s];
            const bool sh = sg.unit == kSharedUnit;
            const int p = sg.start + (m - sg.item0);
            const uint8_t* g = sh ? a.s_gu : a.gu + (size_t)ri.dlist[sg.unit] * 2 * I * RS;
            mbar_arrive_expect_tx(bar, 2u * (uint32_t)RS);
            bulk_g2s(dst, g + (size_t)p * RS, (uint32_t)RS, bar);
            bulk_g2s(dst + RS, g + (size_t)((sh ? Is : I) + p) * RS, (uint32_t)RS, bar);
        } else if constexpr (ROWS) {
            // down item m: rows [R0 + rg (m % ng), + rg) of unit m / ng (the
            // routed experts in list order, then the shared expert)
            const int m = warp + (it - my_g) * kLW;
            const int u = m / ng, r = R0 + (m - u * ng) * a.rg, nr = min(a.rg, R1 - r);
            const bool sh = u == ri.D;
            const int RSu = sh ? RSs : RSr;
            const uint8_t* d = sh ? a.s_down : a.down + (size_t)ri.dlist[u] * H * RSr;
            mbar_arrive_expect_tx(bar, (uint32_t)(nr * RSu));
            bulk_g2s(dst, d + (size_t)r * RSu, (uint32_t)(nr * RSu), bar);
        } else {
            const int m = warp + (it - my_g) * kLW;
            int s = 0;
            while (s + 1 < sm.n_dseg && sm.dseg[s + 1].item0 <= m) ++s;
            const Seg sg = sm.dseg[s];
            const bool sh = sg.unit == kSharedUnit;
            const int RSu = sh ? RSs : RSr;
            const int r = sg.start + (m - sg.item0) * sg.rg, nr = min((int)sg.rg, sg.start + sg.count - r);
            const uint8_t* d = sh ? a.s_down : a.down + (size_t)ri.dlist[sg.unit] * H * RSr;
            mbar_arrive_expect_tx(bar, (uint32_t)(nr * RSu));
            bulk_g2s(dst, d + (size_t)r * RSu, (uint32_t)(nr * RSu), bar);
        }
        sm.issued[warp] = it + 1;
    };
    // Before an early exit: the bulk copies still in flight into this CTA's
    // shared memory land first (bounded; thread 0 for the router rows, lane 0
    // of each warp for its ring).
    auto drain = [&](uint64_t budget_ns) {
        if (tid == 0 && rbar_bytes) mbar_wait_bounded(&sm.rbar, 0, nullptr, 0, budget_ns);
        if (lane == 0) {
            const int n = sm.issued[warp];
            for (int it = max(0, n - NSW); it < n; ++it)
                mbar_wait_bounded(wbar + it % NSW, (uint32_t)(it / NSW) & 1u, nullptr, 0, budget_ns);
        }
    };

    // ---- 0: before the PDL wait: barriers, static weight copies ----------------------
#ifdef FLINT_PHASE_TRACE
    if (tid < kTraceStamps) sm.trace[tid] = 0;
    const uint64_t trace_t0 = globaltimer_ns();
#endif
    FLINT_PHASE(0);
    if (tid < kLW * NSW) mbar_init(&sm.wbar[tid / NSW][tid % NSW], 1);
    if (tid < kLW) sm.issued[tid] = 0;
    if (tid == 0) {
        mbar_init(&sm.rbar, 1);
        sm.fail = 0;
        sm.n_last = 0;
        sm.n_gi = sm.n_di = sm.n_gseg = sm.n_dseg = 0;
        sm.b0 = sm.b1 = 0;
        if (sh_cta) {
            // the shared expert: an even split of its pairs and row blocks
            // (ROWS: no row blocks; its down items come with the routing)
            const int p0 = (int)((long long)c * Is / Gs), p1 = (int)((long long)(c + 1) * Is / Gs);
            const int b0 = ROWS ? 0 : (int)((long long)c * NB / Gs), b1 = ROWS ? 0 : (int)((long long)(c + 1) * NB / Gs);
            build_segs(sm, p0, 0, p1, Is, b0, 0, b1, NB, a.status, true, rows_per_item(RSs, (b1 - b0) * kRowBlock));
        }
    }
    if (tid <= kLW * NSW) fence_mbar_init();
    __syncthreads();
    if (tid == 0) {
        if (rbar_bytes) mbar_arrive_expect_tx(&sm.rbar, rbar_bytes);
        if (nrr > 0) bulk_g2s(smem + L.rows, a.wr + (size_t)r0 * H, (uint32_t)(nrr * H * 2), &sm.rbar);
        if (ts_bulk) bulk_g2s(smem + L.tsall, a.ts, 12u * (uint32_t)E, &sm.rbar);
    }
    if (sh_cta) {
        count_mine();
        if (lane == 0 && !sm.fail)
            for (int it = 0; it < NSW && it < my_g + my_d; ++it) issue(it);
    }
    const StageSrc xsrc[1] = {{a.x, xh, csc, T, H}};
    auto stage_x = [&]() {
        if constexpr (NORM)
            stage_norm_f16<ROWS>(a.norm, xsrc[0], reinterpret_cast<float*>(smem + L.nred), sm.ninv, c, G);
        else
            stage_f16<false>(xsrc, [] {});
    };
    // Given routing right after the router on the same x: the router lets its
    // dependents launch only once its own wait has returned, so x is complete
    // and is staged before this kernel's wait (the ids and weights are not).
    const bool x_early = GIVEN && a.x_early;
    if (x_early) stage_x();
    // Dependents may launch now: their CTAs take SMs as ours exit, and only
    // read static weights before their own wait.
    pdl_launch_dependents();
    pdl_wait();  // x (or the residual stream) comes from the previous kernel
    FLINT_PHASE(1);

    // ---- 1: the call's header, x; this CTA's router scores ---------------------------
    if (tid == 0) {
        const uint4 h0 = ld_cg(reinterpret_cast<const uint4*>(a.hdr));
        const uint4 h1 = ld_cg(reinterpret_cast<const uint4*>(a.hdr) + 1);
        sm.hdr[0] = h0.x; sm.hdr[1] = h0.y; sm.hdr[2] = h0.z; sm.hdr[3] = h0.w;
        sm.hdr[4] = h1.x; sm.hdr[5] = h1.y; sm.hdr[6] = h1.z; sm.hdr[7] = h1.w;
    }
    if (!x_early) stage_x();
    __syncthreads();
    FLINT_PHASE(2);
    const uint64_t budget = sm.hdr[kHdrBudget] ? (uint64_t)sm.hdr[kHdrBudget] * 1000ull : kWaitBudgetNs;
    if (sm.hdr[kHdrStatus] & kStatusPoisonMask) {  // an earlier call failed: re-initialise first
        drain(budget);
        return;
    }
    // test hook: this CTA publishes nothing (no router scores, no h counts)
    const bool withhold = sm.hdr[kHdrLoseCta] == (uint32_t)c + 1u;
    if (nrr > 0) {
        const bool ok = mbar_wait_bounded(&sm.rbar, 0, a.status, kStatusTimeoutLayer, budget);
        if (!ok) sm.fail = 1;
        FLINT_PHASE(35);
        const uint16_t* wrows = reinterpret_cast<const uint16_t*>(smem + L.rows);
        // logits from the staged (exact, chunk-scaled f16) x, one warp per
        // (row, token): lane l takes the 32-value chunks l, l + 32, ...; each
        // chunk's FP32 partial sum is multiplied back by its power-of-two scale
        for (int q = warp; ok && q < nrr * T; q += kLW) {
            const int r = q / T, t = q - r * T;
            const uint4* xb = xh + (size_t)t * (H / 8) + lane;
            const float* cb = csc + (size_t)t * (H / 32) + lane;
            const uint4* wv = reinterpret_cast<const uint4*>(wrows + (size_t)r * H);
            float v = 0.f;
            for (int m = 0; m < H / 1024; ++m) {
                const int ch = lane + 32 * m;
                float s0 = 0.f, s1 = 0.f;
#pragma unroll
                for (int w0 = 0; w0 < 4; ++w0) {
                    // lanes 2i, 2i + 1 start at word i % 4 of their 64-byte chunk,
                    // so that a wavefront's eight 16-byte reads hit distinct banks
                    const int w = (w0 + (lane >> 1)) & 3;
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
            for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(full_mask, v, off);
            if (lane == 0) a.scores[(size_t)t * E + r0 + r] = sigmoid_score(v, a.bias, r0 + r);
        }
        __syncthreads();
        FLINT_PHASE(36);
        if (tid == 0 && ok && !withhold) release_add_gpu(a.hdr + kHdrScoresIn, (uint32_t)nrr);
        FLINT_PHASE(37);
#ifdef FLINT_PHASE_TRACE
        if (tid == 0) sm.trace[26] = globaltimer_ns();
#endif
    }
    FLINT_PHASE(3);
    // The next layer's static weights into L2, issued once this CTA's router
    // scores are out (HBM is otherwise idle while the routing runs; issued
    // before the PDL wait it measured slower, competing with the previous
    // kernel's stream): CTA c takes granules [c n / G, (c + 1) n / G) of the
    // ranges' concatenation (16-byte granules), in bulk L2 prefetches of up
    // to 32 KB.
    if (tid == kLT - 1 && a.pf_granules) {
        const unsigned long long g0 = a.pf_granules * c / G, g1 = a.pf_granules * (c + 1) / G;
        unsigned long long base = 0;
        for (int r = 0; r < 4; ++r) {
            const unsigned long long n = a.pf_bytes[r] / 16;
            const unsigned long long lo = max(g0, base), hi = min(g1, base + n);
            for (unsigned long long q = lo; q < hi;) {
                const unsigned long long m = min(hi - q, 2048ull);
                bulk_prefetch_l2(a.pf_ptr[r] + (q - base) * 16, (uint32_t)(m * 16));
                q += m;
            }
            base += n;
        }
    }

    // Routing in this CTA: once all E router rows are published, all T x E
    // scores into shared memory over the router rows and the top-k of each
    // token (one warp per token). Every thread calls it; false (in every
    // thread) if the scores never came.
    auto route = [&](int stamp) -> bool {
        (void)stamp;
        if constexpr (GIVEN) {
            // the caller's ids and weights (written by an earlier kernel: read
            // through L2); an id outside [0, E) is reported and becomes -1
            if (tid < T * k) {
                int e = ld_cg(a.ids + tid);
                if (e < 0 || e >= E) {
                    atomicOr(a.status, kStatusBadExpertId);
                    e = -1;
                }
                sm.ids[tid] = e;
                sm.w[tid] = ld_cg(a.weights + tid);
            }
            __syncthreads();
            FLINT_PHASE(stamp + 2);
            return !sm.fail;
        }
        if (!cta_wait_count(a.hdr + kHdrScoresIn, (uint32_t)E, a.status, kStatusTimeoutLayer, budget, &sm.ok) ||
            sm.fail)
            return false;
        FLINT_PHASE(stamp);
        FLINT_PHASE(stamp + 1);
        if (warp < T) {  // each token's scores read from L2 by its warp
            const uint32_t* sc = a.scores + (size_t)warp * E;
            if (E <= 256)
                topk_warp<8, true>(sc, E, k, lane, sm.ids + warp * k, sm.w + warp * k);
            else
                topk_warp<FLINT_MAX_EXPERTS / 32, true>(sc, E, k, lane, sm.ids + warp * k, sm.w + warp * k);
        }
        __syncthreads();
        FLINT_PHASE(stamp + 2);
        return true;
    };

    bool failed = false;
    if (!sh_cta) {
        // ---- 2: routing, this CTA's share of the selected experts ---------------
        if (!route(11)) {
            failed = true;
        } else {
            if (!GIVEN && c == G - 1 && tid < T * k) {
                a.ids[tid] = sm.ids[tid];
                a.weights[tid] = sm.w[tid];
            }
            if (warp == 0) {
                route_view_warp(ri, sm.ids, T, k, lane);
                FLINT_PHASE(14);
                int p0, p1, b0, b1, up0, ub0;
                cost_split_warp(ri, I, NB, (uint32_t)(c - Gs), (uint32_t)(G - Gs), lane, p0, p1, b0, b1, up0, ub0);
                if (lane == 0) {
                    if constexpr (ROWS) {
                        build_segs(sm, p0, up0, p1, I, 0, 0, 0, NB, a.status, false, 1);
                        sm.n_di = (ri.D + (has_sh ? 1 : 0)) * ng;
                    } else {
                        build_segs(sm, p0, up0, p1, I, b0, ub0, b1, NB, a.status, false,
                                   rows_per_item(RSr, (b1 - b0) * kRowBlock));
                    }
                }
                FLINT_PHASE(19);
            }
            // the segments are in; the tensor scales of all routed experts too
            // (copied before the PDL wait; the CTAs with router rows waited for
            // them already)
            if (ts_bulk && nrr == 0 && !mbar_wait_bounded(&sm.rbar, 0, a.status, kStatusTimeoutLayer, budget))
                sm.fail = 1;
            __syncthreads();
            FLINT_PHASE(38);
            count_mine();
            if (lane == 0 && !sm.fail)
                for (int it = 0; it < NSW && it < my_g + my_d; ++it) issue(it);
            FLINT_PHASE(39);
        }
    }
    // (no CTA barrier here: each warp goes on to its own items; `failed` is
    // the same in every thread, and sm.fail was last set before the barrier
    // above or is checked per item)
    FLINT_PHASE(4);

    // ---- 3-4: this warp's ring: gate/up items, then (h of the down experts staged) down items --
    if (failed) my_g = my_d = 0;
    bool wfail = false;  // this warp gave up on a copy
#ifdef FLINT_PHASE_TRACE
    unsigned long long wait_gu = 0, wait_dn = 0;  // warp 0: cycles spent waiting for item bytes
    unsigned long long t_math = 0, t_epi = 0;      // warp 0: gate/up arithmetic; epilogue and refill
#endif
    // Waits for item it's bytes (all lanes; false once anything failed).
    auto item_in = [&](int it) {
#ifdef FLINT_PHASE_TRACE
        const unsigned long long tw = clock64();
#endif
        if (!wfail && !sm.fail) {
            if (__all_sync(full_mask, mbar_wait_bounded(wbar + it % NSW, (uint32_t)(it / NSW) & 1u, a.status,
                                                        kStatusTimeoutLayer, budget))) {
#ifdef FLINT_PHASE_TRACE
                (it < my_g ? wait_gu : wait_dn) += clock64() - tw;
#endif
                return true;
            }
            if (lane == 0) sm.fail = 1;
        }
        wfail = true;
        return false;
    };
    // Done with item it: lane 0 refills its slot with item it + NSW.
    auto item_done = [&](int it) {
        __syncwarp();
        if (lane == 0 && it + NSW < my_g + my_d && !sm.fail) issue(it + NSW);
    };
    // The epilogue of a warp's buffered items, one (item, token) per lane:
    // h = bf16(silu(bf16(ts_g g)) bf16(ts_u u)).
    int nb = 0;
    auto epilogue = [&]() {
        __syncwarp();
        for (int e = lane; e < nb * FLINT_MAX_TOKENS; e += 32) {
            const int b = e / FLINT_MAX_TOKENS, t = e % FLINT_MAX_TOKENS;
            const uint32_t key = sm.gkey[warp][b];
            if (!((key >> (24 + t)) & 1u)) continue;
            const int p = (int)(key & 0xFFFFu), ui = (int)((key >> 16) & 0xFFu);
            const bool sh = ui == kShIdx;
            const float g = bf16_round_f32(tscale(sh, ui, 0) * sm.gres[warp][b][0][t]);
            const float u = bf16_round_f32(tscale(sh, ui, 1) * sm.gres[warp][b][1][t]);
            const uint16_t hv = f32_to_bf16_bits(silu_f32(g) * u);
            if (sh) {
                a.h_shared[(size_t)t * Is + p] = hv;
            } else {
                const int j = __ffs(rank_bits(ri.dmask[ui], t)) - 1;
                a.h_routed[((size_t)t * k + j) * I + p] = hv;
            }
        }
        __syncwarp();
        nb = 0;
    };
    // the run the current item falls in, kept from one item to the next
    int cg_s = -1, cg_next = 0, cg_start = 0, cg_item0 = 0, cg_ui = 0;
    uint32_t cg_tm = 0;
    for (int it = 0; it < my_g; ++it) {
        if (!item_in(it)) break;
        if (it == 0) FLINT_PHASE(5);
        const int m = warp + it * kLW;
        while (m >= cg_next) {
            const Seg sg = sm.gseg[++cg_s];
            cg_next = cg_s + 1 < sm.n_gseg ? sm.gseg[cg_s + 1].item0 : INT_MAX;
            cg_start = sg.start;
            cg_item0 = sg.item0;
            const bool sh = sg.unit == kSharedUnit;
            cg_ui = sh ? kShIdx : sg.unit;
            cg_tm = sh ? (1u << T) - 1u : ri.tmask[sg.unit];
        }
        const uint8_t* grow = wring + (size_t)(it % NSW) * a.slot;
#ifdef FLINT_PHASE_TRACE
        const unsigned long long tm0 = clock64();
#endif
        gate_up_item<true>(grow, grow + RS, H, xh, csc, cg_tm, lane, sm.gres[warp][nb][0], sm.gres[warp][nb][1]);
        if (lane == 0)
            sm.gkey[warp][nb] = (uint32_t)(cg_start + (m - cg_item0)) | ((uint32_t)cg_ui << 16) | (cg_tm << 24);
        ++nb;
#ifdef FLINT_PHASE_TRACE
        const unsigned long long tm1 = clock64();
        t_math += tm1 - tm0;
#endif
        item_done(it);  // the slot is free once the sums are out
        if (nb == kEpiBatch) epilogue();
#ifdef FLINT_PHASE_TRACE
        t_epi += clock64() - tm1;
#endif
    }
    if (nb > 0) epilogue();
#ifdef FLINT_PHASE_TRACE
    if (lane == 0) sm.wend[warp] = clock64();
#endif
    // Publish this CTA's h: per expert, the number of its pairs done here.
    if (__syncthreads_or(wfail) && tid == 0) sm.fail = 1;
    if constexpr (ROWS) {
        // ROWS: publish the number of this CTA's pairs done; the shared group
        // learns the routing, and with it its down items; every CTA stages all of
        // h once every pair is published, then computes its rows of every
        // expert's down GEMV and of y.
        if (tid == 0 && !sm.fail && !failed && !withhold && sm.n_gi > 0)
            release_add_gpu(a.hdr + kHdrPairsIn, (uint32_t)sm.n_gi);
        FLINT_PHASE(6);
        if (!__syncthreads_or(failed || sm.fail) && sh_cta) {
            failed = !route(40);
            if (!failed && warp == 0) {
                route_view_warp(ri, sm.ids, T, k, lane);
                if (lane == 0) sm.n_di = (ri.D + (has_sh ? 1 : 0)) * ng;
            }
            __syncthreads();
            FLINT_PHASE(43);
            if (!failed) {
                count_mine();
                if (lane == 0 && !sm.fail)
                    for (int it = my_g; it < my_g + NSW && it < my_g + my_d; ++it) issue(it);
            }
        }
        const int D = ri.D;
        const uint32_t pairs = (uint32_t)D * (uint32_t)I + (has_sh ? (uint32_t)Is : 0u);
        if (failed || sm.fail ||
            !cta_wait_count(a.hdr + kHdrPairsIn, pairs, a.status, kStatusTimeoutLayer, budget, &sm.ok) || sm.fail) {
            drain(budget);
            return;
        }
        // the routed h [T][k][I] (vector t k + j), then the shared h [T][Is]
        const StageSrc hsrc[2] = {{a.h_routed, xh, csc, T * k, I},
                                  {a.h_shared, xh + (size_t)T * k * (I / 8), csc + (size_t)T * k * (I / 32),
                                   has_sh ? T : 0, has_sh ? Is : 32}};
        stage_f16_quarters<true>(hsrc);
        __syncthreads();
        FLINT_PHASE(7);
        float* dres = reinterpret_cast<float*>(smem + L.dres);
        auto dslot = [&](int t, int j, int r) -> float& { return dres[((size_t)t * (k + 1) + j) * a.rows_max + r]; };
        // the unit of the current down item and what it needs, kept from one item
        // to the next
        int cu = -1;
        bool sh = false;
        uint32_t tm = 0;
        float tsd = 0.f;
        unsigned long long dm = 0ull;
        for (int it = my_g; it < my_g + my_d; ++it) {
            if (!item_in(it)) break;
            const int m = warp + (it - my_g) * kLW;
            const int u = m / ng;
            if (u != cu) {
                cu = u;
                sh = u == D;
                tm = sh ? (1u << T) - 1u : ri.tmask[u];
                tsd = tscale(sh, u, 2);
                dm = sh ? 0ull : ri.dmask[u];
            }
            const int rl = (m - u * ng) * a.rg, nrw = min(a.rg, nrows - rl);  // local rows [rl, rl + nrw)
            const int K = sh ? Is : I, RSu = sh ? RSs : RSr;
            const uint8_t* rows = wring + (size_t)(it % NSW) * a.slot;
            // token t's rank of this expert (k: the shared expert) and its staged h
            auto rank = [&](int t) { return sh ? k : __ffs(rank_bits(dm, t)) - 1; };
            auto vec = [&](int t, int j, const uint4*& hv, const float*& cv) {
                if (sh) {
                    hv = hsrc[1].dst + (size_t)t * (Is / 8);
                    cv = hsrc[1].csc + (size_t)t * (Is / 32);
                } else {
                    hv = xh + (size_t)(t * k + j) * (I / 8);
                    cv = csc + (size_t)(t * k + j) * (I / 32);
                }
            };
            auto put = [&](float v, int r, int t, int j) {
                const float d = bf16_round_f32(tsd * v);
                if (GIVEN && !sh) {  // every rank of the token that chose this expert
                    for (uint32_t b = rank_bits(dm, t); b; b &= b - 1u) dslot(t, __ffs(b) - 1, rl + r) = d;
                } else {
                    dslot(t, j, rl + r) = d;
                }
            };
            // rows [0, nrw) against one or two tokens (rows past nrw are skipped inside)
            constexpr int RP = 8;
            uint32_t rest = tm;
            while (rest) {
                const int t0 = __ffs(rest) - 1;
                rest &= rest - 1u;
                const int j0 = rank(t0);
                if (rest) {
                    const int t1 = __ffs(rest) - 1;
                    rest &= rest - 1u;
                    const int j1 = rank(t1);
                    const uint4* hv[2];
                    const float* cv[2];
                    vec(t0, j0, hv[0], cv[0]);
                    vec(t1, j1, hv[1], cv[1]);
                    float acc[2 * RP];
                    down_pass<RP, 2>(rows, RSu, nrw, K, hv, cv, lane, acc);
                    const float v = reduce_scatter<2 * RP>(acc, lane);
                    const int idx = rs_index<2 * RP>(lane), r = idx % RP;
                    if (lane % (16 / RP) == 16 / RP - 1 && r < nrw) {
                        if (idx >= RP) put(v, r, t1, j1);
                        else put(v, r, t0, j0);
                    }
                } else {
                    const uint4* hv[1];
                    const float* cv[1];
                    vec(t0, j0, hv[0], cv[0]);
                    float acc[RP];
                    down_pass<RP, 1>(rows, RSu, nrw, K, hv, cv, lane, acc);
                    const float v = reduce_scatter<RP>(acc, lane);
                    const int r = rs_index<RP>(lane);
                    if (lane % (32 / RP) == 32 / RP - 1 && r < nrw) put(v, r, t0, j0);
                }
            }
            item_done(it);
        }
        if (__syncthreads_or(wfail || sm.fail)) {
            drain(budget);
            return;
        }
        FLINT_PHASE(8);
        // y = bf16(sum_j w_j d_j + d_shared), ranks in order, one (token, row) per thread
        for (int e = tid; e < T * nrows; e += kLT) {
            const int t = e / nrows, r = e - t * nrows;
            float acc = 0.f;
            for (int j = 0; j < k; ++j)
                if (!GIVEN || ri.ids[t * k + j] >= 0) acc = fmaf(sm.w[t * k + j], dslot(t, j, r), acc);
            if (has_sh) acc += dslot(t, k, r);
            a.y[(size_t)t * H + R0 + r] = f32_to_bf16_bits(acc);
        }
        FLINT_PHASE(10);

    } else {
        if (tid == 0 && !sm.fail && !failed && !withhold && sm.n_gseg > 0) {
            fence_acq_rel_gpu();  // one fence for all of them
            for (int s = 0; s < sm.n_gseg; ++s) {
                const int unit = sm.gseg[s].unit;
                red_add_relaxed_gpu(a.unit_counters + (unit == kSharedUnit ? kShIdx : unit), (uint32_t)sm.gseg[s].count);
            }
        }
        FLINT_PHASE(6);
        if (!failed && sm.n_di > 0) {
            // Stage h of this CTA's down experts once every pair of each is published.
            if (tid == 0) {
                int nv = 0, item = 0, off = 0, coff = 0;
                for (int q = 0; q < sm.n_dseg; ++q) {
                    const int unit = sm.dseg[q].unit;
                    const int K = unit == kSharedUnit ? Is : I;
                    const uint32_t tm = unit == kSharedUnit ? (1u << T) - 1u : ri.tmask[unit];
                    for (int t = 0; t < FLINT_MAX_TOKENS; ++t) {
                        sm.vec[q][t] = -1;
                        if (t < T && ((tm >> t) & 1u)) {
                            sm.vec[q][t] = (int16_t)nv;
                            sm.v_item0[nv] = item;
                            sm.v_off[nv] = off;
                            sm.v_coff[nv] = coff;
                            sm.v_q[nv] = (int16_t)q;
                            sm.v_t[nv] = (int16_t)t;
                            item += K / 32;
                            off += 2 * K;
                            coff += 4 * (K / 32);
                            ++nv;
                        }
                    }
                }
                if (off > a.stage_vals || coff > a.stage_scales) {  // the host plans for this not to happen
                    atomicOr(a.status, kStatusLayerPlan);
                    sm.fail = 1;
                    nv = 0;
                    item = 0;
                }
                sm.n_vec = nv;
                sm.v_item0[nv] = item;
            }
            bool ok = true;
            for (int q = 0; q < sm.n_dseg && ok; ++q) {  // sm.n_dseg: written before the earlier barriers
                const int unit = sm.dseg[q].unit;
                ok = cta_wait_count(a.unit_counters + (unit == kSharedUnit ? kShIdx : unit),
                                    (uint32_t)(unit == kSharedUnit ? Is : I), a.status, kStatusTimeoutLayer, budget,
                                    &sm.ok);
            }
            ok = ok && !sm.fail;
            const int n_items = ok ? sm.v_item0[sm.n_vec] : 0;
            for (int q = tid; q < n_items; q += kLT) {
                int v = 0;
                while (sm.v_item0[v + 1] <= q) ++v;
                const int cc = q - sm.v_item0[v], t = sm.v_t[v];
                const int unit = sm.dseg[sm.v_q[v]].unit;
                const bool sh = unit == kSharedUnit;
                const int K = sh ? Is : I;
                const uint16_t* src;
                if (sh) {
                    src = a.h_shared + (size_t)t * Is;
                } else {
                    const int j = __ffs(rank_bits(ri.dmask[unit], t)) - 1;
                    src = a.h_routed + ((size_t)t * k + j) * I;
                }
                const StageSrc ss = {src, reinterpret_cast<uint4*>(smem + L.xs + sm.v_off[v]),
                                     reinterpret_cast<float*>(smem + L.csc + sm.v_coff[v]), 1, K};
                uint4 w4[4];
                stage_load(ss, 0, cc, w4);
                stage_store<true>(ss, 0, cc, w4);
            }
            if (!__syncthreads_and(ok)) wfail = true;
        }
        FLINT_PHASE(7);
        // the run of the current down item and what it needs, kept from one item
        // to the next
        int cd_s = -1, cd_next = 0;
        Seg sg = {};
        bool sh = false;
        uint32_t tm = 0;
        float tsd = 0.f;
        unsigned long long dm = 0ull;
        for (int it = my_g; it < my_g + my_d; ++it) {
            if (!item_in(it)) break;
            const int m = warp + (it - my_g) * kLW;
            while (m >= cd_next) {
                sg = sm.dseg[++cd_s];
                cd_next = cd_s + 1 < sm.n_dseg ? sm.dseg[cd_s + 1].item0 : INT_MAX;
                sh = sg.unit == kSharedUnit;
                tm = sh ? (1u << T) - 1u : ri.tmask[sg.unit];
                tsd = tscale(sh, sg.unit, 2);
                dm = sh ? 0ull : ri.dmask[sg.unit];
            }
            const int row0 = sg.start + (m - sg.item0) * sg.rg;
            const int nrw = min((int)sg.rg, sg.start + sg.count - row0);
            const int K = sh ? Is : I, RSu = sh ? RSs : RSr;
            const uint8_t* rows = wring + (size_t)(it % NSW) * a.slot;
            auto vec = [&](int t, const uint4*& hv, const float*& cv) {
                const int v = sm.vec[sg.q][t];
                hv = reinterpret_cast<const uint4*>(smem + L.xs + sm.v_off[v]);
                cv = reinterpret_cast<const float*>(smem + L.csc + sm.v_coff[v]);
            };
            auto put = [&](float v, int r, int t) {
                const uint16_t d = f32_to_bf16_bits(tsd * v);
                if (sh) {
                    a.d_shared[(size_t)t * H + row0 + r] = d;
                } else if constexpr (GIVEN) {  // every rank of the token that chose this expert
                    for (uint32_t b = rank_bits(dm, t); b; b &= b - 1u)
                        a.d_routed[((size_t)t * k + __ffs(b) - 1) * H + row0 + r] = d;
                } else {
                    const int j = __ffs(rank_bits(dm, t)) - 1;
                    a.d_routed[((size_t)t * k + j) * H + row0 + r] = d;
                }
            };
            // rows [0, nrw) of the item against one or two tokens
            auto rows_pass = [&](auto rp_tag, int t0, int t1) {
                constexpr int RP = decltype(rp_tag)::value;
                if (t1 >= 0) {
                    const uint4* hv[2];
                    const float* cv[2];
                    vec(t0, hv[0], cv[0]);
                    vec(t1, hv[1], cv[1]);
                    float acc[2 * RP];
                    down_pass<RP, 2>(rows, RSu, nrw, K, hv, cv, lane, acc);
                    const float v = reduce_scatter<2 * RP>(acc, lane);
                    const int idx = rs_index<2 * RP>(lane), r = idx % RP;
                    if (lane % (16 / RP) == 16 / RP - 1 && r < nrw) put(v, r, idx >= RP ? t1 : t0);
                } else {
                    const uint4* hv[1];
                    const float* cv[1];
                    vec(t0, hv[0], cv[0]);
                    float acc[RP];
                    down_pass<RP, 1>(rows, RSu, nrw, K, hv, cv, lane, acc);
                    const float v = reduce_scatter<RP>(acc, lane);
                    const int r = rs_index<RP>(lane);
                    if (lane % (32 / RP) == 32 / RP - 1 && r < nrw) put(v, r, t0);
                }
            };
            uint32_t rest = tm;
            while (rest) {
                const int t0 = __ffs(rest) - 1;
                rest &= rest - 1u;
                int t1 = -1;
                if (rest) {
                    t1 = __ffs(rest) - 1;
                    rest &= rest - 1u;
                }
                // one instantiation (rows past nrw are skipped inside); a second,
                // 4-row one measured slower (register spills)
                rows_pass(std::integral_constant<int, 8>(), t0, t1);
            }
            item_done(it);
        }

        // ---- 5: arrivals on the row blocks; the last arriver of a block combines it ------
        FLINT_PHASE(8);
        if (!__syncthreads_or(failed || wfail || sm.fail) && sh_cta) {
            // the shared group learns the routing now (weights, number of experts)
            failed = !route(15);
            if (!failed && warp == 0) route_view_warp(ri, sm.ids, T, k, lane);
            FLINT_PHASE(18);
        }
        if (__syncthreads_or(failed || wfail || sm.fail)) {
            drain(budget);
            return;
        }
        const uint32_t U = (uint32_t)ri.D + (has_sh ? 1u : 0u);
        for (int j = sm.b0 + tid; j < sm.b1; j += kLT) {
            // the release half of the add publishes the CTA's d, ordered before
            // this thread by the barriers above
            const int blk = j % NB;
            if (atom_add_acq_rel_gpu(a.counters + blk, 1u) == U - 1u) sm.last[atomicAdd(&sm.n_last, 1)] = (int16_t)blk;
        }
        __syncthreads();
        FLINT_PHASE(9);
        // the blocks this CTA completed: one thread per 8 rows of one token, the
        // k + 1 expert outputs read as 16-byte words, summed in rank order
        const int n_last = sm.n_last;
        for (int e = tid; e < n_last * T * (kRowBlock / 8); e += kLT) {
            const int qb = e / (T * (kRowBlock / 8)), rem = e - qb * (T * (kRowBlock / 8));
            const int t = rem / (kRowBlock / 8), r = sm.last[qb] * kRowBlock + 8 * (rem - t * (kRowBlock / 8));
            float acc[8];
    #pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = 0.f;
            auto add = [&](float wj, const uint4 dj) {
                const uint32_t dw[4] = {dj.x, dj.y, dj.z, dj.w};
    #pragma unroll
                for (int i = 0; i < 4; ++i) {
                    acc[2 * i] = fmaf(wj, bf16_lo(dw[i]), acc[2 * i]);
                    acc[2 * i + 1] = fmaf(wj, bf16_hi(dw[i]), acc[2 * i + 1]);
                }
            };
            const uint4* dr = reinterpret_cast<const uint4*>(a.d_routed + (size_t)t * k * H + r);
            if constexpr (GIVEN) {  // ranks without an expert add nothing
                for (int j = 0; j < k; ++j)
                    if (ri.ids[t * k + j] >= 0) add(sm.w[t * k + j], __ldcg(dr + (size_t)j * (H / 8)));
            } else {
                for (int j = 0; j < k; j += 2) {  // two loads in flight
                    const uint4 d0 = __ldcg(dr + (size_t)j * (H / 8));
                    const uint4 d1 = j + 1 < k ? __ldcg(dr + (size_t)(j + 1) * (H / 8)) : make_uint4(0u, 0u, 0u, 0u);
                    add(sm.w[t * k + j], d0);
                    if (j + 1 < k) add(sm.w[t * k + j + 1], d1);
                }
            }
            if (has_sh) {
                const uint4 ds = __ldcg(reinterpret_cast<const uint4*>(a.d_shared + (size_t)t * H + r));
                const uint32_t dw[4] = {ds.x, ds.y, ds.z, ds.w};
    #pragma unroll
                for (int i = 0; i < 4; ++i) {
                    acc[2 * i] += bf16_lo(dw[i]);
                    acc[2 * i + 1] += bf16_hi(dw[i]);
                }
            }
            uint32_t o[4];
    #pragma unroll
            for (int i = 0; i < 4; ++i)
                o[i] = (uint32_t)f32_to_bf16_bits(acc[2 * i]) | ((uint32_t)f32_to_bf16_bits(acc[2 * i + 1]) << 16);
            *reinterpret_cast<uint4*>(a.y + (size_t)t * H + r) = make_uint4(o[0], o[1], o[2], o[3]);
        }
        for (int q = tid; q < n_last; q += kLT) a.counters[sm.last[q]] = 0;
        __syncthreads();
        FLINT_PHASE(10);

    }
#ifdef FLINT_PHASE_TRACE
    if (tid == 0) {
        sm.trace[20] = wait_gu;
        sm.trace[21] = t_math;
        sm.trace[22] = t_epi;
        sm.trace[23] = (unsigned long long)my_g | ((unsigned long long)my_d << 16) | (wait_dn << 32);
        unsigned long long lo = ~0ull, hi = 0;
        for (int w = 0; w < kLW; ++w) {
            lo = min(lo, sm.wend[w]);
            hi = max(hi, sm.wend[w]);
        }
        sm.trace[24] = lo;
        sm.trace[25] = hi;
    }
    if (tid == 0 && c < kTraceCtas) {
        unsigned long long* dst = g_phase_trace[sm.hdr[kHdrCalls] % kTraceCalls][c];
        for (int i = 0; i < 27; ++i) dst[i] = sm.trace[i];
        for (int i = 32; i < kTraceStamps; ++i) dst[i] = sm.trace[i];
        uint32_t smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        dst[27] = smid;
        dst[28] = (unsigned long long)sh_cta | ((unsigned long long)(sm.n_gi + sm.n_di) << 8) |
                  ((unsigned long long)sm.n_last << 16) | ((unsigned long long)sm.n_gi << 32);
        dst[29] = trace_t0;
        dst[30] = globaltimer_ns();
        dst[31] = sm.hdr[kHdrCalls] + 1ull;
    }
#endif
    // The last CTA to finish resets the exchange counters for the next call
    // (every other CTA is past all of its waits) and counts the call.
    if (tid == 0 && atomicAdd(a.hdr + kHdrDone, 1u) == (uint32_t)G - 1u) {
        a.hdr[kHdrScoresIn] = 0;
        a.hdr[kHdrPairsIn] = 0;
        for (int u = 0; u < ri.D; ++u) a.unit_counters[u] = 0;
        a.unit_counters[kShIdx] = 0;
        a.hdr[kHdrCalls] = sm.hdr[kHdrCalls] + 1u;
        a.hdr[kHdrDone] = 0;
    }
}

#include "layer_one.cuh"

}  // namespace

size_t layer_smem_bytes(const LayerArgs& a) { return a.one ? one_layout(a).total : layer_layout(a).total; }

namespace {
template <bool NORM, bool ROWS, bool GIVEN>
cudaError_t launch_layer_t(const LayerArgs& a, const DevInfo& d, bool pdl, cudaStream_t s) {
    static int configured_for = -1;
    cudaError_t e = configure_smem(layer_kernel<NORM, ROWS, GIVEN>, d, configured_for);
    if (e != cudaSuccess) return e;
    const size_t smem = layer_smem_bytes(a);
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, layer_kernel<NORM, ROWS, GIVEN>, kLT, smem);
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
    return cudaLaunchKernelEx(&cfg, layer_kernel<NORM, ROWS, GIVEN>, a);
}

template <bool GIVEN>
cudaError_t launch_one_t(const LayerArgs& a, const DevInfo& d, bool pdl, cudaStream_t s) {
    static int configured_for = -1;
    cudaError_t e = configure_smem(layer_one_kernel<GIVEN>, d, configured_for);
    if (e != cudaSuccess) return e;
    const size_t smem = layer_smem_bytes(a);
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, layer_one_kernel<GIVEN>, kOneThreads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)d.sm_count);
    cfg.blockDim = dim3(kOneThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, layer_one_kernel<GIVEN>, a);
}
}  // namespace

cudaError_t launch_layer(const LayerArgs& a, const DevInfo& d, bool pdl, cudaStream_t s) {
    if (a.one) return a.given ? launch_one_t<true>(a, d, pdl, s) : launch_one_t<false>(a, d, pdl, s);
    if (a.given) return a.rows ? launch_layer_t<false, true, true>(a, d, pdl, s) : launch_layer_t<false, false, true>(a, d, pdl, s);
    if (a.rows)
        return a.norm.r ? launch_layer_t<true, true, false>(a, d, pdl, s) : launch_layer_t<false, true, false>(a, d, pdl, s);
    return a.norm.r ? launch_layer_t<true, false, false>(a, d, pdl, s) : launch_layer_t<false, false, false>(a, d, pdl, s);
}

}  // namespace flint

#ifdef FLINT_PHASE_TRACE
// The trace build's reader: copies the ring of phase stamps ([calls][CTAs]
// [stamps] unsigned 64-bit) to host memory `out` of `n` entries; returns the
// entries copied, or -1 on a CUDA error.
extern "C" long long flint_phase_trace_read(unsigned long long* out, size_t n) {
    const size_t total = sizeof(flint::g_phase_trace) / sizeof(unsigned long long);
    if (n > total) n = total;
    if (cudaMemcpyFromSymbol(out, flint::g_phase_trace, n * sizeof(unsigned long long)) != cudaSuccess) return -1;
    return (long long)n;
}
#endif
