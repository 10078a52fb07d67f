// layer_one.cuh -- the decode step of one MoE layer for ONE token, as one
// cooperative kernel laid out for latency (included by layer.cu, whose
// exchange helpers, trace ring and status masks it uses).
//
// "Day-0 Support for Flint on vLLM", section "Optimizations": at batch 1 the
// MoE layer is a chain of short dependent steps (router GEMV, sigmoid top-k,
// gate/up GEMVs of the selected experts, down GEMVs, weighted combine with the
// shared expert), and the pages' low-latency path overlaps each step's weight
// loads with the step before it. At one token every step is small, so the
// time goes to the chain's latencies, not to bytes. This kernel keeps every
// CTA busy on the same fixed share of each step and issues each share's
// copies the moment their addresses are known. It runs 12 warps per CTA, so
// that two CTAs fit on an SM (registers): the next layer's CTAs become
// resident while this layer runs, issue their static copies and wait at the
// PDL wait, instead of starting after this layer's CTAs have left (with 24
// warps the next call's first CTA entered ~2 us after this call's last one
// ended; with 12 it enters ~13 us before, measured on the global timer).
//
//   * CTA c of G owns router rows [c E / G, (c + 1) E / G), shared-expert
//     gate/up pairs [c Is / G, (c + 1) Is / G), routed pairs
//     [c k I / G, (c + 1) k I / G) of the concatenation of the k selected
//     experts in rank order, and output rows [c H / G, (c + 1) H / G) of every
//     expert's down GEMV. No plan depends on the routing beyond "pair q is row
//     q % I of the expert of rank q / I".
//   * Before the PDL wait (static weights): the router rows, the routed
//     experts' tensor scales, the CTA's shared pairs and its shared down rows
//     are copied (1-D bulk copies, one mbarrier per pair, each used once),
//     and x is pulled into L2.
//   * After it: x is staged (chunk-scaled f16), the router warps compute
//     their rows' scores and publish each with a GPU-scope fence and a count;
//     the warps holding shared pairs
//     compute them meanwhile; the last warp waits for all E scores and selects
//     the top k. Then the warps issue the CTA's routed pairs' copies (and one
//     expert's down rows per rank), all at once: the CTA's whole share of the
//     weights is in flight with one round trip.
//   * Each pair's h goes to the workspace; the CTA publishes its count once;
//     every CTA waits for all pairs, stages all of h, computes its rows of the
//     k + 1 down GEMVs (their weights arrived long before) and sums them in
//     rank order into its rows of y. The last CTA to finish resets the counts.
//
// Given routing (GIVEN, behind flint_moe_decode): no router rows, scores or
// top-k; the caller's ids and weights are read after the PDL wait. An id
// outside [0, E) is reported in the status word and its rank adds nothing
// (its pairs and down rows are neither copied nor computed); an expert given
// at two ranks is simply computed for each.
//
// Every wait is bounded by the workspace's budget; on expiry the CTA records
// FLINT_ERR_TIMEOUT, lets its copies in flight land and returns, and the
// workspace must be re-initialised (flint_workspace_check does it).

constexpr int kOneMaxItems = 32;  // gate/up pairs of one CTA (shared + routed)
// pairs per copy of gate rows (and of up rows): two (14.37 against 14.51 us
// per layer with one: half the copies for the SM to take in; four measured
// slower in a 24-warp build, a pair's compute then waiting for its chunk)
constexpr int kOneChunk = 2;

struct OneSmall {
    uint64_t rbar;                        // router rows and tensor scales in
    uint64_t ibar[kOneMaxItems];          // gate/up chunk c in (its gate rows and up rows)
    uint64_t dbar[FLINT_MAX_TOPK + 1];    // down rows of unit u in (u = k: the shared expert)
    uint32_t hdr[8];                      // workspace header at the start of the call
    int32_t ids[FLINT_MAX_TOPK];
    float w[FLINT_MAX_TOPK];
    float ts_sh[3];
    float res[kOneMaxItems][2];           // raw gate / up sums of pair i
    uint32_t issued_chunks, issued_down;  // copies issued (for the drain on failure)
    int fail, ok;
#ifdef FLINT_PHASE_TRACE
    unsigned long long trace[kTraceStamps];
#endif
};

struct OneSmem {
    size_t tsall, xs, csc, hs, hsc, rows, items, down, dres, total;
};

__host__ __device__ inline OneSmem one_layout(const LayerArgs& a) {
    OneSmem L;
    const size_t H = a.H, nh = (size_t)a.k * a.I + a.Is;
    L.tsall = align_up(sizeof(OneSmall), 128);
    L.xs = align_up(L.tsall + 12 * (size_t)a.E, 128);
    L.csc = align_up(L.xs + 2 * H, 128);
    L.hs = align_up(L.csc + 4 * (H / 32), 128);
    L.hsc = align_up(L.hs + 2 * nh, 128);
    L.rows = align_up(L.hsc + 4 * (nh / 32), 128);
    L.items = align_up(L.rows + 2 * (size_t)a.rpc * H, 128);
    L.down = align_up(L.items + (size_t)a.one_items * a.slot, 128);
    L.dres = align_up(L.down + (size_t)(a.k + 1) * a.rows_max * a.one_rsd, 128);
    L.total = align_up(L.dres + 4 * (size_t)(a.k + 1) * a.rows_max, 128);
    return L;
}

// All lanes of the warp wait until *p >= target (each lane's own acquire),
// for at most budget_ns; false in every lane if any gave up (`code` recorded).
__device__ __forceinline__ bool warp_wait_count(const uint32_t* p, uint32_t target, uint32_t* status, uint32_t code,
                                                uint64_t budget_ns) {
    bool ok = true;
    if (ld_acquire_gpu(p) < target) {
        const uint64_t t0 = globaltimer_ns();
        while (ld_acquire_gpu(p) < target) {
            if (globaltimer_ns() - t0 > budget_ns) {
                atomicOr(status, code);
                ok = false;
                break;
            }
        }
    }
    return __all_sync(0xffffffffu, ok);
}

// One token's x (H bf16 values, H % 256 == 0) staged as chunk-scaled f16 in
// the GATE order of stage_f16, four threads per 32-value chunk: thread q takes
// the 16-byte word q % 4 of chunk q / 4, the chunk's largest magnitude comes
// from two shuffles, and each value is converted on its own (the same bits as
// one thread per chunk, with a quarter of the dependent steps).
__device__ __forceinline__ void stage_x_quarters(const uint16_t* x, int H, uint4* xh, float* csc) {
    for (int q = threadIdx.x; q < H / 8; q += blockDim.x) {  // H / 8 is a multiple of 32: whole warps
        const uint4 w = ld_cg(reinterpret_cast<const uint4*>(x) + q);
        uint32_t m2 = __vmaxu2(__vmaxu2(w.x & 0x7FFF7FFFu, w.y & 0x7FFF7FFFu),
                               __vmaxu2(w.z & 0x7FFF7FFFu, w.w & 0x7FFF7FFFu));
        m2 = __vmaxu2(m2, __shfl_xor_sync(0xffffffffu, m2, 1));
        m2 = __vmaxu2(m2, __shfl_xor_sync(0xffffffffu, m2, 2));
        // bf16 exponent field of the largest magnitude -> s with max * 2^-s in [2^14, 2^15)
        const uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
        const int sh = min(126, max(-126, (int)(m >> 7) - 141));
        const float down = __int_as_float((127 - sh) << 23);
        const int c = q >> 2, i = q & 3;
        if (i == 0) csc[c] = __int_as_float((127 + sh) << 23);
        xh[(c / 32) * 128 + i * 32 + c % 32] =
            make_uint4(f32x2_to_f16x2(bf16_lo(w.x) * down, bf16_hi(w.x) * down),
                       f32x2_to_f16x2(bf16_lo(w.y) * down, bf16_hi(w.y) * down),
                       f32x2_to_f16x2(bf16_lo(w.z) * down, bf16_hi(w.z) * down),
                       f32x2_to_f16x2(bf16_lo(w.w) * down, bf16_hi(w.w) * down));
    }
}

// All of h (the routed ranks' [k][I], then the shared expert's [Is]; bf16,
// written by other CTAs: read through L2) staged in the DOWN order of
// stage_f16, four threads per 32-value chunk as above (the same bits).
__device__ __forceinline__ void stage_h_quarters(const uint16_t* hr, const uint16_t* hs, int k, int I, int Is,
                                                 uint4* hh, float* hsc) {
    const int nr = k * I / 8, n = nr + Is / 8;  // 16-byte words; a multiple of 32 (I, Is % 256 == 0)
    for (int q = threadIdx.x; q < n; q += blockDim.x) {
        const bool sh = q >= nr;
        const int K = sh ? Is : I, wq = sh ? q - nr : q % (I / 8), v = sh ? 0 : q / (I / 8);
        const uint4 w = ld_cg(reinterpret_cast<const uint4*>(sh ? hs : hr) + (sh ? wq : q));
        uint32_t m2 = __vmaxu2(__vmaxu2(w.x & 0x7FFF7FFFu, w.y & 0x7FFF7FFFu),
                               __vmaxu2(w.z & 0x7FFF7FFFu, w.w & 0x7FFF7FFFu));
        m2 = __vmaxu2(m2, __shfl_xor_sync(0xffffffffu, m2, 1));
        m2 = __vmaxu2(m2, __shfl_xor_sync(0xffffffffu, m2, 2));
        const uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
        const int s = min(126, max(-126, (int)(m >> 7) - 141));
        const float down = __int_as_float((127 - s) << 23);
        const int c = wq >> 2, i = wq & 3;
        uint4* d = hh + (sh ? (size_t)k * (I / 8) : (size_t)v * (I / 8));
        float* cs = hsc + (sh ? (size_t)k * (I / 32) : (size_t)v * (I / 32));
        if (i == 0) cs[c] = __int_as_float((127 + s) << 23);
        d[(i & 1) * (K / 16) + 2 * c + (i >> 1)] =
            make_uint4(f32x2_to_f16x2(bf16_lo(w.x) * down, bf16_hi(w.x) * down),
                       f32x2_to_f16x2(bf16_lo(w.y) * down, bf16_hi(w.y) * down),
                       f32x2_to_f16x2(bf16_lo(w.z) * down, bf16_hi(w.z) * down),
                       f32x2_to_f16x2(bf16_lo(w.w) * down, bf16_hi(w.w) * down));
    }
}

#ifdef FLINT_PHASE_TRACE
#define ONE_STAMP(i)                                   \
    do {                                               \
        if (lane == 0) sm.trace[(i)] = clock64();      \
    } while (0)
#else
#define ONE_STAMP(i) \
    do {             \
    } while (0)
#endif

template <bool GIVEN>
__global__ void __launch_bounds__(kOneThreads, (kOneWarps <= 12 ? 2 : 1)) layer_one_kernel(const LayerArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const OneSmem L = one_layout(a);
    OneSmall& sm = *reinterpret_cast<OneSmall*>(smem);
    const int H = a.H, E = a.E, k = a.k, I = a.I, Is = a.Is;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = blockIdx.x, G = gridDim.x;
    const bool has_sh = a.s_gu != nullptr;
    const int RS = (int)nvfp4_row_stride(H), RSr = (int)nvfp4_row_stride(I);
    const int RSs = has_sh ? (int)nvfp4_row_stride(Is) : 0;
    uint4* xh = reinterpret_cast<uint4*>(smem + L.xs);
    float* csc = reinterpret_cast<float*>(smem + L.csc);
    uint4* hh = reinterpret_cast<uint4*>(smem + L.hs);
    float* hsc = reinterpret_cast<float*>(smem + L.hsc);
    float* dres = reinterpret_cast<float*>(smem + L.dres);
    const float* tsall = reinterpret_cast<const float*>(smem + L.tsall);
    // this CTA's shares
    const int r0 = (int)((long long)c * E / G), nrr = GIVEN ? 0 : (int)((long long)(c + 1) * E / G) - r0;
    const int s0 = has_sh ? (int)((long long)c * Is / G) : 0;
    const int ns = has_sh ? (int)((long long)(c + 1) * Is / G) - s0 : 0;
    const long long kI = (long long)k * I;
    const int q0 = (int)(c * kI / G), nq = (int)((c + 1) * kI / G) - q0;
    const int n_items = ns + nq;
    // The pairs fall in at most three runs of consecutive rows of one matrix:
    // the shared pairs, then rank j0's routed pairs (n1), then rank j0 + 1's
    // (n2; nq <= I). Each run is copied in chunks of kOneChunk pairs (one
    // mbarrier each): cs0, cs1 and cs2 chunks.
    const int j0 = nq ? q0 / I : 0;
    const int n1 = nq ? min(nq, (j0 + 1) * I - q0) : 0, n2 = nq - n1;
    constexpr int CH = kOneChunk;
    const int cs0 = (ns + CH - 1) / CH, cs1 = (n1 + CH - 1) / CH, cs2 = (n2 + CH - 1) / CH;
    const int R0 = c * H / G, nrows = (c + 1) * H / G - R0;
    const int n_units = k + (has_sh ? 1 : 0);
    constexpr int W = kOneWarps;
    constexpr int TOPW = W - 1;  // waits for the scores and selects
    const bool ts_bulk = (reinterpret_cast<uintptr_t>(a.ts) % 16 == 0) && ((12 * E) % 16 == 0);
    const uint32_t rbar_bytes = (uint32_t)(nrr * H * 2) + (ts_bulk ? 12u * (uint32_t)E : 0u);
    const uint32_t full = 0xffffffffu;
    // pair i's gate row and up row (the CTA's gate rows, then its up rows, each
    // in pair order, so that a chunk of consecutive pairs is two contiguous runs)
    auto gate_dst = [&](int i) { return smem + L.items + (size_t)i * RS; };
    auto up_dst = [&](int i) { return smem + L.items + ((size_t)a.one_items + i) * RS; };
    auto down_dst = [&](int u) { return smem + L.down + (size_t)u * a.rows_max * a.one_rsd; };
    // tensor scale j of routed rank r's expert, or of the shared expert
    auto tscale = [&](int r, int j) -> float {
        if (r == k) return sm.ts_sh[j];
        const int e = sm.ids[r];
        return ts_bulk ? tsall[3 * e + j] : __ldg(a.ts + 3 * e + j);
    };

    // pair i of the CTA (shared pairs first): its rank (k: shared) and row
    auto pair_of = [&](int i, int& r, int& p) {
        if (i < ns) {
            r = k;
            p = s0 + i;
        } else {
            const int q = q0 + i - ns;
            r = q / I;
            p = q - r * I;
        }
    };
    auto chunk_of = [&](int i) {
        if (i < ns) return i / CH;
        i -= ns;
        if (i < n1) return cs0 + i / CH;
        return cs0 + cs1 + (i - n1) / CH;
    };
    // rank r (k: the shared expert) has an expert to compute
    auto live = [&](int r) { return !GIVEN || r == k || sm.ids[r] >= 0; };
    auto chunk_rank = [&](int ch) { return ch < cs0 ? k : (ch < cs0 + cs1 ? j0 : j0 + 1); };
    // chunk ch: its first pair, pair count, rank (k: shared) and first row
    auto chunk_span = [&](int ch, int& i0, int& n, int& r, int& p0) {
        if (ch < cs0) {
            i0 = ch * CH;
            n = min(CH, ns - i0);
            r = k;
            p0 = s0 + i0;
        } else if (ch < cs0 + cs1) {
            const int o = (ch - cs0) * CH;
            i0 = ns + o;
            n = min(CH, n1 - o);
            r = j0;
            p0 = q0 - j0 * I + o;
        } else {
            const int o = (ch - cs0 - cs1) * CH;
            i0 = ns + n1 + o;
            n = min(CH, n2 - o);
            r = j0 + 1;
            p0 = o;
        }
    };
    // one of chunk ch's two copies: its gate rows (half 0) or its up rows
    auto copy_half = [&](int ch, int half) {
        int i0, n, r, p0;
        chunk_span(ch, i0, n, r, p0);
        const uint8_t* g = r == k ? a.s_gu : a.gu + (size_t)sm.ids[r] * 2 * I * RS;
        const int row = half ? (r == k ? Is : I) + p0 : p0;
        bulk_g2s(half ? up_dst(i0) : gate_dst(i0), g + (size_t)row * RS, (uint32_t)(n * RS), &sm.ibar[ch]);
    };
    auto chunk_bytes = [&](int ch) {
        int i0, n, r, p0;
        chunk_span(ch, i0, n, r, p0);
        return 2u * (uint32_t)(n * RS);
    };
    // the CTA's rows of unit u's down matrix (u = k: the shared expert)
    auto issue_down = [&](int u) {
        if (!live(u)) return;
        const bool sh = u == k;
        const int RSu = sh ? RSs : RSr;
        const uint8_t* d = sh ? a.s_down : a.down + (size_t)sm.ids[u] * H * RSr;
        mbar_arrive_expect_tx(&sm.dbar[u], (uint32_t)(nrows * RSu));
        bulk_g2s(down_dst(u), d + (size_t)R0 * RSu, (uint32_t)(nrows * RSu), &sm.dbar[u]);
        atomicOr(&sm.issued_down, 1u << u);
    };
    // chunk ch's two copies (one thread)
    auto issue_chunk = [&](int ch) {
        if (!live(chunk_rank(ch))) return;
        mbar_arrive_expect_tx(&sm.ibar[ch], chunk_bytes(ch));
        copy_half(ch, 0);
        copy_half(ch, 1);
        atomicOr(&sm.issued_chunks, 1u << ch);
    };
    // Before an early exit (every thread, after a CTA barrier): the copies in
    // flight land first (bounded).
    auto drain = [&](uint64_t budget_ns) {
        if (tid == 0) {
            if (rbar_bytes) mbar_wait_bounded(&sm.rbar, 0, nullptr, 0, budget_ns);
            for (uint32_t m = sm.issued_chunks; m; m &= m - 1u) mbar_wait_bounded(&sm.ibar[__ffs(m) - 1], 0, nullptr, 0, budget_ns);
            for (uint32_t m = sm.issued_down; m; m &= m - 1u) mbar_wait_bounded(&sm.dbar[__ffs(m) - 1], 0, nullptr, 0, budget_ns);
        }
        __syncthreads();
    };

    // ---- before the PDL wait: barriers, static weight copies ---------------------------
#ifdef FLINT_PHASE_TRACE
    if (tid < kTraceStamps) sm.trace[tid] = 0;
    const uint64_t trace_t0 = globaltimer_ns();
#endif
    FLINT_PHASE(0);
    if (tid < kOneMaxItems) mbar_init(&sm.ibar[tid], 1);
    if (tid >= 32 && tid < 33 + FLINT_MAX_TOPK) mbar_init(&sm.dbar[tid - 32], 1);
    if (tid == 64) {
        mbar_init(&sm.rbar, 1);
        sm.issued_chunks = sm.issued_down = 0u;
        sm.fail = 0;
    }
    if (tid == 65 && has_sh) {
        sm.ts_sh[0] = __ldg(a.s_ts);
        sm.ts_sh[1] = __ldg(a.s_ts + 1);
        sm.ts_sh[2] = __ldg(a.s_ts + 2);
    }
    if (tid < 65) fence_mbar_init();
    __syncthreads();
    if (tid == 0 && rbar_bytes) {
        mbar_arrive_expect_tx(&sm.rbar, rbar_bytes);
        if (nrr > 0) bulk_g2s(smem + L.rows, a.wr + (size_t)r0 * H, (uint32_t)(nrr * H * 2), &sm.rbar);
        if (ts_bulk) bulk_g2s(smem + L.tsall, a.ts, 12u * (uint32_t)E, &sm.rbar);
    }
    if (lane == 0)
        for (int ch = warp; ch < cs0; ch += W) issue_chunk(ch);
    if (has_sh && warp == TOPW && lane == 0 && nrows > 0) issue_down(k);
    // x and the header into L2: the previous kernel may still be writing them
    // (L2 is where its writes land), so only the address translation and a
    // first copy are warmed, no data is read
    const bool x_early = GIVEN && a.x_early;
    if (warp == TOPW - 1 && !x_early) {
        const size_t xb = (size_t)H * 2;
        for (size_t o = (size_t)lane * 128; o < xb; o += 32 * 128)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char*>(a.x) + o));
        if (lane == 0) asm volatile("prefetch.global.L2 [%0];" ::"l"(a.hdr));
    }
    // given routing right after the router on the same x: the router lets its
    // dependents launch only once its own wait has returned, so x is complete
    if (x_early) stage_x_quarters(a.x, H, xh, csc);
    pdl_launch_dependents();
    pdl_wait();  // x comes from the previous kernel
    FLINT_PHASE(1);

    // ---- x, the header ------------------------------------------------------------------
    if (tid == 0) {
        const uint4 h0 = ld_cg(reinterpret_cast<const uint4*>(a.hdr));
        const uint4 h1 = ld_cg(reinterpret_cast<const uint4*>(a.hdr) + 1);
        sm.hdr[0] = h0.x; sm.hdr[1] = h0.y; sm.hdr[2] = h0.z; sm.hdr[3] = h0.w;
        sm.hdr[4] = h1.x; sm.hdr[5] = h1.y; sm.hdr[6] = h1.z; sm.hdr[7] = h1.w;
    }
    if (!x_early) stage_x_quarters(a.x, H, xh, csc);
    __syncthreads();
    FLINT_PHASE(2);
    const uint64_t budget = sm.hdr[kHdrBudget] ? (uint64_t)sm.hdr[kHdrBudget] * 1000ull : kWaitBudgetNs;
    if (sm.hdr[kHdrStatus] & kStatusPoisonMask) {  // an earlier call failed: re-initialise first
        drain(budget);
        return;
    }
    const bool withhold = sm.hdr[kHdrLoseCta] == (uint32_t)c + 1u;  // test hook: publish nothing
    bool wfail = false;  // this warp gave up on a wait

    // ---- router rows: one warp per row, published one by one -----------------------------
    for (int r = warp; warp < TOPW && r < nrr; r += TOPW) {
        if (!mbar_wait_bounded(&sm.rbar, 0, a.status, kStatusTimeoutLayer, budget)) {
            wfail = true;
            break;
        }
        // lane l takes the 32-value chunks l, l + 32, ...; lanes 2i, 2i + 1 start
        // at word i % 4 of their 64-byte chunk (no bank conflicts); each
        // chunk's FP32 sum is multiplied back by its power-of-two scale
        const uint4* wv = reinterpret_cast<const uint4*>(smem + L.rows + (size_t)r * H * 2);
        float v = 0.f;
        for (int m = 0; m < H / 1024; ++m) {
            const int ch = lane + 32 * m;
            float p0 = 0.f, p1 = 0.f;
#pragma unroll
            for (int w0 = 0; w0 < 4; ++w0) {
                const int w = (w0 + (lane >> 1)) & 3;
                const uint4 xv = xh[(m * 4 + w) * 32 + lane], wq = wv[4 * ch + w];
                const uint32_t xa[4] = {xv.x, xv.y, xv.z, xv.w}, wa[4] = {wq.x, wq.y, wq.z, wq.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 xf = __half22float2(*reinterpret_cast<const __half2*>(&xa[i]));
                    p0 = fmaf(bf16_lo(wa[i]), xf.x, p0);
                    p1 = fmaf(bf16_hi(wa[i]), xf.y, p1);
                }
            }
            v = fmaf(csc[ch], p0 + p1, v);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(full, v, off);
        if (lane == 0) {
            a.scores[r0 + r] = sigmoid_score(v, a.bias, r0 + r);
            if (!withhold) release_add_gpu(a.hdr + kHdrScoresIn, 1u);
#ifdef FLINT_PHASE_TRACE
            if (r == 0) {
                sm.trace[3] = clock64();
                sm.trace[26] = globaltimer_ns();
            }
#endif
        }
    }
    // The next layer's static weights into L2 while the routing runs (CTA c
    // takes granules [c n / G, (c + 1) n / G) of the ranges' concatenation).
    if (tid == (TOPW - 1) * 32 && a.pf_granules) {
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

    // ---- one pair: gate/up sums, then h = bf16(silu(bf16(ts_g g)) bf16(ts_u u)) ----------
    auto compute_item = [&](int i) -> bool {
        if (!live(chunk_rank(chunk_of(i)))) return true;  // an invalid given id: nothing to compute
        if (!__all_sync(full, mbar_wait_bounded(&sm.ibar[chunk_of(i)], 0, a.status, kStatusTimeoutLayer, budget)))
            return false;
        const int tk[1] = {0};
        gate_up_pass<true, 1>(gate_dst(i), up_dst(i), H, xh, csc, tk, lane, &sm.res[i][0], &sm.res[i][1]);
        __syncwarp();
        if (lane == 0) {
            int r, p;
            pair_of(i, r, p);
            const float gv = bf16_round_f32(tscale(r, 0) * sm.res[i][0]);
            const float uv = bf16_round_f32(tscale(r, 1) * sm.res[i][1]);
            const uint16_t hv = f32_to_bf16_bits(silu_f32(gv) * uv);
            if (r == k) a.h_shared[p] = hv;
            else a.h_routed[(size_t)r * I + p] = hv;
        }
        return true;
    };
    // the shared pairs (static: their bytes were requested before the wait)
    for (int i = warp; i < ns && !wfail; i += W)
        if (!compute_item(i)) wfail = true;

    // ---- routing: the last warp waits for all E scores and selects the top k -------------
    if (GIVEN && warp == TOPW && !wfail) {
        // the caller's ids and weights (written by an earlier kernel: read
        // through L2); an id outside [0, E) is reported and becomes -1
        ONE_STAMP(4);
        if (lane < k) {
            int e = ld_cg(a.ids + lane);
            if (e < 0 || e >= E) {
                atomicOr(a.status, kStatusBadExpertId);
                e = -1;
            }
            sm.ids[lane] = e;
            sm.w[lane] = ld_cg(a.weights + lane);
        }
        ONE_STAMP(5);
        if (ts_bulk && !__all_sync(full, mbar_wait_bounded(&sm.rbar, 0, a.status, kStatusTimeoutLayer, budget)))
            wfail = true;
        ONE_STAMP(6);
    }
    if (!GIVEN && warp == TOPW && !wfail) {
        ONE_STAMP(4);
        if (!warp_wait_count(a.hdr + kHdrScoresIn, (uint32_t)E, a.status, kStatusTimeoutLayer, budget)) {
            wfail = true;
        } else {
            ONE_STAMP(5);
            if (E <= 256)
                topk_warp<8, true>(a.scores, E, k, lane, sm.ids, sm.w);
            else
                topk_warp<FLINT_MAX_EXPERTS / 32, true>(a.scores, E, k, lane, sm.ids, sm.w);
            // (lane j wrote rank j's id and weight)
            if (c == G - 1 && lane < k) {
                a.ids[lane] = sm.ids[lane];
                a.weights[lane] = sm.w[lane];
            }
            // the CTAs without router rows still need the tensor scales
            if (ts_bulk && nrr == 0 && !__all_sync(full, mbar_wait_bounded(&sm.rbar, 0, a.status, kStatusTimeoutLayer, budget)))
                wfail = true;
            ONE_STAMP(6);
        }
    }
    if (__syncthreads_or(wfail)) {
        drain(budget);
        return;
    }
    FLINT_PHASE(7);
    // every routed copy of the CTA at once, spread over the warps (a bulk copy
    // instruction holds its thread for up to hundreds of cycles while the SM
    // takes about one copy per hundred cycles, measured): routed chunk m on
    // warp m % W, then one expert's down rows per rank on the following warps
    if (lane == 0) {
        const int nrc = cs1 + cs2;
        for (int m = warp; m < nrc; m += W) issue_chunk(cs0 + m);
        for (int u = 0; u < k; ++u)
            if ((u + nrc) % W == warp && nrows > 0) issue_down(u);
    }
    FLINT_PHASE(8);
    for (int i = warp; i < n_items && !wfail; i += W) {
        if (i < ns) continue;
        if (!compute_item(i)) wfail = true;
        if (i == ns) ONE_STAMP(9);
    }

    // ---- the h exchange: this CTA's count, then every pair's ----------------------------------
    if (__syncthreads_or(wfail)) {
        drain(budget);
        return;
    }
    FLINT_PHASE(10);
    if (tid == 0 && !withhold && n_items > 0) release_add_gpu(a.hdr + kHdrPairsIn, (uint32_t)n_items);
    const uint32_t pairs = (uint32_t)kI + (has_sh ? (uint32_t)Is : 0u);
    if (!cta_wait_count(a.hdr + kHdrPairsIn, pairs, a.status, kStatusTimeoutLayer, budget, &sm.ok)) {
        drain(budget);
        return;
    }
    FLINT_PHASE(11);
    // all of h: the routed ranks' [k][I], then the shared expert's [Is]
    stage_h_quarters(a.h_routed, a.h_shared, k, I, has_sh ? Is : 0, hh, hsc);
    __syncthreads();
    FLINT_PHASE(12);

    // ---- down: the CTA's rows of every unit (unit u's rows are u nrows .. u nrows +
    // nrows - 1 of one list) cut evenly over the warps, in passes of up to 8 rows of
    // one unit (a warp's cut spans at most two units at the Flint shape) -----------
    {
        const int total = n_units * nrows;
        const int w1 = (warp + 1) * total / W;
        for (int q = warp * total / W; q < w1 && !wfail;) {
            const int u = q / nrows, rl = q - u * nrows, nr = min(min(8, nrows - rl), w1 - q);
            q += nr;
            if (!live(u)) continue;
            if (!__all_sync(full, mbar_wait_bounded(&sm.dbar[u], 0, a.status, kStatusTimeoutLayer, budget))) {
                wfail = true;
                break;
            }
            const bool sh = u == k;
            const int K = sh ? Is : I, RSu = sh ? RSs : RSr;
            const uint4* hv[1] = {hh + (size_t)u * (I / 8)};
            const float* cv[1] = {hsc + (size_t)u * (I / 32)};
            float acc[8];
            down_pass<8, 1>(down_dst(u) + (size_t)rl * RSu, RSu, nr, K, hv, cv, lane, acc);
            const float v = reduce_scatter<8>(acc, lane);
            const int r = rs_index<8>(lane);
            if (lane % 4 == 3 && r < nr) dres[u * a.rows_max + rl + r] = bf16_round_f32(tscale(u, 2) * v);
        }
    }
    if (__syncthreads_or(wfail)) {
        drain(budget);
        return;
    }
    FLINT_PHASE(13);
    // y = bf16(sum_j w_j d_j + d_shared), ranks in order
    for (int r = tid; r < nrows; r += kOneThreads) {
        float acc = 0.f;
        for (int j = 0; j < k; ++j)
            if (live(j)) acc = fmaf(sm.w[j], dres[j * a.rows_max + r], acc);
        if (has_sh) acc += dres[k * a.rows_max + r];
        a.y[R0 + r] = f32_to_bf16_bits(acc);
    }
    FLINT_PHASE(14);
#ifdef FLINT_PHASE_TRACE
    if (tid == 0 && c < kTraceCtas) {
        unsigned long long* dst = g_phase_trace[sm.hdr[kHdrCalls] % kTraceCalls][c];
        for (int i = 0; i < 27; ++i) dst[i] = sm.trace[i];
        for (int i = 32; i < kTraceStamps; ++i) dst[i] = sm.trace[i];
        uint32_t smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        dst[27] = smid;
        dst[28] = 2ull | ((unsigned long long)n_items << 8) | ((unsigned long long)ns << 16) |
                  ((unsigned long long)nrr << 32);
        dst[29] = trace_t0;
        dst[30] = globaltimer_ns();
        dst[31] = sm.hdr[kHdrCalls] + 1ull;
    }
#endif
    // The last CTA to finish resets the exchange counts for the next call
    // (every other CTA is past all of its waits) and counts the call.
    if (tid == 0 && atomicAdd(a.hdr + kHdrDone, 1u) == (uint32_t)G - 1u) {
        a.hdr[kHdrScoresIn] = 0;
        a.hdr[kHdrPairsIn] = 0;
        a.hdr[kHdrCalls] = sm.hdr[kHdrCalls] + 1u;
        a.hdr[kHdrDone] = 0;
    }
}
#undef ONE_STAMP
