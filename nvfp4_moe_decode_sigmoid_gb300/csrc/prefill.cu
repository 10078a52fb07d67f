// prefill.cu -- the MoE layer over a long batch of tokens (prefill) on the
// 5th-generation tensor cores.
//
// "Day-0 Support for Flint on vLLM", section "Optimizations": the small-batch
// MoE rewrite (router and expert GEMVs that read only the selected experts'
// weights) was also the largest gain of the 8K-token prefill; section "Model
// architecture": weight-only NVFP4 experts with bf16 activations, sigmoid
// top-6 over 256 experts plus a shared expert. The arithmetic is the decode
// path's (the same rounding points), on many tokens at once:
//   1. router logits = x Wr^T (FP32), a tensor-core GEMM;
//   2. per token: sigmoid, top-k, renormalised weights (one warp per token);
//   3. the (token, rank) pairs sorted by expert, token order kept within an
//      expert (counting sort, deterministic);
//   4. per expert: h = bf16(silu(bf16(ts_g x Wg^T)) bf16(ts_u x Wu^T)) over its
//      gathered token rows, a grouped GEMM whose NVFP4 B tiles are dequantised
//      to bf16 in shared memory (exact: a code times its block scale has at
//      most 6 significant bits); the shared expert over all tokens;
//   5. per expert: d = bf16(ts_d h Wd^T), grouped the same way;
//   6. y = bf16(sum_j w_j d_j + d_shared) per token, ranks in order (a gather,
//      no atomics: deterministic).
//
// GEMM tiles are 128 rows x 128 columns, K in steps of 64, accumulated in
// TMEM by tcgen05.mma (kind::f16, bf16 operands, FP32 accumulator) issued by
// one thread. The operands stream through a ring of shared-memory stages
// filled by TMA (one thread issues cp.async.bulk.tensor 2-D tile copies
// completing on the stage's full mbarrier; 2 stages for the expert GEMMs,
// which take two M-tiles per CTA, 3 for the router's): the A tiles with
// 128-byte swizzle, already in the MMA operand layout, and raw NVFP4 B
// windows (code and scale bytes), which eight dequantising warps expand into
// one of two swizzled bf16 B tiles. Empty mbarriers, committed by the MMA thread, hand
// each stage and B tile back. The expert GEMMs' A rows are the expert-sorted
// copy of the tokens, so every A tile is a plain 2-D tile.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "router_common.cuh"
#include "tcgen05.cuh"

namespace flint {
namespace {

constexpr int kTileM = 128, kStepK = 64;
constexpr int kNTile = 128;  // tile N of the NVFP4 expert GEMMs (256 measured slower: 940 vs 905 us, one CTA per SM)
constexpr int kMT = 2;       // M-tiles per CTA of the expert GEMMs (one dequantised B tile serves both)
constexpr uint32_t kTileBytes = kTileM * kStepK * 2;  // 16 KB

// 8 codes (one 32-bit word: byte b holds columns 2b, 2b + 1) times their
// block scale (f16x2, both halves equal) -> 8 bf16 (exact).
__device__ __forceinline__ uint4 dequant8(uint32_t w, uint32_t s2) {
    uint32_t h[4];
    decode_word_h2(w, h);
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __half2 p = __hmul2(*reinterpret_cast<const __half2*>(&h[i]), *reinterpret_cast<const __half2*>(&s2));
        const float2 f = __half22float2(p);
        const __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
        o[i] = *reinterpret_cast<const uint32_t*>(&b);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.f + expf(-g)); }

// The group (expert) of M-tile `mt` and its first row: tile_start is the
// exclusive prefix of the groups' tile counts (n_groups + 1 entries).
__device__ __forceinline__ int find_group(const int* tile_start, int n_groups, int mt) {
    int lo = 0, hi = n_groups - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tile_start[mid] <= mt) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

enum { kEpiLogits = 0, kEpiSwiglu = 1, kEpiScale = 2 };

// One 128 x 128 output tile of a grouped GEMM (blockIdx.x: N-tile, blockIdx.y:
// M-tile over all groups; the N-tiles of one M-tile run together, so its A
// tile is read from HBM once and from L2 by the others), fed by TMA:
//   warp 8 (one thread) issues each K step's tile loads into a stage of the
//     load ring: the A tile (128 rows x 64 bf16, 128-byte swizzle, exactly the
//     operand layout of the MMA) and either the raw NVFP4 B rows (codes and the
//     16-byte window of scales, two 64-row boxes each) or, for a bf16 B, the B
//     tile itself; completion is counted in bytes on the stage's `full`
//     barrier;
//   warps 0-7 (NVFP4 only) dequantise each step's raw B rows into a B tile of
//     the B ring (each thread half a row: four 8-value chunks, written in the
//     128-byte swizzled layout) and arrive on its barrier;
//   warp 9 (one thread) issues the step's four MMAs (K = 16 each) into the
//     TMEM accumulator and commits them to the `empty` barriers of the load
//     stage and of the B tile, which releases both for reuse;
//   warps 0-7 then run the epilogue from TMEM.
// Every wait is bounded; a timeout is recorded in the status word and the
// tile is skipped.
constexpr int kPT = 320;                // 8 dequantise/epilogue warps, the load warp, the MMA warp
constexpr int kPW = 256;                // dequantise/epilogue threads
constexpr int kPB = 2;                  // B tiles (NVFP4)

// Tile N = TN (128: two CTAs per SM, 3 load stages; 256: one CTA per SM, 4
// load stages, half the A bytes per FLOP); MT M-tiles of 128 rows per CTA (2:
// one dequantised B tile serves both; 2 load stages, so that two CTAs still
// fit an SM: 776 us for the 8192-token layer against 922 with one M-tile,
// and 985 with 3 stages and one CTA per SM).
template <bool NVFP4, int TN, int MT = 1>
struct TmaSmem {
    static constexpr int PL = TN == 256 ? 4 : (MT == 2 ? 2 : 3);         // load stages
    static constexpr size_t raw = (size_t)TN * 48;                        // codes + scale windows of one step
    static constexpr size_t bt = (size_t)TN * kStepK * 2;                 // one B tile
    static constexpr size_t stage = MT * kTileBytes + (NVFP4 ? raw : bt);
    static constexpr size_t load = 0;                                     // PL x (A tile, B raw or B tile)
    static constexpr size_t btile = load + PL * stage;                    // kPB B tiles (NVFP4)
    static constexpr size_t bar = btile + (NVFP4 ? kPB * bt : 0);
    static constexpr int nbar = 2 * PL + 2 * kPB + 1;
    static constexpr size_t tslot = bar + 8 * nbar;
    static constexpr size_t total = tslot + 16 + 1024;                    // + alignment slack
};

template <bool NVFP4, int EPI, int TN, int MT = 1>
__global__ void __launch_bounds__(kPT, TN == 128 ? 2 : 1) prefill_gemm_kernel(
    const __grid_constant__ CUtensorMap tma_a, const __grid_constant__ CUtensorMap tma_b,
    const __grid_constant__ CUtensorMap tma_s, const PrefillGemmArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    using L = TmaSmem<NVFP4, TN, MT>;
    constexpr int kPL = L::PL;
    constexpr int NB = TN / 64;  // 64-row boxes of B per step
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // ---- which tiles: MT consecutive M-tiles of one group (fewer at its end) ----
    int g = 0, row0, nrows;
    const int mt = blockIdx.y;
    if (a.tile_start) {
        const int* starts = MT == 2 ? a.pair_start : a.tile_start;
        if (mt >= ld_cg(starts + a.n_groups)) return;
        g = find_group(starts, a.n_groups, mt);
        const int base = ld_cg(a.seg_base + g);
        row0 = base + (mt - ld_cg(starts + g)) * (MT * kTileM);
        nrows = min(MT * kTileM, base + ld_cg(a.seg_len + g) - row0);
    } else {
        row0 = mt * (MT * kTileM);
        if (row0 >= a.rows) return;
        nrows = min(MT * kTileM, a.rows - row0);
    }
    const int ntile = (nrows + kTileM - 1) / kTileM;  // 1 or MT
    const int nt = blockIdx.x;
    const int K = a.K, nk = K / kStepK;
    uint64_t* fullL = reinterpret_cast<uint64_t*>(smem + L::bar);
    uint64_t* emptyL = fullL + kPL;
    uint64_t* fullB = emptyL + kPL;
    uint64_t* emptyB = fullB + kPB;
    uint64_t* done = emptyB + kPB;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + L::tslot);
    // first B row of 64-row box b: gate rows then up rows (SwiGLU), else consecutive rows
    auto brow = [&](int b) -> int {
        if (EPI == kEpiSwiglu)
            return g * a.b_group_rows + (b < NB / 2 ? nt * (TN / 2) + 64 * b : a.b_up_row0 + nt * (TN / 2) + 64 * (b - NB / 2));
        return g * a.b_group_rows + nt * TN + 64 * b;
    };

    if (tid == 0) {
        for (int i = 0; i < L::nbar; ++i) mbar_init(fullL + i, (i >= 2 * kPL && i < 2 * kPL + kPB) ? kPW : 1);
        fence_mbar_init();
    }
    if (warp == 9) {
        tmem_alloc(tslot, MT * TN);  // accumulator of tile t at columns [t TN, (t + 1) TN)
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tslot;
    bool ok = true;

    if (warp == 8) {
        // ---------------- loads (one thread) ----------------
        if (lane == 0) {
            const uint32_t bytes = (uint32_t)(L::stage - (size_t)(MT - ntile) * kTileBytes);
            for (int j = 0; j < nk && ok; ++j) {
                const int s = j % kPL, k0 = j * kStepK;
                if (j >= kPL) ok = mbar_wait_bounded(emptyL + s, ((j / kPL) - 1) & 1, a.status, kStatusTimeoutPrefill);
                if (!ok) break;
                uint8_t* st = smem + L::load + (size_t)s * L::stage;
                mbar_arrive_expect_tx(fullL + s, bytes);
                for (int t = 0; t < ntile; ++t) tma_load_2d(st + (size_t)t * kTileBytes, &tma_a, k0, row0 + t * kTileM, fullL + s);
                if constexpr (NVFP4) {
                    uint8_t* codes = st + MT * kTileBytes;
                    uint8_t* scales = codes + TN * 32;
                    const int sx = K / 2 + ((k0 / 16) & ~15);
#pragma unroll
                    for (int b = 0; b < NB; ++b) {
                        tma_load_2d(codes + 64 * 32 * b, &tma_b, k0 / 2, brow(b), fullL + s);
                        tma_load_2d(scales + 64 * 16 * b, &tma_s, sx, brow(b), fullL + s);
                    }
                } else {
                    tma_load_2d(st + MT * kTileBytes, &tma_b, k0, nt * TN, fullL + s);
                }
            }
        }
    } else if (warp == 9) {
        // ---------------- MMA issue (one thread) ----------------
        if (lane == 0) {
            const uint32_t idesc = tc_idesc_bf16(kTileM, TN);
            for (int i = 0; i < nk && ok; ++i) {
                const int sl = i % kPL, sb = i % kPB;
                if constexpr (NVFP4)
                    ok = mbar_wait_bounded(fullB + sb, (i / kPB) & 1, a.status, kStatusTimeoutPrefill);
                else
                    ok = mbar_wait_bounded(fullL + sl, (i / kPL) & 1, a.status, kStatusTimeoutPrefill);
                if (!ok) break;
                tc_fence_after_sync();
                const uint8_t* at = smem + L::load + (size_t)sl * L::stage;
                const uint8_t* bt = NVFP4 ? smem + L::btile + (size_t)sb * L::bt : at + MT * kTileBytes;
                for (int t = 0; t < ntile; ++t)
#pragma unroll
                    for (int kk = 0; kk < kStepK / 16; ++kk)
                        tc_mma_bf16(tmem + (uint32_t)(t * TN), tc_smem_desc_sw128(at + (size_t)t * kTileBytes + 32 * kk),
                                    tc_smem_desc_sw128(bt + 32 * kk), idesc, (i > 0 || kk > 0) ? 1u : 0u);
                tc_commit(emptyL + sl);
                if constexpr (NVFP4) tc_commit(emptyB + sb);
            }
            tc_commit(done);  // completes once every MMA issued above has
        }
    } else if constexpr (NVFP4) {
        // ---------------- dequantise (warps 0-7) ----------------
        // half rows u = tid, tid + 256, ...: row u % TN, half u / TN
        for (int i = 0; i < nk && ok; ++i) {
            const int sl = i % kPL, sb = i % kPB;
            ok = mbar_wait_bounded(fullL + sl, (i / kPL) & 1, a.status, kStatusTimeoutPrefill);
            if (ok && i >= kPB) ok = mbar_wait_bounded(emptyB + sb, ((i / kPB) - 1) & 1, a.status, kStatusTimeoutPrefill);
            if (!ok) break;
            const uint8_t* st = smem + L::load + (size_t)sl * L::stage + MT * kTileBytes;
            uint8_t* bt = smem + L::btile + (size_t)sb * L::bt;
#pragma unroll
            for (int u = tid; u < 2 * TN; u += kPW) {
                const int r = u & (TN - 1), hb = u / TN;
                const uint4 cw = *reinterpret_cast<const uint4*>(st + 32 * r + 16 * hb);
                const uint32_t sc = *reinterpret_cast<const uint32_t*>(st + TN * 32 + 16 * r + (((i * kStepK) / 16) & 15));
                const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int kc = 4 * hb + c;
                    const uint32_t sbyte = (sc >> (8 * (kc >> 1))) & 0x7Fu;
                    uint32_t s2;
                    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(s2) : "h"((uint16_t)(sbyte | (sbyte << 8))));
                    *reinterpret_cast<uint4*>(bt + tc_sw128_offset(r, 8 * kc)) = dequant8(words[c], s2);
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(fullB + sb);
        }
    }
    // ---------------- epilogue (warps 0-7) ----------------
    if (warp < 8) {
        if (ok) ok = mbar_wait_bounded(done, 0, a.status, kStatusTimeoutPrefill);
        tc_fence_after_sync();
        for (int t = 0; ok && t < ntile; ++t) {
            const int wq = warp & 3, half = warp >> 2;  // lane quarter, column half
            const int r = 32 * wq + lane;              // the TMEM lane = tile row of this thread
            const uint32_t tl = tmem + (uint32_t)(t * TN) + ((uint32_t)(32 * wq) << 16);
            const bool valid = t * kTileM + r < nrows;
            const int p = row0 + t * kTileM + r;
            if (EPI == kEpiSwiglu) {
                const float tsg = a.ts ? ld_cg(a.ts + (size_t)g * a.ts_stride) : 1.f;
                const float tsu = a.ts ? ld_cg(a.ts + (size_t)g * a.ts_stride + 1) : 1.f;
                for (int c = half * (TN / 4); c < (half + 1) * (TN / 4); c += 16) {
                    uint32_t gv[16], uv[16];
                    tmem_ld16(tl + c, gv);
                    tmem_ld16(tl + TN / 2 + c, uv);
                    tmem_ld_wait();
                    uint32_t o[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        float h2[2];
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const float gg = bf16_round_f32(tsg * __uint_as_float(gv[2 * i + h]));
                            const float uu = bf16_round_f32(tsu * __uint_as_float(uv[2 * i + h]));
                            h2[h] = silu_f(gg) * uu;
                        }
                        o[i] = (uint32_t)f32_to_bf16_bits(h2[0]) | ((uint32_t)f32_to_bf16_bits(h2[1]) << 16);
                    }
                    if (valid) {
                        uint4* dst = reinterpret_cast<uint4*>(a.out_bf16 + (size_t)p * a.ldo + nt * (TN / 2) + c);
                        dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
                        dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
                    }
                }
            } else {
                const float ts = (EPI == kEpiScale && a.ts) ? ld_cg(a.ts + (size_t)g * a.ts_stride + 2) : 1.f;
                for (int c = half * (TN / 2); c < (half + 1) * (TN / 2); c += 16) {
                    uint32_t v[16];
                    tmem_ld16(tl + c, v);
                    tmem_ld_wait();
                    if (!valid) continue;
                    if (EPI == kEpiLogits) {
                        if (a.n_valid && nt * TN + c >= a.n_valid) continue;  // n_valid % 16 == 0
                        float4* dst = reinterpret_cast<float4*>(a.out_f32 + (size_t)p * a.ldo + nt * TN + c);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            dst[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                                 __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
                    } else {
                        uint32_t o[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            o[i] = (uint32_t)f32_to_bf16_bits(ts * __uint_as_float(v[2 * i])) |
                                   ((uint32_t)f32_to_bf16_bits(ts * __uint_as_float(v[2 * i + 1])) << 16);
                        uint4* dst = reinterpret_cast<uint4*>(a.out_bf16 + (size_t)p * a.ldo + nt * TN + c);
                        dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
                        dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
                    }
                }
            }
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 9) tmem_dealloc(tmem, MT * TN);
}

// ---------------------------------------------------------------------------
// Routing: sigmoid top-k per token (one warp per token, 8 tokens per CTA).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) prefill_topk_kernel(const float* logits, const float* bias, int T, int E,
                                                           int k, int32_t* ids, float* weights) {
    // one warp per token: its logits straight from memory into registers, the
    // sigmoid (and bias) applied on load
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (t >= T) return;
    const float* lg = logits + (size_t)t * E;
    if (E <= 256)
        topk_warp_logits<8>(lg, bias, E, k, lane, ids + (size_t)t * k, weights + (size_t)t * k);
    else
        topk_warp_logits<FLINT_MAX_EXPERTS / 32>(lg, bias, E, k, lane, ids + (size_t)t * k, weights + (size_t)t * k);
}

// Counting sort of the (token, rank) pairs q = t k + j by expert, keeping q
// order within an expert, in chunks of kSortChunk pairs:
//   hist:    per chunk, how many of its pairs chose each expert;
//   scan:    per expert, its segment start and the start of each chunk's run
//            inside it; the segments' 128-row tile counts and their prefix;
//   scatter: per chunk, each pair's place = its chunk's run start + the pairs
//            of the same expert before it in the chunk (earlier warps, then
//            earlier lanes of its warp).
constexpr int kSortChunk = 512;

__global__ void __launch_bounds__(kSortChunk) prefill_hist_kernel(const int32_t* ids, int n, int E, int* chunk_hist) {
    extern __shared__ int hist[];
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
    __syncthreads();
    const int q = blockIdx.x * kSortChunk + threadIdx.x;
    if (q < n) atomicAdd(&hist[ids[q]], 1);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) chunk_hist[(size_t)blockIdx.x * E + e] = hist[e];
}

// One CTA of 1024 threads; E <= 1024. Q = 1024 / E threads per expert
// (thread q E + e), each over a contiguous range of the chunks, so that an
// expert's counts are read Q ranges at a time; the ranges' sums meet in
// shared memory.
__global__ void __launch_bounds__(1024) prefill_scan_kernel(const int* chunk_hist, int nch, int E, int* chunk_off,
                                                            int* seg_base, int* seg_len, int* tile_start,
                                                            int* pair_start) {
    __shared__ int part[1024];  // per thread: its range's sum, then the range's first offset
    __shared__ int wsum[32], wtile[32], wpair[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int Q = max(1, 1024 / E), q = tid / E, ex = tid - q * E;
    const bool act = q < Q;
    const int c0 = act ? (int)((long long)q * nch / Q) : 0, c1 = act ? (int)((long long)(q + 1) * nch / Q) : 0;
    int s = 0;
#pragma unroll 8
    for (int c = c0; c < c1; ++c) s += ld_cg(chunk_hist + (size_t)c * E + ex);  // independent loads in flight
    part[tid] = s;
    __syncthreads();
    // threads [0, E): expert e = tid, its total over the Q ranges
    const int e = tid;
    int total = 0;
    if (e < E)
        for (int j = 0; j < Q; ++j) total += part[j * E + e];
    const int tiles = (total + kTileM - 1) / kTileM, pairs = (tiles + 1) / 2;
    // exclusive scans of total, tiles and tile pairs over the experts
    int it = total, tt = tiles, pt = pairs;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int a = __shfl_up_sync(0xffffffffu, it, off), b = __shfl_up_sync(0xffffffffu, tt, off),
                  c2 = __shfl_up_sync(0xffffffffu, pt, off);
        if (lane >= off) {
            it += a;
            tt += b;
            pt += c2;
        }
    }
    if (lane == 31) {
        wsum[warp] = it;
        wtile[warp] = tt;
        wpair[warp] = pt;
    }
    __syncthreads();
    int wb = 0, wt = 0, wp = 0;
    for (int w = 0; w < warp; ++w) {
        wb += wsum[w];
        wt += wtile[w];
        wp += wpair[w];
    }
    const int base = wb + it - total, tbase = wt + tt - tiles, pbase = wp + pt - pairs;
    if (e < E) {
        seg_base[e] = base;
        seg_len[e] = total;
        tile_start[e] = tbase;
        pair_start[e] = pbase;
        if (e == E - 1) {
            tile_start[E] = tbase + tiles;
            pair_start[E] = pbase + pairs;
        }
        int run = base;  // each range's first offset, in chunk order
        for (int j = 0; j < Q; ++j) {
            const int v = part[j * E + e];
            part[j * E + e] = run;
            run += v;
        }
    }
    __syncthreads();
    if (act) {
        int run = part[tid];
#pragma unroll 8
        for (int c = c0; c < c1; ++c) {
            chunk_off[(size_t)c * E + ex] = run;
            run += ld_cg(chunk_hist + (size_t)c * E + ex);
        }
    }
}

__global__ void __launch_bounds__(kSortChunk) prefill_scatter_kernel(const int32_t* ids, int n, int E,
                                                                     const int* chunk_off, int* perm, int* inv) {
    extern __shared__ int cnt[];  // [kSortChunk / 32][E]
    constexpr int NW = kSortChunk / 32;
    for (int i = threadIdx.x; i < NW * E; i += blockDim.x) cnt[i] = 0;
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int q = blockIdx.x * kSortChunk + threadIdx.x;
    const int e = q < n ? ids[q] : -1;
    const uint32_t same = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(same & ((1u << lane) - 1u));
    if (e >= 0 && rank == 0) cnt[warp * E + e] = __popc(same);
    __syncthreads();
    if (e >= 0) {
        int before = 0;
        for (int w = 0; w < warp; ++w) before += cnt[w * E + e];
        const int pos = chunk_off[(size_t)blockIdx.x * E + e] + before + rank;
        perm[pos] = q;
        inv[q] = pos;
    }
}

// y[t] = bf16(sum_j w[t][j] d[inv[t k + j]] + d_shared[t]), ranks in order.
__global__ void __launch_bounds__(256) prefill_combine_kernel(const float* weights, const int* inv, int k,
                                                              const uint16_t* d, const uint16_t* ds, int H,
                                                              uint16_t* y) {
    const int t = blockIdx.x;
    float w[FLINT_MAX_TOPK];
    int pj[FLINT_MAX_TOPK];
    for (int j = 0; j < k; ++j) {
        w[j] = weights[(size_t)t * k + j];
        pj[j] = inv[(size_t)t * k + j];
    }
    for (int c = threadIdx.x * 8; c < H; c += blockDim.x * 8) {
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int j = 0; j < k; ++j) {
            const uint4 v = *reinterpret_cast<const uint4*>(d + (size_t)pj[j] * H + c);
            const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc[2 * i] = fmaf(w[j], bf16_lo(vw[i]), acc[2 * i]);
                acc[2 * i + 1] = fmaf(w[j], bf16_hi(vw[i]), acc[2 * i + 1]);
            }
        }
        if (ds) {
            const uint4 v = *reinterpret_cast<const uint4*>(ds + (size_t)t * H + c);
            const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc[2 * i] += bf16_lo(vw[i]);
                acc[2 * i + 1] += bf16_hi(vw[i]);
            }
        }
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            o[i] = (uint32_t)f32_to_bf16_bits(acc[2 * i]) | ((uint32_t)f32_to_bf16_bits(acc[2 * i + 1]) << 16);
        *reinterpret_cast<uint4*>(y + (size_t)t * H + c) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// x_perm[p] = x[perm[p] / k]: the expert-sorted copy of the token rows (one
// warp per row), so that the routed gate/up GEMM reads its A tiles as plain
// 2-D tiles.
__global__ void __launch_bounds__(256) prefill_gather_kernel(const uint16_t* x, const int* perm, int k, int H, int n,
                                                             uint16_t* x_perm) {
    const int p = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (p >= n) return;
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)(perm[p] / k) * H);
    uint4* dst = reinterpret_cast<uint4*>(x_perm + (size_t)p * H);
    for (int i = lane; i < H / 8; i += 32) dst[i] = src[i];
}

// ---------------------------------------------------------------------------
// Tensor maps (host): 2-D tiled maps for the TMA loads.
// ---------------------------------------------------------------------------
cudaError_t tensor_map(CUtensorMap* m, CUtensorMapDataType type, const void* base, uint64_t rows, uint64_t inner,
                       uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swz) {
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    if (!encode) {
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || !fn || q != cudaDriverEntryPointSuccess) return e != cudaSuccess ? e : cudaErrorNotSupported;
        encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t es[2] = {1, 1};
    const CUresult r = encode(m, type, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              swz, CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// A operand: bf16 [rows, K] row-major -> 128 x 64 tiles, 128-byte swizzle.
cudaError_t map_a(CUtensorMap* m, const uint16_t* A, uint64_t rows, uint64_t K) {
    return tensor_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, A, rows, K, 2 * K, kStepK, kTileM, CU_TENSOR_MAP_SWIZZLE_128B);
}

// One grouped GEMM launch: the A map, the B map(s) and the kernel.
template <bool NVFP4, int EPI, int TN, int MT = 1>
cudaError_t launch_gemm(const PrefillGemmArgs& a, uint64_t a_rows, uint64_t b_rows, const DevInfo& d, int m_tiles,
                        int n_tiles, cudaStream_t s) {
    static int configured_for = -1;
    cudaError_t e = configure_smem(prefill_gemm_kernel<NVFP4, EPI, TN, MT>, d, configured_for);
    if (e != cudaSuccess) return e;
    if (m_tiles <= 0 || n_tiles <= 0) return cudaSuccess;
    CUtensorMap ta, tb, ts;
    if ((e = map_a(&ta, a.A, a_rows, (uint64_t)a.K)) != cudaSuccess) return e;
    if (NVFP4) {
        // packed rows as bytes: 32-byte code windows and 16-byte scale windows of 64 rows
        if ((e = tensor_map(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.B, b_rows, (uint64_t)a.ldb, (uint64_t)a.ldb, 32, 64,
                            CU_TENSOR_MAP_SWIZZLE_NONE)) != cudaSuccess)
            return e;
        if ((e = tensor_map(&ts, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.B, b_rows, (uint64_t)a.ldb, (uint64_t)a.ldb, 16, 64,
                            CU_TENSOR_MAP_SWIZZLE_NONE)) != cudaSuccess)
            return e;
    } else {
        if ((e = tensor_map(&tb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.B, b_rows, (uint64_t)a.K, (uint64_t)a.ldb, kStepK,
                            TN, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
            return e;
        ts = tb;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)n_tiles, (unsigned)m_tiles);
    cfg.blockDim = dim3(kPT);
    cfg.dynamicSmemBytes = TmaSmem<NVFP4, TN, MT>::total;
    cfg.stream = s;
    return cudaLaunchKernelEx(&cfg, prefill_gemm_kernel<NVFP4, EPI, TN, MT>, ta, tb, ts, a);
}

}  // namespace

PrefillWs prefill_ws_layout(int T, int E, int k, int H, int I, int Is) {
    PrefillWs w;
    size_t o = kWsHeader;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = align_up(o + bytes, 256);
        return at;
    };
    w.logits = take(sizeof(float) * (size_t)T * E);
    const size_t nch = ((size_t)T * k + kSortChunk - 1) / kSortChunk;
    w.chunk_hist = take(sizeof(int) * nch * E);
    w.chunk_off = take(sizeof(int) * nch * E);
    w.seg_base = take(sizeof(int) * (size_t)E);
    w.seg_len = take(sizeof(int) * (size_t)E);
    w.tile_start = take(sizeof(int) * (size_t)(E + 1));
    w.pair_start = take(sizeof(int) * (size_t)(E + 1));
    w.perm = take(sizeof(int) * (size_t)T * k);
    w.inv = take(sizeof(int) * (size_t)T * k);
    w.h = take(2 * (size_t)T * k * I);
    w.hs = take(2 * (size_t)T * Is);
    w.d = take(2 * (size_t)T * k * H);
    w.x_perm = take(2 * (size_t)T * k * H);
    w.ds = take(2 * (size_t)T * H);
    w.total = o;
    return w;
}

cudaError_t launch_prefill(const PrefillArgs& p, const DevInfo& d, cudaStream_t s) {
    const PrefillWs W = prefill_ws_layout(p.T, p.E, p.k, p.H, p.I, p.Is);
    uint8_t* ws = static_cast<uint8_t*>(p.ws);
    float* logits = reinterpret_cast<float*>(ws + W.logits);
    int* chunk_hist = reinterpret_cast<int*>(ws + W.chunk_hist);
    int* chunk_off = reinterpret_cast<int*>(ws + W.chunk_off);
    int* seg_base = reinterpret_cast<int*>(ws + W.seg_base);
    int* seg_len = reinterpret_cast<int*>(ws + W.seg_len);
    int* tile_start = reinterpret_cast<int*>(ws + W.tile_start);
    int* pair_start = reinterpret_cast<int*>(ws + W.pair_start);
    int* perm = reinterpret_cast<int*>(ws + W.perm);
    int* inv = reinterpret_cast<int*>(ws + W.inv);
    uint16_t* h = reinterpret_cast<uint16_t*>(ws + W.h);
    uint16_t* hs = reinterpret_cast<uint16_t*>(ws + W.hs);
    uint16_t* dd = reinterpret_cast<uint16_t*>(ws + W.d);
    uint16_t* ds = reinterpret_cast<uint16_t*>(ws + W.ds);
    uint32_t* status = reinterpret_cast<uint32_t*>(ws) + 1;
    const int T = p.T, E = p.E, k = p.k, H = p.H, I = p.I, Is = p.Is;
    const int mt_all = (T + kTileM - 1) / kTileM;
    // the expert GEMMs' CTAs: kMT M-tiles each (bounds for the grouped ones)
    const int mx_all = (T + kMT * kTileM - 1) / (kMT * kTileM);
    const int mx_routed = (T * k + kMT * kTileM - 1) / (kMT * kTileM) + E;
    const long long rs_h = nvfp4_row_stride(H), rs_i = nvfp4_row_stride(I), rs_is = Is ? nvfp4_row_stride(Is) : 0;
    cudaError_t e;

    // 1. router logits (FP32) = x Wr^T
    PrefillGemmArgs r = {};
    r.A = p.x;
    r.lda = H;
    r.rows = T;
    r.K = H;
    r.B = reinterpret_cast<const uint8_t*>(p.router_w);
    r.ldb = 2 * (long long)H;
    r.n_valid = E;
    r.out_f32 = logits;
    r.ldo = E;
    r.status = status;
    if ((e = launch_gemm<false, kEpiLogits, 128>(r, T, E, d, mt_all, (E + 127) / 128, s)) != cudaSuccess) return e;
    // 2. top-k per token
    prefill_topk_kernel<<<(T + 7) / 8, 256, 0, s>>>(logits, p.bias, T, E, k, p.ids, p.weights);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // 3. pairs sorted by expert
    const int nch = (T * k + kSortChunk - 1) / kSortChunk;
    static int scatter_cfg = -1;  // its per-warp tables exceed 48 KB for E > 768
    if (scatter_cfg != d.device) {
        if ((e = cudaFuncSetAttribute(prefill_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)(sizeof(int) * (kSortChunk / 32) * FLINT_MAX_EXPERTS))) != cudaSuccess)
            return e;
        scatter_cfg = d.device;
    }
    prefill_hist_kernel<<<nch, kSortChunk, sizeof(int) * E, s>>>(p.ids, T * k, E, chunk_hist);
    prefill_scan_kernel<<<1, 1024, 0, s>>>(chunk_hist, nch, E, chunk_off, seg_base, seg_len, tile_start, pair_start);
    prefill_scatter_kernel<<<nch, kSortChunk, sizeof(int) * (kSortChunk / 32) * E, s>>>(p.ids, T * k, E, chunk_off,
                                                                                       perm, inv);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // 4. gate/up + SiLU: routed experts over their (expert-sorted) token rows, the shared expert over all
    uint16_t* x_perm = reinterpret_cast<uint16_t*>(ws + W.x_perm);
    prefill_gather_kernel<<<(T * k + 7) / 8, 256, 0, s>>>(p.x, perm, k, H, T * k, x_perm);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    PrefillGemmArgs g = {};
    g.A = x_perm;
    g.lda = H;
    g.tile_start = tile_start;
    g.pair_start = pair_start;
    g.seg_base = seg_base;
    g.seg_len = seg_len;
    g.n_groups = E;
    g.K = H;
    g.B = p.gu;
    g.ldb = rs_h;
    g.b_group_rows = 2 * I;
    g.b_up_row0 = I;
    g.ts = p.ts;
    g.ts_stride = 3;
    g.out_bf16 = h;
    g.ldo = I;
    g.status = status;
    if ((e = launch_gemm<true, kEpiSwiglu, kNTile, kMT>(g, (uint64_t)T * k, (uint64_t)E * 2 * I, d, mx_routed,
                                                         I / (kNTile / 2), s)) != cudaSuccess)
        return e;
    if (p.s_gu) {
        PrefillGemmArgs gs = {};
        gs.A = p.x;
        gs.lda = H;
        gs.rows = T;
        gs.K = H;
        gs.B = p.s_gu;
        gs.ldb = rs_h;
        gs.b_up_row0 = Is;
        gs.ts = p.s_ts;
        gs.out_bf16 = hs;
        gs.ldo = Is;
        gs.status = status;
        if ((e = launch_gemm<true, kEpiSwiglu, kNTile, kMT>(gs, T, 2 * (uint64_t)Is, d, mx_all, Is / (kNTile / 2),
                                                             s)) != cudaSuccess)
            return e;
    }
    // 5. down
    PrefillGemmArgs dn = {};
    dn.A = h;
    dn.lda = I;
    dn.tile_start = tile_start;
    dn.pair_start = pair_start;
    dn.seg_base = seg_base;
    dn.seg_len = seg_len;
    dn.n_groups = E;
    dn.K = I;
    dn.B = p.down;
    dn.ldb = rs_i;
    dn.b_group_rows = H;
    dn.ts = p.ts;
    dn.ts_stride = 3;
    dn.out_bf16 = dd;
    dn.ldo = H;
    dn.status = status;
    if ((e = launch_gemm<true, kEpiScale, kNTile, kMT>(dn, (uint64_t)T * k, (uint64_t)E * H, d, mx_routed, H / kNTile,
                                                        s)) != cudaSuccess)
        return e;
    if (p.s_down) {
        PrefillGemmArgs dsa = {};
        dsa.A = hs;
        dsa.lda = Is;
        dsa.rows = T;
        dsa.K = Is;
        dsa.B = p.s_down;
        dsa.ldb = rs_is;
        dsa.ts = p.s_ts;
        dsa.out_bf16 = ds;
        dsa.ldo = H;
        dsa.status = status;
        if ((e = launch_gemm<true, kEpiScale, kNTile, kMT>(dsa, T, H, d, mx_all, H / kNTile, s)) != cudaSuccess)
            return e;
    }
    // 6. combine
    prefill_combine_kernel<<<T, 256, 0, s>>>(p.weights, inv, k, dd, p.s_down ? ds : nullptr, H, p.y);
    return cudaGetLastError();
}

}  // namespace flint
