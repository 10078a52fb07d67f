// flint_internal.h -- declarations shared by the library's translation units
// (kernel argument blocks, workspace layout, launchers, error reporting).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "flint.h"

#if defined(__CUDACC__)
#define FLINT_HD __host__ __device__
#else
#define FLINT_HD
#endif

namespace flint {

// A bounded device-side wait gives up after this long (a copy of a few KB
// normally lands in microseconds; this only turns a lost copy into an error).
constexpr uint64_t kWaitBudgetNs = 2000000000ull;

// Status-word bits (workspace header, word 1).
enum : uint32_t {
    kStatusTimeoutRoute = 1u << 0,
    kStatusTimeoutGateUp = 1u << 1,
    kStatusTimeoutDown = 1u << 2,
    kStatusTimeoutSelftest = 1u << 3,
    kStatusBadExpertId = 1u << 4,
    kStatusTimeoutLayer = 1u << 5,
    kStatusTimeoutPrefill = 1u << 6,
    kStatusLayerPlan = 1u << 7,  // a fused-layer CTA's work exceeded the shared-memory plan (not expected)
};

constexpr int kThreads = 256;       // router kernel: 8 warps
constexpr int kWarps = kThreads / 32;
// Expert / dense GEMV kernels: 24 warps, each streaming its own share of the
// weight rows through a private ring of shared-memory slots (so 24 warps per
// SM issue copies; 24 measured faster than 16 or 32: deeper rings, same issue).
constexpr int kGemvWarps = 24;
constexpr int kGemvThreads = kGemvWarps * 32;
constexpr int kMaxSlotsPerWarp = 4;
constexpr size_t kWsHeader = 256;   // control words, below
// Workspace header words (uint32): the router's arrival counter, the status
// word, the fused layer's count of completed calls and of finished CTAs, the
// bounded waits' budget in microseconds (0: kWaitBudgetNs), a test hook
// (c + 1: CTA c of the next fused-layer call publishes neither router scores
// nor h counts), and the fused layer's counts of published router rows and
// (one token) of gate/up pairs whose h is written (both 0 between calls).
enum : int {
    kHdrRouteCounter = 0,
    kHdrStatus = 1,
    kHdrCalls = 4,
    kHdrDone = 5,
    kHdrBudget = 6,
    kHdrLoseCta = 7,
    kHdrScoresIn = 8,
    kHdrPairsIn = 9,
};
// Expert GEMV kernels for BF16 weights: 16 warps (a BF16 row is 4x the bytes
// of an NVFP4 row, so fewer, larger ring slots per SM).
constexpr int kBf16Warps = 16;
constexpr int kBf16Threads = kBf16Warps * 32;
// Fused layer kernel: one cooperative CTA per SM.
constexpr int kLayerWarps = 24;
constexpr int kLayerThreads = kLayerWarps * 32;
constexpr int kLayerSlots = 2;           // ring slots of each warp of the fused layer
constexpr int kLayerMaxHidden = 8192;    // largest hidden size of the fused layer
constexpr int kLayerRowsMaxTokens = 1;   // fused layer: down split by output rows up to this many tokens
// One-token layer kernel: 12 warps, so that two CTAs fit on an SM (registers)
// and the next layer's CTA starts its static copies while this one finishes.
constexpr int kOneWarps = 12;
constexpr int kOneThreads = kOneWarps * 32;

FLINT_HD constexpr size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Workspace regions, from the layer shape: the router's FP32 logits [8][E]
// (the fused layer: the sigmoid scores' bits) and the bf16 h of the routed
// [8][k][I] and shared [8][Is] experts; then the fused layer's bf16
// per-expert outputs d of the routed ranks [8][k][H] and of the shared expert
// [8][H], its per-16-row-block arrival counters [H / 16] and its per-expert
// counts of published h pairs [kMaxDistinct + 1] (the shared expert last).
struct WsLayout {
    size_t logits_off, h_routed_off, h_shared_off, d_routed_off, d_shared_off, counters_off, unit_counters_off,
        total;
};
inline WsLayout ws_layout(int E, int k, int H, int I, int Is) {
    WsLayout L;
    const size_t Tm = FLINT_MAX_TOKENS;
    L.logits_off = kWsHeader;
    L.h_routed_off = align_up(L.logits_off + sizeof(float) * Tm * (size_t)E, 256);
    L.h_shared_off = align_up(L.h_routed_off + 2 * Tm * k * (size_t)I, 256);
    L.d_routed_off = align_up(L.h_shared_off + 2 * Tm * (size_t)Is, 256);
    L.d_shared_off = align_up(L.d_routed_off + 2 * Tm * k * (size_t)H, 256);
    L.counters_off = align_up(L.d_shared_off + 2 * Tm * (size_t)H, 256);
    L.unit_counters_off = align_up(L.counters_off + 4 * (size_t)(H / 16), 256);
    L.total = align_up(L.unit_counters_off + 4 * (size_t)(FLINT_MAX_TOKENS * FLINT_MAX_TOPK + 1), 256);
    return L;
}

FLINT_HD inline int64_t nvfp4_row_stride(int64_t cols) { return (int64_t)align_up((size_t)(cols / 2 + cols / 16), 16); }

// ---------------------------------------------------------------------------
// Kernel argument blocks
// ---------------------------------------------------------------------------
struct RouteArgs {
    const uint16_t* x;
    int T, H;
    const uint16_t* wr;
    int E;
    const float* bias;
    int k;
    int32_t* ids;
    float* weights;
    float* logits;     // workspace [8][E]
    uint32_t* counter; // workspace word 0
    uint32_t* status;  // workspace word 1
    int rows_per_cta;
};

// Gate/up + SiLU (pair mode) or plain rows (dense GEMV without epilogue).
// "routed" may be absent (dense); "shared" is the always-on shared expert or
// the dense matrix.
struct GateUpArgs {
    const uint16_t* x;
    int T, H;           // tokens, columns (K)
    const int32_t* ids;
    int k;
    const uint8_t* gu;  // routed: E x [2I, H]
    int E, I;
    const float* ts;    // [E][3]
    const uint8_t* s_gu; // shared: [2Is, H] (pair) or [Is, H] (plain rows), or null
    int Is;
    const float* s_ts;  // [>=2] (pair) or [1]
    uint16_t* h_routed; // [8][k][I]
    uint16_t* h_shared; // [T][Is]: h of the shared expert, or the dense output y
    uint32_t* status;
    int nslots;         // ring slots per warp (one item each)
    int res_items;      // bound on the items of one CTA (shared-memory sums)
    int x_early;        // x is complete before the PDL wait (previous kernel: the router)
};

// Down + combine of the MoE layer.
struct DownArgs {
    const int32_t* ids;
    const float* w;
    int T, k, H;
    const uint8_t* down; // routed: E x [H, I]
    int E, I;
    const float* ts;     // [E][3]; the down scale is index 2
    const uint8_t* s_down; // shared: [H, Is] or null
    int Is;
    const float* s_ts;   // scale s_ts[2]
    const uint16_t* h_routed; // [8][k][I]
    const uint16_t* h_shared; // [T][Is]
    uint16_t* y;              // [T][H]
    uint32_t* status;
    int rg;                   // rows per task: 8 or 16
    int nslots;               // ring slots per warp
    int rows_max;             // largest row slice of any CTA
    int slot_bytes;           // bytes of one slot
};

// Residual add + RMSNorm ahead of a block: per token r' = bf16(r + y) (r' = r
// without y), x = bf16(r' / sqrt(mean(r'^2) + eps) * gamma) (gamma = 1 without
// it). r_out / x_out receive r' / x when given.
struct NormArgs {
    const uint16_t* r;      // [T][H]; null: no norm
    const uint16_t* y;      // [T][H] or null
    const uint16_t* gamma;  // [H] or null
    float eps;
    uint16_t* r_out;        // [T][H] or null
    uint16_t* x_out;        // [T][H] or null
    int T, H;
};

// The whole MoE decode step of one layer (router, gate/up, down, combine).
struct LayerArgs {
    const uint16_t* x;
    int T, H;
    const uint16_t* wr;  // router [E, H] bf16
    int E;
    const float* bias;   // [E] or null
    int k;
    int32_t* ids;        // [T][k] out (given: in)
    float* weights;      // [T][k] out (given: in)
    uint32_t* hdr;       // workspace header (kHdr* words)
    uint32_t* status;    // hdr + kHdrStatus
    uint32_t* scores;    // workspace [8][E]: the bits of the sigmoid scores
    uint16_t* h_routed;  // workspace [8][k][I]: bf16 h
    uint16_t* h_shared;  // workspace [8][Is]
    uint16_t* d_routed;  // workspace [8][k][H]: bf16 d of each rank
    uint16_t* d_shared;  // workspace [8][H]
    uint32_t* counters;  // workspace [H / 16]: arrivals per row block (0 between calls)
    uint32_t* unit_counters;  // workspace [kMaxDistinct + 1]: published h pairs per expert (0 between calls)
    const uint8_t* gu;   // routed E x [2I, H]
    const uint8_t* down; // routed E x [H, I]
    int I;
    const float* ts;     // [E][3]
    const uint8_t* s_gu; // shared [2Is, H] or null
    const uint8_t* s_down;
    int Is;
    const float* s_ts;
    uint16_t* y;         // [T][H] out
    int Gs;              // CTAs [0, Gs) run the shared expert
    int rpc;             // router rows per CTA
    int ns, slot;        // ring slots per warp (kLayerSlots) and bytes per slot
    int stage_vals, stage_scales;  // bytes of the staging region (x, later h) and of its chunk scales
    int rows;            // down split by output rows (the ROWS instantiation)
    const uint8_t* pf_ptr[4];      // the next layer's ranges to pull into L2 before the PDL wait
    unsigned long long pf_bytes[4];
    unsigned long long pf_granules;  // their total in 16-byte granules
    int rows_max;        // ROWS: most output rows of a CTA (ceil(H / G))
    int rg;              // ROWS: rows per down item (a power of two, at most 8)
    NormArgs norm;       // norm.r set: x = the norm of the residual stream (x unused)
    int given;           // ids and weights are inputs (flint_moe_decode): no router
    int x_early;         // given: x is complete before the PDL wait (the router ran on it)
    int one;             // one token: the latency-laid-out kernel (layer_one_kernel)
    int one_items;       // one: most gate/up pairs of a CTA (shared + routed)
    int one_rsd;         // one: bytes of a down-row slot (the larger row stride of I and Is)
};

// One grouped GEMM of the prefill: C[rows of each group] = A B^T on 128 x 128
// tiles, operands loaded by TMA. Groups (experts) are row segments
// [seg_base[g], + seg_len[g]) of A and of the output; tile_start[g] is the
// exclusive prefix of their 128-row tile counts (n_groups + 1 entries).
// Without tile_start there is one group of `rows`.
struct PrefillGemmArgs {
    const uint16_t* A;     // bf16 [rows of all groups, K], lda elements apart
    long long lda;
    const int* tile_start;
    const int* pair_start;   // exclusive prefix of the groups' counts of M-tile pairs (two tiles per CTA)
    const int* seg_base;
    const int* seg_len;
    int n_groups, rows, K;
    const uint8_t* B;      // the groups' B matrices stacked: group g's rows start at row g * b_group_rows
    long long ldb;         // bytes between B rows
    int b_group_rows;
    int b_up_row0;         // SwiGLU: first up row (the gate rows start at 0)
    int n_valid;           // valid B rows (0: all); rows past it read as zero, their columns are not stored
    const float* ts;       // tensor scales of group g at ts + g * ts_stride (gate, up, down), or null
    int ts_stride;
    float* out_f32;        // logits
    uint16_t* out_bf16;    // h or d
    long long ldo;         // output row stride (elements)
    uint32_t* status;
};

// The MoE layer over T tokens (prefill).
struct PrefillArgs {
    const uint16_t* x;      // [T][H]
    int T, H;
    const uint16_t* router_w;  // [E][H]
    int E;
    const float* bias;
    int k;
    const uint8_t* gu;      // routed E x [2I, H] NVFP4
    const uint8_t* down;    // routed E x [H, I]
    int I;
    const float* ts;        // [E][3]
    const uint8_t* s_gu;    // shared [2Is, H] or null
    const uint8_t* s_down;
    int Is;
    const float* s_ts;
    int32_t* ids;           // [T][k] out
    float* weights;         // [T][k] out
    uint16_t* y;            // [T][H] out
    void* ws;
};

struct PrefillWs {
    size_t logits, chunk_hist, chunk_off, seg_base, seg_len, tile_start, pair_start, perm, inv, h, hs, d, x_perm, ds,
        total;
};
PrefillWs prefill_ws_layout(int T, int E, int k, int H, int I, int Is);

// ---------------------------------------------------------------------------
// Launchers (return the CUDA error of the launch)
// ---------------------------------------------------------------------------
struct DevInfo {
    int device;
    int sm_count;
    int cc_major, cc_minor;
    int smem_optin;
};

cudaError_t launch_repack(const uint8_t* src, int64_t n_mats, int64_t rows, int64_t cols, uint8_t* dst,
                          int64_t mat_stride, cudaStream_t s);
cudaError_t launch_unrepack(const uint8_t* dst, int64_t n_mats, int64_t rows, int64_t cols, int64_t mat_stride,
                            uint8_t* src, cudaStream_t s);
cudaError_t launch_dequant(const uint8_t* packed, int64_t rows, int64_t cols, float* out, cudaStream_t s);
cudaError_t launch_route(const RouteArgs& a, const DevInfo& d, bool pdl, cudaStream_t s);
cudaError_t launch_gate_up(const GateUpArgs& a, bool pair, const DevInfo& d, bool pdl, cudaStream_t s);
cudaError_t launch_down(const DownArgs& a, const DevInfo& d, bool pdl, cudaStream_t s);
// BF16 expert weights (same argument blocks; gu/down/s_gu/s_down hold bf16
// matrices, ts/s_ts may be null for 1).
cudaError_t launch_gate_up_bf16(const GateUpArgs& a, const DevInfo& d, bool pdl, cudaStream_t s);
cudaError_t launch_down_bf16(const DownArgs& a, const DevInfo& d, bool pdl, cudaStream_t s);
size_t gate_up_bf16_smem_bytes(const GateUpArgs& a);
size_t down_bf16_smem_bytes(const DownArgs& a);
// Standalone residual add + RMSNorm (x_out required), one CTA per token.
cudaError_t launch_rmsnorm(const NormArgs& a, bool pdl, cudaStream_t s);
// The prefill: router GEMM, top-k, expert sort, grouped gate/up and down
// GEMMs on tcgen05, combine (eight launches in stream order).
cudaError_t launch_prefill(const PrefillArgs& p, const DevInfo& d, cudaStream_t s);
cudaError_t launch_selftest_wait(uint32_t* status, uint64_t budget_ns, cudaStream_t s);
// Cooperative launch of the fused layer kernel, one CTA on every SM (with the
// programmatic-dependent-launch attribute when `pdl`).
cudaError_t launch_layer(const LayerArgs& a, const DevInfo& d, bool pdl, cudaStream_t s);
size_t layer_smem_bytes(const LayerArgs& a);

// Allows `kernel` the device's opt-in dynamic shared memory, less its own
// static shared memory (once per device and kernel).
template <typename K>
cudaError_t configure_smem(K kernel, const DevInfo& d, int& configured_for) {
    if (configured_for == d.device) return cudaSuccess;
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, kernel);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             d.smem_optin - (int)fa.sharedSizeBytes);
    if (e == cudaSuccess) configured_for = d.device;
    return e;
}

size_t gate_up_smem_bytes(const GateUpArgs& a, bool pair);
size_t down_smem_bytes(const DownArgs& a);
size_t route_smem_bytes(const RouteArgs& a);

}  // namespace flint
