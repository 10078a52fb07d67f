// abi.cu -- the extern "C" entry points declared in include/flint.h:
// argument validation on the host, workspace bookkeeping, launch.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "flint_internal.h"

using flint::DevInfo;

namespace {

thread_local char g_err[512] = "";

void set_err(const char* fmt, va_list ap) { vsnprintf(g_err, sizeof g_err, fmt, ap); }

flint_status_t fail(flint_status_t st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    set_err(fmt, ap);
    va_end(ap);
    return st;
}

flint_status_t cuda_fail(cudaError_t e, const char* what) {
    snprintf(g_err, sizeof g_err, "%s: %s", what, cudaGetErrorString(e));
    return FLINT_ERR_CUDA;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// Device facts, cached per device. Only sm_103 devices are accepted.
flint_status_t device_info(DevInfo& d) {
    static std::mutex mu;
    static DevInfo cache[64];
    static bool have[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < 64 && have[dev]) {
        d = cache[dev];
        return FLINT_OK;
    }
    DevInfo n = {};
    n.device = dev;
    if ((e = cudaDeviceGetAttribute(&n.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&n.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&n.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&n.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
        return cuda_fail(e, "cudaDeviceGetAttribute");
    if (n.cc_major != 10 || n.cc_minor != 3)
        return fail(FLINT_ERR_UNSUPPORTED, "device %d is sm_%d%d; the kernels are built for sm_103a only", dev,
                    n.cc_major, n.cc_minor);
    if (dev >= 0 && dev < 64) {
        cache[dev] = n;
        have[dev] = true;
    }
    d = n;
    return FLINT_OK;
}

uint32_t* ws_status(void* ws) { return reinterpret_cast<uint32_t*>(ws) + 1; }

flint_status_t check_experts(const flint_experts* x, const char* name, bool need_down) {
    if (!x) return fail(FLINT_ERR_INVALID_ARG, "%s experts: null", name);
    if (x->dtype != FLINT_DTYPE_NVFP4 && x->dtype != FLINT_DTYPE_BF16)
        return fail(FLINT_ERR_UNSUPPORTED, "%s experts: unknown dtype %d", name, x->dtype);
    if (x->num_experts < 1 || x->num_experts > FLINT_MAX_EXPERTS)
        return fail(FLINT_ERR_UNSUPPORTED, "%s experts: num_experts %d outside 1..%d", name, x->num_experts,
                    FLINT_MAX_EXPERTS);
    if (x->hidden <= 0 || x->hidden % 1024)
        return fail(FLINT_ERR_UNSUPPORTED, "%s experts: hidden %d must be a positive multiple of 1024", name,
                    x->hidden);
    if (x->inter <= 0 || x->inter % 256)
        return fail(FLINT_ERR_UNSUPPORTED, "%s experts: inter %d must be a positive multiple of 256", name, x->inter);
    if ((x->dtype == FLINT_DTYPE_NVFP4 && !x->tensor_scale) || (x->tensor_scale && !aligned(x->tensor_scale, 4)))
        return fail(FLINT_ERR_INVALID_ARG, "%s experts: tensor_scale null or misaligned", name);
    if (!x->gate_up || !aligned(x->gate_up, 16))
        return fail(FLINT_ERR_INVALID_ARG, "%s experts: gate_up null or not 16-byte aligned", name);
    if (need_down && (!x->down || !aligned(x->down, 16)))
        return fail(FLINT_ERR_INVALID_ARG, "%s experts: down null or not 16-byte aligned", name);
    return FLINT_OK;
}

flint_status_t check_ws(const void* ws, size_t ws_bytes, size_t need) {
    if (!ws || !aligned(ws, 256)) return fail(FLINT_ERR_INVALID_ARG, "workspace null or not 256-byte aligned");
    if (ws_bytes < need)
        return fail(FLINT_ERR_INVALID_ARG, "workspace has %zu bytes, needs %zu", ws_bytes, need);
    return FLINT_OK;
}

int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

// Shared memory a launch may take, leaving room for the kernel's static data.
constexpr size_t kSmemSlack = 1024;

// Per-warp ring of the gate/up kernel: up to 4 slots of one item (a copy in
// flight while the previous item is computed), fewer when a warp has less
// work or the CTA would not fit in shared memory. `items` bounds the work
// items of one CTA (their raw sums stay in shared memory). Returns false when
// nothing fits.
bool gate_up_shape(flint::GateUpArgs& a, bool pair, int smem_optin, long long items) {
    a.res_items = (int)items;
    const int per_warp = ceil_div(items, flint::kGemvWarps);
    for (int ns = per_warp < 1 ? 1 : (per_warp > 4 ? 4 : per_warp); ns >= 1; --ns) {
        a.nslots = ns;
        if (flint::gate_up_smem_bytes(a, pair) + kSmemSlack <= (size_t)smem_optin) return true;
    }
    return false;
}

// Shapes of the down kernel: tasks of 16 rows when every task of a warp can
// be in flight at once, else whichever of 16 or 8 rows keeps the larger share
// of a warp's tasks in flight (up to 4 slots per warp). Returns false when
// the layer does not fit.
bool down_shape(flint::DownArgs& a, int sm_count, int smem_optin) {
    a.rows_max = ceil_div(a.H, sm_count);
    const long long rs_r = a.I > 0 ? flint::nvfp4_row_stride(a.I) : 0;
    const long long rs_s = a.Is > 0 ? flint::nvfp4_row_stride(a.Is) : 0;
    const long long rs = rs_r > rs_s ? rs_r : rs_s;
    const int units = (a.T * a.k < a.E ? a.T * a.k : a.E) + (a.Is > 0 ? 1 : 0);
    bool found = false;
    double best_cover = -1.0;
    flint::DownArgs best = a;
    for (int rg : {16, 8}) {
        const int per_warp = ceil_div((long long)units * ceil_div(a.rows_max, rg), flint::kGemvWarps);
        for (int ns = per_warp < 4 ? per_warp : 4; ns >= 1; --ns) {
            flint::DownArgs t = a;
            t.rg = rg;
            t.nslots = ns;
            t.slot_bytes = (int)(rg * rs);
            if (flint::down_smem_bytes(t) + kSmemSlack > (size_t)smem_optin) continue;
            const double cover = (double)ns / per_warp;
            if (cover > best_cover + 1e-9) {
                best = t;
                best_cover = cover;
                found = true;
            }
            break;
        }
    }
    if (found) a = best;
    return found;
}

// BF16 gate/up: ring slots per warp (one row each, up to 4), as many as fit.
bool gate_up_bf16_shape(flint::GateUpArgs& a, int smem_optin, long long pairs) {
    a.res_items = (int)pairs;
    const int per_warp = ceil_div(2 * pairs, flint::kBf16Warps);
    for (int ns = per_warp < 1 ? 1 : (per_warp > 4 ? 4 : per_warp); ns >= 1; --ns) {
        a.nslots = ns;
        if (flint::gate_up_bf16_smem_bytes(a) + kSmemSlack <= (size_t)smem_optin) return true;
    }
    return false;
}

// BF16 down: tasks of 8 or 4 rows; whichever keeps the larger share of a
// warp's tasks in flight (8 on a tie), up to 4 slots per warp.
bool down_bf16_shape(flint::DownArgs& a, int sm_count, int smem_optin) {
    a.rows_max = ceil_div(a.H, sm_count);
    const int kmax = a.I > a.Is ? a.I : a.Is;
    const int units = (a.T * a.k < a.E ? a.T * a.k : a.E) + (a.Is > 0 ? 1 : 0);
    bool found = false;
    double best_cover = -1.0;
    flint::DownArgs best = a;
    for (int rg : {8, 4}) {
        const int per_warp = ceil_div((long long)units * ceil_div(a.rows_max, rg), flint::kBf16Warps);
        for (int ns = per_warp < 4 ? per_warp : 4; ns >= 1; --ns) {
            flint::DownArgs t = a;
            t.rg = rg;
            t.nslots = ns;
            t.slot_bytes = 2 * rg * kmax;
            if (flint::down_bf16_smem_bytes(t) + kSmemSlack > (size_t)smem_optin) continue;
            const double cover = (double)ns / per_warp;
            if (cover > best_cover + 1e-9) {
                best = t;
                best_cover = cover;
                found = true;
            }
            break;
        }
    }
    if (found) a = best;
    return found;
}

// Shapes of the fused layer kernel. The shared expert gets the CTAs
// [0, Gs), in proportion to its cost among all the layer's experts: a row of
// an expert costs ~ 4 + 3 x the tokens that use it (decoding the codes once,
// then a multiply-add per token; measured per-pair times at 1 and 8 tokens),
// with the routed experts' token count at its expected T k / min(E, T k).
bool layer_shape(flint::LayerArgs& a, int sm_count, int smem_optin) {
    const int G = sm_count;
    const int T = a.T, H = a.H;
    const int units = a.T * a.k < a.E ? a.T * a.k : a.E;
    if (a.s_gu) {
        const double n_routed = (double)T * a.k / units;
        const double cs = (4.0 + 3.0 * T) * a.Is, cr = units * (4.0 + 3.0 * n_routed) * a.I;
        int gs = (int)(G * cs / (cs + cr) + 0.5);
        a.Gs = gs < 1 ? 1 : (gs > G / 2 ? G / 2 : gs);
    } else {
        a.Gs = 0;
    }
    a.rpc = a.given ? 0 : ceil_div(a.E, G - a.Gs);  // router rows per routed CTA
    // the kernel splits by cost in 32-bit arithmetic: the total cost of the
    // routed pairs (or blocks) times the group's CTA count must stay below 2^32
    // (an expert's weight is at most 4 + 3 T and the weights sum to at most
    // 4 min(E, T k) + 3 T k)
    const unsigned long long wmax = 4ull * units + 3ull * T * a.k;
    const unsigned long long per = (unsigned long long)(a.I > H / 16 ? a.I : H / 16);
    if (wmax * per * (unsigned long long)(G + 1) >= (1ull << 32)) return false;
    // a ring slot holds one gate/up pair (two rows of H) or a group of down rows
    const int RS = (int)flint::nvfp4_row_stride(H);
    a.slot = 2 * RS;
    const int kmax = a.I > a.Is ? a.I : a.Is;
    if (a.slot < flint::nvfp4_row_stride(kmax)) return false;
    // up to kLayerRowsMaxTokens tokens down is split by output rows: rg rows
    // (a power of two up to 8) of I or Is values per ring slot
    a.rows = T <= flint::kLayerRowsMaxTokens ? 1 : 0;
    a.rows_max = ceil_div(H, G);
    const int RSk = (int)flint::nvfp4_row_stride(kmax);
    a.rg = 8;
    while (a.rg > 1 && a.rg * RSk > a.slot) a.rg >>= 1;
    // staging: x, later the h of at most two routed experts (all tokens) or of
    // the shared expert; split by rows, all of h
    const size_t x_vals = 2 * (size_t)T * H, x_sc = 4 * (size_t)T * (H / 32);
    const size_t h_r = 2 * (2 * (size_t)T * a.I), h_s = 2 * (size_t)T * a.Is;  // two routed experts, or the shared one
    size_t h_vals = h_r > h_s ? h_r : h_s;
    size_t h_sc = 4 * (size_t)T * ((2 * a.I > a.Is ? 2 * a.I : a.Is) / 32);
    if (a.rows) {
        h_vals = 2 * (size_t)T * ((size_t)a.k * a.I + a.Is);
        h_sc = 4 * (size_t)T * ((size_t)a.k * (a.I / 32) + a.Is / 32);
    }
    a.stage_vals = (int)(x_vals > h_vals ? x_vals : h_vals);
    a.stage_scales = (int)(x_sc > h_sc ? x_sc : h_sc);
    // two ring slots per warp (three, where they fit, measured slower at 8
    // tokens: more copies in flight slowed the weight stream)
    a.ns = flint::kLayerSlots;
    return flint::layer_smem_bytes(a) + kSmemSlack <= (size_t)smem_optin;
}

// Shapes of the one-token kernel (layer_one_kernel): CTA c of G takes router
// rows, shared pairs, routed pairs and output rows in equal shares; every
// share of a CTA must fit its shared memory at once (no rings). False where
// it does not (the fused layer kernel then runs the token). Blocks (the norm
// fused in) stay on the fused layer kernel: chained block after block, the
// one-token kernel measured slower (935-940 against 907 us for the 49-block
// stack on one GPU), the plain layer within noise of it or faster.
bool one_shape(flint::LayerArgs& a, int sm_count, int smem_optin) {
    const int G = sm_count;
    if (a.T != 1 || a.norm.r) return false;
    a.rpc = a.given ? 0 : ceil_div(a.E, G);
    if (a.rpc > flint::kOneWarps - 1) return false;  // one router row per warp, the last warp selects
    const int ns_max = a.s_gu ? ceil_div(a.Is, G) : 0;
    a.one_items = ns_max + ceil_div((long long)a.k * a.I, G);
    if (a.one_items > 32) return false;  // one mbarrier bit per pair
    const int RS = (int)flint::nvfp4_row_stride(a.H), RSr = (int)flint::nvfp4_row_stride(a.I);
    const int RSs = a.s_gu ? (int)flint::nvfp4_row_stride(a.Is) : 0;
    a.slot = 2 * RS;
    a.rows_max = ceil_div(a.H, G);
    a.one_rsd = RSr > RSs ? RSr : RSs;
    a.Gs = 0;
    a.rows = 0;
    a.one = 1;
    if (flint::layer_smem_bytes(a) + kSmemSlack <= (size_t)smem_optin) return true;
    a.one = 0;
    return false;
}

}  // namespace

extern "C" {

const char* flint_last_error(void) { return g_err; }

const char* flint_status_string(flint_status_t s) {
    switch (s) {
        case FLINT_OK: return "ok";
        case FLINT_ERR_INVALID_ARG: return "invalid argument";
        case FLINT_ERR_UNSUPPORTED: return "unsupported";
        case FLINT_ERR_CUDA: return "CUDA error";
        case FLINT_ERR_TIMEOUT: return "device wait timed out";
    }
    return "unknown status";
}

int64_t flint_nvfp4_row_stride(int64_t cols) { return cols > 0 ? flint::nvfp4_row_stride(cols) : 0; }

int64_t flint_nvfp4_packed_bytes(int64_t n_mats, int64_t rows, int64_t cols) {
    return n_mats * rows * flint_nvfp4_row_stride(cols);
}

int64_t flint_gguf_nvfp4_bytes(int64_t n_mats, int64_t rows, int64_t cols) { return n_mats * rows * (cols / 64) * 36; }

size_t flint_workspace_bytes(int num_experts, int top_k, int hidden, int inter, int inter_shared) {
    if (num_experts < 0 || top_k < 0 || hidden < 0 || inter < 0 || inter_shared < 0) return 0;
    return flint::ws_layout(num_experts, top_k, hidden, inter, inter_shared).total;
}

flint_status_t flint_workspace_init(void* ws, size_t ws_bytes, void* stream) {
    if (!ws || ws_bytes < flint::kWsHeader) return fail(FLINT_ERR_INVALID_ARG, "workspace null or too small");
    cudaError_t e = cudaMemsetAsync(ws, 0, ws_bytes, as_stream(stream));
    return e == cudaSuccess ? FLINT_OK : cuda_fail(e, "cudaMemsetAsync");
}

flint_status_t flint_workspace_check(void* ws, size_t ws_bytes, void* stream) {
    if (!ws || ws_bytes < flint::kWsHeader) return fail(FLINT_ERR_INVALID_ARG, "workspace null or too small");
    uint32_t st = 0;
    cudaError_t e = cudaMemcpyAsync(&st, ws_status(ws), sizeof st, cudaMemcpyDeviceToHost, as_stream(stream));
    if (e == cudaSuccess) e = cudaStreamSynchronize(as_stream(stream));
    if (e != cudaSuccess) return cuda_fail(e, "reading the workspace status");
    if (!st) return FLINT_OK;
    const bool timeout = (st & (flint::kStatusTimeoutRoute | flint::kStatusTimeoutGateUp | flint::kStatusTimeoutDown |
                                flint::kStatusTimeoutSelftest | flint::kStatusTimeoutLayer |
                                flint::kStatusTimeoutPrefill)) != 0;
    // After a timed-out wait (or a fused-layer CTA that stopped) the counters
    // the kernels synchronise on (the router's arrival counter, the fused
    // layer's call counter and arrival counters) may be left mid-call: the
    // whole workspace is re-initialised, as flint_workspace_init does.
    // Otherwise only the status word is cleared.
    const bool reinit = timeout || (st & flint::kStatusLayerPlan) != 0;
    e = cudaMemsetAsync(reinit ? ws : static_cast<void*>(ws_status(ws)), 0, reinit ? ws_bytes : sizeof st,
                        as_stream(stream));
    if (e == cudaSuccess) e = cudaStreamSynchronize(as_stream(stream));
    if (e != cudaSuccess) return cuda_fail(e, "clearing the workspace status");
    if (timeout) return fail(FLINT_ERR_TIMEOUT, "device wait timed out (status 0x%x); workspace re-initialised", st);
    if (st & flint::kStatusLayerPlan)
        return fail(FLINT_ERR_UNSUPPORTED,
                    "a fused-layer CTA's work exceeded its shared-memory plan (status 0x%x); workspace re-initialised",
                    st);
    return fail(FLINT_ERR_INVALID_ARG, "an expert id was outside [0, num_experts) (status 0x%x)", st);
}

flint_status_t flint_nvfp4_repack(const uint8_t* src, int64_t n_mats, int64_t rows, int64_t cols, uint8_t* dst,
                                  int64_t dst_mat_stride, void* stream) {
    if (n_mats < 0 || rows < 0 || cols <= 0 || cols % 64)
        return fail(FLINT_ERR_INVALID_ARG, "repack: bad shape n_mats=%lld rows=%lld cols=%lld (cols %% 64 == 0)",
                    (long long)n_mats, (long long)rows, (long long)cols);
    const int64_t min_stride = rows * flint::nvfp4_row_stride(cols);
    if (dst_mat_stride == 0) dst_mat_stride = min_stride;
    if (dst_mat_stride < min_stride || dst_mat_stride % 16)
        return fail(FLINT_ERR_INVALID_ARG, "repack: dst_mat_stride %lld below %lld or not a multiple of 16",
                    (long long)dst_mat_stride, (long long)min_stride);
    if (n_mats * rows == 0) return FLINT_OK;
    if (!src || !dst || !aligned(src, 16) || !aligned(dst, 16))
        return fail(FLINT_ERR_INVALID_ARG, "repack: null or misaligned pointer");
    DevInfo d;
    flint_status_t s = device_info(d);
    if (s != FLINT_OK) return s;
    cudaError_t e = flint::launch_repack(src, n_mats, rows, cols, dst, dst_mat_stride, as_stream(stream));
    return e == cudaSuccess ? FLINT_OK : cuda_fail(e, "repack launch");
}

flint_status_t flint_nvfp4_unrepack(const uint8_t* dst, int64_t n_mats, int64_t rows, int64_t cols,
                                    int64_t dst_mat_stride, uint8_t* src, void* stream) {
    if (n_mats < 0 || rows < 0 || cols <= 0 || cols % 64)
        return fail(FLINT_ERR_INVALID_ARG, "unrepack: bad shape");
    const int64_t min_stride = rows * flint::nvfp4_row_stride(cols);
    if (dst_mat_stride == 0) dst_mat_stride = min_stride;
    if (dst_mat_stride < min_stride || dst_mat_stride % 16)
        return fail(FLINT_ERR_INVALID_ARG, "unrepack: bad dst_mat_stride");
    if (n_mats * rows == 0) return FLINT_OK;
    if (!src || !dst || !aligned(src, 16) || !aligned(dst, 16))
        return fail(FLINT_ERR_INVALID_ARG, "unrepack: null or misaligned pointer");
    DevInfo d;
    flint_status_t s = device_info(d);
    if (s != FLINT_OK) return s;
    cudaError_t e = flint::launch_unrepack(dst, n_mats, rows, cols, dst_mat_stride, src, as_stream(stream));
    return e == cudaSuccess ? FLINT_OK : cuda_fail(e, "unrepack launch");
}

flint_status_t flint_nvfp4_dequant(const uint8_t* packed, int64_t rows, int64_t cols, float* out, void* stream) {
    if (rows < 0 || cols <= 0 || cols % 64) return fail(FLINT_ERR_INVALID_ARG, "dequant: bad shape");
    if (rows == 0) return FLINT_OK;
    if (!packed || !out || !aligned(packed, 16) || !aligned(out, 16))
        return fail(FLINT_ERR_INVALID_ARG, "dequant: null or misaligned pointer");
    DevInfo d;
    flint_status_t s = device_info(d);
    if (s != FLINT_OK) return s;
    cudaError_t e = flint::launch_dequant(packed, rows, cols, out, as_stream(stream));
    return e == cudaSuccess ? FLINT_OK : cuda_fail(e, "dequant launch");
}

flint_status_t flint_moe_route(const flint_bf16* x, int T, int H, const flint_bf16* router_w, int E,
                               const float* bias, int k, int32_t* ids, float* weights, void* ws, size_t ws_bytes,
                               unsigned flags, void* stream) {
    if (T < 1 || T > FLINT_MAX_TOKENS) return fail(FLINT_ERR_UNSUPPORTED, "route: T=%d outside 1..%d", T, FLINT_MAX_TOKENS);
    if (H <= 0 || H % 256) return fail(FLINT_ERR_UNSUPPORTED, "route: H=%d must be a positive multiple of 256", H);
    if (E < 1 || E > FLINT_MAX_EXPERTS) return fail(FLINT_ERR_UNSUPPORTED, "route: E=%d outside 1..%d", E, FLINT_MAX_EXPERTS);
    if (k < 1 || k > FLINT_MAX_TOPK || k > E) return fail(FLINT_ERR_UNSUPPORTED, "route: k=%d outside 1..min(%d, E)", k, FLINT_MAX_TOPK);
    if (!x || !router_w || !ids || !weights || !aligned(x, 16) || !aligned(router_w, 16) || !aligned(ids, 4) ||
        !aligned(weights, 4) || (bias && !aligned(bias, 4)))
        return fail(FLINT_ERR_INVALID_ARG, "route: null or misaligned pointer");
    flint_status_t s = check_ws(ws, ws_bytes, flint::ws_layout(E, 0, 0, 0, 0).h_routed_off);
    if (s != FLINT_OK) return s;
    DevInfo d;
    if ((s = device_info(d)) != FLINT_OK) return s;
    flint::RouteArgs a = {};
    a.x = x;
    a.T = T;
    a.H = H;
    a.wr = router_w;
    a.E = E;
    a.bias = bias;
    a.k = k;
    a.ids = ids;
    a.weights = weights;
    a.logits = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + flint::kWsHeader);
    a.counter = reinterpret_cast<uint32_t*>(ws);
    a.status = ws_status(ws);
    a.rows_per_cta = ceil_div(E, d.sm_count);
    const size_t smem = flint::route_smem_bytes(a);
    if (smem + 1024 > (size_t)d.smem_optin || (size_t)a.rows_per_cta * H * 2 >= (1u << 20))
        return fail(FLINT_ERR_UNSUPPORTED, "route: H=%d too large for one CTA's shared memory", H);
    cudaError_t e = flint::launch_route(a, d, (flags & FLINT_PDL) != 0, as_stream(stream));
    return e == cudaSuccess ? FLINT_OK : cuda_fail(e, "route launch");
}

static flint_status_t moe_common(const char* what, int T, int k, const flint_experts* routed,
                                 const flint_experts* shared, bool need_down) {
    if (T < 1 || T > FLINT_MAX_TOKENS) return fail(FLINT_ERR_UNSUPPORTED, "%s: T=%d outside 1..%d", what, T, FLINT_MAX_TOKENS);
    flint_status_t s = check_experts(routed, "routed", need_down);
    if (s != FLINT_OK) return s;
    if (k < 1 || k > FLINT_MAX_TOPK || k > routed->num_experts)
        return fail(FLINT_ERR_UNSUPPORTED, "%s: k=%d outside 1..min(%d, E)", what, k, FLINT_MAX_TOPK);
    if (shared) {
        if ((s = check_experts(shared, "shared", need_down)) != FLINT_OK) return s;
        if (shared->num_experts != 1 || shared->hidden != routed->hidden)
            return fail(FLINT_ERR_INVALID_ARG, "%s: shared expert must have num_experts 1 and the routed hidden size", what);
        if (shared->dtype != routed->dtype)
            return fail(FLINT_ERR_UNSUPPORTED, "%s: shared and routed experts must have the same dtype", what);
    }
    return FLINT_OK;
}

flint_status_t flint_moe_gate_up(const flint_bf16* x, int T, const int32_t* ids, int k, const flint_experts* routed,
                                 const flint_experts* shared, void* ws, size_t ws_bytes, unsigned flags,
                                 void* stream) {
    flint_status_t s = moe_common("gate_up", T, k, routed, shared, false);
    if (s != FLINT_OK) return s;
    if (!x || !ids || !aligned(x, 16) || !aligned(ids, 4))
        return fail(FLINT_ERR_INVALID_ARG, "gate_up: null or misaligned x/ids");
    const int Is = shared ? shared->inter : 0;
    const flint::WsLayout L = flint::ws_layout(routed->num_experts, k, 0, routed->inter, Is);
    if ((s = check_ws(ws, ws_bytes, L.d_routed_off)) != FLINT_OK) return s;
    DevInfo d;
    if ((s = device_info(d)) != FLINT_OK) return s;
    flint::GateUpArgs a = {};
    a.x = x;
    a.T = T;
    a.H = routed->hidden;
    a.ids = ids;
    a.k = k;
    a.gu = static_cast<const uint8_t*>(routed->gate_up);
    a.E = routed->num_experts;
    a.I = routed->inter;
    a.ts = routed->tensor_scale;
    a.s_gu = shared ? static_cast<const uint8_t*>(shared->gate_up) : nullptr;
    a.Is = Is;
    a.s_ts = shared ? shared->tensor_scale : nullptr;
    a.h_routed = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(ws) + L.h_routed_off);
    a.h_shared = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(ws) + L.h_shared_off);
    a.status = ws_status(ws);
    a.x_early = (flags & FLINT_PDL) && (flags & FLINT_PDL_AFTER_ROUTE);
    if (routed->dtype == FLINT_DTYPE_BF16) {
        const long long pairs = ceil_div(a.Is, d.sm_count) +
                                ceil_div((long long)(T * k < a.E ? T * k : a.E) * a.I, d.sm_count);
        if (!gate_up_bf16_shape(a, d.smem_optin, pairs))
            return fail(FLINT_ERR_UNSUPPORTED, "gate_up: shapes exceed one CTA's shared memory");
        cudaError_t e = flint::launch_gate_up_bf16(a, d, (flags & FLINT_PDL) != 0, as_stream(stream));
        return e == cudaSuccess ? FLINT_OK : cuda_fail(e, "gate_up (bf16) launch");
    }
    const long long routed_pairs = (long long)(T * k < a.E ? T * k : a.E) * a.I;
    if (!gate_up_shape(a, true, d.smem_optin,
                       ceil_div(a.Is, d.sm_count) + ceil_div(routed_pairs, d.sm_count)))
        return fail(FLINT_ERR_UNSUPPORTED, "gate_up: shapes exceed one CTA's shared memory");
    cudaError_t e = flint::launch_gate_up(a, true, d, (flags & FLINT_PDL) != 0, as_stream(stream));
    return e == cudaSuccess ? FLINT_OK : cuda_fail(e, "gate_up launch");
}

flint_status_t flint_moe_down_combine(int T, const int32_t* ids, const float* weights, int k,
                                      const flint_experts* routed, const flint_experts* shared, flint_bf16* y,
                                      void* ws, size_t ws_bytes, unsigned flags, void* stream) {
    flint_status_t s = moe_common("down_combine", T, k, routed, shared, true);
    if (s != FLINT_OK) return s;
    if (!ids || !weights || !y || !aligned(ids, 4) || !aligned(weights, 4) || !aligned(y, 16))
        return fail(FLINT_ERR_INVALID_ARG, "down_combine: null or misaligned ids/weights/y");
    const int Is = shared ? shared->inter : 0;
    const flint::WsLayout L = flint::ws_layout(routed->num_experts, k, 0, routed->inter, Is);
    if ((s = check_ws(ws, ws_bytes, L.d_routed_off)) != FLINT_OK) return s;
    DevInfo d;
    if ((s = device_info(d)) != FLINT_OK) return s;
    flint::DownArgs a = {};
    a.ids = ids;
    a.w = weights;
    a.T = T;
    a.k = k;
    a.H = routed->hidden;
    a.down = static_cast<const uint8_t*>(routed->down);
    a.E = routed->num_experts;
    a.I = routed->inter;
    a.ts = routed->tensor_scale;
    a.s_down = shared ? static_cast<const uint8_t*>(shared->down) : nullptr;
    a.Is = Is;
    a.s_ts = shared ? shared->tensor_scale : nullptr;
    a.h_routed = reinterpret_cast<const uint16_t*>(static_cast<uint8_t*>(ws) + L.h_routed_off);
    a.h_shared = reinterpret_cast<const uint16_t*>(static_cast<uint8_t*>(ws) + L.h_shared_off);
    a.y = y;
    a.status = ws_status(ws);
    if (routed->dtype == FLINT_DTYPE_BF16) {
        if (!down_bf16_shape(a, d.sm_count, d.smem_optin))
            return fail(FLINT_ERR_UNSUPPORTED, "down_combine: shapes exceed one CTA's shared memory");
        cudaError_t e = flint::launch_down_bf16(a, d, (flags & FLINT_PDL) != 0, as_stream(stream));
        return e == cudaSuccess ? FLINT_OK : cuda_fail(e, "down_combine (bf16) launch");
    }
    if (!down_shape(a, d.sm_count, d.smem_optin))
        return fail(FLINT_ERR_UNSUPPORTED, "down_combine: shapes exceed one CTA's shared memory");
    cudaError_t e = flint::launch_down(a, d, (flags & FLINT_PDL) != 0, as_stream(stream));
    return e == cudaSuccess ? FLINT_OK : cuda_fail(e, "down_combine launch");
}

static flint_status_t moe_layer_impl(const char* what, const flint_bf16* x, const flint_norm* norm, int T,
                                     const flint_bf16* router_w, int E, const float* bias, int k,
                                     const flint_experts* routed, const flint_experts* shared, int32_t* ids,
                                     float* weights, flint_bf16* y, void* ws, size_t ws_bytes,
                                     const flint_l2_prefetch* next, unsigned flags, void* stream,
                                     bool given = false, bool* no_fit = nullptr);

flint_status_t flint_moe_decode(const flint_bf16* x, int T, const int32_t* ids, const float* weights, int k,
                                const flint_experts* routed, const flint_experts* shared, flint_bf16* y, void* ws,
                                size_t ws_bytes, unsigned flags, void* stream) {
    flint_status_t s = moe_common("decode", T, k, routed, shared, true);
    if (s != FLINT_OK) return s;
    if (!weights || !y || !aligned(weights, 4) || !aligned(y, 16))
        return fail(FLINT_ERR_INVALID_ARG, "decode: null or misaligned weights/y");
    if (routed->dtype == FLINT_DTYPE_NVFP4) {
        // one cooperative launch (the fused layer with the routing given) when
        // the workspace holds the fused layer's regions and the shapes fit
        const int Is = shared ? shared->inter : 0;
        const flint::WsLayout W = flint::ws_layout(routed->num_experts, k, routed->hidden, routed->inter, Is);
        if (ws && ws_bytes >= W.total) {
            bool no_fit = false;
            s = moe_layer_impl("decode", x, nullptr, T, nullptr, routed->num_experts, nullptr, k, routed, shared,
                               const_cast<int32_t*>(ids), const_cast<float*>(weights), y, ws, ws_bytes, nullptr, flags,
                               stream, true, &no_fit);
            if (!no_fit) return s;
        }
    }
    s = flint_moe_gate_up(x, T, ids, k, routed, shared, ws, ws_bytes, flags, stream);
    if (s != FLINT_OK) return s;
    return flint_moe_down_combine(T, ids, weights, k, routed, shared, y, ws, ws_bytes, flags, stream);
}

// Validates a flint_norm for T tokens of H values and fills the kernel's view.
static flint_status_t norm_args(const char* what, const flint_norm* n, int T, int H, bool need_x,
                                flint::NormArgs& a) {
    if (!n) return fail(FLINT_ERR_INVALID_ARG, "%s: norm is null", what);
    if (H <= 0 || H % 256 || H > 32768)
        return fail(FLINT_ERR_UNSUPPORTED, "%s: H=%d must be a multiple of 256 up to 32768", what, H);
    if (!(n->eps >= 0.f)) return fail(FLINT_ERR_INVALID_ARG, "%s: eps must be >= 0", what);
    if (!n->residual || !aligned(n->residual, 16) || (n->y && !aligned(n->y, 16)) ||
        (n->gamma && !aligned(n->gamma, 16)) || (n->residual_out && !aligned(n->residual_out, 16)) ||
        (n->x_out && !aligned(n->x_out, 16)) || (need_x && !n->x_out))
        return fail(FLINT_ERR_INVALID_ARG, "%s: null or misaligned norm pointer", what);
    const size_t bytes = (size_t)T * H * 2;
    auto overlap = [bytes](const void* p, const void* q) {
        if (!p || !q) return false;
        const uint8_t *a = static_cast<const uint8_t*>(p), *b = static_cast<const uint8_t*>(q);
        return a < b + bytes && b < a + bytes;
    };
    if (overlap(n->residual_out, n->residual) || overlap(n->residual_out, n->y))
        return fail(FLINT_ERR_INVALID_ARG, "%s: residual_out overlaps residual or y", what);
    a = {};
    a.r = n->residual;
    a.y = n->y;
    a.gamma = n->gamma;
    a.eps = n->eps;
    a.r_out = n->residual_out;
    a.x_out = n->x_out;
    a.T = T;
    a.H = H;
    return FLINT_OK;
}

flint_status_t flint_residual_rmsnorm(const flint_norm* norm, int T, int H, unsigned flags, void* stream) {
    if (T < 1 || T > FLINT_MAX_TOKENS) return fail(FLINT_ERR_UNSUPPORTED, "rmsnorm: T=%d outside 1..%d", T, FLINT_MAX_TOKENS);
    flint::NormArgs a;
    flint_status_t s = norm_args("rmsnorm", norm, T, H, true, a);
    if (s != FLINT_OK) return s;
    DevInfo d;
    if ((s = device_info(d)) != FLINT_OK) return s;
    cudaError_t e = flint::launch_rmsnorm(a, (flags & FLINT_PDL) != 0, as_stream(stream));
    return e == cudaSuccess ? FLINT_OK : cuda_fail(e, "rmsnorm launch");
}

// The fused layer launch. given: ids and weights are the caller's routing
// (flint_moe_decode; no router, norm or prefetch); *no_fit (when not null) is
// set where the shapes exceed one CTA's shared memory, before anything runs.
static flint_status_t moe_layer_impl(const char* what, const flint_bf16* x, const flint_norm* norm, int T,
                                     const flint_bf16* router_w, int E, const float* bias, int k,
                                     const flint_experts* routed, const flint_experts* shared, int32_t* ids,
                                     float* weights, flint_bf16* y, void* ws, size_t ws_bytes,
                                     const flint_l2_prefetch* next, unsigned flags, void* stream,
                                     bool given, bool* no_fit) {
    if (no_fit) *no_fit = false;
    flint_status_t s = moe_common(what, T, k, routed, shared, true);
    if (s != FLINT_OK) return s;
    unsigned long long pf_granules = 0;
    if (next) {
        for (int r = 0; r < 4; ++r) {
            if (next->bytes[r] == 0) continue;
            if (!next->ptr[r] || !aligned(next->ptr[r], 16) || next->bytes[r] % 16)
                return fail(FLINT_ERR_INVALID_ARG, "%s: prefetch range %d misaligned (16-byte start and size)", what, r);
            pf_granules += next->bytes[r] / 16;
        }
        if (pf_granules >= (1ull << 28))
            return fail(FLINT_ERR_INVALID_ARG, "%s: prefetch ranges sum to 4 GiB or more", what);
    }
    flint::NormArgs na = {};
    if (norm) {
        if ((s = norm_args(what, norm, T, routed->hidden, false, na)) != FLINT_OK) return s;
        const size_t bytes = (size_t)T * routed->hidden * 2;
        for (const void* p : {static_cast<const void*>(norm->residual), static_cast<const void*>(norm->y),
                              static_cast<const void*>(norm->residual_out), static_cast<const void*>(norm->x_out)}) {
            const uint8_t *a = static_cast<const uint8_t*>(p), *b = reinterpret_cast<const uint8_t*>(y);
            if (p && y && a < b + bytes && b < a + bytes)
                return fail(FLINT_ERR_INVALID_ARG, "%s: y overlaps a buffer of the norm", what);
        }
        x = norm->residual;  // checked below like x; the kernel reads the norm's buffers
    }
    if (E != routed->num_experts)
        return fail(FLINT_ERR_INVALID_ARG, "%s: router has %d rows, routed experts %d", what, E, routed->num_experts);
    if (routed->dtype != FLINT_DTYPE_NVFP4)
        return fail(FLINT_ERR_UNSUPPORTED,
                    "%s: the one-kernel layer takes NVFP4 experts; run BF16 experts with flint_moe_route + "
                    "flint_moe_decode", what);
    if (!x || (!given && !router_w) || !ids || !weights || !y || !aligned(x, 16) || !aligned(router_w, 16) ||
        !aligned(ids, 4) || !aligned(weights, 4) || !aligned(y, 16) || (bias && !aligned(bias, 4)))
        return fail(FLINT_ERR_INVALID_ARG, "%s: null or misaligned pointer", what);
    const int Is = shared ? shared->inter : 0;
    const int H = routed->hidden;
    if (H > flint::kLayerMaxHidden) {
        if (no_fit) *no_fit = true;
        return fail(FLINT_ERR_UNSUPPORTED, "%s: hidden %d above %d", what, H, flint::kLayerMaxHidden);
    }
    const flint::WsLayout W = flint::ws_layout(E, k, H, routed->inter, Is);
    if ((s = check_ws(ws, ws_bytes, W.total)) != FLINT_OK) return s;
    DevInfo d;
    if ((s = device_info(d)) != FLINT_OK) return s;
    uint8_t* wb = static_cast<uint8_t*>(ws);
    flint::LayerArgs a = {};
    a.x = x;
    a.T = T;
    a.H = H;
    a.wr = router_w;
    a.E = E;
    a.bias = bias;
    a.k = k;
    a.ids = ids;
    a.weights = weights;
    a.hdr = reinterpret_cast<uint32_t*>(ws);
    a.status = ws_status(ws);
    a.scores = reinterpret_cast<uint32_t*>(wb + W.logits_off);
    a.h_routed = reinterpret_cast<uint16_t*>(wb + W.h_routed_off);
    a.h_shared = reinterpret_cast<uint16_t*>(wb + W.h_shared_off);
    a.d_routed = reinterpret_cast<uint16_t*>(wb + W.d_routed_off);
    a.d_shared = reinterpret_cast<uint16_t*>(wb + W.d_shared_off);
    a.counters = reinterpret_cast<uint32_t*>(wb + W.counters_off);
    a.unit_counters = reinterpret_cast<uint32_t*>(wb + W.unit_counters_off);
    a.gu = static_cast<const uint8_t*>(routed->gate_up);
    a.down = static_cast<const uint8_t*>(routed->down);
    a.I = routed->inter;
    a.ts = routed->tensor_scale;
    a.s_gu = shared ? static_cast<const uint8_t*>(shared->gate_up) : nullptr;
    a.s_down = shared ? static_cast<const uint8_t*>(shared->down) : nullptr;
    a.Is = Is;
    a.s_ts = shared ? shared->tensor_scale : nullptr;
    a.y = y;
    a.norm = na;
    for (int r = 0; r < 4; ++r) {
        a.pf_ptr[r] = next && next->bytes[r] ? static_cast<const uint8_t*>(next->ptr[r]) : nullptr;
        a.pf_bytes[r] = next && next->bytes[r] ? (unsigned long long)next->bytes[r] : 0ull;
    }
    a.pf_granules = pf_granules;
    a.given = given ? 1 : 0;
    a.x_early = given && (flags & FLINT_PDL) && (flags & FLINT_PDL_AFTER_ROUTE) ? 1 : 0;
    if (!one_shape(a, d.sm_count, d.smem_optin) && !layer_shape(a, d.sm_count, d.smem_optin)) {
        if (no_fit) *no_fit = true;
        return fail(FLINT_ERR_UNSUPPORTED, "%s: shapes exceed one CTA's shared memory", what);
    }
    cudaError_t e = flint::launch_layer(a, d, (flags & FLINT_PDL) != 0, as_stream(stream));
    return e == cudaSuccess ? FLINT_OK : cuda_fail(e, "layer launch");
}

flint_status_t flint_moe_layer(const flint_bf16* x, int T, const flint_bf16* router_w, int E, const float* bias, int k,
                               const flint_experts* routed, const flint_experts* shared, int32_t* ids, float* weights,
                               flint_bf16* y, void* ws, size_t ws_bytes, const flint_l2_prefetch* next,
                               unsigned flags, void* stream) {
    return moe_layer_impl("layer", x, nullptr, T, router_w, E, bias, k, routed, shared, ids, weights, y, ws, ws_bytes,
                          next, flags, stream);
}

flint_status_t flint_moe_block(const flint_norm* norm, int T, const flint_bf16* router_w, int E, const float* bias,
                               int k, const flint_experts* routed, const flint_experts* shared, int32_t* ids,
                               float* weights, flint_bf16* y, void* ws, size_t ws_bytes,
                               const flint_l2_prefetch* next, unsigned flags, void* stream) {
    if (!norm) return fail(FLINT_ERR_INVALID_ARG, "block: norm is null");
    return moe_layer_impl("block", nullptr, norm, T, router_w, E, bias, k, routed, shared, ids, weights, y, ws,
                          ws_bytes, next, flags, stream);
}

size_t flint_prefill_workspace_bytes(int tokens, int num_experts, int top_k, int hidden, int inter, int inter_shared) {
    if (tokens < 0 || num_experts < 0 || top_k < 0 || hidden < 0 || inter < 0 || inter_shared < 0) return 0;
    return flint::prefill_ws_layout(tokens, num_experts, top_k, hidden, inter, inter_shared).total;
}

flint_status_t flint_moe_prefill(const flint_bf16* x, int T, const flint_bf16* router_w, int E, const float* bias,
                                 int k, const flint_experts* routed, const flint_experts* shared, int32_t* ids,
                                 float* weights, flint_bf16* y, void* ws, size_t ws_bytes, unsigned flags,
                                 void* stream) {
    (void)flags;
    if (T < 1) return fail(FLINT_ERR_INVALID_ARG, "prefill: T=%d", T);
    flint_status_t s = check_experts(routed, "routed", true);
    if (s != FLINT_OK) return s;
    if (shared && (s = check_experts(shared, "shared", true)) != FLINT_OK) return s;
    if (routed->dtype != FLINT_DTYPE_NVFP4 || (shared && shared->dtype != FLINT_DTYPE_NVFP4))
        return fail(FLINT_ERR_UNSUPPORTED, "prefill: NVFP4 experts only");
    if (shared && (shared->num_experts != 1 || shared->hidden != routed->hidden))
        return fail(FLINT_ERR_INVALID_ARG, "prefill: shared expert must have num_experts 1 and the routed hidden size");
    if (E != routed->num_experts)
        return fail(FLINT_ERR_INVALID_ARG, "prefill: router has %d rows, routed experts %d", E, routed->num_experts);
    if (E % 16 || E > FLINT_MAX_EXPERTS)
        return fail(FLINT_ERR_UNSUPPORTED, "prefill: E=%d must be a multiple of 16 up to %d", E, FLINT_MAX_EXPERTS);
    if (k < 1 || k > FLINT_MAX_TOPK || k > E) return fail(FLINT_ERR_UNSUPPORTED, "prefill: k=%d", k);
    if ((long long)T * k >= (1ll << 30)) return fail(FLINT_ERR_UNSUPPORTED, "prefill: T*k too large");
    if (!x || !router_w || !ids || !weights || !y || !aligned(x, 16) || !aligned(router_w, 16) || !aligned(ids, 4) ||
        !aligned(weights, 4) || !aligned(y, 16) || (bias && !aligned(bias, 4)))
        return fail(FLINT_ERR_INVALID_ARG, "prefill: null or misaligned pointer");
    const int H = routed->hidden, I = routed->inter, Is = shared ? shared->inter : 0;
    if ((s = check_ws(ws, ws_bytes, flint::prefill_ws_layout(T, E, k, H, I, Is).total)) != FLINT_OK) return s;
    DevInfo d;
    if ((s = device_info(d)) != FLINT_OK) return s;
    flint::PrefillArgs p = {};
    p.x = x;
    p.T = T;
    p.H = H;
    p.router_w = router_w;
    p.E = E;
    p.bias = bias;
    p.k = k;
    p.gu = static_cast<const uint8_t*>(routed->gate_up);
    p.down = static_cast<const uint8_t*>(routed->down);
    p.I = I;
    p.ts = routed->tensor_scale;
    p.s_gu = shared ? static_cast<const uint8_t*>(shared->gate_up) : nullptr;
    p.s_down = shared ? static_cast<const uint8_t*>(shared->down) : nullptr;
    p.Is = Is;
    p.s_ts = shared ? shared->tensor_scale : nullptr;
    p.ids = ids;
    p.weights = weights;
    p.y = y;
    p.ws = ws;
    cudaError_t e = flint::launch_prefill(p, d, as_stream(stream));
    return e == cudaSuccess ? FLINT_OK : cuda_fail(e, "prefill launch");
}

flint_status_t flint_dense_gemv(const flint_bf16* x, int T, const flint_packed* W, int epilogue, flint_bf16* y,
                                void* ws, size_t ws_bytes, unsigned flags, void* stream) {
    if (T < 1 || T > FLINT_MAX_TOKENS) return fail(FLINT_ERR_UNSUPPORTED, "dense_gemv: T=%d outside 1..%d", T, FLINT_MAX_TOKENS);
    if (!W) return fail(FLINT_ERR_INVALID_ARG, "dense_gemv: W is null");
    if (W->dtype != FLINT_DTYPE_NVFP4) return fail(FLINT_ERR_UNSUPPORTED, "dense_gemv: only NVFP4 weights");
    const int N = W->rows, K = W->cols;
    if (epilogue != FLINT_EPILOGUE_NONE && epilogue != FLINT_EPILOGUE_SWIGLU)
        return fail(FLINT_ERR_INVALID_ARG, "dense_gemv: unknown epilogue %d", epilogue);
    if (N < 1 || K < 1024 || K % 1024)
        return fail(FLINT_ERR_UNSUPPORTED, "dense_gemv: N=%d, K=%d (K %% 1024 == 0)", N, K);
    if (epilogue == FLINT_EPILOGUE_SWIGLU && N % 2) return fail(FLINT_ERR_UNSUPPORTED, "dense_gemv: SwiGLU needs even N");
    if (!x || !y || !W->data || !W->tensor_scale || !aligned(x, 16) || !aligned(y, 16) || !aligned(W->data, 16) ||
        !aligned(W->tensor_scale, 4))
        return fail(FLINT_ERR_INVALID_ARG, "dense_gemv: null or misaligned pointer");
    if (ws && (ws_bytes < flint::kWsHeader || !aligned(ws, 256)))
        return fail(FLINT_ERR_INVALID_ARG, "dense_gemv: workspace too small or misaligned");
    DevInfo d;
    flint_status_t s = device_info(d);
    if (s != FLINT_OK) return s;
    uint32_t* status = ws ? ws_status(ws) : nullptr;
    const bool pdl = (flags & FLINT_PDL) != 0;
    const bool pair = epilogue == FLINT_EPILOGUE_SWIGLU;
    const int n_out = pair ? N / 2 : N;
    flint::GateUpArgs a = {};
    a.H = K;
    a.s_gu = static_cast<const uint8_t*>(W->data);
    a.Is = n_out;
    a.s_ts = W->tensor_scale;
    a.status = status;
    // Tokens go in groups small enough that their FP32 copy fits beside the ring.
    const int items = ceil_div(n_out, d.sm_count);
    int tg = T;
    for (; tg >= 1; --tg) {
        a.T = tg;
        if (gate_up_shape(a, pair, d.smem_optin, items)) break;
    }
    if (tg < 1) return fail(FLINT_ERR_UNSUPPORTED, "dense_gemv: K=%d exceeds one CTA's shared memory", K);
    cudaError_t e = cudaSuccess;
    for (int t0 = 0; t0 < T && e == cudaSuccess; t0 += tg) {
        a.T = T - t0 < tg ? T - t0 : tg;
        a.x = x + (size_t)t0 * K;
        a.h_shared = y + (size_t)t0 * n_out;
        if (!gate_up_shape(a, pair, d.smem_optin, items))
            return fail(FLINT_ERR_UNSUPPORTED, "dense_gemv: K=%d exceeds one CTA's shared memory", K);
        e = flint::launch_gate_up(a, pair, d, pdl, as_stream(stream));
    }
    return e == cudaSuccess ? FLINT_OK : cuda_fail(e, "dense_gemv launch");
}

flint_status_t flint_selftest_wait_timeout(void* ws, size_t ws_bytes, uint64_t budget_ns, void* stream) {
    flint_status_t s = check_ws(ws, ws_bytes, flint::kWsHeader);
    if (s != FLINT_OK) return s;
    DevInfo d;
    if ((s = device_info(d)) != FLINT_OK) return s;
    cudaError_t e = flint::launch_selftest_wait(ws_status(ws), budget_ns, as_stream(stream));
    return e == cudaSuccess ? FLINT_OK : cuda_fail(e, "selftest launch");
}

// Writes one header word of the workspace (stream-ordered; the source is
// copied before the call returns).
static flint_status_t set_header_word(void* ws, size_t ws_bytes, int word, uint32_t v, void* stream,
                                      const char* what) {
    flint_status_t s = check_ws(ws, ws_bytes, flint::kWsHeader);
    if (s != FLINT_OK) return s;
    cudaError_t e = cudaMemcpyAsync(static_cast<uint32_t*>(ws) + word, &v, sizeof v, cudaMemcpyHostToDevice,
                                    as_stream(stream));
    if (e == cudaSuccess) e = cudaStreamSynchronize(as_stream(stream));
    return e == cudaSuccess ? FLINT_OK : cuda_fail(e, what);
}

flint_status_t flint_workspace_set_wait_budget(void* ws, size_t ws_bytes, uint32_t budget_us, void* stream) {
    return set_header_word(ws, ws_bytes, flint::kHdrBudget, budget_us, stream, "setting the wait budget");
}

flint_status_t flint_selftest_lose_cta(void* ws, size_t ws_bytes, int cta, void* stream) {
    if (cta < 0) return fail(FLINT_ERR_INVALID_ARG, "selftest_lose_cta: cta %d", cta);
    return set_header_word(ws, ws_bytes, flint::kHdrLoseCta, (uint32_t)cta + 1u, stream, "setting the test hook");
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Router without a caller-provided workspace.
//
// Its scratch (the router's arrival counter and status word, then FP32 logits
// for up to FLINT_MAX_TOKENS tokens x FLINT_MAX_EXPERTS experts) lives in the
// array below, which every device that loads this library keeps until the
// process exits. Host code cannot use the array's name as a device address:
// the address comes from cudaGetSymbolAddress, once per device.
// ---------------------------------------------------------------------------
constexpr size_t kRouteStaticScratchBytes =
    flint::kWsHeader + sizeof(float) * FLINT_MAX_TOKENS * FLINT_MAX_EXPERTS;  // 33,024 bytes
static __device__ __align__(256) unsigned char g_route_static_scratch[kRouteStaticScratchBytes];

namespace {

// Device address of the scratch array on the current device (looked up on
// the first call on each device, with that device current).
flint_status_t route_static_scratch(const DevInfo& d, void** out) {
    static std::mutex mu;
    static void* addr[64] = {};
    std::lock_guard<std::mutex> lock(mu);
    if (d.device < 0 || d.device >= 64) return fail(FLINT_ERR_UNSUPPORTED, "device index %d above 63", d.device);
    if (!addr[d.device]) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_route_static_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress of the router scratch");
        addr[d.device] = p;
    }
    *out = addr[d.device];
    return FLINT_OK;
}

}  // namespace

extern "C" flint_status_t flint_moe_route_static(const flint_bf16* x, int T, int H, const flint_bf16* router_w, int E,
                                                 const float* bias, int k, int32_t* ids, float* weights,
                                                 unsigned flags, void* stream) {
    if (T < 1 || T > FLINT_MAX_TOKENS)
        return fail(FLINT_ERR_UNSUPPORTED, "route_static: T=%d outside 1..%d", T, FLINT_MAX_TOKENS);
    if (H <= 0 || H % 256) return fail(FLINT_ERR_UNSUPPORTED, "route_static: H=%d must be a positive multiple of 256", H);
    if (E < 1) return fail(FLINT_ERR_INVALID_ARG, "route_static: E=%d", E);
    // The selection keeps at most FLINT_MAX_EXPERTS scores per token, whatever
    // the scratch could hold.
    if (E > FLINT_MAX_EXPERTS)
        return fail(FLINT_ERR_UNSUPPORTED, "route_static: E=%d above the router's limit of %d experts", E,
                    FLINT_MAX_EXPERTS);
    if (flint::kWsHeader + sizeof(float) * (size_t)T * (size_t)E > kRouteStaticScratchBytes) {
        const int by_scratch = (int)((kRouteStaticScratchBytes - flint::kWsHeader) / sizeof(float) / T);
        return fail(FLINT_ERR_UNSUPPORTED,
                    "route_static: %d tokens x %d experts need %zu bytes of scratch; the static scratch holds %zu "
                    "(at most %d experts for %d tokens)",
                    T, E, flint::kWsHeader + sizeof(float) * (size_t)T * (size_t)E, kRouteStaticScratchBytes,
                    by_scratch < FLINT_MAX_EXPERTS ? by_scratch : FLINT_MAX_EXPERTS, T);
    }
    if (k < 1 || k > FLINT_MAX_TOPK || k > E)
        return fail(FLINT_ERR_UNSUPPORTED, "route_static: k=%d outside 1..min(%d, E)", k, FLINT_MAX_TOPK);
    if (!x || !router_w || !ids || !weights || !aligned(x, 16) || !aligned(router_w, 16) || !aligned(ids, 4) ||
        !aligned(weights, 4) || (bias && !aligned(bias, 4)))
        return fail(FLINT_ERR_INVALID_ARG, "route_static: null or misaligned pointer");
    DevInfo d;
    flint_status_t s = device_info(d);
    if (s != FLINT_OK) return s;
    void* scratch = nullptr;
    if ((s = route_static_scratch(d, &scratch)) != FLINT_OK) return s;
    // The counter must start at zero; the array keeps whatever the last call left.
    cudaError_t e = cudaMemsetAsync(scratch, 0, flint::kWsHeader, as_stream(stream));
    if (e != cudaSuccess) return cuda_fail(e, "route_static: clearing the scratch header");
    flint::RouteArgs a = {};
    a.x = x;
    a.T = T;
    a.H = H;
    a.wr = router_w;
    a.E = E;
    a.bias = bias;
    a.k = k;
    a.ids = ids;
    a.weights = weights;
    a.logits = reinterpret_cast<float*>(static_cast<uint8_t*>(scratch) + flint::kWsHeader);
    a.counter = reinterpret_cast<uint32_t*>(scratch);
    a.status = ws_status(scratch);
    a.rows_per_cta = ceil_div(E, d.sm_count);
    const size_t smem = flint::route_smem_bytes(a);
    if (smem + 1024 > (size_t)d.smem_optin || (size_t)a.rows_per_cta * H * 2 >= (1u << 20))
        return fail(FLINT_ERR_UNSUPPORTED, "route_static: H=%d too large for one CTA's shared memory", H);
    e = flint::launch_route(a, d, (flags & FLINT_PDL) != 0, as_stream(stream));
    return e == cudaSuccess ? FLINT_OK : cuda_fail(e, "route_static launch");
}
