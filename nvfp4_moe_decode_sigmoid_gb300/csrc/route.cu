// route.cu -- router GEMV + sigmoid top-k + renormalisation, one kernel.
//
// "Day-0 Support for Flint on vLLM", section "Model architecture": 256 experts,
// sigmoid top-6; section "Optimizations": the router GEMV is a small-batch
// kernel and routing is fused into the neighbouring GEMV. "vLLM 宣布首日支持
// Recursive 的 Flint ...", section "Flint 是什么": 256 routed experts with
// sigmoid top-6 activation.
//
// Each CTA owns `rows_per_cta` router rows. Before waiting on the previous
// kernel (PDL) it bulk-copies those rows (bf16, static weights) into shared
// memory; after the wait it reads x and computes FP32 logits for all T
// tokens. The last CTA to arrive (atomic ticket) selects the top-k per token,
// one warp per token, and leaves the ticket counter at zero.
#include <cfloat>

#include "flint_device.cuh"

namespace flint {
namespace {

constexpr int kMaxLanesSlots = FLINT_MAX_EXPERTS / 32;  // experts per lane in the top-k warp

__global__ void __launch_bounds__(kThreads, 1) route_kernel(const RouteArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
    float* partial = reinterpret_cast<float*>(smem + 128);  // [kWarps][T][rpc]
    const int rpc = a.rows_per_cta;
    uint16_t* wrows = reinterpret_cast<uint16_t*>(smem + 128 + align_up(sizeof(float) * kWarps * FLINT_MAX_TOKENS * rpc, 128));
    __shared__ int is_last;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r0 = blockIdx.x * rpc;
    const int nrows = min(rpc, a.E - r0);
    const int H = a.H, T = a.T;

    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {
        const uint32_t bytes = (uint32_t)(nrows * H * 2);
        mbar_arrive_expect_tx(bar, bytes);
        bulk_g2s(wrows, a.wr + (size_t)r0 * H, bytes, bar);
    }
    // The gate/up kernel only prefetches static weights before its own wait.
    pdl_launch_dependents();
    pdl_wait();  // x may come from the previous kernel

    const bool ok = mbar_wait_bounded(bar, 0, tid == 0 ? a.status : nullptr, kStatusTimeoutRoute);
    if (!__syncthreads_and(ok)) return;

    // Partial dot products: thread tid covers 8-element chunks tid, tid+256, ...
    float acc[FLINT_MAX_TOKENS][2];
#pragma unroll
    for (int t = 0; t < FLINT_MAX_TOKENS; ++t) acc[t][0] = acc[t][1] = 0.f;
    const int nchunk = H / 8;
    for (int rb = 0; rb < nrows; rb += 2) {  // two router rows at a time
        const bool two = rb + 1 < nrows;
        for (int c = tid; c < nchunk; c += kThreads) {
            const uint4 w0 = reinterpret_cast<const uint4*>(wrows + (size_t)rb * H)[c];
            const uint4 w1 = two ? reinterpret_cast<const uint4*>(wrows + (size_t)(rb + 1) * H)[c] : make_uint4(0, 0, 0, 0);
            const uint32_t wa[4] = {w0.x, w0.y, w0.z, w0.w}, wb[4] = {w1.x, w1.y, w1.z, w1.w};
#pragma unroll
            for (int t = 0; t < FLINT_MAX_TOKENS; ++t) {
                if (t < T) {
                    const uint4 xv = ld_cg(reinterpret_cast<const uint4*>(a.x + (size_t)t * H) + c);
                    const uint32_t xa[4] = {xv.x, xv.y, xv.z, xv.w};
                    float s0 = acc[t][0], s1 = acc[t][1];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float x0 = bf16_lo(xa[i]), x1 = bf16_hi(xa[i]);
                        s0 = fmaf(bf16_lo(wa[i]), x0, s0);
                        s0 = fmaf(bf16_hi(wa[i]), x1, s0);
                        s1 = fmaf(bf16_lo(wb[i]), x0, s1);
                        s1 = fmaf(bf16_hi(wb[i]), x1, s1);
                    }
                    acc[t][0] = s0;
                    acc[t][1] = s1;
                }
            }
        }
        // reduce over the block: warp shuffle, then fixed-order sum over warps
#pragma unroll
        for (int t = 0; t < FLINT_MAX_TOKENS; ++t) {
            if (t < T) {
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    float v = acc[t][q];
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
                    if (lane == 0 && rb + q < nrows) partial[(warp * FLINT_MAX_TOKENS + t) * rpc + rb + q] = v;
                    acc[t][q] = 0.f;
                }
            }
        }
    }
    __syncthreads();
    for (int i = tid; i < T * nrows; i += kThreads) {
        const int t = i / nrows, r = i % nrows;
        float v = 0.f;
        for (int w = 0; w < kWarps; ++w) v += partial[(w * FLINT_MAX_TOKENS + t) * rpc + r];
        a.logits[(size_t)t * a.E + r0 + r] = v;
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) is_last = (atomicAdd(a.counter, 1u) == gridDim.x - 1);
    __syncthreads();
    if (!is_last) return;
    __threadfence();

    // ---- top-k: one warp per token; lane holds experts lane, lane+32, ... ----
    if (warp < T) {
        const int t = warp;
        float s[kMaxLanesSlots];
        const int nslot = (a.E + 31) / 32;
#pragma unroll
        for (int i = 0; i < kMaxLanesSlots; ++i) {
            const int e = lane + 32 * i;
            float v = -FLT_MAX;  // below every sigmoid value
            if (i < nslot && e < a.E) {
                float z = ld_cg(a.logits + (size_t)t * a.E + e);
                if (a.bias) z = z + a.bias[e];
                v = 1.f / (1.f + expf(-z));
            }
            s[i] = v;
        }
        uint32_t taken = 0;
        float sel_s[FLINT_MAX_TOPK];
        int sel_e[FLINT_MAX_TOPK];
        float sum = 0.f;
#pragma unroll
        for (int j = 0; j < FLINT_MAX_TOPK; ++j) {
            if (j < a.k) {
                float bs = -FLT_MAX;
                int be = INT32_MAX;
#pragma unroll
                for (int i = 0; i < kMaxLanesSlots; ++i) {
                    // strict '>' keeps the lower index among equal scores
                    if (i < nslot && !((taken >> i) & 1u) && s[i] > bs) {
                        bs = s[i];
                        be = lane + 32 * i;
                    }
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) {
                    const float os = __shfl_xor_sync(0xffffffffu, bs, off);
                    const int oe = __shfl_xor_sync(0xffffffffu, be, off);
                    if (os > bs || (os == bs && oe < be)) {
                        bs = os;
                        be = oe;
                    }
                }
                if ((be & 31) == lane) taken |= 1u << (be >> 5);
                sel_s[j] = bs;
                sel_e[j] = be;
                sum += bs;
            }
        }
#pragma unroll
        for (int j = 0; j < FLINT_MAX_TOPK; ++j) {
            if (j < a.k && lane == j) {
                a.ids[t * a.k + j] = sel_e[j];
                a.weights[t * a.k + j] = sel_s[j] / sum;
            }
        }
    }
    __syncthreads();
    if (tid == 0) atomicExch(a.counter, 0u);
}

}  // namespace

size_t route_smem_bytes(const RouteArgs& a) {
    return 128 + align_up(sizeof(float) * kWarps * FLINT_MAX_TOKENS * a.rows_per_cta, 128) +
           align_up((size_t)a.rows_per_cta * a.H * 2, 128);
}

cudaError_t launch_route(const RouteArgs& a, const DevInfo& d, bool pdl, cudaStream_t s) {
    const size_t smem = route_smem_bytes(a);
    static int configured_for = -1;
    cudaError_t e = configure_smem(route_kernel, d, configured_for);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((a.E + a.rows_per_cta - 1) / a.rows_per_cta));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, route_kernel, a);
}

}  // namespace flint
