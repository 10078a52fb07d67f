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

#include "expert_common.cuh"
#include "router_common.cuh"

namespace flint {
namespace {

// Shared memory: mbarrier, per-warp partial logits, the CTA's router rows.
__host__ __device__ inline size_t route_scores_offset(const RouteArgs& a) {
    return 128 + align_up(sizeof(float) * kWarps * FLINT_MAX_TOKENS * a.rows_per_cta, 128) +
           align_up((size_t)a.rows_per_cta * a.H * 2, 128);
}

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
        const uint32_t bytes = (uint32_t)(nrows * H * 2);
        mbar_arrive_expect_tx(bar, bytes);
        bulk_g2s(wrows, a.wr + (size_t)r0 * H, bytes, bar);
    }
    if (tid == kThreads - 1) {
        prefetch_range(a.x, 2 * (size_t)T * H);
        prefetch_range(a.bias, 4 * (size_t)a.E);
        prefetch_range(a.logits, 4 * (size_t)T * a.E);
        prefetch_range(a.counter, 8);
        prefetch_range(a.ids, 4 * (size_t)T * a.k);
        prefetch_range(a.weights, 4 * (size_t)T * a.k);
    }
    __syncthreads();  // the barrier is initialised before anyone waits on it
    pdl_wait();  // x may come from the previous kernel
    // Dependents start only now: the gate/up kernel may then read x before its
    // own wait (x is complete once this kernel has passed its wait).
    pdl_launch_dependents();

    const int nchunk = H / 8;
    const bool ok = mbar_wait_bounded(bar, 0, tid == 0 ? a.status : nullptr, kStatusTimeoutRoute);
    if (!__syncthreads_and(ok)) return;

    float acc[FLINT_MAX_TOKENS][2];
#pragma unroll
    for (int t = 0; t < FLINT_MAX_TOKENS; ++t) acc[t][0] = acc[t][1] = 0.f;
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
        // reduce over the block: the 2 x 8 sums reduce-scattered over the warp
        // (two lanes end with each), then a fixed-order sum over the warps
        float v16[2 * FLINT_MAX_TOKENS];
#pragma unroll
        for (int t = 0; t < FLINT_MAX_TOKENS; ++t) {
            v16[2 * t] = acc[t][0];
            v16[2 * t + 1] = acc[t][1];
            acc[t][0] = acc[t][1] = 0.f;
        }
        const float v = reduce_scatter<2 * FLINT_MAX_TOKENS>(v16, lane);
        const int idx = rs_index<2 * FLINT_MAX_TOKENS>(lane), t = idx >> 1, q = idx & 1;
        if ((lane & 1) == 0 && t < T && rb + q < nrows) partial[(warp * FLINT_MAX_TOKENS + t) * rpc + rb + q] = v;
    }
    __syncthreads();
    for (int i = tid; i < T * nrows; i += kThreads) {
        const int t = i / nrows, r = i % nrows;
        float v = 0.f;
        for (int w = 0; w < kWarps; ++w) v += partial[(w * FLINT_MAX_TOKENS + t) * rpc + r];
        a.logits[(size_t)t * a.E + r0 + r] = v;
    }
    // Publish the logits, take a ticket; the last CTA does the selection.
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        is_last = (atomicAdd(a.counter, 1u) == gridDim.x - 1);
        if (is_last) __threadfence();
    }
    __syncthreads();
    if (!is_last) return;

    // one warp per token: its logits straight from L2, the sigmoid on load
    if (warp < T) {
        const float* lg = a.logits + (size_t)warp * a.E;
        if (a.E <= 256)
            topk_warp_logits<8>(lg, a.bias, a.E, a.k, lane, a.ids + warp * a.k, a.weights + warp * a.k);
        else
            topk_warp_logits<FLINT_MAX_EXPERTS / 32>(lg, a.bias, a.E, a.k, lane, a.ids + warp * a.k,
                                                     a.weights + warp * a.k);
    }
    __syncthreads();
    if (tid == 0) atomicExch(a.counter, 0u);
}

}  // namespace

size_t route_smem_bytes(const RouteArgs& a) { return route_scores_offset(a); }

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
