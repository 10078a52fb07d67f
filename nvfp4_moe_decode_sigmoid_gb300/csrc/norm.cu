// norm.cu -- residual add + RMSNorm between the blocks of the decode stack,
// as a kernel of its own (the MoE block fuses the same computation into the
// fused layer kernel's input staging).
//
// "vLLM 宣布首日支持 Recursive 的 Flint ...", section "Flint 是什么": a
// pre-norm Transformer of 49 blocks (2 dense MLP blocks, 47 MoE blocks),
// hidden size 2048. "Day-0 Support for Flint on vLLM", section
// "Optimizations": norm kernels that follow the reference's rounding points.
// Per token: r' = bf16(r + y), x = bf16(r' / sqrt(mean(r'^2) + eps) * gamma),
// FP32 arithmetic, the sum of squares in the same fixed order as the fused
// staging (so both give the same x).
//
// One CTA per token; thread i takes the 32-value chunks i, i + blockDim, ...
#include "expert_common.cuh"

namespace flint {
namespace {

constexpr int kNormThreads = 128;
constexpr int kNormMaxChunks = 1024;  // H <= 32768

__global__ void __launch_bounds__(kNormThreads) rmsnorm_kernel(const NormArgs a) {
    __shared__ float red[kNormMaxChunks];
    __shared__ float inv;
    pdl_launch_dependents();  // dependents wait for this grid before reading x
    pdl_wait();               // r and y come from earlier kernels
    const int t = blockIdx.x, cpv = a.H / 32, tid = threadIdx.x;
    uint4 w0[4] = {};
    for (int c = tid; c < cpv; c += kNormThreads) {
        uint4 w[4];
        const size_t off = (size_t)t * a.H + 32 * c;
        red[c] = norm_residual_chunk(a, off, w);
        if (a.r_out) {
#pragma unroll
            for (int i = 0; i < 4; ++i) reinterpret_cast<uint4*>(a.r_out + off)[i] = w[i];
        }
        if (c == tid) {
#pragma unroll
            for (int i = 0; i < 4; ++i) w0[i] = w[i];
        }
    }
    __syncthreads();
    if (tid < 32) {
        float s = 0.f;
        for (int c = tid; c < cpv; c += 32) s += red[c];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        if (tid == 0) inv = 1.f / sqrtf(s / (float)a.H + a.eps);
    }
    __syncthreads();
    for (int c = tid; c < cpv; c += kNormThreads) {
        uint4 w[4];
        const size_t off = (size_t)t * a.H + 32 * c;
        if (c == tid) {
#pragma unroll
            for (int i = 0; i < 4; ++i) w[i] = w0[i];
        } else {
            norm_residual_chunk(a, off, w);
        }
        norm_scale_chunk(a, 32 * c, inv, w);
#pragma unroll
        for (int i = 0; i < 4; ++i) reinterpret_cast<uint4*>(a.x_out + off)[i] = w[i];
    }
}

}  // namespace

cudaError_t launch_rmsnorm(const NormArgs& a, bool pdl, cudaStream_t s) {
    if (a.H / 32 > kNormMaxChunks) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.T);
    cfg.blockDim = dim3(kNormThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, rmsnorm_kernel, a);
}

}  // namespace flint
