// flint_device.cuh -- device helpers shared by the sm_103a kernels:
// 1-D bulk (TMA) copies into shared memory completed on an mbarrier, bounded
// mbarrier waits, programmatic dependent launch, NVFP4 decode.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "flint_internal.h"

namespace flint {

// ---------------------------------------------------------------------------
// Programmatic dependent launch ("Optimizations": each kernel is launched with
// programmatic dependent launch so it loads weights while the previous one
// still runs). Both are no-ops when the kernel was launched without the PDL
// attribute.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------------------
// Shared-memory addresses, mbarriers, bulk copies
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Adds `bytes` to the barrier's expected transaction count without arriving.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

// Arrives once and adds `bytes` to the expected transaction count.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

// One bounded try: the thread may sleep up to ~20 us inside the instruction
// until the phase completes (so waiting warps do not spin on the issue slots).
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity), "r"(20000)
        : "memory");
    return done != 0;
}

// Orders this thread's earlier generic-proxy accesses of shared memory before
// later async-proxy (bulk copy) writes to it.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Waits for phase `parity` of the barrier, for at most budget_ns. Returns
// false (and records `code` in *status) if the wait gave up.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint32_t* status, uint32_t code,
                                                  uint64_t budget_ns = kWaitBudgetNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > budget_ns) {
            if (status) atomicOr(status, code);
            return false;
        }
    }
}

// Pulls `bytes` (a multiple of 16) from a 16-byte aligned global address into
// L2, asynchronously (no completion to wait for).
__device__ __forceinline__ void bulk_prefetch_l2(const void* gmem_src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(gmem_src), "r"(bytes) : "memory");
}

// 1-D bulk copy global -> shared, completing `bytes` transactions on `bar`.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(smem_dst)),
        "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// ---------------------------------------------------------------------------
// 16-byte asynchronous copies global -> shared (cp.async, L2 only), grouped
// per thread: commit closes a group; wait_groups<N> returns once at most N of
// the thread's groups are still in flight. Both addresses 16-byte aligned.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// Runtime N in 0..4.
__device__ __forceinline__ void cp_async_wait_n(int n) {
    switch (n) {
        case 0: cp_async_wait<0>(); break;
        case 1: cp_async_wait<1>(); break;
        case 2: cp_async_wait<2>(); break;
        case 3: cp_async_wait<3>(); break;
        default: cp_async_wait<4>(); break;
    }
}
// The warp copies `bytes` (a multiple of 16) from src to dst, lane l taking
// the 16-byte words l, l + 32, ...
__device__ __forceinline__ void warp_copy_async(void* dst, const void* src, int bytes, int lane) {
    uint8_t* d = static_cast<uint8_t*>(dst);
    const uint8_t* s = static_cast<const uint8_t*>(src);
    for (int o = 16 * lane; o < bytes; o += 512) cp_async16(d + o, s + o);
}

// Warms the address translation (and L2) for the bytes [p, p + n): a
// prefetch of the first and the last byte, neither of which blocks. Kernels
// issue these at their start for the small buffers they touch late (outputs,
// scales, activations), so the page walks overlap other work instead of
// stalling the first access behind the weight stream.
__device__ __forceinline__ void prefetch_range(const void* p, size_t n) {
    if (!p || n == 0) return;
    const char* c = static_cast<const char*>(p);
    asm volatile("prefetch.global.L2 [%0];" ::"l"(c));
    asm volatile("prefetch.global.L2 [%0];" ::"l"(c + n - 1));
}

// ---------------------------------------------------------------------------
// Loads that bypass L1: data written by another kernel of the PDL chain.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int32_t ld_cg(const int32_t* p) { return __ldcg(p); }
__device__ __forceinline__ float ld_cg(const float* p) { return __ldcg(p); }
__device__ __forceinline__ uint4 ld_cg(const uint4* p) { return __ldcg(p); }
__device__ __forceinline__ uint2 ld_cg(const uint2* p) { return __ldcg(p); }

// Acquire load at GPU scope (a flag written by another CTA).
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}


// ---------------------------------------------------------------------------
// bf16 helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float v) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}
__device__ __forceinline__ float bf16_round_f32(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }

// ---------------------------------------------------------------------------
// NVFP4 decode
// ---------------------------------------------------------------------------
// Two E2M1 codes (one byte: column 2j low nibble, 2j+1 high nibble) -> two
// exact floats, via the hardware FP4 -> f16x2 conversion.
__device__ __forceinline__ float2 e2m1x2_to_float2(uint32_t byte) {
    uint32_t h2;
    asm("{\n .reg .b8 b;\n cvt.u8.u32 b, %1;\n cvt.rn.f16x2.e2m1x2 %0, b;\n}" : "=r"(h2) : "r"(byte));
    return __half22float2(*reinterpret_cast<__half2*>(&h2));
}

// Two UE4M3 scale bytes (low byte = first) -> two exact floats. Bit 7 of each
// byte is not part of the unsigned format and is cleared.
__device__ __forceinline__ float2 ue4m3x2_to_float2(uint32_t two_bytes) {
    uint32_t h2;
    const uint16_t v = static_cast<uint16_t>(two_bytes & 0x7F7Fu);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(v));
    return __half22float2(*reinterpret_cast<__half2*>(&h2));
}

// 8 codes of one 32-bit word (byte b: codes 2b, 2b+1) -> 4 exact float pairs.
__device__ __forceinline__ void decode_word(uint32_t w, float2* f) {
    uint32_t h0, h1, h2, h3;
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
        " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
        " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
        : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
        : "r"(w));
    f[0] = __half22float2(*reinterpret_cast<__half2*>(&h0));
    f[1] = __half22float2(*reinterpret_cast<__half2*>(&h1));
    f[2] = __half22float2(*reinterpret_cast<__half2*>(&h2));
    f[3] = __half22float2(*reinterpret_cast<__half2*>(&h3));
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Barrier among the first `threads` threads of the CTA (hardware barrier `id`).
__device__ __forceinline__ void named_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// 8 codes of one 32-bit word -> 4 f16x2 registers (exact; byte b: codes 2b, 2b+1).
__device__ __forceinline__ void decode_word_h2(uint32_t w, uint32_t (&h)[4]) {
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
        " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
        " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(w));
}

// acc + a.lo * b.lo and acc + a.hi * b.hi for f16x2 operands, FP32 accumulate.
// The f16 x f16 product is exact in FP32, so each step rounds once, like an
// FP32 FMA of the same values.
__device__ __forceinline__ float fma_lo_f16(uint32_t a, uint32_t b, float acc) {
    float d;
    asm("{\n .reg .f16 a0, a1, b0, b1;\n mov.b32 {a0, a1}, %1;\n mov.b32 {b0, b1}, %2;\n"
        " fma.rn.f32.f16 %0, a0, b0, %3;\n}"
        : "=f"(d)
        : "r"(a), "r"(b), "f"(acc));
    return d;
}
__device__ __forceinline__ float fma_hi_f16(uint32_t a, uint32_t b, float acc) {
    float d;
    asm("{\n .reg .f16 a0, a1, b0, b1;\n mov.b32 {a0, a1}, %1;\n mov.b32 {b0, b1}, %2;\n"
        " fma.rn.f32.f16 %0, a1, b1, %3;\n}"
        : "=f"(d)
        : "r"(a), "r"(b), "f"(acc));
    return d;
}

// Two floats -> f16x2 (round to nearest; exact for the scaled activations).
__device__ __forceinline__ uint32_t f32x2_to_f16x2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// One UE4M3 scale byte -> exact float (bit 7 cleared).
__device__ __forceinline__ float ue4m3_to_float(uint32_t byte) { return ue4m3x2_to_float2(byte & 0xFFu).x; }

// 32 codes of one 16-byte chunk -> 32 floats (code values, no scale).
__device__ __forceinline__ void decode_chunk(const uint4 q, float (&w)[32]) {
    const uint32_t words[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const float2 v = e2m1x2_to_float2((words[i] >> (8 * b)) & 0xFFu);
            w[8 * i + 2 * b] = v.x;
            w[8 * i + 2 * b + 1] = v.y;
        }
    }
}

}  // namespace flint
