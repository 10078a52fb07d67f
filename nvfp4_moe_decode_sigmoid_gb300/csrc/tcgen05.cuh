// tcgen05.cuh -- the 5th-generation tensor-core path of sm_103a: tensor-memory
// (TMEM) allocation, tcgen05.mma of kind::f16 from shared-memory operands,
// completion on an mbarrier, and TMEM -> register loads for the epilogue.
//
// Operand layout: K-major tiles without swizzle ("interleaved" canonical
// layout). A tile of R rows x 64 bf16 (one K step) is stored as 8 x 8 core
// matrices of 8 rows x 16 bytes (128 contiguous bytes each): core matrix
// (row group g, K chunk c) at g * 1024 + c * 128, element (r, k) at
// (r / 8) * 1024 + (k / 8) * 128 + (r % 8) * 16 + (k % 8) * 2. The matrix
// descriptor then gives the byte distance of K-adjacent core matrices (128)
// and of row-adjacent ones (1024); one MMA of K = 16 spans two K chunks, so
// the k-th MMA of a step starts 256 * k bytes into the tile.
#pragma once

#include "flint_device.cuh"

namespace flint {

constexpr uint32_t kTcCoreK = 128;    // bytes between K-adjacent core matrices
constexpr uint32_t kTcCoreRow = 1024; // bytes between row-adjacent core matrices (64-wide K step)

// Byte offset of element (r, k) in a K-major tile of 64-wide K (bf16).
__host__ __device__ __forceinline__ uint32_t tc_tile_offset(int r, int k) {
    return (uint32_t)((r >> 3) * kTcCoreRow + (k >> 3) * kTcCoreK + (r & 7) * 16 + (k & 7) * 2);
}

// Shared-memory matrix descriptor (no swizzle): start address, byte offset
// of K-adjacent core matrices (leading), of row-adjacent ones (stride), all
// in 16-byte units; descriptor version 1.
__device__ __forceinline__ uint64_t tc_smem_desc(const void* p, uint32_t lead_bytes, uint32_t stride_bytes) {
    const uint32_t a = smem_u32(p);
    return (uint64_t)((a >> 4) & 0x3FFFu) | ((uint64_t)((lead_bytes >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((stride_bytes >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}

// Shared-memory matrix descriptor of a K-major tile in the 128-byte swizzled
// layout that a TMA tile load with 128-byte swizzle writes: rows of 128 bytes
// (64 bf16 of K), 16-byte chunk c of row r stored at chunk c ^ (r % 8), 8-row
// groups 1024 bytes apart; the tile starts on a 1024-byte boundary and the
// k-th MMA of K = 16 starts 32 * k bytes into it.
__device__ __forceinline__ uint64_t tc_smem_desc_sw128(const void* p) {
    const uint32_t a = smem_u32(p);
    return (uint64_t)((a >> 4) & 0x3FFFu) | (1ull << 16) | ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) |
           (2ull << 61);
}

// Byte offset of element (r, k) (bf16) in a 128-byte-swizzled K-major tile.
__host__ __device__ __forceinline__ uint32_t tc_sw128_offset(int r, int k) {
    return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((((k >> 3) ^ r) & 7) << 4) + (k & 7) * 2);
}

// 2-D TMA tile load global -> shared completing on `bar` (tensor map passed as
// a __grid_constant__ kernel parameter; c0 = innermost coordinate).
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int c0, int c1, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}

// Instruction descriptor of kind::f16 with bf16 A and B, FP32 accumulator,
// both operands K-major, an M x N tile.
__host__ __device__ constexpr uint32_t tc_idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// TMEM allocation of `ncols` columns (a power of two >= 32) by one full warp;
// the address lands in *slot (shared memory).
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D (TMEM) = A B^T (+ D when `accumulate`), one thread issues.
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The mbarrier receives one arrival when every tcgen05 operation this thread
// issued before has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// Lanes [32 (warp % 4), +32) x 16 consecutive 32-bit columns from `taddr`
// (lane in bits 31..16, column in bits 15..0): thread i gets lane base + i.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

}  // namespace flint
