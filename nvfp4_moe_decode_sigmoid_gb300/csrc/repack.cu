// repack.cu -- load-time NVFP4 layout conversion and diagnostics.
//
// "Day-0 Support for Flint on vLLM", section "Model architecture": the GGUF
// blocks are NVIDIA's NVFP4 in a different byte order and are repacked
// losslessly at load time. The source and target layouts are defined in
// include/flint.h. One thread moves one 64-value superblock (36 bytes in,
// 32 code bytes + 4 scale bytes out); this is not on the decode path.
#include "flint_device.cuh"

namespace flint {
namespace {

constexpr int kSbBytes = 36;

__global__ void repack_kernel(const uint8_t* __restrict__ src, int64_t n_sb, int64_t sb_per_row, int64_t rows,
                              int64_t cols, uint8_t* __restrict__ dst, int64_t mat_stride, int64_t row_stride) {
    const int64_t sb = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (sb >= n_sb) return;
    const int64_t row_all = sb / sb_per_row;  // row index across all matrices
    const int64_t j = sb % sb_per_row;        // superblock within the row
    const int64_t m = row_all / rows, r = row_all % rows;
    // 36 bytes = 9 aligned words (the source is 16-byte aligned, 36 = 4 * 9)
    const uint32_t* s32 = reinterpret_cast<const uint32_t*>(src + sb * kSbBytes);
    uint32_t wsrc[9];
#pragma unroll
    for (int i = 0; i < 9; ++i) wsrc[i] = s32[i];
    const uint8_t* bytes = reinterpret_cast<const uint8_t*>(wsrc);
    uint32_t out[8];
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        const uint8_t* cb = bytes + 4 + 8 * s;  // 8 code bytes of sub-block s
        uint32_t lo = 0, hi = 0;                // kernel bytes 0..3 and 4..7 of this sub-block
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
            // kernel byte jj holds sub-block values 2jj (low) and 2jj+1 (high)
            const int v0 = 2 * jj, v1 = 2 * jj + 1;
            const uint32_t c0 = v0 < 8 ? (cb[v0] & 15u) : (cb[v0 - 8] >> 4);
            const uint32_t c1 = v1 < 8 ? (cb[v1] & 15u) : (cb[v1 - 8] >> 4);
            const uint32_t byte = c0 | (c1 << 4);
            if (jj < 4) lo |= byte << (8 * jj);
            else hi |= byte << (8 * (jj - 4));
        }
        out[2 * s] = lo;
        out[2 * s + 1] = hi;
    }
    uint8_t* drow = dst + m * mat_stride + r * row_stride;
    uint4* dcodes = reinterpret_cast<uint4*>(drow + 32 * j);
    dcodes[0] = make_uint4(out[0], out[1], out[2], out[3]);
    dcodes[1] = make_uint4(out[4], out[5], out[6], out[7]);
    *reinterpret_cast<uint32_t*>(drow + cols / 2 + 4 * j) = wsrc[0];
    if (j == sb_per_row - 1) {
        for (int64_t p = cols / 2 + cols / 16; p < row_stride; ++p) drow[p] = 0;
    }
}

__global__ void unrepack_kernel(const uint8_t* __restrict__ dst, int64_t n_sb, int64_t sb_per_row, int64_t rows,
                                int64_t cols, int64_t mat_stride, int64_t row_stride, uint8_t* __restrict__ src) {
    const int64_t sb = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (sb >= n_sb) return;
    const int64_t row_all = sb / sb_per_row;
    const int64_t j = sb % sb_per_row;
    const int64_t m = row_all / rows, r = row_all % rows;
    const uint8_t* drow = dst + m * mat_stride + r * row_stride;
    const uint4* dcodes = reinterpret_cast<const uint4*>(drow + 32 * j);
    const uint4 a = dcodes[0], b = dcodes[1];
    const uint32_t in[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t w[9];
    w[0] = *reinterpret_cast<const uint32_t*>(drow + cols / 2 + 4 * j);
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        // 16 codes of sub-block s, value i in kernel byte i/2 (nibble i%2)
        uint32_t code[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const uint32_t word = in[2 * s + (i / 8)];
            const uint32_t byte = (word >> (8 * ((i / 2) % 4))) & 0xFFu;
            code[i] = (i % 2 == 0) ? (byte & 15u) : (byte >> 4);
        }
        uint32_t lo = 0, hi = 0;  // GGUF bytes b = 0..3 and 4..7: value b low, value b+8 high
#pragma unroll
        for (int bb = 0; bb < 8; ++bb) {
            const uint32_t byte = code[bb] | (code[bb + 8] << 4);
            if (bb < 4) lo |= byte << (8 * bb);
            else hi |= byte << (8 * (bb - 4));
        }
        w[1 + 2 * s] = lo;
        w[2 + 2 * s] = hi;
    }
    uint32_t* s32 = reinterpret_cast<uint32_t*>(src + sb * kSbBytes);
#pragma unroll
    for (int i = 0; i < 9; ++i) s32[i] = w[i];
}

// One thread per 32-value chunk: the same decode the GEMV kernels run.
__global__ void dequant_kernel(const uint8_t* __restrict__ packed, int64_t rows, int64_t cols, int64_t row_stride,
                               float* __restrict__ out) {
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t chunks = cols / 32;
    if (idx >= rows * chunks) return;
    const int64_t r = idx / chunks, c = idx % chunks;
    const uint8_t* row = packed + r * row_stride;
    const uint4 q = *reinterpret_cast<const uint4*>(row + 16 * c);
    const uint32_t sc = *reinterpret_cast<const uint16_t*>(row + cols / 2 + 2 * c);
    const float2 s = ue4m3x2_to_float2(sc);
    float w[32];
    decode_chunk(q, w);
    float* o = out + r * cols + 32 * c;
#pragma unroll
    for (int i = 0; i < 32; ++i) o[i] = w[i] * (i < 16 ? s.x : s.y);
}

// Waits on an mbarrier that nothing completes; gives up after budget_ns.
__global__ void selftest_wait_kernel(uint32_t* status, uint64_t budget_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    mbar_wait_bounded(&bar, 0, threadIdx.x == 0 ? status : nullptr, kStatusTimeoutSelftest, budget_ns);
}

}  // namespace

cudaError_t launch_repack(const uint8_t* src, int64_t n_mats, int64_t rows, int64_t cols, uint8_t* dst,
                          int64_t mat_stride, cudaStream_t s) {
    const int64_t spr = cols / 64, n_sb = n_mats * rows * spr;
    if (n_sb == 0) return cudaSuccess;
    const int64_t blocks = (n_sb + 255) / 256;
    repack_kernel<<<(unsigned)blocks, 256, 0, s>>>(src, n_sb, spr, rows, cols, dst, mat_stride,
                                                   nvfp4_row_stride(cols));
    return cudaGetLastError();
}

cudaError_t launch_unrepack(const uint8_t* dst, int64_t n_mats, int64_t rows, int64_t cols, int64_t mat_stride,
                            uint8_t* src, cudaStream_t s) {
    const int64_t spr = cols / 64, n_sb = n_mats * rows * spr;
    if (n_sb == 0) return cudaSuccess;
    const int64_t blocks = (n_sb + 255) / 256;
    unrepack_kernel<<<(unsigned)blocks, 256, 0, s>>>(dst, n_sb, spr, rows, cols, mat_stride,
                                                     nvfp4_row_stride(cols), src);
    return cudaGetLastError();
}

cudaError_t launch_dequant(const uint8_t* packed, int64_t rows, int64_t cols, float* out, cudaStream_t s) {
    const int64_t n = rows * (cols / 32);
    if (n == 0) return cudaSuccess;
    dequant_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(packed, rows, cols, nvfp4_row_stride(cols), out);
    return cudaGetLastError();
}

cudaError_t launch_selftest_wait(uint32_t* status, uint64_t budget_ns, cudaStream_t s) {
    selftest_wait_kernel<<<1, 32, 0, s>>>(status, budget_ns);
    return cudaGetLastError();
}

}  // namespace flint
