/*
 * flint.h -- C ABI of the GB300 (sm_103a) small-batch decode path of a
 * Flint-style MoE layer with weight-only NVFP4 (W4A16) weights.
 *
 * The method (sources):
 *  - "Day-0 Support for Flint on vLLM", section "Model architecture": 256
 *    routed experts with sigmoid top-6 selection plus a shared expert; the
 *    NVFP4 checkpoint is a GGUF file whose blocks are NVIDIA's NVFP4 format in
 *    a different byte order, repacked losslessly at load time and run
 *    weight-only (W4A16) with BF16 activations; every kernel follows the
 *    reference implementation's rounding points.
 *  - same page, section "Optimizations": router and expert GEMVs that read
 *    only the selected experts' weights; a small-batch dense GEMV on the same
 *    packed NVFP4 weights; for up to 8 requests, routing and the expert
 *    combine fused into the neighbouring GEMV kernels, each launched with
 *    programmatic dependent launch so it loads its weights while the previous
 *    kernel still runs.
 *  - "vLLM 宣布首日支持 Recursive 的 Flint ...", section
 *    "七个内核的依赖链：低延迟路径、无损重排与参考舍入": a 64-value superblock is
 *    4 x [UE4M3 scale + 16 E2M1 codes], with one FP32 scale per tensor (per
 *    expert for MoE weights).
 *
 * Conventions for every call:
 *  - Array pointers are DEVICE pointers owned by the caller, unless a comment
 *    says otherwise. Structs passed by pointer are read on the host during the
 *    call and may be freed when it returns.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream). Calls are
 *    asynchronous on that stream; the library never synchronises it except
 *    in flint_workspace_check.
 *  - The library allocates no memory. Scratch space ("workspace") is passed
 *    in by the caller; see flint_workspace_bytes.
 *  - bf16 values are passed as their 16-bit patterns (flint_bf16).
 *  - Errors are returned, never thrown. Argument errors are detected on the
 *    host before anything is launched. FLINT_ERR_CUDA carries the CUDA error
 *    text in flint_last_error() (thread-local). A device-side wait that gives
 *    up (FLINT_ERR_TIMEOUT) cannot be returned by the launching call; it is
 *    recorded in the workspace's status word and reported by
 *    flint_workspace_check.
 *  - The kernels are built for sm_103a only; any other device gives
 *    FLINT_ERR_UNSUPPORTED. There is no CPU fallback.
 */
#ifndef FLINT_H
#define FLINT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t flint_bf16; /* bfloat16 bit pattern */

typedef enum flint_status {
    FLINT_OK = 0,
    FLINT_ERR_INVALID_ARG = 1, /* null or misaligned pointer, bad size or shape */
    FLINT_ERR_UNSUPPORTED = 2, /* valid but outside what the kernels handle (T > 8, wrong GPU, ...) */
    FLINT_ERR_CUDA = 3,        /* a CUDA runtime call failed; see flint_last_error() */
    FLINT_ERR_TIMEOUT = 4      /* a bounded device-side wait gave up (from flint_workspace_check) */
} flint_status_t;

enum { FLINT_DTYPE_NVFP4 = 0, FLINT_DTYPE_BF16 = 1 };
enum { FLINT_EPILOGUE_NONE = 0, FLINT_EPILOGUE_SWIGLU = 1 };
/* flags: launch with programmatic dependent launch (PDL). The kernel then may
 * start while the previous kernel on the stream still runs; it prefetches
 * weights first and waits for the previous kernel before it reads any input
 * that kernel could have written. */
enum { FLINT_PDL = 1u << 0 };
/* flags, with FLINT_PDL, for flint_moe_gate_up / flint_moe_decode: the
 * previous kernel on the stream is flint_moe_route on the same x. The router
 * triggers its dependents only after its own wait, so x is complete when the
 * gate/up kernel starts and is staged before that kernel's wait. Do not set it
 * after any other kernel. */
enum { FLINT_PDL_AFTER_ROUTE = 1u << 1 };

/* Largest batch of the decode path (the low-latency bound of up to 8 requests). */
#define FLINT_MAX_TOKENS 8
/* Largest top-k and largest routed expert count. */
#define FLINT_MAX_TOPK 8
#define FLINT_MAX_EXPERTS 1024

/* ------------------------------------------------------------------------ */
/* Packed NVFP4 weights                                                      */
/* ------------------------------------------------------------------------ */
/*
 * Source layout (GGUF superblocks), as read by this library: a [rows, cols]
 * matrix (cols % 64 == 0) is rows * cols/64 superblocks of 36 bytes, in row
 * order and along each row. Superblock bytes 0..3 are the UE4M3 scales of its
 * four 16-value sub-blocks; bytes 4+8s .. 4+8s+7 are the E2M1 codes of
 * sub-block s, byte b holding sub-block value b in its low nibble and value
 * b+8 in its high nibble. Matrices are contiguous. The FP32 tensor scale is
 * not part of the blocks; it is passed separately (flint_experts,
 * flint_packed).
 *
 * Kernel layout (the repack target): each row is
 *   bytes [0, cols/2)                 E2M1 codes, byte j = column 2j in the low
 *                                     nibble, column 2j+1 in the high nibble
 *   bytes [cols/2, cols/2 + cols/16)  UE4M3 scales, byte b covers columns
 *                                     16b .. 16b+15
 *   zero padding to the row stride    flint_nvfp4_row_stride(cols), the next
 *                                     multiple of 16 bytes (no padding when
 *                                     cols % 256 == 0)
 * Rows are contiguous; matrix m of a repack starts at m * dst_mat_stride.
 * A row's codes and scales sit together so that a run of rows is one
 * contiguous block for a single bulk (TMA) copy.
 *
 * Element value = E2M1(code) * UE4M3(scale) * tensor_scale. UE4M3 bit 7 is
 * ignored. UE4M3 0x7F (NaN) is outside the supported input domain.
 */
int64_t flint_nvfp4_row_stride(int64_t cols);
int64_t flint_nvfp4_packed_bytes(int64_t n_mats, int64_t rows, int64_t cols);
int64_t flint_gguf_nvfp4_bytes(int64_t n_mats, int64_t rows, int64_t cols);

/*
 * flint_nvfp4_repack -- lossless, bit-exact repack of n_mats GGUF NVFP4
 * matrices [rows, cols] into the kernel layout (load-time step of "Model
 * architecture": the GGUF blocks are repacked losslessly at load time).
 *   src:  n_mats * rows * cols/64 * 36 bytes, 16-byte aligned.
 *   dst:  matrix m at dst + m * dst_mat_stride; 16-byte aligned.
 *         dst_mat_stride = 0 means rows * flint_nvfp4_row_stride(cols);
 *         otherwise it must be >= that and a multiple of 16 (used to place
 *         gate rows and up rows of one expert in a [2I, H] gate/up matrix).
 *         Bytes between matrices are not touched.
 *   Errors: FLINT_ERR_INVALID_ARG (null/misaligned pointer, cols % 64 != 0,
 *   negative sizes, stride too small); FLINT_ERR_CUDA.
 */
flint_status_t flint_nvfp4_repack(const uint8_t* src, int64_t n_mats, int64_t rows, int64_t cols,
                                  uint8_t* dst, int64_t dst_mat_stride, void* stream);

/* Inverse of flint_nvfp4_repack (kernel layout -> GGUF superblocks); same
 * arguments with src as the output. Used to prove the repack lossless. */
flint_status_t flint_nvfp4_unrepack(const uint8_t* dst, int64_t n_mats, int64_t rows, int64_t cols,
                                    int64_t dst_mat_stride, uint8_t* src, void* stream);

/* Dequantise a [rows, cols] kernel-layout matrix to float (without the tensor
 * scale), with the same decode routine the GEMV kernels use.
 *   out: rows * cols floats, row-major. Used to prove the dequant bit-exact. */
flint_status_t flint_nvfp4_dequant(const uint8_t* packed, int64_t rows, int64_t cols, float* out,
                                   void* stream);

/* ------------------------------------------------------------------------ */
/* Workspace                                                                 */
/* ------------------------------------------------------------------------ */
/*
 * One workspace serves flint_moe_route, flint_moe_gate_up,
 * flint_moe_down_combine, flint_moe_decode, flint_moe_layer and
 * flint_moe_block for one layer shape; layers of the same shape may share it
 * when their calls are issued in order on one stream. It holds a control
 * header (router arrival counter, status word, the fused layer's call and
 * finished-CTA counts and published-router-rows count, the wait budget, a
 * test hook), the router's FP32 logits [8, E] and the bf16 SwiGLU activations
 * h of the routed [8, k, I] and shared [8, I_shared] experts (used by
 * flint_moe_route / flint_moe_decode and by the fused layer), then the fused
 * layer's per-expert outputs d [8, k, hidden] and [8, hidden], one arrival
 * counter per 16 output rows and one published-h counter per expert.
 *   - Must be 256-byte aligned and zero-filled before first use
 *     (flint_workspace_init). Every completed call leaves the counters ready
 *     for the next.
 *   - Calls that use one workspace must not overlap on the GPU except as the
 *     PDL chain route -> gate_up -> down_combine -> next route allows (and
 *     fused-layer calls chained with FLINT_PDL, which wait for the previous
 *     kernel before touching the workspace).
 *   - flint_moe_route needs only the regions up to the routed experts' h;
 *     any `hidden` (0 included) sizes a workspace for it. So does
 *     flint_moe_decode, which then runs as two kernels; on a workspace sized
 *     with the experts' hidden size it runs as one (see there).
 */
size_t flint_workspace_bytes(int num_experts, int top_k, int hidden, int inter, int inter_shared);
flint_status_t flint_workspace_init(void* ws, size_t ws_bytes, void* stream);
/* Synchronises `stream`, reads the status word and returns:
 *   FLINT_ERR_TIMEOUT if a kernel recorded a timed-out wait: the whole
 *     workspace is then re-initialised (zero-filled, as flint_workspace_init),
 *     because the counters the kernels synchronise on may have been left
 *     mid-call. Until this check runs, every later fused-layer call on the
 *     workspace returns at once without writing its outputs;
 *   FLINT_ERR_INVALID_ARG if flint_moe_decode was given an expert id outside
 *     [0, num_experts) (the status word is cleared);
 *   FLINT_ERR_UNSUPPORTED if a fused-layer CTA's work exceeded its shared-memory
 *     plan (not expected; the workspace is re-initialised as after a timeout);
 *   FLINT_OK otherwise. */
flint_status_t flint_workspace_check(void* ws, size_t ws_bytes, void* stream);
/* Sets the budget of every bounded device-side wait of the kernels that use
 * this workspace to budget_us microseconds (0 restores the default of 2 s).
 * A wait that runs out records FLINT_ERR_TIMEOUT (see flint_workspace_check).
 * Synchronises `stream`. */
flint_status_t flint_workspace_set_wait_budget(void* ws, size_t ws_bytes, uint32_t budget_us, void* stream);

/* ------------------------------------------------------------------------ */
/* MoE layer                                                                 */
/* ------------------------------------------------------------------------ */

/* Expert weights of one MoE layer (or of its shared expert, with
 * num_experts = 1).
 *
 * FLINT_DTYPE_BF16 ("Day-0 Support for Flint on vLLM", section
 * "Optimizations": the decode path also serves the BF16 checkpoint): gate_up
 * is E bf16 matrices [2I, H] row-major (rows [0, I) gate, [I, 2I) up), down E
 * bf16 matrices [H, I] row-major; tensor_scale may be NULL (every scale 1).
 * The arithmetic and rounding points are those of the NVFP4 path with the
 * weight equal to the bf16 value. Taken by flint_moe_gate_up,
 * flint_moe_down_combine and flint_moe_decode (not by flint_moe_layer);
 * routed and shared experts must have the same dtype. */
typedef struct flint_experts {
    int32_t dtype;        /* FLINT_DTYPE_NVFP4 or FLINT_DTYPE_BF16 */
    int32_t num_experts;  /* E */
    int32_t hidden;       /* H: columns of gate/up, rows of down; % 1024 == 0 */
    int32_t inter;        /* I: intermediate size; % 256 == 0 */
    const void* gate_up;  /* NVFP4: E matrices [2I, H], kernel layout, matrix
                             stride 2I * row_stride(H); rows [0, I) gate, [I, 2I) up */
    const void* down;     /* NVFP4: E matrices [H, I], kernel layout, stride H * row_stride(I) */
    const float* tensor_scale; /* [E][3] FP32: gate, up, down (NVFP4: required) */
} flint_experts;

/*
 * flint_moe_route -- router GEMV, sigmoid, top-k and renormalisation (one
 * kernel; "Model architecture": sigmoid top-6 over 256 experts; "Optimizations":
 * routing fused into the GEMV kernels).
 *   x:        bf16 [T, H] row-major, 16-byte aligned; 1 <= T <= 8; H % 256 == 0.
 *   router_w: bf16 [E, H] row-major, 16-byte aligned; k <= E <= 1024.
 *   bias:     FP32 [E] added to the logits before the sigmoid, or NULL.
 *   ids:      out int32 [T, k]: per token the k experts with the largest
 *             sigmoid(logit + bias), computed in FP32, in descending order,
 *             ties to the lower index.
 *   weights:  out FP32 [T, k]: the selected scores renormalised to sum 1.
 *   ws:       workspace (flint_workspace_bytes(E, k, ...)).
 * Logits are FP32 dot products and are not rounded to bf16. The last CTA to
 * finish its logits performs the selection (no second kernel).
 */
flint_status_t flint_moe_route(const flint_bf16* x, int T, int H, const flint_bf16* router_w, int E,
                               const float* bias, int k, int32_t* ids, float* weights, void* ws,
                               size_t ws_bytes, unsigned flags, void* stream);

/*
 * flint_moe_route_static -- the same router as flint_moe_route, for callers
 * that cannot hand the library any device memory of their own: for example a
 * plug-in whose host framework owns every device allocation and forbids new
 * ones, or a C caller that holds only its input and output buffers and no
 * allocator. The pages describe nothing like it (it has no counterpart in the
 * method); it exists only for such callers.
 *   Arguments as flint_moe_route, without ws/ws_bytes. The results equal those
 *   of flint_moe_route on the same inputs.
 *   Scratch: a 33,024-byte array inside the library (a 256-byte header with
 *   the counter and status word, then FP32 logits for T x E <= 8 x 1024),
 *   held by every device that loads the library until the process exits.
 *   E above 1024 (the selection's limit, as for flint_moe_route), or T x E
 *   beyond the scratch, is rejected with FLINT_ERR_UNSUPPORTED and a message
 *   giving the limit.
 *   The first call on a device looks up the array's device address (with that
 *   device current); make that first call before any stream capture.
 *   Every call clears the 256-byte scratch header (one memset on `stream`)
 *   and then overwrites the logits. All calls share the one array:
 *   calls issued in order on one stream follow each other (the memset waits
 *   for the previous kernel), but calls that can run at the same time on the
 *   GPU (different streams or threads) race on it and must be serialised by
 *   the caller.
 *   A timed-out wait inside the kernel leaves ids/weights unwritten and is not
 *   reported (the status word lives in the shared scratch, which the next
 *   call clears): a caller that must detect it fills ids with -1 first and
 *   checks them after the stream synchronises. No memory is allocated or
 *   freed.
 */
flint_status_t flint_moe_route_static(const flint_bf16* x, int T, int H, const flint_bf16* router_w, int E,
                                      const float* bias, int k, int32_t* ids, float* weights, unsigned flags,
                                      void* stream);

/*
 * flint_moe_gate_up -- for every token and every selected expert (and the
 * shared expert): g = bf16(ts_g * Wg x), u = bf16(ts_u * Wu x),
 * h = bf16(silu(g) * u), with FP32 accumulation. Reads only the distinct
 * selected experts' gate/up rows; writes h into the workspace. One kernel.
 *   x [T, H] bf16; ids [T, k] int32 (as from flint_moe_route); routed
 *   required; shared may be NULL.
 */
flint_status_t flint_moe_gate_up(const flint_bf16* x, int T, const int32_t* ids, int k,
                                 const flint_experts* routed, const flint_experts* shared, void* ws,
                                 size_t ws_bytes, unsigned flags, void* stream);

/*
 * flint_moe_down_combine -- d_j = bf16(ts_d * Wd_j h_j) for every selected
 * expert j and the shared expert, then the combine
 * y = bf16(sum_j weights[j] * d_j + d_shared), FP32 accumulation in rank
 * order then the shared term. Each CTA owns a slice of output rows across all
 * selected experts, so the combine needs no atomics and is deterministic.
 * One kernel. Reads h from the workspace written by flint_moe_gate_up.
 *   weights [T, k] FP32; y out bf16 [T, H].
 */
flint_status_t flint_moe_down_combine(int T, const int32_t* ids, const float* weights, int k,
                                      const flint_experts* routed, const flint_experts* shared,
                                      flint_bf16* y, void* ws, size_t ws_bytes, unsigned flags,
                                      void* stream);

/*
 * flint_moe_decode -- the experts of one MoE layer for a given routing:
 * y = bf16(sum_j weights[j] * d_j + d_shared) with h and d as in
 * flint_moe_gate_up and flint_moe_down_combine ("Optimizations": the expert
 * GEMVs read only the selected experts, the combine fused into the down GEMV).
 *   x [T, H] bf16; ids [T, k] int32 and weights [T, k] FP32 (as from
 *   flint_moe_route; an id may repeat within a token, and an id outside
 *   [0, E) is reported by flint_workspace_check and its rank adds nothing);
 *   y out [T, H] bf16.
 *   - NVFP4 experts and a workspace of at least
 *     flint_workspace_bytes(E, k, hidden, inter, inter_shared) (hidden = the
 *     experts' H): one cooperative kernel, one CTA per SM (the fused layer of
 *     flint_moe_layer with its router left out, its one-token kernel at
 *     T == 1; ids and weights read after its PDL wait). With FLINT_PDL |
 *     FLINT_PDL_AFTER_ROUTE it stages x before that wait. Like flint_moe_layer, it needs every CTA resident (shapes
 *     that do not fit run as below) and a workspace used by one such call at a
 *     time.
 *   - Otherwise (BF16 experts, a smaller workspace, or shapes the one kernel
 *     cannot hold): flint_moe_gate_up then flint_moe_down_combine, two kernels,
 *     the second PDL-chained to the first when flags has FLINT_PDL.
 * Both give the same rounding points and rank order of the combine; the FP32
 * summation order inside the GEMVs differs, so their y may differ in the last
 * bf16 place.
 */
flint_status_t flint_moe_decode(const flint_bf16* x, int T, const int32_t* ids, const float* weights, int k,
                                const flint_experts* routed, const flint_experts* shared, flint_bf16* y,
                                void* ws, size_t ws_bytes, unsigned flags, void* stream);

/*
 * Byte ranges of the NEXT layer's static weights (its router rows, its shared
 * expert) that flint_moe_layer / flint_moe_block pull into L2 while this
 * layer routes (its HBM traffic is low then): those addresses do not depend
 * on data ("Optimizations": each kernel loads its weights while the previous
 * one runs). Up to four ranges; a range has a
 * 16-byte aligned start and a size that is a multiple of 16 (0: unused); the
 * sizes sum to less than 4 GiB. Pass NULL for none.
 */
typedef struct flint_l2_prefetch {
    const void* ptr[4];
    size_t bytes[4];
} flint_l2_prefetch;

/*
 * flint_moe_layer -- the whole decode step of one MoE layer in ONE kernel:
 * router GEMV + sigmoid top-k + renormalisation (as flint_moe_route), the
 * gate/up GEMVs + SiLU and the down GEMVs + combine (as flint_moe_decode).
 * ("Optimizations": the small-batch MoE path fuses the routing and the
 * combine into the neighbouring expert GEMVs and chains them with PDL so that
 * each kernel loads its weights while the previous one runs.) One CTA per SM,
 * all resident (cooperative launch). A group of CTAs runs the shared expert,
 * whose weights they start loading before the PDL wait; the rest split the
 * selected experts' gate/up pairs (and, from two tokens, their down rows) by
 * cost. CTAs exchange the router scores and h through the workspace under
 * release / acquire counts (a CTA waits only for the scores and for the h of
 * the experts it uses; no grid-wide barrier); the combine of each 16-row
 * block of y is done by the CTA that delivers its last expert output. At one
 * token (T == 1) a kernel laid out for latency runs instead: every CTA takes
 * equal fixed shares of the router rows, the shared expert's pairs, the
 * selected experts' pairs (in rank order) and the output rows, and issues its
 * whole share of the weights at once; its CTAs are small enough (12 warps)
 * for two to fit on an SM, so with FLINT_PDL the next layer's CTAs become
 * resident while this one runs. Every CTA then computes its rows of y from
 * all of h, with no exchange of d. Same rounding points either way.
 *   x [T, H] bf16 (H = routed->hidden, H % 1024 == 0, H <= 8192), router_w
 *   [E, H] bf16 with E = routed->num_experts, bias [E] FP32 or NULL,
 *   1 <= k <= min(8, E). ids [T, k] int32 and weights [T, k] FP32 are written
 *   (as flint_moe_route would); y [T, H] bf16 out. shared may be NULL.
 *   ws: the layer's workspace (flint_workspace_bytes(E, k, H, inter,
 *   inter_shared)), initialised once. A wait that runs out (the budget of
 *   flint_workspace_set_wait_budget, 2 s by default) records FLINT_ERR_TIMEOUT
 *   in the status word instead of hanging; flint_workspace_check reports it
 *   and re-initialises the workspace.
 *   flags: FLINT_PDL lets the launch overlap the previous kernel of the stream
 *   (this kernel waits for it before reading x or the workspace).
 *   next: the next layer's ranges to pull into L2 (above), or NULL.
 *   Errors: FLINT_ERR_INVALID_ARG for a misaligned or oversized prefetch
 *   range; FLINT_ERR_UNSUPPORTED when one CTA's shared memory cannot hold
 *   the layer's working set, the device cannot co-schedule one CTA per SM, or
 *   the experts are not NVFP4.
 */
flint_status_t flint_moe_layer(const flint_bf16* x, int T, const flint_bf16* router_w, int E, const float* bias,
                               int k, const flint_experts* routed, const flint_experts* shared, int32_t* ids,
                               float* weights, flint_bf16* y, void* ws, size_t ws_bytes,
                               const flint_l2_prefetch* next, unsigned flags, void* stream);

/* ------------------------------------------------------------------------ */
/* Residual stream of the decode stack                                       */
/* ------------------------------------------------------------------------ */
/*
 * "vLLM 宣布首日支持 Recursive 的 Flint ...", section "Flint 是什么": the model
 * is a pre-norm Transformer of 49 blocks, 2 dense MLP blocks then 47 MoE
 * blocks, on a hidden size of 2048; "Day-0 Support for Flint on vLLM",
 * section "Optimizations": norm kernels that follow the reference's rounding.
 * Ahead of every block, per token:
 *   r' = bf16(r + y)                                 (r' = r when y is NULL)
 *   x  = bf16(r' / sqrt(mean(r'^2) + eps) * gamma)   (gamma = 1 when NULL)
 * in FP32; r' is the residual stream the next block adds its output to.
 */
typedef struct flint_norm {
    const flint_bf16* residual;  /* r [T, H], required */
    const flint_bf16* y;         /* the previous block's output [T, H], or NULL */
    const flint_bf16* gamma;     /* [H], or NULL for all ones */
    float eps;                   /* >= 0 (the workloads use 1e-6) */
    float reserved;
    flint_bf16* residual_out;    /* r' [T, H], or NULL; must not overlap residual or y */
    flint_bf16* x_out;           /* x [T, H], or NULL */
} flint_norm;

/*
 * flint_residual_rmsnorm -- r' and x of the definition above, one small kernel
 * (one CTA per token). x_out is required.
 *   H % 256 == 0, H <= 32768; 1 <= T <= 8; all arrays 16-byte aligned.
 *   flags: FLINT_PDL (the kernel waits for the previous kernel before reading r and y).
 */
flint_status_t flint_residual_rmsnorm(const flint_norm* norm, int T, int H, unsigned flags, void* stream);

/*
 * flint_moe_block -- one pre-norm MoE block in ONE kernel: the residual add +
 * RMSNorm above, fused into the input staging of flint_moe_layer (every CTA
 * normalises the whole input itself; no extra launch, no extra barrier), then
 * the MoE layer on x. Arguments as flint_moe_layer, with `norm` in place of x
 * (norm->x_out may be NULL; when given, x is written too). y must not overlap
 * norm->residual, norm->y or norm->residual_out. Chained blocks alternate two
 * residual buffers (a block reads one and writes the other).
 */
flint_status_t flint_moe_block(const flint_norm* norm, int T, const flint_bf16* router_w, int E, const float* bias,
                               int k, const flint_experts* routed, const flint_experts* shared, int32_t* ids,
                               float* weights, flint_bf16* y, void* ws, size_t ws_bytes,
                               const flint_l2_prefetch* next, unsigned flags, void* stream);

/* ------------------------------------------------------------------------ */
/* Prefill: the MoE layer over many tokens, on the tensor cores               */
/* ------------------------------------------------------------------------ */
/*
 * flint_moe_prefill -- the same MoE layer as flint_moe_layer over T tokens at
 * once ("Day-0 Support for Flint on vLLM", section "Optimizations": the
 * MoE-kernel rewrite that reads only the selected experts' weights was also
 * the largest gain of the 8K-token prefill). Same arithmetic and rounding
 * points as the decode path; the contractions run on the 5th-generation
 * tensor cores (tcgen05.mma, bf16 operands with the NVFP4 weights
 * dequantised exactly in shared memory, FP32 accumulation in tensor memory):
 * router GEMM -> sigmoid top-k per token -> (token, rank) pairs sorted by
 * expert (token order kept within an expert) -> grouped gate/up GEMM + SiLU ->
 * grouped down GEMM -> y = bf16(sum_j w_j d_j + d_shared) gathered per token
 * (no atomics: deterministic). Eight launches in stream order.
 *   x [T, H] bf16, T >= 1; router_w [E, H] bf16, E % 16 == 0, E <= 1024;
 *   bias [E] or NULL; 1 <= k <= min(8, E); NVFP4 experts only (H % 1024 == 0,
 *   I % 256 == 0); shared may be NULL. ids [T, k], weights [T, k], y [T, H] out.
 *   ws: flint_prefill_workspace_bytes(...) bytes, 256-byte aligned,
 *   initialised once (flint_workspace_init); it holds the logits, the sort and
 *   the intermediate h and d of every (token, rank) pair.
 *   flags: 0 (PDL is not used on this path).
 *   A timed-out wait inside a GEMM is reported by flint_workspace_check.
 */
size_t flint_prefill_workspace_bytes(int tokens, int num_experts, int top_k, int hidden, int inter, int inter_shared);
flint_status_t flint_moe_prefill(const flint_bf16* x, int T, const flint_bf16* router_w, int E, const float* bias,
                                 int k, const flint_experts* routed, const flint_experts* shared, int32_t* ids,
                                 float* weights, flint_bf16* y, void* ws, size_t ws_bytes, unsigned flags,
                                 void* stream);

/* ------------------------------------------------------------------------ */
/* Dense GEMV on packed weights                                              */
/* ------------------------------------------------------------------------ */

typedef struct flint_packed {
    int32_t dtype;        /* FLINT_DTYPE_NVFP4 */
    int32_t rows;         /* N */
    int32_t cols;         /* K: % 1024 == 0 */
    int32_t reserved;
    const void* data;     /* [N, K] kernel layout */
    const float* tensor_scale; /* FP32: [1] (epilogue NONE) or [2] gate, up (SWIGLU) */
} flint_packed;

/*
 * flint_dense_gemv -- small-batch dense GEMV on packed NVFP4 weights
 * ("Optimizations": small-batch dense GEMV on the same packed NVFP4 weights).
 *   epilogue NONE:   y [T, N] = bf16(ts * W x)
 *   epilogue SWIGLU: rows [0, N/2) of W are the gate projection, rows
 *                    [N/2, N) the up projection; y [T, N/2] =
 *                    bf16(silu(bf16(ts0 * Wg x)) * bf16(ts1 * Wu x)).
 *   x [T, K] bf16, 1 <= T <= 8. ws may be NULL; when given (any size >= 256
 *   bytes, initialised) a timed-out wait is recorded in its status word.
 *   One kernel per group of tokens whose FP32 copy fits in shared memory
 *   beside the weight ring (all 8 tokens up to K = 4096).
 */
flint_status_t flint_dense_gemv(const flint_bf16* x, int T, const flint_packed* W, int epilogue, flint_bf16* y,
                                void* ws, size_t ws_bytes, unsigned flags, void* stream);

/* ------------------------------------------------------------------------ */
/* Diagnostics                                                               */
/* ------------------------------------------------------------------------ */

/* Text of the last error on this thread ("" if none). */
const char* flint_last_error(void);
const char* flint_status_string(flint_status_t status);

/* Self-test of the bounded-wait path: launches one CTA that waits on an
 * mbarrier nothing will complete, gives up after budget_ns nanoseconds and
 * records a timeout in the workspace status word, which flint_workspace_check
 * then reports as FLINT_ERR_TIMEOUT. Faults nothing; the context stays usable. */
flint_status_t flint_selftest_wait_timeout(void* ws, size_t ws_bytes, uint64_t budget_ns, void* stream);

/*
 * flint_selftest_lose_cta -- test hook for the fused layer's failure path
 * (no counterpart in the method). On the next flint_moe_layer /
 * flint_moe_block call with this workspace (or flint_moe_decode where it runs
 * as one kernel), CTA `cta` publishes neither its
 * router scores nor its count of finished gate/up rows, as if it had been
 * lost: the bounded waits for them (in the other CTAs, and in itself) run out
 * (after the budget of flint_workspace_set_wait_budget), the
 * kernel records FLINT_ERR_TIMEOUT and every CTA returns. Nothing faults or
 * hangs. flint_workspace_check then reports the timeout and re-initialises the
 * workspace, which also clears the hook. Synchronises `stream`.
 */
flint_status_t flint_selftest_lose_cta(void* ws, size_t ws_bytes, int cta, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FLINT_H */
