/*
 * flint_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded CPU statement of what one small-batch decode
 * step of a Flint-style MoE layer with weight-only NVFP4 (W4A16) weights
 * computes. Only the test suite, the smoke check and the CPU-baseline leg of
 * the benchmark may load this library; the product path never does. It
 * shares no code, header, table or helper with the CUDA library.
 *
 * Sources (the pages describing the method):
 *  [Blog]  "Day-0 Support for Flint on vLLM", sections "Model architecture"
 *          (256 experts, sigmoid top-6, plus a shared expert; NVFP4 blocks
 *          repacked losslessly, run weight-only with BF16 activations; every
 *          kernel follows the reference's rounding points) and "Optimizations"
 *          (router and expert GEMVs that read only the selected experts;
 *          routing and the expert combine fused into the neighbouring GEMVs).
 *  [News]  "vLLM 宣布首日支持 Recursive 的 Flint ...", section
 *          "七个内核的依赖链：低延迟路径、无损重排与参考舍入" (64-value superblock =
 *          4 x [UE4M3 scale + 16 E2M1 codes], one FP32 scale per tensor, per
 *          expert for MoE weights; W4A16 with BF16 activations) and section
 *          "Flint 是什么" (256 routed experts, sigmoid top-6, one always-on
 *          shared expert, hidden size 2048).
 *
 * Precision ([Blog] "Model architecture": every kernel follows the
 * reference's rounding points; the reference accumulates in FP32): every dot
 * product is accumulated in FP32 in index order, one rounding per step (each
 * product of a weight and a bf16 activation is exact in FP32, so a fused
 * multiply-add and a multiply followed by an add give the same bits). The
 * per-tensor FP32 scale multiplies the FP32 sum once, in FP32. Values are
 * rounded to bf16, round to nearest even, exactly at the rounding points the
 * method states: after each GEMV (g, u, d), after silu(g)*u (h, with silu and
 * the product in FP32), and for the layer output y, whose combine is an FP32
 * multiply-add per routed expert in rank order, then the shared expert's d
 * added in FP32. Router logits stay FP32 (FP32 sum, FP32 bias add, FP32
 * sigmoid), and the top-k weights are the selected FP32 scores over their
 * FP32 sum in rank order.
 *
 * Readings of points the pages leave open (each listed in the design notes):
 *  - GGUF superblock byte order (36 bytes per 64 values): bytes 0..3 are the
 *    UE4M3 scales of sub-blocks 0..3; sub-block s's codes are bytes
 *    4+8s .. 4+8s+7; byte b of a sub-block holds value b in its low nibble and
 *    value b+8 in its high nibble. Superblocks run along a row; rows and
 *    matrices are contiguous.
 *  - UE4M3 bit 7 is not part of the unsigned format and is ignored.
 *  - Routing weights are the selected sigmoid scores renormalised to sum 1;
 *    the shared expert is added with weight 1.
 *  - Ties in the top-k go to the lower expert index.
 *
 * Parity status: the formats, the repack, the router and the GEMV are pinned
 * by the oracle self-tests (hand-decoded tables, a hand-derived superblock,
 * library routines, brute force and closed forms). The full layer is pinned
 * only through closed-form special cases and invariants.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define FO_OK 0
#define FO_BAD_ARG 1

#define FO_W_NVFP4 0
#define FO_W_BF16 1

#define FO_EPI_NONE 0
#define FO_EPI_SWIGLU 1

/* Threads of the OpenMP build (the same source compiled with -fopenmp, for
 * timing the oracle on all host cores); the plain build ignores them. */
int fo_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* Number formats                                                            */
/* ------------------------------------------------------------------------ */

/* E2M1 (OCP FP4): bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa.
 * Exponent 0 is subnormal: m * 0.5. Otherwise 2^(e-1) * (1 + m/2). */
double fo_e2m1_value(int code) {
    int s = (code >> 3) & 1;
    int e = (code >> 1) & 3;
    int m = code & 1;
    double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -mag : mag;
}

/* UE4M3: unsigned FP8 with a 4-bit exponent (bias 7) and a 3-bit mantissa.
 * Exponent 0 is subnormal: 2^-6 * m/8. Bits 0x7F encode NaN. Bit 7 ignored. */
double fo_ue4m3_value(int byte) {
    int b = byte & 0x7F;
    int e = (b >> 3) & 15;
    int m = b & 7;
    if (b == 0x7F) return NAN;
    if (e == 0) return ldexp(m / 8.0, -6);
    return ldexp(1.0 + m / 8.0, e - 7);
}

/* bfloat16 bits -> exact double. */
double fo_bf16_value(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bfloat16 (ties to even), directly, with no
 * intermediate rounding to float. bf16 keeps 8 significant bits, has the
 * float exponent range (normals down to 2^-126) and subnormals down to
 * 2^-133. */
uint16_t fo_bf16_round(double v) {
    if (isnan(v)) return 0x7FC0;
    int neg = signbit(v) ? 1 : 0;
    double a = fabs(v);
    uint16_t sign = neg ? 0x8000 : 0;
    if (a == 0.0) return sign;
    if (isinf(a)) return sign | 0x7F80;
    int e;
    frexp(a, &e);                 /* a = f * 2^e, f in [0.5, 1) */
    int q = e - 8;                /* weight of the last kept bit */
    if (q < -133) q = -133;       /* subnormal spacing */
    double r = nearbyint(ldexp(a, -q)); /* default mode: nearest, ties even */
    double res = ldexp(r, q);
    /* largest finite bf16 is (2 - 2^-7) * 2^127 */
    if (res > ldexp(2.0 - ldexp(1.0, -7), 127)) return sign | 0x7F80;
    float f = (float)res;         /* exact: res has <= 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | ((u >> 16) & 0x7FFF));
}

/* ------------------------------------------------------------------------ */
/* NVFP4 matrices: GGUF superblocks and the kernel layout                    */
/* ------------------------------------------------------------------------ */

#define FO_SB_VALUES 64
#define FO_SB_BYTES 36

int64_t fo_gguf_matrix_bytes(int64_t rows, int64_t cols) {
    return rows * (cols / FO_SB_VALUES) * FO_SB_BYTES;
}

/* Value (without the tensor scale) of element (row, col) of a GGUF NVFP4
 * matrix with `cols` columns, read straight from its superblock. */
static double gguf_elem(const uint8_t* src, int64_t cols, int64_t row, int64_t col) {
    int64_t sb = row * (cols / FO_SB_VALUES) + col / FO_SB_VALUES;
    const uint8_t* blk = src + sb * FO_SB_BYTES;
    int j = (int)(col % FO_SB_VALUES);
    int s = j / 16;               /* sub-block */
    int b = j % 16;               /* position in the sub-block */
    uint8_t byte = blk[4 + 8 * s + (b % 8)];
    int code = (b < 8) ? (byte & 15) : (byte >> 4);
    return fo_e2m1_value(code) * fo_ue4m3_value(blk[s]);
}

int fo_gguf_decode(const uint8_t* src, int64_t rows, int64_t cols, double* out) {
    if (!src || !out || rows < 0 || cols <= 0 || cols % FO_SB_VALUES) return FO_BAD_ARG;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) out[r * cols + c] = gguf_elem(src, cols, r, c);
    return FO_OK;
}

/* Kernel layout (the repack target), per row of a [rows, cols] matrix:
 *   bytes [0, cols/2)              codes: byte j holds column 2j in its low
 *                                  nibble and column 2j+1 in its high nibble
 *   bytes [cols/2, cols/2+cols/16) scales: byte b is the UE4M3 scale of
 *                                  columns 16b .. 16b+15
 *   zero padding up to the row stride, the next multiple of 16 bytes.
 * Rows are contiguous; matrix m starts at m * mat_stride bytes. */
int64_t fo_packed_row_stride(int64_t cols) {
    int64_t raw = cols / 2 + cols / 16;
    return (raw + 15) / 16 * 16;
}

static double packed_elem(const uint8_t* p, int64_t cols, int64_t row, int64_t col) {
    const uint8_t* r = p + row * fo_packed_row_stride(cols);
    uint8_t byte = r[col / 2];
    int code = (col % 2 == 0) ? (byte & 15) : (byte >> 4);
    return fo_e2m1_value(code) * fo_ue4m3_value(r[cols / 2 + col / 16]);
}

int fo_packed_decode(const uint8_t* p, int64_t rows, int64_t cols, double* out) {
    if (!p || !out || rows < 0 || cols <= 0 || cols % FO_SB_VALUES) return FO_BAD_ARG;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) out[r * cols + c] = packed_elem(p, cols, r, c);
    return FO_OK;
}

/* Lossless repack of n_mats GGUF matrices [rows, cols] into the kernel layout.
 * Moves every code nibble and scale byte; padding bytes are written as 0. */
int fo_repack(const uint8_t* src, int64_t n_mats, int64_t rows, int64_t cols,
              uint8_t* dst, int64_t dst_mat_stride) {
    if (!src || !dst || n_mats < 0 || rows < 0 || cols <= 0 || cols % FO_SB_VALUES) return FO_BAD_ARG;
    int64_t rs = fo_packed_row_stride(cols);
    if (dst_mat_stride == 0) dst_mat_stride = rows * rs;
    if (dst_mat_stride < rows * rs) return FO_BAD_ARG;
    int64_t src_mat = fo_gguf_matrix_bytes(rows, cols);
    for (int64_t m = 0; m < n_mats; ++m) {
        const uint8_t* sm = src + m * src_mat;
        uint8_t* dm = dst + m * dst_mat_stride;
        for (int64_t r = 0; r < rows; ++r) {
            uint8_t* dr = dm + r * rs;
            memset(dr, 0, (size_t)rs);
            for (int64_t c = 0; c < cols; ++c) {
                int64_t sb = r * (cols / FO_SB_VALUES) + c / FO_SB_VALUES;
                const uint8_t* blk = sm + sb * FO_SB_BYTES;
                int j = (int)(c % FO_SB_VALUES), s = j / 16, b = j % 16;
                uint8_t byte = blk[4 + 8 * s + (b % 8)];
                int code = (b < 8) ? (byte & 15) : (byte >> 4);
                if (c % 2 == 0) dr[c / 2] |= (uint8_t)code;
                else dr[c / 2] |= (uint8_t)(code << 4);
                if (b == 0) dr[cols / 2 + c / 16] = blk[s];
            }
        }
    }
    return FO_OK;
}

/* Inverse of fo_repack: kernel layout back to GGUF superblocks. */
int fo_unrepack(const uint8_t* dst, int64_t n_mats, int64_t rows, int64_t cols,
                int64_t dst_mat_stride, uint8_t* src) {
    if (!src || !dst || n_mats < 0 || rows < 0 || cols <= 0 || cols % FO_SB_VALUES) return FO_BAD_ARG;
    int64_t rs = fo_packed_row_stride(cols);
    if (dst_mat_stride == 0) dst_mat_stride = rows * rs;
    int64_t src_mat = fo_gguf_matrix_bytes(rows, cols);
    memset(src, 0, (size_t)(n_mats * src_mat));
    for (int64_t m = 0; m < n_mats; ++m) {
        uint8_t* sm = src + m * src_mat;
        const uint8_t* dm = dst + m * dst_mat_stride;
        for (int64_t r = 0; r < rows; ++r) {
            const uint8_t* dr = dm + r * rs;
            for (int64_t c = 0; c < cols; ++c) {
                int64_t sb = r * (cols / FO_SB_VALUES) + c / FO_SB_VALUES;
                uint8_t* blk = sm + sb * FO_SB_BYTES;
                int j = (int)(c % FO_SB_VALUES), s = j / 16, b = j % 16;
                int code = (c % 2 == 0) ? (dr[c / 2] & 15) : (dr[c / 2] >> 4);
                if (b < 8) blk[4 + 8 * s + b] |= (uint8_t)code;
                else blk[4 + 8 * s + (b - 8)] |= (uint8_t)(code << 4);
                if (b == 0) blk[s] = dr[cols / 2 + c / 16];
            }
        }
    }
    return FO_OK;
}

/* ------------------------------------------------------------------------ */
/* Weight access for a [rows, cols] matrix in either supported source type.  */
/* ------------------------------------------------------------------------ */

static double weight_elem(int wdtype, const void* w, int64_t cols, int64_t row, int64_t col) {
    if (wdtype == FO_W_NVFP4) return gguf_elem((const uint8_t*)w, cols, row, col);
    return fo_bf16_value(((const uint16_t*)w)[row * cols + col]);
}

static int64_t weight_matrix_bytes(int wdtype, int64_t rows, int64_t cols) {
    if (wdtype == FO_W_NVFP4) return fo_gguf_matrix_bytes(rows, cols);
    return rows * cols * 2;
}

/* acc = sum_k W[row, k] * x[k], in FP32, in index order: one rounding per
 * step (the product of a weight and a bf16 value is exact in FP32). */
static float dot_row(int wdtype, const void* w, int64_t cols, int64_t row, const float* x) {
    float acc = 0.0f;
    for (int64_t c = 0; c < cols; ++c) acc = fmaf((float)weight_elem(wdtype, w, cols, row, c), x[c], acc);
    return acc;
}

/* silu(g) = g / (1 + exp(-g)), in FP32. */
static float silu(float g) { return g / (1.0f + expf(-g)); }

/* ------------------------------------------------------------------------ */
/* Router: logits, sigmoid scores, top-k, renormalised weights               */
/* ------------------------------------------------------------------------ */

/* For each token t: logit[e] = sum_h x[t,h] * Wr[e,h] (+ bias[e]);
 * score[e] = sigmoid(logit[e]); ids = the k largest scores, ties to the lower
 * index, in descending score order; weights[j] = score[ids[j]] / sum of the k
 * selected scores. Selection runs on FP32 scores (see the header). */
int fo_router(const uint16_t* x, int T, int H, const uint16_t* wr, int E, const float* bias,
              int k, int32_t* ids, double* weights, float* scores) {
    if (!x || !wr || !ids || !weights || T < 0 || H <= 0 || E <= 0 || k <= 0 || k > E) return FO_BAD_ARG;
    float* s = (float*)malloc(sizeof(float) * (size_t)E);
    char* taken = (char*)malloc((size_t)E);
    if (!s || !taken) { free(s); free(taken); return FO_BAD_ARG; }
    for (int t = 0; t < T; ++t) {
        /* expert rows are independent (the OpenMP build splits them over threads) */
#pragma omp parallel for schedule(static)
        for (int e = 0; e < E; ++e) {
            float z = 0.0f;
            for (int h = 0; h < H; ++h)
                z = fmaf((float)fo_bf16_value(x[(int64_t)t * H + h]), (float)fo_bf16_value(wr[(int64_t)e * H + h]), z);
            if (bias) z = z + bias[e];
            s[e] = 1.0f / (1.0f + expf(-z));
            if (scores) scores[(int64_t)t * E + e] = s[e];
        }
        memset(taken, 0, (size_t)E);
        float sum = 0.0f;
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || s[e] > s[best]) best = e; /* strict: ties keep the lower index */
            }
            taken[best] = 1;
            ids[t * k + j] = best;
            sum += s[best];
        }
        for (int j = 0; j < k; ++j) weights[t * k + j] = (double)(s[ids[t * k + j]] / sum);
    }
    free(s);
    free(taken);
    return FO_OK;
}

/* ------------------------------------------------------------------------ */
/* One SwiGLU expert for one token                                           */
/* ------------------------------------------------------------------------ */

/* g[i] = bf16(ts_g * sum_h Wg[i,h] x[h]);  u[i] = bf16(ts_u * sum_h Wu[i,h] x[h])
 * h[i] = bf16(silu(g[i]) * u[i])
 * d[n] = bf16(ts_d * sum_i Wd[n,i] h[i])
 * (sums, scale products, silu and its product in FP32). Any of g, u, hh may
 * be NULL. */
int fo_expert(const uint16_t* x, int H, int I, int wdtype, const void* gate, const void* up,
              const void* down, double ts_g, double ts_u, double ts_d,
              uint16_t* g, uint16_t* u, uint16_t* hh, uint16_t* d) {
    if (!x || !gate || !up || !down || !d || H <= 0 || I <= 0) return FO_BAD_ARG;
    float* xd = (float*)malloc(sizeof(float) * (size_t)H);
    float* hd = (float*)malloc(sizeof(float) * (size_t)I);
    if (!xd || !hd) { free(xd); free(hd); return FO_BAD_ARG; }
    const float sg = (float)ts_g, su = (float)ts_u, sd = (float)ts_d;
    for (int c = 0; c < H; ++c) xd[c] = (float)fo_bf16_value(x[c]);
    /* Output rows are independent, and each is summed in index order by one
     * thread: the OpenMP build (rows split over threads) gives the same bits. */
#pragma omp parallel for schedule(static)
    for (int i = 0; i < I; ++i) {
        uint16_t gb = fo_bf16_round(sg * dot_row(wdtype, gate, H, i, xd));
        uint16_t ub = fo_bf16_round(su * dot_row(wdtype, up, H, i, xd));
        uint16_t hb = fo_bf16_round(silu((float)fo_bf16_value(gb)) * (float)fo_bf16_value(ub));
        if (g) g[i] = gb;
        if (u) u[i] = ub;
        if (hh) hh[i] = hb;
        hd[i] = (float)fo_bf16_value(hb);
    }
#pragma omp parallel for schedule(static)
    for (int n = 0; n < H; ++n) d[n] = fo_bf16_round(sd * dot_row(wdtype, down, I, n, hd));
    free(xd);
    free(hd);
    return FO_OK;
}

/* ------------------------------------------------------------------------ */
/* Expert part of the layer, given the routing                               */
/* ------------------------------------------------------------------------ */

/* Weights of all E routed experts are contiguous per matrix kind:
 *   gate: E x [I, H], up: E x [I, H], down: E x [H, I]
 * in GGUF NVFP4 (wdtype 0) or bf16 row-major (wdtype 1); ts is [E][3]
 * (gate, up, down) or NULL for 1.0. The shared expert (nullable) has the same
 * shapes with its own intermediate size Is and tensor scales sts[3].
 *
 * For each token t:
 *   y[t] = bf16( sum_{j<k} w[t,j] * d_{ids[t,j]}(x[t])  +  d_shared(x[t]) )
 * accumulated in FP32: a multiply-add per routed expert in rank order (one
 * rounding each), then the shared expert's d added. */
int fo_moe_experts(const uint16_t* x, int T, int H, const int32_t* ids, const float* w, int k,
                   int E, int I, int wdtype, const void* gate, const void* up, const void* down,
                   const float* ts, int Is, const void* sgate, const void* sup, const void* sdown,
                   const float* sts, uint16_t* y) {
    if (!x || !ids || !w || !y || T < 0 || H <= 0 || k <= 0 || E <= 0 || I <= 0) return FO_BAD_ARG;
    int64_t gb = weight_matrix_bytes(wdtype, I, H);
    int64_t db = weight_matrix_bytes(wdtype, H, I);
    uint16_t* d = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)H);
    float* acc = (float*)malloc(sizeof(float) * (size_t)H);
    if (!d || !acc) { free(d); free(acc); return FO_BAD_ARG; }
    int rc = FO_OK;
    for (int t = 0; t < T && rc == FO_OK; ++t) {
        const uint16_t* xt = x + (int64_t)t * H;
        for (int n = 0; n < H; ++n) acc[n] = 0.0f;
        for (int j = 0; j < k; ++j) {
            int e = ids[t * k + j];
            if (e < 0 || e >= E) { rc = FO_BAD_ARG; break; }
            double tg = ts ? ts[3 * e + 0] : 1.0, tu = ts ? ts[3 * e + 1] : 1.0, td = ts ? ts[3 * e + 2] : 1.0;
            rc = fo_expert(xt, H, I, wdtype, (const uint8_t*)gate + e * gb, (const uint8_t*)up + e * gb,
                           (const uint8_t*)down + e * db, tg, tu, td, NULL, NULL, NULL, d);
            if (rc != FO_OK) break;
            for (int n = 0; n < H; ++n) acc[n] = fmaf(w[t * k + j], (float)fo_bf16_value(d[n]), acc[n]);
        }
        if (rc == FO_OK && sgate) {
            double tg = sts ? sts[0] : 1.0, tu = sts ? sts[1] : 1.0, td = sts ? sts[2] : 1.0;
            rc = fo_expert(xt, H, Is, wdtype, sgate, sup, sdown, tg, tu, td, NULL, NULL, NULL, d);
            for (int n = 0; n < H && rc == FO_OK; ++n) acc[n] += (float)fo_bf16_value(d[n]);
        }
        for (int n = 0; n < H; ++n) y[(int64_t)t * H + n] = fo_bf16_round(acc[n]);
    }
    free(d);
    free(acc);
    return rc;
}

/* The whole layer: router, then the experts with the router's own weights. */
int fo_moe_layer(const uint16_t* x, int T, int H, const uint16_t* wr, int E, const float* bias, int k,
                 int I, int wdtype, const void* gate, const void* up, const void* down, const float* ts,
                 int Is, const void* sgate, const void* sup, const void* sdown, const float* sts,
                 int32_t* ids, float* weights, uint16_t* y) {
    if (T <= 0 || k <= 0) return FO_BAD_ARG;
    double* wd = (double*)malloc(sizeof(double) * (size_t)(T * k));
    if (!wd) return FO_BAD_ARG;
    int rc = fo_router(x, T, H, wr, E, bias, k, ids, wd, NULL);
    if (rc == FO_OK) {
        for (int i = 0; i < T * k; ++i) weights[i] = (float)wd[i];
        rc = fo_moe_experts(x, T, H, ids, weights, k, E, I, wdtype, gate, up, down, ts, Is, sgate, sup,
                            sdown, sts, y);
    }
    free(wd);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Dense GEMV on the same packed weights                                     */
/* ------------------------------------------------------------------------ */

/* epilogue NONE:   y[t, n] = bf16(ts[0] * sum_k W[n, k] x[t, k]),  n < N
 * epilogue SWIGLU: W is [N, K] with rows [0, N/2) the gate projection
 *                  (tensor scale ts[0]) and rows [N/2, N) the up projection
 *                  (ts[1]); y[t, i] = bf16(silu(g) * u), g and u rounded to
 *                  bf16 first, i < N/2.
 * Sums, scale products, silu and its product in FP32, as in fo_expert. */
int fo_dense_gemv(const uint16_t* x, int T, int K, int wdtype, const void* W, int N,
                  const float* ts, int epilogue, uint16_t* y) {
    if (!x || !W || !y || T < 0 || K <= 0 || N <= 0) return FO_BAD_ARG;
    if (epilogue == FO_EPI_SWIGLU && N % 2) return FO_BAD_ARG;
    float* xd = (float*)malloc(sizeof(float) * (size_t)K);
    if (!xd) return FO_BAD_ARG;
    for (int t = 0; t < T; ++t) {
        for (int c = 0; c < K; ++c) xd[c] = (float)fo_bf16_value(x[(int64_t)t * K + c]);
        if (epilogue == FO_EPI_NONE) {
            float s = ts ? ts[0] : 1.0f;
            for (int n = 0; n < N; ++n) y[(int64_t)t * N + n] = fo_bf16_round(s * dot_row(wdtype, W, K, n, xd));
        } else {
            int half = N / 2;
            float sg = ts ? ts[0] : 1.0f, su = ts ? ts[1] : 1.0f;
            for (int i = 0; i < half; ++i) {
                float g = (float)fo_bf16_value(fo_bf16_round(sg * dot_row(wdtype, W, K, i, xd)));
                float u = (float)fo_bf16_value(fo_bf16_round(su * dot_row(wdtype, W, K, half + i, xd)));
                y[(int64_t)t * half + i] = fo_bf16_round(silu(g) * u);
            }
        }
    }
    free(xd);
    return FO_OK;
}

/* ------------------------------------------------------------------------ */
/* Residual add + RMSNorm between the blocks of the decode stack             */
/* ------------------------------------------------------------------------ */

/* [News] section "Flint 是什么": Flint is a pre-norm Transformer of 49 blocks
 * (2 dense MLP blocks, then 47 MoE blocks) on a hidden size of 2048; [Blog]
 * section "Optimizations": norm kernels that follow the reference's rounding
 * points. The pages fix neither the norm's epsilon nor its scale vector, nor
 * its internal precision (the workloads use eps = 1e-6 and gamma = 1).
 * Per token t:
 *   r'[h] = bf16(r[h] + y[h])                  (r' = r when y is NULL)
 *   x[h]  = bf16(r'[h] / sqrt(mean_h(r'^2) + eps) * gamma[h])   (gamma = 1 when NULL)
 * in FP32 like every other step: the residual add, the sum of squares in
 * index order, the mean, the square root, its reciprocal and the products.
 * r_out (may be NULL) receives r'; x_out receives x. */
int fo_residual_rmsnorm(const uint16_t* r, const uint16_t* y, int T, int H, const uint16_t* gamma, double eps,
                        uint16_t* r_out, uint16_t* x_out) {
    if (!r || !x_out || T < 0 || H <= 0 || eps < 0.0) return FO_BAD_ARG;
    float* rr = (float*)malloc(sizeof(float) * (size_t)H);
    if (!rr) return FO_BAD_ARG;
    const float epsf = (float)eps;
    for (int t = 0; t < T; ++t) {
        float ss = 0.0f;
        for (int h = 0; h < H; ++h) {
            int64_t i = (int64_t)t * H + h;
            float v = (float)fo_bf16_value(r[i]);
            if (y) v = (float)fo_bf16_value(fo_bf16_round(v + (float)fo_bf16_value(y[i])));
            rr[h] = v;
            ss = fmaf(v, v, ss);
            if (r_out) r_out[i] = fo_bf16_round(v);
        }
        float inv = 1.0f / sqrtf(ss / (float)H + epsf);
        for (int h = 0; h < H; ++h) {
            float g = gamma ? (float)fo_bf16_value(gamma[h]) : 1.0f;
            x_out[(int64_t)t * H + h] = fo_bf16_round(rr[h] * inv * g);
        }
    }
    free(rr);
    return FO_OK;
}
