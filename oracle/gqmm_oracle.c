/*
 * gqmm_oracle.c -- plain, slow CPU oracle for the quantized MoE gather matmul.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call this
 * file: only the test suite, the package's smoke check and the benchmark's CPU-baseline
 * leg use it.  It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes, step by step, as the pages state the problem:
 *
 *  1. Affine group quantization.  The issue "[CUDA] gather_qmm ~24x slower than
 *     equal-FLOPs quantized_matmul on GB10 (sm_121)" (ml-explore/mlx #4339), section
 *     "Kernel microbenchmark", quantizes W with mx.quantize(w, group_size=64, bits=4).
 *     The pages never print that function's formula; the reading taken here is the
 *     standard affine min/max one: for each group of 64 consecutive weights along H,
 *         scale = (max - min) / 15,  bias = min,
 *         q     = clamp(round((w - bias) / scale), 0, 15),
 *     two 4-bit codes per byte, the even element in the low nibble, and w ~ scale*q + bias.
 *     Arithmetic is IEEE float32; scale and bias are stored as bfloat16 (round to nearest
 *     even) and the codes are computed from the STORED scale and bias; round() is
 *     round-half-to-even; a constant group (max == min) stores scale 0 and codes 0.
 *
 *  2. Dequantization in float64:  w_hat = (double)scale * q + (double)bias.
 *
 *  3. Routing sort.  mlxcel #629 "perf(cuda/moe): fix MoE prefill collapse", implementation
 *     plan item 4b: sort tokens by expert so each expert owns one contiguous block.  Here:
 *     a stable counting sort of the flat rows i = t*A + a by key idx[i]; keys >= E (invalid
 *     routing) are collected after every valid row, in row order.  offsets[e] is the number
 *     of valid rows whose expert is < e, offsets[E] the number of valid rows, and
 *     perm[offsets[e] + k] is the k-th smallest flat row routed to expert e.
 *
 *  4. Gather matmul (mlx #4339, "Kernel microbenchmark": mx.gather_qmm(x, wq, sc, bs,
 *     rhs_indices=idx, transpose=True, ...)): for every flat row i and output column f,
 *         y[i, f] = sum_h (double)x[i, h] * w_hat[idx[i], f, h],
 *     accumulated in float64 in increasing h.  A row whose index is >= E yields zeros.
 *     The sorted_indices flag is a performance hint only (same issue, "Describe the bug":
 *     it makes no measurable difference), so the oracle has no such argument.
 *
 * Threads split the rows of step 4 and the groups of step 1; that changes no arithmetic.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define EXPORT __attribute__((visibility("default")))

/* ---- bfloat16 <-> float32, written from the IEEE-754 definitions ------------------------- */

static float bf16_to_f32(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round a float32 to the nearest bfloat16, ties to even (keeps the top 16 bits). */
static uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u); /* quiet NaN */
    uint32_t lower = u & 0xffffu;
    uint32_t upper = u >> 16;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
    return (uint16_t)upper;
}

EXPORT int oracle_nthreads_default(void) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/* ---- 1. quantize -------------------------------------------------------------------------- */

typedef struct {
    const uint16_t* w;
    int64_t H, gs, n_groups_total, g_begin, g_end;
    uint8_t* wq;
    uint16_t* scales;
    uint16_t* biases;
} quant_job;

static void quantize_group(const quant_job* J, int64_t gi) {
    const int64_t G = J->H / J->gs;
    const int64_t row = gi / G, g = gi % G;
    const uint16_t* src = J->w + row * J->H + g * J->gs;

    float mn = bf16_to_f32(src[0]), mx = mn;
    for (int64_t k = 1; k < J->gs; ++k) {
        float v = bf16_to_f32(src[k]);
        if (v < mn) mn = v;
        if (v > mx) mx = v;
    }
    float range = mx - mn;              /* float32 subtraction */
    float scale32 = range / 15.0f;      /* float32 IEEE division */
    uint16_t s_b = f32_to_bf16_rne(scale32);
    uint16_t b_b = f32_to_bf16_rne(mn); /* mn is already a bfloat16 value: exact */
    float s = bf16_to_f32(s_b), b = bf16_to_f32(b_b);
    J->scales[gi] = s_b;
    J->biases[gi] = b_b;

    uint8_t* dst = J->wq + row * (J->H / 2) + g * (J->gs / 2);
    for (int64_t k = 0; k < J->gs; k += 2) {
        int q[2];
        for (int j = 0; j < 2; ++j) {
            if (s == 0.0f) {
                q[j] = 0;
            } else {
                float v = bf16_to_f32(src[k + j]);
                float t = (v - b) / s;  /* float32 subtract, float32 divide */
                float r = rintf(t);     /* round half to even (default rounding mode) */
                int qi = (int)r;
                if (qi < 0) qi = 0;
                if (qi > 15) qi = 15;
                q[j] = qi;
            }
        }
        dst[k / 2] = (uint8_t)(q[0] | (q[1] << 4));
    }
}

static void* quant_worker(void* arg) {
    quant_job* J = (quant_job*)arg;
    for (int64_t gi = J->g_begin; gi < J->g_end; ++gi) quantize_group(J, gi);
    return NULL;
}

/* w: bf16 [rows, H]; wq: u8 [rows, H/2]; scales, biases: bf16 [rows, H/gs]. bits must be 4.
 * Returns 0, or -1 on a bad argument. */
EXPORT int oracle_quantize(const uint16_t* w, int64_t rows, int64_t H, int group_size, int bits,
                           uint8_t* wq, uint16_t* scales, uint16_t* biases, int nthreads) {
    if (bits != 4 || group_size <= 0 || group_size % 2 || H % group_size || rows < 0) return -1;
    const int64_t total = rows * (H / group_size);
    if (nthreads <= 0) nthreads = oracle_nthreads_default();
    if (nthreads > 256) nthreads = 256;
    if (total < 4096) nthreads = 1;
    pthread_t th[256];
    quant_job jobs[256];
    for (int t = 0; t < nthreads; ++t) {
        quant_job J = {w, H, group_size, total, total * t / nthreads, total * (t + 1) / nthreads,
                       wq, scales, biases};
        jobs[t] = J;
    }
    if (nthreads == 1) {
        quant_worker(&jobs[0]);
        return 0;
    }
    for (int t = 0; t < nthreads; ++t) pthread_create(&th[t], NULL, quant_worker, &jobs[t]);
    for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
    return 0;
}

/* ---- 2. dequantize ------------------------------------------------------------------------ */

static inline double dequant_one(const uint8_t* wq_row, const uint16_t* s_row, const uint16_t* b_row,
                                 int64_t h, int64_t gs) {
    uint8_t byte = wq_row[h / 2];
    int q = (h % 2 == 0) ? (byte & 0x0f) : (byte >> 4);
    double s = (double)bf16_to_f32(s_row[h / gs]);
    double b = (double)bf16_to_f32(b_row[h / gs]);
    return s * (double)q + b;
}

/* w_hat: float64 [rows, H] */
EXPORT int oracle_dequantize(const uint8_t* wq, const uint16_t* scales, const uint16_t* biases,
                             int64_t rows, int64_t H, int group_size, double* w_hat) {
    if (group_size <= 0 || H % group_size) return -1;
    const int64_t G = H / group_size;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t h = 0; h < H; ++h)
            w_hat[r * H + h] = dequant_one(wq + r * (H / 2), scales + r * G, biases + r * G, h, group_size);
    return 0;
}

/* ---- 3. route sort ------------------------------------------------------------------------ */

/* idx: u32 [n]; perm: i32 [n]; offsets: i32 [E+1].  Returns the number of rows whose
 * index is >= E (0 when the routing is valid), or -1 on a bad argument. */
EXPORT int64_t oracle_route_sort(const uint32_t* idx, int64_t n, int E, int32_t* perm, int32_t* offsets) {
    if (E <= 0 || n < 0) return -1;
    int64_t* count = (int64_t*)calloc((size_t)E + 1, sizeof(int64_t));
    int64_t* next = (int64_t*)calloc((size_t)E + 1, sizeof(int64_t));
    if (!count || !next) { free(count); free(next); return -1; }
    for (int64_t i = 0; i < n; ++i) {
        int64_t key = idx[i] < (uint32_t)E ? (int64_t)idx[i] : (int64_t)E;
        count[key] += 1;
    }
    int64_t run = 0;
    for (int e = 0; e <= E; ++e) {
        next[e] = run;
        if (e < E) offsets[e] = (int32_t)run;
        run += count[e];
    }
    offsets[E] = (int32_t)next[E];
    for (int64_t i = 0; i < n; ++i) {
        int64_t key = idx[i] < (uint32_t)E ? (int64_t)idx[i] : (int64_t)E;
        perm[next[key]++] = (int32_t)i;
    }
    int64_t bad = count[E];
    free(count);
    free(next);
    return bad;
}

/* ---- 4. gather matmul --------------------------------------------------------------------- */

typedef struct {
    const uint16_t* x;
    const uint8_t* wq;
    const uint16_t* scales;
    const uint16_t* biases;
    const uint32_t* idx; /* NULL: every row uses expert 0 */
    const int64_t* rows; /* NULL: rows 0..n_rows-1 */
    int64_t n_rows, H, F, E, gs;
    double* y;           /* [n_rows, F] */
    int64_t r_begin, r_end;
} gemm_job;

static void* gemm_worker(void* arg) {
    gemm_job* J = (gemm_job*)arg;
    const int64_t H = J->H, F = J->F, G = H / J->gs;
    double* xrow = (double*)malloc(sizeof(double) * (size_t)H);
    if (!xrow) return NULL;
    for (int64_t rr = J->r_begin; rr < J->r_end; ++rr) {
        const int64_t i = J->rows ? J->rows[rr] : rr;
        double* out = J->y + rr * F;
        const uint32_t e = J->idx ? J->idx[i] : 0u;
        if (e >= (uint32_t)J->E) {
            for (int64_t f = 0; f < F; ++f) out[f] = 0.0;
            continue;
        }
        for (int64_t h = 0; h < H; ++h) xrow[h] = (double)bf16_to_f32(J->x[i * H + h]);
        for (int64_t f = 0; f < F; ++f) {
            const int64_t wr = (int64_t)e * F + f;
            const uint8_t* wq_row = J->wq + wr * (H / 2);
            const uint16_t* s_row = J->scales + wr * G;
            const uint16_t* b_row = J->biases + wr * G;
            double acc = 0.0;
            for (int64_t h = 0; h < H; ++h) acc += xrow[h] * dequant_one(wq_row, s_row, b_row, h, J->gs);
            out[f] = acc;
        }
    }
    free(xrow);
    return NULL;
}

static int run_gemm(gemm_job base, int64_t n_rows, int nthreads) {
    if (nthreads <= 0) nthreads = oracle_nthreads_default();
    if (nthreads > 256) nthreads = 256;
    if (nthreads > n_rows) nthreads = (int)(n_rows > 0 ? n_rows : 1);
    pthread_t th[256];
    gemm_job jobs[256];
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = base;
        jobs[t].r_begin = n_rows * t / nthreads;
        jobs[t].r_end = n_rows * (t + 1) / nthreads;
    }
    if (nthreads == 1) {
        gemm_worker(&jobs[0]);
        return 1;
    }
    for (int t = 0; t < nthreads; ++t) pthread_create(&th[t], NULL, gemm_worker, &jobs[t]);
    for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
    return nthreads;
}

/* x: bf16 [n, H]; wq: u8 [E, F, H/2]; scales, biases: bf16 [E, F, H/gs]; idx: u32 [n] or NULL
 * (then E must be 1); y: float64 [n, F].  Returns the thread count used, or -1. */
EXPORT int oracle_gather_qmm(const uint16_t* x, const uint8_t* wq, const uint16_t* scales,
                             const uint16_t* biases, const uint32_t* idx, int64_t n, int64_t H,
                             int64_t F, int64_t E, int group_size, int bits, double* y, int nthreads) {
    if (bits != 4 || group_size <= 0 || H % group_size || E <= 0 || (idx == NULL && E != 1)) return -1;
    gemm_job base = {x, wq, scales, biases, idx, NULL, n, H, F, E, group_size, y, 0, 0};
    return run_gemm(base, n, nthreads);
}

/* Same as oracle_gather_qmm for the listed flat rows only: y_rows is float64 [n_rows, F]. */
EXPORT int oracle_gather_qmm_rows(const uint16_t* x, const uint8_t* wq, const uint16_t* scales,
                                  const uint16_t* biases, const uint32_t* idx, int64_t H, int64_t F,
                                  int64_t E, int group_size, int bits, const int64_t* rows,
                                  int64_t n_rows, double* y_rows, int nthreads) {
    if (bits != 4 || group_size <= 0 || H % group_size || E <= 0 || (idx == NULL && E != 1)) return -1;
    gemm_job base = {x, wq, scales, biases, idx, rows, n_rows, H, F, E, group_size, y_rows, 0, 0};
    return run_gemm(base, n_rows, nthreads);
}
