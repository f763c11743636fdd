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
 * Other affine bit widths (mlx PR #4023 "Pick BM from rows per expert in gather_qmm_rhs_nax",
 * the author's follow-up: the upstream tests run every mode, group size and bit width).  For
 * bits b in {2, 3, 4, 5, 6, 8} the same steps hold with 2^b - 1 levels in place of 15:
 *     scale = (max - min) / (2^b - 1),  q = clamp(round((w - bias) / scale), 0, 2^b - 1),
 * and a row's codes form one little-endian bit stream: element k occupies bits
 * [k*b, (k+1)*b) of the row, bit j of the stream being bit (j mod 8) of byte j / 8 (for
 * b = 4 this is the two-nibbles-per-byte layout above).  A row of H weights takes H*b/8 bytes.
 *
 * Block-scaled floating-point modes (mlx #4339, comment by nastya236 under "Activity": the
 * CUDA back end is to support mxfp8 and nvfp4 rather than affine).  The pages name the modes
 * without their definitions; these follow the published formats:
 *   element types  E2M1 (1 sign, 2 exponent, 1 mantissa bit, bias 1, largest 6, no inf/NaN) and
 *                  E4M3 (1 sign, 4 exponent, 3 mantissa bits, bias 7, largest 448, S.1111.111 NaN,
 *                  no inf), each with subnormals; scale types E8M0 (2^(c - 127), 255 = NaN) and E4M3.
 *   mxfp4 / mxfp8  (OCP Microscaling Formats v1.0): blocks of 32 consecutive weights along H share
 *                  an E8M0 scale X = 2^(floor(log2(amax)) - emax), emax = 2 for E2M1, 8 for E4M3
 *                  (X = 1 for an all-zero block); each element is w / X rounded to the element type,
 *                  to nearest with ties to even, saturating at the largest finite value.
 *   nvfp4          (NVIDIA's NVFP4): blocks of 16 share an E4M3 scale, and each tensor (each
 *                  expert's F x H weight here) has a float32 scale t = amax_tensor / (6 * 448)
 *                  (t = 1 for an all-zero tensor).  In float32: s = (amax_block / 6) / t, rounded to
 *                  E4M3 (nearest, ties to even, saturating) giving S; then each element is
 *                  w / (S * t) (float32 product and quotient) rounded to E2M1 (codes 0 when S * t
 *                  is 0).
 *   Dequantization in float64: w_hat = element * X  (mx) or element * S * t  (nvfp4).
 *   Codes: E2M1 two per byte as the 4-bit affine codes, E4M3 one per byte; scales one byte each,
 *   [rows, H/32] (mx) or [rows, H/16] (nvfp4); the nvfp4 tensor scales are float32, one per tensor.
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
    int bits;
} quant_job;

/* Bit stream of a row of codes: element k occupies bits [k*b, (k+1)*b), bit j of the stream
 * being bit (j mod 8) of byte j / 8.  The destination bits must start cleared. */
static void put_bits(uint8_t* row, int64_t bit0, int nbits, uint32_t value) {
    for (int i = 0; i < nbits; ++i)
        if ((value >> i) & 1u) row[(bit0 + i) / 8] |= (uint8_t)(1u << ((bit0 + i) % 8));
}

static uint32_t get_bits(const uint8_t* row, int64_t bit0, int nbits) {
    uint32_t v = 0;
    for (int i = 0; i < nbits; ++i) v |= (uint32_t)((row[(bit0 + i) / 8] >> ((bit0 + i) % 8)) & 1u) << i;
    return v;
}

static int bits_supported(int bits) {
    return bits == 2 || bits == 3 || bits == 4 || bits == 5 || bits == 6 || bits == 8;
}

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
    const int levels = (1 << J->bits) - 1;
    float range = mx - mn;              /* float32 subtraction */
    float scale32 = range / (float)levels;  /* float32 IEEE division */
    uint16_t s_b = f32_to_bf16_rne(scale32);
    uint16_t b_b = f32_to_bf16_rne(mn); /* mn is already a bfloat16 value: exact */
    float s = bf16_to_f32(s_b), b = bf16_to_f32(b_b);
    J->scales[gi] = s_b;
    J->biases[gi] = b_b;

    uint8_t* dst_row = J->wq + row * (J->H * J->bits / 8);
    for (int64_t k = 0; k < J->gs; ++k) {
        int q = 0;
        if (s != 0.0f) {
            float v = bf16_to_f32(src[k]);
            float t = (v - b) / s;  /* float32 subtract, float32 divide */
            float r = rintf(t);     /* round half to even (default rounding mode) */
            q = (int)r;
            if (q < 0) q = 0;
            if (q > levels) q = levels;
        }
        put_bits(dst_row, (g * J->gs + k) * J->bits, J->bits, (uint32_t)q);
    }
}

static void* quant_worker(void* arg) {
    quant_job* J = (quant_job*)arg;
    for (int64_t gi = J->g_begin; gi < J->g_end; ++gi) quantize_group(J, gi);
    return NULL;
}

/* w: bf16 [rows, H]; wq: u8 [rows, H*bits/8]; scales, biases: bf16 [rows, H/gs];
 * bits in {2, 3, 4, 5, 6, 8}.  Returns 0, or -1 on a bad argument. */
EXPORT int oracle_quantize(const uint16_t* w, int64_t rows, int64_t H, int group_size, int bits,
                           uint8_t* wq, uint16_t* scales, uint16_t* biases, int nthreads) {
    if (!bits_supported(bits) || group_size <= 0 || group_size % 8 || H % group_size || rows < 0) return -1;
    memset(wq, 0, (size_t)(rows * H * bits / 8));
    const int64_t total = rows * (H / group_size);
    if (nthreads <= 0) nthreads = oracle_nthreads_default();
    if (nthreads > 256) nthreads = 256;
    if (total < 4096) nthreads = 1;
    pthread_t th[256];
    quant_job jobs[256];
    for (int t = 0; t < nthreads; ++t) {
        quant_job J = {w, H, group_size, total, total * t / nthreads, total * (t + 1) / nthreads,
                       wq, scales, biases, bits};
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
                                 int64_t h, int64_t gs, int bits) {
    int q = (int)get_bits(wq_row, h * bits, bits);
    double s = (double)bf16_to_f32(s_row[h / gs]);
    double b = (double)bf16_to_f32(b_row[h / gs]);
    return s * (double)q + b;
}

/* w_hat: float64 [rows, H] */
EXPORT int oracle_dequantize(const uint8_t* wq, const uint16_t* scales, const uint16_t* biases,
                             int64_t rows, int64_t H, int group_size, int bits, double* w_hat) {
    if (!bits_supported(bits) || group_size <= 0 || H % group_size) return -1;
    const int64_t G = H / group_size;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t h = 0; h < H; ++h)
            w_hat[r * H + h] = dequant_one(wq + r * (H * bits / 8), scales + r * G, biases + r * G, h, group_size,
                                           bits);
    return 0;
}

/* ---- 1b, 2b. block-scaled floating-point formats ------------------------------------------ */

enum { MODE_AFFINE = 0, MODE_MXFP4 = 1, MODE_NVFP4 = 2, MODE_MXFP8 = 3 };

/* E2M1: sign bit 3, exponent bits 2-1 (bias 1), mantissa bit 0; exponent 0 is subnormal. */
static double e2m1_value(unsigned c) {
    const unsigned e = (c >> 1) & 3u, m = c & 1u;
    const double mag = e == 0 ? 0.5 * (double)m : ldexp(1.0 + 0.5 * (double)m, (int)e - 1);
    return (c & 8u) ? -mag : mag;
}

/* E4M3: sign bit 7, exponent bits 6-3 (bias 7), mantissa bits 2-0; exponent 0 is subnormal;
 * exponent 15 with mantissa 7 is NaN, and there are no infinities. */
static double e4m3_value(unsigned c) {
    const unsigned e = (c >> 3) & 15u, m = c & 7u;
    if (e == 15u && m == 7u) return NAN;
    const double mag = e == 0 ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, (int)e - 7);
    return (c & 0x80u) ? -mag : mag;
}

/* E8M0: 2^(c - 127); 255 is NaN. */
static double e8m0_value(unsigned c) { return c == 255u ? NAN : ldexp(1.0, (int)c - 127); }

/* The value nearest to v (ties to the even significand) of a binary floating-point type with
 * `man` stored mantissa bits and smallest normal exponent `emin` (below which the spacing stays
 * 2^(emin - man): subnormals), saturating at +-maxv.  Every step is exact in double for the
 * types used here. */
static double round_to_type(double v, int man, int emin, double maxv) {
    const double a = fabs(v);
    if (a == 0.0) return v;
    if (a >= maxv) return copysign(maxv, v);
    int ex;
    frexp(a, &ex);          /* a = f * 2^ex, f in [0.5, 1): floor(log2 a) = ex - 1 */
    int e = ex - 1;
    if (e < emin) e = emin;
    const double quantum = ldexp(1.0, e - man);
    double r = rint(a / quantum) * quantum;  /* a / quantum is exact; rint rounds half to even */
    if (r > maxv) r = maxv;
    return copysign(r, v);
}

/* Codes of finite values of each element type (the sign of a zero is kept). */
static unsigned e2m1_code(double r) {
    const unsigned sign = signbit(r) ? 8u : 0u;
    for (unsigned c = 0; c < 8; ++c)
        if (e2m1_value(c) == fabs(r)) return sign | c;
    return sign | 7u; /* not reached for values from round_to_type */
}

static unsigned e4m3_code(double r) {
    const unsigned sign = signbit(r) ? 0x80u : 0u;
    const double a = fabs(r);
    if (a == 0.0) return sign;
    int ex;
    frexp(a, &ex);
    const int e = ex - 1;
    if (e < -6) return sign | (unsigned)(a / ldexp(1.0, -9));             /* subnormal: m * 2^-9 */
    return sign | ((unsigned)(e + 7) << 3) | (unsigned)((a / ldexp(1.0, e) - 1.0) * 8.0);
}

static int mode_block(int mode) { return mode == MODE_NVFP4 ? 16 : 32; }
static int64_t mode_row_bytes(int mode, int64_t H) { return mode == MODE_MXFP8 ? H : H / 2; }

static unsigned fp_code_at(int mode, const uint8_t* row, int64_t h) {
    if (mode == MODE_MXFP8) return row[h];
    return (unsigned)get_bits(row, h * 4, 4);
}

static void fp_put_code(int mode, uint8_t* row, int64_t h, unsigned c) {
    if (mode == MODE_MXFP8) row[h] = (uint8_t)c;
    else put_bits(row, h * 4, 4, c);
}

/* One block of one row: amax, scale code, element codes. */
static void quantize_fp_block(int mode, const uint16_t* src, int nb, float tscale, uint8_t* row, int64_t h0,
                              uint8_t* scale_out) {
    float amax = 0.0f;
    for (int k = 0; k < nb; ++k) {
        const float a = fabsf(bf16_to_f32(src[k]));
        if (a > amax) amax = a;
    }
    if (mode == MODE_NVFP4) {
        const float s = (amax / 6.0f) / tscale;            /* float32 quotients */
        const double S = round_to_type((double)s, 3, -6, 448.0);
        *scale_out = (uint8_t)e4m3_code(S);
        const float denom = (float)S * tscale;             /* float32 product */
        for (int k = 0; k < nb; ++k) {
            unsigned c = 0;
            if (denom != 0.0f) c = e2m1_code(round_to_type((double)(bf16_to_f32(src[k]) / denom), 1, 0, 6.0));
            fp_put_code(mode, row, h0 + k, c);
        }
        return;
    }
    const int emax = mode == MODE_MXFP8 ? 8 : 2;
    int k_exp = 0;
    if (amax > 0.0f) {
        int ex;
        frexp((double)amax, &ex);
        k_exp = (ex - 1) - emax;
        if (k_exp < -127) k_exp = -127;
        if (k_exp > 127) k_exp = 127;
    }
    *scale_out = (uint8_t)(k_exp + 127);
    const double X = ldexp(1.0, k_exp);
    for (int k = 0; k < nb; ++k) {
        const double v = (double)bf16_to_f32(src[k]) / X;  /* exact: a power of two */
        const unsigned c = mode == MODE_MXFP8 ? e4m3_code(round_to_type(v, 3, -6, 448.0))
                                              : e2m1_code(round_to_type(v, 1, 0, 6.0));
        fp_put_code(mode, row, h0 + k, c);
    }
}

/* w: bf16 [rows, H]; wq: u8 [rows, H/2] (mxfp4, nvfp4) or [rows, H] (mxfp8); scales: u8
 * [rows, H/32] (mx) or [rows, H/16] (nvfp4); tscale: float32 [rows / rows_per_tensor] (nvfp4,
 * written here; NULL otherwise).  Returns 0, or -1 on a bad argument. */
EXPORT int oracle_quantize_fp(const uint16_t* w, int64_t rows, int64_t H, int mode, int64_t rows_per_tensor,
                              uint8_t* wq, uint8_t* scales, float* tscale) {
    if (mode < MODE_MXFP4 || mode > MODE_MXFP8 || rows < 0 || H <= 0) return -1;
    const int nb = mode_block(mode);
    if (H % nb) return -1;
    if (mode == MODE_NVFP4 && (!tscale || rows_per_tensor <= 0 || rows % rows_per_tensor)) return -1;
    const int64_t rb = mode_row_bytes(mode, H);
    memset(wq, 0, (size_t)(rows * rb));
    for (int64_t r0 = 0; r0 < rows; r0 += (mode == MODE_NVFP4 ? rows_per_tensor : rows)) {
        const int64_t r1 = mode == MODE_NVFP4 ? r0 + rows_per_tensor : rows;
        float t = 1.0f;
        if (mode == MODE_NVFP4) {
            float amax = 0.0f;
            for (int64_t i = r0 * H; i < r1 * H; ++i) {
                const float a = fabsf(bf16_to_f32(w[i]));
                if (a > amax) amax = a;
            }
            t = amax > 0.0f ? amax / 2688.0f : 1.0f;  /* 6 * 448, float32 quotient */
            tscale[r0 / rows_per_tensor] = t;
        }
        for (int64_t r = r0; r < r1; ++r)
            for (int64_t h0 = 0; h0 < H; h0 += nb)
                quantize_fp_block(mode, w + r * H + h0, nb, t, wq + r * rb, h0, scales + r * (H / nb) + h0 / nb);
    }
    return 0;
}

/* Dequantized weight h of row `row` in any mode, float64. */
typedef struct {
    int mode, bits;
    int64_t H, gs;
    const uint8_t* wq;
    const void* scales;   /* bf16 (affine) or u8 (floating-point modes) */
    const uint16_t* biases;
    const float* tscale;  /* nvfp4: one per rows_per_tensor rows */
    int64_t rows_per_tensor;
} qweights;

static double w_hat_at(const qweights* W, int64_t row, int64_t h) {
    const int64_t H = W->H;
    if (W->mode == MODE_AFFINE) {
        const int64_t G = H / W->gs;
        return dequant_one(W->wq + row * (H * W->bits / 8), (const uint16_t*)W->scales + row * G, W->biases + row * G,
                           h, W->gs, W->bits);
    }
    const int nb = mode_block(W->mode);
    const uint8_t* row_codes = W->wq + row * mode_row_bytes(W->mode, H);
    const unsigned c = fp_code_at(W->mode, row_codes, h);
    const unsigned sc = ((const uint8_t*)W->scales)[row * (H / nb) + h / nb];
    if (W->mode == MODE_MXFP4) return e2m1_value(c) * e8m0_value(sc);
    if (W->mode == MODE_MXFP8) return e4m3_value(c) * e8m0_value(sc);
    return e2m1_value(c) * e4m3_value(sc) * (double)W->tscale[row / W->rows_per_tensor];
}

/* w_hat: float64 [rows, H] */
EXPORT int oracle_dequantize_fp(const uint8_t* wq, const uint8_t* scales, const float* tscale, int64_t rows, int64_t H,
                                int mode, int64_t rows_per_tensor, double* w_hat) {
    if (mode < MODE_MXFP4 || mode > MODE_MXFP8 || H % mode_block(mode)) return -1;
    if (mode == MODE_NVFP4 && (!tscale || rows_per_tensor <= 0)) return -1;
    qweights W = {mode, 0, H, mode_block(mode), wq, scales, NULL, tscale, rows_per_tensor};
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t h = 0; h < H; ++h) w_hat[r * H + h] = w_hat_at(&W, r, h);
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
    qweights W;          /* the experts' weights: row e*F + f */
    const uint32_t* idx; /* NULL: every row uses expert 0 */
    const int64_t* rows; /* NULL: rows 0..n_rows-1 */
    int64_t n_rows, H, F, E;
    double* y;           /* [n_rows, F] */
    int64_t r_begin, r_end;
} gemm_job;

static void* gemm_worker(void* arg) {
    gemm_job* J = (gemm_job*)arg;
    const int64_t H = J->H, F = J->F;
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
            double acc = 0.0;
            for (int64_t h = 0; h < H; ++h) acc += xrow[h] * w_hat_at(&J->W, wr, h);
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

/* x: bf16 [n, H]; wq: u8 [E, F, H*bits/8]; scales, biases: bf16 [E, F, H/gs]; idx: u32 [n] or
 * NULL (then E must be 1); y: float64 [n, F].  Returns the thread count used, or -1. */
EXPORT int oracle_gather_qmm(const uint16_t* x, const uint8_t* wq, const uint16_t* scales,
                             const uint16_t* biases, const uint32_t* idx, int64_t n, int64_t H,
                             int64_t F, int64_t E, int group_size, int bits, double* y, int nthreads) {
    if (!bits_supported(bits) || group_size <= 0 || H % group_size || E <= 0 || (idx == NULL && E != 1)) return -1;
    qweights W = {MODE_AFFINE, bits, H, group_size, wq, scales, biases, NULL, 1};
    gemm_job base = {x, W, idx, NULL, n, H, F, E, y, 0, 0};
    return run_gemm(base, n, nthreads);
}

/* Same as oracle_gather_qmm for the listed flat rows only: y_rows is float64 [n_rows, F]. */
EXPORT int oracle_gather_qmm_rows(const uint16_t* x, const uint8_t* wq, const uint16_t* scales,
                                  const uint16_t* biases, const uint32_t* idx, int64_t H, int64_t F,
                                  int64_t E, int group_size, int bits, const int64_t* rows,
                                  int64_t n_rows, double* y_rows, int nthreads) {
    if (!bits_supported(bits) || group_size <= 0 || H % group_size || E <= 0 || (idx == NULL && E != 1)) return -1;
    qweights W = {MODE_AFFINE, bits, H, group_size, wq, scales, biases, NULL, 1};
    gemm_job base = {x, W, idx, rows, n_rows, H, F, E, y_rows, 0, 0};
    return run_gemm(base, n_rows, nthreads);
}

/* The gather matmul on weights in a floating-point mode (wq, scales, tscale as written by
 * oracle_quantize_fp over E*F rows with rows_per_tensor = F: one nvfp4 tensor scale per expert).
 * rows: NULL for all n rows, else the listed flat rows (y is [n_rows, F]). */
EXPORT int oracle_gather_qmm_fp(const uint16_t* x, const uint8_t* wq, const uint8_t* scales, const float* tscale,
                                const uint32_t* idx, int64_t n, int64_t H, int64_t F, int64_t E, int mode,
                                const int64_t* rows, int64_t n_rows, double* y, int nthreads) {
    if (mode < MODE_MXFP4 || mode > MODE_MXFP8 || H % mode_block(mode) || E <= 0 || (idx == NULL && E != 1)) return -1;
    if (mode == MODE_NVFP4 && !tscale) return -1;
    qweights W = {mode, 0, H, mode_block(mode), wq, scales, NULL, tscale, F};
    gemm_job base = {x, W, idx, rows, rows ? n_rows : n, H, F, E, y, 0, 0};
    return run_gemm(base, rows ? n_rows : n, nthreads);
}
