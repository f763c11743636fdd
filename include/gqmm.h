/*
 * gqmm.h -- C ABI of libgqmm, the affine-4-bit quantized mixture-of-experts gather matmul
 * for NVIDIA GB300 (sm_103a).
 *
 * The operation is the one the mlx issue "[CUDA] gather_qmm ~24x slower than equal-FLOPs
 * quantized_matmul on GB10 (sm_121)" (ml-explore/mlx #4339) benchmarks in its section
 * "Kernel microbenchmark":
 *
 *     wq, sc, bs = mx.quantize(w, group_size=64, bits=4)
 *     y = mx.gather_qmm(x, wq, sc, bs, rhs_indices=idx, transpose=True,
 *                       group_size=64, bits=4, mode="affine", sorted_indices=...)
 *
 * i.e. for every routed row (t, a):  y[t, a, :] = x[t, a, :] . deq(W[idx[t, a]])^T.
 *
 * Entry points: gqmm_quantize (the weight format below), gqmm_route_sort, gqmm_gather_qmm
 * (the operation; gqmm_gather_qmm_noalloc without a workspace), gqmm_moe_mlp (the expert MLP
 * built on it: gate/up, SiLU or GELU gating, down), gqmm_gather_qmm_nn (transpose=False),
 * gqmm_gather_qmm_simt and gqmm_gather_qmm_nn_simt (CUDA-core cross-checks), and status /
 * instrumentation calls.
 *
 * Conventions shared by every entry point
 *  - All tensor arguments are DEVICE pointers on the current CUDA device, except where a
 *    comment says otherwise.  The caller allocates and owns every buffer (outputs and the
 *    workspace included); the library allocates no device memory, keeps no pointer after
 *    a call returns, and never synchronizes the stream (gqmm_device_status excepted).
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Work is enqueued on it
 *    asynchronously; results are valid once the stream reaches that point.
 *  - bfloat16 tensors are passed as void* holding IEEE bfloat16 values.  All tensors are
 *    dense and row-major (last dimension contiguous).
 *  - Return value: GQMM_OK (0) or a positive GQMM_ERR_* code from argument validation or
 *    from the CUDA launch; nothing is enqueued when validation fails.  Conditions only the
 *    device can see (an expert index >= E, a false `sorted` promise, a wait that timed
 *    out) set bits in a status word inside the workspace; gqmm_device_status reads them.
 *  - gqmm_last_error() returns a short human-readable message for the calling thread's
 *    most recent non-OK return.
 *
 * Quantized weight format (the reading this library takes of mx.quantize(..., 64, 4); the
 * pages name the call but do not print its formula): for each group of group_size (64; also
 * 32 or 128) consecutive weights along H,
 *     scale = bf16((max - min) / 15)  (IEEE float32 division, round to nearest even)
 *     bias  = min                     (exact)
 *     q     = clamp(round_half_even((w - bias) / scale), 0, 15)  using the stored scale
 *             and bias as float32; q = 0 for a constant group (scale 0)
 *     byte j of a row = q[2j] | (q[2j + 1] << 4)
 * and deq(q) = scale * q + bias.  Shapes for E experts of F x H weights:
 *     wq      uint8     [E, F, H/2]
 *     scales  bfloat16  [E, F, H/group_size]
 *     biases  bfloat16  [E, F, H/group_size]
 * Other bit widths (mlx PR #4023 "Pick BM from rows per expert", the author's follow-up: every
 * mode, group size and bit width): bits b in {2, 3, 5, 6, 8} with 64-wide groups keep the steps
 * above with 2^b - 1 levels in place of 15; a row's codes are one little-endian bit stream
 * (element k in bits [k*b, (k+1)*b), bit j of the stream in bit j%8 of byte j/8; at b = 4 this is
 * the layout above), so wq is uint8 [E, F, H*b/8].
 *
 * Block-scaled floating-point modes (mlx #4339, Activity, nastya236: mxfp8 and nvfp4 are what the
 * CUDA back end is to support); the pages give no formulas, so these are the published formats:
 *   GQMM_MODE_MXFP4  OCP MX v1.0: E2M1 codes (two per byte as above), one E8M0 scale per 32
 *                    weights: X = 2^(floor(log2 amax) - 2), element = nearest E2M1 to w / X
 *                    (ties to even, saturating at 6).   wq [E, F, H/2], scales uint8 [E, F, H/32]
 *   GQMM_MODE_MXFP8  the same with E4M3 codes (one per byte), X = 2^(floor(log2 amax) - 8),
 *                    saturating at 448.                 wq [E, F, H],   scales uint8 [E, F, H/32]
 *   GQMM_MODE_NVFP4  NVFP4: E2M1 codes, one E4M3 scale per 16 weights and a float32 scale t per
 *                    expert: t = amax_expert / 2688, S = E4M3((amax_block / 6) / t), element =
 *                    E2M1(w / (S t)), all float32 operations.
 *                                                       wq [E, F, H/2], scales uint8 [E, F, H/16],
 *                                                       tscale float32 [E]
 *   and deq = element * X (mx) or element * S * t (nvfp4).
 */
#ifndef GQMM_H
#define GQMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define GQMM_API __attribute__((visibility("default")))
#else
#define GQMM_API
#endif

typedef struct CUstream_st* gqmm_stream_t; /* identical to cudaStream_t */

/* Synchronous return codes. */
#define GQMM_OK 0
#define GQMM_ERR_NULL 1         /* a required pointer is NULL */
#define GQMM_ERR_SHAPE 2        /* a size is out of range (see each entry point) */
#define GQMM_ERR_UNSUPPORTED 3  /* a format the call does not take, or E above GQMM_MAX_EXPERTS */
#define GQMM_ERR_ALIGN 4        /* a pointer is not aligned as required */
#define GQMM_ERR_WORKSPACE 5    /* workspace too small or misaligned */
#define GQMM_ERR_CUDA 6         /* a CUDA runtime/driver call or a kernel launch failed */
#define GQMM_ERR_DEVICE 7       /* the current device is not an sm_103 (GB300-class) GPU */

/* Device-side status bits (returned by gqmm_device_status, OR-ed across calls). */
#define GQMM_STATUS_BAD_INDEX 0x100u  /* some idx value was >= E; those rows of y are zero */
#define GQMM_STATUS_NOT_SORTED 0x200u /* sorted=1 but idx decreased somewhere: y unspecified */
#define GQMM_STATUS_TIMEOUT 0x400u    /* a bounded device-side wait gave up: y unspecified */

#define GQMM_MAX_EXPERTS 1024

/* Block-scaled floating-point modes of gqmm_quantize_fp and gqmm_gather_qmm_fp. */
#define GQMM_MODE_MXFP4 1
#define GQMM_MODE_NVFP4 2
#define GQMM_MODE_MXFP8 3

/* Gate activations of gqmm_moe_mlp. */
#define GQMM_ACT_SILU 0
#define GQMM_ACT_GELU 1
#define GQMM_ACT_GELU_TANH 2

/*
 * gqmm_quantize -- affine 4-bit group quantization (mx.quantize(w, group_size=64, bits=4)
 * in mlx #4339 "Kernel microbenchmark"), format as stated at the top of this header.
 *
 *  w       bfloat16 [rows, H] (for E experts of F x H weights, rows = E*F), 16-byte aligned
 *  rows    >= 0;  H > 0 and H % group_size == 0 (the quantized axis; gqmm_gather_qmm also needs
 *          its K a multiple of 64)
 *  group_size, bits   4-bit codes with 32-, 64- or 128-wide groups (64 is the pages' setting), or
 *          2-, 3-, 5-, 6- or 8-bit codes with 64-wide groups
 *  wq      out: uint8 [rows, H*bits/8], 16-byte aligned
 *  scales  out: bfloat16 [rows, H/group_size];  biases  out: bfloat16 [rows, H/group_size]
 * Results are bit-identical to the float32 reference formula above (no fast math).
 * Errors: GQMM_ERR_NULL, GQMM_ERR_SHAPE, GQMM_ERR_UNSUPPORTED, GQMM_ERR_ALIGN, GQMM_ERR_CUDA.
 */
GQMM_API int gqmm_quantize(const void* w, int64_t rows, int64_t H, int group_size, int bits, void* wq,
                  void* scales, void* biases, gqmm_stream_t stream);

/*
 * gqmm_quantize_fp -- block-scaled floating-point quantization (GQMM_MODE_*, formats at the top
 * of this header; mlx #4339, Activity).
 *  w       bfloat16 [rows, H], 16-byte aligned; H a positive multiple of 64
 *  rows_per_tensor  nvfp4: rows sharing one float32 scale (F for an [E, F, H] expert stack;
 *          rows a multiple of it, at most 65535 tensors); ignored otherwise
 *  wq      out: uint8 [rows, H/2] (mxfp4, nvfp4) or [rows, H] (mxfp8), 16-byte aligned
 *  scales  out: uint8 [rows, H/32] (mx) or [rows, H/16] (nvfp4)
 *  tscale  out: float32 [rows / rows_per_tensor] (nvfp4; may be NULL otherwise)
 * Codes and scales are bit-identical to the float32 steps stated above.  nvfp4 runs three kernels
 * (the tensors' largest magnitudes, their scales, the blocks).
 * Errors: GQMM_ERR_NULL, GQMM_ERR_SHAPE, GQMM_ERR_UNSUPPORTED, GQMM_ERR_ALIGN, GQMM_ERR_CUDA.
 */
GQMM_API int gqmm_quantize_fp(const void* w, int64_t rows, int64_t H, int64_t rows_per_tensor, int mode, void* wq,
                              void* scales, float* tscale, gqmm_stream_t stream);

/*
 * gqmm_workspace_size -- bytes of device workspace gqmm_gather_qmm and gqmm_route_sort
 * need for n = T*A routed rows, F output columns and E experts.  The workspace must be
 * 256-byte aligned and MUST BE ZERO-FILLED ONCE before its first use (it carries the
 * device status word, which gqmm_device_status clears after reading); afterwards it can be
 * reused by any number of calls on the same stream whose own gqmm_workspace_size is at
 * most its size.  For decode-sized calls with few work units the size includes float32
 * planes for split-K partial sums (ksplit x n x F, ksplit <= 16), so it is not monotone
 * in n: a workspace shared by several shapes takes the maximum over them.
 * Returns 0 for invalid sizes.
 */
GQMM_API size_t gqmm_workspace_size(int64_t n, int F, int E);

/*
 * gqmm_route_sort -- on-device stable counting sort of the routing entries by expert
 * (mlxcel #629 "perf(cuda/moe): fix MoE prefill collapse", implementation plan item 4b:
 * token sorting by expert on device so each expert owns one contiguous block).
 *
 *  idx      uint32 [n] expert index of each flat row i = t*A + a
 *  n        number of rows, 0 <= n <= 2^31 - 1;  E in [1, GQMM_MAX_EXPERTS]
 *  perm     out: int32 [n]; perm[offsets[e] + k] is the k-th smallest row routed to e;
 *           rows with idx >= E follow all valid rows, in row order
 *  offsets  out: int32 [E + 1]; offsets[e] = number of valid rows with expert < e,
 *           offsets[E] = number of valid rows (n when the routing is valid)
 *  ws       workspace of at least gqmm_workspace_size(n, 1, E) bytes (see above)
 * Two kernels (tile histograms; scan + stable scatter), no host round trip.  The output
 * is unique (stable order).
 * Errors: GQMM_ERR_NULL, GQMM_ERR_SHAPE, GQMM_ERR_UNSUPPORTED, GQMM_ERR_WORKSPACE,
 * GQMM_ERR_CUDA; idx >= E sets GQMM_STATUS_BAD_INDEX.
 */
GQMM_API int gqmm_route_sort(const uint32_t* idx, int64_t n, int E, int32_t* perm, int32_t* offsets,
                    void* ws, size_t ws_bytes, gqmm_stream_t stream);

/*
 * gqmm_gather_qmm -- y[t, a, :] = x[t, a, :] . deq(W[idx[t, a]])^T  (mx.gather_qmm with
 * transpose=True, mode="affine", mlx #4339 "Kernel microbenchmark"), float32
 * accumulation, bfloat16 output rounded to nearest even once.
 *
 *  x        bfloat16 [T, A, H] (the issue's (T, A, 1, H)), 16-byte aligned
 *  wq, scales, biases   the quantized weights of E experts, [E, F, ...] as above;
 *           wq, scales and biases 16-byte aligned
 *  idx      uint32 [T, A] expert per row, or NULL for the dense quantized matmul
 *           (mx.quantized_matmul, same issue), which requires E == 1
 *  T, A     T >= 1, A >= 1, T*A <= 2^31 - 1
 *  H        > 0, multiple of 64 and of group_size;   F > 0, multiple of 16;   E in [1, GQMM_MAX_EXPERTS]
 *  group_size, bits   as for gqmm_quantize; a row's codes (H*bits/8 bytes) must be a multiple
 *           of 16 bytes (for 3- and 5-bit codes: H a multiple of 128).  The weight-streaming
 *           kernels of decode-sized calls take 4-bit codes in 64-wide groups (the CUDA-core one
 *           H a multiple of 128 up to 8192, the MMA one H of 1024, 2048 or 4096); other formats
 *           and sizes run decode-sized calls on the tensor-core GEMM's narrow variant
 *  x_shared 0: x is [T, A, H], one row per (t, a);  1: x is [T, H], the A routed rows of
 *           token t all read x[t] (the x of an MoE layer, broadcast over its A experts;
 *           needs idx != NULL)
 *  sorted   0: idx in any order (the library sorts rows by expert on device);
 *           1: the caller promises idx is nondecreasing in flat order (the issue's
 *              sorted_indices=True).  The result is identical either way; a broken
 *              promise sets GQMM_STATUS_NOT_SORTED, computes nothing and writes y as zeros.
 *  y        out: bfloat16 [T, A, F] in (t, a) order, 16-byte aligned
 *  ws       workspace of at least gqmm_workspace_size(T*A, F, E) bytes (see above)
 * Rows whose idx is >= E are written as zeros and set GQMM_STATUS_BAD_INDEX.
 * Errors: GQMM_ERR_NULL, GQMM_ERR_SHAPE, GQMM_ERR_UNSUPPORTED, GQMM_ERR_ALIGN,
 * GQMM_ERR_WORKSPACE, GQMM_ERR_DEVICE, GQMM_ERR_CUDA.
 */
GQMM_API int gqmm_gather_qmm(const void* x, const void* wq, const void* scales, const void* biases,
                    const uint32_t* idx, int64_t T, int A, int H, int F, int E, int group_size,
                    int bits, int sorted, int x_shared, void* y, void* ws, size_t ws_bytes,
                    gqmm_stream_t stream);

/*
 * gqmm_gather_qmm_fp -- gqmm_gather_qmm on weights in a block-scaled floating-point mode
 * (mx.gather_qmm with mode "mxfp4", "nvfp4" or "mxfp8"; mlx #4339, Activity):
 *     y[t, a, :] = x[t, a, :] . deq(W[idx[t, a]])^T,
 * x bfloat16, each weight decoded exactly and scaled in float32 to one bfloat16 rounding
 * (like the affine path's dequantized weights), float32 accumulation, bfloat16 y.
 *  wq, scales, tscale   as gqmm_quantize_fp writes them for rows = E*F, rows_per_tensor = F;
 *           scales and tscale 4-byte aligned
 *  mode     GQMM_MODE_MXFP4, GQMM_MODE_NVFP4 (needs tscale) or GQMM_MODE_MXFP8
 *  the rest as for gqmm_gather_qmm (H a positive multiple of 64; the same workspace size).
 * Every mode runs on the wide tensor-core variant and on the narrow one (at most 32 rows per
 * expert on average).
 * Errors: as gqmm_gather_qmm.
 */
GQMM_API int gqmm_gather_qmm_fp(const void* x, const void* wq, const void* scales, const float* tscale,
                                const uint32_t* idx, int64_t T, int A, int H, int F, int E, int mode, int sorted,
                                int x_shared, void* y, void* ws, size_t ws_bytes, gqmm_stream_t stream);

/*
 * gqmm_moe_mlp_workspace_size -- bytes of workspace for gqmm_moe_mlp with n = T*A rows,
 * model width H, expert intermediate width I and E experts (256-byte aligned pointer
 * required).  Holds the route sort, the work list and the two bf16 intermediates
 * ([n, 2I] and [n, I]); 0 for invalid sizes.
 */
GQMM_API size_t gqmm_moe_mlp_workspace_size(int64_t n, int H, int I, int E);

/*
 * gqmm_moe_mlp -- the MoE expert MLP on the routed rows, the two quantized projections
 * chained through one route sort (mlx PR #4023 "Pick BM from rows per expert", Measurement:
 * chained up and down projection pairs; mlxcel #629 References: a fused switch MLP over
 * gather_qmm):
 *     g = x[t, a, :] . deq(W_gu[e])[0 : I]^T,   u = x[t, a, :] . deq(W_gu[e])[I : 2I]^T,
 *     y[t, a, :] = (act(g) * u) . deq(W_dn[e])^T,   e = idx[t, a],
 * with the gate activation act chosen by `activation` (the switch-GeGLU of mlxcel #629
 * References and the SwiGLU of most MoE models):
 *     GQMM_ACT_SILU       act(v) = v / (1 + e^-v)                                  (SwiGLU)
 *     GQMM_ACT_GELU       act(v) = v/2 (1 + erf(v / sqrt 2))                       (GeGLU)
 *     GQMM_ACT_GELU_TANH  act(v) = v/2 (1 + tanh(sqrt(2/pi) (v + 0.044715 v^3)))   (GeGLU, tanh form)
 * g and u are rounded to bfloat16 as the first projection writes them, act(g) * u is
 * computed in float32 and rounded to bfloat16, and each projection accumulates in float32.
 *
 *  x        bfloat16 [T, A, H], 16-byte aligned
 *  wq_gu, sc_gu, bs_gu   W_gu = [W_gate; W_up] quantized, [E, 2I, ...] (gate rows 0 .. I-1,
 *           up rows I .. 2I-1), as gqmm_quantize writes for rows = E*2I
 *  wq_dn, sc_dn, bs_dn   W_dn quantized, [E, H, ...] with K = I
 *  idx, T, A, E, group_size, bits, sorted   as for gqmm_gather_qmm
 *  H        > 0, multiple of 64;   I > 0, multiple of 64 (it is the down projection's K)
 *  activation  GQMM_ACT_SILU, GQMM_ACT_GELU or GQMM_ACT_GELU_TANH (else GQMM_ERR_UNSUPPORTED)
 *  x_shared as for gqmm_gather_qmm (x [T, H] shared by a token's A experts)
 *  y        out: bfloat16 [T, A, H] in (t, a) order, 16-byte aligned
 *  ws       workspace of at least gqmm_moe_mlp_workspace_size(T*A, H, I, E) bytes
 * Rows whose idx is >= E are written as zeros and set GQMM_STATUS_BAD_INDEX.
 * Errors: as gqmm_gather_qmm, for both projections' shapes.
 */
GQMM_API int gqmm_moe_mlp(const void* x, const void* wq_gu, const void* sc_gu, const void* bs_gu,
                          const void* wq_dn, const void* sc_dn, const void* bs_dn, const uint32_t* idx,
                          int64_t T, int A, int H, int I, int E, int group_size, int bits, int activation,
                          int sorted, int x_shared, void* y, void* ws, size_t ws_bytes, gqmm_stream_t stream);

/*
 * gqmm_gather_qmm_nn -- gather_qmm with transpose=False (mlx PR #4023 "Pick BM from rows per
 * expert in gather_qmm_rhs_nax", the author's follow-up: the shape of the backward pass and of
 * fine-tuning):
 *     y[t, a, :] = x[t, a, :] . deq(W[idx[t, a]]),   W[e] of shape [K, N], quantized along N
 * (mx.quantize applied to an [E, K, N] weight, the format at the top of this header with H := N).
 * The same route step and tcgen05 grouped GEMM as gqmm_gather_qmm: a unit is 256 output columns
 * of one expert; each k-block's codes are 64 k-rows of the unit's columns, dequantized column by
 * column into the same K-major bf16 operand (one rounding per weight), float32 accumulation,
 * bf16 output.
 *
 *  x        bfloat16 [T, A, K] (or [T, K] with x_shared = 1), 16-byte aligned
 *  wq       uint8 [E, K, N/2] (element n of a k-row in the low nibble when n is even), 16-byte
 *           aligned;  scales, biases  bfloat16 [E, K, N/group_size], 2-byte aligned
 *  idx, T, A, E, sorted, x_shared, ws, ws_bytes, stream   as for gqmm_gather_qmm, with the
 *           workspace sized by gqmm_workspace_size(T*A, N, E)
 *  K        a positive multiple of 64;  N  a positive multiple of 32 and of group_size
 *  group_size 32, 64 or 128;  bits 4;  E*K and E*N below 2^31
 *  y        out: bfloat16 [T, A, N], 16-byte aligned
 * Invalid indices, the status word and the sorted-promise rule: as gqmm_gather_qmm.
 * Errors: GQMM_ERR_NULL, GQMM_ERR_SHAPE, GQMM_ERR_UNSUPPORTED, GQMM_ERR_ALIGN,
 * GQMM_ERR_WORKSPACE, GQMM_ERR_DEVICE, GQMM_ERR_CUDA.
 */
GQMM_API int gqmm_gather_qmm_nn(const void* x, const void* wq, const void* scales, const void* biases,
                               const uint32_t* idx, int64_t T, int A, int K, int N, int E, int group_size,
                               int bits, int sorted, int x_shared, void* y, void* ws, size_t ws_bytes,
                               gqmm_stream_t stream);

/*
 * gqmm_gather_qmm_nn_simt -- the transpose=False operation on CUDA cores: every routed row
 * streams its expert's [K, N] codes (from L2 after the first row of an expert); float32
 * dequantization and accumulation, bf16 output.  A slow, independent GPU cross-check of
 * gqmm_gather_qmm_nn, never used by it; needs no workspace.
 *  x        bfloat16 [T, A, K] (or [T, K] with x_shared = 1), 2-byte aligned
 *  K        in [1, 2^24];   N  positive multiple of group_size, at most 2^24
 *  other arguments as gqmm_gather_qmm_nn (no sorted flag: rows are independent)
 * Rows whose idx is >= E are written as zeros (no status word: this call takes no workspace).
 * Errors: GQMM_ERR_NULL, GQMM_ERR_SHAPE, GQMM_ERR_UNSUPPORTED, GQMM_ERR_ALIGN, GQMM_ERR_CUDA.
 */
GQMM_API int gqmm_gather_qmm_nn_simt(const void* x, const void* wq, const void* scales, const void* biases,
                                    const uint32_t* idx, int64_t T, int A, int K, int N, int E,
                                    int group_size, int bits, int x_shared, void* y, gqmm_stream_t stream);

/*
 * gqmm_gather_qmm_simt -- the same operation computed on CUDA cores, one thread per output
 * element with float32 accumulation; needs no workspace.  A slow, independent GPU
 * cross-check of gqmm_gather_qmm's data handling, never used by it.  Same argument rules
 * (sorted is not needed: each row reads its own index).  Rows with idx >= E are zero.
 */
GQMM_API int gqmm_gather_qmm_simt(const void* x, const void* wq, const void* scales, const void* biases,
                         const uint32_t* idx, int64_t T, int A, int H, int F, int E,
                         int group_size, int bits, int x_shared, void* y, gqmm_stream_t stream);

/*
 * gqmm_gather_qmm_noalloc -- the pages have no counterpart to this entry point; it is a
 * convenience of this library.  Same operation, arguments and results as gqmm_gather_qmm
 * with x_shared = 0 (x [T, A, H]), but without a workspace argument: the scratch it needs is a
 * fixed array of
 * GQMM_NOALLOC_SCRATCH_BYTES inside the library's device code, and the call allocates
 * nothing (no cudaMalloc, no cudaFree, no allocating library routine).  It is meant for
 * callers that cannot allocate device memory or keep a workspace: a plugin whose host
 * framework owns all device memory, or a latency-critical path that must not call
 * cudaMalloc (which can synchronize the device).
 *  - The scratch covers any call with T*A <= 131072 rows (and E <= GQMM_MAX_EXPERTS); larger
 *    calls return GQMM_ERR_WORKSPACE with a message and enqueue nothing.  Calls with few
 *    work units, which gqmm_gather_qmm runs with K split into slices, are split here only
 *    when the float32 partial-sum planes also fit; otherwise they run unsplit (equal
 *    within rounding, less parallelism).
 *  - The array occupies device memory on every GPU that loads the library, until exit.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress); make that first call before any stream capture.
 *  - Every call on a device shares the one array: calls whose GPU work overlaps (different
 *    streams, no ordering between them) race and give undefined results.  Calls on one
 *    stream are ordered and safe.
 *  - Each call clears the scratch's status word (after validating its arguments: a refused
 *    call enqueues nothing), and nothing reads it back, so device-detected conditions are
 *    NOT reported and the call still returns GQMM_OK: rows with an index >= E come out as
 *    zeros, a false sorted = 1 promise gives a y of all zeros, and a bounded wait that ran
 *    out leaves y undefined.  Use gqmm_gather_qmm with gqmm_device_status when these
 *    conditions must be seen.
 *  - The device address of the array is cached per device ordinal for the life of the
 *    process; after cudaDeviceReset on a device, do not call this entry point on it again.
 */
#define GQMM_NOALLOC_SCRATCH_BYTES (1u << 20)
GQMM_API int gqmm_gather_qmm_noalloc(const void* x, const void* wq, const void* scales, const void* biases,
                                     const uint32_t* idx, int64_t T, int A, int H, int F, int E,
                                     int group_size, int bits, int sorted, void* y, gqmm_stream_t stream);

/*
 * gqmm_device_status -- synchronizes `stream`, returns the device status bits
 * (GQMM_STATUS_*) accumulated in workspace `ws` since the last call, and clears them.
 * Returns a negative value if the synchronization or the copy fails.
 */
GQMM_API int gqmm_device_status(void* ws, gqmm_stream_t stream);

/* Short description of a return code or status bit. Never NULL. */
GQMM_API const char* gqmm_status_string(int status);

/* Message describing the calling thread's most recent failing call ("" if none). */
GQMM_API const char* gqmm_last_error(void);

/*
 * Instrumentation (host side only; nothing here changes what the kernels compute).
 *  gqmm_launch_count      kernels this library has launched in this process.
 *  gqmm_kernel_timer      capacity > 0: time the next `capacity` grouped-GEMM launches of
 *                         gqmm_gather_qmm with CUDA events on the call's stream (events are
 *                         created by this call; not for use during stream capture);
 *                         capacity 0: stop timing.
 *  gqmm_kernel_timer_read synchronizes the recorded events and returns the number of timed
 *                         launches and their total duration in milliseconds, then resets.
 *  gqmm_dispatch_count    how many times each internal variant ran (GQMM_VARIANT_*).
 */
GQMM_API int64_t gqmm_launch_count(void);
GQMM_API void gqmm_kernel_timer(int capacity);
GQMM_API int gqmm_kernel_timer_read(int64_t* launches, double* total_ms);

/*
 * gqmm_test_stall_next -- failure-path test hook.  The next n tensor-core GEMM launches leave
 * their first k-block's codes uncopied, so the dequant warps' bounded wait for them runs out
 * (after 2 s): the launch sets GQMM_STATUS_TIMEOUT, every role unwinds (waits, each bounded,
 * for its own copies and MMAs in flight) and the tensor memory is freed, so the context and the
 * next calls stay usable.  y of a stalled call is undefined.  n = 0 disarms.  No fault, trap or
 * unbounded wait is involved.
 */
GQMM_API void gqmm_test_stall_next(int n);

#define GQMM_VARIANT_ROUTE_UNSORTED 0 /* histogram + scatter route sort */
#define GQMM_VARIANT_ROUTE_SORTED 1   /* segment boundaries from caller-sorted idx */
#define GQMM_VARIANT_ROUTE_DENSE 2    /* idx == NULL, E == 1 */
#define GQMM_VARIANT_GEMM_TC 3        /* tcgen05 grouped GEMM, chunks of up to 256 rows (mid variant: 128;
                                         CTA pairs, above 256 rows per expert: 512) */
#define GQMM_VARIANT_GEMM_NARROW 4    /* tcgen05 grouped GEMM, chunks of up to 32 rows */
#define GQMM_VARIANT_SPLIT_K 5        /* K split into slices, fp32 partial sums + finalize */
#define GQMM_VARIANT_GEMV 6           /* weight-streaming CUDA-core kernel: routed chunks of 1-2 rows, dense 1 row */
#define GQMM_VARIANT_GEMV_MMA 7       /* weight-streaming MMA kernel, dense calls of 2 to 8 rows */
#define GQMM_VARIANT_NN 8             /* gqmm_gather_qmm_nn (transpose=False) calls, on the tcgen05 GEMM */
#define GQMM_VARIANT_ROUTE_FUSED 9    /* unsorted routed decode (<= 64 rows) planned inside the streaming kernel */
#define GQMM_VARIANT_COUNT 10
GQMM_API int64_t gqmm_dispatch_count(int variant);

#ifdef __cplusplus
}
#endif

#endif /* GQMM_H */
