// Weight formats of the grouped GEMM: how one 64-wide k-block of one weight row is stored, where
// the TMA copies its codes from, and how a dequant thread turns them into 64 bfloat16 values.
//
//   FmtAffine<GS, BITS>  affine groups of GS weights (scale and bias bfloat16), BITS-bit codes in a
//                        little-endian bit stream per row (element k in bits [k*BITS, (k+1)*BITS));
//                        BITS = 4 is the format of mx.quantize(w, group_size, 4) as the mlx issue
//                        "[CUDA] gather_qmm ~24x slower ..." (Kernel microbenchmark) calls it; the
//                        other widths are the rest of mlx PR #4023's "all modes, group sizes and bit
//                        widths" (the author's follow-up).
//   FmtMx<ELEM8>         OCP microscaling: E2M1 codes two per byte (mxfp4) or E4M3 codes one per
//                        byte (mxfp8), one E8M0 scale byte per 32 weights.
//   FmtNv                NVFP4: E2M1 codes two per byte, one E4M3 scale byte per 16 weights and a
//                        float32 scale per expert.
// (mlx #4339, Activity, nastya236: mxfp8 and nvfp4 are the modes the CUDA back end is to support.)
//
// A k-block's codes take CB = 64 * BITS / 8 bytes of the row.  TMA boxes must start on a 16-byte
// boundary, so the code tile of a k-block is a window of W bytes per row starting at
// (kb * CB) rounded down to 16; the k-block's codes start OFF = (kb * CB) mod 16 bytes into it
// (0 or 8 for 3- and 5-bit codes, 0 otherwise).  32-byte windows are copied with the 32-byte
// swizzle (16-byte chunk c of row r at chunk c ^ ((r >> 2) & 1)), other widths unswizzled.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace gqmm {

enum WeightKind { kAffine = 0, kMxfp4 = 1, kNvfp4 = 2, kMxfp8 = 3, kAffineNn = 4 };

template <int GS_, int BITS_>
struct FmtAffine {
  static constexpr int KIND = kAffine;
  static constexpr int GS = GS_;
  static constexpr int BITS = BITS_;
  static constexpr int CB = 64 * BITS / 8;
  static constexpr int W = BITS == 3 || BITS == 5 ? 48 : CB;
  static_assert(BITS == 2 || BITS == 3 || BITS == 4 || BITS == 5 || BITS == 6 || BITS == 8, "bit widths");
};

template <bool ELEM8>
struct FmtMx {
  static constexpr int KIND = ELEM8 ? kMxfp8 : kMxfp4;
  static constexpr int GS = 32;  // weights per scale
  static constexpr int BITS = ELEM8 ? 8 : 4;
  static constexpr int CB = 64 * BITS / 8;
  static constexpr int W = CB;
};

struct FmtNv {
  static constexpr int KIND = kNvfp4;
  static constexpr int GS = 16;
  static constexpr int BITS = 4;
  static constexpr int CB = 32;
  static constexpr int W = CB;
};

// transpose=False (mlx PR #4023, the author's follow-up): W[e] is [K, N] with 4-bit affine codes
// in groups of GS along N, so one k-block of a unit is a tile of 64 k-rows x 256 n-codes (128
// bytes each, 8 KB like the other 4-bit stages), copied unswizzled; a dequant thread builds the
// K-major row of one output column n from one nibble of each of the 64 k-rows, with the scale and
// bias of (k, n / GS).  The same MMA, gather and epilogue then compute y[:, n] for the unit's n.
template <int GS_>
struct FmtNn {
  static constexpr int KIND = kAffineNn;
  static constexpr int GS = GS_;
  static constexpr int BITS = 4;
  static constexpr int CB = 32;
  static constexpr int W = 32;  // code stage bytes = 256 rows x 32 = 64 k-rows x 128 bytes
};

// TMA x coordinate (bytes) of k-block kb's code window, and the codes' offset in it.
template <class FMT>
__host__ __device__ __forceinline__ int code_window_x(int kb) {
  return (kb * FMT::CB) & ~15;
}
template <class FMT>
__host__ __device__ __forceinline__ int code_window_off(int kb) {
  return (kb * FMT::CB) & 15;
}

#if defined(__CUDACC__)

// ---- affine codes of any width: bf16 pairs (128 + q) into the scale/bias FMA ----------------

// bits [pos, pos + n) of the little-endian word array (pos + n <= 32 * N), n <= 8
template <int N>
__device__ __forceinline__ uint32_t bits_at(const uint32_t (&w)[N], int pos, int n) {
  const int i = pos >> 5, sh = pos & 31;
  const uint32_t lo = w[i];
  const uint32_t hi = i + 1 < N ? w[i + 1] : 0u;
  return __funnelshift_r(lo, hi, sh) & ((1u << n) - 1u);
}

// (s, s) and (b, b) applied to two codes held as bfloat16 128 + q: the first FMA removes 128
// exactly, the second rounds s * q + b once to bfloat16.
__device__ __forceinline__ uint32_t affine_pair(uint32_t p, uint32_t s2, uint32_t b2) {
  uint32_t q, r;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(q) : "r"(p), "r"(0x3F803F80u), "r"(0xC300C300u));
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(q), "r"(s2), "r"(b2));
  return r;
}

// 64 weights of an affine row from codes at bit offset OFF*8 of the window words cw (BITS <= 7:
// codes as bfloat16 128 + q; BITS == 8: q itself, exact in bfloat16, through float32).
template <int BITS, int OFF, int NW>
__device__ __forceinline__ void dequant_affine(const uint32_t (&cw)[NW], uint32_t s2, uint32_t b2, uint4 (&o)[8]) {
  uint32_t* out = reinterpret_cast<uint32_t*>(o);
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const uint32_t q0 = bits_at(cw, OFF * 8 + (2 * j) * BITS, BITS);
    const uint32_t q1 = bits_at(cw, OFF * 8 + (2 * j + 1) * BITS, BITS);
    if (BITS <= 7) {
      out[j] = affine_pair(q0 | (q1 << 16) | 0x43004300u, s2, b2);
    } else {
      const float f0 = __uint_as_float(0x4B000000u | q0) - 8388608.0f;  // q exactly
      const float f1 = __uint_as_float(0x4B000000u | q1) - 8388608.0f;
      const __nv_bfloat162 qq = __floats2bfloat162_rn(f0, f1);           // exact: q < 256
      uint32_t r;
      asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(*reinterpret_cast<const uint32_t*>(&qq)), "r"(s2), "r"(b2));
      out[j] = r;
    }
  }
}

// ---- E2M1 / E4M3 codes: hardware conversion to f16 pairs, float32 scale, one rounding ------

// four f16 pairs from the 8 E2M1 codes of a word (element 2j in the low nibble of byte j)
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

// two f16 pairs from the 4 E4M3 codes of a word (element j in byte j)
__device__ __forceinline__ void e4m3x4_to_f16x2(uint32_t w, uint32_t (&h)[2]) {
  asm("{\n\t.reg .b16 s0, s1;\n\tmov.b32 {s0, s1}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, s0;\n\tcvt.rn.f16x2.e4m3x2 %1, s1;\n\t}"
      : "=r"(h[0]), "=r"(h[1])
      : "r"(w));
}

// an f16 pair times a float32 scale, as a bfloat16 pair (one rounding)
__device__ __forceinline__ uint32_t scaled_pair(uint32_t h2, float sc) {
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2));
  const __nv_bfloat162 r = __floats2bfloat162_rn(f.x * sc, f.y * sc);
  return *reinterpret_cast<const uint32_t*>(&r);
}

// E8M0 scale byte -> 2^(c - 127) as float32 (c = 0: 2^-127, a float32 subnormal; 255: NaN)
__device__ __forceinline__ float e8m0_to_f32(uint32_t c) {
  return c == 0u ? __uint_as_float(0x00400000u) : c == 255u ? __uint_as_float(0x7FC00000u) : __uint_as_float(c << 23);
}

// E4M3 scale byte -> float32, from the format's definition (exact): exponent field e (bias 7)
// and mantissa m give (8 + m) 2^(e - 10), or m 2^-9 when e = 0.
__device__ __forceinline__ float e4m3_to_f32(uint32_t c) {
  const uint32_t e = (c >> 3) & 15u, m = c & 7u;
  const float v = e == 0u ? (float)m * 0.001953125f : (float)(8u + m) * __uint_as_float((e + 117u) << 23);
  return (c & 0x80u) ? -v : v;
}

// 64 weights of a 4-bit E2M1 row (32 bytes of codes in cw) with per-16 scales sc[4]
// (element k uses sc[k / 16]).
__device__ __forceinline__ void dequant_e2m1(const uint32_t (&cw)[8], const float (&sc)[4], uint4 (&o)[8]) {
  uint32_t* out = reinterpret_cast<uint32_t*>(o);
#pragma unroll
  for (int i = 0; i < 8; ++i) {  // word i holds elements 8 i .. 8 i + 7
    uint32_t h[4];
    e2m1x8_to_f16x2(cw[i], h);
#pragma unroll
    for (int j = 0; j < 4; ++j) out[4 * i + j] = scaled_pair(h[j], sc[(8 * i) / 16]);
  }
}

// 64 weights of an E4M3 row (64 bytes of codes in cw) with per-16 scales sc[4] (element k uses
// sc[k / 16]; the mx formats repeat each per-32 scale twice)
__device__ __forceinline__ void dequant_e4m3(const uint32_t (&cw)[16], const float (&sc)[4], uint4 (&o)[8]) {
  uint32_t* out = reinterpret_cast<uint32_t*>(o);
#pragma unroll
  for (int i = 0; i < 16; ++i) {  // word i holds elements 4 i .. 4 i + 3
    uint32_t h[2];
    e4m3x4_to_f16x2(cw[i], h);
#pragma unroll
    for (int j = 0; j < 2; ++j) out[2 * i + j] = scaled_pair(h[j], sc[(4 * i) / 16]);
  }
}

#endif  // __CUDACC__

}  // namespace gqmm
