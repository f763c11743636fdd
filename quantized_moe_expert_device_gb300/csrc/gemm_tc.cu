// Persistent grouped GEMM for the quantized MoE gather matmul on tcgen05 tensor cores.
//
// Work unit = (chunk of one expert's sorted rows, 128-row tile of the expert's F outputs).
// The product is computed transposed ("swap A/B"): the UMMA M slot (128) holds weight rows
// f, the N slot holds the chunk's tokens, so N = round_up(rows, 16) follows the rows per
// expert.  This is the tensor-core form of the lesson in mlx PR #4023 "Pick BM from rows
// per expert in gather_qmm_rhs_nax" (useful arithmetic ~ min(1, run / BM)): a 4-row run
// costs an N=16 MMA instead of most of a 64- or 128-row tile, and each expert's weight
// tile is read and dequantized once per chunk of up to 256 rows instead of once per row
// (mlx #4339 comment by manunicholasjacob: one CTA per token-expert pair, 15 of 16 tile
// rows empty, the 4-bit slab dequantized once per row).
//
// Per CTA (one per SM, persistent, static round-robin over units), warp roles:
//   warps 0-7   dequant:  read packed nibbles from shared memory, w = scale*q + bias in
//                         bf16x2, write the bf16 A tile in the 128-byte-swizzle K-major layout
//   warps 8-11  epilogue: TMEM -> registers -> bf16 -> shared transpose -> 16-byte stores
//                         to y rows perm[j] (the scatter back to (t, a) order)
//   warp 12     TMA:      one thread streams 128 x 32-byte nibble tiles (one 64-wide group)
//   warp 13     MMA:      allocates TMEM (2 x 256 columns), one thread issues
//                         tcgen05.mma 128xNx16 x4 per stage, commits to mbarriers
//   warps 14-15 gather:   cp.async 16-byte copies of x rows perm[j] into the swizzled B tile
// Pipeline depth: 4 stages of (A 16 KB, B 32 KB, nibbles 4 KB).  TMEM accumulators are double
// buffered so the epilogue of unit i overlaps the mainloop of unit i+1.
//
// Every wait is bounded (mbar_wait): on expiry the CTA raises GQMM_STATUS_TIMEOUT, unwinds,
// waits (bounded) for its own copies and MMAs in flight and frees its TMEM.
#include "gqmm_internal.cuh"

namespace gqmm {
namespace {

constexpr int BM = 128;                 // weight rows per tile (UMMA M)
constexpr int BK = 64;                  // K per stage = one quantization group
constexpr int NMAX = kChunkMaxRows;     // tokens per unit, UMMA N <= 256
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;    // 16 KB bf16
constexpr int B_BYTES = NMAX * BK * 2;  // 32 KB bf16
constexpr int NIB_BYTES = BM * BK / 2;  // 4 KB packed codes
constexpr int EPI_WARP_BYTES = 16 * 32 * 2;

constexpr int kThreads = 512;
constexpr int kDeqThreads = 256;        // warps 0-7
constexpr int kEpiWarp0 = 8;            // warps 8-11
constexpr int kTmaWarp = 12;
constexpr int kMmaWarp = 13;
constexpr int kGatherWarp0 = 14;        // warps 14-15
constexpr int kGatherThreads = 64;
constexpr int kGatherLag = 2;           // cp.async groups kept in flight per gather thread
constexpr uint32_t kTmemCols = 512;     // two 256-column fp32 accumulators

constexpr int OFF_A = 0;
constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
constexpr int OFF_NIB = OFF_B + STAGES * B_BYTES;
constexpr int OFF_EPI = OFF_NIB + STAGES * NIB_BYTES;
constexpr int OFF_BAR = OFF_EPI + 4 * EPI_WARP_BYTES;
constexpr int NUM_BARS = 5 * STAGES + 5;
constexpr int OFF_MISC = OFF_BAR + ((NUM_BARS * 8 + 127) / 128) * 128;
constexpr int SMEM_USED = OFF_MISC + 16;
constexpr int SMEM_DYN = SMEM_USED + 1024;  // room to align the base to 1024 bytes
static_assert(SMEM_DYN <= 232448, "fits the 227 KB opt-in shared memory of one CTA");

// barrier slots
__device__ __forceinline__ int b_nib_full(int s) { return s; }
__device__ __forceinline__ int b_nib_empty(int s) { return STAGES + s; }
__device__ __forceinline__ int b_a_full(int s) { return 2 * STAGES + s; }
__device__ __forceinline__ int b_b_full(int s) { return 3 * STAGES + s; }
__device__ __forceinline__ int b_ab_empty(int s) { return 4 * STAGES + s; }
__device__ __forceinline__ int b_tmem_full(int b) { return 5 * STAGES + b; }
__device__ __forceinline__ int b_tmem_empty(int b) { return 5 * STAGES + 2 + b; }
__device__ __forceinline__ int b_unwind() { return 5 * STAGES + 4; }

struct Unit {
  int expert, start, rows, f0;
};

__device__ __forceinline__ Unit decode_unit(const Chunk* chunks, int u, int n_ftiles) {
  const int c = u / n_ftiles;
  const int ft = u - c * n_ftiles;
  const int4 ch = __ldg(reinterpret_cast<const int4*>(chunks) + c);
  Unit U;
  U.expert = ch.x;
  U.start = ch.y;
  U.rows = ch.z;
  U.f0 = ft * BM;
  return U;
}

// (s, s) and (b, b) as bf16x2 from one 16-bit pattern each.
__device__ __forceinline__ uint32_t splat16(uint32_t v16) { return (v16 & 0xFFFFu) * 0x00010001u; }

// Two codes, as bf16 128+q in each half, to bf16 scale*q + bias: the first FMA subtracts
// 128 exactly, the second rounds scale*q + bias once to bf16.
__device__ __forceinline__ uint32_t deq_pair(uint32_t p, uint32_t s2, uint32_t b2) {
  uint32_t q, r;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(q) : "r"(p), "r"(0x3F803F80u), "r"(0xC300C300u));
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(q), "r"(s2), "r"(b2));
  return r;
}

// 8 codes (one 32-bit word, element k in bits 4k..4k+3) -> 8 bf16 in element order.
__device__ __forceinline__ uint4 deq8(uint32_t w, uint32_t s2, uint32_t b2) {
  constexpr uint32_t kMask = 0x000F000Fu, kMagic = 0x43004300u;  // bf16 128.0 in each half
  const uint32_t t0 = (w & kMask) | kMagic;          // elements 0, 4
  const uint32_t t1 = ((w >> 4) & kMask) | kMagic;   // elements 1, 5
  const uint32_t t2 = ((w >> 8) & kMask) | kMagic;   // elements 2, 6
  const uint32_t t3 = ((w >> 12) & kMask) | kMagic;  // elements 3, 7
  uint4 o;
  o.x = deq_pair(__byte_perm(t0, t1, 0x5410), s2, b2);  // (0, 1)
  o.y = deq_pair(__byte_perm(t2, t3, 0x5410), s2, b2);  // (2, 3)
  o.z = deq_pair(__byte_perm(t0, t1, 0x7632), s2, b2);  // (4, 5)
  o.w = deq_pair(__byte_perm(t2, t3, 0x7632), s2, b2);  // (6, 7)
  return o;
}

// Byte offset of 16-byte chunk c (0..7) of row r in a 128-byte-swizzled K-major tile.
__device__ __forceinline__ uint32_t swz128(int r, int c) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint16_t pick16(const uint4& v, int g) {
  const uint32_t w = (g & 4) ? ((g & 2) ? v.w : v.z) : ((g & 2) ? v.y : v.x);
  return (uint16_t)((g & 1) ? (w >> 16) : (w & 0xFFFFu));
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmap_wq, const GemmArgs p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
  uint32_t* status = &p.header->status;
  auto bar = [&](int i) -> uint32_t { return sbase + OFF_BAR + 8u * (uint32_t)i; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar(b_nib_full(s)), 1);
      mbar_init(bar(b_nib_empty(s)), kDeqThreads);
      mbar_init(bar(b_a_full(s)), kDeqThreads);
      mbar_init(bar(b_b_full(s)), kGatherThreads);
      mbar_init(bar(b_ab_empty(s)), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(b_tmem_full(b)), 1);
      mbar_init(bar(b_tmem_empty(b)), 128);
    }
    mbar_init(bar(b_unwind()), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kTmaWarp && lane == 0) prefetch_tensormap(&tmap_wq);
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int H = p.H, F = p.F;
  const int G = H / BK;
  const int num_kb = G;
  const int n_ftiles = (F + BM - 1) / BM;
  const int n_units = p.header->n_chunks * n_ftiles;

  if (warp == kTmaWarp) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < n_units; u += gridDim.x) {
        const Unit U = decode_unit(p.chunks, u, n_ftiles);
        const int row0 = U.expert * F + U.f0;
        for (int kb = 0; kb < num_kb; ++kb) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
          if (!mbar_wait(bar(b_nib_empty(s)), ph ^ 1u, abort_flag, status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar(b_nib_full(s)), NIB_BYTES);
          tma_load_2d(sbase + OFF_NIB + s * NIB_BYTES, &tmap_wq, bar(b_nib_full(s)), kb * (BK / 2), row0);
          ++it;
        }
      }
      if (!ok) {  // unwinding: let the copies already issued land before the CTA exits
        const uint32_t first = it > STAGES ? it - STAGES : 0;
        for (uint32_t j = first; j < it; ++j)
          mbar_wait_unwind(bar(b_nib_full(j % STAGES)), (j / STAGES) & 1u, 100000000ull);
      }
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t it = 0, lu = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < n_units; u += gridDim.x, ++lu) {
        const Unit U = decode_unit(p.chunks, u, n_ftiles);
        const int N = (U.rows + 15) & ~15;
        const uint32_t idesc = umma_idesc_bf16(BM, N);
        const uint32_t ab = lu & 1u, aph = (lu >> 1) & 1u;
        if (!mbar_wait(bar(b_tmem_empty(ab)), aph ^ 1u, abort_flag, status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + ab * 256u;
        for (int kb = 0; kb < num_kb; ++kb) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
          if (!mbar_wait(bar(b_a_full(s)), ph, abort_flag, status) ||
              !mbar_wait(bar(b_b_full(s)), ph, abort_flag, status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc = umma_desc_sw128(sbase + OFF_A + s * A_BYTES);
          const uint64_t bdesc = umma_desc_sw128(sbase + OFF_B + s * B_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)  // advance 16 elements = 32 bytes along K
            tc_mma_bf16(d_tmem, adesc + 2u * k, bdesc + 2u * k, idesc, (kb > 0 || k > 0) ? 1u : 0u);
          tc_commit(bar(b_ab_empty(s)));
          ++it;
        }
        if (!ok) break;
        tc_commit(bar(b_tmem_full(ab)));
      }
      // every MMA issued above completes before this barrier's phase 0 completes
      tc_commit(bar(b_unwind()));
      mbar_wait_unwind(bar(b_unwind()), 0, 100000000ull);
      // and the stage-release arrivals of the last STAGES iterations have landed
      const uint32_t first = it > STAGES ? it - STAGES : 0;
      for (uint32_t j = first; j < it; ++j)
        mbar_wait_unwind(bar(b_ab_empty(j % STAGES)), (j / STAGES) & 1u, 100000000ull);
    }
  } else if (warp >= kGatherWarp0) {
    // ---------------------------------------------------------------- x row gather
    const int g = threadIdx.x - kGatherWarp0 * 32;
    const int cidx = g & 7;    // 16-byte chunk of the 128-byte row slice
    const int jrow0 = g >> 3;  // this thread handles rows jrow0 + 8 m
    uint32_t it = 0, issued = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < n_units; u += gridDim.x) {
      const Unit U = decode_unit(p.chunks, u, n_ftiles);
      int src_row[NMAX / 8];
#pragma unroll
      for (int m = 0; m < NMAX / 8; ++m) {
        const int j = jrow0 + 8 * m;
        src_row[m] = j < U.rows ? (p.perm ? __ldg(p.perm + U.start + j) : U.start + j) : -1;
      }
      for (int kb = 0; kb < num_kb; ++kb) {
        const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
        if (!mbar_wait(bar(b_ab_empty(s)), ph ^ 1u, abort_flag, status)) {
          ok = false;
          break;
        }
        const uint32_t bs = sbase + OFF_B + s * B_BYTES + jrow0 * 128 + ((cidx ^ jrow0) << 4);
        const __nv_bfloat16* xk = p.x + kb * BK + cidx * 8;
#pragma unroll
        for (int m = 0; m < NMAX / 8; ++m)
          if (src_row[m] >= 0) cp_async_16(bs + m * 1024, xk + (int64_t)src_row[m] * H);
        cp_async_commit();
        ++it;
        ++issued;
        if (issued > kGatherLag) {
          cp_async_wait<kGatherLag>();
          fence_proxy_async_smem();
          mbar_arrive(bar(b_b_full((it - 1 - kGatherLag) % STAGES)));
        }
      }
    }
    cp_async_wait<0>();
    fence_proxy_async_smem();
    if (ok) {
      const uint32_t first = it > (uint32_t)kGatherLag ? it - kGatherLag : 0;
      for (uint32_t j = first; j < it; ++j) mbar_arrive(bar(b_b_full(j % STAGES)));
    }
  } else if (warp >= kEpiWarp0) {
    // ---------------------------------------------------------------- epilogue
    const int ew = warp - kEpiWarp0;  // TMEM lanes 32 ew .. 32 ew + 31
    uint16_t* epi = reinterpret_cast<uint16_t*>(smem + OFF_EPI + ew * EPI_WARP_BYTES);
    const uint32_t epi_addr = sbase + OFF_EPI + ew * EPI_WARP_BYTES;
    uint32_t lu = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++lu) {
      const Unit U = decode_unit(p.chunks, u, n_ftiles);
      const int N = (U.rows + 15) & ~15;
      const uint32_t ab = lu & 1u, aph = (lu >> 1) & 1u;
      const bool okl = mbar_wait(bar(b_tmem_full(ab)), aph, abort_flag, status);
      if (!__all_sync(0xffffffffu, okl)) break;
      tc_fence_after();
      const uint32_t trow = tmem_base + ((uint32_t)(ew * 32) << 16) + ab * 256u;
      const int q = lane & 3;
      const int fcol = U.f0 + ew * 32 + q * 8;
      for (int c0 = 0; c0 < N; c0 += 16) {
        uint32_t v[16];
        tc_ld_32x32b_x16(trow + (uint32_t)c0, v);
        tc_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j)
          epi[j * 32 + lane] = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(v[j])));
        __syncwarp();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int jj = (lane >> 2) + 8 * h;
          const int tok = c0 + jj;
          if (tok < U.rows && fcol < F) {
            const int row = p.perm ? __ldg(p.perm + U.start + tok) : U.start + tok;
            uint4 val;
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(val.x), "=r"(val.y), "=r"(val.z), "=r"(val.w)
                         : "r"(epi_addr + (uint32_t)(jj * 64 + q * 16))
                         : "memory");
            *reinterpret_cast<uint4*>(p.y + (int64_t)row * F + fcol) = val;
          }
        }
        __syncwarp();
      }
      tc_fence_before();
      mbar_arrive(bar(b_tmem_empty(ab)));
    }
  } else {
    // ---------------------------------------------------------------- dequant
    const int t = threadIdx.x;  // 0..255
    const int r = t & (BM - 1);  // weight row within the tile
    const int half = t >> 7;     // which 32 of the 64 codes of the group
    const bool vec8 = (G & 7) == 0;  // scales/biases fetched 8 groups (16 bytes) at a time
    const int blk = vec8 ? 8 : 1;
    uint32_t it = 0;

    auto load_sb = [&](const Unit& U, int kb, uint4& s_out, uint4& b_out) {
      s_out = make_uint4(0, 0, 0, 0);
      b_out = make_uint4(0, 0, 0, 0);
      if (U.f0 + r < F) {
        const int64_t off = ((int64_t)U.expert * F + U.f0 + r) * G + kb;
        if (vec8) {
          s_out = __ldg(reinterpret_cast<const uint4*>(p.scales + off));
          b_out = __ldg(reinterpret_cast<const uint4*>(p.biases + off));
        } else {
          s_out.x = __ldg(reinterpret_cast<const uint16_t*>(p.scales) + off);
          b_out.x = __ldg(reinterpret_cast<const uint16_t*>(p.biases) + off);
        }
      }
    };

    int u = blockIdx.x;
    Unit U;
    uint4 s_cur, b_cur, s_nxt = make_uint4(0, 0, 0, 0), b_nxt = make_uint4(0, 0, 0, 0);
    if (u < n_units) {
      U = decode_unit(p.chunks, u, n_ftiles);
      load_sb(U, 0, s_cur, b_cur);
    }
    int kb = 0;
    while (u < n_units) {
      if (kb % blk == 0) {  // prefetch the next block of scales/biases
        int nkb = kb + blk, nu = u;
        if (nkb >= num_kb) {
          nkb = 0;
          nu = u + gridDim.x;
        }
        if (nu < n_units) {
          const Unit NU = (nu == u) ? U : decode_unit(p.chunks, nu, n_ftiles);
          load_sb(NU, nkb, s_nxt, b_nxt);
        }
      }
      const int gsel = vec8 ? (kb & 7) : 0;
      const uint32_t s2 = splat16(pick16(s_cur, gsel));
      const uint32_t b2 = splat16(pick16(b_cur, gsel));

      const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
      if (!mbar_wait(bar(b_nib_full(s)), ph, abort_flag, status)) break;
      uint4 nib;
      asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(nib.x), "=r"(nib.y), "=r"(nib.z), "=r"(nib.w)
                   : "r"(sbase + OFF_NIB + s * NIB_BYTES + r * 32 + half * 16)
                   : "memory");
      // The nibble stage is released only after the proxy fence below: the next TMA into
      // it is an async-proxy write, which is not ordered after these generic-proxy reads
      // by the mbarrier alone.
      const uint4 o0 = deq8(nib.x, s2, b2);
      const uint4 o1 = deq8(nib.y, s2, b2);
      const uint4 o2 = deq8(nib.z, s2, b2);
      const uint4 o3 = deq8(nib.w, s2, b2);
      if (!mbar_wait(bar(b_ab_empty(s)), ph ^ 1u, abort_flag, status)) break;
      const uint32_t a_tile = sbase + OFF_A + s * A_BYTES;
      const int c0 = half * 4;
      asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a_tile + swz128(r, c0 + 0)),
                   "r"(o0.x), "r"(o0.y), "r"(o0.z), "r"(o0.w) : "memory");
      asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a_tile + swz128(r, c0 + 1)),
                   "r"(o1.x), "r"(o1.y), "r"(o1.z), "r"(o1.w) : "memory");
      asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a_tile + swz128(r, c0 + 2)),
                   "r"(o2.x), "r"(o2.y), "r"(o2.z), "r"(o2.w) : "memory");
      asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a_tile + swz128(r, c0 + 3)),
                   "r"(o3.x), "r"(o3.y), "r"(o3.z), "r"(o3.w) : "memory");
      fence_proxy_async_smem();  // orders the A writes and the nibble reads before async-proxy use
      mbar_arrive(bar(b_a_full(s)));
      mbar_arrive(bar(b_nib_empty(s)));
      ++it;

      ++kb;
      if (kb % blk == 0) {
        s_cur = s_nxt;
        b_cur = b_nxt;
      }
      if (kb == num_kb) {
        kb = 0;
        u += gridDim.x;
        if (u < n_units) U = decode_unit(p.chunks, u, n_ftiles);
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem_base, kTmemCols);
}

struct DeviceInfo {
  int sms = 0;
  bool configured = false;
};

DeviceInfo g_dev[64];

}  // namespace

cudaError_t launch_gemm_tc(const GemmArgs& a, cudaStream_t s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  DeviceInfo& di = g_dev[dev];
  if (!di.configured) {
    e = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_DYN);
    if (e != cudaSuccess) return e;
    di.configured = true;
  }

  static decltype(&cuTensorMapEncodeTiled) encode = nullptr;
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
    encode = reinterpret_cast<decltype(&cuTensorMapEncodeTiled)>(fn);
  }
  CUtensorMap map;
  const cuuint64_t dims[2] = {(cuuint64_t)(a.H / 2), (cuuint64_t)a.E * (cuuint64_t)a.F};
  const cuuint64_t strides[1] = {(cuuint64_t)(a.H / 2)};
  const cuuint32_t box[2] = {BK / 2, BM};
  const cuuint32_t estr[2] = {1, 1};
  CUresult cr = encode(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(a.wq),
                                       dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                       CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return cudaErrorInvalidValue;
  gemm_tc_kernel<<<di.sms, kThreads, SMEM_DYN, s>>>(map, a);
  return cudaGetLastError();
}

}  // namespace gqmm
