// Persistent grouped GEMM for the quantized MoE gather matmul on tcgen05 tensor cores.
//
// Work unit = (chunk of one expert's sorted rows, pair of 128-row tiles of the expert's F
// outputs).  The product is computed transposed ("swap A/B"): the UMMA M slot (128) holds
// weight rows f, the N slot holds the chunk's tokens, so N = round_up(rows, 16) follows the
// rows per expert.  This is the tensor-core form of the lesson in mlx PR #4023 "Pick BM from
// rows per expert in gather_qmm_rhs_nax" (useful arithmetic ~ min(1, run / BM)): a 4-row run
// costs an N=16 MMA instead of most of a 64- or 128-row tile, and each expert's weight tile is
// read and dequantized once per chunk of up to 256 rows instead of once per row (mlx #4339,
// comment by manunicholasjacob: one CTA per token-expert pair, 15 of 16 tile rows empty, the
// 4-bit slab dequantized once per row).  The two tiles of a unit share every x tile, which
// halves the x bytes moved per FLOP compared with one tile per unit.
//
// Per CTA (one per SM, persistent, static round-robin over units), warp roles:
//   warps 0-15  dequant:  two groups of 256 threads take alternate k-blocks; a thread owns one
//                         of the unit's 256 weight rows: reads its 32 bytes of codes, computes
//                         w = scale*q + bias in bf16x2 and writes the 64 bf16 in the
//                         128-byte-swizzle K-major A layout
//   warps 16-23 epilogue: warp 16+e drains TMEM lanes 32(e%4).. of tile e/4: TMEM -> registers
//                         -> bf16 -> shared transpose -> 16-byte stores to y rows perm[j]
//   warp 24     TMA:      one thread streams the unit's 256 x 32-byte nibble tile per k-block
//   warp 25     MMA:      allocates TMEM (two 256-column fp32 accumulators), one thread issues
//                         tcgen05.mma 128xNx16, four per tile per k-block, commits to mbarriers
//   warps 26-31 gather:   warps 26+2s and 27+2s own pipeline stage s: whenever the stage is free
//                         they copy the chunk's x rows perm[j] (128 bytes each) with 16-byte
//                         cp.async into the swizzled B tile, wait for their own copies, fence
//                         them for the tensor core and mark the stage full.  Each lane keeps its
//                         32 source rows in registers for the whole unit, so a stage's copies
//                         issue back to back.  (TMA tile::gather4 was measured at ~80 cycles per
//                         512-byte gather per SM: too slow for 128-byte rows.)
// Pipeline depth: 3 stages of (A 2 x 16 KB, B 32 KB, nibbles 8 KB).  The accumulators use all
// 512 TMEM columns, so the MMA of a unit starts once the epilogue has drained the previous one;
// the producers keep filling stages meanwhile.
//
// Every wait is bounded (mbar_wait): on expiry the CTA raises GQMM_STATUS_TIMEOUT, unwinds,
// waits (bounded) for its own copies and MMAs in flight and frees its TMEM.
#include "gqmm_internal.cuh"

namespace gqmm {
namespace {

constexpr int BM = 128;                  // weight rows per tile (UMMA M)
constexpr int NT = 2;                    // tiles per unit
constexpr int UM = BM * NT;              // weight rows per unit
constexpr int BK = 64;                   // K per stage = one quantization group
constexpr int NMAX = kChunkMaxRows;      // tokens per unit, UMMA N <= 256
constexpr int STAGES = 3;
constexpr int A_TILE_BYTES = BM * BK * 2;      // 16 KB bf16
constexpr int A_BYTES = NT * A_TILE_BYTES;     // 32 KB
constexpr int B_BYTES = NMAX * BK * 2;         // 32 KB bf16
constexpr int NIB_BYTES = UM * BK / 2;         // 8 KB packed codes
constexpr int EPI_WARP_BYTES = 16 * 32 * 2;

constexpr int kThreads = 1024;
constexpr int kDeqGroup = UM;            // threads per dequant group (one per weight row)
constexpr int kDeqGroups = 2;            // warps 0-15
constexpr int kEpiWarp0 = 16;            // warps 16-23
constexpr int kEpiWarps = 4 * NT;
constexpr int kTmaWarp = 24;
constexpr int kMmaWarp = 25;
constexpr int kGatherWarp0 = 26;         // warps 26 .. 31, a pair per stage
constexpr uint32_t kTmemCols = 512;      // NT accumulators of NMAX fp32 columns
static_assert(kGatherWarp0 + 2 * STAGES == kThreads / 32, "warp roles fill the block");
static_assert(kDeqGroup * kDeqGroups == kEpiWarp0 * 32, "dequant warps");

constexpr int OFF_A = 0;
constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
constexpr int OFF_NIB = OFF_B + STAGES * B_BYTES;
constexpr int OFF_EPI = OFF_NIB + STAGES * NIB_BYTES;
constexpr int OFF_BAR = OFF_EPI + kEpiWarps * EPI_WARP_BYTES;
constexpr int NUM_BARS = 5 * STAGES + 3;
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
__device__ __forceinline__ int b_tmem_full() { return 5 * STAGES; }
__device__ __forceinline__ int b_tmem_empty() { return 5 * STAGES + 1; }
__device__ __forceinline__ int b_unwind() { return 5 * STAGES + 2; }

struct Unit {
  int expert, start, rows, f0;
};

__device__ __forceinline__ Unit decode_unit(const Chunk* chunks, int u, int n_fpairs) {
  const int c = u / n_fpairs;
  const int fp = u - c * n_fpairs;
  const int4 ch = __ldg(reinterpret_cast<const int4*>(chunks) + c);
  Unit U;
  U.expert = ch.x;
  U.start = ch.y;
  U.rows = ch.z;
  U.f0 = fp * UM;
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
      mbar_init(bar(b_nib_empty(s)), kDeqGroup);  // the dequant group that consumed it
      mbar_init(bar(b_a_full(s)), kDeqGroup);
      mbar_init(bar(b_b_full(s)), 64);            // every lane of the stage's two gather warps
      mbar_init(bar(b_ab_empty(s)), 1);
    }
    mbar_init(bar(b_tmem_full()), 1);
    mbar_init(bar(b_tmem_empty()), kEpiWarps * 32);
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
  const int n_fpairs = (F + UM - 1) / UM;
  const int n_units = p.header->n_chunks * n_fpairs;

  if (warp == kTmaWarp) {
    // ---------------------------------------------------------------- TMA producer (nibbles)
    // Besides the stage loads, the tile kPrefetchAhead k-blocks ahead (possibly in the next
    // unit) is prefetched into L2, so stage loads see L2 rather than HBM latency: with only
    // three stages the loads themselves cannot run far enough ahead.
    if (lane == 0) {
      constexpr int kPrefetchAhead = 6;
      auto prefetch = [&](int u, int kb) {
        while (kb >= num_kb && u < n_units) {
          kb -= num_kb;
          u += gridDim.x;
        }
        if (u < n_units) {
          const Unit V = decode_unit(p.chunks, u, n_fpairs);
          tma_prefetch_l2_2d(&tmap_wq, kb * (BK / 2), V.expert * F + V.f0);
        }
      };
      for (int j = 0; j < kPrefetchAhead; ++j) prefetch(blockIdx.x, j);
      uint32_t it = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < n_units; u += gridDim.x) {
        const Unit U = decode_unit(p.chunks, u, n_fpairs);
        const int row0 = U.expert * F + U.f0;
        for (int kb = 0; kb < num_kb; ++kb) {
          prefetch(u, kb + kPrefetchAhead);
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
        const Unit U = decode_unit(p.chunks, u, n_fpairs);
        const int N = (U.rows + 15) & ~15;
        const uint32_t idesc = umma_idesc_bf16(BM, N);
        if (!mbar_wait(bar(b_tmem_empty()), (lu & 1u) ^ 1u, abort_flag, status)) break;
        tc_fence_after();
        for (int kb = 0; kb < num_kb; ++kb) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
          if (!mbar_wait(bar(b_a_full(s)), ph, abort_flag, status) ||
              !mbar_wait(bar(b_b_full(s)), ph, abort_flag, status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t bdesc = umma_desc_sw128(sbase + OFF_B + s * B_BYTES);
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            const uint64_t adesc = umma_desc_sw128(sbase + OFF_A + s * A_BYTES + t * A_TILE_BYTES);
#pragma unroll
            for (int k = 0; k < BK / 16; ++k)  // advance 16 elements = 32 bytes along K
              tc_mma_bf16(tmem_base + (uint32_t)(t * NMAX), adesc + 2u * k, bdesc + 2u * k, idesc,
                          (kb > 0 || k > 0) ? 1u : 0u);
          }
          tc_commit(bar(b_ab_empty(s)));
          ++it;
        }
        if (!ok) break;
        tc_commit(bar(b_tmem_full()));
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
    const uint32_t gs = (uint32_t)(warp - kGatherWarp0) >> 1;  // the stage this warp pair fills
    const int h = (warp - kGatherWarp0) & 1;
    const int cidx = lane & 7;                 // 16-byte chunk of a 128-byte row slice
    const int rlow = 4 * h + (lane >> 3);      // rows 8 q + rlow, q = 0..31
    const uint32_t dst_lane = (uint32_t)(rlow * 128 + ((cidx ^ rlow) << 4));
    uint32_t it = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < n_units; u += gridDim.x) {
      const Unit U = decode_unit(p.chunks, u, n_fpairs);
      int src[NMAX / 8];
#pragma unroll
      for (int q = 0; q < NMAX / 8; ++q) {
        const int row = 8 * q + rlow;
        src[q] = row < U.rows ? (p.perm ? __ldg(p.perm + U.start + row) : U.start + row) : -1;
      }
      for (int kb = 0; kb < num_kb; ++kb, ++it) {
        if (it % STAGES != gs) continue;
        const uint32_t ph = (it / STAGES) & 1u;
        const bool okl = mbar_wait(bar(b_ab_empty(gs)), ph ^ 1u, abort_flag, status);
        if (!__all_sync(0xffffffffu, okl)) {
          ok = false;
          break;
        }
        const uint32_t b_lane = sbase + OFF_B + gs * B_BYTES + dst_lane;
        const __nv_bfloat16* xk = p.x + kb * BK + cidx * 8;
#pragma unroll
        for (int q = 0; q < NMAX / 8; ++q)
          if (src[q] >= 0) cp_async_16(b_lane + q * 1024, xk + (int64_t)src[q] * H);
        cp_async_commit();
        cp_async_wait<0>();
        fence_proxy_async_smem();  // this lane's copies, made visible to the tensor core
        mbar_arrive(bar(b_b_full(gs)));
      }
    }
    cp_async_wait<0>();
  } else if (warp >= kEpiWarp0) {
    // ---------------------------------------------------------------- epilogue
    const int ew = warp - kEpiWarp0;
    const int tile = ew >> 2;          // accumulator (weight-row tile) this warp drains
    const int quarter = ew & 3;        // TMEM lanes 32 quarter .. 32 quarter + 31 (= warp % 4)
    uint16_t* epi = reinterpret_cast<uint16_t*>(smem + OFF_EPI + ew * EPI_WARP_BYTES);
    const uint32_t epi_addr = sbase + OFF_EPI + ew * EPI_WARP_BYTES;
    uint32_t lu = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++lu) {
      const Unit U = decode_unit(p.chunks, u, n_fpairs);
      const int N = (U.rows + 15) & ~15;
      const bool okl = mbar_wait(bar(b_tmem_full()), lu & 1u, abort_flag, status);
      if (!__all_sync(0xffffffffu, okl)) break;
      tc_fence_after();
      const uint32_t trow = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(tile * NMAX);
      const int q = lane & 3;
      const int fcol = U.f0 + tile * BM + quarter * 32 + q * 8;
      for (int c0 = 0; c0 < N; c0 += 16) {
        uint32_t v[16];
        tc_ld_32x32b_x16(trow + (uint32_t)c0, v);
        tc_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j)
          epi[j * 32 + lane] = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(v[j])));
        __syncwarp();
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int jj = (lane >> 2) + 8 * hh;
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
      mbar_arrive(bar(b_tmem_empty()));
    }
  } else {
    // ---------------------------------------------------------------- dequant
    const int t = threadIdx.x;                   // 0 .. 2 * UM - 1
    const int r = t % UM;                        // weight row within the unit
    const uint32_t grp = (uint32_t)(t / UM);     // handles the steps with it % 2 == grp
    const int tile = r >> 7, rr = r & (BM - 1);
    // nibble tile rows are 32 bytes, TMA-swizzled in 32-byte mode: 16-byte chunk c of row r
    // sits at chunk position c ^ ((r >> 2) & 1)
    const uint32_t nib_row = (uint32_t)(r * 32);
    const uint32_t nib_c0 = (uint32_t)(((r >> 2) & 1) << 4), nib_c1 = nib_c0 ^ 16u;
    const uint32_t a_off = (uint32_t)(tile * A_TILE_BYTES + (rr >> 3) * 1024 + (rr & 7) * 128);
    const uint16_t* sc16 = reinterpret_cast<const uint16_t*>(p.scales);
    const uint16_t* bs16 = reinterpret_cast<const uint16_t*>(p.biases);
    // Flat walk over (unit, k-block); this group processes every second step.  The scale and
    // bias of the next step it processes are loaded one processed step ahead.
    struct Step {
      int u, kb;
      Unit U;
    };
    auto advance = [&](Step& st, int by) {
      st.kb += by;
      while (st.kb >= num_kb && st.u < n_units) {
        st.kb -= num_kb;
        st.u += gridDim.x;
        if (st.u < n_units) st.U = decode_unit(p.chunks, st.u, n_fpairs);
      }
    };
    auto load_sb = [&](const Step& st, uint32_t& sv, uint32_t& bv) {
      sv = 0;
      bv = 0;
      if (st.u < n_units && st.U.f0 + r < F) {
        const int64_t off = ((int64_t)st.U.expert * F + st.U.f0 + r) * G + st.kb;
        sv = __ldg(sc16 + off);
        bv = __ldg(bs16 + off);
      }
    };
    Step cur;
    cur.u = blockIdx.x;
    cur.kb = 0;
    if (cur.u < n_units) cur.U = decode_unit(p.chunks, cur.u, n_fpairs);
    advance(cur, (int)grp);
    uint32_t it = grp;  // global step index of cur
    uint32_t s_cur, b_cur;
    load_sb(cur, s_cur, b_cur);
    while (cur.u < n_units) {
      Step nxt = cur;
      advance(nxt, kDeqGroups);
      uint32_t s_nxt, b_nxt;
      load_sb(nxt, s_nxt, b_nxt);
      const uint32_t s2 = splat16(s_cur), b2 = splat16(b_cur);
      const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
      if (!mbar_wait(bar(b_nib_full(s)), ph, abort_flag, status)) break;
      const uint32_t nib_tile = sbase + OFF_NIB + s * NIB_BYTES + nib_row;
      uint4 n0, n1;
      asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(n0.x), "=r"(n0.y), "=r"(n0.z), "=r"(n0.w)
                   : "r"(nib_tile + nib_c0)
                   : "memory");
      asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(n1.x), "=r"(n1.y), "=r"(n1.z), "=r"(n1.w)
                   : "r"(nib_tile + nib_c1)
                   : "memory");
      // The nibble stage is released only after the proxy fence below: the next TMA into
      // it is an async-proxy write, which is not ordered after these generic-proxy reads
      // by the mbarrier alone.
      uint4 o[8];
      o[0] = deq8(n0.x, s2, b2);
      o[1] = deq8(n0.y, s2, b2);
      o[2] = deq8(n0.z, s2, b2);
      o[3] = deq8(n0.w, s2, b2);
      o[4] = deq8(n1.x, s2, b2);
      o[5] = deq8(n1.y, s2, b2);
      o[6] = deq8(n1.z, s2, b2);
      o[7] = deq8(n1.w, s2, b2);
      if (!mbar_wait(bar(b_ab_empty(s)), ph ^ 1u, abort_flag, status)) break;
      const uint32_t a_row = sbase + OFF_A + s * A_BYTES + a_off;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a_row + (uint32_t)((c ^ (rr & 7)) << 4)),
                     "r"(o[c].x), "r"(o[c].y), "r"(o[c].z), "r"(o[c].w)
                     : "memory");
      fence_proxy_async_smem();  // orders the A writes and the nibble reads before async-proxy use
      mbar_arrive(bar(b_a_full(s)));
      mbar_arrive(bar(b_nib_empty(s)));
      cur = nxt;
      s_cur = s_nxt;
      b_cur = b_nxt;
      it += kDeqGroups;
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
  // Packed codes as a [E*F, H/2] byte matrix; one box = the unit's 256 rows x 32 bytes (one
  // 64-wide group), 32-byte swizzled so the dequant threads read it without bank conflicts.
  CUtensorMap map_wq;
  const cuuint64_t dims[2] = {(cuuint64_t)(a.H / 2), (cuuint64_t)a.E * (cuuint64_t)a.F};
  const cuuint64_t strides[1] = {(cuuint64_t)(a.H / 2)};
  const cuuint32_t box[2] = {BK / 2, UM};
  const cuuint32_t estr[2] = {1, 1};
  CUresult cr = encode(&map_wq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(a.wq), dims, strides, box,
                       estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return cudaErrorInvalidValue;
  gemm_tc_kernel<<<di.sms, kThreads, SMEM_DYN, s>>>(map_wq, a);
  return cudaGetLastError();
}

}  // namespace gqmm
