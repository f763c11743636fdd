// Persistent grouped GEMM for the quantized MoE gather matmul on tcgen05 tensor cores.
//
// Work unit = (chunk of one expert's sorted rows, pair of 128-row tiles of the expert's F
// outputs, K slice).  The product is computed transposed ("swap A/B"): the UMMA M slot (128)
// holds weight rows f, the N slot holds the chunk's tokens, so N = round_up(rows, 16) follows
// the rows per expert.  This is the tensor-core form of the lesson in mlx PR #4023 "Pick BM
// from rows per expert in gather_qmm_rhs_nax" (useful arithmetic ~ min(1, run / BM)): a 4-row
// run costs an N=16 MMA instead of most of a 64- or 128-row tile, and each expert's weight
// tile is read and dequantized once per chunk instead of once per row (mlx #4339, comment by
// manunicholasjacob: one CTA per token-expert pair, 15 of 16 tile rows empty, the 4-bit slab
// dequantized once per row).  The two tiles of a unit share every x tile, which halves the x
// bytes moved per FLOP compared with one tile per unit.  For decode-sized calls (mlxcel #725
// "amortizing small-M quantized GEMM": per-row qmv re-reads the weights, a 128-wide tile is
// 94% wasted) the same kernel reads each weight tile once per call for all of its M <= 8 rows.
//
// Three variants (template Cfg), chosen on the host from the rows per expert:
//   wide    chunks of <= 256 rows; 3 stages of (A 2 x 16 KB, x 32 KB) and 3 of codes (8 KB); the
//           MMA is M = 128 weight rows x N = the chunk's rows, two tiles per unit
//   narrow  chunks of <= 32 rows, and mid chunks of <= 128 rows (4-bit affine codes): the operands
//           swap places (SWAP: M = 128 token rows, N = the unit's 256 weight rows), so a k-block
//           is 4 full-size MMAs instead of 8 small ones, and a unit's accumulator (token lanes x
//           256 columns) takes half of tensor memory: the epilogue of one unit runs under the
//           MMAs of the next.  4 (mid: 3) stages of (A 32 KB, x 4 KB (mid: 16 KB)), 9 of codes.
// The kernel is also templated on the weight format (formats.cuh: affine codes of 2-8 bits,
// mxfp4 / nvfp4 / mxfp8, and transpose=False affine weights), which sets the code tile of a
// k-block and the dequant arithmetic; the rest is shared.
// Calls with too few units for the GPU (dense decode: F/256 units) split K into slices; each
// slice stores its fp32 partial sums in its own plane of a workspace buffer, and a second
// kernel adds the planes in slice order (so results are deterministic) into bf16 y.
//
// Per CTA (one per SM, persistent; units taken from a call-wide counter), warp roles (the
// warp numbers are the wide variant's; the narrow and mid ones have 3 dequant groups, warps
// 0-23, 4 epilogue warps (one per TMEM lane quarter: 32 tokens each), and 2 gather warps):
//   warps 0-15  dequant:  two groups of 256 threads take alternate k-blocks; a thread owns one
//                         of the unit's 256 weight rows: reads its 32 bytes of codes, turns each
//                         nibble pair into bf16 128 + q (one byte permute and one mask per pair),
//                         computes w = scale*q + bias in bf16x2 and writes the 64 bf16 into the
//                         K-major A tile (unswizzled core-matrix layout)
//   warps 16-23 epilogue: warp 16+e drains TMEM lanes 32(e%4).. of tile e/4: TMEM -> registers
//                         -> bf16 -> shared transpose -> 16-byte stores to y rows perm[j]
//                         (or fp32 stores into the slice's plane of the split-K sums)
//   warp 24     scheduler + TMA: one thread takes the next unit from the call-wide counter,
//                         pushes it into the CTA's unit queue (read by every other warp) and
//                         streams the unit's 256 x 32-byte code tile per k-block
//   warp 25     MMA:      allocates TMEM (two 256-column fp32 accumulators), one thread issues
//                         tcgen05.mma 128xNx16, four per tile per k-block, commits to mbarriers
//   warps 26-31 gather:   the chunk's x rows perm[j] (128 bytes per k-block) come by TMA
//                         tile::gather4, four rows per copy, into the 128-byte-swizzled x tile;
//                         the copies of a stage are spread over the six warps (one per lane), so
//                         the TMA engine gets many issuers, and no warp waits for its data: the
//                         copies complete the stage's full barrier.  (Measured on all SMs with
//                         random 128-byte rows: cp.async from 2 warps moves ~9 B/clk/SM and from
//                         16 warps ~23; gather4 from one thread ~7, from 8 warps ~26.)
// The wide variant's accumulators use all 512 TMEM columns, so the MMA of a unit starts once the
// epilogue has drained the previous one; the producers keep filling stages meanwhile.
//
// Every wait is bounded (mbar_wait): on expiry the CTA raises GQMM_STATUS_TIMEOUT, unwinds,
// waits (bounded) for its own copies and MMAs in flight and frees its TMEM.
#include "formats.cuh"
#include "gqmm_internal.cuh"

namespace gqmm {
namespace {

constexpr int BM = 128;                  // weight rows per tile (UMMA M)
constexpr int NT = 2;                    // tiles per unit
constexpr int UM = BM * NT;              // weight rows per unit
static_assert(UM == kUnitRows, "unit height");
constexpr int BK = 64;                   // K per stage = one quantization group
constexpr int A_TILE_BYTES = BM * BK * 2;      // 16 KB bf16
constexpr int EPI_WARP_BYTES = 16 * 32 * 2;

constexpr int kThreads = 1024;
constexpr uint32_t kTmemCols = 512;      // the whole tensor memory of the SM

// A work unit as the scheduler hands it to the CTA's roles (one entry of the unit queue), or
// the end of the work (valid == 0).
struct UnitEntry {
  int expert, start, rows;  // chunk: expert id, first sorted position, rows
  int f0;                   // first weight row (output column) of the unit's 256
  int kb0, kb1;             // k-blocks [kb0, kb1) of the unit's K slice
  int ks;                   // K slice index when K is split, else -1
  int valid;
};
constexpr int kUnitQ = 8;  // queue depth: how far the scheduler may run ahead of the epilogue

// Variant: largest chunk (UMMA N), code ring depth, and the warp roles: DEQ_GROUPS groups of 8
// dequant warps (warps 0 ..), EPI_WARPS epilogue warps, then the scheduler/TMA warp, the MMA
// warp and the gather warps.  PAIR: a cluster of two CTAs computes each unit with cta_group::2
// MMAs of M = 256 and units of up to 512 tokens (see the pair notes at the top of the kernel).
// SWAP: the operands trade places: the chunk's x rows are the MMA's A (M = 128 token rows; rows
// past the chunk's end are never stored) and the unit's 256 dequantized weight rows its B (N = 256),
// so a k-block takes 4 MMAs of 128 x 256 x 16 instead of 8 of 128 x NMAX x 16, and each unit's
// accumulator (token lanes x 256 weight-row columns) takes 256 columns: two fit in tensor memory,
// so the epilogue of one unit overlaps the MMAs of the next.
template <int NMAX_, int NIB_STAGES_, int DEQ_GROUPS_, int EPI_WARPS_, int AB_STAGES_, int W_ = 32,
          bool SWAP_ = false, bool PAIR_ = false>
struct Cfg {
  static constexpr bool SWAP = SWAP_;
  static constexpr bool PAIR = PAIR_;
  static constexpr int NMAX = NMAX_;              // rows per chunk = largest UMMA N (SWAP: at most M)
  static constexpr int NIB_STAGES = NIB_STAGES_;  // code ring depth
  static constexpr int W = W_;                    // bytes of a weight row's code window per k-block
  static constexpr int ROWS = PAIR ? BM : UM;     // weight rows of a unit this CTA dequantizes
  static constexpr int CT = PAIR ? 1 : NT;        // A tiles of a stage in this CTA
  static constexpr int A_BYTES = CT * A_TILE_BYTES;
  static constexpr int NIB_BYTES = ROWS * W;      // one code stage: this CTA's rows' windows
  // AB_STAGES = depth of the A (dequantized weights) / x ring.  Tensor memory: accumulators of
  // NMAX columns per tile at column tile * ACC_COLS (SWAP: one accumulator of 256 columns per
  // unit, in one of two slots; PAIR: this CTA's 128 weight rows x the unit's up to 512 tokens,
  // column = token).
  static constexpr int AB_STAGES = AB_STAGES_;
  static constexpr int ACC_COLS = SWAP ? UM : NMAX;
  static constexpr int SLOTS = SWAP ? 2 : 1;
  static_assert((SWAP ? SLOTS : PAIR ? 1 : NT) * ACC_COLS <= (int)kTmemCols, "accumulators fit in tensor memory");
  static_assert(!SWAP || NMAX <= BM, "SWAP: chunks of at most M rows");
  static_assert(!PAIR || (!SWAP && NMAX == 2 * UM), "PAIR: units of up to 512 tokens, two N tiles of 256");
  static constexpr int DEQ_GROUPS = DEQ_GROUPS_;  // dequant groups of ROWS threads, alternate steps
  static constexpr int EPI_WARPS = EPI_WARPS_;    // 4 * NT (one tile each) or 4 (both tiles each)
  static constexpr int EPI_WARP0 = DEQ_GROUPS * ROWS / 32;
  static constexpr int TMA_WARP = EPI_WARP0 + EPI_WARPS;
  static constexpr int MMA_WARP = TMA_WARP + 1;
  static constexpr int GATHER_WARP0 = MMA_WARP + 1;
  static constexpr int GATHER_WARPS = kThreads / 32 - GATHER_WARP0;
  static constexpr int TILES_PER_EPI_WARP = NT * 4 / EPI_WARPS;
  // warps that pop every unit: all but the scheduler's
  static constexpr int UNIT_CONSUMER_WARPS = EPI_WARP0 + EPI_WARPS + GATHER_WARPS + 1;
  static_assert(GATHER_WARPS >= 1 && UNIT_CONSUMER_WARPS == kThreads / 32 - 1, "warp roles fill the block");
  // releases of a unit-queue entry the scheduler waits for (PAIR: the odd CTA's warps too, its
  // scheduler warp among them, which loads that CTA's codes)
  static constexpr int UQ_RELEASES = PAIR ? UNIT_CONSUMER_WARPS + kThreads / 32 : UNIT_CONSUMER_WARPS;
  static_assert(EPI_WARPS % 4 == 0 && (NT * 4) % EPI_WARPS == 0, "epilogue warps cover the TMEM lane quarters");
  static_assert(NIB_STAGES > DEQ_GROUPS && AB_STAGES >= DEQ_GROUPS, "a step advances the rings by DEQ_GROUPS");
  // x rows of a stage in this CTA (PAIR: its halves of the two N tiles, 128 rows apart)
  static constexpr int B_ROWS = PAIR ? NMAX / 2 : NMAX;
  static constexpr int B_BYTES = B_ROWS * BK * 2;
  // SWAP: the x stages come first: the MMA reads 128 rows (16 KB) from an x stage's start, past its
  // NMAX written rows into the following stages (rows whose results are never stored), which keeps
  // every read inside the block's shared memory
  static constexpr int OFF_A = SWAP ? AB_STAGES * B_BYTES : 0;
  static constexpr int OFF_B = SWAP ? 0 : OFF_A + AB_STAGES * A_BYTES;
  static constexpr int OFF_NIB = SWAP ? OFF_A + AB_STAGES * A_BYTES : OFF_B + AB_STAGES * B_BYTES;
  static_assert(!SWAP || (AB_STAGES - 1) * B_BYTES + BM * BK * 2 <= OFF_NIB, "SWAP: the A reads stay inside");
  static constexpr int OFF_EPI = OFF_NIB + NIB_STAGES * NIB_BYTES;
  static constexpr int OFF_BAR = OFF_EPI + EPI_WARPS * EPI_WARP_BYTES;
  static constexpr int NUM_BARS = 2 * NIB_STAGES + 2 * AB_STAGES + 5 + 2 * kUnitQ;
  static constexpr int OFF_MISC = OFF_BAR + ((NUM_BARS * 8 + 127) / 128) * 128;
  static constexpr int OFF_UQ = OFF_MISC + 16;
  static constexpr int SMEM_DYN = OFF_UQ + kUnitQ * 32 + 1024;  // room to align the base to 1024 bytes
  static_assert(SMEM_DYN <= 232448, "fits the 227 KB opt-in shared memory of one CTA");
  static_assert(B_BYTES % 1024 == 0, "x tiles stay 1024-byte aligned");
  // barrier slots
  __device__ static int nib_full(int s) { return s; }
  __device__ static int nib_empty(int s) { return NIB_STAGES + s; }
  // A tile and x tile of a stage are both written: the stage's dequant group (256 arrivals)
  // and the six gather warps (one arrival with their byte count each, plus the copies'
  // completed bytes) arrive on one barrier, so the MMA thread probes once per
  // k-block (a probe costs ~160 cycles even when the phase is already complete, which at
  // N=16 is more than half the MMA time of the k-block).
  __device__ static int ab_full(int s) { return 2 * NIB_STAGES + s; }
  __device__ static int ab_empty(int s) { return 2 * NIB_STAGES + AB_STAGES + s; }
  __device__ static int tmem_full(int slot) { return 2 * NIB_STAGES + 2 * AB_STAGES + slot; }
  __device__ static int tmem_empty(int slot) { return 2 * NIB_STAGES + 2 * AB_STAGES + 2 + slot; }
  __device__ static int unwind() { return 2 * NIB_STAGES + 2 * AB_STAGES + 4; }
  __device__ static int uq_full(int q) { return 2 * NIB_STAGES + 2 * AB_STAGES + 5 + q; }
  __device__ static int uq_empty(int q) { return 2 * NIB_STAGES + 2 * AB_STAGES + 5 + kUnitQ + q; }
};
// wide: 2 dequant groups, 8 epilogue warps, 6 gather warps (x tiles of up to 256 rows need
// many TMA issuers).  narrow / mid: the x tile is at most 32 / 128 rows, so 2 gather warps and 4
// epilogue warps suffice and a third dequant group takes the rest.
using CfgWide = Cfg<kChunkRowsWide, 3, 2, 8, 3>;
// Other code-window widths (formats.cuh): 16 bytes (2-bit affine); 48 and 64 bytes (3-, 5-, 6-
// and 8-bit affine, mxfp8).  The wide variants for 48- and 64-byte windows have a two-stage A / x
// ring, which leaves room for the larger code stages (4 x 12 KB, 3 x 16 KB).
using CfgWide16 = Cfg<kChunkRowsWide, 3, 2, 8, 3, 16>;
using CfgWide48 = Cfg<kChunkRowsWide, 4, 2, 8, 2, 48>;
using CfgWide64 = Cfg<kChunkRowsWide, 3, 2, 8, 2, 64>;
// narrow (SWAP): x stages of 4 KB ahead of 32 KB weight stages, a 4-deep ring, and as many code
// stages as fit
using CfgSwap = Cfg<kChunkRowsNarrow, 9, 3, 4, 4, 32, true>;
using CfgSwap16 = Cfg<kChunkRowsNarrow, 12, 3, 4, 4, 16, true>;
using CfgSwap48 = Cfg<kChunkRowsNarrow, 4, 3, 4, 4, 48, true>;
using CfgSwap64 = Cfg<kChunkRowsNarrow, 4, 3, 4, 4, 64, true>;
// mid (SWAP, 4-bit affine codes): the same with 16 KB x stages and a 3-deep ring
using CfgSwapMid = Cfg<kChunkRowsMid, 9, 3, 4, 3, 32, true>;
// CTA pairs (4-bit affine, chunks of up to 512 rows): per CTA 128 weight rows and up to 256 x rows a
// unit, so a stage is 16 + 32 KB: a 4-deep ring, a 5-deep code ring, four dequant groups of 128
using CfgPair = Cfg<kChunkRowsPair, 5, 4, 8, 4, 32, false, true>;

__device__ __forceinline__ UnitEntry decode_unit(const Chunk* chunks, int u, int n_fpairs, int ksplit, int num_kb) {
  const int ks = u % ksplit;
  const int t = u / ksplit;
  const int c = t / n_fpairs;
  const int fp = t - c * n_fpairs;
  const int4 ch = __ldg(reinterpret_cast<const int4*>(chunks) + c);
  UnitEntry U;
  U.expert = ch.x;
  U.start = ch.y;
  U.rows = ch.z;
  U.f0 = fp * UM;
  U.kb0 = (int)((int64_t)num_kb * ks / ksplit);
  U.kb1 = (int)((int64_t)num_kb * (ks + 1) / ksplit);
  U.ks = ksplit > 1 ? ks : -1;
  U.valid = 1;
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

// 8 codes (one 32-bit word, element k in bits 4k..4k+3) -> 8 bf16 in element order.  Output
// pair j takes byte j of w (elements 2j, 2j+1 in its nibbles) into byte 0 and byte j of w >> 4
// (element 2j+1 in its low nibble) into byte 2; the mask keeps the two low nibbles and the
// magic makes them bf16 128 + q.
__device__ __forceinline__ uint4 deq8(uint32_t w, uint32_t s2, uint32_t b2) {
  constexpr uint32_t kMask = 0x000F000Fu, kMagic = 0x43004300u;  // bf16 128.0 in each half
  const uint32_t ws = w >> 4;
  uint4 o;
  o.x = deq_pair((__byte_perm(w, ws, 0x0400) & kMask) | kMagic, s2, b2);  // (0, 1)
  o.y = deq_pair((__byte_perm(w, ws, 0x0501) & kMask) | kMagic, s2, b2);  // (2, 3)
  o.z = deq_pair((__byte_perm(w, ws, 0x0602) & kMask) | kMagic, s2, b2);  // (4, 5)
  o.w = deq_pair((__byte_perm(w, ws, 0x0703) & kMask) | kMagic, s2, b2);  // (6, 7)
  return o;
}

template <class C, class FMT>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmap_wq, const __grid_constant__ CUtensorMap tmap_x,
                   const GemmArgs p) {
  constexpr int NIB_STAGES = C::NIB_STAGES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  volatile UnitEntry* uq = reinterpret_cast<volatile UnitEntry*>(smem + C::OFF_UQ);
  uint32_t* status = &p.header->status;
  auto bar = [&](int i) -> uint32_t { return sbase + C::OFF_BAR + 8u * (uint32_t)i; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // CTA pairs: rank 0 (the even CTA) schedules the units and issues the MMAs; rank 1 holds weight
  // rows 128.. of each unit and the second half of each N tile's x rows.  The unit queue's entries
  // are written into the odd CTA by the even one, so its barriers are released and acquired at
  // cluster scope; the per-stage and per-accumulator handshakes are plain remote arrivals.
  constexpr bool PAIR = C::PAIR;
  const uint32_t crank = PAIR ? cluster_ctarank() : 0u;
  const bool leader = crank == 0;
  const int rbase = PAIR ? (int)crank * BM : 0;  // first weight row of the unit in this CTA
  auto peer_bar = [&](int i) -> uint32_t { return mapa_shared(bar(i), crank ^ 1u); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < NIB_STAGES; ++s) {
      mbar_init(bar(C::nib_full(s)), 1);
      mbar_init(bar(C::nib_empty(s)), C::ROWS / 32);  // one arrival per warp of the group that consumed it
    }
    for (int s = 0; s < C::AB_STAGES; ++s) {
      // one arrival per warp of the dequant group that wrote A and per gather warp (PAIR, even
      // CTA: and one from the odd CTA when its A and x of the stage are written)
      mbar_init(bar(C::ab_full(s)), C::ROWS / 32 + C::GATHER_WARPS + (PAIR && leader ? 1 : 0));
      mbar_init(bar(C::ab_empty(s)), 1);
    }
    for (int q = 0; q < kUnitQ; ++q) {
      mbar_init(bar(C::uq_full(q)), 1);
      mbar_init(bar(C::uq_empty(q)), C::UQ_RELEASES);
    }
    for (int slot = 0; slot < 2; ++slot) {
      mbar_init(bar(C::tmem_full(slot)), 1);
      // one arrival per epilogue warp (PAIR: of both CTAs)
      mbar_init(bar(C::tmem_empty(slot)), PAIR ? 2 * C::EPI_WARPS : C::EPI_WARPS);
    }
    mbar_init(bar(C::unwind()), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == C::TMA_WARP && lane == 0) prefetch_tensormap(&tmap_wq);
  if (warp == C::GATHER_WARP0 && lane == 0) prefetch_tensormap(&tmap_x);
  if (warp == C::MMA_WARP) {
    if constexpr (PAIR) {
      tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_slot), kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  // PAIR: neither CTA touches the other's barriers before both have initialized them
  if constexpr (PAIR) cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  grid_dependents_launch();  // the split-K finalize may be scheduled; it waits for this grid

  const int H = p.H, F = p.F;
  static_assert(FMT::W == C::W, "the code stages hold this format's windows");
  // transpose=False on the wide variant: A (the dequantized weights) is MN-major, each k-row of a
  // 128-row tile two 64-wide atoms (8 KB apart) of 8 k-rows each (1 KB apart)
  constexpr bool kAmn = FMT::KIND == kAffineNn;
  constexpr uint32_t kAmnAtomPitch = 8192u;
  constexpr int GS = FMT::GS;
  static_assert(FMT::KIND != kAffine || GS == 32 || GS == 64 || GS == 128, "group sizes");
  const int num_kb = H / BK;
  // scale groups per weight row (transpose=False: per k-row, along the N = F output columns)
  const int G = (FMT::KIND == kAffineNn ? F : H) / GS;

  // Unit queue: the scheduler (TMA thread) pushes decoded units; every consumer warp pops
  // each entry in order and releases it once its lanes hold a copy.
  auto pop = [&](uint32_t qi, UnitEntry& U) -> bool {
    const uint32_t slot = qi % kUnitQ;
    if (!mbar_wait<PAIR>(bar(C::uq_full(slot)), (qi / kUnitQ) & 1u, abort_flag, status)) return false;
    U.expert = uq[slot].expert;
    U.start = uq[slot].start;
    U.rows = uq[slot].rows;
    U.f0 = uq[slot].f0;
    U.kb0 = uq[slot].kb0;
    U.kb1 = uq[slot].kb1;
    U.ks = uq[slot].ks;
    U.valid = uq[slot].valid;
    return true;
  };
  // one release of entry qi (PAIR: the odd CTA's releases go to the even CTA's scheduler; the
  // entry was read into registers before, and the slot is rewritten kUnitQ entries later)
  auto release_one = [&](uint32_t qi) {
    if (PAIR && !leader)
      mbar_arrive_remote(peer_bar(C::uq_empty(qi % kUnitQ)));
    else
      mbar_arrive(bar(C::uq_empty(qi % kUnitQ)));
  };
  auto release_warp = [&](uint32_t qi) {  // all 32 lanes of the warp call this
    __syncwarp();
    if (lane == 0) release_one(qi);
  };

  if (warp == C::TMA_WARP) {
    // ---------------------------------------------------------------- scheduler + TMA (codes)
    // Units are taken from the call-wide counter one at a time, largest first (the plan
    // orders chunks by size), so CTAs that finish early take more.  (An L2 prefetch of the
    // code tiles several k-blocks ahead was measured: no gain with three stages, a loss with
    // thirteen, so there is none.)
    if (lane == 0) {
      // The kernel may start while the route step that wrote the plan is still running
      // (programmatic dependent launch).  Only this thread reads the plan directly; every
      // other read of routing output (perm) follows a pop from the unit queue, so it comes
      // after this wait.  (PAIR: the odd CTA's scheduler warp only pops the units, in the
      // even CTA's order, and loads its own rows' codes.)
      grid_dependency_wait();
      const int ksplit = p.header->ksplit;
      const int n_fpairs = (F + UM - 1) / UM;
      const int n_units = p.header->n_chunks * n_fpairs * ksplit;
      // the first unit of a CTA (PAIR: of a pair) is its own index (the counter starts at the
      // number of CTAs, or pairs), which saves the counter's round trip on the way to the first MMA
      const int first_unit = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
      uint32_t itn = 0, qi = 0;
      bool ok = true;
      for (;;) {
        const uint32_t slot = qi % kUnitQ;
        UnitEntry U;
        if (PAIR && !leader) {
          if (!pop(qi, U)) {
            ok = false;
            break;
          }
          release_one(qi);
        } else {
          if (!mbar_wait<PAIR>(bar(C::uq_empty(slot)), ((qi / kUnitQ) & 1u) ^ 1u, abort_flag, status)) {
            ok = false;
            break;
          }
          const int u = qi == 0 ? first_unit : atomicAdd(&p.header->next_unit, 1);
          U.valid = u < n_units ? 1 : 0;
          if (U.valid) {
            U = decode_unit(p.chunks, u, n_fpairs, ksplit, num_kb);
          } else {
            U.expert = U.start = U.rows = U.f0 = U.kb0 = U.kb1 = 0;
            U.ks = -1;
          }
          uq[slot].expert = U.expert;
          uq[slot].start = U.start;
          uq[slot].rows = U.rows;
          uq[slot].f0 = U.f0;
          uq[slot].kb0 = U.kb0;
          uq[slot].kb1 = U.kb1;
          uq[slot].ks = U.ks;
          uq[slot].valid = U.valid;
          mbar_arrive(bar(C::uq_full(slot)));  // release: the entry is visible to the waiters
          if constexpr (PAIR) {
            // the same entry into the odd CTA's queue, then its full barrier (release at cluster
            // scope orders the remote stores before the arrival)
            const uint32_t e0 = mapa_shared(smem_u32(const_cast<UnitEntry*>(&uq[slot])), crank ^ 1u);
            const int vals[8] = {U.expert, U.start, U.rows, U.f0, U.kb0, U.kb1, U.ks, U.valid};
#pragma unroll
            for (int j = 0; j < 8; ++j) st_cluster_u32(e0 + 4u * (uint32_t)j, (uint32_t)vals[j]);
            mbar_arrive_cluster(peer_bar(C::uq_full(slot)));
          }
        }
        ++qi;
        if (!U.valid) break;
        const int urows = F - U.f0 < UM ? F - U.f0 : UM;  // the unit's weight rows (a multiple of 16)
        const int crows = min(C::ROWS, urows - rbase);    // this CTA's (none: past F)
        if constexpr (FMT::KIND == kAffine) {
          // The unit's scales and biases (its rows are contiguous, rows x H/GS bf16 each) are
          // pulled into L2 now, so the dequant threads' loads a step ahead hit L2 rather
          // than HBM when they reach this unit.  (The other formats' scales are fetched on
          // demand: their scale arrays are only 4-byte aligned, and bulk prefetches want 16.)
          if (crows > 0) {
            const int64_t off = ((int64_t)U.expert * F + U.f0 + rbase) * G;
            prefetch_l2_bulk(p.scales + off, (uint32_t)(crows * G * 2));
            prefetch_l2_bulk(p.biases + off, (uint32_t)(crows * G * 2));
          }
        }
        // codes of k-block kb: rows row0.. of the [E*F, row bytes] code matrix at byte
        // code_window_x(kb); transpose=False: k-rows U.expert*H + 64 kb.. of the [E*K, N/2]
        // code matrix at byte U.f0 / 2
        const int row0 = U.expert * F + U.f0 + rbase;
        for (int kb = U.kb0; kb < U.kb1; ++kb) {
          const uint32_t s = itn % NIB_STAGES, ph = (itn / NIB_STAGES) & 1u;
          if (!mbar_wait(bar(C::nib_empty(s)), ph ^ 1u, abort_flag, status)) {
            ok = false;
            break;
          }
          if (p.test_stall && itn == 0) {  // failure-path test: this stage's codes never arrive
            ++itn;
            continue;
          }
          mbar_arrive_expect_tx(bar(C::nib_full(s)), C::NIB_BYTES);
          if constexpr (FMT::KIND == kAffineNn)
            tma_load_2d(sbase + C::OFF_NIB + s * C::NIB_BYTES, &tmap_wq, bar(C::nib_full(s)), U.f0 / 2,
                        U.expert * H + kb * BK);
          else
            tma_load_2d(sbase + C::OFF_NIB + s * C::NIB_BYTES, &tmap_wq, bar(C::nib_full(s)), code_window_x<FMT>(kb),
                        row0);
          ++itn;
        }
        if (!ok) break;
      }
      if (!ok) {  // unwinding: let the copies already issued land before the CTA exits
        const uint32_t first = itn > NIB_STAGES ? itn - NIB_STAGES : 0;
        for (uint32_t j = first; j < itn; ++j)
          mbar_wait_unwind(bar(C::nib_full(j % NIB_STAGES)), (j / NIB_STAGES) & 1u, 100000000ull);
      }
    }
  } else if (warp == C::MMA_WARP) {
    // ---------------------------------------------------------------- MMA issuer
    // (PAIR: the even CTA's thread issues the pair's MMAs once both CTAs' A and x of a stage are
    // written, and its commits release the stage and signal the accumulator in both CTAs; the
    // odd CTA's thread forwards the completion of each of its own stages to the even CTA's
    // barrier of that stage, whose phase then completes with the even CTA's own arrivals.)
    if (lane == 0 && PAIR && !leader) {
      uint32_t it = 0, qi = 0;
      bool ok = true;
      for (;;) {
        UnitEntry U;
        if (!pop(qi, U)) break;
        release_one(qi);
        ++qi;
        if (!U.valid) break;
        for (int kb = U.kb0; kb < U.kb1; ++kb, ++it) {
          const uint32_t s = it % C::AB_STAGES, ph = (it / C::AB_STAGES) & 1u;
          if (!mbar_wait(bar(C::ab_full(s)), ph, abort_flag, status)) {
            ok = false;
            break;
          }
          mbar_arrive_remote(peer_bar(C::ab_full(s)));
        }
        if (!ok) break;
      }
      // the even CTA's stage-release commits of the last stages have landed here
      const uint32_t first = it > C::AB_STAGES ? it - C::AB_STAGES : 0;
      for (uint32_t j = first; j < it; ++j)
        mbar_wait_unwind(bar(C::ab_empty(j % C::AB_STAGES)), (j / C::AB_STAGES) & 1u, 100000000ull);
    } else if (lane == 0) {
      uint32_t it = 0, lu = 0, qi = 0;
      bool ok = true;
      for (;; ++lu) {
        UnitEntry U;
        if (!pop(qi, U)) break;
        release_one(qi);  // the only lane of this role
        ++qi;
        if (!U.valid) break;
        const int N = (U.rows + 15) & ~15;
        // PAIR: M = 256 (both CTAs' weight rows) x the chunk's tokens in N tiles of up to 256
        const int N0 = N < UM ? N : UM, N1 = N - N0;
        // SWAP: M = 128 token rows x N = 256 weight rows, the weights (B) MN-major for transpose=False
        const uint32_t idesc = C::SWAP ? umma_idesc_bf16(BM, UM) | (kAmn ? kIdescTransposeB : 0u)
                                       : umma_idesc_bf16(BM, N) | (kAmn ? kIdescTransposeA : 0u);
        const uint32_t slot = lu % C::SLOTS, use = lu / C::SLOTS;
        if (!mbar_wait(bar(C::tmem_empty(slot)), (use & 1u) ^ 1u, abort_flag, status)) break;
        tc_fence_after();
        for (int kb = U.kb0; kb < U.kb1; ++kb) {
          const uint32_t s = it % C::AB_STAGES, ph = (it / C::AB_STAGES) & 1u;
          if (!mbar_wait(bar(C::ab_full(s)), ph, abort_flag, status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t bdesc = umma_desc_sw128(sbase + C::OFF_B + s * C::B_BYTES);
          if constexpr (PAIR) {
            // N tile t: accumulator columns 256 t.. (column = token), x rows 128 t.. of each CTA's
            // stage (its half of the tile's tokens)
            const uint64_t adesc = umma_desc_kmajor_interleave(sbase + C::OFF_A + s * C::A_BYTES);
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              const int Nt = t == 0 ? N0 : N1;
              if (Nt == 0) break;
              const uint32_t idt = umma_idesc_bf16(2 * BM, Nt);
              const uint64_t bdt = bdesc + (uint64_t)((t * BM * BK * 2) >> 4);
#pragma unroll
              for (int k = 0; k < BK / 16; ++k)
                tc_mma_bf16_pair(tmem_base + (uint32_t)(t * UM), adesc + (256u >> 4) * k, bdt + 2u * k, idt,
                                 (kb > U.kb0 || k > 0) ? 1u : 0u);
            }
            tc_commit_pair_mc(bar(C::ab_empty(s)), 0x3);
          } else if constexpr (C::SWAP) {
            // A = the x tile (128-byte-swizzled K-major), B = the 256 weight rows of the stage
            const uint32_t w_addr = sbase + C::OFF_A + s * C::A_BYTES;
            const uint64_t wdesc =
                kAmn ? umma_desc_sw128_mn(w_addr, kAmnAtomPitch, 1024u) : umma_desc_kmajor_interleave(w_addr);
            const uint32_t wstep = kAmn ? 2048u >> 4 : 256u >> 4;
            const uint32_t d_tmem = tmem_base + slot * (uint32_t)C::ACC_COLS;
#pragma unroll
            for (int k = 0; k < BK / 16; ++k)
              tc_mma_bf16(d_tmem, bdesc + 2u * k, wdesc + wstep * k, idesc, (kb > U.kb0 || k > 0) ? 1u : 0u);
          } else {
#pragma unroll
            for (int t = 0; t < NT; ++t) {
              const uint32_t d_tmem = tmem_base + (uint32_t)(t * C::ACC_COLS);
              const uint32_t a_addr = sbase + C::OFF_A + s * C::A_BYTES + t * A_TILE_BYTES;
              // K-major (unswizzled): 16 elements = two 16-byte chunks, 256 bytes on; MN-major: two
              // 8-row atoms (2048 bytes)
              const uint64_t adesc =
                  kAmn ? umma_desc_sw128_mn(a_addr, kAmnAtomPitch, 1024u) : umma_desc_kmajor_interleave(a_addr);
              const uint32_t astep = kAmn ? 2048u >> 4 : 256u >> 4;
#pragma unroll
              for (int k = 0; k < BK / 16; ++k)
                tc_mma_bf16(d_tmem, adesc + astep * k, bdesc + 2u * k, idesc, (kb > U.kb0 || k > 0) ? 1u : 0u);
            }
          }
          if constexpr (!PAIR) tc_commit(bar(C::ab_empty(s)));
          ++it;
        }
        if (!ok) break;
        if constexpr (PAIR)
          tc_commit_pair_mc(bar(C::tmem_full(slot)), 0x3);
        else
          tc_commit(bar(C::tmem_full(slot)));
      }
      // every MMA issued above completes before this barrier's phase 0 completes
      if constexpr (PAIR)
        tc_commit_pair(bar(C::unwind()));
      else
        tc_commit(bar(C::unwind()));
      mbar_wait_unwind(bar(C::unwind()), 0, 100000000ull);
      // and the stage-release arrivals of the last stages have landed
      const uint32_t first = it > C::AB_STAGES ? it - C::AB_STAGES : 0;
      for (uint32_t j = first; j < it; ++j)
        mbar_wait_unwind(bar(C::ab_empty(j % C::AB_STAGES)), (j / C::AB_STAGES) & 1u, 100000000ull);
    }
  } else if (warp >= C::GATHER_WARP0) {
    // ---------------------------------------------------------------- x row gather (TMA)
    // The unit's x tile (N rows x 64 columns per k-block) is fetched with tile::gather4, four
    // rows per copy, straight into the 128-byte-swizzled K-major layout the MMA reads.  Copy g
    // (rows 4g .. 4g+3 of the tile) belongs to lane g / 6 of gather warp g % 6, so every warp
    // issues a few copies per stage and none waits for its data: each warp's lane 0 arrives on
    // the stage's full barrier with the bytes its lanes will deliver.  Rows past the chunk's
    // end (up to N) repeat its first row; the MMA columns they feed are never stored.
    const int gw = warp - C::GATHER_WARP0;
    const int g = lane * C::GATHER_WARPS + gw;
    uint32_t it = 0, qi = 0;
    bool ok = true;
    while (ok) {
      UnitEntry U;
      // a warp-uniform decision: lanes whose bounded wait ran out must not leave the others
      // waiting in the warp synchronization below
      if (!__all_sync(0xffffffffu, pop(qi, U))) break;
      release_warp(qi);
      ++qi;
      if (!U.valid) break;
      // PAIR: this CTA's half of each N tile (tile 0: tokens 0 .. N0-1, tile 1: 256 .. N-1; the odd
      // CTA takes the second half of each), tile 1's rows 128 rows into the stage
      const int N = (U.rows + 15) & ~15;
      const int N0 = N < UM ? N : UM;
      const int ops0 = PAIR ? N0 / 8 : N / 4;
      const int nops = PAIR ? ops0 + (N - N0) / 8 : ops0;
      const bool mine = g < nops;
      const bool t1 = PAIR && g >= ops0;
      const int tok0 = !PAIR ? 4 * g
                       : t1 ? UM + (int)crank * ((N - N0) / 2) + 4 * (g - ops0)
                            : (int)crank * (N0 / 2) + 4 * g;
      const uint32_t soff = t1 ? (uint32_t)(BM * BK * 2) + (uint32_t)(g - ops0) * 512u : (uint32_t)g * 512u;
      int rr[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int pos = tok0 + j < U.rows ? tok0 + j : 0;
        rr[j] = mine ? (p.perm ? __ldg(p.perm + U.start + pos) : U.start + pos) : 0;
        if (p.x_div != 1) rr[j] /= p.x_div;  // a token's A rows share one x row
      }
      const int wops = nops > gw ? min(32, (nops - gw + C::GATHER_WARPS - 1) / C::GATHER_WARPS) : 0;
      for (int kb = U.kb0; kb < U.kb1; ++kb, ++it) {
        const uint32_t s = it % C::AB_STAGES, ph = (it / C::AB_STAGES) & 1u;
        const bool okl = mbar_wait(bar(C::ab_empty(s)), ph ^ 1u, abort_flag, status);
        if (!__all_sync(0xffffffffu, okl)) {
          ok = false;
          break;
        }
        if (lane == 0) mbar_arrive_expect_tx(bar(C::ab_full(s)), (uint32_t)wops * 512u);
        __syncwarp();
        if (mine)
          tma_gather4(sbase + C::OFF_B + s * C::B_BYTES + soff, &tmap_x, bar(C::ab_full(s)), kb * BK, rr[0], rr[1],
                      rr[2], rr[3]);
      }
    }
    if (!ok && lane == 0) {  // unwinding: let this warp's copies of the last stages land
      const uint32_t first = it > C::AB_STAGES ? it - C::AB_STAGES : 0;
      for (uint32_t j = first; j < it; ++j)
        mbar_wait_unwind(bar(C::ab_full(j % C::AB_STAGES)), (j / C::AB_STAGES) & 1u, 100000000ull);
    }
  } else if (warp >= C::EPI_WARP0) {
    // ---------------------------------------------------------------- epilogue
    const int ew = warp - C::EPI_WARP0;
    const int quarter = ew & 3;        // TMEM lanes 32 quarter .. 32 quarter + 31 (= warp % 4)
    uint16_t* epi = reinterpret_cast<uint16_t*>(smem + C::OFF_EPI + ew * EPI_WARP_BYTES);
    const uint32_t epi_addr = sbase + C::OFF_EPI + ew * EPI_WARP_BYTES;
    uint32_t lu = 0, qi = 0;
    for (;; ++lu) {
      UnitEntry U;
      // a warp-uniform decision: lanes whose bounded wait ran out must not leave the others
      // waiting in the warp synchronization below
      if (!__all_sync(0xffffffffu, pop(qi, U))) break;
      release_warp(qi);
      ++qi;
      if (!U.valid) break;
      const int N = (U.rows + 15) & ~15;
      // destination rows of the unit's tokens, loaded before the accumulator is ready: lane l
      // holds the rows of tokens l, l + 32, ...; an iteration's 16 tokens share one register
      int prow[C::NMAX / 32];
#pragma unroll
      for (int q = 0; q < C::NMAX / 32; ++q) {
        const int tok = q * 32 + lane;
        prow[q] = tok < U.rows ? (p.y_perm ? __ldg(p.y_perm + U.start + tok) : U.start + tok) : 0;
      }
      const uint32_t slot = lu % C::SLOTS, use = lu / C::SLOTS;
      const bool okl = mbar_wait(bar(C::tmem_full(slot)), use & 1u, abort_flag, status);
      if (!__all_sync(0xffffffffu, okl)) break;
      tc_fence_after();
      if constexpr (C::SWAP) {
        // lane = token 32 quarter + lane of the chunk, columns = the unit's 256 weight rows: each
        // 16-column load is one token's 16 consecutive outputs (32 bytes of y, or 64 of a split-K
        // plane), stored straight from registers
        const int tok = quarter * 32 + lane;
        if (quarter * 32 < U.rows) {  // warp-uniform: the warp's lanes hold tokens of the chunk
          const bool live = tok < U.rows;
          const int64_t yrow = live ? (p.y_perm ? __ldg(p.y_perm + U.start + tok) : U.start + tok) : 0;
          const uint32_t tcol = tmem_base + ((uint32_t)(quarter * 32) << 16) + slot * (uint32_t)C::ACC_COLS;
          float* plane = U.ks >= 0 ? p.acc + (int64_t)U.ks * p.n * F + (int64_t)(U.start + tok) * F : nullptr;
          for (int c0 = 0; c0 < UM && U.f0 + c0 < F; c0 += 16) {
            uint32_t v[16];
            tc_ld_32x32b_x16(tcol + (uint32_t)c0, v);
            tc_wait_ld_regs(v);
            if (!live) continue;
            const int f = U.f0 + c0;  // F is a multiple of 16: the 16 columns are all in range
            if (U.ks >= 0) {
              uint4* dst = reinterpret_cast<uint4*>(plane + f);
#pragma unroll
              for (int q = 0; q < 4; ++q) dst[q] = make_uint4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
            } else {
              uint32_t h[8];
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                const __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(v[2 * q]), __uint_as_float(v[2 * q + 1]));
                h[q] = *reinterpret_cast<const uint32_t*>(&b2);
              }
              uint4* dst = reinterpret_cast<uint4*>(p.y + yrow * F + f);
              dst[0] = make_uint4(h[0], h[1], h[2], h[3]);
              dst[1] = make_uint4(h[4], h[5], h[6], h[7]);
            }
          }
        }
      } else {
      // PAIR: one accumulator of this CTA's 128 weight rows x the unit's tokens (column = token); the
      // two warps of a lane quarter take alternate 16-column blocks
      constexpr int kTiles = PAIR ? 1 : C::TILES_PER_EPI_WARP;
      const int half = ew >> 2;
      for (int tt = 0; tt < kTiles; ++tt) {
        const int tile = PAIR ? 0 : (ew >> 2) * C::TILES_PER_EPI_WARP + tt;  // accumulator (weight-row tile)
        const uint32_t trow = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(tile * C::ACC_COLS);
        const int frow = U.f0 + rbase + tile * BM + quarter * 32;  // weight row of the warp's lane 0
        if (U.ks >= 0) {
          // partial sums of this K slice into its own plane: thread = weight row f, 16 tokens
          // per TMEM load; a warp's stores for one token are 32 consecutive f (128 bytes)
          const int f = frow + lane;
          float* plane = p.acc + (int64_t)U.ks * p.n * F;
          for (int c0 = PAIR ? 16 * half : 0; c0 < N; c0 += PAIR ? 32 : 16) {
            uint32_t v[16];
            tc_ld_32x32b_x16(trow + (uint32_t)c0, v);
            tc_wait_ld_regs(v);
            if (f < F) {
#pragma unroll
              for (int j = 0; j < 16; ++j)
                if (c0 + j < U.rows) plane[(int64_t)(U.start + c0 + j) * F + f] = __uint_as_float(v[j]);
            }
          }
        } else {
          const int q = lane & 3;
          const int fcol = frow + q * 8;
#pragma unroll
          for (int c0 = 0; c0 < C::NMAX; c0 += 16) {
            if (c0 >= N) break;
            if (PAIR && ((c0 >> 4) & 1) != half) continue;
            uint32_t v[16];
            tc_ld_32x32b_x16(trow + (uint32_t)c0, v);
            tc_wait_ld_regs(v);
#pragma unroll
            for (int j = 0; j < 16; ++j)
              epi[j * 32 + lane] = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(v[j])));
            __syncwarp();
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const int jj = (lane >> 2) + 8 * hh;
              const int tok = c0 + jj;
              const int row = __shfl_sync(0xffffffffu, prow[c0 >> 5], (c0 & 16) + jj);
              if (tok < U.rows && fcol < F) {
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
        }
      }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (PAIR && !leader)
          mbar_arrive_remote(peer_bar(C::tmem_empty(slot)));
        else
          mbar_arrive(bar(C::tmem_empty(slot)));
      }
    }
  } else {
    // ---------------------------------------------------------------- dequant
    static_assert(!PAIR || (FMT::KIND == kAffine && FMT::BITS == 4), "pairs: 4-bit affine codes");
    const int t = threadIdx.x;                     // 0 .. DEQ_GROUPS * ROWS - 1
    const int r = t % C::ROWS;                     // weight row within this CTA's rows of the unit
    const uint32_t grp = (uint32_t)(t / C::ROWS);  // handles the steps with it % DEQ_GROUPS == grp
    const int tile = PAIR ? 0 : r >> 7, rr = r & (BM - 1);
    // code tile rows are W bytes; 32-byte rows are TMA-swizzled in 32-byte mode (16-byte chunk c
    // of row r at chunk position c ^ ((r >> 2) & 1)), other widths are not swizzled
    const uint32_t nib_row = sbase + C::OFF_NIB + (uint32_t)(r * C::W);
    const uint32_t nib_c0 = (uint32_t)(((r >> 2) & 1) << 4), nib_c1 = nib_c0 ^ 16u;
    // the row in A stage 0 (shared-memory A is K-major and unswizzled: core matrices of 8 rows x
    // 16 bytes): chunk c of the row is at a_row + 128 c, so the 8 stores take immediate offsets
    const uint32_t a_row0 = sbase + C::OFF_A + (uint32_t)(tile * A_TILE_BYTES + (rr >> 3) * 1024 + (rr & 7) * 16);
    // transpose=False, wide variant (MN-major A, 128-byte swizzled): thread = (k-row kq, 64-column
    // chunk cq) of the k-block; its 64 bf16 go to one 128-byte k-row of an atom, with the swizzle
    // XOR folded in: chunk c of the k-row is at a_row ^ (c << 4)
    const int kq = r >> 2, cq = r & 3;
    const uint32_t a_nn0 = sbase + C::OFF_A +
                           (uint32_t)((cq >> 1) * A_TILE_BYTES + (cq & 1) * (int)kAmnAtomPitch + (kq >> 3) * 1024 +
                                      (kq & 7) * 128 + ((kq & 7) << 4));
    const uint16_t* sc16 = reinterpret_cast<const uint16_t*>(p.scales);
    const uint16_t* bs16 = reinterpret_cast<const uint16_t*>(p.biases);
    // Flat walk over (unit, k-block) steps in queue order; this group processes every
    // DEQ_GROUPS-th step.  Scales and biases come one step ahead: when the row's group count
    // H/GS is a multiple of 8, as one 16-byte load each covering eight groups of the thread's
    // row (reloaded when the step leaves the block of eight); else 2-byte loads per step (two
    // each for 32-wide groups).
    const bool sb_vec = (G & 7) == 0;
    uint32_t qi = 0;
    bool ok = true;
    auto next_unit = [&](UnitEntry& U) {
      if (!__all_sync(0xffffffffu, pop(qi, U))) {  // warp-uniform, see the gather role
        ok = false;
        U.valid = 0;
      }
      release_warp(qi);
      ++qi;
    };
    // carry kb past the unit's end into the following units
    auto normalize = [&](UnitEntry& U, int& kb) {
      while (U.valid && kb >= U.kb1) {
        const int over = kb - U.kb1;
        next_unit(U);
        kb = U.kb0 + over;
      }
    };
    // scale / bias block of the thread's row in unit U: eight bf16 (sb_vec) or one (low half
    // of .x); zero for rows past F (their outputs are dropped)
    uint4 sblk = make_uint4(0, 0, 0, 0), bblk = make_uint4(0, 0, 0, 0);
    // The scale group of k-block kb's codes: kb for 64-wide groups, kb / 2 for 128-wide ones;
    // for 32-wide groups the block's first 32 codes are group 2 kb and the other 32 group 2 kb + 1.
    auto grp_of = [](int kb) -> int { return GS == 64 ? kb : GS == 128 ? (kb >> 1) : (kb << 1); };
    // Floating-point formats keep the k-block's scale bytes in sblk.x (two E8M0 bytes, or four
    // E4M3 bytes for nvfp4 with the expert's float32 scale in sblk.y).
    auto load_sb = [&](const UnitEntry& U, int kb) {
      if constexpr (kAmn) {
        // the (k-row, chunk) thread's group(s): one scale and bias, or two for 32-wide groups
        const int n = U.f0 + 64 * cq;
        if (!U.valid || n >= F) {
          sblk = bblk = make_uint4(0, 0, 0, 0);
          return;
        }
        const int64_t at = ((int64_t)U.expert * H + (int64_t)kb * BK + kq) * G + n / GS;
        sblk.x = __ldg(sc16 + at);
        bblk.x = __ldg(bs16 + at);
        if (GS == 32) {
          const bool hi = n + 32 < F;
          sblk.y = hi ? __ldg(sc16 + at + 1) : 0u;
          bblk.y = hi ? __ldg(bs16 + at + 1) : 0u;
        }
        return;
      }
      if (!U.valid || U.f0 + rbase + r >= F) {
        sblk = bblk = make_uint4(0, 0, 0, 0);
        return;
      }
      const int64_t row = (int64_t)(U.expert * F + U.f0 + rbase) + r;  // E * F fits in int
      if constexpr (FMT::KIND != kAffine) {
        const uint8_t* sc8 = reinterpret_cast<const uint8_t*>(p.scales);
        if constexpr (FMT::KIND == kNvfp4) {
          sblk.x = __ldg(reinterpret_cast<const uint32_t*>(sc8 + row * (H / 16) + 4 * kb));
          sblk.y = __float_as_uint(__ldg(p.tscale + U.expert));
        } else {
          sblk.x = __ldg(reinterpret_cast<const uint16_t*>(sc8 + row * (H / 32) + 2 * kb));
        }
        return;
      }
      const int g = grp_of(kb);
      if (sb_vec) {
        sblk = __ldg(reinterpret_cast<const uint4*>(sc16 + row * G) + (g >> 3));
        bblk = __ldg(reinterpret_cast<const uint4*>(bs16 + row * G) + (g >> 3));
      } else {
        sblk.x = __ldg(sc16 + row * G + g);
        bblk.x = __ldg(bs16 + row * G + g);
        if (GS == 32) {
          sblk.y = __ldg(sc16 + row * G + g + 1);
          bblk.y = __ldg(bs16 + row * G + g + 1);
        }
      }
    };
    // (v, v) as bf16x2 for the block's element of group g (second: the block's second group,
    // g + 1, of a 32-wide k-block)
    auto pick = [&](const uint4& blk, int g, bool second) -> uint32_t {
      if (!sb_vec) return splat16(second ? blk.y : blk.x);
      const int j = g & 7;
      const uint32_t w = (j & 4) ? ((j & 2) ? blk.w : blk.z) : ((j & 2) ? blk.y : blk.x);
      return __byte_perm(w, 0, (j & 1) ? 0x3232 : 0x1010);
    };
    UnitEntry U;
    next_unit(U);
    int kb = U.kb0 + (int)grp;
    normalize(U, kb);
    load_sb(U, kb);
    // stage indices and phase parities of the current step (global step index grp, grp+2, ...)
    uint32_t sn = grp, phn = 0, sa = grp, pha = 0;
    while (ok && U.valid) {
      const int g = grp_of(kb);
      const uint32_t s2 = pick(sblk, g, false), b2 = pick(bblk, g, false);
      // transpose=False: this thread's group(s)
      const uint32_t nn_s = sblk.x, nn_b = bblk.x, nn_s2 = sblk.y, nn_b2 = bblk.y;
      // floating-point formats: the float32 scale of each 16 weights of the k-block
      float sc4[4] = {0.f, 0.f, 0.f, 0.f};
      if constexpr (FMT::KIND == kNvfp4) {
        const float tsc = __uint_as_float(sblk.y);
#pragma unroll
        for (int j = 0; j < 4; ++j) sc4[j] = e4m3_to_f32((sblk.x >> (8 * j)) & 0xFFu) * tsc;
      } else if constexpr (FMT::KIND != kAffine) {
        sc4[0] = sc4[1] = e8m0_to_f32(sblk.x & 0xFFu);
        sc4[2] = sc4[3] = e8m0_to_f32((sblk.x >> 8) & 0xFFu);
      }
      // 32-wide groups: the row's second 32 codes (n1 below) have their own scale and bias
      const uint32_t s2b = GS == 32 ? pick(sblk, g + 1, true) : s2;
      const uint32_t b2b = GS == 32 ? pick(bblk, g + 1, true) : b2;
      // the next step of this group: same unit, or carried into the following ones
      int kbn = kb + C::DEQ_GROUPS;
      UnitEntry Un;
      const bool cross = kbn >= U.kb1;
      if (cross) {
        Un = U;
        normalize(Un, kbn);
        load_sb(Un, kbn);
      } else if (FMT::KIND != kAffine || !sb_vec || (grp_of(kbn) >> 3) != (g >> 3)) {
        load_sb(U, kbn);
      }
      if (!__all_sync(0xffffffffu, mbar_wait(bar(C::nib_full(sn)), phn, abort_flag, status))) break;
      const uint32_t nib_tile = nib_row + sn * C::NIB_BYTES;
      // The code stage is released only after the proxy fence below: the next TMA into it
      // is an async-proxy write, which is not ordered after these generic-proxy reads by the
      // mbarrier alone.
      uint4 o[8];
      if constexpr (kAmn) {
        // k-row kq, columns 64 cq .. 64 cq + 63: 32 bytes of the k-row in the 128-byte-swizzled
        // code tile (16-byte chunk c of k-row k at chunk c ^ (k % 8)), 8 words of 8 codes in
        // column order, dequantized like a transpose=True row and stored as they are computed
        const uint32_t rowa = nib_tile - (uint32_t)(r * C::W) + (uint32_t)(kq * 128);
        const uint32_t x7 = (uint32_t)(kq & 7);
        uint4 n0, n1;
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(n0.x), "=r"(n0.y), "=r"(n0.z), "=r"(n0.w)
                     : "r"(rowa + ((((uint32_t)(2 * cq)) ^ x7) << 4))
                     : "memory");
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(n1.x), "=r"(n1.y), "=r"(n1.z), "=r"(n1.w)
                     : "r"(rowa + ((((uint32_t)(2 * cq + 1)) ^ x7) << 4))
                     : "memory");
        const uint32_t cw[8] = {n0.x, n0.y, n0.z, n0.w, n1.x, n1.y, n1.z, n1.w};
        const uint32_t sa2 = splat16(nn_s), ba2 = splat16(nn_b);
        const uint32_t sb2 = GS == 32 ? splat16(nn_s2) : sa2, bb2 = GS == 32 ? splat16(nn_b2) : ba2;
        if (!__all_sync(0xffffffffu, mbar_wait(bar(C::ab_empty(sa)), pha ^ 1u, abort_flag, status))) break;
        const uint32_t a_row = a_nn0 + sa * C::A_BYTES;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 v = deq8(cw[c], c < 4 ? sa2 : sb2, c < 4 ? ba2 : bb2);
          asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a_row ^ (uint32_t)(c << 4)), "r"(v.x),
                       "r"(v.y), "r"(v.z), "r"(v.w)
                       : "memory");
        }
      } else if constexpr (FMT::KIND == kAffine && FMT::BITS == 4) {
        uint4 n0, n1;
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(n0.x), "=r"(n0.y), "=r"(n0.z), "=r"(n0.w)
                     : "r"(nib_tile + nib_c0)
                     : "memory");
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(n1.x), "=r"(n1.y), "=r"(n1.z), "=r"(n1.w)
                     : "r"(nib_tile + nib_c1)
                     : "memory");
        const uint32_t cw[8] = {n0.x, n0.y, n0.z, n0.w, n1.x, n1.y, n1.z, n1.w};
        // wait for the A stage first and store each 8-weight piece as soon as it is computed, so
        // the row's 64 bf16 are never all live in registers at once
        if (!__all_sync(0xffffffffu, mbar_wait(bar(C::ab_empty(sa)), pha ^ 1u, abort_flag, status))) break;
        const uint32_t a_row = a_row0 + sa * C::A_BYTES;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 v = deq8(cw[c], c < 4 ? s2 : s2b, c < 4 ? b2 : b2b);
          asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a_row + (uint32_t)(c * 128)), "r"(v.x),
                       "r"(v.y), "r"(v.z), "r"(v.w)
                       : "memory");
        }
      } else {
        // the row's code window: W / 4 words (for 32-byte windows through the swizzle)
        uint32_t cw[C::W / 4];
#pragma unroll
        for (int c = 0; c < C::W / 16; ++c) {
          const uint32_t at = C::W == 32 ? (c == 0 ? nib_c0 : nib_c1) : (uint32_t)(16 * c);
          asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(cw[4 * c]), "=r"(cw[4 * c + 1]), "=r"(cw[4 * c + 2]), "=r"(cw[4 * c + 3])
                       : "r"(nib_tile + at)
                       : "memory");
        }
        if constexpr (FMT::KIND == kAffine) {
          if constexpr (C::W == 48 && (FMT::BITS == 3 || FMT::BITS == 5)) {
            if (code_window_off<FMT>(kb) == 0)
              dequant_affine<FMT::BITS, 0>(cw, s2, b2, o);
            else
              dequant_affine<FMT::BITS, 8>(cw, s2, b2, o);
          } else {
            dequant_affine<FMT::BITS, 0>(cw, s2, b2, o);
          }
        } else if constexpr (FMT::KIND == kMxfp8) {
          dequant_e4m3(cw, sc4, o);
        } else {
          dequant_e2m1(cw, sc4, o);
        }
      }
      // (the 4-bit affine and transpose=False rows are already stored)
      constexpr bool kStored = (FMT::KIND == kAffine && FMT::BITS == 4) || FMT::KIND == kAffineNn;
      if (!kStored && !__all_sync(0xffffffffu, mbar_wait(bar(C::ab_empty(sa)), pha ^ 1u, abort_flag, status))) break;
      if (!kStored) {
        const uint32_t a_row = a_row0 + sa * C::A_BYTES;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a_row + (uint32_t)(c * 128)), "r"(o[c].x),
                       "r"(o[c].y), "r"(o[c].z), "r"(o[c].w)
                       : "memory");
      }
      // Every thread orders its A writes and code reads before async-proxy use; the warp then
      // synchronizes and one lane arrives for it (an arrival per thread costs the barrier
      // unit 32 updates per warp).
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar(C::ab_full(sa)));
        mbar_arrive(bar(C::nib_empty(sn)));
      }
      if (cross) U = Un;
      kb = kbn;
      sn += C::DEQ_GROUPS;
      if (sn >= (uint32_t)NIB_STAGES) {
        sn -= NIB_STAGES;
        phn ^= 1u;
      }
      sa += C::DEQ_GROUPS;
      if (sa >= (uint32_t)C::AB_STAGES) {
        sa -= C::AB_STAGES;
        pha ^= 1u;
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) {
    // neither CTA leaves (or frees the pair's tensor memory) while the other may still read its
    // shared memory through the MMAs or arrive on its barriers
    cluster_sync();
    tc_fence_after();
    if (warp == C::MMA_WARP) tmem_dealloc_pair(tmem_base, kTmemCols);
  } else {
    tc_fence_after();
    if (warp == C::MMA_WARP) tmem_dealloc(tmem_base, kTmemCols);
  }
}

// Split-K epilogue: y[row(p), f] = bf16(sum over slices ks of acc[ks, p, f]), added in slice
// order, for every valid sorted position p (rows with an invalid index keep the zeros the
// route step wrote).  One thread per 8 consecutive outputs.
__global__ void __launch_bounds__(256) splitk_finalize(const GemmArgs p) {
  grid_dependency_wait();  // launched to overlap the GEMM's tail; the planes are complete here
  const int ksplit = p.header->ksplit;  // chosen by the plan step; 1: the GEMM wrote y itself
  if (ksplit <= 1) return;
  int64_t n_valid = __ldg(p.offsets + p.E);
  n_valid = n_valid < 0 ? 0 : (n_valid > p.n ? p.n : n_valid);
  const int oct = p.F / 8;
  const int64_t n_oct = n_valid * oct;
  const int64_t plane = p.n * (int64_t)p.F;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_oct; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t pos = i / oct;
    const int f = (int)(i - pos * oct) * 8;
    const float4* a = reinterpret_cast<const float4*>(p.acc + pos * p.F + f);
    float4 s0 = __ldg(a), s1 = __ldg(a + 1);
    for (int ks = 1; ks < ksplit; ++ks) {
      const float4* b = reinterpret_cast<const float4*>(p.acc + ks * plane + pos * p.F + f);
      const float4 t0 = __ldg(b), t1 = __ldg(b + 1);
      s0.x += t0.x; s0.y += t0.y; s0.z += t0.z; s0.w += t0.w;
      s1.x += t1.x; s1.y += t1.y; s1.z += t1.z; s1.w += t1.w;
    }
    const int row = p.y_perm ? __ldg(p.y_perm + pos) : (int)pos;
    uint4 o;
    o.x = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(s0.x)) |
          ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(s0.y)) << 16);
    o.y = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(s0.z)) |
          ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(s0.w)) << 16);
    o.z = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(s1.x)) |
          ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(s1.y)) << 16);
    o.w = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(s1.z)) |
          ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(s1.w)) << 16);
    *reinterpret_cast<uint4*>(p.y + (int64_t)row * p.F + f) = o;
  }
}

struct DeviceInfo {
  int sms = 0;
  int pairs = 0;  // CTA pairs of the pair instances resident at once (0: those are not used)
  bool configured = false;
};

DeviceInfo g_dev[64];

template <class C, class FMT>
cudaError_t set_smem() {
  return cudaFuncSetAttribute(gemm_tc_kernel<C, FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_DYN);
}

cudaError_t configure_all() {
  cudaError_t e = cudaSuccess;
  auto need = [&](cudaError_t r) {
    if (e == cudaSuccess) e = r;
  };
  need(set_smem<CfgWide, FmtAffine<32, 4>>());
  need(set_smem<CfgWide, FmtAffine<64, 4>>());
  need(set_smem<CfgWide, FmtAffine<128, 4>>());
  need(set_smem<CfgWide16, FmtAffine<64, 2>>());
  need(set_smem<CfgWide, FmtMx<false>>());
  need(set_smem<CfgWide, FmtNv>());
  need(set_smem<CfgWide48, FmtAffine<64, 3>>());
  need(set_smem<CfgWide48, FmtAffine<64, 5>>());
  need(set_smem<CfgWide48, FmtAffine<64, 6>>());
  need(set_smem<CfgWide64, FmtAffine<64, 8>>());
  need(set_smem<CfgWide64, FmtMx<true>>());
  need(set_smem<CfgWide, FmtNn<32>>());
  need(set_smem<CfgWide, FmtNn<64>>());
  need(set_smem<CfgWide, FmtNn<128>>());
  need(set_smem<CfgSwapMid, FmtAffine<32, 4>>());
  need(set_smem<CfgSwapMid, FmtAffine<64, 4>>());
  need(set_smem<CfgSwapMid, FmtAffine<128, 4>>());
  need(set_smem<CfgSwap, FmtAffine<32, 4>>());
  need(set_smem<CfgSwap, FmtAffine<64, 4>>());
  need(set_smem<CfgSwap, FmtAffine<128, 4>>());
  need(set_smem<CfgSwap16, FmtAffine<64, 2>>());
  need(set_smem<CfgSwap48, FmtAffine<64, 3>>());
  need(set_smem<CfgSwap48, FmtAffine<64, 5>>());
  need(set_smem<CfgSwap48, FmtAffine<64, 6>>());
  need(set_smem<CfgSwap64, FmtAffine<64, 8>>());
  need(set_smem<CfgSwap, FmtMx<false>>());
  need(set_smem<CfgSwap, FmtNv>());
  need(set_smem<CfgSwap64, FmtMx<true>>());
  need(set_smem<CfgSwap, FmtNn<32>>());
  need(set_smem<CfgSwap, FmtNn<64>>());
  need(set_smem<CfgSwap, FmtNn<128>>());
  need(set_smem<CfgPair, FmtAffine<32, 4>>());
  need(set_smem<CfgPair, FmtAffine<64, 4>>());
  need(set_smem<CfgPair, FmtAffine<128, 4>>());
  return e;
}

// Launch attribute of the pair instances: clusters of two CTAs.
cudaLaunchAttribute pair_cluster_attr() {
  cudaLaunchAttribute a;
  a.id = cudaLaunchAttributeClusterDimension;
  a.val.clusterDim.x = 2;
  a.val.clusterDim.y = 1;
  a.val.clusterDim.z = 1;
  return a;
}

// How many CTA pairs of the pair instances the device holds at once (one CTA per SM); 0 if the
// occupancy query fails, and the single-CTA wide instances are used instead.
int query_pairs(int sms) {
  cudaLaunchAttribute ca[1] = {pair_cluster_attr()};
  cudaLaunchConfig_t qc = {};
  qc.gridDim = dim3((unsigned)(sms - sms % 2));
  qc.blockDim = dim3(kThreads);
  qc.dynamicSmemBytes = (size_t)CfgPair::SMEM_DYN;
  qc.attrs = ca;
  qc.numAttrs = 1;
  int nc = 0;
  if (cudaOccupancyMaxActiveClusters(&nc, gemm_tc_kernel<CfgPair, FmtAffine<64, 4>>, &qc) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return nc < sms / 2 ? nc : sms / 2;
}

// The device's info, configuring the kernel instances on first use.
cudaError_t device_info(DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  DeviceInfo& di = g_dev[dev];
  if (!di.configured) {
    e = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if ((e = configure_all()) != cudaSuccess) return e;
    di.pairs = query_pairs(di.sms);
    di.configured = true;
  }
  *out = &di;
  return cudaSuccess;
}

// Calls whose plan has chunks of up to 512 rows (4-bit affine) run on CTA pairs.
bool uses_pairs(const DeviceInfo& di, int kind, int bits, int chunk_rows) {
  return di.pairs > 0 && kind == kAffine && bits == 4 && chunk_rows == kChunkRowsPair;
}

using GemmKernel = decltype(&gemm_tc_kernel<CfgWide, FmtAffine<64, 4>>);

// The kernel instance and its shared-memory size for a format and a variant (nullptr: no
// instance for the format).
using FmtA4g32 = FmtAffine<32, 4>;
using FmtA4g64 = FmtAffine<64, 4>;
using FmtA4g128 = FmtAffine<128, 4>;
using FmtA2 = FmtAffine<64, 2>;
using FmtA3 = FmtAffine<64, 3>;
using FmtA5 = FmtAffine<64, 5>;
using FmtA6 = FmtAffine<64, 6>;
using FmtA8 = FmtAffine<64, 8>;
using FmtMxfp4 = FmtMx<false>;
using FmtMxfp8 = FmtMx<true>;
using FmtNn32 = FmtNn<32>;
using FmtNn64 = FmtNn<64>;
using FmtNn128 = FmtNn<128>;

GemmKernel pick_instance(const GemmArgs& a, bool narrow, bool mid, bool pair, int* smem) {
#define GQMM_PICK(CFG, FMT)      \
  do {                           \
    *smem = CFG::SMEM_DYN;       \
    return gemm_tc_kernel<CFG, FMT>; \
  } while (0)
  if (a.kind == kAffine && a.bits == 4) {
    if (pair) {
      if (a.group_size == 32) GQMM_PICK(CfgPair, FmtA4g32);
      if (a.group_size == 128) GQMM_PICK(CfgPair, FmtA4g128);
      GQMM_PICK(CfgPair, FmtA4g64);
    }
    if (narrow) {
      if (a.group_size == 32) GQMM_PICK(CfgSwap, FmtA4g32);
      if (a.group_size == 128) GQMM_PICK(CfgSwap, FmtA4g128);
      GQMM_PICK(CfgSwap, FmtA4g64);
    }
    if (mid) {
      if (a.group_size == 32) GQMM_PICK(CfgSwapMid, FmtA4g32);
      if (a.group_size == 128) GQMM_PICK(CfgSwapMid, FmtA4g128);
      GQMM_PICK(CfgSwapMid, FmtA4g64);
    }
    if (a.group_size == 32) GQMM_PICK(CfgWide, FmtA4g32);
    if (a.group_size == 128) GQMM_PICK(CfgWide, FmtA4g128);
    GQMM_PICK(CfgWide, FmtA4g64);
  }
  if (a.kind == kAffineNn) {
    if (narrow) {
      if (a.group_size == 32) GQMM_PICK(CfgSwap, FmtNn32);
      if (a.group_size == 128) GQMM_PICK(CfgSwap, FmtNn128);
      GQMM_PICK(CfgSwap, FmtNn64);
    }
    if (a.group_size == 32) GQMM_PICK(CfgWide, FmtNn32);
    if (a.group_size == 128) GQMM_PICK(CfgWide, FmtNn128);
    GQMM_PICK(CfgWide, FmtNn64);
  }
  if (a.kind == kAffine && a.bits == 2) {
    if (narrow) GQMM_PICK(CfgSwap16, FmtA2);
    GQMM_PICK(CfgWide16, FmtA2);
  }
  if (a.kind == kMxfp4) {
    if (narrow) GQMM_PICK(CfgSwap, FmtMxfp4);
    GQMM_PICK(CfgWide, FmtMxfp4);
  }
  if (a.kind == kNvfp4) {
    if (narrow) GQMM_PICK(CfgSwap, FmtNv);
    GQMM_PICK(CfgWide, FmtNv);
  }
  if (a.kind == kMxfp8) {
    if (narrow) GQMM_PICK(CfgSwap64, FmtMxfp8);
    GQMM_PICK(CfgWide64, FmtMxfp8);
  }
  if (a.kind == kAffine && a.bits == 8) {
    if (narrow) GQMM_PICK(CfgSwap64, FmtA8);
    GQMM_PICK(CfgWide64, FmtA8);
  }
  if (a.kind == kAffine && a.bits == 3) {
    if (narrow) GQMM_PICK(CfgSwap48, FmtA3);
    GQMM_PICK(CfgWide48, FmtA3);
  }
  if (a.kind == kAffine && a.bits == 5) {
    if (narrow) GQMM_PICK(CfgSwap48, FmtA5);
    GQMM_PICK(CfgWide48, FmtA5);
  }
  if (a.kind == kAffine && a.bits == 6) {
    if (narrow) GQMM_PICK(CfgSwap48, FmtA6);
    GQMM_PICK(CfgWide48, FmtA6);
  }
#undef GQMM_PICK
  return nullptr;
}

}  // namespace

cudaError_t gemm_tc_workers(int kind, int bits, int chunk_rows, int* workers) {
  DeviceInfo* di = nullptr;
  cudaError_t e = device_info(&di);
  if (e != cudaSuccess) return e;
  *workers = uses_pairs(*di, kind, bits, chunk_rows) ? di->pairs : di->sms;
  return cudaSuccess;
}

cudaError_t gemm_tc_chunk_rows(int kind, int bits, int chunk_rows, int64_t n, int E, int* out) {
  DeviceInfo* di = nullptr;
  cudaError_t e = device_info(&di);
  if (e != cudaSuccess) return e;
  const int64_t busy = n < E ? n : E;  // experts that can have rows
  const bool big = busy > 0 && n > busy * kChunkRowsWide;
  *out = di->pairs > 0 && kind == kAffine && bits == 4 && chunk_rows == kChunkRowsWide && big ? kChunkRowsPair
                                                                                            : chunk_rows;
  return cudaSuccess;
}

cudaError_t device_sm_count(int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  DeviceInfo& di = g_dev[dev];
  if (di.sms == 0) {
    e = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
  }
  *sms = di.sms;
  return cudaSuccess;
}

cudaError_t launch_gemm_tc(const GemmArgs& a, cudaStream_t s, int* launched) {
  *launched = 0;
  DeviceInfo* dip = nullptr;
  cudaError_t e = device_info(&dip);
  if (e != cudaSuccess) return e;
  const DeviceInfo& di = *dip;

  static decltype(&cuTensorMapEncodeTiled) encode = nullptr;
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
    encode = reinterpret_cast<decltype(&cuTensorMapEncodeTiled)>(fn);
  }
  const bool narrow = a.chunk_rows <= kChunkRowsNarrow;
  const bool mid = !narrow && a.chunk_rows <= kChunkRowsMid;
  const bool pair = uses_pairs(di, a.kind, a.bits, a.chunk_rows);
  int smem = 0;
  GemmKernel kern = pick_instance(a, narrow, mid, pair, &smem);
  if (kern == nullptr) return cudaErrorInvalidValue;
  // Packed codes as an [E*F, row bytes] byte matrix; one box = the unit's 256 rows x one k-block's
  // code window (W bytes: formats.cuh), 32-byte swizzled when W is 32 so the dequant threads read
  // it without bank conflicts.  Every window starts on a 16-byte boundary.
  // transpose=False: codes as an [E*K, N/2] byte matrix; one box = 64 k-rows (one k-block) x the
  // unit's 256 columns (128 bytes), 128-byte swizzled; columns past N read as zero.
  const bool nn = a.kind == kAffineNn;
  const int code_bits = a.kind == kMxfp8 ? 8 : a.kind == kAffine ? a.bits : 4;
  const int W = code_bits == 3 || code_bits == 5 ? 48 : 8 * code_bits;
  const int64_t row_bytes = nn ? (int64_t)a.F / 2 : (int64_t)a.H * code_bits / 8;
  const int64_t code_rows = (int64_t)a.E * (nn ? a.H : a.F);
  CUtensorMap map_wq;
  const cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)code_rows};
  const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  const cuuint32_t box[2] = {nn ? (cuuint32_t)(UM / 2) : (cuuint32_t)W,
                             nn ? (cuuint32_t)BK : (cuuint32_t)(pair ? CfgPair::ROWS : UM)};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapSwizzle swz = nn ? CU_TENSOR_MAP_SWIZZLE_128B
                                : W == 32 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_NONE;
  CUresult cr = encode(&map_wq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(a.wq), dims, strides, box,
                       estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return cudaErrorInvalidValue;
  // x as a [n, H] bf16 matrix; one box = 64 columns (one k-block, 128 bytes) of one row, for
  // tile::gather4 into the 128-byte-swizzled B tile.
  CUtensorMap map_x;
  const cuuint64_t xdims[2] = {(cuuint64_t)a.H, (cuuint64_t)(a.n / a.x_div)};
  const cuuint64_t xstrides[1] = {(cuuint64_t)a.H * 2};
  const cuuint32_t xbox[2] = {BK, 1};
  cr = encode(&map_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<__nv_bfloat16*>(a.x), xdims, xstrides, xbox,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return cudaErrorInvalidValue;
  // Both kernels are launched with programmatic stream serialization: the GEMM's prologue
  // (barriers, TMEM, tensor maps) overlaps the route step, and the finalize's launch the
  // GEMM's tail.  Each waits (griddepcontrol.wait) before reading its predecessor's output.
  // The pair instances are launched as clusters of two CTAs, one pair per unit worker.
  cudaLaunchAttribute pdl[2];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  pdl[1] = pair_cluster_attr();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(pair ? 2 * di.pairs : di.sms));
  cfg.blockDim = dim3(kThreads);
  cfg.stream = s;
  cfg.attrs = pdl;
  cfg.numAttrs = pair ? 2 : 1;
  cfg.dynamicSmemBytes = (size_t)smem;
  e = cudaLaunchKernelEx(&cfg, kern, map_wq, map_x, a);
  if (e != cudaSuccess) return e;
  *launched = 1;
  if (a.ks_cap > 1) {
    const int64_t n_oct = a.n * (a.F / 8);
    const int64_t blocks = (n_oct + 255) / 256;
    cfg.gridDim = dim3((unsigned)(blocks < 4 * di.sms ? blocks : 4 * di.sms));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, splitk_finalize, a);
    if (e != cudaSuccess) return e;
    *launched = 2;
  }
  return cudaSuccess;
}

}  // namespace gqmm
