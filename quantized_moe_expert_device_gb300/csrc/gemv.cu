// Weight-streaming gather matmul for calls with at most 2 rows per chunk (decode): every weight
// byte is read from HBM once per chunk and applied to the chunk's M <= 2 rows on the CUDA cores.
//
// Small-M decode is bandwidth-bound: with M rows a weight is used M times, so forming 128-row
// tensor-core tiles would only add a pipeline between roles (mlxcel #725 "amortizing small-M
// quantized GEMM", sections The gap and What's needed: load each weight tile once and apply it
// across the small batch).  Design:
//   - work item = (chunk, batch of RB weight rows of the chunk's expert).  The RB rows are
//     contiguous in wq, scales and biases, so one item is three 1-D bulk copies (plus the
//     chunk's rows of x when the chunk changes) into a stage of a 3- or 4-deep shared-memory
//     ring (4 where it fits two blocks per SM); a dense call copies its x rows once into a buffer
//     of their own, so its stages hold weights only and its ring is 5-6 deep;
//   - one producer warp issues the copies up to a ring's depth ahead; eight consumer warps
//     compute;
//   - consumer thread = (row group, k slice of 32 elements), R = 4 rows per item; a row group
//     is the next power of two (>= 32) of the row's slice count, the threads past the last slice
//     adding zeros (H a multiple of 128, at most 8192).  The x slice
//     stays in registers as bf16 pairs for as long as the block works on the chunk;
//   - per row the thread reads 16 bytes of codes and the group's scale s and bias b from shared
//     memory, accumulates acc_t = sum_k x_tk (128 + q_k) with the codes made into exact bf16
//     values by the magic-number trick and multiplied in a mixed bf16 x bf16 + fp32 FMA, then
//     adds s acc_t + (b - 128 s) X_t with X_t = sum_k x_tk over the slice (the slice lies in one
//     quantization group), all accumulated in fp32;
//   - the partial sums are reduced across the row's threads (warp reduce-scatter, then shared
//     memory, double-buffered so one consumer barrier per item suffices) and written as bf16.
// Items are split into one contiguous range per block, two blocks per SM.
#include "gqmm_internal.cuh"

namespace gqmm {
namespace {

constexpr int kStreamConsumers = 256;                  // 8 consumer warps
constexpr int kStreamThreads = kStreamConsumers + 32;  // + the producer warp
constexpr int kStreamKS = 32;                          // k elements per consumer thread
constexpr int kStreamR = 4;                            // weight rows per consumer thread and item
constexpr int kStreamStages = 4;                       // ring depth when it fits the budget, else 3
constexpr int kStreamMaxStages = 6;                    // dense calls: as many weight-only stages as fit
constexpr int kStreamSmemBudget = 110 * 1024;          // ring bytes per block: two blocks per SM
constexpr int kStreamMaxXElems = 8192;                 // M * H bound: the x rows of a stage <= 16 KB
constexpr uint32_t kStreamBarId = 1;                   // named barrier of the consumer warps

// Rows per item: kStreamConsumers / (H / KS) row groups of kStreamR rows.
// Consumer threads per weight row: one per 32-element k slice, rounded up to a power of two of at
// least a warp (threads past the row's last slice add zeros), so a row group is whole warps.
__host__ __device__ constexpr int stream_lanes(int H) {
  return H / kStreamKS <= 32 ? 32 : H / kStreamKS <= 64 ? 64 : H / kStreamKS <= 128 ? 128 : 256;
}
__host__ __device__ constexpr int stream_rows_per_item(int H) {
  return kStreamConsumers / stream_lanes(H) * kStreamR;
}
// Bytes of one ring stage: codes, scales, biases of the item's rows, then M rows of x.
__host__ __device__ constexpr int stream_stage_bytes(int H, int M) {
  return stream_rows_per_item(H) * (H / 2 + 2 * (H / 64) * 2) + M * H * 2;
}

__host__ __device__ constexpr int stream_stages(int H, int M) {
  return kStreamStages * stream_stage_bytes(H, M) <= kStreamSmemBudget ? kStreamStages : kStreamStages - 1;
}
// A dense call has one chunk, so its x rows are copied once, with the first item, into a buffer of
// their own after the ring; its stages hold weights only, and more of them fit.
__host__ __device__ constexpr int stream_weight_bytes(int H) { return stream_stage_bytes(H, 0); }
__host__ __device__ constexpr int stream_stages_dense(int H, int M) {
  return (kStreamSmemBudget - M * H * 2) / stream_weight_bytes(H) < kStreamMaxStages
             ? (kStreamSmemBudget - M * H * 2) / stream_weight_bytes(H)
             : kStreamMaxStages;
}

// Routed calls of at most this many rows (decode: M tokens x A experts) are planned inside the
// kernel: every block sorts the call's routing entries into chunks itself, so no route kernel runs
// in front of it.
constexpr int kFusedPlanRows = 64;
static_assert(kFusedPlanRows == kFusedPlanMaxRows, "one bound for the host and the kernel");

// The chunk list of a routed call of n <= 64 rows, computed by one warp: the rows of each expert
// in flat-row order, in chunks of at most two rows (the first and second, third and fourth, ...
// occurrences of the expert), numbered in the flat order of their first rows.  Each lane holds
// entries lane and 32 + lane; a match within each half of the entries and, when there is a second
// half, one unrolled pass of shuffles across the halves give an entry's occurrence rank, its
// expert's total and its next occurrence.  plan[c] = (expert, first row, second row
// (= first row for a one-row chunk), rows).  Rows whose index is >= E are in no chunk; block 0
// writes them as zeros and records GQMM_STATUS_BAD_INDEX.  Returns the number of chunks (lane 0).
__device__ __forceinline__ int fused_plan(const GemmArgs& p, int4* plan, uint32_t* status) {
  const int lane = threadIdx.x & 31;
  const int n = (int)p.n;
  uint32_t key[2];
  int rank[2], tot[2], next[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int i = 32 * r + lane;
    key[r] = i < n ? __ldg(p.idx + i) : 0xFFFFFFFFu;
  }
  // Within each half: the lanes holding the same key (padding keys 0xFFFFFFFF match only one
  // another, never a valid index), their count, the ones below this lane and the next one above.
  const uint32_t lt = (1u << lane) - 1u, le = lt | (1u << lane);
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const uint32_t m = __match_any_sync(0xffffffffu, key[r]);
    tot[r] = __popc(m);
    rank[r] = __popc(m & lt);
    const uint32_t above = m & ~le;
    next[r] = above ? 32 * r + __ffs(above) - 1 : -1;
  }
  if (n > 32) {  // uniform: entries 32.. exist; count each half's key in the other half
    int c0 = 0, c1 = 0, first1 = -1;
#pragma unroll
    for (int jl = 0; jl < 32; ++jl) {
      const uint32_t k1 = __shfl_sync(0xffffffffu, key[1], jl);  // entry 32 + jl
      const uint32_t k0 = __shfl_sync(0xffffffffu, key[0], jl);  // entry jl
      if (k1 == key[0]) {
        ++c0;
        if (first1 < 0) first1 = 32 + jl;
      }
      if (k0 == key[1]) ++c1;
    }
    tot[0] += c0;
    if (next[0] < 0) next[0] = first1;
    tot[1] += c1;
    rank[1] += c1;  // every entry of the first half comes before the second half
  }
  bool lead[2], bad[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int i = 32 * r + lane;
    bad[r] = i < n && key[r] >= (uint32_t)p.E;
    lead[r] = i < n && !bad[r] && (rank[r] & 1) == 0;
  }
  const uint32_t b0 = __ballot_sync(0xffffffffu, lead[0]), b1 = __ballot_sync(0xffffffffu, lead[1]);
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    if (lead[r]) {
      const int i = 32 * r + lane;
      const int id = r == 0 ? __popc(b0 & lt) : __popc(b0) + __popc(b1 & lt);
      const int rows = tot[r] - rank[r] >= 2 ? 2 : 1;
      plan[id] = make_int4((int)key[r], i, rows == 2 ? next[r] : i, rows);
    }
  }
  if (blockIdx.x == 0) {
    bool any = false;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      if (bad[r]) {
        uint4* row = reinterpret_cast<uint4*>(p.y + (int64_t)(32 * r + lane) * p.F);
        for (int c = 0; c < p.F / 8; ++c) row[c] = make_uint4(0u, 0u, 0u, 0u);
        any = true;
      }
    }
    if (__any_sync(0xffffffffu, any) && lane == 0) atomicOr(status, GQMM_STATUS_BAD_INDEX);
  }
  return __popc(b0) + __popc(b1);
}

// Per-stage item description written by the producer before it arms the stage's barrier.
struct StageMeta {
  int rows;     // rows of the chunk (1..M)
  int fb;       // first weight row of the item within the expert
  int newx;     // 1: the stage holds the chunk's rows of x (first item of a chunk in this block)
  int trow[2];  // output rows of y
};

// Sum of v[0..V) over the 32 lanes, scattered: on return lane l holds in v[0 .. max(V/32,1))
// the totals of the indices scatter_index(l, j); lanes that share an index hold equal totals.
template <int V>
__device__ __forceinline__ void warp_reduce_scatter(float (&v)[V]) {
  const int lane = threadIdx.x & 31;
  int cnt = V;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    if (cnt > 1) {
      const int half = cnt / 2;
      const bool up = (lane & off) != 0;
#pragma unroll
      for (int j = 0; j < V / 2; ++j) {
        if (j < half) {
          const float mine = up ? v[half + j] : v[j];
          const float give = up ? v[j] : v[half + j];
          v[j] = mine + __shfl_xor_sync(0xffffffffu, give, off);
        }
      }
      cnt = half;
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
    }
  }
}

// index held in v[j] after warp_reduce_scatter<V> by lane l
template <int V>
__device__ __forceinline__ int scatter_index(int lane, int j) {
  int idx = 0, span = V;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    if (span > 1) {
      span /= 2;
      if (lane & off) idx += span;
    }
  }
  return idx + j;
}

// The rows' bf16 pairs (x[8w + j], x[8w + j + 4]) for w < 4, j < 4, from 32 bf16 at `src`
// (shared memory), and their fp32 sum.
__device__ __forceinline__ float load_x_pairs(uint32_t (&xp)[16], const __nv_bfloat16* src) {
  float sum = 0.f;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const uint4 u = reinterpret_cast<const uint4*>(src)[w];
    xp[4 * w + 0] = __byte_perm(u.x, u.z, 0x5410);
    xp[4 * w + 1] = __byte_perm(u.x, u.z, 0x7632);
    xp[4 * w + 2] = __byte_perm(u.y, u.w, 0x5410);
    xp[4 * w + 3] = __byte_perm(u.y, u.w, 0x7632);
    const uint32_t h[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) sum += __uint_as_float(h[q] << 16) + __uint_as_float(h[q] & 0xFFFF0000u);
  }
  return sum;
}

// acc += x.lo * w.lo + x.hi * w.hi, each product of two bf16 exact and added in fp32 (a mixed
// precision FMA, one rounding per add).
__device__ __forceinline__ float fma2_bf16(uint32_t x2, uint32_t w2, float acc) {
  asm("{\n\t.reg .b16 xl, xh, wl, wh;\n\t"
      "mov.b32 {xl, xh}, %1;\n\t"
      "mov.b32 {wl, wh}, %2;\n\t"
      "fma.rn.f32.bf16 %0, xl, wl, %0;\n\t"
      "fma.rn.f32.bf16 %0, xh, wh, %0;\n\t}\n"
      : "+f"(acc)
      : "r"(x2), "r"(w2));
  return acc;
}

// Partial sums of one item for MU of the M x rows: part[r * M + t] for the thread's rows r.
template <int M, int MU>
__device__ __forceinline__ void item_partials(float (&part)[kStreamR * M], const uint8_t* codes,
                                              const uint16_t* sc, const uint16_t* bs, const uint32_t (&xp)[M][16],
                                              const float (&X)[M], int row0, int lr, int H, int valid_rows) {
  const int G = H / 64;
#pragma unroll
  for (int r = 0; r < kStreamR; ++r) {
    const int row = row0 + r;
    const uint4 u = *reinterpret_cast<const uint4*>(codes + (size_t)row * (H / 2) + lr * (kStreamKS / 2));
    const uint32_t s16 = sc[row * G + lr / 2], b16 = bs[row * G + lr / 2];
    const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
    float acc[M];
#pragma unroll
    for (int t = 0; t < M; ++t) acc[t] = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      // word w holds elements 8 w .. 8 w + 7 (element j in bits 4j .. 4j + 3); t_j holds the
      // bf16 values 128 + q of elements (8 w + j, 8 w + j + 4)
      constexpr uint32_t kMask = 0x000F000Fu, kMagic = 0x43004300u;
      const uint32_t c = wv[w];
      const uint32_t tj[4] = {(c & kMask) | kMagic, ((c >> 4) & kMask) | kMagic, ((c >> 8) & kMask) | kMagic,
                              ((c >> 12) & kMask) | kMagic};
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int t = 0; t < MU; ++t) acc[t] = fma2_bf16(xp[t][4 * w + j], tj[j], acc[t]);
    }
    const float s = __uint_as_float(s16 << 16), b = __uint_as_float(b16 << 16);
    const float cb = fmaf(-128.f, s, b);  // b - 128 s (exact in fp32 for bf16 s and b)
    const bool ok = row < valid_rows;
#pragma unroll
    for (int t = 0; t < M; ++t) part[r * M + t] = (ok && t < MU) ? fmaf(s, acc[t], cb * X[t]) : 0.f;
  }
}

template <int M>
__global__ void __launch_bounds__(kStreamThreads, 2) gemv_fma_kernel(const GemmArgs p) {
  constexpr int V = kStreamR * M;  // partial sums per consumer thread and item
  constexpr int VL = V >= 32 ? V / 32 : 1;
  constexpr int NW = kStreamConsumers / 32;
  extern __shared__ __align__(128) uint8_t stream_smem[];
  __shared__ __align__(8) uint64_t full_bar[kStreamMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kStreamMaxStages];
  __shared__ StageMeta meta[kStreamMaxStages];
  __shared__ float red[2][NW][V];
  __shared__ int abort_flag;
  __shared__ int4 plan[kFusedPlanRows];  // the in-kernel chunk list of a fused-plan call
  __shared__ int plan_n;

  const int H = p.H, F = p.F, G = H / 64;
  const int RB = stream_rows_per_item(H);
  const bool dense = p.dense_plan != 0;
  const int stage_bytes = dense ? stream_weight_bytes(H) : stream_stage_bytes(H, M);
  const int NS = dense ? stream_stages_dense(H, M) : stream_stages(H, M);
  // where a stage's x rows are: the stage's own tail, or (dense) the buffer after the ring
  auto x_at = [&](int s) -> int { return dense ? NS * stage_bytes : s * stage_bytes + RB * (H / 2 + 4 * G); };
  const int n_batches = (F + RB - 1) / RB;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t* status = &p.header->status;

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  // The next call's kernel may be scheduled as this one's blocks retire: it waits for this grid
  // to finish (griddepcontrol.wait) before it reads or writes anything of the call.
  grid_dependents_launch();

  // The kernel may start while the previous kernel on the stream is still running
  // (programmatic dependent launch), and that kernel may be writing this call's x, weights or
  // y.  A dense call knows its items without the route step, so before the wait its producer
  // only asks L2 to pull in the block's share of the weights (a prefetch is a hint served by
  // L2, the point of coherence, so it cannot hand back stale bytes); every copy into shared
  // memory and every store to y comes after the wait.
  if (p.dense_plan && warp == NW && lane == 0) {
    const int per0 = (n_batches + (int)gridDim.x - 1) / (int)gridDim.x;
    const int f0 = min(F, (int)blockIdx.x * per0 * RB), f1 = min(F, f0 + per0 * RB);
    // the rows beyond the ring's first fill: those are copied (from HBM) as soon as the wait returns,
    // and a prefetch of them would only sit ahead of those copies in the block's copy engine
    const int fs = min(f1, f0 + NS * RB);
    if (f1 > fs) {
      prefetch_l2_bulk(p.wq + (int64_t)fs * (H / 2), (uint32_t)(f1 - fs) * (H / 2));
      prefetch_l2_bulk(p.scales + (int64_t)fs * G, (uint32_t)(f1 - fs) * G * 2);
      prefetch_l2_bulk(p.biases + (int64_t)fs * G, (uint32_t)(f1 - fs) * G * 2);
    }
  }
  grid_dependency_wait();
  if (p.fused_plan) {
    if (warp == 0) {
      const int nc = fused_plan(p, plan, status);
      if (lane == 0) plan_n = nc;
    }
    __syncthreads();
  }
  const int n_chunks = p.dense_plan ? 1 : p.fused_plan ? plan_n : p.header->n_chunks;
  const int n_items = n_chunks * n_batches;
  const int per = (n_items + (int)gridDim.x - 1) / (int)gridDim.x;
  const int it0 = min(n_items, (int)blockIdx.x * per);
  const int it1 = min(n_items, it0 + per);

  if (warp == NW) {
    // ---------------- producer ----------------
    if (lane == 0) {
      int prev_c = -1;
      int4 rec = make_int4(0, 0, 0, 0);
      int trow[2] = {0, 0};  // rows of y
      int xrow[2] = {0, 0};  // rows of x
      bool ok = true;
      int issued = 0;
      for (int j = it0; j < it1 && ok; ++j) {
        const int k = j - it0, s = k % NS, u = k / NS;
        if (u > 0 && !mbar_wait(smem_u32(&empty_bar[s]), (u - 1) & 1, &abort_flag, status)) {
          ok = false;
          break;
        }
        const int c = j / n_batches, b = j - c * n_batches;
        const bool newx = c != prev_c;
        if (newx) {
          if (p.fused_plan) {
            const int4 pc = plan[c];  // (expert, first row, second row, rows)
            rec = make_int4(pc.x, 0, pc.w, 0);
            trow[0] = pc.y;
            trow[1] = M > 1 && pc.w > 1 ? pc.z : 0;
#pragma unroll
            for (int t = 0; t < 2; ++t) xrow[t] = trow[t] / p.x_div;
          } else {
            rec = p.dense_plan ? make_int4(0, 0, (int)p.n, 0) : __ldg(reinterpret_cast<const int4*>(p.chunks) + c);
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              const bool live = t < M && t < rec.z;
              trow[t] = live ? (p.y_perm ? __ldg(p.y_perm + rec.y + t) : rec.y + t) : 0;
              xrow[t] = live ? (p.perm ? __ldg(p.perm + rec.y + t) : rec.y + t) / p.x_div : 0;
            }
          }
          prev_c = c;
        }
        const int fb = b * RB;
        const int nr = min(RB, F - fb);
        StageMeta& m = meta[s];
        m.rows = rec.z;
        m.fb = fb;
        m.newx = newx ? 1 : 0;
        m.trow[0] = trow[0];
        m.trow[1] = trow[1];
        const uint32_t code_bytes = (uint32_t)nr * (H / 2), sb_bytes = (uint32_t)nr * G * 2;
        const int xr = min(rec.z, M);
        const uint32_t x_bytes = newx ? (uint32_t)xr * H * 2 : 0u;
        const uint32_t base = smem_u32(stream_smem) + (uint32_t)(s * stage_bytes);
        const uint32_t bar = smem_u32(&full_bar[s]);
        mbar_arrive_expect_tx(bar, code_bytes + 2 * sb_bytes + x_bytes);
        const int64_t row = (int64_t)rec.x * F + fb;
        bulk_load(base, p.wq + row * (H / 2), code_bytes, bar);
        bulk_load(base + RB * (H / 2), p.scales + row * G, sb_bytes, bar);
        bulk_load(base + RB * (H / 2) + RB * G * 2, p.biases + row * G, sb_bytes, bar);
        if (newx)
          for (int t = 0; t < xr; ++t)
            bulk_load(smem_u32(stream_smem) + (uint32_t)(x_at(s) + t * H * 2), p.x + (int64_t)xrow[t] * H, H * 2, bar);
        ++issued;
      }
      if (!ok || abort_flag) {
        // unwinding: wait (bounded) for the copies still in flight into this block's memory
        for (int k = max(0, issued - NS); k < issued; ++k)
          mbar_wait_unwind(smem_u32(&full_bar[k % NS]), (k / NS) & 1, 100000000ull);
      }
    }
    return;
  }

  // ---------------- consumers ----------------
  const int L = stream_lanes(H);  // threads per row
  const int rg = tid / L, lr = tid - rg * L;
  const bool active = lr < H / kStreamKS;  // the thread has a k slice of the row
  const int W = L / 32;         // warps per row group
  const int RG = kStreamConsumers / L;
  uint32_t xp[M][16];
  float X[M];
#pragma unroll
  for (int t = 0; t < M; ++t) {
    X[t] = 0.f;
#pragma unroll
    for (int q = 0; q < 16; ++q) xp[t][q] = 0u;
  }
  int rows = 0;
  for (int j = it0; j < it1; ++j) {
    const int k = j - it0, s = k % NS;
    bool failed = !mbar_wait(smem_u32(&full_bar[s]), (k / NS) & 1, &abort_flag, status);
    const uint8_t* st = stream_smem + (size_t)s * stage_bytes;
    const StageMeta m = meta[s];
    if (!failed && m.newx) {
      rows = m.rows;
#pragma unroll
      for (int t = 0; t < M; ++t) {
        if (t < rows && active) {
          X[t] = load_x_pairs(xp[t], reinterpret_cast<const __nv_bfloat16*>(stream_smem + x_at(s) + t * H * 2) +
                                         lr * kStreamKS);
        } else {
          X[t] = 0.f;
#pragma unroll
          for (int q = 0; q < 16; ++q) xp[t][q] = 0u;
        }
      }
    }
    float part[V];
    const int valid_rows = min(RB, F - m.fb);
    const uint16_t* sc = reinterpret_cast<const uint16_t*>(st + RB * (H / 2));
    const uint16_t* bs = sc + RB * G;
    if (!active) {
#pragma unroll
      for (int q = 0; q < V; ++q) part[q] = 0.f;
    } else if (M == 1 || rows == 1) {
      item_partials<M, 1>(part, st, sc, bs, xp, X, rg * kStreamR, lr, H, valid_rows);
    } else {
      item_partials<M, M>(part, st, sc, bs, xp, X, rg * kStreamR, lr, H, valid_rows);
    }
    warp_reduce_scatter<V>(part);
    const bool writer = V >= 32 || (lane & (32 / V - 1)) == 0;
    float (*rb)[V] = red[k & 1];
    if (writer) {
#pragma unroll
      for (int q = 0; q < VL; ++q) rb[warp][scatter_index<V>(lane, q)] = part[q];
    }
    // all consumers are done with stage s and have written their sums
    failed = named_barrier_or(kStreamBarId, kStreamConsumers, failed);
    if (failed) break;
    if (tid == 0) mbar_arrive(smem_u32(&empty_bar[s]));
    if (tid < RG * V) {
      const int g = tid / V, idx = tid - g * V;  // row group; (row r, x row t) = (idx / M, idx % M)
      float sum = 0.f;
      for (int w2 = 0; w2 < W; ++w2) sum += rb[g * W + w2][idx];
      const int r = idx / M, t = idx - r * M;
      const int f = m.fb + g * kStreamR + r;
      if (f < F && t < rows) p.y[(int64_t)(t == 0 ? m.trow[0] : m.trow[1]) * F + f] = __float2bfloat16_rn(sum);
    }
  }
}

}  // namespace

bool gemv_fma_supported(int rows, int H) {
  // H a multiple of 128 keeps every bulk copy a multiple of 16 bytes (an item's scale rows are
  // 4096 H / (32 stream_lanes(H)) bytes)
  return (rows == 1 || rows == 2) && H > 0 && H % 128 == 0 && H / kStreamKS <= kStreamConsumers &&
         rows * H <= kStreamMaxXElems;
}

cudaError_t launch_gemv_fma(const GemmArgs& a, int rows, int sms, cudaStream_t s) {
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  const int smem = a.dense_plan ? stream_stages_dense(a.H, rows) * stream_weight_bytes(a.H) + rows * a.H * 2
                                 : stream_stages(a.H, rows) * stream_stage_bytes(a.H, rows);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * sms));  // two blocks per SM
  cfg.blockDim = dim3(kStreamThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = s;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  // The shared-memory opt-in is set once per device and instance, to the largest size asked so
  // far (a host call per launch would cost more than a decode-sized kernel takes).
  static int smem_set[64][2] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int& set = smem_set[dev][rows == 1 ? 0 : 1];
  if (smem > set) {
    e = rows == 1 ? cudaFuncSetAttribute(gemv_fma_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)
                  : cudaFuncSetAttribute(gemv_fma_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    set = smem;
  }
  return rows == 1 ? cudaLaunchKernelEx(&cfg, gemv_fma_kernel<1>, a) : cudaLaunchKernelEx(&cfg, gemv_fma_kernel<2>, a);
}

// The weight-streaming path: dense calls of 2 to 8 rows run on the MMA kernel (gemv_mma.cu),
// whose cost does not grow with the rows; single-row dense calls and routed chunks of 1 or 2
// rows on the CUDA-core kernel above.
bool gemv_uses_mma(int rows, int H, int E) { return E == 1 && rows >= 2 && gemv_mma_supported(rows, H); }

bool gemv_supported(int rows, int H, int E) {
  return gemv_uses_mma(rows, H, E) || (rows <= 2 && gemv_fma_supported(rows, H));
}

cudaError_t launch_gemv(const GemmArgs& a, int rows, int sms, cudaStream_t s) {
  if (gemv_uses_mma(rows, a.H, a.E)) return launch_gemv_mma(a, rows, sms, s);
  return launch_gemv_fma(a, rows, sms, s);
}

}  // namespace gqmm
