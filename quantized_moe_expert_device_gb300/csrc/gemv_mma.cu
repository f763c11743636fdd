// Weight-streaming gather matmul for dense calls of 3 to 8 rows (decode with a small batch):
// every weight byte is read from HBM once and applied to all rows of x.
//
// Small-M decode is bandwidth-bound (mlxcel #725 "amortizing small-M quantized GEMM", sections
// The gap and What's needed: load each weight tile once and apply it across the small batch).
// On the CUDA cores the arithmetic grows with the rows (one FMA per weight and row), so here the
// products go to a warp-level MMA instead and the cost per weight is the 4-bit decode alone:
//   - a code word (8 nibbles) becomes four bf16 pairs 128 + q by the magic-number trick (one
//     mask-and-or per pair, no scale applied);
//   - the pairs go straight into a bf16 MMA (m16n8k16, fp32 accumulate) as its A fragment,
//     with the rows of x (up to 8) as B, so D = sum_k (128 + q) x per quantization group.  The
//     MMA's k order is a permutation of the group's elements, the same for A and B;
//   - per group, y += s D + (b - 128 s) X with X = sum_k x over the group (fp32 FMAs).
// Work item = (chunk, 16 weight rows).  The item's code rows, scales and biases are contiguous
// in global memory; one producer warp copies them with 1-D bulk copies (one row per lane) into
// a shared-memory ring, code rows padded so that the fragment loads are free of bank conflicts.
// 16 consumer warps split K: warp w takes H/16 elements, keeps its slice of x in registers as
// MMA B fragments, and the 16 partial 16 x 8 tiles are summed in shared memory behind one
// named barrier per item.  Items are split into one contiguous range per block, one block per SM.
#include "gqmm_internal.cuh"

namespace gqmm {
namespace {

constexpr int kMmaWarps = 16;                        // consumer warps (K split 16 ways)
constexpr int kMmaConsumers = kMmaWarps * 32;
constexpr int kMmaThreads = kMmaConsumers + 32;      // + the producer warp
constexpr int kItemRows = 16;                        // weight rows per item (the MMA's M)
constexpr int kMaxTokens = 8;                        // rows of x per chunk (the MMA's N)
constexpr int kCodePad = 32;                         // bytes of padding after each staged code row
constexpr int kXPad = 16;                            // bytes of padding after each staged x row
constexpr int kMaxStages = 8;
constexpr int kDynSmemBudget = 200 * 1024;           // ring + x buffer (static smem holds ~17 KB)
constexpr uint32_t kConsumerBar = 1;                 // named barrier of the consumer warps

__host__ __device__ constexpr int code_stride(int H) { return H / 2 + kCodePad; }
// One ring stage: kItemRows padded code rows, then their scales, then their biases.
__host__ __device__ constexpr int stage_bytes(int H) { return kItemRows * (code_stride(H) + 2 * (H / 64) * 2); }
__host__ __device__ constexpr int xbuf_bytes(int H, int mcap) { return mcap * (2 * H + kXPad); }
__host__ __device__ constexpr int ring_stages(int H, int mcap) {
  return (kDynSmemBudget - xbuf_bytes(H, mcap)) / stage_bytes(H) < kMaxStages
             ? (kDynSmemBudget - xbuf_bytes(H, mcap)) / stage_bytes(H)
             : kMaxStages;
}

// Per-stage item description written by the producer before it arms the stage's barrier.
struct StageMeta {
  int rows;               // rows of x in the chunk (1..8)
  int fb;                 // first weight row of the item within the expert
  int newx;               // 1: first item of a chunk in this block (x buffer refilled)
  int trow[kMaxTokens];   // output rows of y
};

// The four bf16 pairs (128 + q_j, 128 + q_{j+4}) of the code word c (element e in bits 4e..4e+3).
__device__ __forceinline__ void decode_word(uint32_t c, uint32_t (&t)[4]) {
  constexpr uint32_t kMask = 0x000F000Fu, kMagic = 0x43004300u;
  t[0] = (c & kMask) | kMagic;
  t[1] = ((c >> 4) & kMask) | kMagic;
  t[2] = ((c >> 8) & kMask) | kMagic;
  t[3] = ((c >> 12) & kMask) | kMagic;
}

// D += A B for one m16n8k16 bf16 MMA with fp32 accumulators.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// GW consecutive bf16 values (scales or biases of GW groups) from shared memory.
template <int GW>
struct Bf16Run {
  uint32_t v[(GW + 1) / 2];
  __device__ __forceinline__ void load(const uint16_t* p) {
    if constexpr (GW == 1) v[0] = *p;
    else if constexpr (GW == 2) v[0] = *reinterpret_cast<const uint32_t*>(p);
    else if constexpr (GW == 4) {
      const uint2 u = *reinterpret_cast<const uint2*>(p);
      v[0] = u.x;
      v[1] = u.y;
    } else {
      const uint4 u = *reinterpret_cast<const uint4*>(p);
      v[0] = u.x;
      v[1] = u.y;
      v[2] = u.z;
      v[3] = u.w;
    }
  }
  __device__ __forceinline__ float get(int i) const {
    return (i & 1) ? __uint_as_float(v[i >> 1] & 0xFFFF0000u) : __uint_as_float(v[i >> 1] << 16);
  }
};

// GW = quantization groups per consumer warp = H / 1024.
template <int GW>
__global__ void __launch_bounds__(kMmaThreads, 1) gemv_mma_kernel(const GemmArgs p) {
  extern __shared__ __align__(128) uint8_t dsmem[];
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ __align__(8) uint64_t xfull_bar, xempty_bar;
  __shared__ StageMeta meta[kMaxStages];
  __shared__ __align__(16) float red[2][kMmaWarps][kItemRows][kMaxTokens];
  __shared__ int abort_flag;

  const int H = p.H, F = p.F, G = H / 64;
  const int mcap = p.chunk_rows;
  const int CS = code_stride(H);
  const int SB = stage_bytes(H);
  const int NS = ring_stages(H, mcap);
  const int XS = 2 * H + kXPad;  // staged x row stride
  uint8_t* ring = dsmem;
  uint8_t* xbuf = dsmem + (size_t)NS * SB;
  const int n_batches = (F + kItemRows - 1) / kItemRows;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t* status = &p.header->status;

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    mbar_init(smem_u32(&xfull_bar), 1);
    mbar_init(smem_u32(&xempty_bar), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();

  // The next call's kernel may be scheduled as this one's blocks retire: it waits for this grid
  // to finish (griddepcontrol.wait) before it reads or writes anything of the call.
  grid_dependents_launch();

  // The kernel may start while the previous kernel on the stream is still running
  // (programmatic dependent launch), and that kernel may be writing this call's x, weights or
  // y.  The dense plan is known without the route step, so before the wait the producer only
  // asks L2 to pull in the block's share of the weights (a hint served by L2, the point of
  // coherence: it cannot hand back stale bytes); every copy into shared memory and every
  // store to y comes after the wait.
  if (p.dense_plan && warp == kMmaWarps && lane == 0) {
    const int per0 = (n_batches + (int)gridDim.x - 1) / (int)gridDim.x;
    const int f0 = min(F, (int)blockIdx.x * per0 * kItemRows), f1 = min(F, f0 + per0 * kItemRows);
    // the rows beyond the ring's first fill (those are copied as soon as the wait returns, and a
    // prefetch of them would only sit ahead of those copies in the block's copy engine)
    const int fs = min(f1, f0 + NS * kItemRows);
    if (f1 > fs) {
      prefetch_l2_bulk(p.wq + (int64_t)fs * (H / 2), (uint32_t)(f1 - fs) * (H / 2));
      prefetch_l2_bulk(p.scales + (int64_t)fs * G, (uint32_t)(f1 - fs) * G * 2);
      prefetch_l2_bulk(p.biases + (int64_t)fs * G, (uint32_t)(f1 - fs) * G * 2);
    }
  }
  grid_dependency_wait();
  const int n_chunks = p.dense_plan ? 1 : p.header->n_chunks;
  const int n_items = n_chunks * n_batches;
  const int per = (n_items + (int)gridDim.x - 1) / (int)gridDim.x;
  const int it0 = min(n_items, (int)blockIdx.x * per);
  const int it1 = min(n_items, it0 + per);

  if (warp == kMmaWarps) {
    // ---------------- producer warp (all lanes run the loop in step) ----------------
    int prev_c = -1, xq = 0, issued = 0, x_issued = 0;
    int4 rec = make_int4(0, 0, 0, 0);
    int trow_lane = 0, xrow_lane = 0;  // lane t < 8: row t of the chunk in y and in x
    bool ok = true;
    for (int j = it0; j < it1; ++j) {
      const int k = j - it0, s = k % NS, u = k / NS;
      if (u > 0) {
        ok = mbar_wait(smem_u32(&empty_bar[s]), (u - 1) & 1, &abort_flag, status);
        if (!__all_sync(0xffffffffu, ok)) break;
      }
      const int c = j / n_batches, b = j - c * n_batches;
      const bool newx = c != prev_c;
      if (newx) {
        rec = p.dense_plan ? make_int4(0, 0, (int)p.n, 0) : __ldg(reinterpret_cast<const int4*>(p.chunks) + c);
        const int xr = min(rec.z, mcap);
        if (xq > 0) {  // the consumers have moved the previous chunk's x into registers
          ok = mbar_wait(smem_u32(&xempty_bar), (xq - 1) & 1, &abort_flag, status);
          if (!__all_sync(0xffffffffu, ok)) break;
        }
        trow_lane = lane < xr ? (p.y_perm ? __ldg(p.y_perm + rec.y + lane) : rec.y + lane) : 0;
        xrow_lane = lane < xr ? (p.perm ? __ldg(p.perm + rec.y + lane) : rec.y + lane) / p.x_div : 0;
        if (lane == 0) mbar_arrive_expect_tx(smem_u32(&xfull_bar), (uint32_t)xr * H * 2);
        __syncwarp();
        if (lane < xr)
          bulk_load(smem_u32(xbuf + lane * XS), p.x + (int64_t)xrow_lane * H, H * 2, smem_u32(&xfull_bar));
        prev_c = c;
        ++xq;
        x_issued = 1;
      }
      const int fb = b * kItemRows;
      const int nr = min(kItemRows, F - fb);
      int trows[kMaxTokens];
#pragma unroll
      for (int t = 0; t < kMaxTokens; ++t) trows[t] = __shfl_sync(0xffffffffu, trow_lane, t);
      const uint32_t bar = smem_u32(&full_bar[s]);
      if (lane == 0) {
        StageMeta& m = meta[s];
        m.rows = rec.z;
        m.fb = fb;
        m.newx = newx ? 1 : 0;
#pragma unroll
        for (int t = 0; t < kMaxTokens; ++t) m.trow[t] = trows[t];
        mbar_arrive_expect_tx(bar, (uint32_t)nr * (H / 2) + 2u * nr * G * 2);
      }
      __syncwarp();
      uint8_t* st = ring + (size_t)s * SB;
      const int64_t row0 = (int64_t)rec.x * F + fb;
      if (lane < nr) bulk_load(smem_u32(st + lane * CS), p.wq + (row0 + lane) * (H / 2), H / 2, bar);
      if (lane == 16) bulk_load(smem_u32(st + kItemRows * CS), p.scales + row0 * G, nr * G * 2, bar);
      if (lane == 17)
        bulk_load(smem_u32(st + kItemRows * CS + kItemRows * G * 2), p.biases + row0 * G, nr * G * 2, bar);
      ++issued;
    }
    if (lane == 0 && (!ok || abort_flag)) {
      // unwinding: wait (bounded) for the copies still in flight into this block's memory
      for (int k = max(0, issued - NS); k < issued; ++k)
        mbar_wait_unwind(smem_u32(&full_bar[k % NS]), (k / NS) & 1, 100000000ull);
      if (x_issued) mbar_wait_unwind(smem_u32(&xfull_bar), (xq - 1) & 1, 100000000ull);
    }
    return;
  }

  // ---------------- consumers ----------------
  const int g = lane >> 2, t4 = lane & 3;  // fragment row group and thread-in-group
  const int grp0 = warp * GW;              // this warp's first quantization group
  uint32_t xb[GW][8];                      // B fragments: x pairs of token g for the warp's groups
  float Xs[GW][2];                         // group sums of x for tokens 2 t4 and 2 t4 + 1
#pragma unroll
  for (int gi = 0; gi < GW; ++gi) {
    Xs[gi][0] = Xs[gi][1] = 0.f;
#pragma unroll
    for (int q = 0; q < 8; ++q) xb[gi][q] = 0u;
  }
  int rows = 0, xq = 0;
  for (int j = it0; j < it1; ++j) {
    const int k = j - it0, s = k % NS;
    bool failed = !mbar_wait(smem_u32(&full_bar[s]), (k / NS) & 1, &abort_flag, status);
    const int fb = meta[s].fb;
    const int newx = meta[s].newx;
    const int my_trow = meta[s].trow[tid & 7];
    if (newx) {
      rows = meta[s].rows;
      failed = failed || !mbar_wait(smem_u32(&xfull_bar), xq & 1, &abort_flag, status);
      ++xq;
      // this thread's 16 elements per group of token g (elements 16 t4 .. 16 t4 + 15)
#pragma unroll
      for (int gi = 0; gi < GW; ++gi) {
        float part = 0.f;
        if (g < rows && !failed) {
          const uint4* src = reinterpret_cast<const uint4*>(xbuf + g * XS + (grp0 + gi) * 128 + t4 * 32);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint4 u = src[h];
            xb[gi][4 * h + 0] = __byte_perm(u.x, u.z, 0x5410);
            xb[gi][4 * h + 1] = __byte_perm(u.x, u.z, 0x7632);
            xb[gi][4 * h + 2] = __byte_perm(u.y, u.w, 0x5410);
            xb[gi][4 * h + 3] = __byte_perm(u.y, u.w, 0x7632);
            const uint32_t hw[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) part += __uint_as_float(hw[q] << 16) + __uint_as_float(hw[q] & 0xFFFF0000u);
          }
        } else {
#pragma unroll
          for (int q = 0; q < 8; ++q) xb[gi][q] = 0u;
        }
        part += __shfl_xor_sync(0xffffffffu, part, 1);
        part += __shfl_xor_sync(0xffffffffu, part, 2);  // group sum for token g, in its 4 lanes
        Xs[gi][0] = __shfl_sync(0xffffffffu, part, 8 * t4);      // token 2 t4
        Xs[gi][1] = __shfl_sync(0xffffffffu, part, 8 * t4 + 4);  // token 2 t4 + 1
      }
    }
    const uint8_t* st = ring + (size_t)s * SB;
    const uint8_t* crow0 = st + g * CS + grp0 * 32 + t4 * 8;  // rows g and g + 8
    const uint8_t* crow1 = crow0 + 8 * CS;
    const uint16_t* sc = reinterpret_cast<const uint16_t*>(st + kItemRows * CS);
    const uint16_t* bs = sc + kItemRows * G;
    Bf16Run<GW> s0, s1, b0, b1;
    s0.load(sc + g * G + grp0);
    s1.load(sc + (g + 8) * G + grp0);
    b0.load(bs + g * G + grp0);
    b1.load(bs + (g + 8) * G + grp0);
    float Y[4] = {0.f, 0.f, 0.f, 0.f};  // (row g | g + 8) x (token 2 t4 | 2 t4 + 1)
#pragma unroll
    for (int gi = 0; gi < GW; ++gi) {
      const uint2 w0 = *reinterpret_cast<const uint2*>(crow0 + gi * 32);
      const uint2 w1 = *reinterpret_cast<const uint2*>(crow1 + gi * 32);
      float D[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t ta[4], tb[4];
        decode_word(h ? w0.y : w0.x, ta);
        decode_word(h ? w1.y : w1.x, tb);
        mma_bf16_16816(D, ta[0], tb[0], ta[1], tb[1], xb[gi][4 * h + 0], xb[gi][4 * h + 1]);
        mma_bf16_16816(D, ta[2], tb[2], ta[3], tb[3], xb[gi][4 * h + 2], xb[gi][4 * h + 3]);
      }
      const float sg0 = s0.get(gi), sg1 = s1.get(gi);
      const float cg0 = fmaf(-128.f, sg0, b0.get(gi)), cg1 = fmaf(-128.f, sg1, b1.get(gi));  // b - 128 s
      Y[0] = fmaf(sg0, D[0], fmaf(cg0, Xs[gi][0], Y[0]));
      Y[1] = fmaf(sg0, D[1], fmaf(cg0, Xs[gi][1], Y[1]));
      Y[2] = fmaf(sg1, D[2], fmaf(cg1, Xs[gi][0], Y[2]));
      Y[3] = fmaf(sg1, D[3], fmaf(cg1, Xs[gi][1], Y[3]));
    }
    float (*rb)[kItemRows][kMaxTokens] = red[k & 1];
    *reinterpret_cast<float2*>(&rb[warp][g][2 * t4]) = make_float2(Y[0], Y[1]);
    *reinterpret_cast<float2*>(&rb[warp][g + 8][2 * t4]) = make_float2(Y[2], Y[3]);
    // all consumers are done with stage s (and, on a chunk's first item, the x buffer)
    failed = named_barrier_or(kConsumerBar, kMmaConsumers, failed);
    if (failed) break;
    if (tid == 0) {
      mbar_arrive(smem_u32(&empty_bar[s]));
      if (newx) mbar_arrive(smem_u32(&xempty_bar));
    }
    if (tid < kItemRows * kMaxTokens) {
      const int r = tid >> 3, col = tid & 7;
      if (col < rows && fb + r < F) {
        float sum = 0.f;
#pragma unroll
        for (int w2 = 0; w2 < kMmaWarps; ++w2) sum += rb[w2][r][col];
        p.y[(int64_t)my_trow * F + fb + r] = __float2bfloat16_rn(sum);
      }
    }
  }
}

}  // namespace

bool gemv_mma_supported(int rows, int H) {
  const int gw = H / 1024;
  return rows >= 1 && rows <= kMaxTokens && H % 1024 == 0 && (gw == 1 || gw == 2 || gw == 4) &&
         ring_stages(H, rows) >= 2;
}

cudaError_t launch_gemv_mma(const GemmArgs& a, int rows, int sms, cudaStream_t s) {
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  const int smem = ring_stages(a.H, rows) * stage_bytes(a.H) + xbuf_bytes(a.H, rows);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)sms);  // one block per SM
  cfg.blockDim = dim3(kMmaThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = s;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  GemmArgs args = a;
  args.chunk_rows = rows;
  // The shared-memory opt-in is set once per device and instance, to the largest size asked so
  // far (a host call per launch would cost more than a decode-sized kernel takes).
  static int smem_set[64][3] = {};
  int dev = 0;
  cudaError_t e0 = cudaGetDevice(&dev);
  if (e0 != cudaSuccess) return e0;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const int inst = a.H / 1024 == 1 ? 0 : a.H / 1024 == 2 ? 1 : 2;
  auto run = [&](auto kern) {
    int& set = smem_set[dev][inst];
    if (smem > set) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return e;
      set = smem;
    }
    return cudaLaunchKernelEx(&cfg, kern, args);
  };
  switch (inst) {
    case 0: return run(gemv_mma_kernel<1>);
    case 1: return run(gemv_mma_kernel<2>);
    default: return run(gemv_mma_kernel<4>);
  }
}

}  // namespace gqmm
