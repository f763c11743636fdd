// gqmm_gather_qmm_noalloc: gqmm_gather_qmm with its scratch in a fixed, statically sized
// device array owned by this library, for callers that cannot allocate device memory.
//
// gqmm_gather_qmm asks its caller for a workspace (routing permutation, expert offsets,
// histograms, the work list and a status word).  Some callers cannot provide one: code that
// runs where device allocation is unavailable or forbidden (a plugin whose host framework
// owns every byte of device memory, a real-time path that may not block in cudaMalloc, which
// can synchronize the whole device), or a caller with no place to keep a buffer between
// calls.  This entry point uses the array below instead and allocates nothing itself.
//
// The array lives in device memory of every GPU on which this library's kernels are loaded,
// from module load until the process exits.  Host code must not use the array's name as a
// device address (on the host it names a host-side placeholder); the device address is
// obtained once per device with cudaGetSymbolAddress and cached.
#include <mutex>

#include "gqmm_internal.cuh"

namespace {

constexpr size_t kScratchBytes = GQMM_NOALLOC_SCRATCH_BYTES;
static_assert(kScratchBytes % 256 == 0, "scratch is a whole number of 256-byte lines");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_dev_ptr[64] = {};  // device address of g_noalloc_scratch, per device ordinal

// Device address of the scratch array on the current device (looked up on first use).
int scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return gqmm::report_error(GQMM_ERR_CUDA, "gqmm_gather_qmm_noalloc: cudaGetDevice failed");
  if (dev < 0 || dev >= 64) return gqmm::report_error(GQMM_ERR_DEVICE, "gqmm_gather_qmm_noalloc: device ordinal >= 64");
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_dev_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr)
      return gqmm::report_error(GQMM_ERR_CUDA, "gqmm_gather_qmm_noalloc: cudaGetSymbolAddress failed");
    g_scratch_dev_ptr[dev] = p;
  }
  *out = g_scratch_dev_ptr[dev];
  return GQMM_OK;
}

}  // namespace

extern "C" int gqmm_gather_qmm_noalloc(const void* x, const void* wq, const void* scales, const void* biases,
                                       const uint32_t* idx, int64_t T, int A, int H, int F, int E, int group_size,
                                       int bits, int sorted, void* y, gqmm_stream_t stream) {
  // Split K (used when a call has too few work units for the GPU) needs partial-sum planes
  // in the scratch; it is used only when those fit too, else the call runs unsplit.
  // Sizes the C ABI rejects anyway are passed through for gather_qmm_impl to report.
  bool allow_split = true;
  const bool sizes_ok = T >= 1 && A >= 1 && T * (int64_t)A <= 2147483647LL && F > 0 && E >= 1 &&
                        E <= GQMM_MAX_EXPERTS;
  if (sizes_ok) {
    const int64_t n = T * (int64_t)A;
    if (gqmm::ws_layout(n, F, E, true).total > kScratchBytes) {
      allow_split = false;
      const size_t need = gqmm::ws_layout(n, F, E, false).total;
      if (need > kScratchBytes)
        return gqmm::report_error(GQMM_ERR_WORKSPACE,
                                  "gqmm_gather_qmm_noalloc: T*A=%lld rows with E=%d need %zu bytes of scratch, "
                                  "more than the built-in %zu bytes (GQMM_NOALLOC_SCRATCH_BYTES); "
                                  "use gqmm_gather_qmm with a caller workspace",
                                  (long long)n, E, need, kScratchBytes);
    }
  }
  void* ws = nullptr;
  int rc = scratch_for_current_device(&ws);
  if (rc != GQMM_OK) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // The header at the start of the scratch (status word included) is cleared on every call,
  // after the arguments have been validated (a refused call enqueues nothing): nothing reads
  // the status back through this entry point, and it must not carry bits from earlier calls.
  return gqmm::gather_qmm_impl(x, wq, scales, biases, idx, T, A, H, F, E, group_size, bits, sorted, 0, y, ws,
                               kScratchBytes, s, allow_split, /*clear_header=*/true);
}
