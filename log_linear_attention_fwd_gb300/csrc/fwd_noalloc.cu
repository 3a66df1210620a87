// loglinear_fwd_noalloc: the forward with its scratch in a fixed device array.
//
// Some callers cannot allocate device memory: a plugin inside a host application that
// owns every byte of device memory and gives extensions no allocator, or a real-time loop
// in which cudaMalloc (which may synchronise the whole device) is not allowed.  For them
// this entry point takes the same inputs and output as loglinear_fwd but no workspace:
// the forward's scratch (per-chunk states, Fenwick block states, per-chunk log decays)
// lives in g_noalloc_scratch below, a file-scope device array of kNoallocScratchBytes.
//
// Facts a caller must know:
//   * Every GPU on which the library's device code is loaded holds this array until the
//     process exits.
//   * The first call on a device, with that device current, looks the array's device
//     address up (cudaGetSymbolAddress) and caches it; that first call should come before
//     any stream capture.
//   * All calls share the one array, and it keeps the last call's contents.  The forward
//     writes every scratch entry before it reads it, so nothing needs clearing between
//     calls; but two calls whose work overlaps on the GPU (different streams, or different
//     host threads) race on the array and give wrong results.  Serialise them.
//   * Problems whose scratch would exceed kNoallocScratchBytes are rejected with
//     LL_ERR_WORKSPACE before anything is launched.
#include <mutex>

#include "ll_internal.cuh"

namespace ll {
namespace {

constexpr size_t kNoallocScratchBytes = LL_FWD_NOALLOC_SCRATCH_BYTES;  // 32 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// Device address of g_noalloc_scratch, looked up once per device.  In host code the
// array's name only stands in for the symbol; it is not a device address.
constexpr int kMaxDevices = 128;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

cudaError_t scratch_on_current_device(void** addr) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *addr = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace ll

extern "C" {

int loglinear_fwd_noalloc(const void* q, const void* k, const void* v, const float* log_a,
                          const float* lambda, void* out, int64_t B, int64_t T, int64_t H,
                          int64_t Hqk, int64_t dk, int64_t dv, int64_t L, int chunk, int in_dtype,
                          int out_dtype, int path, ll_stream_t stream) {
  size_t need = 0;
  const int st = loglinear_fwd_workspace_size(B, T, H, dk, dv, chunk, in_dtype, path, &need);
  if (st != LL_OK) return st;
  if (need > ll::kNoallocScratchBytes) return LL_ERR_WORKSPACE;
  void* scratch = nullptr;
  const cudaError_t e = ll::scratch_on_current_device(&scratch);
  if (e != cudaSuccess) return ll::report_cuda_error(e);
  return loglinear_fwd(q, k, v, log_a, lambda, out, B, T, H, Hqk, dk, dv, L, chunk, in_dtype,
                       out_dtype, path, scratch, ll::kNoallocScratchBytes, stream);
}

}  // extern "C"
