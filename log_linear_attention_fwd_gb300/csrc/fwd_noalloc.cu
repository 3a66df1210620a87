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
//     address up (cudaGetSymbolAddress, which also loads the module on that device) and
//     caches it together with the unique ID of the current CUDA context; that first call
//     should come before any stream capture.  A later call under another context (after
//     cudaDeviceReset, or once the application replaced the primary context) looks the
//     address up again, since the module, and the array with it, moved.
//   * All calls share the one array, and it keeps the last call's contents.  The forward
//     writes every scratch entry before it reads it, so nothing needs clearing between
//     calls; but two calls whose work overlaps on the GPU (different streams, or different
//     host threads) race on the array and give wrong results.  Serialise them.
//   * Problems whose scratch would exceed kNoallocScratchBytes are rejected with
//     LL_ERR_WORKSPACE before anything is launched.
#include <cuda.h>

#include <mutex>

#include "ll_internal.cuh"

namespace ll {
namespace {

constexpr size_t kNoallocScratchBytes = LL_FWD_NOALLOC_SCRATCH_BYTES;  // 32 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// Device address of g_noalloc_scratch, looked up once per device and context.  In host
// code the array's name only stands in for the symbol; it is not a device address.
constexpr int kMaxDevices = 128;
struct ScratchAddr {
  unsigned long long ctx_id;  // unique ID of the context the address belongs to (0: none)
  void* addr;
};
std::mutex g_scratch_mu;
ScratchAddr g_scratch_addr[kMaxDevices] = {};

// Unique ID of the calling thread's current CUDA context, or 0 when there is none or the
// driver does not offer the query.  Context IDs are never reused within a process, unlike
// context handles.
unsigned long long current_context_id() {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(p);
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

cudaError_t scratch_on_current_device(void** addr) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  const unsigned long long id = current_context_id();
  ScratchAddr& c = g_scratch_addr[dev];
  if (!c.addr || id == 0 || c.ctx_id != id) {
    // first call on this device, or another context than the cached address belongs to
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    c.addr = p;
    c.ctx_id = current_context_id();  // the lookup made a context current if none was
  }
  *addr = c.addr;
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
