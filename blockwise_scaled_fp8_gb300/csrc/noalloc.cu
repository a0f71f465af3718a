// bfp8_linear_fwd_static: the blockwise-FP8 linear forward for callers that
// cannot allocate device memory.
//
// bfp8_linear_fwd needs a caller-provided workspace for the quantised x and W
// and their scales.  Some callers cannot provide one: plugins hosted by a
// framework that owns every allocation and hands them no allocator, and
// latency-critical paths that must not enter the driver's allocator (a
// cudaMalloc can synchronise the device and take milliseconds).  This entry
// point takes the same inputs and output as bfp8_linear_fwd, runs the same
// launches, and keeps its scratch in one fixed array in device memory that
// the library reserves when it is loaded.
//
// Limits and sharing:
//   - the scratch holds at most kNoAllocScratchBytes (32 MiB); problems whose
//     quantised operands do not fit are rejected with BFP8_ERR_INVALID_ARG;
//   - every GPU that loads the library keeps these 32 MiB until the process
//     exits;
//   - all calls share the one array, on every stream: two calls whose work
//     overlaps on the GPU race on it and produce wrong results; order them on
//     one stream (or with events);
//   - the array keeps the previous call's contents; nothing in it has to start
//     at zero, because every byte the kernels read is written earlier in the
//     same call;
//   - the first call in each CUDA context (normally: once per device) looks up
//     the array's device address (cudaGetSymbolAddress) with that device
//     current, and remembers it for that context.  A new context on the same
//     device (after cudaDeviceReset, or a driver-API context made current by
//     the caller) loads the library's module again, possibly at another
//     address, and is looked up again on its first call.
#include <cudaTypedefs.h>

#include <mutex>

#include <stdio.h>

#include "../../include/bfp8.h"
#include "index.cuh"
#include "kernels.h"

static constexpr size_t kNoAllocScratchBytes = (size_t)32 << 20;

// The scratch itself.  In host code this name is only a stand-in for the
// symbol: its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

// The current context's unique id (cuCtxGetId: never reused within a
// process), or 0 when it cannot be read.
unsigned long long current_context_id() {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// The array's device address in each context seen so far.
struct ScratchAddr {
  unsigned long long ctx_id;
  void* ptr;
};
std::mutex g_noalloc_mu;
ScratchAddr g_noalloc_addr[64];
int g_noalloc_next = 0;

// Set-up, with the device current: the array's address in the current
// context, looked up once per context.
bfp8_status scratch_address(void** out) {
  const unsigned long long id = current_context_id();
  if (id == 0) {
    bfp8::set_last_error("bfp8_linear_fwd_static: cannot identify the current CUDA context");
    return BFP8_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  for (const ScratchAddr& a : g_noalloc_addr)
    if (a.ctx_id == id) {
      *out = a.ptr;
      return BFP8_OK;
    }
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess || p == nullptr) {
    char msg[256];
    snprintf(msg, sizeof msg, "bfp8_linear_fwd_static: cudaGetSymbolAddress of the scratch array failed: %s",
             cudaGetErrorString(e));
    bfp8::set_last_error(msg);
    return BFP8_ERR_CUDA;
  }
  g_noalloc_addr[g_noalloc_next] = ScratchAddr{id, p};
  g_noalloc_next = (g_noalloc_next + 1) % 64;
  *out = p;
  return BFP8_OK;
}

}  // namespace

extern "C" bfp8_status bfp8_linear_fwd_static(const void* x, const void* w, void* y, int64_t M, int64_t N, int64_t K,
                                              bfp8_stream_t stream) {
  if (M < 0 || N < 0 || K < 0) {
    bfp8::set_last_error("bfp8_linear_fwd_static: negative dimension");
    return BFP8_ERR_INVALID_ARG;
  }
  if (M == 0 || N == 0 || K == 0) return bfp8_linear_fwd(x, w, y, M, N, K, nullptr, 0, stream);
  if (!x || !w || !y) {
    bfp8::set_last_error("bfp8_linear_fwd_static: null pointer");
    return BFP8_ERR_INVALID_ARG;
  }
  if (M >= ((int64_t)1 << 31) || N >= ((int64_t)1 << 31) || K >= ((int64_t)1 << 31)) {
    bfp8::set_last_error("bfp8_linear_fwd_static: dimension >= 2^31");
    return BFP8_ERR_INVALID_ARG;
  }
  const size_t need = bfp8::linear_fwd_scratch_bytes(M, N, K);
  if (need > kNoAllocScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof msg,
             "bfp8_linear_fwd_static: M=%lld N=%lld K=%lld needs %zu bytes of scratch, above its fixed %zu",
             (long long)M, (long long)N, (long long)K, need, kNoAllocScratchBytes);
    bfp8::set_last_error(msg);
    return BFP8_ERR_INVALID_ARG;
  }
  int sms = 0;
  bfp8_status st = bfp8::check_current_device(&sms);  // sm_103a, and the thread's device current
  if (st != BFP8_OK) return st;
  void* base = nullptr;
  if ((st = scratch_address(&base)) != BFP8_OK) return st;
  return bfp8::linear_fwd_into(x, w, y, M, N, K, static_cast<uint8_t*>(base), sms, stream);
}
