// bfp8_linear_fwd_static: the blockwise-FP8 linear forward for callers that
// cannot allocate device memory.
//
// bfp8_linear_fwd needs a caller-provided workspace for the quantised x and W
// and their scales.  Some callers cannot provide one: code that runs inside a
// CUDA stream capture (where cudaMalloc is not allowed), plugins hosted by a
// framework that owns every allocation and exposes no allocator, or
// latency-critical paths that must not enter the driver's allocator.  This
// entry point takes the same inputs and output as bfp8_linear_fwd but keeps
// its scratch in one fixed array in device memory that the library reserves
// when it is loaded.
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
//   - the first call on each device looks up the array's device address
//     (cudaGetSymbolAddress) with that device current; make that first call
//     before any stream capture, since the lookup may not be capturable.
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

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64];  // device address of g_noalloc_scratch, per device ordinal

size_t a256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

extern "C" bfp8_status bfp8_linear_fwd_static(const void* x, const void* w, void* y, int64_t M, int64_t N, int64_t K,
                                              bfp8_stream_t stream) {
  using bfp8::cdiv;
  if (M < 0 || N < 0 || K < 0) {
    bfp8::set_last_error("bfp8_linear_fwd_static: negative dimension");
    return BFP8_ERR_INVALID_ARG;
  }
  if (M == 0 || N == 0 || K == 0) return bfp8_linear_fwd(x, w, y, M, N, K, nullptr, 0, stream);
  // layout of the quantised operands inside the scratch (as in bfp8_linear_fwd)
  const int64_t ldK = cdiv(K, 16) * 16, ldsM = cdiv(M, 4) * 4, Kb = cdiv(K, 128), Nb = cdiv(N, 128);
  size_t o = 0;
  const size_t qx = o;
  o = a256(o + (size_t)M * ldK);
  const size_t sx = o;
  o = a256(o + (size_t)Kb * ldsM * 4);
  const size_t qw = o;
  o = a256(o + (size_t)N * ldK);
  const size_t sw = o;
  o = a256(o + (size_t)Nb * Kb * 4);
  if (o > kNoAllocScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof msg,
             "bfp8_linear_fwd_static: M=%lld N=%lld K=%lld needs %zu bytes of scratch, above its fixed %zu",
             (long long)M, (long long)N, (long long)K, o, kNoAllocScratchBytes);
    bfp8::set_last_error(msg);
    return BFP8_ERR_INVALID_ARG;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    bfp8::set_last_error("bfp8_linear_fwd_static: no usable current device");
    return BFP8_ERR_CUDA;
  }
  void* base = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (g_noalloc_ptr[dev] == nullptr) {
      void* p = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess || p == nullptr) {
        bfp8::set_last_error("bfp8_linear_fwd_static: cudaGetSymbolAddress of the scratch array failed");
        return BFP8_ERR_CUDA;
      }
      g_noalloc_ptr[dev] = p;
    }
    base = g_noalloc_ptr[dev];
  }
  uint8_t* b = static_cast<uint8_t*>(base);
  bfp8_status st = bfp8_quant_lhs(x, M, K, K, 0, b + qx, ldK, reinterpret_cast<float*>(b + sx), ldsM, stream);
  if (st != BFP8_OK) return st;
  st = bfp8_quant_weight(w, N, K, K, b + qw, ldK, nullptr, 0, reinterpret_cast<float*>(b + sw), Kb, stream);
  if (st != BFP8_OK) return st;
  return bfp8_gemm_1x128_128x128(b + qx, ldK, reinterpret_cast<const float*>(b + sx), ldsM, b + qw, ldK,
                                 reinterpret_cast<const float*>(b + sw), Kb, 0, y, N, M, N, K, stream);
}
