// C ABI of the library (declared in include/bfp8.h): argument validation,
// device checks, the linear-layer composition and the host-side index replay.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>
#include <vector>

#include "../../include/bfp8.h"
#include "index.cuh"
#include "kernels.h"

using namespace bfp8;

namespace {

thread_local char g_msg[512] = "";

bfp8_status fail(bfp8_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof g_msg, fmt, ap);
  va_end(ap);
  return st;
}

bfp8_status cuda_fail(cudaError_t e, const char* where) {
  return fail(BFP8_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

struct DevInfo {
  int checked = 0;
  int ok = 0;
  int sms = 0;
  int major = 0, minor = 0;
};
DevInfo g_dev[64];
std::mutex g_dev_mu;

// A host thread that never selected a device (an autograd worker, a thread
// pool) reports device 0 without having its primary context current, and an
// extensible launch from it fails with "invalid argument".  Selecting the
// device once per thread makes the context current.
bfp8_status bind_thread_device(int* dev_out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  thread_local int bound = -1;
  if (bound != dev) {
    e = cudaSetDevice(dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaSetDevice");
    bound = dev;
  }
  *dev_out = dev;
  return BFP8_OK;
}

// The kernels are built for sm_103a only.  Returns the SM count via *sms.
bfp8_status check_device(int* sms) {
  int dev = 0;
  bfp8_status st = bind_thread_device(&dev);
  if (st != BFP8_OK) return st;
  if (dev < 0 || dev >= 64) return fail(BFP8_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DevInfo& d = g_dev[dev];
  if (!d.checked) {
    cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    d.ok = (d.major == 10 && d.minor == 3);
    d.checked = 1;
  }
  if (!d.ok)
    return fail(BFP8_ERR_UNSUPPORTED, "bfp8 kernels are built for sm_103a (GB300); device %d is sm_%d%d",
                dev, d.major, d.minor);
  *sms = d.sms;
  return BFP8_OK;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool al4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
bool al2(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 1u) == 0; }
constexpr int64_t kMaxDim = (int64_t)1 << 31;  // TMA coordinates are 32-bit signed
int64_t rup(int64_t a, int64_t b) { return cdiv(a, b) * b; }

#define CHECK_ARG(cond, ...)                                  \
  do {                                                        \
    if (!(cond)) return fail(BFP8_ERR_INVALID_ARG, __VA_ARGS__); \
  } while (0)

bfp8_status check_dims(const char* fn, int64_t a, int64_t b, int64_t c = 1) {
  CHECK_ARG(a >= 0 && b >= 0 && c >= 0, "%s: negative dimension", fn);
  CHECK_ARG(a < kMaxDim && b < kMaxDim && c < kMaxDim, "%s: dimension >= 2^31", fn);
  return BFP8_OK;
}

}  // namespace

void bfp8::set_last_error(const char* msg) { snprintf(g_msg, sizeof g_msg, "%s", msg); }

extern "C" {

const char* bfp8_last_error(void) { return g_msg; }

bfp8_status bfp8_quant_lhs(const void* x, int64_t M, int64_t K, int64_t ldx, int x_transposed, void* q,
                           int64_t ldq, float* s, int64_t lds, bfp8_stream_t stream) {
  bfp8_status st = check_dims("bfp8_quant_lhs", M, K);
  if (st != BFP8_OK) return st;
  if (M == 0 || K == 0) return BFP8_OK;
  CHECK_ARG(x && q && s, "bfp8_quant_lhs: null pointer");
  CHECK_ARG(al2(x) && al16(q) && al4(s), "bfp8_quant_lhs: x must be 2-byte, q 16-byte, s 4-byte aligned");
  CHECK_ARG(ldx >= (x_transposed ? M : K), "bfp8_quant_lhs: ldx=%lld < %s=%lld", (long long)ldx,
            x_transposed ? "M" : "K", (long long)(x_transposed ? M : K));
  CHECK_ARG(ldq >= K && ldq % 16 == 0, "bfp8_quant_lhs: ldq=%lld must be >= K=%lld and a multiple of 16",
            (long long)ldq, (long long)K);
  CHECK_ARG(lds >= M, "bfp8_quant_lhs: lds=%lld < M=%lld", (long long)lds, (long long)M);
  int sms = 0;
  if ((st = check_device(&sms)) != BFP8_OK) return st;
  cudaError_t e;
  const uint16_t* xb = (const uint16_t*)x;
  const bool tiled = x_transposed ? quant_tile_supported(x, ldx, nullptr, 0, q, ldq)
                                   : quant_tile_supported(x, ldx, q, ldq, nullptr, 0);
  if (tiled) {
    if (x_transposed)  // x is [K, M]: 128x1 groups of x along K are 1x128 groups of A = x^T
      e = launch_quant_tile(
          QuantTileArgs{kQuantTileCol, xb, K, M, ldx, nullptr, 0, nullptr, 0, (uint8_t*)q, ldq, s, lds}, sms,
          (cudaStream_t)stream);
    else
      e = launch_quant_tile(
          QuantTileArgs{kQuantTileRow, xb, M, K, ldx, (uint8_t*)q, ldq, s, lds, nullptr, 0, nullptr, 0}, sms,
          (cudaStream_t)stream);
  } else if (x_transposed) {
    e = launch_quant_cols(xb, K, M, ldx, (uint8_t*)q, ldq, s, lds, (cudaStream_t)stream);
  } else {
    e = launch_quant_rows(xb, M, K, ldx, (uint8_t*)q, ldq, s, lds, sms, (cudaStream_t)stream);
  }
  return e == cudaSuccess ? BFP8_OK : cuda_fail(e, "bfp8_quant_lhs launch");
}

bfp8_status bfp8_quant_rhs(const void* x, int64_t K, int64_t N, int64_t ldx, void* qT, int64_t ldq, float* s,
                           int64_t lds, bfp8_stream_t stream) {
  bfp8_status st = check_dims("bfp8_quant_rhs", K, N);
  if (st != BFP8_OK) return st;
  if (K == 0 || N == 0) return BFP8_OK;
  CHECK_ARG(x && qT && s, "bfp8_quant_rhs: null pointer");
  CHECK_ARG(al2(x) && al16(qT) && al4(s), "bfp8_quant_rhs: x must be 2-byte, qT 16-byte, s 4-byte aligned");
  CHECK_ARG(ldx >= N, "bfp8_quant_rhs: ldx=%lld < N=%lld", (long long)ldx, (long long)N);
  CHECK_ARG(ldq >= K && ldq % 16 == 0, "bfp8_quant_rhs: ldq=%lld must be >= K=%lld and a multiple of 16",
            (long long)ldq, (long long)K);
  CHECK_ARG(lds >= N, "bfp8_quant_rhs: lds=%lld < N=%lld", (long long)lds, (long long)N);
  int sms = 0;
  if ((st = check_device(&sms)) != BFP8_OK) return st;
  cudaError_t e;
  if (quant_tile_supported(x, ldx, nullptr, 0, qT, ldq))
    e = launch_quant_tile(QuantTileArgs{kQuantTileCol, (const uint16_t*)x, K, N, ldx, nullptr, 0, nullptr, 0,
                                        (uint8_t*)qT, ldq, s, lds},
                          sms, (cudaStream_t)stream);
  else
    e = launch_quant_cols((const uint16_t*)x, K, N, ldx, (uint8_t*)qT, ldq, s, lds, (cudaStream_t)stream);
  return e == cudaSuccess ? BFP8_OK : cuda_fail(e, "bfp8_quant_rhs launch");
}

bfp8_status bfp8_quant_weight(const void* w, int64_t N, int64_t K, int64_t ldw, void* q, int64_t ldq, void* qt,
                              int64_t ldqt, float* s, int64_t lds, bfp8_stream_t stream) {
  bfp8_status st = check_dims("bfp8_quant_weight", N, K);
  if (st != BFP8_OK) return st;
  if (N == 0 || K == 0) return BFP8_OK;
  CHECK_ARG(w && s && (q || qt), "bfp8_quant_weight: null pointer (w, s, and one of q/qt are required)");
  CHECK_ARG(al2(w) && al4(s), "bfp8_quant_weight: w must be 2-byte, s 4-byte aligned");
  CHECK_ARG(ldw >= K, "bfp8_quant_weight: ldw=%lld < K=%lld", (long long)ldw, (long long)K);
  if (q) {
    CHECK_ARG(al16(q), "bfp8_quant_weight: q must be 16-byte aligned");
    CHECK_ARG(ldq >= K && ldq % 16 == 0, "bfp8_quant_weight: ldq=%lld must be >= K=%lld and a multiple of 16",
              (long long)ldq, (long long)K);
  }
  if (qt) {
    CHECK_ARG(al16(qt), "bfp8_quant_weight: qt must be 16-byte aligned");
    CHECK_ARG(ldqt >= N && ldqt % 16 == 0,
              "bfp8_quant_weight: ldqt=%lld must be >= N=%lld and a multiple of 16", (long long)ldqt, (long long)N);
  }
  CHECK_ARG(lds >= cdiv(K, kBlock), "bfp8_quant_weight: lds=%lld < ceil(K/128)=%lld", (long long)lds,
            (long long)cdiv(K, kBlock));
  int sms = 0;
  if ((st = check_device(&sms)) != BFP8_OK) return st;
  cudaError_t e;
  if (quant_tile_supported(w, ldw, q, ldq, qt, ldqt))
    e = launch_quant_tile(QuantTileArgs{kQuantTileScale, (const uint16_t*)w, N, K, ldw, (uint8_t*)q, ldq, s, lds,
                                        (uint8_t*)qt, ldqt, nullptr, 0},
                          sms, (cudaStream_t)stream);
  else
    e = launch_quant_weight((const uint16_t*)w, N, K, ldw, (uint8_t*)q, ldq, (uint8_t*)qt, ldqt, s, lds,
                            (cudaStream_t)stream);
  return e == cudaSuccess ? BFP8_OK : cuda_fail(e, "bfp8_quant_weight launch");
}

bfp8_status bfp8_quant_dual(const void* x, int64_t T, int64_t C, int64_t ldx, void* q_row, int64_t ldq_row,
                            float* s_row, int64_t lds_row, void* q_col, int64_t ldq_col, float* s_col,
                            int64_t lds_col, bfp8_stream_t stream) {
  bfp8_status st = check_dims("bfp8_quant_dual", T, C);
  if (st != BFP8_OK) return st;
  if (T == 0 || C == 0) return BFP8_OK;
  CHECK_ARG(x && q_row && s_row && q_col && s_col, "bfp8_quant_dual: null pointer");
  CHECK_ARG(al2(x) && al16(q_row) && al16(q_col) && al4(s_row) && al4(s_col),
            "bfp8_quant_dual: x must be 2-byte, q_row/q_col 16-byte, scales 4-byte aligned");
  CHECK_ARG(ldx >= C, "bfp8_quant_dual: ldx=%lld < C=%lld", (long long)ldx, (long long)C);
  CHECK_ARG(ldq_row >= C && ldq_row % 16 == 0, "bfp8_quant_dual: ldq_row=%lld must be >= C and a multiple of 16",
            (long long)ldq_row);
  CHECK_ARG(ldq_col >= T && ldq_col % 16 == 0, "bfp8_quant_dual: ldq_col=%lld must be >= T and a multiple of 16",
            (long long)ldq_col);
  CHECK_ARG(lds_row >= T, "bfp8_quant_dual: lds_row=%lld < T=%lld", (long long)lds_row, (long long)T);
  CHECK_ARG(lds_col >= C, "bfp8_quant_dual: lds_col=%lld < C=%lld", (long long)lds_col, (long long)C);
  int sms = 0;
  if ((st = check_device(&sms)) != BFP8_OK) return st;
  cudaError_t e;
  const uint16_t* xb = (const uint16_t*)x;
  if (quant_tile_supported(x, ldx, q_row, ldq_row, q_col, ldq_col)) {
    e = launch_quant_tile(QuantTileArgs{kQuantTileRow | kQuantTileCol, xb, T, C, ldx, (uint8_t*)q_row, ldq_row, s_row,
                                        lds_row, (uint8_t*)q_col, ldq_col, s_col, lds_col},
                          sms, (cudaStream_t)stream);
  } else {
    e = launch_quant_rows(xb, T, C, ldx, (uint8_t*)q_row, ldq_row, s_row, lds_row, sms, (cudaStream_t)stream);
    if (e == cudaSuccess)
      e = launch_quant_cols(xb, T, C, ldx, (uint8_t*)q_col, ldq_col, s_col, lds_col, (cudaStream_t)stream);
  }
  return e == cudaSuccess ? BFP8_OK : cuda_fail(e, "bfp8_quant_dual launch");
}

bfp8_status bfp8_quant_dual_weight(const void* x, int64_t T, int64_t C, int64_t ldx, void* q_row, int64_t ldq_row,
                                   float* s_row, int64_t lds_row, void* q_col, int64_t ldq_col, float* s_col,
                                   int64_t lds_col, const void* w, int64_t N, int64_t ldw, void* qw, int64_t ldqw,
                                   void* qwt, int64_t ldqwt, float* sw, int64_t ldsw, bfp8_stream_t stream) {
  bfp8_status st = check_dims("bfp8_quant_dual_weight", T, C, N);
  if (st != BFP8_OK) return st;
  CHECK_ARG(x && q_row && s_row && q_col && s_col && w && qw && qwt && sw, "bfp8_quant_dual_weight: null pointer");
  CHECK_ARG(al2(x) && al2(w) && al16(q_row) && al16(q_col) && al16(qw) && al16(qwt) && al4(s_row) && al4(s_col) &&
                al4(sw),
            "bfp8_quant_dual_weight: x, w 2-byte, codes 16-byte, scales 4-byte aligned");
  CHECK_ARG(ldx >= C && ldw >= C, "bfp8_quant_dual_weight: ldx=%lld / ldw=%lld < C=%lld", (long long)ldx,
            (long long)ldw, (long long)C);
  CHECK_ARG(ldq_row >= C && ldq_row % 16 == 0 && ldqw >= C && ldqw % 16 == 0,
            "bfp8_quant_dual_weight: ldq_row and ldqw must be >= C and multiples of 16");
  CHECK_ARG(ldq_col >= T && ldq_col % 16 == 0, "bfp8_quant_dual_weight: ldq_col=%lld must be >= T and a multiple of 16",
            (long long)ldq_col);
  CHECK_ARG(ldqwt >= N && ldqwt % 16 == 0, "bfp8_quant_dual_weight: ldqwt=%lld must be >= N and a multiple of 16",
            (long long)ldqwt);
  CHECK_ARG(lds_row >= T && lds_col >= C && ldsw >= cdiv(C, kBlock), "bfp8_quant_dual_weight: scale stride too small");
  // one of the inputs empty, or an input the TMA tile path cannot read (not
  // 16-byte aligned, or rows not of 16-byte multiples): the two calls on their own
  if (T == 0 || C == 0 || N == 0 || !quant_tile_supported(x, ldx, q_row, ldq_row, q_col, ldq_col) ||
      !quant_tile_supported(w, ldw, qw, ldqw, qwt, ldqwt)) {
    if ((st = bfp8_quant_dual(x, T, C, ldx, q_row, ldq_row, s_row, lds_row, q_col, ldq_col, s_col, lds_col, stream)) !=
        BFP8_OK)
      return st;
    return bfp8_quant_weight(w, N, C, ldw, qw, ldqw, qwt, ldqwt, sw, ldsw, stream);
  }
  int sms = 0;
  if ((st = check_device(&sms)) != BFP8_OK) return st;
  const cudaError_t e = launch_quant_tile_pair(
      QuantTileArgs{kQuantTileRow | kQuantTileCol, (const uint16_t*)x, T, C, ldx, (uint8_t*)q_row, ldq_row, s_row,
                    lds_row, (uint8_t*)q_col, ldq_col, s_col, lds_col},
      QuantTileArgs{kQuantTileScale, (const uint16_t*)w, N, C, ldw, (uint8_t*)qw, ldqw, sw, ldsw, (uint8_t*)qwt, ldqwt,
                    nullptr, 0},
      sms, (cudaStream_t)stream);
  return e == cudaSuccess ? BFP8_OK : cuda_fail(e, "bfp8_quant_dual_weight launch");
}

bfp8_status bfp8_mx_cast(const void* x, int64_t M, int64_t K, int64_t ldx, void* q0, int64_t ldq0, void* e0,
                         int64_t lde0, void* q1, int64_t ldq1, void* e1, int64_t lde1, bfp8_stream_t stream) {
  bfp8_status st = check_dims("bfp8_mx_cast", M, K);
  if (st != BFP8_OK) return st;
  if (M == 0 || K == 0) return BFP8_OK;
  CHECK_ARG(x && (q0 || q1), "bfp8_mx_cast: null input or no output asked for");
  CHECK_ARG(!q0 == !e0 && !q1 == !e1, "bfp8_mx_cast: each cast needs its codes and its exponents");
  CHECK_ARG(ldx >= K, "bfp8_mx_cast: ldx=%lld < K=%lld", (long long)ldx, (long long)K);
  if (q0) {
    CHECK_ARG(ldq0 >= K && ldq0 % 16 == 0, "bfp8_mx_cast: ldq0=%lld must be >= K and a multiple of 16",
              (long long)ldq0);
    CHECK_ARG(lde0 >= cdiv(K, 32), "bfp8_mx_cast: lde0=%lld < ceil(K/32)", (long long)lde0);
  }
  if (q1) {
    CHECK_ARG(ldq1 >= M && ldq1 % 16 == 0, "bfp8_mx_cast: ldq1=%lld must be >= M and a multiple of 16",
              (long long)ldq1);
    CHECK_ARG(lde1 >= cdiv(M, 32), "bfp8_mx_cast: lde1=%lld < ceil(M/32)", (long long)lde1);
  }
  CHECK_ARG(quant_tile_supported(x, ldx, q0, ldq0, q1, ldq1),
            "bfp8_mx_cast: x and the codes must be 16-byte aligned, ldx a multiple of 8");
  int sms = 0;
  if ((st = check_device(&sms)) != BFP8_OK) return st;
  QuantTileArgs a{kQuantTileMx | (q0 ? kQuantTileRow : 0) | (q1 ? kQuantTileCol : 0),
                  (const uint16_t*)x, M, K, ldx, (uint8_t*)q0, ldq0, nullptr, 0, (uint8_t*)q1, ldq1, nullptr, 0,
                  (uint8_t*)e0, lde0, (uint8_t*)e1, lde1};
  const cudaError_t e = launch_quant_tile(a, sms, (cudaStream_t)stream);
  return e == cudaSuccess ? BFP8_OK : cuda_fail(e, "bfp8_mx_cast launch");
}

static bfp8_status gemm_common(const char* fn, const GemmArgs& a, bfp8_stream_t stream,
                               uint64_t wait_limit_ns = kWaitLimitNs, int debug_stall = 0) {
  bfp8_status st = check_dims(fn, a.M, a.N, a.K);
  if (st != BFP8_OK) return st;
  if (a.M == 0 || a.N == 0) return BFP8_OK;
  CHECK_ARG(a.qa && a.qb && a.sa && a.sb && a.c, "%s: null pointer", fn);
  if (a.K == 0) {  // empty reduction: C = 0 on the logical [M,N] region
    CHECK_ARG(a.ldc >= a.N, "%s: ldc=%lld < N=%lld", fn, (long long)a.ldc, (long long)a.N);
    cudaError_t e = cudaMemset2DAsync(a.c, (size_t)a.ldc * 2, 0, (size_t)a.N * 2, (size_t)a.M,
                                      (cudaStream_t)stream);
    return e == cudaSuccess ? BFP8_OK : cuda_fail(e, fn);
  }
  CHECK_ARG(al16(a.qa) && al16(a.qb), "%s: qa and qb must be 16-byte aligned", fn);
  CHECK_ARG(al4(a.sa) && al4(a.sb) && al2(a.c), "%s: sa/sb must be 4-byte and c 2-byte aligned", fn);
  CHECK_ARG(a.lda >= a.K && a.lda % 16 == 0, "%s: lda=%lld must be >= K=%lld and a multiple of 16", fn,
            (long long)a.lda, (long long)a.K);
  CHECK_ARG(a.ldb >= a.K && a.ldb % 16 == 0, "%s: ldb=%lld must be >= K=%lld and a multiple of 16", fn,
            (long long)a.ldb, (long long)a.K);
  CHECK_ARG(a.ldsa >= a.M, "%s: ldsa=%lld < M=%lld", fn, (long long)a.ldsa, (long long)a.M);
  const int64_t Kb = cdiv(a.K, kBlock), Nb = cdiv(a.N, kBlock);
  if (a.sb_mode == kSbTile)
    CHECK_ARG(a.ldsb >= Kb, "%s: ldsb=%lld < ceil(K/128)=%lld", fn, (long long)a.ldsb, (long long)Kb);
  else if (a.sb_mode == kSbTileT)
    CHECK_ARG(a.ldsb >= Nb, "%s: ldsb=%lld < ceil(N/128)=%lld", fn, (long long)a.ldsb, (long long)Nb);
  else
    CHECK_ARG(a.ldsb >= a.N, "%s: ldsb=%lld < N=%lld", fn, (long long)a.ldsb, (long long)a.N);
  CHECK_ARG(a.ldc >= a.N, "%s: ldc=%lld < N=%lld", fn, (long long)a.ldc, (long long)a.N);
  int sms = 0;
  if ((st = check_device(&sms)) != BFP8_OK) return st;
  const char* msg = nullptr;
  cudaError_t e = launch_gemm(a, sms, (cudaStream_t)stream, &msg, wait_limit_ns, debug_stall);
  if (e != cudaSuccess) {
    if (msg) return fail(BFP8_ERR_INVALID_ARG, "%s: %s", fn, msg);
    return cuda_fail(e, fn);
  }
  return BFP8_OK;
}

bfp8_status bfp8_gemm_1x128_128x128(const void* qa, int64_t lda, const float* sa, int64_t ldsa, const void* qb,
                                    int64_t ldb, const float* sb, int64_t ldsb, int sb_transposed, void* c,
                                    int64_t ldc, int64_t M, int64_t N, int64_t K, bfp8_stream_t stream) {
  GemmArgs a{qa, lda, sa, ldsa, qb, ldb, sb, ldsb, sb_transposed ? kSbTileT : kSbTile, c, ldc, M, N, K};
  return gemm_common("bfp8_gemm_1x128_128x128", a, stream);
}

bfp8_status bfp8_gemm_1x128_128x1(const void* qa, int64_t lda, const float* sa, int64_t ldsa, const void* qb,
                                  int64_t ldb, const float* sb, int64_t ldsb, void* c, int64_t ldc, int64_t M,
                                  int64_t N, int64_t K, bfp8_stream_t stream) {
  GemmArgs a{qa, lda, sa, ldsa, qb, ldb, sb, ldsb, kSbCol, c, ldc, M, N, K};
  return gemm_common("bfp8_gemm_1x128_128x1", a, stream);
}

bfp8_status bfp8_gemm_1x128_128x128_xq(const void* x, int64_t ldx, const void* qb, int64_t ldb, const float* sb,
                                       int64_t ldsb, void* c, int64_t ldc, int64_t M, int64_t N, int64_t K,
                                       bfp8_stream_t stream) {
  const char* fn = "bfp8_gemm_1x128_128x128_xq";
  bfp8_status st = check_dims(fn, M, N, K);
  if (st != BFP8_OK) return st;
  if (M == 0 || N == 0) return BFP8_OK;
  CHECK_ARG(c, "%s: null pointer", fn);
  if (K == 0) {  // empty reduction (x, qb, sb are not read): C = 0 on the logical [M,N] region
    CHECK_ARG(ldc >= N, "%s: ldc=%lld < N=%lld", fn, (long long)ldc, (long long)N);
    cudaError_t e = cudaMemset2DAsync(c, (size_t)ldc * 2, 0, (size_t)N * 2, (size_t)M, (cudaStream_t)stream);
    return e == cudaSuccess ? BFP8_OK : cuda_fail(e, fn);
  }
  CHECK_ARG(x && qb && sb, "%s: null pointer", fn);
  CHECK_ARG(al16(x) && al16(qb), "%s: x and qb must be 16-byte aligned", fn);
  CHECK_ARG(al4(sb) && al2(c), "%s: sb must be 4-byte and c 2-byte aligned", fn);
  CHECK_ARG(ldx >= K && ldx % 8 == 0, "%s: ldx=%lld must be >= K=%lld and a multiple of 8", fn, (long long)ldx,
            (long long)K);
  CHECK_ARG(ldb >= K && ldb % 16 == 0, "%s: ldb=%lld must be >= K=%lld and a multiple of 16", fn, (long long)ldb,
            (long long)K);
  const int64_t Kb = cdiv(K, kBlock);
  CHECK_ARG(ldsb >= Kb, "%s: ldsb=%lld < ceil(K/128)=%lld", fn, (long long)ldsb, (long long)Kb);
  CHECK_ARG(ldc >= N, "%s: ldc=%lld < N=%lld", fn, (long long)ldc, (long long)N);
  int sms = 0;
  if ((st = check_device(&sms)) != BFP8_OK) return st;
  const char* msg = nullptr;
  cudaError_t e = launch_gemm_xq(GemmXqArgs{x, ldx, qb, ldb, sb, ldsb, c, ldc, M, N, K}, sms, (cudaStream_t)stream,
                                 &msg);
  if (e != cudaSuccess) {
    if (msg) return fail(BFP8_ERR_INVALID_ARG, "%s: %s", fn, msg);
    return cuda_fail(e, fn);
  }
  return BFP8_OK;
}

bfp8_status bfp8_gemm_1x128_128x1_xq(const void* qa, int64_t lda, const float* sa, int64_t ldsa, const void* x,
                                     int64_t ldx, void* c, int64_t ldc, int64_t M, int64_t N, int64_t K,
                                     bfp8_stream_t stream) {
  const char* fn = "bfp8_gemm_1x128_128x1_xq";
  bfp8_status st = check_dims(fn, M, N, K);
  if (st != BFP8_OK) return st;
  if (M == 0 || N == 0) return BFP8_OK;
  CHECK_ARG(c, "%s: null pointer", fn);
  if (K == 0) {  // empty reduction (qa, sa, x are not read): C = 0 on the logical [M,N] region
    CHECK_ARG(ldc >= N, "%s: ldc=%lld < N=%lld", fn, (long long)ldc, (long long)N);
    cudaError_t e = cudaMemset2DAsync(c, (size_t)ldc * 2, 0, (size_t)N * 2, (size_t)M, (cudaStream_t)stream);
    return e == cudaSuccess ? BFP8_OK : cuda_fail(e, fn);
  }
  CHECK_ARG(qa && sa && x, "%s: null pointer", fn);
  CHECK_ARG(al16(qa) && al16(x), "%s: qa and x must be 16-byte aligned", fn);
  CHECK_ARG(al4(sa) && al2(c), "%s: sa must be 4-byte and c 2-byte aligned", fn);
  CHECK_ARG(lda >= K && lda % 16 == 0, "%s: lda=%lld must be >= K=%lld and a multiple of 16", fn, (long long)lda,
            (long long)K);
  CHECK_ARG(ldsa >= M, "%s: ldsa=%lld < M=%lld", fn, (long long)ldsa, (long long)M);
  CHECK_ARG(ldx >= N && ldx % 8 == 0, "%s: ldx=%lld must be >= N=%lld and a multiple of 8", fn, (long long)ldx,
            (long long)N);
  CHECK_ARG(ldc >= N, "%s: ldc=%lld < N=%lld", fn, (long long)ldc, (long long)N);
  int sms = 0;
  if ((st = check_device(&sms)) != BFP8_OK) return st;
  const char* msg = nullptr;
  cudaError_t e = launch_gemm_wgrad_xq(GemmWxqArgs{qa, lda, sa, ldsa, x, ldx, c, ldc, M, N, K}, sms,
                                       (cudaStream_t)stream, &msg);
  if (e != cudaSuccess) {
    if (msg) return fail(BFP8_ERR_INVALID_ARG, "%s: %s", fn, msg);
    return cuda_fail(e, fn);
  }
  return BFP8_OK;
}

// ---------------------------------------------------------------------------
// Grouped (mixture-of-experts) GEMMs
// ---------------------------------------------------------------------------

static bfp8_status grouped_common(const char* fn, const GemmGroupArgs& ga, bfp8_stream_t stream) {
  const GemmArgs& a = ga.g;
  CHECK_ARG(ga.E >= 1 && ga.E <= kMaxGroups, "%s: E=%lld must be in [1, %d]", fn, (long long)ga.E, kMaxGroups);
  CHECK_ARG(ga.offs && al4(ga.offs), "%s: offs must be a 4-byte aligned device pointer", fn);
  const bool rows = ga.kind == kGroupRows;
  bfp8_status st = check_dims(fn, ga.M_total, a.N, rows ? a.K : a.M);
  if (st != BFP8_OK) return st;
  const int64_t K = rows ? a.K : ga.M_total;  // the reduction extent of the maps
  if ((rows ? ga.M_total : a.M) == 0 || a.N == 0) return BFP8_OK;
  // (an empty reduction is the kernel's job too: every tile then has no
  // K-blocks and its outputs are written as zeros)
  CHECK_ARG(a.qa && a.qb && a.sa && a.sb && a.c, "%s: null pointer", fn);
  CHECK_ARG(al16(a.qa) && al16(a.qb), "%s: qa and qb must be 16-byte aligned", fn);
  CHECK_ARG(al4(a.sa) && al4(a.sb) && al2(a.c), "%s: sa/sb must be 4-byte and c 2-byte aligned", fn);
  // input gradient: expert e's B starts at K column e*K of the map, and a TMA
  // load must start on a 16-byte boundary
  CHECK_ARG(!(rows && ga.b_k_step && ga.E > 1 && K % 16 != 0),
            "%s: the input-gradient form needs K %% 16 == 0 (K=%lld) when E > 1", fn, (long long)K);
  const int64_t b_inner = rows && ga.b_k_step ? ga.E * K : K;
  CHECK_ARG(a.lda >= K && a.lda % 16 == 0, "%s: lda=%lld must be >= %lld and a multiple of 16", fn,
            (long long)a.lda, (long long)K);
  CHECK_ARG(a.ldb >= b_inner && a.ldb % 16 == 0, "%s: ldb=%lld must be >= %lld and a multiple of 16", fn,
            (long long)a.ldb, (long long)b_inner);
  CHECK_ARG(a.ldsa >= (rows ? ga.M_total : a.M), "%s: ldsa=%lld too small", fn, (long long)a.ldsa);
  const int64_t Kb = cdiv(K, kBlock), Nb = cdiv(a.N, kBlock);
  if (a.sb_mode == kSbTile)
    CHECK_ARG(a.ldsb >= Kb, "%s: ldsb=%lld < ceil(K/128)=%lld", fn, (long long)a.ldsb, (long long)Kb);
  else if (a.sb_mode == kSbTileT)
    CHECK_ARG(a.ldsb >= Nb, "%s: ldsb=%lld < ceil(N/128)=%lld", fn, (long long)a.ldsb, (long long)Nb);
  else
    CHECK_ARG(a.ldsb >= a.N, "%s: ldsb=%lld < N=%lld", fn, (long long)a.ldsb, (long long)a.N);
  CHECK_ARG(a.ldc >= a.N, "%s: ldc=%lld < N=%lld", fn, (long long)a.ldc, (long long)a.N);
  if (!rows)
    CHECK_ARG(ga.c_step >= a.M * a.ldc, "%s: c_expert_stride=%lld < M*ldc=%lld", fn, (long long)ga.c_step,
              (long long)(a.M * a.ldc));
  int sms = 0;
  if ((st = check_device(&sms)) != BFP8_OK) return st;
  const char* msg = nullptr;
  cudaError_t e = launch_gemm_grouped(ga, sms, (cudaStream_t)stream, &msg);
  if (e != cudaSuccess) {
    if (msg) return fail(BFP8_ERR_INVALID_ARG, "%s: %s", fn, msg);
    return cuda_fail(e, fn);
  }
  return BFP8_OK;
}

bfp8_status bfp8_gemm_grouped_1x128_128x128(const void* qa, int64_t lda, const float* sa, int64_t ldsa,
                                            const void* qb, int64_t ldb, const float* sb, int64_t ldsb,
                                            int sb_transposed, const int32_t* offs, int64_t E, void* c,
                                            int64_t ldc, int64_t M_total, int64_t N, int64_t K,
                                            bfp8_stream_t stream) {
  GemmGroupArgs ga;
  ga.g = GemmArgs{qa, lda, sa, ldsa, qb, ldb, sb, ldsb, sb_transposed ? kSbTileT : kSbTile, c, ldc, 0, N, K};
  ga.kind = kGroupRows;
  ga.offs = offs;
  ga.E = E;
  ga.M_total = M_total;
  // forward: expert e's weight rows e*N ..; input gradient: its K columns e*K ..
  ga.b_row_step = sb_transposed ? 0 : N;
  ga.b_k_step = sb_transposed ? K : 0;
  ga.sb_step = sb_transposed ? cdiv(K, kBlock) * ldsb : cdiv(N, kBlock) * ldsb;
  ga.c_step = 0;
  return grouped_common("bfp8_gemm_grouped_1x128_128x128", ga, stream);
}

bfp8_status bfp8_gemm_grouped_1x128_128x1(const void* qa, int64_t lda, const float* sa, int64_t ldsa,
                                          const void* qb, int64_t ldb, const float* sb, int64_t ldsb,
                                          const int32_t* offs, int64_t E, void* c, int64_t ldc,
                                          int64_t c_expert_stride, int64_t M, int64_t N, int64_t T,
                                          bfp8_stream_t stream) {
  GemmGroupArgs ga;
  ga.g = GemmArgs{qa, lda, sa, ldsa, qb, ldb, sb, ldsb, kSbCol, c, ldc, M, N, 0};
  ga.kind = kGroupRed;
  ga.offs = offs;
  ga.E = E;
  ga.M_total = T;
  ga.b_row_step = ga.b_k_step = 0;
  ga.sb_step = 0;
  ga.c_step = c_expert_stride;
  return grouped_common("bfp8_gemm_grouped_1x128_128x1", ga, stream);
}

bfp8_status bfp8_debug_gemm_stall(const void* qa, int64_t lda, const float* sa, int64_t ldsa, const void* qb,
                                  int64_t ldb, const float* sb, int64_t ldsb, void* c, int64_t ldc, int64_t M,
                                  int64_t N, int64_t K, int64_t wait_limit_us, bfp8_stream_t stream) {
  CHECK_ARG(wait_limit_us > 0 && wait_limit_us <= 2000000, "bfp8_debug_gemm_stall: wait limit must be in (0, 2 s]");
  CHECK_ARG(M > 0 && N > 0 && K > 0, "bfp8_debug_gemm_stall: needs a non-empty problem");
  GemmArgs a{qa, lda, sa, ldsa, qb, ldb, sb, ldsb, kSbTile, c, ldc, M, N, K};
  return gemm_common("bfp8_debug_gemm_stall", a, stream, (uint64_t)wait_limit_us * 1000ull, 1);
}

bfp8_status bfp8_cast_e4m3(const float* x, int64_t n, void* q, bfp8_stream_t stream) {
  CHECK_ARG(n >= 0, "bfp8_cast_e4m3: negative size");
  if (n == 0) return BFP8_OK;
  CHECK_ARG(x && q, "bfp8_cast_e4m3: null pointer");
  CHECK_ARG(al4(x), "bfp8_cast_e4m3: x must be 4-byte aligned");
  int sms = 0;
  bfp8_status st = check_device(&sms);
  if (st != BFP8_OK) return st;
  cudaError_t e = launch_cast(x, n, (uint8_t*)q, sms, (cudaStream_t)stream);
  return e == cudaSuccess ? BFP8_OK : cuda_fail(e, "bfp8_cast_e4m3 launch");
}

bfp8_status bfp8_check_device_errors(bfp8_stream_t stream) {
  int dev = 0;
  bfp8_status st = bind_thread_device(&dev);
  if (st != BFP8_OK) return st;
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "bfp8_check_device_errors: stream synchronize");
  uint32_t bits = 0, qbits = 0;
  e = gemm_read_errors(&bits);
  if (e != cudaSuccess) return cuda_fail(e, "bfp8_check_device_errors: read flag");
  e = quant_read_errors(&qbits);
  if (e != cudaSuccess) return cuda_fail(e, "bfp8_check_device_errors: read flag");
  if (qbits) return fail(BFP8_ERR_TIMEOUT, "quantisation kernel gave up waiting for its TMA tile loads");
  if (bits & 64u)  // kErrGroupOffsets
    return fail(BFP8_ERR_INVALID_ARG,
                "grouped GEMM: expert offsets decreasing, outside [0, total tokens], or (weight gradient) "
                "not on a 128-token boundary; the affected experts were computed with clamped offsets");
  if (bits) {
    return fail(BFP8_ERR_TIMEOUT,
                "GEMM kernel gave up on a bounded wait (flags 0x%x: %s%s%s%s%s)", bits,
                (bits & 1) ? "smem-stage-release " : "", (bits & 2) ? "tma-arrival " : "",
                (bits & 4) ? "tmem-release " : "", (bits & 8) ? "partial-product " : "",
                (bits & 16) ? "teardown-drain " : "");
  }
  return BFP8_OK;
}

// ---------------------------------------------------------------------------
// Linear layer
// ---------------------------------------------------------------------------

namespace {
size_t a256(size_t x) { return (x + 255) & ~(size_t)255; }

struct FwdLayout {
  size_t qx, sx, qw, sw, total;
  int64_t ldK, ldsM;
};
FwdLayout fwd_layout(int64_t M, int64_t N, int64_t K) {
  FwdLayout L;
  L.ldK = rup(K, 16);
  L.ldsM = rup(M, 4);
  const int64_t Kb = cdiv(K, kBlock), Nb = cdiv(N, kBlock);
  size_t o = 0;
  L.qx = o; o = a256(o + (size_t)M * L.ldK);
  L.sx = o; o = a256(o + (size_t)Kb * L.ldsM * 4);
  L.qw = o; o = a256(o + (size_t)N * L.ldK);
  L.sw = o; o = a256(o + (size_t)Nb * Kb * 4);
  L.total = o;
  return L;
}

struct BwdLayout {
  size_t qdy, sdy, qwt, sw, qdyt, sdyt, qxt, sxt, total;
  int64_t ldN, ldM, ldsM, ldsN, ldsK;
};
BwdLayout bwd_layout(int64_t M, int64_t N, int64_t K) {
  BwdLayout L;
  L.ldN = rup(N, 16);
  L.ldM = rup(M, 16);
  L.ldsM = rup(M, 4);
  L.ldsN = rup(N, 4);
  L.ldsK = rup(K, 4);
  const int64_t Kb = cdiv(K, kBlock), Nb = cdiv(N, kBlock), Mb = cdiv(M, kBlock);
  size_t o = 0;
  L.qdy = o; o = a256(o + (size_t)M * L.ldN);          // dY, 1x128 along N
  L.sdy = o; o = a256(o + (size_t)Nb * L.ldsM * 4);
  L.qwt = o; o = a256(o + (size_t)K * L.ldN);          // W^T bytes
  L.sw = o; o = a256(o + (size_t)Nb * Kb * 4);
  L.qdyt = o; o = a256(o + (size_t)N * L.ldM);         // dY^T, 1x128 along M
  L.sdyt = o; o = a256(o + (size_t)Mb * L.ldsN * 4);
  L.qxt = o; o = a256(o + (size_t)K * L.ldM);          // X, 128x1 along M, transposed
  L.sxt = o; o = a256(o + (size_t)Mb * L.ldsK * 4);
  L.total = o;
  return L;
}
}  // namespace

size_t bfp8_linear_workspace_size(int64_t M, int64_t N, int64_t K) {
  if (M <= 0 || N <= 0 || K <= 0) return 0;
  const size_t f = fwd_layout(M, N, K).total, b = bwd_layout(M, N, K).total;
  return f > b ? f : b;
}

bfp8_status bfp8_linear_fwd(const void* x, const void* w, void* y, int64_t M, int64_t N, int64_t K, void* ws,
                            size_t ws_bytes, bfp8_stream_t stream) {
  bfp8_status st = check_dims("bfp8_linear_fwd", M, N, K);
  if (st != BFP8_OK) return st;
  if (M == 0 || N == 0 || K == 0) {
    if (M > 0 && N > 0 && y) {
      cudaError_t e = cudaMemsetAsync(y, 0, (size_t)M * N * 2, (cudaStream_t)stream);
      if (e != cudaSuccess) return cuda_fail(e, "bfp8_linear_fwd");
    }
    return BFP8_OK;
  }
  CHECK_ARG(x && w && y && ws, "bfp8_linear_fwd: null pointer");
  CHECK_ARG((reinterpret_cast<uintptr_t>(ws) & 255u) == 0, "bfp8_linear_fwd: workspace must be 256-byte aligned");
  CHECK_ARG(ws_bytes >= bfp8_linear_workspace_size(M, N, K), "bfp8_linear_fwd: workspace too small (%zu < %zu)",
            ws_bytes, bfp8_linear_workspace_size(M, N, K));
  int sms = 0;
  if ((st = check_device(&sms)) != BFP8_OK) return st;
  return bfp8::linear_fwd_into(x, w, y, M, N, K, (uint8_t*)ws, sms, stream);
}

}  // extern "C"

size_t bfp8::linear_fwd_scratch_bytes(int64_t M, int64_t N, int64_t K) { return fwd_layout(M, N, K).total; }

bfp8_status bfp8::check_current_device(int* sms) { return check_device(sms); }

// The forward's quantisations and GEMM into scratch at base (laid out by
// fwd_layout, 256-byte aligned), after the caller validated the arguments.
bfp8_status bfp8::linear_fwd_into(const void* x, const void* w, void* y, int64_t M, int64_t N, int64_t K,
                                  uint8_t* base, int sms, bfp8_stream_t stream) {
  bfp8_status st;
  const FwdLayout L = fwd_layout(M, N, K);
  const int64_t Kb = cdiv(K, kBlock);
  if (quant_tile_supported(x, K, base + L.qx, L.ldK, nullptr, 0) && quant_tile_supported(w, K, base + L.qw, L.ldK,
                                                                                          nullptr, 0)) {
    // x's 1x128 groups and W's tiles in one launch
    const cudaError_t e = launch_quant_tile_pair(
        QuantTileArgs{kQuantTileRow, (const uint16_t*)x, M, K, K, base + L.qx, L.ldK, (float*)(base + L.sx), L.ldsM,
                      nullptr, 0, nullptr, 0},
        QuantTileArgs{kQuantTileScale, (const uint16_t*)w, N, K, K, base + L.qw, L.ldK, (float*)(base + L.sw), Kb,
                      nullptr, 0, nullptr, 0},
        sms, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "bfp8_linear_fwd quantisation launch");
  } else {
    if ((st = bfp8_quant_lhs(x, M, K, K, 0, base + L.qx, L.ldK, (float*)(base + L.sx), L.ldsM, stream)) != BFP8_OK)
      return st;
    if ((st = bfp8_quant_weight(w, N, K, K, base + L.qw, L.ldK, nullptr, 0, (float*)(base + L.sw), Kb, stream)) !=
        BFP8_OK)
      return st;
  }
  return bfp8_gemm_1x128_128x128(base + L.qx, L.ldK, (const float*)(base + L.sx), L.ldsM, base + L.qw, L.ldK,
                                 (const float*)(base + L.sw), Kb, 0, y, N, M, N, K, stream);
}

extern "C" {

bfp8_status bfp8_linear_bwd(const void* dy, const void* x, const void* w, void* dx, void* dw, int64_t M, int64_t N,
                            int64_t K, void* ws, size_t ws_bytes, bfp8_stream_t stream) {
  bfp8_status st = check_dims("bfp8_linear_bwd", M, N, K);
  if (st != BFP8_OK) return st;
  if (M == 0 || N == 0 || K == 0) {
    cudaError_t e = cudaSuccess;
    if (M > 0 && K > 0 && dx) e = cudaMemsetAsync(dx, 0, (size_t)M * K * 2, (cudaStream_t)stream);
    if (e == cudaSuccess && N > 0 && K > 0 && dw) e = cudaMemsetAsync(dw, 0, (size_t)N * K * 2, (cudaStream_t)stream);
    return e == cudaSuccess ? BFP8_OK : cuda_fail(e, "bfp8_linear_bwd");
  }
  CHECK_ARG(dy && x && w && dx && dw && ws, "bfp8_linear_bwd: null pointer");
  CHECK_ARG((reinterpret_cast<uintptr_t>(ws) & 255u) == 0, "bfp8_linear_bwd: workspace must be 256-byte aligned");
  CHECK_ARG(ws_bytes >= bfp8_linear_workspace_size(M, N, K), "bfp8_linear_bwd: workspace too small (%zu < %zu)",
            ws_bytes, bfp8_linear_workspace_size(M, N, K));
  const BwdLayout L = bwd_layout(M, N, K);
  uint8_t* base = (uint8_t*)ws;
  const int64_t Kb = cdiv(K, kBlock), Nb = cdiv(N, kBlock);
  (void)Nb;
  // dX = dY W : dY 1x128 along N (reduction), W's tiles read transposed.
  if ((st = bfp8_quant_lhs(dy, M, N, N, 0, base + L.qdy, L.ldN, (float*)(base + L.sdy), L.ldsM, stream)) != BFP8_OK)
    return st;
  if ((st = bfp8_quant_weight(w, N, K, K, nullptr, 0, base + L.qwt, L.ldN, (float*)(base + L.sw), Kb, stream)) !=
      BFP8_OK)
    return st;
  if ((st = bfp8_gemm_1x128_128x128(base + L.qdy, L.ldN, (const float*)(base + L.sdy), L.ldsM, base + L.qwt, L.ldN,
                                    (const float*)(base + L.sw), Kb, 1, dx, K, M, K, N, stream)) != BFP8_OK)
    return st;
  // dW = dY^T X : dY^T 1x128 along M, X 128x1 along M (both written K-major).
  if ((st = bfp8_quant_lhs(dy, N, M, N, 1, base + L.qdyt, L.ldM, (float*)(base + L.sdyt), L.ldsN, stream)) !=
      BFP8_OK)
    return st;
  if ((st = bfp8_quant_rhs(x, M, K, K, base + L.qxt, L.ldM, (float*)(base + L.sxt), L.ldsK, stream)) != BFP8_OK)
    return st;
  return bfp8_gemm_1x128_128x1(base + L.qdyt, L.ldM, (const float*)(base + L.sdyt), L.ldsN, base + L.qxt, L.ldM,
                               (const float*)(base + L.sxt), L.ldsK, dw, K, N, K, M, stream);
}

// ---------------------------------------------------------------------------
// Linear layer, training form: the forward keeps what the backward needs
// ---------------------------------------------------------------------------

namespace {
struct TrainLayout {
  size_t qx, sx, qxt, sxt, qw, qwt, sw, qdy, sdy, qdyt, sdyt, total;
  int64_t ldK, ldN, ldM, ldsM, ldsN, ldsK;
};
TrainLayout train_layout(int64_t M, int64_t N, int64_t K) {
  TrainLayout L;
  L.ldK = rup(K, 16);
  L.ldN = rup(N, 16);
  L.ldM = rup(M, 16);
  L.ldsM = rup(M, 4);
  L.ldsN = rup(N, 4);
  L.ldsK = rup(K, 4);
  const int64_t Kb = cdiv(K, kBlock), Nb = cdiv(N, kBlock), Mb = cdiv(M, kBlock);
  size_t o = 0;
  L.qx = o; o = a256(o + (size_t)M * L.ldK);            // x, 1x128 along K (forward lhs)
  L.sx = o; o = a256(o + (size_t)Kb * L.ldsM * 4);
  L.qxt = o; o = a256(o + (size_t)K * L.ldM);           // x, 128x1 along M, transposed (wgrad rhs)
  L.sxt = o; o = a256(o + (size_t)Mb * L.ldsK * 4);
  L.qw = o; o = a256(o + (size_t)N * L.ldK);            // W tiles (forward rhs)
  L.qwt = o; o = a256(o + (size_t)K * L.ldN);           // W tiles transposed (dgrad rhs)
  L.sw = o; o = a256(o + (size_t)Nb * Kb * 4);
  L.qdy = o; o = a256(o + (size_t)M * L.ldN);           // dY, 1x128 along N (dgrad lhs)
  L.sdy = o; o = a256(o + (size_t)Nb * L.ldsM * 4);
  L.qdyt = o; o = a256(o + (size_t)N * L.ldM);          // dY^T, 1x128 along M (wgrad lhs)
  L.sdyt = o; o = a256(o + (size_t)Mb * L.ldsN * 4);
  L.total = o;
  return L;
}
}  // namespace

size_t bfp8_linear_train_workspace_size(int64_t M, int64_t N, int64_t K) {
  if (M <= 0 || N <= 0 || K <= 0) return 0;
  return train_layout(M, N, K).total;
}

bfp8_status bfp8_linear_fwd_train(const void* x, const void* w, void* y, int64_t M, int64_t N, int64_t K, void* ws,
                                  size_t ws_bytes, bfp8_stream_t stream) {
  bfp8_status st = check_dims("bfp8_linear_fwd_train", M, N, K);
  if (st != BFP8_OK) return st;
  CHECK_ARG(M > 0 && N > 0 && K > 0, "bfp8_linear_fwd_train: dimensions must be positive");
  CHECK_ARG(x && w && y && ws, "bfp8_linear_fwd_train: null pointer");
  CHECK_ARG((reinterpret_cast<uintptr_t>(ws) & 255u) == 0, "bfp8_linear_fwd_train: workspace must be 256-byte aligned");
  const TrainLayout L = train_layout(M, N, K);
  CHECK_ARG(ws_bytes >= L.total, "bfp8_linear_fwd_train: workspace too small (%zu < %zu)", ws_bytes, L.total);
  uint8_t* b = (uint8_t*)ws;
  const int64_t Kb = cdiv(K, kBlock);
  // one launch, one read of x and of W: x's 1x128 groups (forward) and 128x1
  // groups along M (weight gradient); W's 128x128 tiles as is (forward) and
  // transposed (input gradient)
  if ((st = bfp8_quant_dual_weight(x, M, K, K, b + L.qx, L.ldK, (float*)(b + L.sx), L.ldsM, b + L.qxt, L.ldM,
                                   (float*)(b + L.sxt), L.ldsK, w, N, K, b + L.qw, L.ldK, b + L.qwt, L.ldN,
                                   (float*)(b + L.sw), Kb, stream)) != BFP8_OK)
    return st;
  return bfp8_gemm_1x128_128x128(b + L.qx, L.ldK, (const float*)(b + L.sx), L.ldsM, b + L.qw, L.ldK,
                                 (const float*)(b + L.sw), Kb, 0, y, N, M, N, K, stream);
}

bfp8_status bfp8_linear_bwd_saved(const void* dy, void* dx, void* dw, int64_t M, int64_t N, int64_t K, void* ws,
                                  size_t ws_bytes, bfp8_stream_t stream) {
  bfp8_status st = check_dims("bfp8_linear_bwd_saved", M, N, K);
  if (st != BFP8_OK) return st;
  CHECK_ARG(M > 0 && N > 0 && K > 0, "bfp8_linear_bwd_saved: dimensions must be positive");
  CHECK_ARG(dy && dx && dw && ws, "bfp8_linear_bwd_saved: null pointer");
  CHECK_ARG((reinterpret_cast<uintptr_t>(ws) & 255u) == 0, "bfp8_linear_bwd_saved: workspace must be 256-byte aligned");
  const TrainLayout L = train_layout(M, N, K);
  CHECK_ARG(ws_bytes >= L.total, "bfp8_linear_bwd_saved: workspace too small (%zu < %zu)", ws_bytes, L.total);
  uint8_t* b = (uint8_t*)ws;
  const int64_t Kb = cdiv(K, kBlock);
  // one read of dY: 1x128 along N (input gradient) and 1x128 along M of dY^T (weight gradient)
  if ((st = bfp8_quant_dual(dy, M, N, N, b + L.qdy, L.ldN, (float*)(b + L.sdy), L.ldsM, b + L.qdyt, L.ldM,
                            (float*)(b + L.sdyt), L.ldsN, stream)) != BFP8_OK)
    return st;
  if ((st = bfp8_gemm_1x128_128x128(b + L.qdy, L.ldN, (const float*)(b + L.sdy), L.ldsM, b + L.qwt, L.ldN,
                                    (const float*)(b + L.sw), Kb, 1, dx, K, M, K, N, stream)) != BFP8_OK)
    return st;
  return bfp8_gemm_1x128_128x1(b + L.qdyt, L.ldM, (const float*)(b + L.sdyt), L.ldsN, b + L.qxt, L.ldM,
                               (const float*)(b + L.sxt), L.ldsK, dw, K, N, K, M, stream);
}

// ---------------------------------------------------------------------------
// One training step from host memory, copies overlapped with the kernels
// ---------------------------------------------------------------------------

namespace {
struct HostStepLayout {
  size_t x, w, dy, y, dx, dw, train, total;
};
HostStepLayout host_step_layout(int64_t M, int64_t N, int64_t K) {
  HostStepLayout H;
  size_t o = 0;
  H.x = o; o = a256(o + (size_t)M * K * 2);
  H.w = o; o = a256(o + (size_t)N * K * 2);
  H.dy = o; o = a256(o + (size_t)M * N * 2);
  H.y = o; o = a256(o + (size_t)M * N * 2);
  H.dx = o; o = a256(o + (size_t)M * K * 2);
  H.dw = o; o = a256(o + (size_t)N * K * 2);
  H.train = o; o += train_layout(M, N, K).total;
  H.total = o;
  return H;
}

constexpr int kMaxStepChunks = 64;
constexpr int kMaxDgradPieces = 4;

// Columns of W / dY per pipeline chunk when the caller passes 0: about an
// eighth of N, at least 1024 (2-D copies of narrower column chunks move
// slower, device to host most of all), a multiple of 128 (one weight tile row).
int64_t step_chunk_n(int64_t N) { return rup(cdiv(N, 8) > 1024 ? cdiv(N, 8) : 1024, kBlock); }

// The copy streams and events of the host step on one device: created on the
// first call, kept for the life of the process.  Calls on one device enqueue
// under the mutex; a wait binds to the event's latest record at enqueue time,
// so reusing the events across calls is safe.
struct HostStepCtx {
  std::mutex mu;
  bool ready = false;
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start, x_in, in_end, out_end;
  cudaEvent_t chunk_in[kMaxStepChunks], y_done[kMaxStepChunks], dw_done[kMaxStepChunks];
  cudaEvent_t dx_done[kMaxDgradPieces];
  cudaEvent_t slot_free[2];  // per-expert steps: a device slot's last copy out
};
HostStepCtx g_step[64];

cudaError_t host_step_init(HostStepCtx& C) {
  if (C.ready) return cudaSuccess;
  cudaError_t e;
  if ((e = cudaStreamCreateWithFlags(&C.in, cudaStreamNonBlocking)) != cudaSuccess) return e;
  if ((e = cudaStreamCreateWithFlags(&C.out, cudaStreamNonBlocking)) != cudaSuccess) return e;
  std::vector<cudaEvent_t*> evs = {&C.start, &C.x_in, &C.in_end, &C.out_end};
  for (int i = 0; i < kMaxStepChunks; ++i) {
    evs.push_back(&C.chunk_in[i]);
    evs.push_back(&C.y_done[i]);
    evs.push_back(&C.dw_done[i]);
  }
  for (int i = 0; i < kMaxDgradPieces; ++i) evs.push_back(&C.dx_done[i]);
  evs.push_back(&C.slot_free[0]);
  evs.push_back(&C.slot_free[1]);
  for (cudaEvent_t* ev : evs)
    if ((e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming)) != cudaSuccess) return e;
  C.ready = true;
  return cudaSuccess;
}
}  // namespace

namespace {
// Enqueues one step (copies on C.in / C.out, kernels on s) into the device
// buffers at `base` (host_step_layout(M, N, K)).  The caller records the start
// and joins the streams afterwards, whatever this returns.
bfp8_status host_step_enqueue(HostStepCtx& C, cudaStream_t s, bfp8_stream_t stream, const void* x, const void* w,
                              const void* dy, void* y, void* dx, void* dw, int64_t M, int64_t N, int64_t K,
                              int64_t Nc, uint8_t* base) {
  bfp8_status st = BFP8_OK;
  const HostStepLayout H = host_step_layout(M, N, K);
  const int64_t nc = cdiv(N, Nc);
  uint16_t *d_x = (uint16_t*)(base + H.x), *d_w = (uint16_t*)(base + H.w), *d_dy = (uint16_t*)(base + H.dy);
  uint16_t *d_y = (uint16_t*)(base + H.y), *d_dx = (uint16_t*)(base + H.dx), *d_dw = (uint16_t*)(base + H.dw);
  const TrainLayout L = train_layout(M, N, K);
  uint8_t* b = base + H.train;
  const int64_t Kb = cdiv(K, kBlock);
  const size_t row_x = (size_t)K * 2, row_y = (size_t)N * 2;
  const char* h_x = (const char*)x;
  const char* h_w = (const char*)w;
  const char* h_dy = (const char*)dy;

  // Enqueue everything, stopping at the first failure; the caller's stream
  // then waits on both copy streams either way, so later work stays ordered.
  cudaError_t ce = cudaSuccess;
  const char* what = nullptr;
  auto cu = [&](cudaError_t r, const char* w_) {
    if (ce == cudaSuccess && r != cudaSuccess) {
      ce = r;
      what = w_;
    }
    return ce == cudaSuccess;
  };
  auto ok = [&](bfp8_status r) {
    if (st == BFP8_OK) st = r;
    return st == BFP8_OK;
  };

  bool go = true;
  // inputs, in the order the kernels need them: x, then W and dY chunk by chunk
  go = go && cu(cudaMemcpyAsync(d_x, h_x, (size_t)M * row_x, cudaMemcpyDefault, C.in), "copy x in") &&
       cu(cudaEventRecord(C.x_in, C.in), "event record");
  for (int64_t j = 0; go && j < nc; ++j) {
    const int64_t n0 = j * Nc, nj = (N - n0 < Nc) ? N - n0 : Nc;
    go = cu(cudaMemcpyAsync((char*)d_w + n0 * row_x, h_w + n0 * row_x, (size_t)nj * row_x, cudaMemcpyDefault, C.in),
            "copy W in") &&
         cu(cudaMemcpy2DAsync((char*)d_dy + n0 * 2, row_y, h_dy + n0 * 2, row_y, (size_t)nj * 2, (size_t)M,
                              cudaMemcpyDefault, C.in),
            "copy dY in") &&
         cu(cudaEventRecord(C.chunk_in[j], C.in), "event record");
  }

  // x in both forms: 1x128 along K (forward lhs), 128x1 along M (weight-gradient rhs)
  go = go && cu(cudaStreamWaitEvent(s, C.x_in, 0), "wait") &&
       ok(bfp8_quant_dual(d_x, M, K, K, b + L.qx, L.ldK, (float*)(b + L.sx), L.ldsM, b + L.qxt, L.ldM,
                          (float*)(b + L.sxt), L.ldsK, stream));
  for (int64_t j = 0; go && j < nc; ++j) {
    const int64_t n0 = j * Nc, nj = (N - n0 < Nc) ? N - n0 : Nc, nb0 = n0 / kBlock;
    go = cu(cudaStreamWaitEvent(s, C.chunk_in[j], 0), "wait") &&
         // W rows n0..n0+nj: tiles as is and transposed, tile scales at tile row nb0
         ok(bfp8_quant_weight(d_w + n0 * K, nj, K, K, b + L.qw + n0 * L.ldK, L.ldK, b + L.qwt + n0, L.ldN,
                              (float*)(b + L.sw) + nb0 * Kb, Kb, stream)) &&
         // y[:, n0..n0+nj] = x W_j^T
         ok(bfp8_gemm_1x128_128x128(b + L.qx, L.ldK, (const float*)(b + L.sx), L.ldsM, b + L.qw + n0 * L.ldK,
                                    L.ldK, (const float*)(b + L.sw) + nb0 * Kb, Kb, 0, d_y + n0, N, M, nj, K,
                                    stream)) &&
         cu(cudaEventRecord(C.y_done[j], s), "event record") && cu(cudaStreamWaitEvent(C.out, C.y_done[j], 0), "wait") &&
         cu(cudaMemcpy2DAsync((char*)y + n0 * 2, row_y, (const char*)d_y + n0 * 2, row_y, (size_t)nj * 2, (size_t)M,
                              cudaMemcpyDefault, C.out),
            "copy y out") &&
         // dY[:, n0..n0+nj] in both forms: 1x128 along N (input-gradient lhs), along M of dY^T (weight-gradient lhs)
         ok(bfp8_quant_dual(d_dy + n0, M, nj, N, b + L.qdy + n0, L.ldN, (float*)(b + L.sdy) + nb0 * L.ldsM, L.ldsM,
                            b + L.qdyt + n0 * L.ldM, L.ldM, (float*)(b + L.sdyt) + n0, L.ldsN, stream)) &&
         // dW[n0..n0+nj, :] = dY_j^T x
         ok(bfp8_gemm_1x128_128x1(b + L.qdyt + n0 * L.ldM, L.ldM, (const float*)(b + L.sdyt) + n0, L.ldsN,
                                  b + L.qxt, L.ldM, (const float*)(b + L.sxt), L.ldsK, d_dw + n0 * K, K, nj, K, M,
                                  stream)) &&
         cu(cudaEventRecord(C.dw_done[j], s), "event record") &&
         cu(cudaStreamWaitEvent(C.out, C.dw_done[j], 0), "wait") &&
         cu(cudaMemcpyAsync((char*)dw + n0 * row_x, (const char*)d_dw + n0 * row_x, (size_t)nj * row_x,
                            cudaMemcpyDefault, C.out),
            "copy dW out");
  }
  // dX = dY W, needing every chunk, in row pieces so that the first pieces
  // leave while the last ones run
  const int np = M >= 1024 ? kMaxDgradPieces : (M >= 512 ? 2 : 1);
  const int64_t Mp = rup(cdiv(M, np), kBlock);
  for (int p = 0; go && p < np && p * Mp < M; ++p) {
    const int64_t m0 = p * Mp, mp = (M - m0 < Mp) ? M - m0 : Mp;
    go = ok(bfp8_gemm_1x128_128x128(b + L.qdy + m0 * L.ldN, L.ldN, (const float*)(b + L.sdy) + m0, L.ldsM,
                                    b + L.qwt, L.ldN, (const float*)(b + L.sw), Kb, 1, d_dx + m0 * K, K, mp, K, N,
                                    stream)) &&
         cu(cudaEventRecord(C.dx_done[p], s), "event record") &&
         cu(cudaStreamWaitEvent(C.out, C.dx_done[p], 0), "wait") &&
         cu(cudaMemcpyAsync((char*)dx + m0 * row_x, (const char*)d_dx + m0 * row_x, (size_t)mp * row_x,
                            cudaMemcpyDefault, C.out),
            "copy dX out");
  }
  if (st != BFP8_OK) return st;
  if (ce != cudaSuccess) return cuda_fail(ce, what);
  return BFP8_OK;
}

// Records the step's start on the caller's stream for both copy streams.
cudaError_t host_step_start(HostStepCtx& C, cudaStream_t s) {
  cudaError_t e = cudaEventRecord(C.start, s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(C.in, C.start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(C.out, C.start, 0);
  return e;
}

// The caller's stream continues after every copy of the step.
cudaError_t host_step_join(HostStepCtx& C, cudaStream_t s) {
  cudaEventRecord(C.in_end, C.in);
  cudaEventRecord(C.out_end, C.out);
  cudaStreamWaitEvent(s, C.in_end, 0);
  return cudaStreamWaitEvent(s, C.out_end, 0);
}
}  // namespace

size_t bfp8_linear_step_host_workspace_size(int64_t M, int64_t N, int64_t K) {
  if (M <= 0 || N <= 0 || K <= 0) return 0;
  return host_step_layout(M, N, K).total;
}

bfp8_status bfp8_linear_step_host(const void* x, const void* w, const void* dy, void* y, void* dx, void* dw,
                                  int64_t M, int64_t N, int64_t K, int64_t chunk_n, void* ws, size_t ws_bytes,
                                  bfp8_stream_t stream) {
  const char* fn = "bfp8_linear_step_host";
  bfp8_status st = check_dims(fn, M, N, K);
  if (st != BFP8_OK) return st;
  CHECK_ARG(M > 0 && N > 0 && K > 0, "%s: dimensions must be positive", fn);
  CHECK_ARG(x && w && dy && y && dx && dw && ws, "%s: null pointer", fn);
  CHECK_ARG((reinterpret_cast<uintptr_t>(ws) & 255u) == 0, "%s: workspace must be 256-byte aligned", fn);
  CHECK_ARG(chunk_n >= 0 && chunk_n % kBlock == 0, "%s: chunk_n=%lld must be 0 (automatic) or a multiple of 128", fn,
            (long long)chunk_n);
  const HostStepLayout H = host_step_layout(M, N, K);
  CHECK_ARG(ws_bytes >= H.total, "%s: workspace too small (%zu < %zu)", fn, ws_bytes, H.total);
  const int64_t Nc = chunk_n ? chunk_n : step_chunk_n(N);
  const int64_t nc = cdiv(N, Nc);
  CHECK_ARG(nc <= kMaxStepChunks, "%s: %lld chunks of %lld columns exceed %d; pass a larger chunk_n", fn,
            (long long)nc, (long long)Nc, kMaxStepChunks);
  int sms = 0, dev = 0;
  if ((st = check_device(&sms)) != BFP8_OK) return st;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  HostStepCtx& C = g_step[dev];
  std::lock_guard<std::mutex> lk(C.mu);
  if ((e = host_step_init(C)) != cudaSuccess) return cuda_fail(e, "bfp8_linear_step_host: stream/event creation");

  const cudaStream_t s = (cudaStream_t)stream;
  if ((e = host_step_start(C, s)) != cudaSuccess) return cuda_fail(e, "bfp8_linear_step_host: start");
  st = host_step_enqueue(C, s, stream, x, w, dy, y, dx, dw, M, N, K, Nc, (uint8_t*)ws);
  const cudaError_t je = host_step_join(C, s);
  if (st != BFP8_OK) return st;
  return je == cudaSuccess ? BFP8_OK : cuda_fail(je, "bfp8_linear_step_host: join");
}

size_t bfp8_moe_step_host_workspace_size(int64_t M_max, int64_t N, int64_t K) {
  if (N <= 0 || K <= 0 || M_max < 0) return 0;
  return 2 * a256(host_step_layout(M_max > 0 ? M_max : 1, N, K).total);
}

bfp8_status bfp8_moe_step_host(const void* x, const void* w, const void* dy, const int32_t* offs, int64_t E,
                               void* y, void* dx, void* dw, int64_t T, int64_t N, int64_t K, int64_t chunk_n,
                               void* ws, size_t ws_bytes, bfp8_stream_t stream) {
  const char* fn = "bfp8_moe_step_host";
  bfp8_status st = check_dims(fn, T, N, K);
  if (st != BFP8_OK) return st;
  CHECK_ARG(N > 0 && K > 0, "%s: N and K must be positive", fn);
  CHECK_ARG(E >= 1 && E <= 4096, "%s: E=%lld experts out of [1, 4096]", fn, (long long)E);
  CHECK_ARG(offs, "%s: null offsets", fn);
  CHECK_ARG(offs[0] >= 0 && offs[E] <= T, "%s: offsets must lie in [0, T=%lld]", fn, (long long)T);
  int64_t M_max = 0;
  for (int64_t e = 0; e < E; ++e) {
    CHECK_ARG(offs[e + 1] >= offs[e], "%s: offsets decrease at expert %lld", fn, (long long)e);
    if (offs[e + 1] - offs[e] > M_max) M_max = offs[e + 1] - offs[e];
  }
  CHECK_ARG(w && dw && ws, "%s: null pointer", fn);
  CHECK_ARG(M_max == 0 || (x && dy && y && dx), "%s: null pointer", fn);
  CHECK_ARG((reinterpret_cast<uintptr_t>(ws) & 255u) == 0, "%s: workspace must be 256-byte aligned", fn);
  CHECK_ARG(chunk_n >= 0 && chunk_n % kBlock == 0, "%s: chunk_n=%lld must be 0 (automatic) or a multiple of 128", fn,
            (long long)chunk_n);
  const size_t slot = a256(host_step_layout(M_max > 0 ? M_max : 1, N, K).total);
  CHECK_ARG(ws_bytes >= 2 * slot, "%s: workspace too small (%zu < %zu)", fn, ws_bytes, 2 * slot);
  const int64_t Nc = chunk_n ? chunk_n : step_chunk_n(N);
  CHECK_ARG(cdiv(N, Nc) <= kMaxStepChunks, "%s: %lld chunks of %lld columns exceed %d; pass a larger chunk_n", fn,
            (long long)cdiv(N, Nc), (long long)Nc, kMaxStepChunks);
  int sms = 0, dev = 0;
  if ((st = check_device(&sms)) != BFP8_OK) return st;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  HostStepCtx& C = g_step[dev];
  std::lock_guard<std::mutex> lk(C.mu);
  if ((e = host_step_init(C)) != cudaSuccess) return cuda_fail(e, "bfp8_moe_step_host: stream/event creation");

  const cudaStream_t s = (cudaStream_t)stream;
  if ((e = host_step_start(C, s)) != cudaSuccess) return cuda_fail(e, "bfp8_moe_step_host: start");
  uint8_t* base = (uint8_t*)ws;
  const size_t wbytes = (size_t)N * K * 2;
  // Each expert with tokens is one dense step on its rows, in two device
  // slots used in turn: expert k's inputs enter slot k % 2 once expert k-2's
  // outputs have left it, so copies of one expert overlap kernels of another.
  int64_t k = 0;
  for (int64_t ex = 0; st == BFP8_OK && ex < E; ++ex) {
    const int64_t m0 = offs[ex], Me = offs[ex + 1] - offs[ex];
    if (Me == 0) continue;
    const int sl = (int)(k & 1);
    if (k >= 2 && (e = cudaStreamWaitEvent(C.in, C.slot_free[sl], 0)) != cudaSuccess) {
      st = cuda_fail(e, "bfp8_moe_step_host: wait");
      break;
    }
    st = host_step_enqueue(C, s, stream, (const char*)x + m0 * K * 2, (const char*)w + ex * wbytes,
                           (const char*)dy + m0 * N * 2, (char*)y + m0 * N * 2, (char*)dx + m0 * K * 2,
                           (char*)dw + ex * wbytes, Me, N, K, Nc, base + sl * slot);
    if (st == BFP8_OK && (e = cudaEventRecord(C.slot_free[sl], C.out)) != cudaSuccess)
      st = cuda_fail(e, "bfp8_moe_step_host: event record");
    ++k;
  }
  // experts without tokens: dW = 0, copied out of a zeroed device region
  // (slot 0's weight-gradient buffer, after every earlier copy out of it)
  bool zeroed = false;
  for (int64_t ex = 0; st == BFP8_OK && ex < E; ++ex) {
    if (offs[ex + 1] != offs[ex]) continue;
    const HostStepLayout H = host_step_layout(M_max > 0 ? M_max : 1, N, K);
    uint8_t* zero = base + H.dw;
    if (!zeroed && (e = cudaMemsetAsync(zero, 0, wbytes, C.out)) != cudaSuccess) {
      st = cuda_fail(e, "bfp8_moe_step_host: memset");
      break;
    }
    zeroed = true;
    if ((e = cudaMemcpyAsync((char*)dw + ex * wbytes, zero, wbytes, cudaMemcpyDefault, C.out)) != cudaSuccess)
      st = cuda_fail(e, "bfp8_moe_step_host: copy dW out");
  }
  const cudaError_t je = host_step_join(C, s);
  if (st != BFP8_OK) return st;
  return je == cudaSuccess ? BFP8_OK : cuda_fail(je, "bfp8_moe_step_host: join");
}

// ---------------------------------------------------------------------------
// Host replay of the kernels' index arithmetic
// ---------------------------------------------------------------------------

namespace {
// Replays the stores of the TMA-staged tile kernel over a [T, C] input.
// rows_out: q_row [T, C]; cols_out: q_col [C, T]; scale_kind: 0 none,
// 1 row scales [Cb, T], 2 column scales [Tb, C], 3 tile scales [Tb, Cb].
void replay_tile(int64_t T, int64_t C, bool rows_out, bool cols_out, int scale_kind, uint32_t* counts,
                 uint32_t* scounts, int64_t* oob, int sms) {
  // scale_kind: 0 none, 1 row scales s_row[c/128][t], 2 column scales
  // s_col[t/128][c], 3 tile scales s_row[t/128][c/128]
  auto hit = [&](uint32_t* arr, int64_t r, int64_t c, int64_t rows, int64_t cols) {
    if (r < 0 || r >= rows || c < 0 || c >= cols) {
      ++*oob;
      return;
    }
    if (arr) arr[r * cols + c]++;
  };
  const int64_t tiles_c = cdiv(C, 128), num_tiles = cdiv(T, 128) * tiles_c;
  const int64_t grid = qt_grid(num_tiles, sms), Tb = cdiv(T, 128), Cb = cdiv(C, 128);
  for (int64_t cta = 0; cta < grid; ++cta)
    for (int64_t tile = cta; tile < num_tiles; tile += grid) {
      const int64_t t0 = qt_tile_t0(tile, tiles_c), c0 = qt_tile_c0(tile, tiles_c);
      // TMA stores: one 128 x 128 box per output, clipped to the 16-byte-
      // aligned extent of the inner dimension (C_al for q_row, T_al for q_col)
      const int64_t C_al = C & ~(int64_t)15, T_al = T & ~(int64_t)15;
      if (rows_out && c0 < C_al)
        for (int64_t t = t0; t < t0 + 128 && t < T; ++t)
          for (int64_t c = c0; c < c0 + 128 && c < C_al; ++c) hit(counts, t, c, T, C);
      if (cols_out && t0 < T_al)
        for (int64_t c = c0; c < c0 + 128 && c < C; ++c)
          for (int64_t t = t0; t < t0 + 128 && t < T_al; ++t) hit(counts, c, t, C, T);
      for (int tid = 0; tid < kQtThreads; ++tid) {
        // the ragged bytes past the aligned extents, stored by the threads
        const int gr = qt_scale_group(tid), b0 = 4 * (tid & 3);
        for (int b = 0; b < 4; ++b) {
          if (rows_out && c0 + 128 > C_al && C_al < C && t0 + gr < T && C_al + b0 + b < C)
            hit(counts, t0 + gr, C_al + b0 + b, T, C);
          if (cols_out && t0 + 128 > T_al && T_al < T && c0 + gr < C && T_al + b0 + b < T)
            hit(counts, c0 + gr, T_al + b0 + b, C, T);
        }
        if (!qt_scale_writer(tid)) continue;
        const int g = qt_scale_group(tid);
        if (scale_kind == 1 && t0 + g < T) hit(scounts, c0 / 128, t0 + g, Cb, T);
        if (scale_kind == 2 && c0 + g < C) hit(scounts, t0 / 128, c0 + g, Tb, C);
      }
      if (scale_kind == 3) hit(scounts, t0 / 128, c0 / 128, Tb, Cb);
    }
}
}  // namespace

int bfp8_debug_launch_pdl(int kind, int64_t a, int64_t b, int64_t c) {
  if (a < 0 || b < 0 || c < 0) return -1;
  if (kind == 0) return pdl_for_gemm(a, b, c) ? 1 : 0;
  if (kind == 1) return pdl_for_quant(a) ? 1 : 0;
  return -1;
}

int bfp8_debug_gemm_pick_bn(int64_t M, int64_t N, int col_scales, int num_sms) {
  if (M <= 0 || N <= 0 || num_sms <= 0) return 0;
  return gemm_pick_bn(M, N, col_scales != 0, num_sms);
}

bfp8_status bfp8_debug_write_counts(int kind, int64_t M, int64_t N, int64_t K, int flag, uint32_t* counts,
                                    uint32_t* scale_counts, int64_t* oob) {
  CHECK_ARG(counts && oob, "bfp8_debug_write_counts: null pointer");
  CHECK_ARG(M >= 0 && N >= 0 && K >= 0, "bfp8_debug_write_counts: negative size");
  const int sms = 152;  // GB300
  *oob = 0;
  const bool plain = (flag & 2) != 0;  // replay the untiled fallback kernels instead of the TMA-staged one
  if (!plain) {
    switch (kind) {
      case 0:
        if (flag & 1) replay_tile(K, M, false, true, 2, counts, scale_counts, oob, sms);   // x is [K, M]
        else replay_tile(M, K, true, false, 1, counts, scale_counts, oob, sms);
        return BFP8_OK;
      case 1: replay_tile(K, N, false, true, 2, counts, scale_counts, oob, sms); return BFP8_OK;
      case 2: replay_tile(N, K, true, false, 3, counts, scale_counts, oob, sms); return BFP8_OK;
      case 4: replay_tile(N, K, false, true, 0, counts, nullptr, oob, sms); return BFP8_OK;
      case 5: replay_tile(M, K, true, false, 1, counts, scale_counts, oob, sms); return BFP8_OK;
      case 6: replay_tile(M, K, false, true, 2, counts, scale_counts, oob, sms); return BFP8_OK;
      default: break;
    }
  }
  auto hit = [&](uint32_t* arr, int64_t r, int64_t c, int64_t rows, int64_t cols) {
    if (r < 0 || r >= rows || c < 0 || c >= cols) {
      ++*oob;
      return;
    }
    if (arr) arr[r * cols + c]++;
  };
  if (kind == 0 && !(flag & 1)) {  // quant_lhs, row-major input [M,K]
    const int64_t Kb = cdiv(K, kBlock), groups = M * Kb;
    if (groups == 0) return BFP8_OK;
    const int64_t grid = quant_rows_grid(M, K, sms);
    const int64_t nhw = grid * (kRowThreads / 16);
    const int64_t iters = cdiv(groups, nhw * kRowUnroll);
    for (int64_t hw = 0; hw < nhw; ++hw)
      for (int64_t it = 0; it < iters; ++it)
        for (int u = 0; u < kRowUnroll; ++u) {
          const int64_t g = row_group(hw, nhw, it, u);
          if (g >= groups) continue;
          for (int l16 = 0; l16 < 16; ++l16) {
            const RowChunk c = row_chunk(g, l16, Kb);
            for (int b = 0; b < 8; ++b)
              if (c.k + b < K) hit(counts, c.m, c.k + b, M, K);
            if (l16 == 0) hit(scale_counts, c.k / kBlock, c.m, Kb, M);
          }
        }
    return BFP8_OK;
  }
  if ((kind == 0 && (flag & 1)) || kind == 1) {  // transposed-read groups: T = grouped dim, C = columns
    // kind 0 (x is [K,M]): T = K, C = M, logical q [M,K].  kind 1 (x is [K,N]): T = K, C = N, qT [N,K].
    const int64_t T = K, C = (kind == 0) ? M : N;
    const int64_t grid = cdiv(T, kColTileT) * cdiv(C, kColTileC);
    for (int64_t blk = 0; blk < grid; ++blk) {
      const ColTile tile = col_tile(blk, C);
      for (int ch = 0; ch < kColTileC * kColTileT / 16; ++ch) {
        const int64_t c = col_store_c(tile, ch), t = col_store_t(tile, ch);
        if (c < C)
          for (int b = 0; b < 16; ++b)
            if (t + b < T) hit(counts, c, t + b, C, T);
      }
      for (int warp = 0; warp < kColThreads / 32; ++warp)
        for (int j = 0; j < 8; ++j) {
          const int64_t c = col_elem_c(tile, warp, j);
          if (c < C) hit(scale_counts, tile.t0 / kBlock, c, cdiv(T, kBlock), C);
        }
    }
    return BFP8_OK;
  }
  if (kind == 2 || kind == 4) {  // quant_weight: q (kind 2) or qt (kind 4)
    const int64_t Kb = cdiv(K, kBlock), grid = cdiv(N, kBlock) * Kb;
    for (int64_t blk = 0; blk < grid; ++blk) {
      const WTile tile = w_tile(blk, Kb);
      if (kind == 2) {
        for (int warp = 0; warp < kWThreads / 32; ++warp)
          for (int cc = 0; cc < 2; ++cc)
            for (int lane = 0; lane < 32; ++lane)
              for (int i = 0; i < 4; ++i) {
                const int64_t n = w_elem_n(tile, lane, i), k = w_elem_k(tile, warp + 8 * cc, 0);
                if (n < N)
                  for (int b = 0; b < 8; ++b)
                    if (k + b < K) hit(counts, n, k + b, N, K);
              }
        hit(scale_counts, tile.nb, tile.kb, cdiv(N, kBlock), Kb);
      } else {
        for (int ch = 0; ch < kBlock * kBlock / 16; ++ch) {
          const int64_t k = w_tstore_k(tile, ch), n = w_tstore_n(tile, ch);
          if (k < K)
            for (int b = 0; b < 16; ++b)
              if (n + b < N) hit(counts, k, n + b, K, N);
        }
      }
    }
    return BFP8_OK;
  }
  if (kind == 3) {  // GEMM output C [M,N]; flag bit 3: the 1x128 x 128x1 GEMM
    if (smallm_eligible(M, N, (flag & 8) != 0, sms)) {
      // small-M kernel: the leader CTA of tile t, thread nl, stores column 128t + nl of every row
      for (int64_t t = 0; t < cdiv(N, kBM); ++t)
        for (int nl = 0; nl < kBM; ++nl) {
          const int64_t n = t * kBM + nl;
          if (n >= N) continue;
          for (int m = 0; m < 16; ++m)
            if (m < M) hit(counts, m, n, M, N);
        }
      return BFP8_OK;
    }
    const int bn = gemm_pick_bn(M, N, (flag & 8) != 0, sms);
    const int ew = gemm_epi_warps((flag & 8) != 0, bn);
    const int num_m = (int)cdiv(M, kBM), num_n = (int)cdiv(N, bn), tiles = num_m * num_n;
    const int grid = (int)gemm_grid(M, N, bn, sms);
    for (int cta = 0; cta < grid; ++cta)
      for (int tile = cta; tile < tiles; tile += grid) {
        const GemmTile g = gemm_tile(tile, num_m, num_n, bn);
        const int G = epi_group(bn, ew);
        for (int e = 0; e < ew; ++e)
          for (int lane = 0; lane < 32 && (gemm_a_rows(M, bn) == kBM || e % 4 == 0); ++lane)
            for (int sg = 0; sg < epi_passes(bn, ew); ++sg)
              for (int i = 0; i < G && G * sg + lane % G < epi_chunks(bn, ew); ++i) {
                const int64_t m = g.m0 + epi_store_row(e, lane, i, G);
                const int64_t n0 = g.n0 + epi_store_col(e, lane, sg, G, bn, ew);
                if (m >= M) continue;
                for (int b = 0; b < 8; ++b)
                  if (n0 + b < N) hit(counts, m, n0 + b, M, N);
              }
      }
    return BFP8_OK;
  }
  return fail(BFP8_ERR_INVALID_ARG, "bfp8_debug_write_counts: unknown kind %d", kind);
}

}  // extern "C"
