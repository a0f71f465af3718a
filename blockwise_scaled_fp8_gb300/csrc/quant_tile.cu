// TMA-staged blockwise e4m3 quantisation of 128x128 bf16 tiles.
//
// One kernel serves every quantisation of the method ("Enable blockwise FP8
// dense training kernels on ROCm": act_quant_lhs 1x128, act_quant_rhs 128x1,
// weight_quant_rhs 128x128; s = amax/448, q = RNE_e4m3(clamp(x/s, +-448))),
// and can produce two of them from a single read of the input:
//   kTileRow   1x128 groups along the contiguous dim C:
//              q_row[t*ldq_row + c], s_row[(c/128)*lds_row + t]
//   kTileCol   128x1 groups along the row dim T, written transposed:
//              q_col[c*ldq_col + t], s_col[(t/128)*lds_col + c]
//   kTileScale one scale per 128x128 tile: q_row and/or q_col (either may
//              be null), s_row[(t/128)*lds_row + c/128]
// The input [T, C] (row stride ldx) is read by TMA as two 64-column boxes per
// tile with 128-byte swizzling into a two-stage ring per CTA; persistent CTAs
// (two per SM) walk the tiles, so the next tile's load overlaps this tile's
// arithmetic.  Rows / columns outside [T, C] arrive as zeros (TMA fill) and
// every store is masked to the logical tensor.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace bfp8 {

static __device__ uint32_t g_quant_error;

namespace {

constexpr int kTileRow = kQuantTileRow, kTileCol = kQuantTileCol, kTileScale = kQuantTileScale;
constexpr int kQtBoxBytes = 128 * 128;               // 64 bf16 columns x 128 rows
constexpr int kQtStageBytes = 2 * kQtBoxBytes;       // one 128x128 bf16 tile
constexpr int kQtOffTout = 2 * kQtStageBytes;        // transposed byte tile, 128 x 128
constexpr int kQtOffBar = kQtOffTout + 128 * 128;
constexpr int kQtSmemBytes = kQtOffBar + 64 + 4 * (kQtThreads / 32) + 1024;  // + alignment slack

struct TileQuantParams {
  int64_t T, C;
  uint8_t* q_row;
  int64_t ldq_row;
  float* s_row;
  int64_t lds_row;
  uint8_t* q_col;
  int64_t ldq_col;
  float* s_col;
  int64_t lds_col;
  int64_t tiles_c, num_tiles;
  uint64_t wait_limit_ns;
};

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

// 16-byte chunk `chunk` (0..15, 8 columns each) of tile row `r` in a stage
// written by two 64-column TMA boxes with 128-byte swizzling.
__device__ __forceinline__ uint32_t tile_chunk_addr(uint32_t stage, int r, int chunk) {
  return stage + (uint32_t)((chunk >> 3) * kQtBoxBytes + r * 128 + (((chunk & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint32_t absmax2(uint32_t acc, uint32_t w) { return __vmaxu2(acc, w & 0x7FFF7FFFu); }

__device__ __forceinline__ uint32_t word_of(const uint4& v, int q) {
  return q == 0 ? v.x : q == 1 ? v.y : q == 2 ? v.z : v.w;
}

// x/s for the two bf16 values of `w` (Markstein-corrected product, as
// quotient()), on packed fp32x2 lanes; returns the two e4m3 bytes.  The
// sign of a zero result may come out positive; sign_bytes() restores it.
__device__ __forceinline__ uint32_t quant2(uint32_t w, uint64_t ns2, uint64_t y2) {
  const uint64_t x2 = f2_pack(bf16_lo(w), bf16_hi(w));
  const uint64_t q0 = f2_mul(x2, y2);
  const uint64_t r0 = f2_fma(ns2, q0, x2);
  const uint64_t q1 = f2_fma(r0, y2, q0);
  const uint64_t r1 = f2_fma(ns2, q1, x2);
  const uint64_t q2 = f2_fma(r1, y2, q1);
  return cvt_e4m3x2(__uint_as_float((uint32_t)q2), __uint_as_float((uint32_t)(q2 >> 32)));
}

// The four e4m3 sign bits of the bf16 values in words a (values 0, 1) and b
// (values 2, 3), placed at bit 7 of bytes 0..3: x/s keeps the sign of x, so
// ORing these into the codes fixes zero codes and leaves the others as they are.
__device__ __forceinline__ uint32_t sign_bytes(uint32_t a, uint32_t b) {
  return __byte_perm(a, b, 0x7531) & 0x80808080u;
}

// eight values (one 16-byte chunk) -> eight bytes, as two words
__device__ __forceinline__ uint2 quant8(const uint4& v, float sc, float rc) {
  const uint64_t ns2 = f2_pack(-sc, -sc), y2 = f2_pack(rc, rc);
  uint2 o;
  o.x = (quant2(v.x, ns2, y2) | (quant2(v.y, ns2, y2) << 16)) | sign_bytes(v.x, v.y);
  o.y = (quant2(v.z, ns2, y2) | (quant2(v.w, ns2, y2) << 16)) | sign_bytes(v.z, v.w);
  return o;
}

}  // namespace

template <int MODE>
__global__ void __launch_bounds__(kQtThreads, 2)
    quant_tile_kernel(const __grid_constant__ CUtensorMap tmap, const TileQuantParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t tout = sbase + kQtOffTout;
  const uint32_t bar0 = sbase + kQtOffBar;
  volatile int* never = reinterpret_cast<volatile int*>(smem + kQtOffBar + 16);
  float* red = reinterpret_cast<float*>(smem + kQtOffBar + 64);  // one partial per warp
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    mbar_init(bar0, 1);
    mbar_init(bar0 + 8, 1);
    *never = 0;
    fence_barrier_init();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tma_prefetch_desc(&tmap);
  }
  __syncthreads();

  auto issue = [&](int64_t tile, int s) {
    const int32_t t0 = (int32_t)qt_tile_t0(tile, p.tiles_c), c0 = (int32_t)qt_tile_c0(tile, p.tiles_c);
    const uint32_t st = sbase + (uint32_t)(s * kQtStageBytes);
    mbar_arrive_expect_tx(bar0 + 8u * s, (uint32_t)kQtStageBytes);
    tma_load_2d(st, &tmap, bar0 + 8u * s, c0, t0);
    tma_load_2d(st + kQtBoxBytes, &tmap, bar0 + 8u * s, c0 + 64, t0);
  };
  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      const int64_t tile = blockIdx.x + (int64_t)s * gridDim.x;
      if (tile < p.num_tiles) issue(tile, s);
    }
  }

  int it = 0;
  for (int64_t tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++it) {
    const int s = it & 1;
    const uint32_t stage = sbase + (uint32_t)(s * kQtStageBytes);
    const bool ok = mbar_wait_bounded(bar0 + 8u * s, (uint32_t)((it >> 1) & 1), p.wait_limit_ns, never);
    if (!__syncthreads_and(ok)) {
      if (tid == 0) {
        atomicOr(&g_quant_error, 1u);
        // the other stage's copy (if issued) must land before the CTA exits
        if (tile + gridDim.x < p.num_tiles)
          mbar_wait_bounded(bar0 + 8u * (s ^ 1), (uint32_t)(((it + 1) >> 1) & 1), p.wait_limit_ns, never);
      }
      break;
    }
    const int64_t t0 = qt_tile_t0(tile, p.tiles_c), c0 = qt_tile_c0(tile, p.tiles_c);
    float tile_sc = 0.0f, tile_rc = 0.0f;

    // ------------------------------------------------------------ row pass
    if (MODE & (kTileRow | kTileScale)) {
      const int lane16 = lane & 15, half = lane >> 4;
      uint4 v[kQtRowPasses];
#pragma unroll
      for (int ps = 0; ps < kQtRowPasses; ++ps) v[ps] = lds128(tile_chunk_addr(stage, qt_rowpass_row(ps, warp, half), lane16));
      float sc[kQtRowPasses], rc[kQtRowPasses];
      if (MODE & kTileRow) {
        float a[kQtRowPasses];
#pragma unroll
        for (int ps = 0; ps < kQtRowPasses; ++ps) {
          const uint32_t m2 = absmax2(absmax2(absmax2(absmax2(0u, v[ps].x), v[ps].y), v[ps].z), v[ps].w);
          a[ps] = fmaxf(bf16_lo(m2), bf16_hi(m2));
#pragma unroll
          for (int off = 8; off >= 1; off >>= 1) a[ps] = fmaxf(a[ps], __shfl_xor_sync(0xffffffffu, a[ps], off));
        }
        // lane (half*16 + j), j < kQtRowPasses, computes the scale of pass j; then broadcast
        float amine = a[0];
#pragma unroll
        for (int ps = 1; ps < kQtRowPasses; ++ps) amine = (lane16 == ps) ? a[ps] : amine;
        const float scm = group_scale(amine), rcm = recip_rn(scm);
#pragma unroll
        for (int ps = 0; ps < kQtRowPasses; ++ps) {
          sc[ps] = __shfl_sync(0xffffffffu, scm, half * 16 + ps);
          rc[ps] = __shfl_sync(0xffffffffu, rcm, half * 16 + ps);
        }
      } else {
        uint32_t m2 = 0;
#pragma unroll
        for (int ps = 0; ps < kQtRowPasses; ++ps)
          m2 = absmax2(absmax2(absmax2(absmax2(m2, v[ps].x), v[ps].y), v[ps].z), v[ps].w);
        float a = fmaxf(bf16_lo(m2), bf16_hi(m2));
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
        if (lane == 0) red[warp] = a;
        __syncthreads();
        a = red[0];
#pragma unroll
        for (int w = 1; w < kQtThreads / 32; ++w) a = fmaxf(a, red[w]);
        tile_sc = group_scale(a);
        tile_rc = recip_rn(tile_sc);
#pragma unroll
        for (int ps = 0; ps < kQtRowPasses; ++ps) {
          sc[ps] = tile_sc;
          rc[ps] = tile_rc;
        }
        if (tid == 0) p.s_row[(t0 / 128) * p.lds_row + c0 / 128] = tile_sc;
      }
      if ((MODE & kTileRow) || p.q_row != nullptr) {
        const int64_t c = c0 + qt_rowpass_col(lane16);
#pragma unroll
        for (int ps = 0; ps < kQtRowPasses; ++ps) {
          const int64_t t = t0 + qt_rowpass_row(ps, warp, half);
          const uint2 o = quant8(v[ps], sc[ps], rc[ps]);
          if (t < p.T) {
            uint8_t* dst = p.q_row + t * p.ldq_row + c;
            if (c + 8 <= p.C) {
              *reinterpret_cast<uint2*>(dst) = o;
            } else {
#pragma unroll
              for (int b = 0; b < 8; ++b)
                if (c + b < p.C) dst[b] = (uint8_t)(((b < 4) ? o.x : o.y) >> (8 * (b & 3)));
            }
            if ((MODE & kTileRow) && lane16 == 0) p.s_row[(c0 / 128) * p.lds_row + t] = sc[ps];
          }
        }
      }
    }

    // ------------------------------------------------------------ column pass
    if ((MODE & kTileCol) || ((MODE & kTileScale) && p.q_col != nullptr)) {
#pragma unroll
      for (int h = 0; h < kQtColChunks; ++h) {
        const int chunk = qt_colpass_chunk(warp, h);
        uint4 v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = lds128(tile_chunk_addr(stage, qt_colpass_row(lane, i), chunk));
        float sc[8], rc[8];
        if (MODE & kTileCol) {
          uint32_t m2[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            m2[q] = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) m2[q] = absmax2(m2[q], word_of(v[i], q));
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) m2[q] = __vmaxu2(m2[q], __shfl_xor_sync(0xffffffffu, m2[q], off));
          }
          // lane j < 8 computes the scale of column j of the chunk; then broadcast
          float amine = 0.0f;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float aj = (j & 1) ? bf16_hi(m2[j >> 1]) : bf16_lo(m2[j >> 1]);
            amine = ((lane & 7) == j) ? aj : amine;
          }
          const float scm = group_scale(amine), rcm = recip_rn(scm);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            sc[j] = __shfl_sync(0xffffffffu, scm, j);
            rc[j] = __shfl_sync(0xffffffffu, rcm, j);
          }
          const int64_t cg = c0 + 8 * chunk + lane;  // lanes 0..7 hold the chunk's 8 column scales
          if (lane < 8 && cg < p.C) p.s_col[(t0 / 128) * p.lds_col + cg] = scm;
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            sc[j] = tile_sc;
            rc[j] = tile_rc;
          }
        }
        // quantise column by column; byte (row r, column j) -> tout[8*chunk + j][r]
#pragma unroll
        for (int i = 0; i < 4; ++i) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t wq = word_of(v[i], q);
            const uint64_t x2 = f2_pack(bf16_lo(wq), bf16_hi(wq));
            // the two columns of this word have different scales
            const uint64_t ns2 = f2_pack(-sc[2 * q], -sc[2 * q + 1]), y2 = f2_pack(rc[2 * q], rc[2 * q + 1]);
            const uint64_t q0 = f2_mul(x2, y2);
            const uint64_t r0 = f2_fma(ns2, q0, x2);
            const uint64_t q1 = f2_fma(r0, y2, q0);
            const uint64_t r1 = f2_fma(ns2, q1, x2);
            const uint64_t q2 = f2_copysign(f2_fma(r1, y2, q1), x2);
            const uint32_t bb = cvt_e4m3x2(__uint_as_float((uint32_t)q2), __uint_as_float((uint32_t)(q2 >> 32)));
            const uint32_t r = (uint32_t)qt_colpass_row(lane, i);
            asm volatile("st.shared.u8 [%0], %1;" ::"r"(tout + (uint32_t)((8 * chunk + 2 * q) * 128) + r), "r"(bb & 0xFF));
            asm volatile("st.shared.u8 [%0], %1;" ::"r"(tout + (uint32_t)((8 * chunk + 2 * q + 1) * 128) + r),
                         "r"(bb >> 8));
          }
        }
      }
      __syncthreads();
#pragma unroll
      for (int k = 0; k < (128 * 128 / 16) / kQtThreads; ++k) {
        const int ch = tid + k * kQtThreads;
        const int64_t cg = c0 + qt_store_col(ch), tg = t0 + qt_store_row(ch);
        if (cg < p.C) {
          const uint4 val = lds128(tout + (uint32_t)(qt_store_col(ch) * 128 + qt_store_row(ch)));
          uint8_t* dst = p.q_col + cg * p.ldq_col + tg;
          if (tg + 16 <= p.T) {
            *reinterpret_cast<uint4*>(dst) = val;
          } else {
            const uint32_t w[4] = {val.x, val.y, val.z, val.w};
#pragma unroll
            for (int b = 0; b < 16; ++b)
              if (tg + b < p.T) dst[b] = (uint8_t)(w[b >> 2] >> (8 * (b & 3)));
          }
        }
      }
    }
    __syncthreads();  // the stage and the transposed tile are free again
    if (tid == 0) {
      const int64_t next = tile + 2 * (int64_t)gridDim.x;
      if (next < p.num_tiles) issue(next, s);
    }
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

static PFN_cuTensorMapEncodeTiled_v12000 qt_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

bool quant_tile_supported(const void* x, int64_t ldx) {
  return ((reinterpret_cast<uintptr_t>(x) & 15u) == 0) && (ldx % 8 == 0) && qt_encode_fn() != nullptr;
}

template <int MODE>
static cudaError_t run_tile(const CUtensorMap& m, const TileQuantParams& p, int64_t grid, cudaStream_t st) {
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [] {
    attr = cudaFuncSetAttribute(quant_tile_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, kQtSmemBytes);
  });
  if (attr != cudaSuccess) return attr;
  quant_tile_kernel<MODE><<<(unsigned)grid, kQtThreads, kQtSmemBytes, st>>>(m, p);
  return cudaGetLastError();
}

cudaError_t launch_quant_tile(int mode, const uint16_t* x, int64_t T, int64_t C, int64_t ldx, uint8_t* q_row,
                              int64_t ldq_row, float* s_row, int64_t lds_row, uint8_t* q_col, int64_t ldq_col,
                              float* s_col, int64_t lds_col, int num_sms, cudaStream_t st) {
  CUtensorMap m;
  cuuint64_t dims[2] = {(cuuint64_t)C, (cuuint64_t)T};
  cuuint64_t strides[1] = {(cuuint64_t)ldx * 2};
  cuuint32_t box[2] = {64, 128};
  cuuint32_t elem[2] = {1, 1};
  if (qt_encode_fn()(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(x), dims, strides, box, elem,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  TileQuantParams p;
  p.T = T;
  p.C = C;
  p.q_row = q_row;
  p.ldq_row = ldq_row;
  p.s_row = s_row;
  p.lds_row = lds_row;
  p.q_col = q_col;
  p.ldq_col = ldq_col;
  p.s_col = s_col;
  p.lds_col = lds_col;
  p.tiles_c = cdiv(C, 128);
  p.num_tiles = cdiv(T, 128) * p.tiles_c;
  p.wait_limit_ns = kWaitLimitNs;
  const int64_t grid = qt_grid(p.num_tiles, num_sms);
  switch (mode) {
    case kTileRow: return run_tile<kTileRow>(m, p, grid, st);
    case kTileCol: return run_tile<kTileCol>(m, p, grid, st);
    case kTileRow | kTileCol: return run_tile<kTileRow | kTileCol>(m, p, grid, st);
    case kTileScale: return run_tile<kTileScale>(m, p, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t quant_read_errors(uint32_t* out) {
  uint32_t zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_quant_error, sizeof(uint32_t));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_quant_error, &zero, sizeof(uint32_t));
}

}  // namespace bfp8
