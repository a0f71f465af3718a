// Blockwise e4m3 quantisation kernels (1x128 rows, 128x1 columns written
// transposed, 128x128 weight tiles) and the elementwise cast.
//
// Method ("Enable blockwise FP8 dense training kernels on ROCm", quantization
// kernel correctness table and summary; the lhs scale-store fix of its
// root-cause comment): per group amax = max|x| over in-range elements,
// s = max(amax, 1e-12)/448, q = RNE_e4m3(clamp(x/s, +-448)).  Every load,
// byte store and scale store is masked to the logical tensor.
//
// These kernels are HBM-bound (about 3 bytes moved per element): 16-byte
// vector loads, packed-bf16 amax, warp-shuffle reductions, one reciprocal per
// group and a corrected product per element for x/s, packed e4m3 stores.
#include "common.cuh"
#include "kernels.h"

namespace bfp8 {

// max(|a|, |b|) of packed bf16 pairs: on non-negative bf16 bit patterns the
// unsigned 16-bit order is the value order.
__device__ __forceinline__ uint32_t absmax2(uint32_t acc, uint32_t w) {
  return __vmaxu2(acc, w & 0x7FFF7FFFu);
}
__device__ __forceinline__ float absmax2_to_float(uint32_t m2) {
  return fmaxf(bf16_lo(m2), bf16_hi(m2));
}

// ---------------------------------------------------------------------------
// 1x128 groups along the contiguous dimension of a row-major [M,K] input.
// ---------------------------------------------------------------------------
template <bool kVec>
__global__ void __launch_bounds__(kRowThreads) quant_rows_kernel(
    const uint16_t* __restrict__ x, int64_t M, int64_t K, int64_t ldx, uint8_t* __restrict__ q,
    int64_t ldq, float* __restrict__ s, int64_t lds, int64_t Kb, int64_t num_groups,
    int64_t iters) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane16 = threadIdx.x & 15;
  const int64_t hw = ((int64_t)blockIdx.x * kRowThreads + threadIdx.x) >> 4;
  const int64_t nhw = ((int64_t)gridDim.x * kRowThreads) >> 4;

  for (int64_t it = 0; it < iters; ++it) {
    uint32_t v[kRowUnroll][4];
    int64_t mm[kRowUnroll], kk[kRowUnroll];
    bool gv[kRowUnroll];
#pragma unroll
    for (int u = 0; u < kRowUnroll; ++u) {
      const int64_t g = row_group(hw, nhw, it, u);
      gv[u] = g < num_groups;
      const RowChunk c = row_chunk(gv[u] ? g : 0, lane16, Kb);
      mm[u] = c.m;
      kk[u] = c.k;
      const uint16_t* src = x + c.m * ldx + c.k;
      if (kVec && gv[u] && c.k + 8 <= K) {
        const uint4 w = ld_nc_v4(src);
        v[u][0] = w.x; v[u][1] = w.y; v[u][2] = w.z; v[u][3] = w.w;
      } else {
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const uint32_t lo = (gv[u] && c.k + 2 * p < K) ? src[2 * p] : 0u;
          const uint32_t hi = (gv[u] && c.k + 2 * p + 1 < K) ? src[2 * p + 1] : 0u;
          v[u][p] = lo | (hi << 16);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kRowUnroll; ++u) {
      uint32_t m2 = 0;
#pragma unroll
      for (int p = 0; p < 4; ++p) m2 = absmax2(m2, v[u][p]);
      float amax = absmax2_to_float(m2);
#pragma unroll
      for (int off = 8; off >= 1; off >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
      const float sc = group_scale(amax);
      const float rc = recip_rn(sc);
      uint32_t out[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t w0 = v[u][2 * h], w1 = v[u][2 * h + 1];
        out[h] = cvt_e4m3x2(quotient(bf16_lo(w0), sc, rc), quotient(bf16_hi(w0), sc, rc)) |
                 (cvt_e4m3x2(quotient(bf16_lo(w1), sc, rc), quotient(bf16_hi(w1), sc, rc)) << 16);
      }
      if (gv[u]) {
        uint8_t* dst = q + mm[u] * ldq + kk[u];
        if (kk[u] + 8 <= K) {
          *reinterpret_cast<uint2*>(dst) = make_uint2(out[0], out[1]);
        } else {
#pragma unroll
          for (int b = 0; b < 8; ++b)
            if (kk[u] + b < K) dst[b] = (uint8_t)(out[b >> 2] >> (8 * (b & 3)));
        }
        if (lane16 == 0) s[(kk[u] / kBlock) * lds + mm[u]] = sc;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Groups of 128 consecutive rows of one column of a row-major [T,C] input,
// written transposed: qT[c*ldq + t], s[(t/128)*lds + c].
// ---------------------------------------------------------------------------
template <bool kVec>
__global__ void __launch_bounds__(kColThreads) quant_cols_kernel(
    const uint16_t* __restrict__ x, int64_t T, int64_t C, int64_t ldx, uint8_t* __restrict__ qT,
    int64_t ldq, float* __restrict__ s, int64_t lds) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ __align__(16) uint32_t tout[kColTileC][kColTileT / 4];  // 64 rows of 128 bytes
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const ColTile tile = col_tile(blockIdx.x, C);
  const int64_t c_first = col_elem_c(tile, warp, 0);

  uint32_t v[4][4];  // [row i][column pair p]
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t t = col_elem_t(tile, lane, i);
    const uint16_t* src = x + t * ldx + c_first;
    if (kVec && t < T && c_first + 8 <= C) {
      const uint4 w = ld_nc_v4(src);
      v[i][0] = w.x; v[i][1] = w.y; v[i][2] = w.z; v[i][3] = w.w;
    } else {
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const uint32_t lo = (t < T && c_first + 2 * p < C) ? src[2 * p] : 0u;
        const uint32_t hi = (t < T && c_first + 2 * p + 1 < C) ? src[2 * p + 1] : 0u;
        v[i][p] = lo | (hi << 16);
      }
    }
  }
  // column amax over the 4 rows of this lane, then over the 32 lanes (128 rows)
  uint32_t m2[4];
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    m2[p] = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) m2[p] = absmax2(m2[p], v[i][p]);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) m2[p] = __vmaxu2(m2[p], __shfl_xor_sync(0xffffffffu, m2[p], off));
  }
  float sc[8], rc[8];
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    sc[2 * p] = group_scale(bf16_lo(m2[p]));
    sc[2 * p + 1] = group_scale(bf16_hi(m2[p]));
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) rc[j] = recip_rn(sc[j]);
  // quantise; one 32-bit word per column = the column's 4 rows, in row order
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    float r[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t w = v[i][j >> 1];
      r[i] = quotient((j & 1) ? bf16_hi(w) : bf16_lo(w), sc[j], rc[j]);
    }
    tout[8 * warp + j][lane] = cvt_e4m3x2(r[0], r[1]) | (cvt_e4m3x2(r[2], r[3]) << 16);
  }
  {
    const int64_t tb = tile.t0 / kBlock;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (lane == j && c_first + j < C) s[tb * lds + c_first + j] = sc[j];
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < (kColTileC * kColTileT / 16) / kColThreads; ++r) {
    const int ch = threadIdx.x + r * kColThreads;
    const int64_t c = col_store_c(tile, ch), t = col_store_t(tile, ch);
    if (c < C) {
      const uint4 val = *reinterpret_cast<const uint4*>(&tout[ch / 8][(ch % 8) * 4]);
      uint8_t* dst = qT + c * ldq + t;
      if (t + 16 <= T) {
        *reinterpret_cast<uint4*>(dst) = val;
      } else {
        const uint32_t w[4] = {val.x, val.y, val.z, val.w};
#pragma unroll
        for (int b = 0; b < 16; ++b)
          if (t + b < T) dst[b] = (uint8_t)(w[b >> 2] >> (8 * (b & 3)));
      }
    }
  }
}

// ---------------------------------------------------------------------------
// 128x128 weight tiles; q written as is, qt (optional) transposed.
// ---------------------------------------------------------------------------
template <bool kVec>
__global__ void __launch_bounds__(kWThreads) quant_weight_kernel(
    const uint16_t* __restrict__ w, int64_t N, int64_t K, int64_t ldw, uint8_t* __restrict__ q,
    int64_t ldq, uint8_t* __restrict__ qt, int64_t ldqt, float* __restrict__ s, int64_t lds,
    int64_t Kb) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ __align__(16) uint32_t tout[kBlock][kBlock / 4];  // 128 k-rows of 128 n-bytes
  __shared__ float red[kWThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const WTile tile = w_tile(blockIdx.x, Kb);

  uint32_t v[2][4][4];  // [chunk][row i][column pair]
  uint32_t m2 = 0;
#pragma unroll
  for (int cc = 0; cc < 2; ++cc) {
    const int chunk = warp + 8 * cc;
    const int64_t k = w_elem_k(tile, chunk, 0);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t n = w_elem_n(tile, lane, i);
      const uint16_t* src = w + n * ldw + k;
      if (kVec && n < N && k + 8 <= K) {
        const uint4 u = ld_nc_v4(src);
        v[cc][i][0] = u.x; v[cc][i][1] = u.y; v[cc][i][2] = u.z; v[cc][i][3] = u.w;
      } else {
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const uint32_t lo = (n < N && k + 2 * p < K) ? src[2 * p] : 0u;
          const uint32_t hi = (n < N && k + 2 * p + 1 < K) ? src[2 * p + 1] : 0u;
          v[cc][i][p] = lo | (hi << 16);
        }
      }
#pragma unroll
      for (int p = 0; p < 4; ++p) m2 = absmax2(m2, v[cc][i][p]);
    }
  }
  float amax = absmax2_to_float(m2);
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if (lane == 0) red[warp] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int i = 1; i < kWThreads / 32; ++i) amax = fmaxf(amax, red[i]);
  const float sc = group_scale(amax);
  const float rc = recip_rn(sc);
  if (threadIdx.x == 0) s[tile.nb * lds + tile.kb] = sc;

#pragma unroll
  for (int cc = 0; cc < 2; ++cc) {
    const int chunk = warp + 8 * cc;
    const int64_t k = w_elem_k(tile, chunk, 0);
    uint32_t row_words[4][2];  // [row i][columns 0-3 / 4-7]
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t a = v[cc][i][2 * h], b = v[cc][i][2 * h + 1];
        row_words[i][h] = cvt_e4m3x2(quotient(bf16_lo(a), sc, rc), quotient(bf16_hi(a), sc, rc)) |
                          (cvt_e4m3x2(quotient(bf16_lo(b), sc, rc), quotient(bf16_hi(b), sc, rc)) << 16);
      }
      const int64_t n = w_elem_n(tile, lane, i);
      if (q != nullptr && n < N) {
        uint8_t* dst = q + n * ldq + k;
        if (k + 8 <= K) {
          *reinterpret_cast<uint2*>(dst) = make_uint2(row_words[i][0], row_words[i][1]);
        } else {
#pragma unroll
          for (int b = 0; b < 8; ++b)
            if (k + b < K) dst[b] = (uint8_t)(row_words[i][b >> 2] >> (8 * (b & 3)));
        }
      }
    }
    if (qt != nullptr) {
      // 4x4 byte transposes: rows i = 0..3 of this lane -> one word per column
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t t0 = __byte_perm(row_words[0][h], row_words[1][h], 0x5140);
        const uint32_t t1 = __byte_perm(row_words[0][h], row_words[1][h], 0x7362);
        const uint32_t t2 = __byte_perm(row_words[2][h], row_words[3][h], 0x5140);
        const uint32_t t3 = __byte_perm(row_words[2][h], row_words[3][h], 0x7362);
        tout[8 * chunk + 4 * h + 0][lane] = __byte_perm(t0, t2, 0x5410);
        tout[8 * chunk + 4 * h + 1][lane] = __byte_perm(t0, t2, 0x7632);
        tout[8 * chunk + 4 * h + 2][lane] = __byte_perm(t1, t3, 0x5410);
        tout[8 * chunk + 4 * h + 3][lane] = __byte_perm(t1, t3, 0x7632);
      }
    }
  }
  if (qt != nullptr) {
    __syncthreads();
#pragma unroll
    for (int r = 0; r < (kBlock * kBlock / 16) / kWThreads; ++r) {
      const int ch = threadIdx.x + r * kWThreads;
      const int64_t k = w_tstore_k(tile, ch), n = w_tstore_n(tile, ch);
      if (k < K) {
        const uint4 val = *reinterpret_cast<const uint4*>(&tout[ch / 8][(ch % 8) * 4]);
        uint8_t* dst = qt + k * ldqt + n;
        if (n + 16 <= N) {
          *reinterpret_cast<uint4*>(dst) = val;
        } else {
          const uint32_t wv[4] = {val.x, val.y, val.z, val.w};
#pragma unroll
          for (int b = 0; b < 16; ++b)
            if (n + b < N) dst[b] = (uint8_t)(wv[b >> 2] >> (8 * (b & 3)));
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Elementwise fp32 -> e4m3 (the rounding step alone).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) cast_kernel(const float* __restrict__ x, int64_t n,
                                                   uint8_t* __restrict__ q, int vec) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i * 8 < n; i += stride) {
    const int64_t e = i * 8;
    if (vec && e + 8 <= n) {
      const float4 a = *reinterpret_cast<const float4*>(x + e);
      const float4 b = *reinterpret_cast<const float4*>(x + e + 4);
      const uint32_t w0 = cvt_e4m3x2(a.x, a.y) | (cvt_e4m3x2(a.z, a.w) << 16);
      const uint32_t w1 = cvt_e4m3x2(b.x, b.y) | (cvt_e4m3x2(b.z, b.w) << 16);
      *reinterpret_cast<uint2*>(q + e) = make_uint2(w0, w1);
    } else {
      for (int64_t j = e; j < n && j < e + 8; ++j) q[j] = (uint8_t)cvt_e4m3x2(x[j], 0.0f);
    }
  }
}

// ---------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

cudaError_t launch_quant_rows(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q,
                              int64_t ldq, float* s, int64_t lds, int num_sms, cudaStream_t st) {
  const int64_t Kb = cdiv(K, kBlock);
  const int64_t groups = M * Kb;
  const int64_t groups_per_cta = (kRowThreads / 16) * kRowUnroll;
  int64_t grid = cdiv(groups, groups_per_cta);
  const int64_t cap = (int64_t)num_sms * 8;  // 8 resident CTAs of 256 threads per SM
  if (grid > cap) grid = cap;
  const int64_t nhw = grid * (kRowThreads / 16);
  const int64_t iters = cdiv(groups, nhw * kRowUnroll);
  const bool vec = (ldx % 8 == 0) && aligned16(x);
  return launch_pdl(vec ? quant_rows_kernel<true> : quant_rows_kernel<false>, (unsigned)grid, kRowThreads, 0, st, x,
                    M, K, ldx, q, ldq, s, lds, Kb, groups, iters);
}

int64_t quant_rows_grid(int64_t M, int64_t K, int num_sms) {
  const int64_t groups = M * cdiv(K, kBlock);
  int64_t grid = cdiv(groups, (int64_t)(kRowThreads / 16) * kRowUnroll);
  const int64_t cap = (int64_t)num_sms * 8;
  return grid > cap ? cap : grid;
}

cudaError_t launch_quant_cols(const uint16_t* x, int64_t T, int64_t C, int64_t ldx, uint8_t* qT,
                              int64_t ldq, float* s, int64_t lds, cudaStream_t st) {
  const int64_t grid = cdiv(T, kColTileT) * cdiv(C, kColTileC);
  const bool vec = (ldx % 8 == 0) && aligned16(x);
  return launch_pdl(vec ? quant_cols_kernel<true> : quant_cols_kernel<false>, (unsigned)grid, kColThreads, 0, st, x, T,
                    C, ldx, qT, ldq, s, lds);
}

cudaError_t launch_quant_weight(const uint16_t* w, int64_t N, int64_t K, int64_t ldw, uint8_t* q,
                                int64_t ldq, uint8_t* qt, int64_t ldqt, float* s, int64_t lds,
                                cudaStream_t st) {
  const int64_t Kb = cdiv(K, kBlock);
  const int64_t grid = cdiv(N, kBlock) * Kb;
  const bool vec = (ldw % 8 == 0) && aligned16(w);
  return launch_pdl(vec ? quant_weight_kernel<true> : quant_weight_kernel<false>, (unsigned)grid, kWThreads, 0, st, w,
                    N, K, ldw, q, ldq, qt, ldqt, s, lds, Kb);
}

cudaError_t launch_cast(const float* x, int64_t n, uint8_t* q, int num_sms, cudaStream_t st) {
  int64_t grid = cdiv(cdiv(n, 8), 256);
  const int64_t cap = (int64_t)num_sms * 8;
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  const int vec = aligned16(x) && aligned16(q);
  return launch_pdl(cast_kernel, (unsigned)grid, 256, 0, st, x, n, q, vec);
}

}  // namespace bfp8
