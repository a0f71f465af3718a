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
//
// Data flow of one tile (persistent CTAs, two per SM, 16 warps each):
//   1. TMA loads the tile as two 64-column boxes (128-byte swizzle) into one
//      of two stages.
//   2. Warp w takes the 8-column chunk w, lane l the four rows 4l..4l+3 (read
//      in a lane-rotated order so that the 16-byte reads of a quarter-warp hit
//      eight different bank groups).
//   3. Group maxima: |x| maxima on packed bf16 pairs inside each thread; the
//      16 chunk maxima of a row and the 32 lane maxima of a column meet in
//      shared memory, where four threads per row / column finish them and
//      compute the scale and the negated reciprocal.
//   4. Every value is divided by its scale(s) and rounded to e4m3; the codes
//      are written into the spent input stage, row-major (128-byte swizzled)
//      and transposed (the four codes of a thread's rows in one column are one
//      32-bit word, assembled with byte permutes).
//   5. One TMA store per output writes the tile.  A TMA store clips the
//      innermost dimension in whole 16-byte units, so the maps cover only the
//      16-byte-aligned part of each row (q_row: columns < C & ~15, q_col:
//      rows < T & ~15) and the threads store the last C % 16 (T % 16) bytes of
//      each row of an edge tile from the staged tile themselves; nothing
//      outside the logical [T, C] (or [C, T]) region is written.
// Rows / columns outside [T, C] arrive as zeros (TMA fill) and cannot raise
// a maximum.  Inputs are finite bf16 values (the method's domain).
#include <cudaTypedefs.h>

#include <string.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace bfp8 {

static __device__ uint32_t g_quant_error;

namespace {

constexpr int kTileRow = kQuantTileRow, kTileCol = kQuantTileCol, kTileScale = kQuantTileScale;
constexpr int kTileMx = kQuantTileMx;
constexpr int kQtBoxBytes = 128 * 128;               // 64 bf16 columns x 128 rows
constexpr int kQtStageBytes = 2 * kQtBoxBytes;       // one 128x128 bf16 tile
// once the tile is in registers its stage holds the outputs:
constexpr int kQtOutRow = 0;                         // q_row tile: 128 rows x 128 B, 128-byte swizzled
constexpr int kQtOutCol = 128 * 128;                 // q_col tile: 128 columns x 128 B (input rows)
constexpr int kQtOffRowRed = 2 * kQtStageBytes;      // [16 chunks][128 rows] bf16x2 row maxima
constexpr int kQtOffColRed = kQtOffRowRed + 16 * 128 * 4;  // [16 chunks][32 lanes] 4 x bf16x2 column maxima
constexpr int kQtOffRowSc = kQtOffColRed + 16 * 32 * 16;   // [128 rows] (s, -1/s)
constexpr int kQtOffColSc = kQtOffRowSc + 128 * 8;         // [64 column pairs] (s0, s1, -1/s0, -1/s1)
constexpr int kQtOffBar = kQtOffColSc + 64 * 16;
constexpr int kQtSmemBytes = kQtOffBar + 64 + 1024;        // + alignment slack

struct TileQuantParams {
  int64_t T, C;
  uint8_t* q_row;   // for the ragged bytes only; the rest goes through the tensor maps
  int64_t ldq_row;
  uint8_t* q_col;
  int64_t ldq_col;
  int64_t C_al, T_al;  // C & ~15, T & ~15: extents of the two store maps
  float* s_row;
  int64_t lds_row;
  float* s_col;
  int64_t lds_col;
  int has_q_row, has_q_col;
  int64_t tiles_c, num_tiles;
  uint64_t wait_limit_ns;
  int pdl;  // launched with programmatic dependent launch: let the next kernel start early
  uint8_t* e_row;  // MXFP8: biased exponents of the dim0 and dim1 casts
  int64_t lde_row;
  uint8_t* e_col;
  int64_t lde_col;
};

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ void sts32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void sts64(uint32_t addr, uint32_t a, uint32_t b) {
  asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(addr), "r"(a), "r"(b) : "memory");
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int q) {
  return q == 0 ? v.x : q == 1 ? v.y : q == 2 ? v.z : v.w;
}

// MXFP8 (OCP Microscaling v1.0, FLOOR scale): for a block maximum amax (a
// bf16 value, here its 15 magnitude bits), e = floor(log2(amax)) - 8 clamped
// to [-127, 127]: amax's exponent field E gives e = max(E - 135, -127) (zero
// and subnormals included: they clamp).  Returns the biased byte e + 127, and
// in *mult the fp32 2^-e (a normal float: e <= 119 for bf16 inputs).
__device__ __forceinline__ uint32_t mx_exponent(uint32_t amax_bits15, float* mult) {
  const int E = (int)(amax_bits15 >> 7);
  const int e = max(E - 135, -127);
  *mult = __uint_as_float((uint32_t)(127 - e) << 23);
  return (uint32_t)(e + 127);
}

// e4m3 codes of x * mult for the two bf16 values of `w` (mult2 = (m, m')):
// one exact power-of-two product per value, rounded to nearest even and
// saturated at 448 by the conversion.
__device__ __forceinline__ uint32_t mx_codes2(uint32_t w, uint64_t mult2) {
  const uint64_t r = f2_mul(f2_pack(bf16_lo(w), bf16_hi(w)), mult2);
  return cvt_e4m3x2(__uint_as_float((uint32_t)r), __uint_as_float((uint32_t)(r >> 32)));
}

}  // namespace

// Phase 1 of a tile: this thread's 4 x 8 input values from the stage into
// registers, and its partial row / column (or tile) maxima into shared memory.
template <int MODE>
__device__ __forceinline__ void qt_load_reduce(uint32_t stage, uint4 (&v)[4], uint32_t (&cm)[4], int warp, int lane,
                                               int rot, uint32_t rowred, uint32_t colred) {
  constexpr bool kRow = (MODE & kTileRow) != 0, kCol = (MODE & kTileCol) != 0, kScale = (MODE & kTileScale) != 0;
  constexpr bool kMx = (MODE & kTileMx) != 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = 4 * lane + ((i + rot) & 3);
    v[i] = lds128(stage + (uint32_t)((warp >> 3) * kQtBoxBytes + r * 128 + (((warp & 7) ^ (r & 7)) << 4)));
  }
  uint32_t rm[4];  // per row: (max |even column|, max |odd column|)
#pragma unroll
  for (int i = 0; i < 4; ++i) rm[i] = amax2(amax2(v[i].x, v[i].y), amax2(v[i].z, v[i].w));
  if (kScale) {
    uint32_t m = amax2(amax2(rm[0], rm[1]), amax2(rm[2], rm[3]));
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) m = amax2(m, __shfl_xor_sync(0xffffffffu, m, off));
    if (lane == 0) sts32(rowred + 4u * warp, m);
  } else {
    if (kRow) {
#pragma unroll
      for (int i = 0; i < 4; ++i) sts32(rowred + 4u * (uint32_t)(warp * 128 + 4 * lane + ((i + rot) & 3)), rm[i]);
    }
    if (kCol) {
      // per column pair of the chunk, over this thread's 4 rows
#pragma unroll
      for (int q = 0; q < 4; ++q)
        cm[q] = amax2(amax2(word_of(v[0], q), word_of(v[1], q)), amax2(word_of(v[2], q), word_of(v[3], q)));
      if (kMx) {
        // MXFP8: a 32-row block is the 4 rows of 8 consecutive lanes
#pragma unroll
        for (int off = 1; off <= 4; off <<= 1)
#pragma unroll
          for (int q = 0; q < 4; ++q) cm[q] = amax2(cm[q], __shfl_xor_sync(0xffffffffu, cm[q], off));
      } else {
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(colred + 16u * (uint32_t)(warp * 32 + lane)),
                     "r"(cm[0]), "r"(cm[1]), "r"(cm[2]), "r"(cm[3])
                     : "memory");
      }
    }
  }
}

// Phase 2 of a tile (after the maxima are visible): the scales, the codes into
// the spent stage, and the TMA stores (plus the ragged bytes of edge tiles).
template <int MODE>
__device__ __forceinline__ void qt_scale_store(const CUtensorMap* tmap_qrow, const CUtensorMap* tmap_qcol,
                                               const TileQuantParams& p, int64_t tile, uint32_t stage,
                                               const uint4 (&v)[4], const uint32_t (&cm)[4], int tid, int warp,
                                               int lane, int rot, uint32_t sel_e, uint32_t sel_o, uint32_t sbase,
                                               uint32_t rowred, uint32_t colred) {
  constexpr bool kRow = (MODE & kTileRow) != 0, kCol = (MODE & kTileCol) != 0, kScale = (MODE & kTileScale) != 0;
  constexpr bool kMx = (MODE & kTileMx) != 0;
  const bool out_row = kRow || (kScale && p.has_q_row);
  const bool out_col = kCol || (kScale && p.has_q_col);
  const int64_t t0 = qt_tile_t0(tile, p.tiles_c), c0 = qt_tile_c0(tile, p.tiles_c);
  if constexpr (kMx) {
    // ------------------------------------------------ MXFP8 exponents
    if (kRow) {  // dim0: thread tid takes row tid & 127, 32-column block tid >> 7
      const int r = tid & 127, g = tid >> 7;
      uint32_t m = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t w;
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w) : "r"(rowred + 4u * (uint32_t)((4 * g + j) * 128 + r)));
        m = amax2(m, w);
      }
      m = amax2(m, __byte_perm(m, 0, 0x1032));
      float mult;
      const uint32_t eb = mx_exponent((m >> 16) & 0x7FFFu, &mult);
      asm volatile("st.shared.f32 [%0], %1;" ::"r"(sbase + kQtOffRowSc + 4u * (uint32_t)(g * 128 + r)), "f"(mult)
                   : "memory");
      if (t0 + r < p.T && c0 + 32 * g < p.C) p.e_row[(t0 + r) * p.lde_row + c0 / 32 + g] = (uint8_t)eb;
    }
    float cmult[8];  // dim1: the 2^-e of this thread's 8 columns over its lane group's 32 rows
    if (kCol) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        mx_exponent(cm[q] & 0x7FFFu, &cmult[2 * q]);
        mx_exponent((cm[q] >> 16) & 0x7FFFu, &cmult[2 * q + 1]);
      }
      // lane l of the 8-lane group h = l / 8 stores the exponent of column 8*warp + l % 8
      const int j = lane & 7, h = lane >> 3;
      const uint32_t w = j < 2 ? cm[0] : j < 4 ? cm[1] : j < 6 ? cm[2] : cm[3];
      float unused;
      const uint32_t eb = mx_exponent(((j & 1) ? (w >> 16) : w) & 0x7FFFu, &unused);
      if (c0 + 8 * warp + j < p.C && t0 + 32 * h < p.T)
        p.e_col[(c0 + 8 * warp + j) * p.lde_col + t0 / 32 + h] = (uint8_t)eb;
    }
    __syncthreads();  // the row multipliers are visible

    // ------------------------------------------------ codes into the spent stage
    if (kCol) {
      const uint32_t dst = stage + kQtOutCol + (uint32_t)(8 * warp * 128 + 4 * lane);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint64_t mult2 = f2_pack(cmult[2 * q], cmult[2 * q + 1]);
        uint32_t cc[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) cc[i] = mx_codes2(word_of(v[i], q), mult2);
        const uint32_t X = __byte_perm(cc[0], cc[1], 0x5140), Y = __byte_perm(cc[2], cc[3], 0x5140);
        sts32(dst + (uint32_t)((2 * q) * 128), __byte_perm(X, Y, sel_e));
        sts32(dst + (uint32_t)((2 * q + 1) * 128), __byte_perm(X, Y, sel_o));
      }
    }
    if (kRow) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = 4 * lane + ((i + rot) & 3);
        float mult;
        asm volatile("ld.shared.f32 %0, [%1];"
                     : "=f"(mult)
                     : "r"(sbase + kQtOffRowSc + 4u * (uint32_t)((warp >> 2) * 128 + r)));
        const uint64_t mult2 = f2_pack(mult, mult);
        const uint32_t c01 = mx_codes2(v[i].x, mult2), c23 = mx_codes2(v[i].y, mult2);
        const uint32_t c45 = mx_codes2(v[i].z, mult2), c67 = mx_codes2(v[i].w, mult2);
        sts64(stage + kQtOutRow + (uint32_t)(r * 128 + ((((warp >> 1) ^ (r & 7)) << 4) | ((warp & 1) << 3))),
              __byte_perm(c01, c23, 0x5410), __byte_perm(c45, c67, 0x5410));
      }
    }
  } else {
  // ------------------------------------------------ scales
  float tile_s = 0.0f, tile_ny = 0.0f;
  if (kScale) {
    uint32_t m = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint4 a = lds128(rowred + 16u * k);
      m = amax2(m, amax2(amax2(a.x, a.y), amax2(a.z, a.w)));
    }
    m = amax2(m, __byte_perm(m, 0, 0x1032));
    tile_s = scale_of(__uint_as_float(m & 0x7FFF0000u));
    tile_ny = neg_rcp(tile_s);
    if (tid == 0) p.s_row[(t0 / 128) * p.lds_row + c0 / 128] = tile_s;
  } else {
    const int g = qt_scale_group(tid), qd = tid & 3;  // four threads per row / column g of the tile
    if (kRow) {
      uint32_t m = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t w;
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w) : "r"(rowred + 4u * (uint32_t)((4 * qd + j) * 128 + g)));
        m = amax2(m, w);
      }
      m = amax2(m, __shfl_xor_sync(0xffffffffu, m, 1));
      m = amax2(m, __shfl_xor_sync(0xffffffffu, m, 2));
      m = amax2(m, __byte_perm(m, 0, 0x1032));
      const float sc = scale_of(__uint_as_float(m & 0x7FFF0000u));
      if (qt_scale_writer(tid)) {
        const float ny = neg_rcp(sc);
        asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(sbase + kQtOffRowSc + 8u * g), "f"(sc), "f"(ny)
                     : "memory");
        if (t0 + g < p.T) p.s_row[(c0 / 128) * p.lds_row + t0 + g] = sc;
      }
    }
    if (kCol) {
      const int w = g >> 3, q = (g & 7) >> 1;
      uint32_t m = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint32_t x;
        asm volatile("ld.shared.u32 %0, [%1];"
                     : "=r"(x)
                     : "r"(colred + 16u * (uint32_t)(w * 32 + 8 * qd + j) + 4u * q));
        m = amax2(m, x);
      }
      m = amax2(m, __shfl_xor_sync(0xffffffffu, m, 1));
      m = amax2(m, __shfl_xor_sync(0xffffffffu, m, 2));
      const uint32_t bits = (g & 1) ? (m & 0x7FFF0000u) : ((m << 16) & 0x7FFF0000u);
      const float sc = scale_of(__uint_as_float(bits));
      if (qt_scale_writer(tid)) {
        const uint32_t slot = sbase + kQtOffColSc + 16u * (uint32_t)(g >> 1) + 4u * (g & 1);
        asm volatile("st.shared.f32 [%0], %1;" ::"r"(slot), "f"(sc) : "memory");
        asm volatile("st.shared.f32 [%0], %1;" ::"r"(slot + 8u), "f"(neg_rcp(sc)) : "memory");
        if (c0 + g < p.C) p.s_col[(t0 / 128) * p.lds_col + c0 + g] = sc;
      }
    }
    __syncthreads();  // scales visible
  }

  // ------------------------------------------------ codes into the spent stage
  if (out_col) {
    // column pair q of the chunk: the four rows' codes of each column -> one word
    const uint32_t dst = stage + kQtOutCol + (uint32_t)(8 * warp * 128 + 4 * lane);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint64_t s2, ny2;
      if (kScale) {
        s2 = f2_pack(tile_s, tile_s);
        ny2 = f2_pack(tile_ny, tile_ny);
      } else {
        // (s, s', -1/s, -1/s') of columns 8*warp + 2q, +1
        asm volatile("ld.shared.v2.u64 {%0, %1}, [%2];"
                     : "=l"(s2), "=l"(ny2)
                     : "r"(sbase + kQtOffColSc + 16u * (uint32_t)(4 * warp + q)));
      }
      uint32_t cc[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) cc[i] = neg_codes2(word_of(v[i], q), s2, ny2);
      const uint32_t X = __byte_perm(cc[0], cc[1], 0x5140), Y = __byte_perm(cc[2], cc[3], 0x5140);
      sts32(dst + (uint32_t)((2 * q) * 128), __byte_perm(X, Y, sel_e) ^ 0x80808080u);
      sts32(dst + (uint32_t)((2 * q + 1) * 128), __byte_perm(X, Y, sel_o) ^ 0x80808080u);
    }
  }
  if (out_row) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = 4 * lane + ((i + rot) & 3);
      uint64_t s2, ny2;
      if (kScale) {
        s2 = f2_pack(tile_s, tile_s);
        ny2 = f2_pack(tile_ny, tile_ny);
      } else {
        float rs, rny;
        asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(rs), "=f"(rny) : "r"(sbase + kQtOffRowSc + 8u * r));
        s2 = f2_pack(rs, rs);
        ny2 = f2_pack(rny, rny);
      }
      const uint32_t c01 = neg_codes2(v[i].x, s2, ny2), c23 = neg_codes2(v[i].y, s2, ny2);
      const uint32_t c45 = neg_codes2(v[i].z, s2, ny2), c67 = neg_codes2(v[i].w, s2, ny2);
      const uint32_t lo = __byte_perm(c01, c23, 0x5410) ^ 0x80808080u;
      const uint32_t hi = __byte_perm(c45, c67, 0x5410) ^ 0x80808080u;
      sts64(stage + kQtOutRow + (uint32_t)(r * 128 + ((((warp >> 1) ^ (r & 7)) << 4) | ((warp & 1) << 3))), lo, hi);
    }
  }
  }  // blockwise scales
  fence_proxy_async_shared();
  __syncthreads();  // the output tiles are complete
  if (tid == 0) {
    if (out_row && c0 < p.C_al) tma_store_2d(tmap_qrow, stage + kQtOutRow, (int32_t)c0, (int32_t)t0);
    if (out_col && t0 < p.T_al) tma_store_2d(tmap_qcol, stage + kQtOutCol, (int32_t)t0, (int32_t)c0);
    bulk_commit();
  }
  // ragged bytes past the maps' 16-byte-aligned extents (edge tiles only):
  // thread tid covers row / column qt_scale_group(tid) of the tile and
  // four of the (at most 15) trailing positions
  const int g = qt_scale_group(tid), b0 = 4 * (tid & 3);
  if (out_row && c0 + 128 > p.C_al && p.C_al < p.C && t0 + g < p.T) {
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int64_t c = p.C_al + b0 + b;
      if (c < p.C) {
        const int cl = (int)(c - c0);
        uint32_t b8;
        asm volatile("ld.shared.u8 %0, [%1];"
                     : "=r"(b8)
                     : "r"(stage + kQtOutRow + (uint32_t)(g * 128 + ((((cl >> 4) ^ (g & 7)) << 4) | (cl & 15)))));
        p.q_row[(t0 + g) * p.ldq_row + c] = (uint8_t)b8;
      }
    }
  }
  if (out_col && t0 + 128 > p.T_al && p.T_al < p.T && c0 + g < p.C) {
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int64_t t = p.T_al + b0 + b;
      if (t < p.T) {
        uint32_t b8;
        asm volatile("ld.shared.u8 %0, [%1];" : "=r"(b8) : "r"(stage + kQtOutCol + (uint32_t)(g * 128 + (t - t0))));
        p.q_col[(c0 + g) * p.ldq_col + t] = (uint8_t)b8;
      }
    }
  }
}

// One launch quantises the tiles of up to two inputs (A's tiles first, then
// B's), e.g. both forms of x and the weight's tiles for a forward step: one
// pipeline ramp-up and drain instead of two.  A single input passes B with no
// tiles.
template <int MODE_A, int MODE_B>
__global__ void __launch_bounds__(kQtThreads, 2)
    quant_tile_kernel(const __grid_constant__ CUtensorMap tmap_xa, const __grid_constant__ CUtensorMap tmap_qrow_a,
                      const __grid_constant__ CUtensorMap tmap_qcol_a, const __grid_constant__ CUtensorMap tmap_xb,
                      const __grid_constant__ CUtensorMap tmap_qrow_b, const __grid_constant__ CUtensorMap tmap_qcol_b,
                      const TileQuantParams pa, const TileQuantParams pb) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + kQtOffBar;
  volatile int* never = reinterpret_cast<volatile int*>(smem + kQtOffBar + 16);
  const uint32_t rowred = sbase + kQtOffRowRed;  // also the per-warp tile maxima (kTileScale)
  const uint32_t colred = sbase + kQtOffColRed;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t na = pa.num_tiles, num_tiles = pa.num_tiles + pb.num_tiles;
  // only a kernel launched with programmatic dependent launch lets the next
  // one start early; otherwise the next kernel starts once this one completes
  if (pa.pdl) pdl_launch_dependents();

  if (tid == 0) {
    mbar_init(bar0, 1);
    mbar_init(bar0 + 8, 1);
    *never = 0;
    fence_barrier_init();
    fence_proxy_async_shared();
    tma_prefetch_desc(&tmap_xa);
    if (pa.has_q_row && pa.C_al > 0) tma_prefetch_desc(&tmap_qrow_a);
    if (pa.has_q_col && pa.T_al > 0) tma_prefetch_desc(&tmap_qcol_a);
    if (pb.num_tiles > 0) {
      tma_prefetch_desc(&tmap_xb);
      if (pb.has_q_row && pb.C_al > 0) tma_prefetch_desc(&tmap_qrow_b);
      if (pb.has_q_col && pb.T_al > 0) tma_prefetch_desc(&tmap_qcol_b);
    }
  }
  __syncthreads();
  pdl_wait();  // the previous kernel's writes are visible from here on

  // Lane l reads its rows in the order 4l + rho(i), rho(i) = (i + rot) & 3.
  const int rot = (lane >> 1) & 3;
  // Byte selectors that put the codes of rows 4l..4l+3 of one column, in row
  // order, into one word (see the column store below): in the 8 bytes
  // (X, Y), slot i's code of the even column sits at {0, 1, 4, 5}[i], of the
  // odd column at {2, 3, 6, 7}[i].
  uint32_t sel_e = 0, sel_o = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int i = (k - rot) & 3;
    sel_e |= (uint32_t)((i & 1) + 4 * (i >> 1)) << (4 * k);
    sel_o |= (uint32_t)(2 + (i & 1) + 4 * (i >> 1)) << (4 * k);
  }

  auto issue = [&](int64_t tile, int s) {
    const bool in_a = tile < na;
    const int64_t local = in_a ? tile : tile - na, tiles_c = in_a ? pa.tiles_c : pb.tiles_c;
    const int32_t t0 = (int32_t)qt_tile_t0(local, tiles_c), c0 = (int32_t)qt_tile_c0(local, tiles_c);
    const CUtensorMap* mx = in_a ? &tmap_xa : &tmap_xb;
    const uint32_t st = sbase + (uint32_t)(s * kQtStageBytes);
    mbar_arrive_expect_tx(bar0 + 8u * s, (uint32_t)kQtStageBytes);
    tma_load_2d(st, mx, bar0 + 8u * s, c0, t0);
    tma_load_2d(st + kQtBoxBytes, mx, bar0 + 8u * s, c0 + 64, t0);
  };
  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      const int64_t tile = blockIdx.x + (int64_t)s * gridDim.x;
      if (tile < num_tiles) issue(tile, s);
    }
  }

  int it = 0;
  for (int64_t tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++it) {
    const int s = it & 1;
    const uint32_t stage = sbase + (uint32_t)(s * kQtStageBytes);
    const bool ok = mbar_wait_bounded(bar0 + 8u * s, (uint32_t)((it >> 1) & 1), pa.wait_limit_ns, never);
    if (!__syncthreads_and(ok)) {
      if (tid == 0) {
        atomicOr(&g_quant_error, 1u);
        // tile 1's copy, issued at the start, must land before the CTA exits
        if (it == 0 && tile + gridDim.x < num_tiles)
          mbar_wait_bounded(bar0 + 8u, 0u, pa.wait_limit_ns, never);
      }
      break;
    }
    const bool in_a = tile < na;
    uint4 v[4];
    uint32_t cm[4];  // MXFP8: the column maxima of this lane group's 32 rows
    if (in_a) qt_load_reduce<MODE_A>(stage, v, cm, warp, lane, rot, rowred, colred);
    else qt_load_reduce<MODE_B>(stage, v, cm, warp, lane, rot, rowred, colred);
    __syncthreads();  // partial maxima visible; the input tile is in registers
    if (tid == 0 && it >= 1) {
      // the other stage held the previous tile's outputs: once their stores
      // have read it, it takes the next tile
      bulk_wait_read_all();
      const int64_t next = tile + gridDim.x;
      if (next < num_tiles) issue(next, s ^ 1);
    }

    if (in_a)
      qt_scale_store<MODE_A>(&tmap_qrow_a, &tmap_qcol_a, pa, tile, stage, v, cm, tid, warp, lane, rot, sel_e,
                             sel_o, sbase, rowred, colred);
    else
      qt_scale_store<MODE_B>(&tmap_qrow_b, &tmap_qcol_b, pb, tile - na, stage, v, cm, tid, warp, lane, rot, sel_e,
                             sel_o, sbase, rowred, colred);
  }
  if (tid == 0) bulk_wait_all();  // stores complete before the CTA exits
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

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool quant_tile_supported(const void* x, int64_t ldx, const void* q_row, int64_t ldq_row, const void* q_col,
                          int64_t ldq_col) {
  if (!aligned16(x) || ldx % 8 != 0 || qt_encode_fn() == nullptr) return false;
  if (q_row && (!aligned16(q_row) || ldq_row % 16 != 0)) return false;  // TMA store: 16-byte rows
  if (q_col && (!aligned16(q_col) || ldq_col % 16 != 0)) return false;
  return true;
}

// u8 matrix [rows, inner] with row stride ld bytes, written by 128 x 128-byte boxes.
static bool make_store_map(CUtensorMap* m, void* base, int64_t inner, int64_t rows, int64_t ld, bool swizzle) {
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld};
  cuuint32_t box[2] = {128, 128};
  cuuint32_t elem[2] = {1, 1};
  return qt_encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, elem,
                        CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MODE_A, int MODE_B>
static cudaError_t run_tile(const CUtensorMap (&ma)[3], const CUtensorMap (&mb)[3], const TileQuantParams& pa,
                            const TileQuantParams& pb, int64_t grid, cudaStream_t st) {
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [] {
    attr = cudaFuncSetAttribute(quant_tile_kernel<MODE_A, MODE_B>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kQtSmemBytes);
  });
  if (attr != cudaSuccess) return attr;
  const int64_t bytes_read = 2 * (pa.T * pa.C + (pb.num_tiles > 0 ? pb.T * pb.C : 0));
  TileQuantParams qa = pa, qb = pb;
  qa.pdl = qb.pdl = pdl_for_quant(bytes_read);
  return launch_kernel(qa.pdl != 0, quant_tile_kernel<MODE_A, MODE_B>, (unsigned)grid, kQtThreads, kQtSmemBytes, st,
                       ma[0], ma[1], ma[2], mb[0], mb[1], mb[2], qa, qb);
}

// Tensor maps (input, q_row store, q_col store) and parameters of one input.
static bool prepare_tile(const QuantTileArgs& a, CUtensorMap (&m)[3], TileQuantParams* p) {
  memset(m, 0, sizeof(m));
  cuuint64_t dims[2] = {(cuuint64_t)a.C, (cuuint64_t)a.T};
  cuuint64_t strides[1] = {(cuuint64_t)a.ldx * 2};
  cuuint32_t box[2] = {64, 128};
  cuuint32_t elem[2] = {1, 1};
  if (qt_encode_fn()(&m[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(a.x), dims, strides, box, elem,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  const int64_t C_al = a.C & ~(int64_t)15, T_al = a.T & ~(int64_t)15;
  if (a.q_row && C_al > 0 && !make_store_map(&m[1], a.q_row, C_al, a.T, a.ldq_row, true)) return false;
  if (a.q_col && T_al > 0 && !make_store_map(&m[2], a.q_col, T_al, a.C, a.ldq_col, false)) return false;
  p->T = a.T;
  p->C = a.C;
  p->q_row = a.q_row;
  p->ldq_row = a.ldq_row;
  p->q_col = a.q_col;
  p->ldq_col = a.ldq_col;
  p->C_al = C_al;
  p->T_al = T_al;
  p->s_row = a.s_row;
  p->lds_row = a.lds_row;
  p->s_col = a.s_col;
  p->lds_col = a.lds_col;
  p->has_q_row = a.q_row != nullptr;
  p->has_q_col = a.q_col != nullptr;
  p->tiles_c = cdiv(a.C, 128);
  p->num_tiles = cdiv(a.T, 128) * p->tiles_c;
  p->wait_limit_ns = kWaitLimitNs;
  p->pdl = 1;
  p->e_row = a.e_row;
  p->lde_row = a.lde_row;
  p->e_col = a.e_col;
  p->lde_col = a.lde_col;
  return true;
}

cudaError_t launch_quant_tile(const QuantTileArgs& a, int num_sms, cudaStream_t st) {
  CUtensorMap m[3];
  TileQuantParams p;
  if (!prepare_tile(a, m, &p)) return cudaErrorInvalidValue;
  TileQuantParams none = p;  // no second input
  none.num_tiles = 0;
  const int64_t grid = qt_grid(p.num_tiles, num_sms);
  switch (a.mode) {
    case kTileRow: return run_tile<kTileRow, kTileRow>(m, m, p, none, grid, st);
    case kTileCol: return run_tile<kTileCol, kTileCol>(m, m, p, none, grid, st);
    case kTileRow | kTileCol: return run_tile<kTileRow | kTileCol, kTileRow | kTileCol>(m, m, p, none, grid, st);
    case kTileScale: return run_tile<kTileScale, kTileScale>(m, m, p, none, grid, st);
    case kTileMx | kTileRow | kTileCol:
      return run_tile<kTileMx | kTileRow | kTileCol, kTileMx | kTileRow | kTileCol>(m, m, p, none, grid, st);
    case kTileMx | kTileRow: return run_tile<kTileMx | kTileRow, kTileMx | kTileRow>(m, m, p, none, grid, st);
    case kTileMx | kTileCol: return run_tile<kTileMx | kTileCol, kTileMx | kTileCol>(m, m, p, none, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_quant_tile_pair(const QuantTileArgs& a, const QuantTileArgs& b, int num_sms, cudaStream_t st) {
  if (b.mode != kTileScale) return cudaErrorInvalidValue;
  CUtensorMap ma[3], mb[3];
  TileQuantParams pa, pb;
  if (!prepare_tile(a, ma, &pa) || !prepare_tile(b, mb, &pb)) return cudaErrorInvalidValue;
  const int64_t grid = qt_grid(pa.num_tiles + pb.num_tiles, num_sms);
  switch (a.mode) {
    case kTileRow | kTileCol: return run_tile<kTileRow | kTileCol, kTileScale>(ma, mb, pa, pb, grid, st);
    case kTileRow: return run_tile<kTileRow, kTileScale>(ma, mb, pa, pb, grid, st);
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
