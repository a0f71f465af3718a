// Launch geometry and index arithmetic of the kernels, as __host__ __device__
// functions so that the host can replay exactly what a launch would touch
// (the scale-bounds test idea of "Mask a_s/b_s scale loads in blockwise FP8
// training GEMM kernels": check the offs -> index arithmetic on tail shapes
// without running the kernel).
#pragma once

#include <stdint.h>

#ifndef BFP8_HD
#define BFP8_HD __host__ __device__ __forceinline__
#endif

namespace bfp8 {

constexpr int kBlock = 128;            // group / tile edge (block_size = 128)
constexpr float kE4m3Max = 448.0f;     // FP8_MAX of float8_e4m3fn
constexpr float kAmaxFloor = 1e-12f;   // keeps an all-zero group's scale finite

BFP8_HD int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// ---------------------------------------------------------------------------
// quant_lhs, row-major input: 16 threads per 1x128 group, 8 elements each.
// ---------------------------------------------------------------------------
constexpr int kRowThreads = 256;       // threads per CTA
constexpr int kRowUnroll = 4;          // groups per half-warp per iteration

struct RowChunk {
  int64_t m, k;  // first element of the thread's 8-element chunk
};

// Group g (row-major over [M, Kb]) and the thread's lane within its half-warp.
BFP8_HD RowChunk row_chunk(int64_t g, int lane16, int64_t Kb) {
  RowChunk c;
  c.m = g / Kb;
  c.k = (g % Kb) * kBlock + (int64_t)lane16 * 8;
  return c;
}

// Group processed by half-warp `hw` (of `nhw`) in iteration `it`, unroll slot `u`.
BFP8_HD int64_t row_group(int64_t hw, int64_t nhw, int64_t it, int u) {
  return hw + (it * kRowUnroll + u) * nhw;
}

// ---------------------------------------------------------------------------
// Column groups (128 consecutive rows of one column) written transposed:
// CTA tile of 128 rows x 64 columns; warp w owns columns 8w..8w+7, lane l owns
// rows 4l..4l+3 of the tile.  Used by quant_lhs(x_transposed) and quant_rhs.
// ---------------------------------------------------------------------------
constexpr int kColThreads = 256;
constexpr int kColTileT = 128;   // rows (the grouped dimension)
constexpr int kColTileC = 64;    // columns

struct ColTile {
  int64_t t0, c0;
};
BFP8_HD ColTile col_tile(int64_t block, int64_t C) {
  const int64_t nct = cdiv(C, kColTileC);
  ColTile t;
  t.t0 = (block / nct) * kColTileT;
  t.c0 = (block % nct) * kColTileC;
  return t;
}
// Element (row t, column c) of value (i, j) held by (warp, lane).
BFP8_HD int64_t col_elem_t(const ColTile& tile, int lane, int i) { return tile.t0 + 4 * lane + i; }
BFP8_HD int64_t col_elem_c(const ColTile& tile, int warp, int j) { return tile.c0 + 8 * warp + j; }
// Store phase: 16-byte chunk `ch` (0..511) of the transposed 64 x 128-byte tile.
BFP8_HD int64_t col_store_c(const ColTile& tile, int ch) { return tile.c0 + ch / 8; }
BFP8_HD int64_t col_store_t(const ColTile& tile, int ch) { return tile.t0 + (ch % 8) * 16; }

// ---------------------------------------------------------------------------
// quant_weight: one CTA per 128x128 tile; warp w owns 8-column chunks w and
// w+8, lane l owns rows 4l..4l+3.
// ---------------------------------------------------------------------------
constexpr int kWThreads = 256;

struct WTile {
  int64_t nb, kb;
};
BFP8_HD WTile w_tile(int64_t block, int64_t Kb) {
  WTile t;
  t.nb = block / Kb;
  t.kb = block % Kb;
  return t;
}
BFP8_HD int64_t w_elem_n(const WTile& t, int lane, int i) { return t.nb * kBlock + 4 * lane + i; }
BFP8_HD int64_t w_elem_k(const WTile& t, int chunk, int j) { return t.kb * kBlock + 8 * chunk + j; }
// transposed store phase: 16-byte chunk `ch` (0..1023) of the 128 x 128-byte qt tile
BFP8_HD int64_t w_tstore_k(const WTile& t, int ch) { return t.kb * kBlock + ch / 8; }
BFP8_HD int64_t w_tstore_n(const WTile& t, int ch) { return t.nb * kBlock + (ch % 8) * 16; }

// ---------------------------------------------------------------------------
// TMA-staged tile quantisation: persistent CTAs (two per SM, 16 warps each)
// over 128x128 tiles of a [T, C] input, tile index = blockIdx.x + k * gridDim.x,
// walked C-fastest.  Row pass: 16 threads per tile row, thread lane16 owns
// columns 8*lane16..+7, pass ps (0..3) of warp w covers row 32*ps + 2*w + half.
// Column pass: warp w owns 8-column chunk w, lane l owns rows l + 32*i.  The
// transposed tile is stored as 16-byte chunks: chunk ch -> column ch/8,
// rows 16*(ch%8)..+15.
// ---------------------------------------------------------------------------
constexpr int kQtThreads = 512;
constexpr int kQtRowPasses = 4;     // tile rows per thread in the row pass
constexpr int kQtColChunks = 1;     // 8-column chunks per warp in the column pass
constexpr int kQtCtasPerSm = 2;

BFP8_HD int64_t qt_grid(int64_t num_tiles, int num_sms) {
  const int64_t cap = (int64_t)kQtCtasPerSm * num_sms;
  return num_tiles < cap ? num_tiles : cap;
}
BFP8_HD int64_t qt_tile_t0(int64_t tile, int64_t tiles_c) { return (tile / tiles_c) * 128; }
BFP8_HD int64_t qt_tile_c0(int64_t tile, int64_t tiles_c) { return (tile % tiles_c) * 128; }
BFP8_HD int qt_rowpass_row(int ps, int warp, int half) { return 32 * ps + 2 * warp + half; }
BFP8_HD int qt_rowpass_col(int lane16) { return 8 * lane16; }
BFP8_HD int qt_colpass_chunk(int warp, int h) { return warp + 16 * h; }
BFP8_HD int qt_colpass_row(int lane, int i) { return lane + 32 * i; }
BFP8_HD int qt_store_col(int ch) { return ch / 8; }
BFP8_HD int qt_store_row(int ch) { return 16 * (ch % 8); }

// ---------------------------------------------------------------------------
// GEMM: persistent CTAs over BM x BN output tiles.
// ---------------------------------------------------------------------------
constexpr int kBM = 128;
constexpr int kBK = 128;          // one scale block per pipeline stage
constexpr int kGroupM = 16;       // tile rasterisation: bands of 16 M-blocks
constexpr size_t kGemmFlagBytes = 4096;  // stream-K workspace: per-CTA flags, then partial tiles

struct GemmTile {
  int64_t m0, n0;
};

// Output tile of linear tile index `t`: tiles are walked N-fastest inside
// bands of kGroupM M-blocks so that concurrently running CTAs share A rows
// and B columns in L2.
BFP8_HD GemmTile gemm_tile(int64_t t, int64_t num_m, int64_t num_n, int bn) {
  const int64_t per_band = (int64_t)kGroupM * num_n;
  const int64_t band = t / per_band;
  const int64_t first_m = band * kGroupM;
  const int64_t rows = (num_m - first_m) < kGroupM ? (num_m - first_m) : kGroupM;
  const int64_t r = t % per_band;
  GemmTile g;
  g.m0 = (first_m + r % rows) * kBM;
  g.n0 = (r / rows) * bn;
  return g;
}

// Work of one persistent CTA, as segments (tile, K-blocks [kb0, kb1)).
// Tile-parallel: tiles cta, cta + grid, ... each with all K-blocks.
// Stream-K: the units (tile, K-block) in tile-major order are split into
// `grid` equal contiguous ranges; a CTA's range may begin inside one tile
// (finishing it: kb0 > 0, kb1 = Kb) and end inside another (starting it:
// kb0 = 0, kb1 < Kb).  The host enables stream-K only when every range holds
// at least Kb units, so a tile is split between at most two CTAs.
struct GemmSeg {
  int64_t tile;
  int kb0, kb1;
};
struct GemmWork {
  int64_t a, b, step;  // tile-parallel: next tile, tile count, stride; stream-K: next unit, end, Kb
  bool sk;
  BFP8_HD void init(bool stream_k, int64_t cta, int64_t grid, int64_t num_tiles, int64_t Kb) {
    sk = stream_k;
    if (sk) {
      const int64_t units = num_tiles * Kb;
      a = units * cta / grid;
      b = units * (cta + 1) / grid;
      step = Kb;
    } else {
      a = cta;
      b = num_tiles;
      step = grid;
    }
  }
  BFP8_HD bool next(GemmSeg& s, int64_t Kb) {
    if (a >= b) return false;
    if (sk) {
      s.tile = a / Kb;
      s.kb0 = (int)(a % Kb);
      const int64_t left = b - a;
      s.kb1 = (int)((Kb - s.kb0) < left ? Kb : s.kb0 + left);
      a += s.kb1 - s.kb0;
    } else {
      s.tile = a;
      s.kb0 = 0;
      s.kb1 = (int)Kb;
      a += step;
    }
    return true;
  }
};

// Epilogue warp e (0-based among the epilogue warps; CTA warp id = e + 4):
// tensor-memory lane quarter = CTA warp id % 4, column half = e / 4.
BFP8_HD int epi_row(int e, int lane) { return 32 * ((e + 4) % 4) + lane; }
BFP8_HD int epi_col0(int e) { return 128 * (e / 4); }

}  // namespace bfp8
