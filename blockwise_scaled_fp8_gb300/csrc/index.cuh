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
// walked C-fastest.  Warp w owns the 8-column chunk w of the tile, lane l the
// rows 4l..4l+3.  Scales: thread tid joins the maximum of row / column
// qt_scale_group(tid) of the tile (four threads each), and the thread with
// qt_scale_writer(tid) stores its scale.  Codes leave by one TMA store per
// output and tile (a 128 x 128-byte box, clipped to the tensor).
// ---------------------------------------------------------------------------
// Programmatic dependent launch pays where kernels are short (the next
// kernel's set-up hides behind the end of the one before: a 2048 x 4096 x
// 4096 linear step 1% faster, small quantise-then-GEMM pairs up to 6%) and
// costs 1-3% in a step of long ones (8192 tokens x 4096 x 4096, MLP-up
// 16384 x 14336 x 4096, their MoE form: measured without it 1.3%, 3.0% and
// 2.1% faster).  GEMMs of at least 2^37 FLOPs and quantisations reading at
// least 64 MiB of bf16 are launched without it.
BFP8_HD bool pdl_for_gemm(int64_t M, int64_t N, int64_t K) {
  return 2.0 * (double)M * (double)N * (double)K < 137438953472.0;
}
BFP8_HD bool pdl_for_quant(int64_t bytes_read) { return bytes_read < ((int64_t)64 << 20); }

constexpr int kQtThreads = 512;
constexpr int kQtCtasPerSm = 2;

BFP8_HD int64_t qt_grid(int64_t num_tiles, int num_sms) {
  const int64_t cap = (int64_t)kQtCtasPerSm * num_sms;
  return num_tiles < cap ? num_tiles : cap;
}
BFP8_HD int64_t qt_tile_t0(int64_t tile, int64_t tiles_c) { return (tile / tiles_c) * 128; }
BFP8_HD int64_t qt_tile_c0(int64_t tile, int64_t tiles_c) { return (tile % tiles_c) * 128; }
BFP8_HD int qt_scale_group(int tid) { return tid >> 2; }
BFP8_HD bool qt_scale_writer(int tid) { return (tid & 3) == 0; }

// ---------------------------------------------------------------------------
// GEMM: persistent CTAs over BM x BN output tiles.
// ---------------------------------------------------------------------------
constexpr int kBM = 128;
constexpr int kBK = 128;          // one scale block per pipeline stage
constexpr int kGroupM = 16;       // tile rasterisation: bands of 16 M-blocks

struct GemmTile {
  int m0, n0;
};

// Output tile of linear tile index `t`: tiles are walked N-fastest inside
// bands of kGroupM M-blocks so that concurrently running CTAs share A rows
// and B columns in L2.  (Sizes are below 2^31; the host checks.)
BFP8_HD GemmTile gemm_tile(int t, int num_m, int num_n, int bn) {
  const int per_band = kGroupM * num_n;
  const int band = t / per_band;
  const int first_m = band * kGroupM;
  const int rows = (num_m - first_m) < kGroupM ? (num_m - first_m) : kGroupM;
  const int r = t % per_band;
  GemmTile g;
  g.m0 = (first_m + r % rows) * kBM;
  g.n0 = (r / rows) * bn;
  return g;
}

// Grouped (mixture-of-experts) GEMMs.  kGroupRows (forward, input gradient):
// expert e owns token rows offs[e] .. offs[e+1] of A and C, and its tiles are
// gemm_tile(t - start[e], cdiv(rows of e, 128), num_n) for start[e] <= t <
// start[e+1], start[] the running sum of the experts' tile counts.  kGroupRed
// (weight gradient): expert e reduces over tokens offs[e] .. offs[e+1]; each
// expert has num_m x num_n tiles, expert e the tiles e*num_m*num_n onwards.
enum : int { kGroupNone = 0, kGroupRows = 1, kGroupRed = 2 };
constexpr int kMaxGroups = 1024;
// experts a grouped GEMM can have and still take the staged TMA-store epilogue
// (its expert table shares shared memory with the staging buffers)
constexpr int kStageGroups = 256;

// The expert holding tile t: the largest e < E with start[e] <= t, given
// start non-decreasing and start[0] <= t < start[E] (empty experts skipped).
BFP8_HD int group_of_tile(const int* start, int E, int t) {
  int lo = 0, hi = E;  // start[lo] <= t < start[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (start[mid] <= t) lo = mid;
    else hi = mid;
  }
  return lo;
}

// Promotion / epilogue warp e (0-based, CTA warp id = e + 4) of `ew` (8 or
// 16): tensor-memory lane quarter e % 4 (the quarter a warp may access is its
// CTA warp id % 4), column block e / 4 of epi_cols(bn, ew) columns.  The
// 1x128 x 128x128 GEMMs use 8 promotion warps (16 with 224- and 256-column
// tiles), the 1x128 x 128x1 GEMM 16.
BFP8_HD int gemm_epi_warps(bool col_scales, int bn) { return (col_scales || bn >= 224) ? 16 : 8; }
// Rows of A one pipeline stage loads: 16 for the 64-column tiles of problems
// of at most 16 rows, else 128.  With 16, only the promotion warps of lane
// quarter 0 (e % 4 == 0) hold rows of the problem; the others store nothing.
BFP8_HD int gemm_a_rows(int64_t M, int bn) { return bn == 64 && M <= 16 ? 16 : kBM; }
// Small-M GEMMs (at most 32 rows, tile-scale modes) whose 128-column tiles
// fit in one wave take the operand-swapped kernel: W as the MMA's 128-row A,
// the rows of A as its B (R = 16 or 32 rows: smallm_rows), and each tile's
// K-blocks split over a cluster of CTAs.  Split s of S takes K-blocks
// [smallm_kb_lo(s), smallm_kb_lo(s + 1)).
BFP8_HD bool smallm_eligible(int64_t M, int64_t N, bool col_scales, int num_sms) {
  return M >= 1 && M <= 32 && !col_scales && (N + kBM - 1) / kBM <= num_sms;
}
BFP8_HD int smallm_rows(int64_t M) { return M <= 16 ? 16 : 32; }
BFP8_HD int smallm_kb_lo(int s, int splits, int Kb) { return (int)((int64_t)s * Kb / splits); }
BFP8_HD int epi_row(int e, int lane) { return 32 * (e % 4) + lane; }
BFP8_HD int epi_cols(int bn, int ew) { return bn / (ew / 4); }
BFP8_HD int epi_col0(int e, int bn, int ew) { return epi_cols(bn, ew) * (e / 4); }
// Epilogue stores: G x G blocks of 16-byte (8-column) chunks are transposed
// within groups of G lanes, G = the warp's chunk count epi_cols / 8 rounded up
// to a power of two, at most 8; in pass sg (of epi_passes), lane (grp =
// lane / G, pos = lane % G) stores chunk G*sg + pos of tile rows
// 32*(e%4) + G*grp + i, i < G, if that chunk exists (a share of 56 columns has
// 7 chunks: the eighth position of each group stores nothing).
BFP8_HD int epi_chunks(int bn, int ew) { return epi_cols(bn, ew) / 8; }
BFP8_HD int epi_group(int bn, int ew) {
  const int c = epi_chunks(bn, ew);
  return c > 4 ? 8 : c > 2 ? 4 : c;
}
BFP8_HD int epi_passes(int bn, int ew) { return (epi_chunks(bn, ew) + epi_group(bn, ew) - 1) / epi_group(bn, ew); }
BFP8_HD int epi_store_row(int e, int lane, int i, int G) { return 32 * (e % 4) + G * (lane / G) + i; }
BFP8_HD int epi_store_col(int e, int lane, int sg, int G, int bn, int ew) {
  return epi_col0(e, bn, ew) + 8 * (G * sg + lane % G);
}

}  // namespace bfp8
