// Internal launchers (host side) shared by the C-ABI translation unit.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/bfp8.h"

namespace bfp8 {

constexpr uint64_t kWaitLimitNs = 4000000000ull;  // 4 s per wait: far above any legitimate stall

// Sets the message bfp8_last_error() returns on the calling thread.
void set_last_error(const char* msg);

cudaError_t launch_quant_rows(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q,
                              int64_t ldq, float* s, int64_t lds, int num_sms, cudaStream_t st);
int64_t quant_rows_grid(int64_t M, int64_t K, int num_sms);
cudaError_t launch_quant_cols(const uint16_t* x, int64_t T, int64_t C, int64_t ldx, uint8_t* qT,
                              int64_t ldq, float* s, int64_t lds, cudaStream_t st);
cudaError_t launch_quant_weight(const uint16_t* w, int64_t N, int64_t K, int64_t ldw, uint8_t* q,
                                int64_t ldq, uint8_t* qt, int64_t ldqt, float* s, int64_t lds,
                                cudaStream_t st);
cudaError_t launch_cast(const float* x, int64_t n, uint8_t* q, int num_sms, cudaStream_t st);

// TMA-staged tile quantisation (quant_tile.cu): which outputs one read makes.
// kQuantTileMx: MXFP8 instead (blocks of 32, E8M0 exponents): with kQuantTileRow the dim0
// cast (q_row, e_row), with kQuantTileCol the transposed dim1 cast (q_col, e_col)
enum : int { kQuantTileRow = 1, kQuantTileCol = 2, kQuantTileScale = 4, kQuantTileMx = 8 };
// x: 16-byte aligned, ldx % 8 == 0; each non-null output: 16-byte aligned, ld % 16 == 0
bool quant_tile_supported(const void* x, int64_t ldx, const void* q_row, int64_t ldq_row, const void* q_col,
                          int64_t ldq_col);
// One input of the tile quantisation kernel (quant_tile.cu).
struct QuantTileArgs {
  int mode;  // kQuantTileRow, kQuantTileCol, both, or kQuantTileScale
  const uint16_t* x;
  int64_t T, C, ldx;
  uint8_t* q_row;
  int64_t ldq_row;
  float* s_row;
  int64_t lds_row;
  uint8_t* q_col;
  int64_t ldq_col;
  float* s_col;
  int64_t lds_col;
  uint8_t* e_row;  // kQuantTileMx: biased exponents, e_row[t * lde_row + c / 32]
  int64_t lde_row;
  uint8_t* e_col;  //                                  e_col[c * lde_col + t / 32]
  int64_t lde_col;
};
cudaError_t launch_quant_tile(const QuantTileArgs& a, int num_sms, cudaStream_t st);
// x's 1x128 groups (kQuantTileRow), or both its forms (kQuantTileRow |
// kQuantTileCol), and a weight's tiles (kQuantTileScale) in one launch.
cudaError_t launch_quant_tile_pair(const QuantTileArgs& x, const QuantTileArgs& w, int num_sms, cudaStream_t st);
cudaError_t quant_read_errors(uint32_t* out);

enum SbMode : int { kSbTile = 0, kSbTileT = 1, kSbCol = 2 };

struct GemmArgs {
  const void* qa;
  int64_t lda;
  const float* sa;
  int64_t ldsa;
  const void* qb;
  int64_t ldb;
  const float* sb;
  int64_t ldsb;
  int sb_mode;
  void* c;
  int64_t ldc;
  int64_t M, N, K;
};

// Returns cudaSuccess or the launch error; *msg gets a static description of
// a host-side failure (tensor-map encoding) when the return is not success.
cudaError_t launch_gemm(const GemmArgs& a, int num_sms, cudaStream_t st, const char** msg,
                        uint64_t wait_limit_ns = kWaitLimitNs, int debug_stall = 0);
// Tile width the launcher picks for an M x N output (col_scales: the 1x128 x
// 128x1 GEMM), and the grid it uses.
int gemm_pick_bn(int64_t M, int64_t N, bool col_scales, int num_sms);
int64_t gemm_grid(int64_t M, int64_t N, int bn, int num_sms);
// Grouped (mixture-of-experts) GEMM, kind kGroupRows or kGroupRed (index.cuh).
//   kGroupRows: g.qa [M_total, K] token rows, C [M_total, N]; expert e's rows
//               offs[e] .. offs[e+1] against its B: rows e * b_row_step of the B
//               map (b_row_step = N: forward) or K columns e * b_k_step
//               (b_k_step = K: input gradient, B map [N, E*K]); its b_s at
//               g.sb + e * sb_step.  g.M is unused.
//   kGroupRed:  g.qa [M, T], g.qb [N, T] (T = M_total tokens), C_e [M, N] at
//               g.c + e * c_step; expert e reduces over tokens offs[e] ..
//               offs[e+1] (offs[e] % 128 == 0).  g.K is unused.
// offs is a device array of E + 1 int32 (1 <= E <= kMaxGroups).
struct GemmGroupArgs {
  GemmArgs g;
  int kind;
  const int32_t* offs;
  int64_t E;
  int64_t M_total;
  int64_t b_row_step, b_k_step;
  int64_t sb_step, c_step;
};
cudaError_t launch_gemm_grouped(const GemmGroupArgs& a, int num_sms, cudaStream_t st, const char** msg);
// The forward GEMM (1x128 x 128x128) with A quantised inside the kernel: x
// bf16 [M, K] (ldx elements, ldx % 8 == 0, 16-byte aligned), qb the weight's
// e4m3 bytes [N, K] (ldb % 16 == 0), sb its tile scales [Nb, Kb] (row-major,
// ldsb), c bf16 [M, N].
struct GemmXqArgs {
  const void* x;
  int64_t ldx;
  const void* qb;
  int64_t ldb;
  const float* sb;
  int64_t ldsb;
  void* c;
  int64_t ldc;
  int64_t M, N, K;
};
cudaError_t launch_gemm_xq(const GemmXqArgs& a, int num_sms, cudaStream_t st, const char** msg);
// The weight-gradient GEMM (1x128 x 128x1) with its rhs quantised 128x1 inside
// the kernel: qa e4m3 [M, K] (lda % 16 == 0), sa its 1x128 scales sa[kb*ldsa + m],
// x bf16 [K, N] row-major (ldx elements, ldx % 8 == 0, 16-byte aligned), c bf16 [M, N].
struct GemmWxqArgs {
  const void* qa;
  int64_t lda;
  const float* sa;
  int64_t ldsa;
  const void* x;
  int64_t ldx;
  void* c;
  int64_t ldc;
  int64_t M, N, K;
};
cudaError_t launch_gemm_wgrad_xq(const GemmWxqArgs& a, int num_sms, cudaStream_t st, const char** msg);

// Reads and clears the device error word of the GEMM kernels (synchronous).
cudaError_t gemm_read_errors(uint32_t* out);

// The linear forward (api.cu), shared with the entry that keeps its scratch
// in a library-owned array (noalloc.cu): the bytes its scratch needs, the
// sm_103a check of the current device (SM count via *sms), and the forward's
// launches into scratch at `base` (256-byte aligned, linear_fwd_scratch_bytes
// long) once the arguments are validated.
size_t linear_fwd_scratch_bytes(int64_t M, int64_t N, int64_t K);
bfp8_status check_current_device(int* sms);
bfp8_status linear_fwd_into(const void* x, const void* w, void* y, int64_t M, int64_t N, int64_t K, uint8_t* base,
                            int sms, bfp8_stream_t stream);

}  // namespace bfp8
