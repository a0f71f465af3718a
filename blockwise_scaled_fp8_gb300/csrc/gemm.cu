// Blockwise-scaled FP8 GEMMs on the 5th-generation tensor cores (sm_103a).
//
// C[m,n] = sum_kb a_s[m,kb] * b_s(n,kb) * P_kb[m,n],  P_kb = the e4m3 x e4m3
// partial product of one 128-wide K-block ("Mask a_s/b_s scale loads in
// blockwise FP8 training GEMM kernels", Summary: 1x128 x 128x128 and
// 1x128 x 128x1 kernels with per-tile a_s/b_s; Fix: scale loads masked to
// offs_m < M and offs_n < N like every other load and the output store).
//
// Design (one persistent CTA per SM, warp-specialised):
//   warp 0      TMA producer: 128x128-byte A and BNx128-byte B tiles of one
//               K-block per stage, 128-byte swizzled, into an S-stage ring.
//   warps 1, 3  MMA issuers: 4 x tcgen05.mma.kind::f8f6f4 (K = 32 each) per
//               K-block into one of two tensor-memory partial buffers, then
//               tcgen05.commit to release the smem stage and publish the partial.
//               Warp 1 takes the even K-block steps (buffer 0), warp 3 the odd
//               ones (buffer 1): a thread issuing MMAs blocks while the tensor
//               pipe drains its short queue, so with one issuer the pipe sat
//               idle during every wait for the next buffer and stage.
//   warp 2      scale loader: per K-block, a_s of the tile's 128 rows and b_s
//               (BN column scales, or the tile scales) into a shared-memory
//               ring of two slots of four K-blocks each, with cp.async, running
//               ahead of the promotion so that no promotion warp waits on a
//               global load; one wait and one release per four K-blocks.
//   warps 4..   promotion/epilogue, EW/4 per tensor-memory lane quarter, each
//               owning 32 rows x BN/(EW/4) columns of the tile: tcgen05.ld the
//               K-block's fp32 partial, release the tensor-memory buffer,
//               acc += (a_s*b_s) * partial in registers; at tile end round to
//               bf16, transpose 16-byte chunks across lanes with shuffles and
//               store whole row segments (only rows m < M, columns n < N).
// The two tensor-memory buffers let the promotion of K-block kb overlap the
// MMAs of K-block kb+1.  Tails: TMA zero-fills rows/columns outside M, N, K;
// scale copies are zero-filled past M / N; the epilogue store is masked.
// Every mbarrier wait is bounded in time; a timeout records an error bit,
// lets every role leave its loop, waits for its own copies/MMAs in flight and
// frees tensor memory before the CTA exits.
// gemm_grouped_kernel runs the same pipeline for the mixture-of-experts forms
// (token rows or the reduction grouped by expert; see GemmJob).
#include <cudaTypedefs.h>

#include <string.h>

#include <mutex>

#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace bfp8 {

static __device__ uint32_t g_gemm_error;

enum : uint32_t {
  kErrWaitEmpty = 1u << 0,      // producer: a smem stage was never released
  kErrWaitFull = 1u << 1,       // MMA: a stage's TMA bytes never landed
  kErrWaitTmemEmpty = 1u << 2,  // MMA: a tensor-memory buffer was never released
  kErrWaitTmemFull = 1u << 3,   // epilogue: a partial product never arrived
  kErrWaitDrain = 1u << 4,      // teardown: MMAs or copies in flight never finished
  kErrWaitScale = 1u << 5,      // scale ring: a slot was never filled / released
  kErrGroupOffsets = 1u << 6,   // grouped GEMM: expert offsets decreasing, out of range or misaligned
};

struct GemmParams {
  const float* sa;
  int64_t ldsa;
  const float* sb;
  int64_t ldsb;
  uint16_t* c;
  int64_t ldc;
  int64_t M, N, K;
  int num_m, num_n, num_tiles, Kb, Nb;  // below 2^31, as is num_tiles * Kb (checked by the host)
  int c_vec;   // 16-byte output stores allowed (ldc % 8 == 0, c 16-byte aligned)
  int sa_vec;  // 16-byte a_s copies allowed (ldsa % 4 == 0, sa 16-byte aligned)
  int sb_vec;  // 16-byte b_s copies allowed (ldsb % 4 == 0, sb 16-byte aligned)
  uint64_t wait_limit_ns;
  int debug_stall;  // test hook: the promotion warps wait on a barrier nothing arrives on
  int c_tma = 0;    // (dense kernel, 256-column tiles) the epilogue stores through the C tensor map
  int pdl = 1;      // launched with programmatic dependent launch: let the next kernel start early
};

// What the grouped (mixture-of-experts) forms add.  A separate kernel
// parameter: growing GemmParams alone changed the dense kernels' register
// allocation (more spills in the weight-gradient form).
struct GemmGroupParams {
  const int32_t* offs;  // [E+1] token offsets of the experts (device memory)
  int E;
  int M_total;          // kGroupRows: token rows of A and C;  kGroupRed: token extent of A and B
  int b_row_step;       // per expert: first row of its B in the B map (forward)
  int b_k_step;         // per expert: first K column of its B in the B map (input gradient)
  int64_t sb_step;      // per expert: offset of its b_s (elements)
  int64_t c_step;       // per expert: offset of its C (elements; weight gradient)
  int c_rows = 0;       // c_step / ldc where the epilogue stores through the C map (weight gradient)
};

// One output tile's work: where its operands sit in the two tensor maps, its
// K-blocks, and where its scales and outputs are.
struct GemmJob {
  int a_row, b_row;  // first rows of the tile in the A and B maps
  int a_k, b_k;      // first K columns (elements) in the A and B maps
  int kb_s;          // first K-block index in a_s / b_s
  int kbn;           // K-blocks of the tile (0: the tile is all zeros)
  int rows;          // valid rows from a_row (>= 1; rows past 128 belong to other tiles)
  int n0;            // first output column
  int e;             // expert (b_s at sb + e * sb_step)
  int64_t c_off;     // element offset of the output C[first row][n0]
};

constexpr int gcd_c(int a, int b) { return b ? gcd_c(b, a % b) : a; }

template <int BN, int STAGES, int EW, int A_ROWS = 128>
struct GemmCfg {
  static constexpr int kEpiWarps = EW;
  static constexpr int kCols = BN / (EW / 4);  // tile columns per promotion warp
  static constexpr int kThreads = 128 + 32 * EW;
  // Register split: the control warpgroup drops to kCtrlRegs and the promotion
  // warpgroups rise to kEpiRegs, within what the launch holds (threads x
  // registers per thread at launch, 65536 / threads rounded down to 8):
  //   EW = 16: 128*56 + 512*104 = 60416 <= 640*96;  EW = 8: 128*40 + 256*224 = 62464 <= 384*168.
  // (With 40 the weight-gradient form's control warps spilled.)
  static constexpr int kLaunchRegs = (65536 / kThreads) / 8 * 8;
  static constexpr int kCtrlRegs = EW == 16 ? 56 : 40;
  static constexpr int kEpiRegs = EW == 16 ? 104 : 224;
  static_assert(128 * kCtrlRegs + 32 * EW * kEpiRegs <= kThreads * kLaunchRegs, "register split");
  static constexpr int kABytes = kBM * kBK;  // what one MMA reads of A: 128 rows x 128 B
  // A_ROWS = 16 (problems of at most 16 rows): A stages hold 16-row boxes and
  // sit 2 KiB apart; an MMA still reads 128 rows from its stage's start, and
  // rows 16..127 (bytes of the following stages) only feed accumulator rows
  // >= M, which are never read.  The room saved holds more stages of B, the
  // operand streamed from DRAM.
  static_assert(A_ROWS == 128 || A_ROWS == 16, "A box rows");
  static constexpr int kAStride = A_ROWS == 16 ? 16 * kBK : kABytes;
  static constexpr int kBBytes = BN * kBK;
  static constexpr int kStageBytes = A_ROWS * kBK + kBBytes;  // what one stage's copies bring
  // fp32 partial buffers in tensor memory: two of BN >= 128 columns, or (the
  // narrow tiles of problems that fill few SMs) as many as fit in 512
  // columns, so that the MMAs run several K-blocks ahead of the promotion
  static constexpr int kBufs = BN >= 128 ? 2 : 512 / BN;
  static constexpr int kTmemCols = kBufs * BN;
  // the allocation: a power of two of at least kTmemCols columns
  static constexpr int kTmemAlloc = kTmemCols <= 256 ? 256 : 512;
  // promotion warps that hold rows of the tile: all, or with A_ROWS = 16 the
  // EW / 4 warps of tensor-memory lanes 0..31
  static constexpr int kActiveEpi = A_ROWS == 16 ? EW / 4 : EW;
  // tile scales (1x128 x 128x128 modes) a K-block needs: one per 128-column
  // block its columns touch.  Tiles start on multiples of BN, so a tile starts
  // at most 128 - gcd(BN, 128) columns into a block (224-column tiles: 96,
  // three blocks).
  static constexpr int kTileScales = (128 - gcd_c(BN, 128) + BN + 127) / 128;
  static constexpr int kOffB = ((STAGES - 1) * kAStride + kABytes + 1023) / 1024 * 1024;
  static constexpr int kOffC = kOffB + STAGES * kBBytes;
  // scale ring: kScaleSlots slots of kScaleGroup K-blocks, each K-block
  // a_s[128 rows] then b_s (BN column scales or up to BN/128 tile scales)
  static constexpr int kScaleSlots = 2;
  static constexpr int kScaleGroup = 4;
  static constexpr int kScaleKbBytes = 128 * 4 + BN * 4;
  static constexpr int kScaleBytes = kScaleGroup * kScaleKbBytes;
  static constexpr int kOffScale = kOffC;
  static constexpr int kOffBar = kOffScale + kScaleSlots * kScaleBytes;
  static constexpr int kNumBars = 2 * STAGES + 2 * kBufs + 2 + 2 * kScaleSlots;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + slack for 1024-byte alignment
  // Dense kernel, 256-column tiles: the epilogue of the tile-scale modes can
  // leave through TMA stores, each promotion warp staging its 32 rows x 64
  // columns of bf16 (4 KiB, 128-byte swizzled rows) in a buffer of its own.
  // (The column-scale mode measured 7% slower with it: its promotion loop,
  // not its few tiles' epilogues, sets its pace.)
  static constexpr bool kEpiTma = BN == 256 && EW == 16 && A_ROWS == 128;
  static constexpr int kOffStage = (kOffMisc + 16 + 1023) / 1024 * 1024;
  static constexpr int kDenseSmemBytes = kEpiTma ? kOffStage + EW * 4096 + 1024 : kSmemBytes;
  // grouped forms only: the experts' offsets and first tiles
  static constexpr int kGroupTabBytes = 2 * (kMaxGroups + 1) * 4;
  static_assert(kSmemBytes + kGroupTabBytes <= 227 * 1024, "shared memory budget");
  static_assert(kTmemCols <= kTmemAlloc && kTmemAlloc <= 512, "tensor-memory allocation");
};

// L consecutive columns of a warp's tensor-memory lanes into r (L a multiple
// of 8 up to 64; 24 = 16 + 8 and so on, several loads before one wait).
template <int L>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t* r) {
  if constexpr (L == 64) {
    tmem_ld_32x32b_x64(taddr, *reinterpret_cast<uint32_t(*)[64]>(r));
  } else if constexpr (L == 32) {
    tmem_ld_32x32b_x32(taddr, *reinterpret_cast<uint32_t(*)[32]>(r));
  } else if constexpr (L == 16) {
    tmem_ld_32x32b_x16(taddr, *reinterpret_cast<uint32_t(*)[16]>(r));
  } else if constexpr (L == 8) {
    tmem_ld_32x32b_x8(taddr, *reinterpret_cast<uint32_t(*)[8]>(r));
  } else {
    static_assert(L % 8 == 0 && L > 16 && L < 64, "tensor-memory load width");
    tmem_ld_cols<16>(taddr, r);
    tmem_ld_cols<L - 16>(taddr + 16u, r + 16);
  }
}

__device__ __forceinline__ void gemm_fail(uint32_t code, volatile int* abort_flag) {
  atomicOr(&g_gemm_error, code);
  *abort_flag = 1;
}

// Four consecutive fp32 scales v[i0 .. i0+3] (of a row of n) into shared
// memory at dst by cp.async; past n zero-filled.
__device__ __forceinline__ void copy_scales4(uint32_t dst, const float* v, int i0, int64_t n, bool vec) {
  if (vec) {
    const int64_t left = n - i0;
    const uint32_t bytes = left >= 4 ? 16u : left > 0 ? (uint32_t)left * 4u : 0u;
    cp_async_16(dst, bytes ? v + i0 : v, bytes);
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const bool in = i0 + q < n;
      cp_async_4(dst + 4u * q, in ? v + i0 + q : v, in ? 4u : 0u);
    }
  }
}

// The experts' clamped offsets o[0..E] (running maximum of offs, within
// [0, M_total]) and, for kGroupRows, the first tile of each expert, built by
// one warp into shared memory.  Offsets that had to be clamped, and (kGroupRed)
// experts not starting on a 128-token boundary, set kErrGroupOffsets.
template <int GROUP>
__device__ void gemm_build_groups(const GemmParams& p, const GemmGroupParams& gp, int* s_offs, int* s_start,
                                  int lane) {
  const int n = gp.E + 1;
  const int per = (n + 31) / 32;
  const int i0 = min(lane * per, n), i1 = min(i0 + per, n);
  int run = 0;
  for (int i = i0; i < i1; ++i) {
    run = max(run, min(max(gp.offs[i], 0), gp.M_total));
    s_offs[i] = run;
  }
  int incl = run;  // running maximum over the chunks of lanes <= this one
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl = max(incl, y);
  }
  int excl = __shfl_up_sync(0xffffffffu, incl, 1);
  if (lane == 0) excl = 0;
  bool bad = false;
  for (int i = i0; i < i1; ++i) {
    const int raw = gp.offs[i];
    const int v = max(s_offs[i], excl);
    s_offs[i] = v;
    bad |= raw != v;
    if (GROUP == kGroupRed && i < gp.E) bad |= (v % kBK) != 0;
  }
  __syncwarp();
  if (GROUP == kGroupRows) {
    int cnt = 0;  // tiles of this lane's experts
    for (int i = i0; i < i1 && i < gp.E; ++i) cnt += (int)cdiv(s_offs[i + 1] - s_offs[i], kBM) * p.num_n;
    int sum = cnt;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, sum, off);
      if (lane >= off) sum += y;
    }
    int acc = sum - cnt;
    for (int i = i0; i < i1; ++i) {
      s_start[i] = acc;
      if (i < gp.E) acc += (int)cdiv(s_offs[i + 1] - s_offs[i], kBM) * p.num_n;
    }
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0 && blockIdx.x == 0) atomicOr(&g_gemm_error, kErrGroupOffsets);
}

template <int GROUP, int BN>
__device__ __forceinline__ GemmJob gemm_job(int tile, const GemmParams& p, const GemmGroupParams& gp, const int* s_offs,
                                            const int* s_start) {
  GemmJob j;
  if constexpr (GROUP == kGroupRows) {
    const int e = group_of_tile(s_start, gp.E, tile);
    const int r0 = s_offs[e], re = s_offs[e + 1] - r0;
    const GemmTile g = gemm_tile(tile - s_start[e], (int)cdiv(re, kBM), p.num_n, BN);
    j.a_row = r0 + g.m0;
    j.rows = re - g.m0;
    j.b_row = e * gp.b_row_step + g.n0;
    j.a_k = 0;
    j.b_k = e * gp.b_k_step;
    j.kb_s = 0;
    j.kbn = p.Kb;
    j.n0 = g.n0;
    j.e = e;
    j.c_off = (int64_t)j.a_row * p.ldc + g.n0;
  } else {  // kGroupRed
    const int per = p.num_m * p.num_n;
    const int e = tile / per;
    const GemmTile g = gemm_tile(tile - e * per, p.num_m, p.num_n, BN);
    const int t0 = s_offs[e], t1 = s_offs[e + 1];
    j.kb_s = t0 / kBK;
    j.kbn = t1 > t0 ? (int)cdiv(t1, kBK) - j.kb_s : 0;
    j.a_k = j.kb_s * kBK;
    j.b_k = j.a_k;
    j.a_row = g.m0;
    j.rows = (int)p.M - g.m0;
    j.b_row = g.n0;
    j.n0 = g.n0;
    j.e = e;
    j.c_off = (int64_t)e * gp.c_step + (int64_t)g.m0 * p.ldc + g.n0;
  }
  return j;
}

template <int BN, int STAGES, int SB_MODE, int LDW, int EW, int A_ROWS = 128>
__global__ void __launch_bounds__(GemmCfg<BN, STAGES, EW, A_ROWS>::kThreads, 1)
    gemm_blockwise_kernel(const __grid_constant__ CUtensorMap tma_a, const __grid_constant__ CUtensorMap tma_b,
                          const __grid_constant__ CUtensorMap tma_c, const GemmParams p) {
  using Cfg = GemmCfg<BN, STAGES, EW, A_ROWS>;
  constexpr int kCols = Cfg::kCols;
  constexpr int NT = Cfg::kBufs;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sA = sbase;
  const uint32_t sB = sbase + Cfg::kOffB;
  const uint32_t sScale = sbase + Cfg::kOffScale;
  const uint32_t bar0 = sbase + Cfg::kOffBar;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + Cfg::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::kOffMisc + 4);
  volatile int* never = reinterpret_cast<volatile int*>(smem + Cfg::kOffMisc + 8);

  // barriers: full[S], empty[S], tfull[NT], tempty[NT], drain (both issuers), stall, sfull[2], sempty[2]
  auto full_bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  auto empty_bar = [&](int i) { return bar0 + 8u * (uint32_t)(STAGES + i); };
  auto tfull_bar = [&](int i) { return bar0 + 8u * (uint32_t)(2 * STAGES + i); };
  auto tempty_bar = [&](int i) { return bar0 + 8u * (uint32_t)(2 * STAGES + NT + i); };
  const uint32_t drain_bar = bar0 + 8u * (uint32_t)(2 * STAGES + 2 * NT);
  const uint32_t stall_bar = bar0 + 8u * (uint32_t)(2 * STAGES + 2 * NT + 1);  // never arrived on
  auto sfull_bar = [&](int i) { return bar0 + 8u * (uint32_t)(2 * STAGES + 2 * NT + 2 + i); };
  auto sempty_bar = [&](int i) {
    return bar0 + 8u * (uint32_t)(2 * STAGES + 2 * NT + 2 + Cfg::kScaleSlots + i);
  };

  const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);
  const int lane = (int)(threadIdx.x & 31);
  // only a kernel launched with programmatic dependent launch lets the next
  // one start early; otherwise the next kernel starts once this one completes
  if (p.pdl) pdl_launch_dependents();

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(full_bar(i), 1);
      mbar_init(empty_bar(i), 1);
    }
    for (int i = 0; i < NT; ++i) {
      mbar_init(tfull_bar(i), 1);
      mbar_init(tempty_bar(i), Cfg::kActiveEpi);
    }
    mbar_init(drain_bar, 2);
    mbar_init(stall_bar, 1);
    for (int i = 0; i < Cfg::kScaleSlots; ++i) {
      mbar_init(sfull_bar(i), 32);  // one cp.async arrival per loader lane
      mbar_init(sempty_bar(i), Cfg::kActiveEpi);
    }
    *abort_flag = 0;
    *never = 0;
    fence_barrier_init();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), Cfg::kTmemAlloc);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tma_a);
    tma_prefetch_desc(&tma_b);
    if (Cfg::kEpiTma && SB_MODE != kSbCol && p.c_tma) tma_prefetch_desc(&tma_c);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_wait();  // the previous kernel's writes are visible from here on
  const uint32_t tmem_base = *tmem_holder;
  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(Cfg::kCtrlRegs));
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
        const GemmTile g = gemm_tile(tile, p.num_m, p.num_n, BN);
        for (int kb = 0; kb < p.Kb; ++kb, ++it) {
          const int st = (int)(it % STAGES);
          const uint32_t ph = (it / STAGES) & 1u;
          if (!mbar_wait_bounded(empty_bar(st), ph ^ 1u, p.wait_limit_ns, abort_flag)) {
            gemm_fail(kErrWaitEmpty, abort_flag);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full_bar(st), (uint32_t)Cfg::kStageBytes);
          tma_load_2d(sA + (uint32_t)(st * Cfg::kAStride), &tma_a, full_bar(st), kb * kBK, g.m0);
          tma_load_2d(sB + (uint32_t)(st * Cfg::kBBytes), &tma_b, full_bar(st), kb * kBK, g.n0);
        }
      }
      if (!ok) {
        // copies already issued must land before this CTA's smem goes away
        for (uint32_t j = (it > STAGES ? it - STAGES : 0); j < it; ++j)
          if (!mbar_wait_bounded(full_bar((int)(j % STAGES)), (j / STAGES) & 1u,
                                 p.wait_limit_ns, never))
            atomicOr(&g_gemm_error, kErrWaitDrain);
      }
    }
  } else if (warp == 1 || warp == 3) {
    // ------------------------------------------------------------ MMA issuers
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_e4m3_f32(kBM, BN);
      const uint32_t mine = warp == 1 ? 0u : 1u;  // the K-block steps (and TMEM buffer) of this issuer
      uint32_t it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
        for (int kb = 0; kb < p.Kb; ++kb, ++it) {
          if ((it & 1u) != mine) continue;
          const int st = (int)(it % STAGES);
          const uint32_t ph = (it / STAGES) & 1u;
          const int buf = (int)(it % NT);
          const uint32_t tph = (it / NT) & 1u;
          if (!mbar_spin_bounded(tempty_bar(buf), tph ^ 1u, p.wait_limit_ns, abort_flag)) {
            gemm_fail(kErrWaitTmemEmpty, abort_flag);
            ok = false;
            break;
          }
          if (!mbar_spin_bounded(full_bar(st), ph, p.wait_limit_ns, abort_flag)) {
            gemm_fail(kErrWaitFull, abort_flag);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t da = desc_kmajor_sw128(sA + (uint32_t)(st * Cfg::kAStride));
          const uint64_t db = desc_kmajor_sw128(sB + (uint32_t)(st * Cfg::kBBytes));
          const uint32_t d_tmem = tmem_base + (uint32_t)(buf * BN);
#pragma unroll
          for (int k = 0; k < kBK / 32; ++k)  // advance 32 bytes of K inside the swizzled row
            mma_e4m3(d_tmem, da + (uint64_t)(2 * k), db + (uint64_t)(2 * k), idesc, k > 0 ? 1u : 0u);
          mma_commit(empty_bar(st));
          mma_commit(tfull_bar(buf));
        }
      }
      // every MMA issued by both issuers completes before tensor memory is released
      mma_commit(drain_bar);
      if (!mbar_wait_bounded(drain_bar, 0, p.wait_limit_ns, never))
        gemm_fail(kErrWaitDrain, abort_flag);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ scale loader
    uint32_t it = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
      const GemmTile g = gemm_tile(tile, p.num_m, p.num_n, BN);
      const bool last_tile = tile + (int)gridDim.x >= p.num_tiles;
      for (int kb = 0; kb < p.Kb; ++kb, ++it) {
        const uint32_t grp = it / Cfg::kScaleGroup, sub = it % Cfg::kScaleGroup;
        const int sl = (int)(grp % Cfg::kScaleSlots);
        if (sub == 0) {
          const uint32_t ph = (grp / Cfg::kScaleSlots) & 1u;
          const bool got = mbar_wait_bounded(sempty_bar(sl), ph ^ 1u, p.wait_limit_ns, abort_flag);
          if (!__all_sync(0xffffffffu, got)) {
            if (lane == 0) gemm_fail(kErrWaitScale, abort_flag);
            ok = false;
            break;
          }
        }
        const uint32_t slot = sScale + (uint32_t)(sl * Cfg::kScaleBytes + sub * Cfg::kScaleKbBytes);
        // a_s of rows m0 + 4*lane .. +3 (zero past M)
        copy_scales4(slot + 16u * lane, p.sa + (int64_t)kb * p.ldsa, g.m0 + 4 * lane, p.M, p.sa_vec);
        if (SB_MODE == kSbCol) {  // b_s of columns n0 + 128h + 4*lane .. +3 < n0 + BN (zero past N)
#pragma unroll
          for (int h = 0; h < (BN + 127) / 128; ++h)
            if (128 * h + 4 * lane < BN)
              copy_scales4(slot + 512u + 512u * h + 16u * lane, p.sb + (int64_t)kb * p.ldsb, g.n0 + 128 * h + 4 * lane,
                           p.N, p.sb_vec);
        } else if (lane < Cfg::kTileScales) {  // tile scale of the 128 columns n0 + 128*lane (zero past N)
          const int nb = g.n0 / kBlock + lane;
          const bool in = nb < p.Nb;
          const float* src = SB_MODE == kSbTile ? p.sb + (int64_t)nb * p.ldsb + kb : p.sb + (int64_t)kb * p.ldsb + nb;
          cp_async_4(slot + 512u + 4u * lane, in ? src : p.sb, in ? 4u : 0u);
        }
        // the slot is published once its group is complete (or the CTA's K-blocks end)
        if (sub == Cfg::kScaleGroup - 1 || (last_tile && kb == p.Kb - 1)) cp_async_mbar_arrive(sfull_bar(sl));
      }
    }
    // let this lane's copies land before the CTA can exit
    asm volatile("cp.async.wait_all;" ::: "memory");
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(Cfg::kEpiRegs));
    // ------------------------------------------------------------ promotion + epilogue
    const int e = warp - 4;
    const int row = epi_row(e, lane);
    const int col0 = epi_col0(e, BN, EW);
    const uint32_t lane_base = (uint32_t)(32 * (warp % 4)) << 16;
    uint32_t it = 0;
    // (A_ROWS = 16: warps of lanes 32..127 hold no row of the problem and skip the loop)
    bool ok = A_ROWS == 128 || warp % 4 == 0;
    for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
      const GemmTile g = gemm_tile(tile, p.num_m, p.num_n, BN);
      const bool last_tile = tile + (int)gridDim.x >= p.num_tiles;
      float acc[kCols];
#pragma unroll
      for (int j = 0; j < kCols; ++j) acc[j] = 0.0f;

      for (int kb = 0; kb < p.Kb; ++kb, ++it) {
        const uint32_t grp = it / Cfg::kScaleGroup, sub = it % Cfg::kScaleGroup;
        const int sl = (int)(grp % Cfg::kScaleSlots);
        const uint32_t slot = sScale + (uint32_t)(sl * Cfg::kScaleBytes + sub * Cfg::kScaleKbBytes);
        // once per group: the loader runs ahead, so the slot is almost always ready (poll)
        const bool sgot = sub != 0 || mbar_spin_bounded(sfull_bar(sl), (grp / Cfg::kScaleSlots) & 1u,
                                                        p.wait_limit_ns, abort_flag);
        const int buf = (int)(it % NT);
        const uint32_t tph = (it / NT) & 1u;
        const bool got = sgot && mbar_wait_bounded(p.debug_stall ? stall_bar : tfull_bar(buf), tph, p.wait_limit_ns,
                                                   abort_flag);
        if (!__all_sync(0xffffffffu, got)) {
          if (lane == 0) gemm_fail(sgot ? kErrWaitTmemFull : kErrWaitScale, abort_flag);
          ok = false;
          break;
        }
        tc_fence_after();
        float sa_cur, sb_cur = 0.0f;
        asm volatile("ld.shared.f32 %0, [%1];" : "=f"(sa_cur) : "r"(slot + 4u * row));
        if (SB_MODE != kSbCol)
          asm volatile("ld.shared.f32 %0, [%1];" : "=f"(sb_cur) : "r"(slot + 512u + 4u * (uint32_t)(col0 >> 7)));
        const float scale = sa_cur * sb_cur;
        const uint64_t scale2 = f2_pack(scale, scale);
        const uint32_t taddr = tmem_base + lane_base + (uint32_t)(buf * BN + col0);
        if constexpr (kCols % LDW != 0) {
          // 224-column tiles (column scales): a warp's 56 columns are
          // segments of LDW columns and a last one of kCols % LDW, one
          // tensor-memory round trip each
          static_assert(kCols == 56 && BN == 224 && SB_MODE == kSbCol, "segmented promotion: 224-column tiles");
          auto segment = [&](auto len, int c0, bool last) {
            constexpr int L = decltype(len)::value;
            uint32_t r[L];
            tmem_ld_cols<L>(taddr + (uint32_t)c0, r);
            tmem_ld_wait();
            tmem_regs_after_wait(r);
            if (last) {
              // this warp's share of the partial is in registers: release the buffer
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(tempty_bar(buf));
            }
            // acc[n] += (a_s * b_s[n]) * P[n] on fp32x2 lanes, as below
            const uint64_t sa2 = f2_pack(sa_cur, sa_cur);
#pragma unroll
            for (int j4 = 0; j4 < L / 4; ++j4) {
              float4 sb4;
              asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                           : "=f"(sb4.x), "=f"(sb4.y), "=f"(sb4.z), "=f"(sb4.w)
                           : "r"(slot + 512u + 4u * (uint32_t)(col0 + c0 + 4 * j4)));
              const uint64_t t2[2] = {f2_mul(sa2, f2_pack(sb4.x, sb4.y)), f2_mul(sa2, f2_pack(sb4.z, sb4.w))};
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const int j = c0 + 4 * j4 + 2 * h;
                const uint64_t p2 =
                    f2_pack(__uint_as_float(r[4 * j4 + 2 * h]), __uint_as_float(r[4 * j4 + 2 * h + 1]));
                f2_unpack(f2_fma(t2[h], p2, f2_pack(acc[j], acc[j + 1])), acc[j], acc[j + 1]);
              }
            }
          };
#pragma unroll
          for (int c = 0; c < kCols / LDW; ++c) segment(std::integral_constant<int, LDW>{}, LDW * c, false);
          segment(std::integral_constant<int, kCols % LDW>{}, kCols / LDW * LDW, true);
        } else {
        // LDW columns of the partial per tensor-memory load round trip (one wait)
#pragma unroll
        for (int c = 0; c < kCols / LDW; ++c) {
          uint32_t r[LDW];
          if constexpr (LDW == 64)
            tmem_ld_32x32b_x64(taddr + (uint32_t)(LDW * c), r);
          else if constexpr (LDW == 32)
            tmem_ld_32x32b_x32(taddr + (uint32_t)(LDW * c), r);
          else
            tmem_ld_32x32b_x16(taddr + (uint32_t)(LDW * c), r);
          tmem_ld_wait();
          tmem_regs_after_wait(r);
          if (c == kCols / LDW - 1) {
            // this warp's share of the partial is in registers: release the buffer
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty_bar(buf));
          }
          if (SB_MODE == kSbCol) {
            // acc[n] += (a_s * b_s[n]) * P[n] on fp32x2 lanes (two columns per instruction)
            const uint64_t sa2 = f2_pack(sa_cur, sa_cur);
#pragma unroll
            for (int j4 = 0; j4 < LDW / 4; ++j4) {
              float4 sb4;
              asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                           : "=f"(sb4.x), "=f"(sb4.y), "=f"(sb4.z), "=f"(sb4.w)
                           : "r"(slot + 512u + 4u * (uint32_t)(col0 + LDW * c + 4 * j4)));
              const uint64_t t2[2] = {f2_mul(sa2, f2_pack(sb4.x, sb4.y)), f2_mul(sa2, f2_pack(sb4.z, sb4.w))};
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const int j = LDW * c + 4 * j4 + 2 * h;
                const uint64_t p2 =
                    f2_pack(__uint_as_float(r[4 * j4 + 2 * h]), __uint_as_float(r[4 * j4 + 2 * h + 1]));
                f2_unpack(f2_fma(t2[h], p2, f2_pack(acc[j], acc[j + 1])), acc[j], acc[j + 1]);
              }
            }
          } else {
#pragma unroll
            for (int j = 0; j < LDW; j += 2) {  // acc += (a_s * b_s) * P, two columns per fp32x2 FMA
              const uint64_t p2 = f2_pack(__uint_as_float(r[j]), __uint_as_float(r[j + 1]));
              f2_unpack(f2_fma(scale2, p2, f2_pack(acc[LDW * c + j], acc[LDW * c + j + 1])), acc[LDW * c + j],
                        acc[LDW * c + j + 1]);
            }
          }
        }
        }
        // the slot's scales are no longer needed by this warp (end of its group)
        if (sub == Cfg::kScaleGroup - 1 || (last_tile && kb == p.Kb - 1)) {
          __syncwarp();
          if (lane == 0) mbar_arrive(sempty_bar(sl));
        }
      }
      if (!ok) break;

      // Epilogue: round to bf16, transpose G x G blocks of 16-byte chunks (8
      // columns) within groups of G lanes (xor shuffles), so that lane pos of a
      // group holds chunk pos of the group's G rows; each store instruction of
      // the warp then writes 32/G row segments of 16*G contiguous bytes.  Only
      // rows < M and columns < N are written.
      if (Cfg::kEpiTma && SB_MODE != kSbCol && p.c_tma) {
        // TMA-store epilogue: this warp's 32 rows x 64 columns, rounded to
        // bf16, into its staging buffer (16-byte chunk c of row r at c ^ (r & 7):
        // the 128-byte swizzle of the map, and conflict-free for the eight rows
        // of a quarter-warp), then one store of the box at (n0 + col0, m0 + 32 *
        // (warp % 4)); the map clips rows >= M and columns >= N (N % 8 == 0).
        const uint32_t stg = sbase + (uint32_t)(Cfg::kOffStage + e * 4096);
        if (lane == 0) bulk_wait_read_all();  // the previous tile's store has read the buffer
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 8; ++c)
          asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(stg + 128u * lane + ((uint32_t)(c ^ (lane & 7)) << 4)),
                       "r"(pack_bf16x2(acc[8 * c], acc[8 * c + 1])), "r"(pack_bf16x2(acc[8 * c + 2], acc[8 * c + 3])),
                       "r"(pack_bf16x2(acc[8 * c + 4], acc[8 * c + 5])), "r"(pack_bf16x2(acc[8 * c + 6], acc[8 * c + 7]))
                       : "memory");
        fence_proxy_async_shared();
        __syncwarp();
        const int bm = g.m0 + 32 * (warp % 4), bn0 = g.n0 + col0;
        if (lane == 0 && bm < p.M && bn0 < p.N) {
          tma_store_2d(&tma_c, stg, bn0, bm);
          bulk_commit();
        }
      } else {
        // chunks per transposed block and passes (epi_group, epi_passes): a
        // share of 56 columns is 7 chunks in one block of 8, the eighth empty
        constexpr int kChunks = kCols / 8;
        constexpr int kG = kChunks > 4 ? 8 : kChunks > 2 ? 4 : kChunks;
        const int pos = lane % kG;
#pragma unroll
        for (int sg = 0; sg < (kChunks + kG - 1) / kG; ++sg) {
          uint32_t X[kG][4];
#pragma unroll
          for (int j = 0; j < kG; ++j)
#pragma unroll
            for (int q = 0; q < 4; ++q)
              X[j][q] = kG * sg + j < kChunks
                            ? pack_bf16x2(acc[8 * (kG * sg + j) + 2 * q], acc[8 * (kG * sg + j) + 2 * q + 1])
                            : 0u;
#pragma unroll
          for (int msk = kG / 2; msk >= 1; msk >>= 1) {
            const bool hi = (pos & msk) != 0;
#pragma unroll
            for (int j = 0; j < kG; ++j) {
              if (j & msk) continue;
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const uint32_t send = hi ? X[j][q] : X[j | msk][q];
                const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, msk);
                if (hi) X[j][q] = recv;
                else X[j | msk][q] = recv;
              }
            }
          }
          const int n = g.n0 + epi_store_col(e, lane, sg, kG, BN, EW);
          const bool has_chunk = kG * sg + pos < kChunks;
#pragma unroll
          for (int i = 0; i < kG; ++i) {
            const int mr = g.m0 + epi_store_row(e, lane, i, kG);
            if (!has_chunk || mr >= p.M || n >= p.N) continue;
            uint16_t* dst = p.c + (int64_t)mr * p.ldc + n;
            if (p.c_vec && n + 8 <= p.N) {
              *reinterpret_cast<uint4*>(dst) = make_uint4(X[i][0], X[i][1], X[i][2], X[i][3]);
            } else {
#pragma unroll
              for (int b = 0; b < 8; ++b)
                if (n + b < p.N) dst[b] = (uint16_t)(X[i][b >> 1] >> (16 * (b & 1)));
            }
          }
        }
      }
    }
    // this warp's TMA stores complete before the CTA's shared memory goes away
    if (Cfg::kEpiTma && SB_MODE != kSbCol && p.c_tma && lane == 0) bulk_wait_all();
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::kTmemAlloc);
  }
}

// The grouped (mixture-of-experts) forms: the same pipeline as
// gemm_blockwise_kernel, with each tile's operands, K-blocks, scales and
// output found through its GemmJob.  (The dense GEMM keeps its own kernel:
// its weight-gradient form sits at the register limit of the promotion warps,
// and the job indirection measured 10-17% slower there.)
template <int BN, int STAGES, int SB_MODE, int LDW, int EW, int GROUP, bool STG = false>
__global__ void __launch_bounds__(GemmCfg<BN, STAGES, EW>::kThreads, 1)
    gemm_grouped_kernel(const __grid_constant__ CUtensorMap tma_a, const __grid_constant__ CUtensorMap tma_b,
                        const __grid_constant__ CUtensorMap tma_c, const GemmParams p, const GemmGroupParams gp) {
  static_assert(GROUP == kGroupRows || GROUP == kGroupRed, "a grouped form");
  using Cfg = GemmCfg<BN, STAGES, EW>;
  // STG: the epilogue may store through the C map from per-warp staging
  // buffers placed after an expert table of at most kStageGroups experts
  static_assert(!STG || Cfg::kEpiTma, "staged epilogue: 64 columns per promotion warp");
  constexpr int kTab = STG ? kStageGroups : kMaxGroups;
  constexpr uint32_t kOffStageG = (uint32_t)((Cfg::kOffMisc + 16 + 2 * (kTab + 1) * 4 + 1023) / 1024 * 1024);
  static_assert(Cfg::kBufs == 2 && Cfg::kTileScales == BN / 128, "the grouped forms use tiles of 128 or 256 columns");
  constexpr int kCols = Cfg::kCols;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sA = sbase;
  const uint32_t sB = sbase + Cfg::kOffB;
  const uint32_t sScale = sbase + Cfg::kOffScale;
  const uint32_t bar0 = sbase + Cfg::kOffBar;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + Cfg::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::kOffMisc + 4);
  volatile int* never = reinterpret_cast<volatile int*>(smem + Cfg::kOffMisc + 8);
  // grouped forms: the experts' offsets and first tiles (kGroupTabBytes past the barriers)
  int* s_offs = reinterpret_cast<int*>(smem + Cfg::kOffMisc + 16);
  int* s_start = s_offs + (kTab + 1);

  // barriers: full[S], empty[S], tfull[2], tempty[2], drain (both issuers), stall, sfull[2], sempty[2]
  auto full_bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  auto empty_bar = [&](int i) { return bar0 + 8u * (uint32_t)(STAGES + i); };
  auto tfull_bar = [&](int i) { return bar0 + 8u * (uint32_t)(2 * STAGES + i); };
  auto tempty_bar = [&](int i) { return bar0 + 8u * (uint32_t)(2 * STAGES + 2 + i); };
  const uint32_t drain_bar = bar0 + 8u * (uint32_t)(2 * STAGES + 4);
  const uint32_t stall_bar = bar0 + 8u * (uint32_t)(2 * STAGES + 5);  // never arrived on
  auto sfull_bar = [&](int i) { return bar0 + 8u * (uint32_t)(2 * STAGES + 6 + i); };
  auto sempty_bar = [&](int i) { return bar0 + 8u * (uint32_t)(2 * STAGES + 6 + Cfg::kScaleSlots + i); };

  const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);
  const int lane = (int)(threadIdx.x & 31);
  // only a kernel launched with programmatic dependent launch lets the next
  // one start early; otherwise the next kernel starts once this one completes
  if (p.pdl) pdl_launch_dependents();

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(full_bar(i), 1);
      mbar_init(empty_bar(i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(tfull_bar(i), 1);
      mbar_init(tempty_bar(i), Cfg::kEpiWarps);
    }
    mbar_init(drain_bar, 2);
    mbar_init(stall_bar, 1);
    for (int i = 0; i < Cfg::kScaleSlots; ++i) {
      mbar_init(sfull_bar(i), 32);  // one cp.async arrival per loader lane
      mbar_init(sempty_bar(i), Cfg::kEpiWarps);
    }
    *abort_flag = 0;
    *never = 0;
    fence_barrier_init();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), Cfg::kTmemAlloc);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tma_a);
    tma_prefetch_desc(&tma_b);
  }
  pdl_wait();  // the previous kernel's writes (the offsets among them) are visible from here on
  if (warp == 2) gemm_build_groups<GROUP>(p, gp, s_offs, s_start, lane);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int num_tiles = GROUP == kGroupRows ? s_start[gp.E] : p.num_tiles;
  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(Cfg::kCtrlRegs));
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
        const GemmJob j = gemm_job<GROUP, BN>(tile, p, gp, s_offs, s_start);
        for (int kb = 0; kb < j.kbn; ++kb, ++it) {
          const int st = (int)(it % STAGES);
          const uint32_t ph = (it / STAGES) & 1u;
          if (!mbar_wait_bounded(empty_bar(st), ph ^ 1u, p.wait_limit_ns, abort_flag)) {
            gemm_fail(kErrWaitEmpty, abort_flag);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full_bar(st), (uint32_t)Cfg::kStageBytes);
          tma_load_2d(sA + (uint32_t)(st * Cfg::kABytes), &tma_a, full_bar(st), j.a_k + kb * kBK, j.a_row);
          tma_load_2d(sB + (uint32_t)(st * Cfg::kBBytes), &tma_b, full_bar(st), j.b_k + kb * kBK, j.b_row);
        }
      }
      if (!ok) {
        // copies already issued must land before this CTA's smem goes away
        for (uint32_t j = (it > STAGES ? it - STAGES : 0); j < it; ++j)
          if (!mbar_wait_bounded(full_bar((int)(j % STAGES)), (j / STAGES) & 1u,
                                 p.wait_limit_ns, never))
            atomicOr(&g_gemm_error, kErrWaitDrain);
      }
    }
  } else if (warp == 1 || warp == 3) {
    // ------------------------------------------------------------ MMA issuers
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_e4m3_f32(kBM, BN);
      const uint32_t mine = warp == 1 ? 0u : 1u;  // the K-block steps (and TMEM buffer) of this issuer
      uint32_t it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
        const int kbn = gemm_job<GROUP, BN>(tile, p, gp, s_offs, s_start).kbn;
        for (int kb = 0; kb < kbn; ++kb, ++it) {
          if ((it & 1u) != mine) continue;
          const int st = (int)(it % STAGES);
          const uint32_t ph = (it / STAGES) & 1u;
          const int buf = (int)(it & 1u);
          const uint32_t tph = (it >> 1) & 1u;
          if (!mbar_spin_bounded(tempty_bar(buf), tph ^ 1u, p.wait_limit_ns, abort_flag)) {
            gemm_fail(kErrWaitTmemEmpty, abort_flag);
            ok = false;
            break;
          }
          if (!mbar_spin_bounded(full_bar(st), ph, p.wait_limit_ns, abort_flag)) {
            gemm_fail(kErrWaitFull, abort_flag);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t da = desc_kmajor_sw128(sA + (uint32_t)(st * Cfg::kABytes));
          const uint64_t db = desc_kmajor_sw128(sB + (uint32_t)(st * Cfg::kBBytes));
          const uint32_t d_tmem = tmem_base + (uint32_t)(buf * BN);
#pragma unroll
          for (int k = 0; k < kBK / 32; ++k)  // advance 32 bytes of K inside the swizzled row
            mma_e4m3(d_tmem, da + (uint64_t)(2 * k), db + (uint64_t)(2 * k), idesc, k > 0 ? 1u : 0u);
          mma_commit(empty_bar(st));
          mma_commit(tfull_bar(buf));
        }
      }
      // every MMA issued by both issuers completes before tensor memory is released
      mma_commit(drain_bar);
      if (!mbar_wait_bounded(drain_bar, 0, p.wait_limit_ns, never))
        gemm_fail(kErrWaitDrain, abort_flag);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ scale loader
    // Scale groups: the tiles have different K-block counts (some none), so a
    // group of up to kScaleGroup K-blocks never spans two tiles; grp counts
    // the groups published so far.
    uint32_t grp = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
      const GemmJob j = gemm_job<GROUP, BN>(tile, p, gp, s_offs, s_start);
      const bool sa_vec = p.sa_vec && (j.a_row & 3) == 0;
      const float* sbe = p.sb + (int64_t)j.e * gp.sb_step;
      for (int kb = 0; kb < j.kbn; ++kb) {
        const uint32_t sub = (uint32_t)kb % Cfg::kScaleGroup;
        const int sl = (int)(grp % Cfg::kScaleSlots);
        const int kbs = j.kb_s + kb;
        if (sub == 0) {
          const uint32_t ph = (grp / Cfg::kScaleSlots) & 1u;
          const bool got = mbar_wait_bounded(sempty_bar(sl), ph ^ 1u, p.wait_limit_ns, abort_flag);
          if (!__all_sync(0xffffffffu, got)) {
            if (lane == 0) gemm_fail(kErrWaitScale, abort_flag);
            ok = false;
            break;
          }
        }
        const uint32_t slot = sScale + (uint32_t)(sl * Cfg::kScaleBytes + sub * Cfg::kScaleKbBytes);
        // a_s of the tile's rows 4*lane .. +3 (zero past its valid rows)
        copy_scales4(slot + 16u * lane, p.sa + (int64_t)kbs * p.ldsa + j.a_row, 4 * lane, j.rows, sa_vec);
        if (SB_MODE == kSbCol) {  // b_s of columns n0 + 128h + 4*lane .. +3 (zero past N)
#pragma unroll
          for (int h = 0; h < BN / 128; ++h)
            copy_scales4(slot + 512u + 512u * h + 16u * lane, sbe + (int64_t)kbs * p.ldsb, j.n0 + 128 * h + 4 * lane,
                         p.N, p.sb_vec);
        } else if (lane < BN / 128) {  // tile scale of the 128 columns n0 + 128*lane (zero past N)
          const int nb = j.n0 / kBlock + lane;
          const bool in = nb < p.Nb;
          const float* src = SB_MODE == kSbTile ? sbe + (int64_t)nb * p.ldsb + kbs : sbe + (int64_t)kbs * p.ldsb + nb;
          cp_async_4(slot + 512u + 4u * lane, in ? src : p.sb, in ? 4u : 0u);
        }
        // the slot is published once its group is complete (or the K-blocks end)
        if (sub == Cfg::kScaleGroup - 1 || kb == j.kbn - 1) {
          cp_async_mbar_arrive(sfull_bar(sl));
          ++grp;
        }
      }
    }
    // let this lane's copies land before the CTA can exit
    asm volatile("cp.async.wait_all;" ::: "memory");
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(Cfg::kEpiRegs));
    // ------------------------------------------------------------ promotion + epilogue
    const int e = warp - 4;
    const int row = epi_row(e, lane);
    const int col0 = epi_col0(e, BN, EW);
    const uint32_t lane_base = (uint32_t)(32 * (warp % 4)) << 16;
    uint32_t it = 0, grp = 0;  // K-block steps; scale groups as the loader counts them
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
      // (the rest of the tile's job is recomputed for the epilogue: fewer live registers)
      const int kbn = gemm_job<GROUP, BN>(tile, p, gp, s_offs, s_start).kbn;
      float acc[kCols];
#pragma unroll
      for (int j = 0; j < kCols; ++j) acc[j] = 0.0f;

      for (int kb = 0; kb < kbn; ++kb, ++it) {
        const uint32_t sub = (uint32_t)kb % Cfg::kScaleGroup;
        const int sl = (int)(grp % Cfg::kScaleSlots);
        const uint32_t slot = sScale + (uint32_t)(sl * Cfg::kScaleBytes + sub * Cfg::kScaleKbBytes);
        // once per group: the loader runs ahead, so the slot is almost always ready (poll)
        const bool sgot = sub != 0 || mbar_spin_bounded(sfull_bar(sl), (grp / Cfg::kScaleSlots) & 1u,
                                                        p.wait_limit_ns, abort_flag);
        const int buf = (int)(it & 1u);
        const uint32_t tph = (it >> 1) & 1u;
        const bool got = sgot && mbar_wait_bounded(p.debug_stall ? stall_bar : tfull_bar(buf), tph, p.wait_limit_ns,
                                                   abort_flag);
        if (!__all_sync(0xffffffffu, got)) {
          if (lane == 0) gemm_fail(sgot ? kErrWaitTmemFull : kErrWaitScale, abort_flag);
          ok = false;
          break;
        }
        tc_fence_after();
        float sa_cur, sb_cur = 0.0f;
        asm volatile("ld.shared.f32 %0, [%1];" : "=f"(sa_cur) : "r"(slot + 4u * row));
        if (SB_MODE != kSbCol)
          asm volatile("ld.shared.f32 %0, [%1];" : "=f"(sb_cur) : "r"(slot + 512u + 4u * (uint32_t)(col0 >> 7)));
        const float scale = sa_cur * sb_cur;
        const uint64_t scale2 = f2_pack(scale, scale);
        const uint32_t taddr = tmem_base + lane_base + (uint32_t)(buf * BN + col0);
        // LDW columns of the partial per tensor-memory load round trip (one wait)
#pragma unroll
        for (int c = 0; c < kCols / LDW; ++c) {
          uint32_t r[LDW];
          if constexpr (LDW == 64)
            tmem_ld_32x32b_x64(taddr + (uint32_t)(LDW * c), r);
          else if constexpr (LDW == 32)
            tmem_ld_32x32b_x32(taddr + (uint32_t)(LDW * c), r);
          else
            tmem_ld_32x32b_x16(taddr + (uint32_t)(LDW * c), r);
          tmem_ld_wait();
          tmem_regs_after_wait(r);
          if (c == kCols / LDW - 1) {
            // this warp's share of the partial is in registers: release the buffer
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty_bar(buf));
          }
          if (SB_MODE == kSbCol) {
            // acc[n] += (a_s * b_s[n]) * P[n] on fp32x2 lanes (two columns per instruction)
            const uint64_t sa2 = f2_pack(sa_cur, sa_cur);
#pragma unroll
            for (int j4 = 0; j4 < LDW / 4; ++j4) {
              float4 sb4;
              asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                           : "=f"(sb4.x), "=f"(sb4.y), "=f"(sb4.z), "=f"(sb4.w)
                           : "r"(slot + 512u + 4u * (uint32_t)(col0 + LDW * c + 4 * j4)));
              const uint64_t t2[2] = {f2_mul(sa2, f2_pack(sb4.x, sb4.y)), f2_mul(sa2, f2_pack(sb4.z, sb4.w))};
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const int j = LDW * c + 4 * j4 + 2 * h;
                const uint64_t p2 =
                    f2_pack(__uint_as_float(r[4 * j4 + 2 * h]), __uint_as_float(r[4 * j4 + 2 * h + 1]));
                f2_unpack(f2_fma(t2[h], p2, f2_pack(acc[j], acc[j + 1])), acc[j], acc[j + 1]);
              }
            }
          } else {
#pragma unroll
            for (int j = 0; j < LDW; j += 2) {  // acc += (a_s * b_s) * P, two columns per fp32x2 FMA
              const uint64_t p2 = f2_pack(__uint_as_float(r[j]), __uint_as_float(r[j + 1]));
              f2_unpack(f2_fma(scale2, p2, f2_pack(acc[LDW * c + j], acc[LDW * c + j + 1])), acc[LDW * c + j],
                        acc[LDW * c + j + 1]);
            }
          }
        }
        // the slot's scales are no longer needed by this warp (end of its group)
        if (sub == Cfg::kScaleGroup - 1 || kb == kbn - 1) {
          __syncwarp();
          if (lane == 0) mbar_arrive(sempty_bar(sl));
          ++grp;
        }
      }
      if (!ok) break;

      // Epilogue: round to bf16, transpose G x G blocks of 16-byte chunks (8
      // columns) within groups of G lanes (xor shuffles), so that lane pos of a
      // group holds chunk pos of the group's G rows; each store instruction of
      // the warp then writes 32/G row segments of 16*G contiguous bytes.  Only
      // rows < M and columns < N are written.
      const GemmJob job = gemm_job<GROUP, BN>(tile, p, gp, s_offs, s_start);
      if (STG && p.c_tma && 32 * (warp % 4) + 32 <= job.rows) {
        // all 32 of this warp's rows belong to the job: stage them as bf16
        // (128-byte swizzled rows) and store the block through the C map at
        // (n0 + col0, the rows' first row of C); the map clips columns >= N
        const uint32_t stg = sbase + kOffStageG + (uint32_t)(e * 4096);
        if (lane == 0) bulk_wait_read_all();  // the previous tile's store has read the buffer
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 8; ++c)
          asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(stg + 128u * lane + ((uint32_t)(c ^ (lane & 7)) << 4)),
                       "r"(pack_bf16x2(acc[8 * c], acc[8 * c + 1])), "r"(pack_bf16x2(acc[8 * c + 2], acc[8 * c + 3])),
                       "r"(pack_bf16x2(acc[8 * c + 4], acc[8 * c + 5])), "r"(pack_bf16x2(acc[8 * c + 6], acc[8 * c + 7]))
                       : "memory");
        fence_proxy_async_shared();
        __syncwarp();
        const int crow = (GROUP == kGroupRows ? job.a_row : job.e * gp.c_rows + job.a_row) + 32 * (warp % 4);
        if (lane == 0 && job.n0 + col0 < p.N) {
          tma_store_2d(&tma_c, stg, job.n0 + col0, crow);
          bulk_commit();
        }
      } else {
        constexpr int kG = kCols / 8 >= 8 ? 8 : kCols / 8;  // chunks per transposed block (epi_group)
        const int pos = lane % kG;
#pragma unroll
        for (int sg = 0; sg < kCols / (8 * kG); ++sg) {
          uint32_t X[kG][4];
#pragma unroll
          for (int j = 0; j < kG; ++j)
#pragma unroll
            for (int q = 0; q < 4; ++q)
              X[j][q] = pack_bf16x2(acc[8 * (kG * sg + j) + 2 * q], acc[8 * (kG * sg + j) + 2 * q + 1]);
#pragma unroll
          for (int msk = kG / 2; msk >= 1; msk >>= 1) {
            const bool hi = (pos & msk) != 0;
#pragma unroll
            for (int j = 0; j < kG; ++j) {
              if (j & msk) continue;
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const uint32_t send = hi ? X[j][q] : X[j | msk][q];
                const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, msk);
                if (hi) X[j][q] = recv;
                else X[j | msk][q] = recv;
              }
            }
          }
          const int nl = epi_store_col(e, lane, sg, kG, BN, EW);  // tile-local
#pragma unroll
          for (int i = 0; i < kG; ++i) {
            const int ml = epi_store_row(e, lane, i, kG);
            const int ncols = (int)p.N - job.n0;
            if (ml >= job.rows || nl >= ncols) continue;
            uint16_t* dst = p.c + job.c_off + (int64_t)ml * p.ldc + nl;
            const int left = ncols - nl;  // valid columns from this chunk's first one
            if (p.c_vec && left >= 8) {
              *reinterpret_cast<uint4*>(dst) = make_uint4(X[i][0], X[i][1], X[i][2], X[i][3]);
            } else {
#pragma unroll
              for (int b = 0; b < 8; ++b)
                if (b < left) dst[b] = (uint16_t)(X[i][b >> 1] >> (16 * (b & 1)));
            }
          }
        }
      }
    }
    // this warp's TMA stores complete before the CTA's shared memory goes away
    if (STG && p.c_tma && lane == 0) bulk_wait_all();
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::kTmemAlloc);
  }
}


// ---------------------------------------------------------------------------
// The forward GEMM (1x128 x 128x128) with its A operand quantised inside the
// kernel: A is the bf16 activation x, read through TMA, and a quantiser
// warpgroup forms each row's 1x128 group maximum, scale and e4m3 codes for
// the K-block into the MMA's shared-memory stage, with the same arithmetic as
// the quantisation kernels (so the bytes, scales and output equal those of
// quantising x first).  B is a weight already quantised in 128x128 tiles.
// For small M the separate quantisation launch of x and its HBM round trip go
// away ("Enable blockwise FP8 dense training kernels on ROCm", perf table:
// FP8 behind BF16 at M = 128 and 512).
//
//   warp 0      producer: raw bf16 x tiles (two 64-column boxes) into a
//               ring (two slots of 128 rows, or eight of 16 when M <= 16),
//               B tiles into the stage ring
//   warps 1, 3  MMA issuers: as the dense kernel, also waiting for the
//               stage's quantised A
//   warp 2      b_s of each K-block into the scale ring
//   warps 4-7   quantisers, two halves taking alternate K-blocks (two
//               K-blocks quantised at once): thread (row, 16-column chunk);
//               a row's 8 chunks are 8 lanes of one warp, which combine their
//               maxima by shuffles; the chunk-0 lane writes a_s into a ring
//   warps 8-15  promotion + epilogue, as the dense kernel (8 warps; with
//               M <= 16 only the two of lanes 0..31 hold rows)
// ---------------------------------------------------------------------------
template <int BN, int STAGES, int RAW_ROWS>
struct XqCfg {
  static constexpr int kEpiWarps = 8;
  static constexpr int kCols = BN / (kEpiWarps / 4);
  static constexpr int kThreads = 128 + 128 + 32 * kEpiWarps;  // 512
  // registers: 128 per thread at launch; control 56, quantisers 72, promotion 192
  static constexpr int kCtrlRegs = 56, kQuantRegs = 72, kEpiRegs = 192;
  static_assert(128 * kCtrlRegs + 128 * kQuantRegs + 32 * kEpiWarps * kEpiRegs <= kThreads * 128, "register split");
  static constexpr int kABytes = kBM * kBK;                 // e4m3 A stage: 128 rows x 128 B
  // With RAW_ROWS == 16 (M <= 16) only the first 16 rows of an A stage are
  // written, so the stages sit 2 KB apart and the MMA's reads of rows 16..127
  // fall on neighbouring stages: in-bounds shared memory whose rows only feed
  // output rows >= M, which are never stored.  That leaves room for more
  // stages of B, the operand streamed from DRAM.
  static constexpr int kAStride = RAW_ROWS == 16 ? 16 * kBK : kABytes;
  static constexpr int kBBytes = BN * kBK;
  // bf16 x tile of RAW_ROWS rows: two 64-column boxes.  128 rows in two slots,
  // or (M <= 16) 16 rows in eight, so that small problems keep eight x tiles
  // in flight against the DRAM latency
  static constexpr int kRawBytes = RAW_ROWS * kBK * 2;
  static constexpr int kRawSlots = RAW_ROWS == 16 ? 8 : 2;
  static constexpr int kOffB = ((STAGES - 1) * kAStride + kABytes + 1023) / 1024 * 1024;
  static constexpr int kOffRaw = kOffB + STAGES * kBBytes;
  static constexpr int kOffScale = kOffRaw + kRawSlots * kRawBytes;
  static constexpr int kScaleSlots = 2, kScaleGroup = 4;
  static constexpr int kScaleKbBytes = 128 * 4 + BN * 4;
  static constexpr int kScaleBytes = kScaleGroup * kScaleKbBytes;
  // fp32 partial buffers in tensor memory: two of 128 columns, or eight of
  // 64 (the narrow tiles of problems that fill few SMs, as the dense GEMM)
  static constexpr int kBufs = BN >= 128 ? 2 : 512 / BN;
  static constexpr int kTmemCols = kBufs * BN;
  // promotion warps that hold rows of the problem: all, or with M <= 16 the
  // two of tensor-memory lanes 0..31
  static constexpr int kActiveEpi = RAW_ROWS == 16 ? kEpiWarps / 4 : kEpiWarps;
  static constexpr int kTileScales = BN >= 128 ? BN / 128 : 1;
  // a_s of each K-block, written by the quantisers into a ring of kAsSlots
  // entries: they run at most STAGES units ahead of the MMAs, which run at
  // most kBufs ahead of the promotion, and a promotion warp reads its a_s
  // before releasing the buffer, so an entry is never rewritten before it has
  // been read
  static constexpr int kAsSlots = BN >= 128 ? 16 : 32;
  static_assert(kAsSlots >= STAGES + kBufs, "a_s ring depth");
  static constexpr int kOffAs = kOffScale + kScaleSlots * kScaleBytes;
  static constexpr int kOffBar = kOffAs + kAsSlots * kBM * 4;
  // full[S] empty[S] afull[S] rfull[R] rempty[R] tfull[T] tempty[T] drain stall sfull[2] sempty[2]
  static constexpr int kNumBars = 3 * STAGES + 2 * kRawSlots + 2 * kBufs + 2 + 2 * kScaleSlots;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

template <int BN, int STAGES, int LDW, int RAW_ROWS>
__global__ void __launch_bounds__(XqCfg<BN, STAGES, RAW_ROWS>::kThreads, 1)
    gemm_xq_kernel(const __grid_constant__ CUtensorMap tma_x, const __grid_constant__ CUtensorMap tma_b,
                   const GemmParams p) {
  using Cfg = XqCfg<BN, STAGES, RAW_ROWS>;
  constexpr int NR = Cfg::kRawSlots;
  constexpr int NT = Cfg::kBufs;
  constexpr int EW = Cfg::kEpiWarps;
  constexpr int kCols = Cfg::kCols;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sA = sbase, sB = sbase + Cfg::kOffB, sRaw = sbase + Cfg::kOffRaw;
  const uint32_t sScale = sbase + Cfg::kOffScale;
  const uint32_t bar0 = sbase + Cfg::kOffBar;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + Cfg::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::kOffMisc + 4);
  volatile int* never = reinterpret_cast<volatile int*>(smem + Cfg::kOffMisc + 8);

  auto full_bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  auto empty_bar = [&](int i) { return bar0 + 8u * (uint32_t)(STAGES + i); };
  auto afull_bar = [&](int i) { return bar0 + 8u * (uint32_t)(2 * STAGES + i); };
  auto rfull_bar = [&](int i) { return bar0 + 8u * (uint32_t)(3 * STAGES + i); };
  auto rempty_bar = [&](int i) { return bar0 + 8u * (uint32_t)(3 * STAGES + NR + i); };
  auto tfull_bar = [&](int i) { return bar0 + 8u * (uint32_t)(3 * STAGES + 2 * NR + i); };
  auto tempty_bar = [&](int i) { return bar0 + 8u * (uint32_t)(3 * STAGES + 2 * NR + NT + i); };
  const uint32_t drain_bar = bar0 + 8u * (uint32_t)(3 * STAGES + 2 * NR + 2 * NT);
  const uint32_t stall_bar = bar0 + 8u * (uint32_t)(3 * STAGES + 2 * NR + 2 * NT + 1);  // never arrived on
  auto sfull_bar = [&](int i) { return bar0 + 8u * (uint32_t)(3 * STAGES + 2 * NR + 2 * NT + 2 + i); };
  auto sempty_bar = [&](int i) { return bar0 + 8u * (uint32_t)(3 * STAGES + 2 * NR + 2 * NT + 4 + i); };

  const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);
  const int lane = (int)(threadIdx.x & 31);
  pdl_launch_dependents();

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(full_bar(i), 1);
      mbar_init(empty_bar(i), 1);
      mbar_init(afull_bar(i), 64);  // every thread of the quantiser half that takes the stage
    }
    for (int i = 0; i < Cfg::kRawSlots; ++i) {
      mbar_init(rfull_bar(i), 1);
      mbar_init(rempty_bar(i), 64);
    }
    for (int i = 0; i < NT; ++i) {
      mbar_init(tfull_bar(i), 1);
      mbar_init(tempty_bar(i), Cfg::kActiveEpi);
    }
    mbar_init(drain_bar, 2);
    mbar_init(stall_bar, 1);
    for (int i = 0; i < Cfg::kScaleSlots; ++i) {
      mbar_init(sfull_bar(i), 32);  // one cp.async arrival per b_s loader lane
      mbar_init(sempty_bar(i), Cfg::kActiveEpi);
    }
    *abort_flag = 0;
    *never = 0;
    fence_barrier_init();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), Cfg::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tma_x);
    tma_prefetch_desc(&tma_b);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_wait();  // the previous kernel's writes are visible from here on
  const uint32_t tmem_base = *tmem_holder;
  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(Cfg::kCtrlRegs));
    if (warp == 0) {
      // ---------------------------------------------------------- producer
      if (lane == 0) {
        uint32_t it = 0, n_raw = 0, n_b = 0;  // units; raw x and B copies issued
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
          const GemmTile g = gemm_tile(tile, p.num_m, p.num_n, BN);
          for (int kb = 0; kb < p.Kb; ++kb, ++it) {
            const int r = (int)(it % Cfg::kRawSlots);
            if (!mbar_wait_bounded(rempty_bar(r), ((it / Cfg::kRawSlots) & 1u) ^ 1u, p.wait_limit_ns, abort_flag)) {
              gemm_fail(kErrWaitEmpty, abort_flag);
              ok = false;
              break;
            }
            const uint32_t raw = sRaw + (uint32_t)(r * Cfg::kRawBytes);
            mbar_arrive_expect_tx(rfull_bar(r), (uint32_t)Cfg::kRawBytes);
            tma_load_2d(raw, &tma_x, rfull_bar(r), kb * kBK, g.m0);
            tma_load_2d(raw + (uint32_t)(Cfg::kRawBytes / 2), &tma_x, rfull_bar(r), kb * kBK + 64, g.m0);
            ++n_raw;
            const int st = (int)(it % STAGES);
            if (!mbar_wait_bounded(empty_bar(st), ((it / STAGES) & 1u) ^ 1u, p.wait_limit_ns, abort_flag)) {
              gemm_fail(kErrWaitEmpty, abort_flag);
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(full_bar(st), (uint32_t)Cfg::kBBytes);
            tma_load_2d(sB + (uint32_t)(st * Cfg::kBBytes), &tma_b, full_bar(st), kb * kBK, g.n0);
            ++n_b;
          }
        }
        if (!ok) {
          // copies already issued land before this CTA's shared memory goes away
          for (uint32_t j = (n_raw > Cfg::kRawSlots ? n_raw - Cfg::kRawSlots : 0); j < n_raw; ++j)
            if (!mbar_wait_bounded(rfull_bar((int)(j % Cfg::kRawSlots)), (j / Cfg::kRawSlots) & 1u, p.wait_limit_ns,
                                   never))
              atomicOr(&g_gemm_error, kErrWaitDrain);
          for (uint32_t j = (n_b > STAGES ? n_b - STAGES : 0); j < n_b; ++j)
            if (!mbar_wait_bounded(full_bar((int)(j % STAGES)), (j / STAGES) & 1u, p.wait_limit_ns, never))
              atomicOr(&g_gemm_error, kErrWaitDrain);
        }
      }
    } else if (warp == 1 || warp == 3) {
      // ---------------------------------------------------------- MMA issuers
      if (lane == 0) {
        constexpr uint32_t idesc = idesc_e4m3_f32(kBM, BN);
        const uint32_t mine = warp == 1 ? 0u : 1u;
        uint32_t it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
          for (int kb = 0; kb < p.Kb; ++kb, ++it) {
            if ((it & 1u) != mine) continue;
            const int st = (int)(it % STAGES);
            const uint32_t ph = (it / STAGES) & 1u;
            const int buf = (int)(it % NT);
            const uint32_t tph = (it / NT) & 1u;
            if (!mbar_spin_bounded(tempty_bar(buf), tph ^ 1u, p.wait_limit_ns, abort_flag)) {
              gemm_fail(kErrWaitTmemEmpty, abort_flag);
              ok = false;
              break;
            }
            if (!mbar_spin_bounded(full_bar(st), ph, p.wait_limit_ns, abort_flag) ||
                !mbar_spin_bounded(afull_bar(st), ph, p.wait_limit_ns, abort_flag)) {
              gemm_fail(kErrWaitFull, abort_flag);
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t da = desc_kmajor_sw128(sA + (uint32_t)(st * Cfg::kAStride));
            const uint64_t db = desc_kmajor_sw128(sB + (uint32_t)(st * Cfg::kBBytes));
            const uint32_t d_tmem = tmem_base + (uint32_t)(buf * BN);
#pragma unroll
            for (int k = 0; k < kBK / 32; ++k)
              mma_e4m3(d_tmem, da + (uint64_t)(2 * k), db + (uint64_t)(2 * k), idesc, k > 0 ? 1u : 0u);
            mma_commit(empty_bar(st));
            mma_commit(tfull_bar(buf));
          }
        }
        mma_commit(drain_bar);
        if (!mbar_wait_bounded(drain_bar, 0, p.wait_limit_ns, never)) gemm_fail(kErrWaitDrain, abort_flag);
      }
    } else {
      // ---------------------------------------------------------- b_s loader (warp 2)
      uint32_t it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
        const GemmTile g = gemm_tile(tile, p.num_m, p.num_n, BN);
        const bool last_tile = tile + (int)gridDim.x >= p.num_tiles;
        for (int kb = 0; kb < p.Kb; ++kb, ++it) {
          const uint32_t grp = it / Cfg::kScaleGroup, sub = it % Cfg::kScaleGroup;
          const int sl = (int)(grp % Cfg::kScaleSlots);
          if (sub == 0) {
            const bool got =
                mbar_wait_bounded(sempty_bar(sl), ((grp / Cfg::kScaleSlots) & 1u) ^ 1u, p.wait_limit_ns, abort_flag);
            if (!__all_sync(0xffffffffu, got)) {
              if (lane == 0) gemm_fail(kErrWaitScale, abort_flag);
              ok = false;
              break;
            }
          }
          const uint32_t slot = sScale + (uint32_t)(sl * Cfg::kScaleBytes + sub * Cfg::kScaleKbBytes);
          if (lane < Cfg::kTileScales) {  // tile scale of the 128 columns n0 + 128*lane (zero past N)
            const int nb = g.n0 / kBlock + lane;
            const bool in = nb < p.Nb;
            cp_async_4(slot + 512u + 4u * lane, in ? p.sb + (int64_t)nb * p.ldsb + kb : p.sb, in ? 4u : 0u);
          }
          if (sub == Cfg::kScaleGroup - 1 || (last_tile && kb == p.Kb - 1)) cp_async_mbar_arrive(sfull_bar(sl));
        }
      }
      asm volatile("cp.async.wait_all;" ::: "memory");
    }
  } else if (warp < 8) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(Cfg::kQuantRegs));
    // ------------------------------------------------------------ quantisers
    const int qt = (int)threadIdx.x - 128;
    const uint32_t half = (uint32_t)(qt >> 6);  // takes the K-block steps it with it % 2 == half
    const int hq = qt & 63;
    const int chunk = hq & 7;          // 16 columns of the K-block
    const int row0 = hq >> 3;          // rows row0 + 8 i
    const uint32_t gmask = 0xFFu << (8 * (lane >> 3));  // the 8 lanes of this thread's row
    const uint32_t sAs = sbase + Cfg::kOffAs;
    uint32_t it = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
      const GemmTile g = gemm_tile(tile, p.num_m, p.num_n, BN);
      const int rows_valid = (int)min((int64_t)RAW_ROWS, p.M - g.m0);
      for (int kb = 0; kb < p.Kb; ++kb, ++it) {
        if ((it & 1u) != half) continue;
        const int r = (int)(it % Cfg::kRawSlots);
        const int st = (int)(it % STAGES);
        const bool got = mbar_wait_bounded(rfull_bar(r), (it / Cfg::kRawSlots) & 1u, p.wait_limit_ns, abort_flag) &&
                         mbar_wait_bounded(empty_bar(st), ((it / STAGES) & 1u) ^ 1u, p.wait_limit_ns, abort_flag);
        if (!__all_sync(0xffffffffu, got)) {
          if (lane == 0) gemm_fail(kErrWaitFull, abort_flag);
          ok = false;
          break;
        }
        const uint32_t raw = sRaw + (uint32_t)(r * Cfg::kRawBytes);
        const uint32_t adst = sA + (uint32_t)(st * Cfg::kAStride);
        const uint32_t as_slot = sAs + (uint32_t)((it % Cfg::kAsSlots) * kBM * 4);
#pragma unroll 1
        for (int i = 0; i < RAW_ROWS / 8; ++i) {
          const int row = row0 + 8 * i;
          if (row >= rows_valid) continue;  // the 8 lanes of a row agree
          // 16 bf16 values: 16-byte chunks 2*(chunk%4) and +1 of box chunk/4 (128-byte swizzle)
          const uint32_t rbase = raw + (uint32_t)((chunk >> 2) * (Cfg::kRawBytes / 2) + row * 128);
          const int c0 = 2 * (chunk & 3);
          uint4 v0, v1;
          asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                       : "=r"(v0.x), "=r"(v0.y), "=r"(v0.z), "=r"(v0.w)
                       : "r"(rbase + (uint32_t)(((c0) ^ (row & 7)) << 4)));
          asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                       : "=r"(v1.x), "=r"(v1.y), "=r"(v1.z), "=r"(v1.w)
                       : "r"(rbase + (uint32_t)(((c0 + 1) ^ (row & 7)) << 4)));
          uint32_t m = amax2(amax2(amax2(v0.x, v0.y), amax2(v0.z, v0.w)), amax2(amax2(v1.x, v1.y), amax2(v1.z, v1.w)));
          m = amax2(m, __shfl_xor_sync(gmask, m, 1));
          m = amax2(m, __shfl_xor_sync(gmask, m, 2));
          m = amax2(m, __shfl_xor_sync(gmask, m, 4));
          m = amax2(m, __byte_perm(m, 0, 0x1032));
          const float sc = scale_of(__uint_as_float(m & 0x7FFF0000u));
          const float ny = neg_rcp(sc);
          const uint64_t s2 = f2_pack(sc, sc), ny2 = f2_pack(ny, ny);
          const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
          uint32_t q[4];
#pragma unroll
          for (int k = 0; k < 4; ++k)
            q[k] = __byte_perm(neg_codes2(w[2 * k], s2, ny2), neg_codes2(w[2 * k + 1], s2, ny2), 0x5410) ^ 0x80808080u;
          asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(adst + (uint32_t)(row * 128) +
                                                                      (uint32_t)((chunk ^ (row & 7)) << 4)),
                       "r"(q[0]), "r"(q[1]), "r"(q[2]), "r"(q[3])
                       : "memory");
          if (chunk == 0) asm volatile("st.shared.f32 [%0], %1;" ::"r"(as_slot + 4u * (uint32_t)row), "f"(sc) : "memory");
        }
        fence_proxy_async_shared();  // the codes, for the MMA (async proxy)
        mbar_arrive(afull_bar(st));
        mbar_arrive(rempty_bar(r));
      }
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(Cfg::kEpiRegs));
    // ------------------------------------------------------------ promotion + epilogue
    const int e = warp - 8;
    const int row = epi_row(e, lane);
    const int col0 = epi_col0(e, BN, EW);
    const uint32_t lane_base = (uint32_t)(32 * (warp % 4)) << 16;
    uint32_t it = 0;
    // (M <= 16: warps of lanes 32..127 hold no row of the problem and skip the loop)
    bool ok = RAW_ROWS == 128 || warp % 4 == 0;
    for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
      const GemmTile g = gemm_tile(tile, p.num_m, p.num_n, BN);
      const bool last_tile = tile + (int)gridDim.x >= p.num_tiles;
      float acc[kCols];
#pragma unroll
      for (int j = 0; j < kCols; ++j) acc[j] = 0.0f;
      for (int kb = 0; kb < p.Kb; ++kb, ++it) {
        const uint32_t grp = it / Cfg::kScaleGroup, sub = it % Cfg::kScaleGroup;
        const int sl = (int)(grp % Cfg::kScaleSlots);
        const uint32_t slot = sScale + (uint32_t)(sl * Cfg::kScaleBytes + sub * Cfg::kScaleKbBytes);
        const bool sgot = sub != 0 || mbar_spin_bounded(sfull_bar(sl), (grp / Cfg::kScaleSlots) & 1u,
                                                        p.wait_limit_ns, abort_flag);
        const int buf = (int)(it % NT);
        const uint32_t tph = (it / NT) & 1u;
        const bool got = sgot && mbar_wait_bounded(p.debug_stall ? stall_bar : tfull_bar(buf), tph, p.wait_limit_ns,
                                                   abort_flag);
        if (!__all_sync(0xffffffffu, got)) {
          if (lane == 0) gemm_fail(sgot ? kErrWaitTmemFull : kErrWaitScale, abort_flag);
          ok = false;
          break;
        }
        tc_fence_after();
        float sa_cur, sb_cur;
        asm volatile("ld.shared.f32 %0, [%1];"
                     : "=f"(sa_cur)
                     : "r"(sbase + Cfg::kOffAs + (uint32_t)((it % Cfg::kAsSlots) * kBM * 4) + 4u * row));
        asm volatile("ld.shared.f32 %0, [%1];" : "=f"(sb_cur) : "r"(slot + 512u + 4u * (uint32_t)(col0 >> 7)));
        const float scale = sa_cur * sb_cur;
        const uint64_t scale2 = f2_pack(scale, scale);
        const uint32_t taddr = tmem_base + lane_base + (uint32_t)(buf * BN + col0);
#pragma unroll
        for (int c = 0; c < kCols / LDW; ++c) {
          uint32_t rr[LDW];
          if constexpr (LDW == 64)
            tmem_ld_32x32b_x64(taddr + (uint32_t)(LDW * c), rr);
          else
            tmem_ld_32x32b_x32(taddr + (uint32_t)(LDW * c), rr);
          tmem_ld_wait();
          tmem_regs_after_wait(rr);
          if (c == kCols / LDW - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty_bar(buf));
          }
#pragma unroll
          for (int j = 0; j < LDW; j += 2) {  // acc += (a_s * b_s) * P, two columns per fp32x2 FMA
            const uint64_t p2 = f2_pack(__uint_as_float(rr[j]), __uint_as_float(rr[j + 1]));
            f2_unpack(f2_fma(scale2, p2, f2_pack(acc[LDW * c + j], acc[LDW * c + j + 1])), acc[LDW * c + j],
                      acc[LDW * c + j + 1]);
          }
        }
        if (sub == Cfg::kScaleGroup - 1 || (last_tile && kb == p.Kb - 1)) {
          __syncwarp();
          if (lane == 0) mbar_arrive(sempty_bar(sl));
        }
      }
      if (!ok) break;
      // epilogue (as the dense kernel): rows < M and columns < N only
      constexpr int kG = kCols / 8 >= 8 ? 8 : kCols / 8;
      const int pos = lane % kG;
#pragma unroll
      for (int sg = 0; sg < kCols / (8 * kG); ++sg) {
        uint32_t X[kG][4];
#pragma unroll
        for (int j = 0; j < kG; ++j)
#pragma unroll
          for (int q = 0; q < 4; ++q)
            X[j][q] = pack_bf16x2(acc[8 * (kG * sg + j) + 2 * q], acc[8 * (kG * sg + j) + 2 * q + 1]);
#pragma unroll
        for (int msk = kG / 2; msk >= 1; msk >>= 1) {
          const bool hi = (pos & msk) != 0;
#pragma unroll
          for (int j = 0; j < kG; ++j) {
            if (j & msk) continue;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint32_t send = hi ? X[j][q] : X[j | msk][q];
              const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, msk);
              if (hi) X[j][q] = recv;
              else X[j | msk][q] = recv;
            }
          }
        }
        const int n = g.n0 + epi_store_col(e, lane, sg, kG, BN, EW);
#pragma unroll
        for (int i = 0; i < kG; ++i) {
          const int mr = g.m0 + epi_store_row(e, lane, i, kG);
          if (mr >= p.M || n >= p.N) continue;
          uint16_t* dst = p.c + (int64_t)mr * p.ldc + n;
          if (p.c_vec && n + 8 <= p.N) {
            *reinterpret_cast<uint4*>(dst) = make_uint4(X[i][0], X[i][1], X[i][2], X[i][3]);
          } else {
#pragma unroll
            for (int b = 0; b < 8; ++b)
              if (n + b < p.N) dst[b] = (uint16_t)(X[i][b >> 1] >> (16 * (b & 1)));
          }
        }
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// The weight-gradient GEMM (1x128 x 128x1) with its rhs quantised inside the
// kernel: B arrives as the bf16 activation X[K tokens, N features] and eight
// quantiser warps form, per K-block, each feature column's 128x1 group
// maximum over the block's 128 tokens, its scale and the e4m3 codes, written
// transposed (K-major, the layout the MMA reads) into the stage, with the
// quantisation kernels' arithmetic: the result equals quant_rhs followed by
// the 1x128 x 128x1 GEMM bit for bit.  This is the optional fused
// quantisation in the GEMM prologue for the weight gradient's rhs that the
// method allows ("Enable blockwise FP8 dense training kernels on ROCm":
// act_quant_rhs 128x1 and the 1x128 x 128x1 GEMM); every 128-row tile of the
// output quantises the X columns it reads again, so it trades the separate
// quantisation's HBM round trip for ceil(M/128)-fold quantisation work.
//
//   warp 0       producer: raw X tiles (two 64-feature boxes of 128 tokens)
//                into a ring of three slots, A tiles (dY^T codes) into four
//                stages
//   warps 1, 3   MMA issuers on alternate K-blocks, each waiting for the
//                K-block's A bytes and its quantised B
//   warp 2       a_s of each K-block into the scale ring
//   warps 4-11   quantisers, all eight on every K-block: warp w takes the
//                16 features 16w..16w+15 over the 128 tokens, lane (chunk c,
//                token group g) the 8 features 16w+8c.. over tokens 8g..8g+7,
//                read once into registers (in a lane-rotated token order, so
//                that a warp's 16-byte reads spread over every bank); the
//                16 token groups combine their maxima by shuffles; the codes
//                of a feature's 8 tokens are one 8-byte store into the
//                double-buffered B stage, b_s goes into a ring
//   warps 12-15  promotion (per-column scales, 128 columns a warp) + epilogue
// ---------------------------------------------------------------------------
struct WxqCfg {
  static constexpr int BN = 128;
  static constexpr int kAStages = 4;  // A tiles
  static constexpr int kBStages = 2;  // quantised B tiles
  static constexpr int kRawSlots = 3; // raw X tiles
  static constexpr int kBufs = 4;     // 128-column fp32 partial buffers in tensor memory
  static constexpr int kTmemCols = kBufs * BN;
  static constexpr int kQuantWarps = 8;
  static constexpr int kEpiWarps = 4;
  static constexpr int kCols = BN / (kEpiWarps / 4);  // 128 columns per promotion thread
  static constexpr int kThreads = 128 + 32 * kQuantWarps + 32 * kEpiWarps;  // 512
  // registers: 128 per thread at launch; control 56, quantisers 88, promotion 248
  static constexpr int kCtrlRegs = 56, kQuantRegs = 88, kEpiRegs = 248;
  static_assert(128 * kCtrlRegs + 32 * kQuantWarps * kQuantRegs + 32 * kEpiWarps * kEpiRegs <= kThreads * 128,
                "register split");
  static constexpr int kABytes = kBM * kBK;      // 16 KiB
  static constexpr int kBBytes = BN * kBK;       // 16 KiB of codes
  static constexpr int kRawBytes = kBK * BN * 2; // 128 tokens x 128 features bf16 = 32 KiB
  static constexpr int kOffB = kAStages * kABytes;
  static constexpr int kOffRaw = kOffB + kBStages * kBBytes;
  static constexpr int kScaleSlots = 2, kScaleGroup = 4;
  static constexpr int kScaleKbBytes = kBM * 4;  // a_s of the K-block's 128 rows
  static constexpr int kScaleBytes = kScaleGroup * kScaleKbBytes;
  static constexpr int kOffScale = kOffRaw + kRawSlots * kRawBytes;
  // b_s of each K-block, written by the quantisers into a ring of kBsSlots
  // entries.  The quantisers write entry `it` after the MMAs of K-block
  // it - kBStages completed; those were issued after the promotion released
  // the buffer of K-block it - kBStages - kBufs, which each promotion warp
  // does only after its last read of that K-block's b_s.  So the entry's
  // previous K-block (it - kBsSlots) has been read by then.
  static constexpr int kBsSlots = 8;
  static_assert(kBsSlots >= kBStages + kBufs, "b_s ring depth");
  static constexpr int kOffBs = kOffScale + kScaleSlots * kScaleBytes;
  static constexpr int kOffBar = kOffBs + kBsSlots * BN * 4;
  // afull[SA] aempty[SA] bfull[SB] bempty[SB] rfull[R] rempty[R] tfull[T] tempty[T] drain stall sfull[2] sempty[2]
  static constexpr int kNumBars = 2 * kAStages + 2 * kBStages + 2 * kRawSlots + 2 * kBufs + 2 + 2 * kScaleSlots;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

// 64-bit rotate left by 8*r bits (r in 0..7) of the pair (hi:lo).
__device__ __forceinline__ void rotl_bytes64(uint32_t& lo, uint32_t& hi, int r) {
  const uint32_t a = (r & 4) ? hi : lo, b = (r & 4) ? lo : hi;  // rotated by 32 when r >= 4
  const uint32_t s = 8u * (uint32_t)(r & 3);
  hi = __funnelshift_l(a, b, s);
  lo = __funnelshift_l(b, a, s);
}

__global__ void __launch_bounds__(WxqCfg::kThreads, 1)
    gemm_wgrad_xq_kernel(const __grid_constant__ CUtensorMap tma_a, const __grid_constant__ CUtensorMap tma_x,
                         const GemmParams p) {
  using Cfg = WxqCfg;
  constexpr int BN = Cfg::BN, SA = Cfg::kAStages, SB = Cfg::kBStages, NR = Cfg::kRawSlots, NT = Cfg::kBufs;
  constexpr int EW = Cfg::kEpiWarps, QW = Cfg::kQuantWarps, kCols = Cfg::kCols, LDW = 32;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sA = sbase, sB = sbase + Cfg::kOffB, sRaw = sbase + Cfg::kOffRaw;
  const uint32_t sScale = sbase + Cfg::kOffScale, sBs = sbase + Cfg::kOffBs;
  const uint32_t bar0 = sbase + Cfg::kOffBar;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + Cfg::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::kOffMisc + 4);
  volatile int* never = reinterpret_cast<volatile int*>(smem + Cfg::kOffMisc + 8);

  auto afull_bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  auto aempty_bar = [&](int i) { return bar0 + 8u * (uint32_t)(SA + i); };
  auto bfull_bar = [&](int i) { return bar0 + 8u * (uint32_t)(2 * SA + i); };
  auto bempty_bar = [&](int i) { return bar0 + 8u * (uint32_t)(2 * SA + SB + i); };
  auto rfull_bar = [&](int i) { return bar0 + 8u * (uint32_t)(2 * SA + 2 * SB + i); };
  auto rempty_bar = [&](int i) { return bar0 + 8u * (uint32_t)(2 * SA + 2 * SB + NR + i); };
  auto tfull_bar = [&](int i) { return bar0 + 8u * (uint32_t)(2 * SA + 2 * SB + 2 * NR + i); };
  auto tempty_bar = [&](int i) { return bar0 + 8u * (uint32_t)(2 * SA + 2 * SB + 2 * NR + NT + i); };
  const uint32_t drain_bar = bar0 + 8u * (uint32_t)(2 * SA + 2 * SB + 2 * NR + 2 * NT);
  const uint32_t stall_bar = drain_bar + 8u;  // never arrived on
  auto sfull_bar = [&](int i) { return drain_bar + 16u + 8u * (uint32_t)i; };
  auto sempty_bar = [&](int i) { return drain_bar + 32u + 8u * (uint32_t)i; };

  const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);
  const int lane = (int)(threadIdx.x & 31);
  pdl_launch_dependents();

  if (threadIdx.x == 0) {
    for (int i = 0; i < SA; ++i) {
      mbar_init(afull_bar(i), 1);
      mbar_init(aempty_bar(i), 1);
    }
    for (int i = 0; i < SB; ++i) {
      mbar_init(bfull_bar(i), QW);  // one arrival per quantiser warp
      mbar_init(bempty_bar(i), 1);
    }
    for (int i = 0; i < NR; ++i) {
      mbar_init(rfull_bar(i), 1);
      mbar_init(rempty_bar(i), QW);
    }
    for (int i = 0; i < NT; ++i) {
      mbar_init(tfull_bar(i), 1);
      mbar_init(tempty_bar(i), EW);
    }
    mbar_init(drain_bar, 2);
    mbar_init(stall_bar, 1);
    for (int i = 0; i < Cfg::kScaleSlots; ++i) {
      mbar_init(sfull_bar(i), 32);  // one cp.async arrival per a_s loader lane
      mbar_init(sempty_bar(i), EW);
    }
    *abort_flag = 0;
    *never = 0;
    fence_barrier_init();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), Cfg::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tma_a);
    tma_prefetch_desc(&tma_x);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_wait();  // the previous kernel's writes are visible from here on
  const uint32_t tmem_base = *tmem_holder;
  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(Cfg::kCtrlRegs));
    if (warp == 0) {
      // ---------------------------------------------------------- producer
      if (lane == 0) {
        uint32_t it = 0, n_raw = 0, n_a = 0;  // K-block steps; raw X and A copies issued
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
          const GemmTile g = gemm_tile(tile, p.num_m, p.num_n, BN);
          for (int kb = 0; kb < p.Kb; ++kb, ++it) {
            const int r = (int)(it % NR);
            if (!mbar_wait_bounded(rempty_bar(r), ((it / NR) & 1u) ^ 1u, p.wait_limit_ns, abort_flag)) {
              gemm_fail(kErrWaitEmpty, abort_flag);
              ok = false;
              break;
            }
            const uint32_t raw = sRaw + (uint32_t)(r * Cfg::kRawBytes);
            mbar_arrive_expect_tx(rfull_bar(r), (uint32_t)Cfg::kRawBytes);
            tma_load_2d(raw, &tma_x, rfull_bar(r), g.n0, kb * kBK);
            tma_load_2d(raw + (uint32_t)(Cfg::kRawBytes / 2), &tma_x, rfull_bar(r), g.n0 + 64, kb * kBK);
            ++n_raw;
            const int sa = (int)(it % SA);
            if (!mbar_wait_bounded(aempty_bar(sa), ((it / SA) & 1u) ^ 1u, p.wait_limit_ns, abort_flag)) {
              gemm_fail(kErrWaitEmpty, abort_flag);
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(afull_bar(sa), (uint32_t)Cfg::kABytes);
            tma_load_2d(sA + (uint32_t)(sa * Cfg::kABytes), &tma_a, afull_bar(sa), kb * kBK, g.m0);
            ++n_a;
          }
        }
        if (!ok) {
          // copies already issued land before this CTA's shared memory goes away
          for (uint32_t j = (n_raw > NR ? n_raw - NR : 0); j < n_raw; ++j)
            if (!mbar_wait_bounded(rfull_bar((int)(j % NR)), (j / NR) & 1u, p.wait_limit_ns, never))
              atomicOr(&g_gemm_error, kErrWaitDrain);
          for (uint32_t j = (n_a > SA ? n_a - SA : 0); j < n_a; ++j)
            if (!mbar_wait_bounded(afull_bar((int)(j % SA)), (j / SA) & 1u, p.wait_limit_ns, never))
              atomicOr(&g_gemm_error, kErrWaitDrain);
        }
      }
    } else if (warp == 1 || warp == 3) {
      // ---------------------------------------------------------- MMA issuers
      if (lane == 0) {
        constexpr uint32_t idesc = idesc_e4m3_f32(kBM, BN);
        const uint32_t mine = warp == 1 ? 0u : 1u;
        uint32_t it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
          for (int kb = 0; kb < p.Kb; ++kb, ++it) {
            if ((it & 1u) != mine) continue;
            const int sa = (int)(it % SA), sb = (int)(it % SB), buf = (int)(it % NT);
            if (!mbar_spin_bounded(tempty_bar(buf), ((it / NT) & 1u) ^ 1u, p.wait_limit_ns, abort_flag)) {
              gemm_fail(kErrWaitTmemEmpty, abort_flag);
              ok = false;
              break;
            }
            if (!mbar_spin_bounded(afull_bar(sa), (it / SA) & 1u, p.wait_limit_ns, abort_flag) ||
                !mbar_spin_bounded(bfull_bar(sb), (it / SB) & 1u, p.wait_limit_ns, abort_flag)) {
              gemm_fail(kErrWaitFull, abort_flag);
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t da = desc_kmajor_sw128(sA + (uint32_t)(sa * Cfg::kABytes));
            const uint64_t db = desc_kmajor_sw128(sB + (uint32_t)(sb * Cfg::kBBytes));
            const uint32_t d_tmem = tmem_base + (uint32_t)(buf * BN);
#pragma unroll
            for (int k = 0; k < kBK / 32; ++k)
              mma_e4m3(d_tmem, da + (uint64_t)(2 * k), db + (uint64_t)(2 * k), idesc, k > 0 ? 1u : 0u);
            mma_commit(aempty_bar(sa));
            mma_commit(bempty_bar(sb));
            mma_commit(tfull_bar(buf));
          }
        }
        mma_commit(drain_bar);
        if (!mbar_wait_bounded(drain_bar, 0, p.wait_limit_ns, never)) gemm_fail(kErrWaitDrain, abort_flag);
      }
    } else {
      // ---------------------------------------------------------- a_s loader (warp 2)
      uint32_t it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
        const GemmTile g = gemm_tile(tile, p.num_m, p.num_n, BN);
        const bool last_tile = tile + (int)gridDim.x >= p.num_tiles;
        for (int kb = 0; kb < p.Kb; ++kb, ++it) {
          const uint32_t grp = it / Cfg::kScaleGroup, sub = it % Cfg::kScaleGroup;
          const int sl = (int)(grp % Cfg::kScaleSlots);
          if (sub == 0) {
            const bool got =
                mbar_wait_bounded(sempty_bar(sl), ((grp / Cfg::kScaleSlots) & 1u) ^ 1u, p.wait_limit_ns, abort_flag);
            if (!__all_sync(0xffffffffu, got)) {
              if (lane == 0) gemm_fail(kErrWaitScale, abort_flag);
              ok = false;
              break;
            }
          }
          const uint32_t slot = sScale + (uint32_t)(sl * Cfg::kScaleBytes + sub * Cfg::kScaleKbBytes);
          // a_s of rows m0 + 4*lane .. +3 (zero past M)
          copy_scales4(slot + 16u * lane, p.sa + (int64_t)kb * p.ldsa, g.m0 + 4 * lane, p.M, p.sa_vec);
          if (sub == Cfg::kScaleGroup - 1 || (last_tile && kb == p.Kb - 1)) cp_async_mbar_arrive(sfull_bar(sl));
        }
      }
      asm volatile("cp.async.wait_all;" ::: "memory");
    }
  } else if (warp < 4 + QW) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(Cfg::kQuantRegs));
    // ------------------------------------------------------------ quantisers
    const int chunk = 2 * (warp - 4) + (lane >> 4);  // features 8*chunk .. +7
    const int g = lane & 15;                         // tokens 8g .. 8g+7
    const int rot = g & 7;                           // token order rotation of this lane
    const int jb = chunk & 7;                        // 16-byte chunk of the features in their box row
    uint32_t it = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
      for (int kb = 0; kb < p.Kb; ++kb, ++it) {
        const int r = (int)(it % NR), sb = (int)(it % SB);
        bool got = mbar_wait_bounded(rfull_bar(r), (it / NR) & 1u, p.wait_limit_ns, abort_flag);
        if (!__all_sync(0xffffffffu, got)) {
          if (lane == 0) gemm_fail(kErrWaitFull, abort_flag);
          ok = false;
          break;
        }
        // box chunk/8 of the raw tile: token t's 64 features at t*128 bytes, 16-byte chunk c at (c ^ (t & 7)).
        // Step i reads token 8g + ((i + rot) & 7): the 16 token groups of a warp then hit 8 chunk positions.
        const uint32_t box = sRaw + (uint32_t)(r * Cfg::kRawBytes + (chunk >> 3) * (Cfg::kRawBytes / 2));
        uint4 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int ph = (i + rot) & 7;
          asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                       : "=r"(v[i].x), "=r"(v[i].y), "=r"(v[i].z), "=r"(v[i].w)
                       : "r"(box + (uint32_t)((8 * g + ph) * 128) + (uint32_t)((jb ^ ph) << 4)));
        }
        // the values are in registers: the raw slot can be refilled
        __syncwarp();
        if (lane == 0) mbar_arrive(rempty_bar(r));
        // |x| maxima of the 8 features (packed bf16 pairs) over the 128 tokens
        uint32_t m[4];
        m[0] = amax2(amax2(amax2(v[0].x, v[1].x), amax2(v[2].x, v[3].x)), amax2(amax2(v[4].x, v[5].x), amax2(v[6].x, v[7].x)));
        m[1] = amax2(amax2(amax2(v[0].y, v[1].y), amax2(v[2].y, v[3].y)), amax2(amax2(v[4].y, v[5].y), amax2(v[6].y, v[7].y)));
        m[2] = amax2(amax2(amax2(v[0].z, v[1].z), amax2(v[2].z, v[3].z)), amax2(amax2(v[4].z, v[5].z), amax2(v[6].z, v[7].z)));
        m[3] = amax2(amax2(amax2(v[0].w, v[1].w), amax2(v[2].w, v[3].w)), amax2(amax2(v[4].w, v[5].w), amax2(v[6].w, v[7].w)));
        uint64_t s2[4], ny2[4];  // (s, s') and (-1/s, -1/s') of features 8*chunk + 2q, +1
#pragma unroll
        for (int q = 0; q < 4; ++q) {
#pragma unroll
          for (int d = 1; d < 16; d <<= 1) m[q] = amax2(m[q], __shfl_xor_sync(0xffffffffu, m[q], d));
          const float s_lo = scale_of(__uint_as_float((m[q] << 16) & 0x7FFF0000u));
          const float s_hi = scale_of(__uint_as_float(m[q] & 0x7FFF0000u));
          s2[q] = f2_pack(s_lo, s_hi);
          ny2[q] = f2_pack(neg_rcp(s_lo), neg_rcp(s_hi));
        }
        // the B stage and the b_s ring entry are free once the MMAs of K-block it - kBStages completed
        got = mbar_wait_bounded(bempty_bar(sb), ((it / SB) & 1u) ^ 1u, p.wait_limit_ns, abort_flag);
        if (!__all_sync(0xffffffffu, got)) {
          if (lane == 0) gemm_fail(kErrWaitEmpty, abort_flag);
          ok = false;
          break;
        }
        if (g == 0) {
          const uint32_t bs = sBs + (uint32_t)((it % Cfg::kBsSlots) * BN * 4 + 4 * (8 * chunk));
          float lo[4], hi[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) f2_unpack(s2[q], lo[q], hi[q]);
          asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(bs), "f"(lo[0]), "f"(hi[0]), "f"(lo[1]),
                       "f"(hi[1])
                       : "memory");
          asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(bs + 16u), "f"(lo[2]), "f"(hi[2]),
                       "f"(lo[3]), "f"(hi[3])
                       : "memory");
        }
        // codes: per feature pair q, the 8 steps' codes -> one 8-byte word per feature, in step order
        // (byte i = token 8g + ((i + rot) & 7)), rotated into token order, stored at row f, bytes 8g..8g+7
        const uint32_t bdst = sB + (uint32_t)(sb * Cfg::kBBytes);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t fe[2], fo[2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t cc[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint4& w4 = v[4 * h + i];
              const uint32_t w = q == 0 ? w4.x : q == 1 ? w4.y : q == 2 ? w4.z : w4.w;
              cc[i] = neg_codes2(w, s2[q], ny2[q]);  // byte 0: feature 8*chunk+2q, byte 1: +1
            }
            const uint32_t X = __byte_perm(cc[0], cc[1], 0x5140), Y = __byte_perm(cc[2], cc[3], 0x5140);
            fe[h] = __byte_perm(X, Y, 0x5410) ^ 0x80808080u;
            fo[h] = __byte_perm(X, Y, 0x7632) ^ 0x80808080u;
          }
          rotl_bytes64(fe[0], fe[1], rot);
          rotl_bytes64(fo[0], fo[1], rot);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int f = 8 * chunk + 2 * q + h;
            const uint32_t lo = h ? fo[0] : fe[0], hi = h ? fo[1] : fe[1];
            asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(bdst + (uint32_t)(f * 128) +
                                                                 (uint32_t)(((g >> 1) ^ (f & 7)) << 4) +
                                                                 (uint32_t)(8 * (g & 1))),
                         "r"(lo), "r"(hi)
                         : "memory");
          }
        }
        fence_proxy_async_shared();  // the codes, for the MMA (async proxy)
        __syncwarp();
        if (lane == 0) mbar_arrive(bfull_bar(sb));
      }
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(Cfg::kEpiRegs));
    // ------------------------------------------------------------ promotion + epilogue
    const int e = warp - 4 - QW;
    const int row = epi_row(e, lane);
    const int col0 = epi_col0(e, BN, EW);
    const uint32_t lane_base = (uint32_t)(32 * (warp % 4)) << 16;
    uint32_t it = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
      const GemmTile gt = gemm_tile(tile, p.num_m, p.num_n, BN);
      const bool last_tile = tile + (int)gridDim.x >= p.num_tiles;
      float acc[kCols];
#pragma unroll
      for (int jj = 0; jj < kCols; ++jj) acc[jj] = 0.0f;
      for (int kb = 0; kb < p.Kb; ++kb, ++it) {
        const uint32_t grp = it / Cfg::kScaleGroup, sub = it % Cfg::kScaleGroup;
        const int sl = (int)(grp % Cfg::kScaleSlots);
        const uint32_t slot = sScale + (uint32_t)(sl * Cfg::kScaleBytes + sub * Cfg::kScaleKbBytes);
        const bool sgot = sub != 0 || mbar_spin_bounded(sfull_bar(sl), (grp / Cfg::kScaleSlots) & 1u,
                                                        p.wait_limit_ns, abort_flag);
        const int buf = (int)(it % NT);
        const bool got = sgot && mbar_wait_bounded(p.debug_stall ? stall_bar : tfull_bar(buf), (it / NT) & 1u,
                                                   p.wait_limit_ns, abort_flag);
        if (!__all_sync(0xffffffffu, got)) {
          if (lane == 0) gemm_fail(sgot ? kErrWaitTmemFull : kErrWaitScale, abort_flag);
          ok = false;
          break;
        }
        tc_fence_after();
        float sa_cur;
        asm volatile("ld.shared.f32 %0, [%1];" : "=f"(sa_cur) : "r"(slot + 4u * row));
        const uint64_t sa2 = f2_pack(sa_cur, sa_cur);
        const uint32_t bs = sBs + (uint32_t)((it % Cfg::kBsSlots) * BN * 4);
        const uint32_t taddr = tmem_base + lane_base + (uint32_t)(buf * BN + col0);
#pragma unroll
        for (int c = 0; c < kCols / LDW; ++c) {
          uint32_t rr[LDW];
          tmem_ld_32x32b_x32(taddr + (uint32_t)(LDW * c), rr);
          tmem_ld_wait();
          tmem_regs_after_wait(rr);
          // acc[n] += (a_s * b_s[n]) * P[n] on fp32x2 lanes, as the 1x128 x 128x1 GEMM
#pragma unroll
          for (int j4 = 0; j4 < LDW / 4; ++j4) {
            float4 sb4;
            asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                         : "=f"(sb4.x), "=f"(sb4.y), "=f"(sb4.z), "=f"(sb4.w)
                         : "r"(bs + 4u * (uint32_t)(col0 + LDW * c + 4 * j4)));
            const uint64_t t2[2] = {f2_mul(sa2, f2_pack(sb4.x, sb4.y)), f2_mul(sa2, f2_pack(sb4.z, sb4.w))};
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int jj = LDW * c + 4 * j4 + 2 * h;
              const uint64_t p2 = f2_pack(__uint_as_float(rr[4 * j4 + 2 * h]), __uint_as_float(rr[4 * j4 + 2 * h + 1]));
              f2_unpack(f2_fma(t2[h], p2, f2_pack(acc[jj], acc[jj + 1])), acc[jj], acc[jj + 1]);
            }
          }
        }
        // the partial and this K-block's b_s have been read: release the buffer
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty_bar(buf));
        if (sub == Cfg::kScaleGroup - 1 || (last_tile && kb == p.Kb - 1)) {
          __syncwarp();
          if (lane == 0) mbar_arrive(sempty_bar(sl));
        }
      }
      if (!ok) break;
      // epilogue (as the dense kernel): rows < M and columns < N only
      constexpr int kG = 8;
      const int pos = lane % kG;
#pragma unroll
      for (int sg = 0; sg < kCols / (8 * kG); ++sg) {
        uint32_t X[kG][4];
#pragma unroll
        for (int jj = 0; jj < kG; ++jj)
#pragma unroll
          for (int q = 0; q < 4; ++q)
            X[jj][q] = pack_bf16x2(acc[8 * (kG * sg + jj) + 2 * q], acc[8 * (kG * sg + jj) + 2 * q + 1]);
#pragma unroll
        for (int msk = kG / 2; msk >= 1; msk >>= 1) {
          const bool hi = (pos & msk) != 0;
#pragma unroll
          for (int jj = 0; jj < kG; ++jj) {
            if (jj & msk) continue;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint32_t send = hi ? X[jj][q] : X[jj | msk][q];
              const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, msk);
              if (hi) X[jj][q] = recv;
              else X[jj | msk][q] = recv;
            }
          }
        }
        const int n = gt.n0 + epi_store_col(e, lane, sg, kG, BN, EW);
#pragma unroll
        for (int i = 0; i < kG; ++i) {
          const int mr = gt.m0 + epi_store_row(e, lane, i, kG);
          if (mr >= p.M || n >= p.N) continue;
          uint16_t* dst = p.c + (int64_t)mr * p.ldc + n;
          if (p.c_vec && n + 8 <= p.N) {
            *reinterpret_cast<uint4*>(dst) = make_uint4(X[i][0], X[i][1], X[i][2], X[i][3]);
          } else {
#pragma unroll
            for (int b = 0; b < 8; ++b)
              if (n + b < p.N) dst[b] = (uint16_t)(X[i][b >> 1] >> (16 * (b & 1)));
          }
        }
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// Small-M GEMM (1x128 x 128x128, at most 32 rows of A): the operands swap
// places in the MMA.  W's 128 rows of a tile are the instruction's A (M = 128)
// and the R rows of A (R = 16 or 32, the smaller that holds them) its B
// (N = R), so that every instruction consumes 4 KiB of the weight, the
// operand streamed from DRAM, and the partial product of a K-block is a
// 128 x R block of tensor memory: lane n, column m.  Each tile's K-blocks are
// split over the S CTAs of a cluster (contiguous ranges); every CTA promotes
// its range as the dense kernel does (acc += (a_s * b_s) * P per K-block, the
// same fp32 operations).  With S > 1 every CTA then leaves its 128 x R
// partial sums in its idle W stages, and CTA s of the cluster adds rows
// s R/S .. (s+1) R/S - 1 of all S partials in rank order through distributed
// shared memory and stores them (bf16), between two cluster barriers.  With
// XQ the rows of A arrive as bf16 x and four quantiser warps form their 1x128
// groups in the kernel (the forward that quantises x itself), with the
// quantisation kernels' arithmetic.  (Measured with R = 64 and 128 as well,
// this form was slower than the dense kernel's tiles beyond 32 rows.)
//
//   warp 0       producer: W tiles (128 rows) and A tiles (R rows; bf16 x
//                with XQ) of the CTA's K-range into the stage ring
//   warps 1, 3   MMA issuers (M = 128, N = R) on alternate K-blocks
//   warp 2       a_s (without XQ) and the tile's b_s of each K-block
//   warps 4-7    promotion (lane n: column n of C, its R rows), reduction,
//                stores
//   warps 8-11   (XQ) quantisers: thread (row, 16-column chunk) for each group
//                of 16 rows, as the dense forward's quantiser for 16 rows
// ---------------------------------------------------------------------------
template <bool XQ, int R>
struct SmallCfg {
  static_assert(R == 16 || R == 32, "rows of A");
  static constexpr int kRows = R;                   // the MMA's N
  static constexpr int kStages = XQ && R == 32 ? 6 : 8;
  static constexpr int kBufs = 8;                   // R-column partial buffers in tensor memory
  static constexpr int kTmemCols = kBufs * R;       // 128 or 256
  static constexpr int kPromoWarps = 4;
  static constexpr int kCols = R;                   // rows of A per promotion thread
  static constexpr int kChunk = R;                  // columns per tensor-memory load
  static constexpr int kThreads = 128 + 32 * kPromoWarps + (XQ ? 128 : 0);
  static constexpr int kWBytes = kBM * kBK;                  // 16 KiB
  static constexpr int kXBytes = R * kBK;                    // codes of the R rows
  static constexpr int kRawBytes = XQ ? R * kBK * 2 : 0;     // bf16 x (two 64-column boxes)
  static constexpr int kSlotBytes = (4 * R + 16 + 127) / 128 * 128;  // a_s[R], then b_s at byte 4R
  static constexpr int kOffX = kStages * kWBytes;
  static constexpr int kOffRaw = kOffX + kStages * kXBytes;
  static constexpr int kOffSlot = kOffRaw + kStages * kRawBytes;
  static constexpr int kOffBar = kOffSlot + kStages * kSlotBytes;
  // full[S] empty[S] sfull[S] sempty[S] qfull[S] rfull[S] tfull[T] tempty[T] drain stall
  static constexpr int kNumBars = 6 * kStages + 2 * kBufs + 2;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;
  // once the K-loop is over, the 128 x R partial sums sit in the W stages
  static_assert(kBM * R * 4 <= kStages * kWBytes, "partial sums fit in the W stages");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

// Splits the reduction supports: S = 2, 4 or 8 divides R, and each promotion
// thread's share of a CTA's rows is at least two values (8-byte loads).
constexpr int kSmallMaxSplits = 8;

// The partial sums of lane n: R fp32 in 16-byte chunks, chunk c stored at
// position c ^ smallm_swz(n), so that a warp's 32 lanes (rows R*4 bytes
// apart) spread over all eight 16-byte bank groups.
template <int R>
__device__ __forceinline__ uint32_t smallm_part_addr(uint32_t part, int n, int m) {
  const int swz = R >= 32 ? (n & 7) : ((n >> 1) & (R / 4 - 1));
  return part + (uint32_t)(n * R * 4) + (uint32_t)((((m >> 2) ^ swz) << 4) + (m & 3) * 4);
}

// CTA `rank` of S: rows rank R/S .. of the tile, summed over the S partials
// (at `part` in every CTA's shared memory, 128 x R fp32 by lane n, chunks
// swizzled) in rank order and stored as bf16.  Thread (nl, h): column
// n0 + nl, rows rank R/S + h CW .. + CW - 1.
template <int R, int PW, int S>
__device__ __forceinline__ void smallm_reduce_store(uint32_t part, int rank, int nl, int h, int n0, const GemmParams& p) {
  constexpr int CW = R / S / (PW / 4);
  static_assert(CW % 2 == 0, "whole 8-byte loads");
  const int m0 = rank * (R / S) + h * CW;
  float v[S][CW];
#pragma unroll
  for (int s = 0; s < S; ++s) {
    if constexpr (CW % 4 == 0) {
#pragma unroll
      for (int q = 0; q < CW / 4; ++q) {
        const float4 t = lds128_cluster(mapa_shared(smallm_part_addr<R>(part, nl, m0 + 4 * q), (uint32_t)s));
        v[s][4 * q] = t.x;
        v[s][4 * q + 1] = t.y;
        v[s][4 * q + 2] = t.z;
        v[s][4 * q + 3] = t.w;
      }
    } else {
#pragma unroll
      for (int q = 0; q < CW / 2; ++q) {
        const float2 t = lds64_cluster(mapa_shared(smallm_part_addr<R>(part, nl, m0 + 2 * q), (uint32_t)s));
        v[s][2 * q] = t.x;
        v[s][2 * q + 1] = t.y;
      }
    }
  }
  const int64_t n = n0 + nl;
  if (n >= p.N) return;
#pragma unroll
  for (int j = 0; j < CW; ++j) {
    float sum = v[0][j];
#pragma unroll
    for (int s = 1; s < S; ++s) sum += v[s][j];
    const int64_t m = m0 + j;
    if (m < p.M) p.c[m * p.ldc + n] = (uint16_t)(pack_bf16x2(sum, 0.0f) & 0xFFFFu);
  }
}

template <int SB_MODE, bool XQ, int R>
__global__ void __launch_bounds__(SmallCfg<XQ, R>::kThreads, 1)
    gemm_smallm_kernel(const __grid_constant__ CUtensorMap tma_w, const __grid_constant__ CUtensorMap tma_x,
                       const GemmParams p, const int splits) {
  using Cfg = SmallCfg<XQ, R>;
  static_assert(SB_MODE == kSbTile || SB_MODE == kSbTileT, "tile-scale modes");
  constexpr int ST = Cfg::kStages, NT = Cfg::kBufs, PW = Cfg::kPromoWarps;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sW = sbase, sX = sbase + Cfg::kOffX, sRaw = sbase + Cfg::kOffRaw;
  const uint32_t sSlot = sbase + Cfg::kOffSlot;
  const uint32_t bar0 = sbase + Cfg::kOffBar;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + Cfg::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::kOffMisc + 4);
  volatile int* never = reinterpret_cast<volatile int*>(smem + Cfg::kOffMisc + 8);
  auto full_bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  auto empty_bar = [&](int i) { return bar0 + 8u * (uint32_t)(ST + i); };
  auto sfull_bar = [&](int i) { return bar0 + 8u * (uint32_t)(2 * ST + i); };
  auto sempty_bar = [&](int i) { return bar0 + 8u * (uint32_t)(3 * ST + i); };
  auto qfull_bar = [&](int i) { return bar0 + 8u * (uint32_t)(4 * ST + i); };
  auto rfull_bar = [&](int i) { return bar0 + 8u * (uint32_t)(5 * ST + i); };
  auto tfull_bar = [&](int i) { return bar0 + 8u * (uint32_t)(6 * ST + i); };
  auto tempty_bar = [&](int i) { return bar0 + 8u * (uint32_t)(6 * ST + NT + i); };
  const uint32_t drain_bar = bar0 + 8u * (uint32_t)(6 * ST + 2 * NT);
  const uint32_t stall_bar = drain_bar + 8u;  // never arrived on

  const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);
  const int lane = (int)(threadIdx.x & 31);
  const int tile = (int)blockIdx.x / splits, split = (int)blockIdx.x % splits;  // split = rank in the cluster
  const int n0 = tile * kBM;
  const int kb0 = smallm_kb_lo(split, splits, p.Kb), kbn = smallm_kb_lo(split + 1, splits, p.Kb) - kb0;
  pdl_launch_dependents();
  // copy issue of K-block j of the CTA's range (producer thread)
  auto issue = [&](int j) {
    const int st = j % ST, kb = kb0 + j;
    mbar_arrive_expect_tx(full_bar(st), (uint32_t)(Cfg::kWBytes + (XQ ? 0 : Cfg::kXBytes)));
    tma_load_2d(sW + (uint32_t)(st * Cfg::kWBytes), &tma_w, full_bar(st), kb * kBK, n0);
    if constexpr (XQ) {
      const uint32_t raw = sRaw + (uint32_t)(st * Cfg::kRawBytes);
      mbar_arrive_expect_tx(rfull_bar(st), (uint32_t)Cfg::kRawBytes);
      tma_load_2d(raw, &tma_x, rfull_bar(st), kb * kBK, 0);
      tma_load_2d(raw + (uint32_t)(Cfg::kRawBytes / 2), &tma_x, rfull_bar(st), kb * kBK + 64, 0);
    } else {
      tma_load_2d(sX + (uint32_t)(st * Cfg::kXBytes), &tma_x, full_bar(st), kb * kBK, 0);
    }
  };
  const int first = kbn < ST ? kbn : ST;  // K-blocks whose stages are fresh
  if (threadIdx.x == 0) {
    for (int i = 0; i < ST; ++i) {
      mbar_init(full_bar(i), 1);
      mbar_init(empty_bar(i), 1);
      mbar_init(sfull_bar(i), 32);  // one cp.async arrival per loader lane
      mbar_init(sempty_bar(i), PW); // the promotion warps
      mbar_init(qfull_bar(i), 128); // the quantiser threads (XQ)
      mbar_init(rfull_bar(i), 1);
    }
    for (int i = 0; i < NT; ++i) {
      mbar_init(tfull_bar(i), 1);
      mbar_init(tempty_bar(i), PW);
    }
    mbar_init(drain_bar, 2);  // one commit per issuer
    mbar_init(stall_bar, 1);
    *abort_flag = 0;
    *never = 0;
    fence_barrier_init();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    // the first stages' copies go out before the CTA-wide set-up completes
    tma_prefetch_desc(&tma_w);
    tma_prefetch_desc(&tma_x);
    pdl_wait();  // the previous kernel's writes are visible from here on
    for (int j = 0; j < first; ++j) issue(j);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_wait();
  const uint32_t tmem_base = *tmem_holder;
  const bool promo = warp >= 4 && warp < 4 + PW;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int j = first;
      bool ok = true;
      for (; j < kbn; ++j) {
        if (!mbar_wait_bounded(empty_bar(j % ST), ((j / ST) & 1) ^ 1, p.wait_limit_ns, abort_flag)) {
          gemm_fail(kErrWaitEmpty, abort_flag);
          ok = false;
          break;
        }
        issue(j);
      }
      if (!ok) {
        // copies already issued land before this CTA's shared memory goes away
        for (int i = (j > ST ? j - ST : 0); i < j; ++i) {
          if (!mbar_wait_bounded(full_bar(i % ST), (i / ST) & 1, p.wait_limit_ns, never))
            atomicOr(&g_gemm_error, kErrWaitDrain);
          if (XQ && !mbar_wait_bounded(rfull_bar(i % ST), (i / ST) & 1, p.wait_limit_ns, never))
            atomicOr(&g_gemm_error, kErrWaitDrain);
        }
      }
    }
  } else if (warp == 1 || warp == 3) {
    // ------------------------------------------------------------ MMA issuers (alternate K-blocks)
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_e4m3_f32(kBM, R);
      for (int j = warp == 1 ? 0 : 1; j < kbn; j += 2) {
        const int st = j % ST, buf = j % NT;
        if (!mbar_spin_bounded(tempty_bar(buf), ((j / NT) & 1) ^ 1, p.wait_limit_ns, abort_flag)) {
          gemm_fail(kErrWaitTmemEmpty, abort_flag);
          break;
        }
        if (!mbar_spin_bounded(full_bar(st), (j / ST) & 1, p.wait_limit_ns, abort_flag) ||
            (XQ && !mbar_spin_bounded(qfull_bar(st), (j / ST) & 1, p.wait_limit_ns, abort_flag))) {
          gemm_fail(kErrWaitFull, abort_flag);
          break;
        }
        tc_fence_after();
        const uint64_t da = desc_kmajor_sw128(sW + (uint32_t)(st * Cfg::kWBytes));
        const uint64_t db = desc_kmajor_sw128(sX + (uint32_t)(st * Cfg::kXBytes));
        const uint32_t d_tmem = tmem_base + (uint32_t)(buf * R);
#pragma unroll
        for (int k = 0; k < kBK / 32; ++k)
          mma_e4m3(d_tmem, da + (uint64_t)(2 * k), db + (uint64_t)(2 * k), idesc, k > 0 ? 1u : 0u);
        mma_commit(empty_bar(st));
        mma_commit(tfull_bar(buf));
      }
      // every MMA issued completes before tensor memory is released
      mma_commit(drain_bar);
      if (!mbar_wait_bounded(drain_bar, 0, p.wait_limit_ns, never)) gemm_fail(kErrWaitDrain, abort_flag);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ scale loader
    const int nbk = n0 / kBlock;
    const bool nin = nbk < p.Nb;
    for (int j = 0; j < kbn; ++j) {
      const int st = j % ST, kb = kb0 + j;
      const bool got = mbar_wait_bounded(sempty_bar(st), ((j / ST) & 1) ^ 1, p.wait_limit_ns, abort_flag);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) gemm_fail(kErrWaitScale, abort_flag);
        break;
      }
      const uint32_t slot = sSlot + (uint32_t)(st * Cfg::kSlotBytes);
      // a_s of rows 4*lane .. +3 (zero past M)
      if (!XQ && lane < R / 4) copy_scales4(slot + 16u * lane, p.sa + (int64_t)kb * p.ldsa, 4 * lane, p.M, p.sa_vec);
      if (lane == 0) {  // the tile scale of W's 128 x 128 block (nbk, kb)
        const float* src = SB_MODE == kSbTile ? p.sb + (int64_t)nbk * p.ldsb + kb : p.sb + (int64_t)kb * p.ldsb + nbk;
        cp_async_4(slot + 4u * R, nin ? src : p.sb, nin ? 4u : 0u);
      }
      cp_async_mbar_arrive(sfull_bar(st));
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (promo) {
    // ------------------------------------------------------------ promotion
    const int e = warp - 4;
    const int nl = 32 * (e % 4) + lane;  // tensor-memory lane = column n0 + nl
    const int h = e / 4;                 // rows h * kCols .. of A
    const uint32_t lane_base = (uint32_t)(32 * (e % 4)) << 16;
    float acc[Cfg::kCols];
#pragma unroll
    for (int m = 0; m < Cfg::kCols; ++m) acc[m] = 0.0f;
    bool ok = true;
    for (int j = 0; j < kbn; ++j) {
      const int st = j % ST, buf = j % NT;
      const bool sgot = mbar_wait_bounded(sfull_bar(st), (j / ST) & 1, p.wait_limit_ns, abort_flag);
      const bool got = sgot && mbar_wait_bounded(p.debug_stall ? stall_bar : tfull_bar(buf), (j / NT) & 1,
                                                 p.wait_limit_ns, abort_flag);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) gemm_fail(sgot ? kErrWaitTmemFull : kErrWaitScale, abort_flag);
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t slot = sSlot + (uint32_t)(st * Cfg::kSlotBytes) + 4u * (uint32_t)(h * Cfg::kCols);
      float bsc;
      asm volatile("ld.shared.f32 %0, [%1];" : "=f"(bsc) : "r"(sSlot + (uint32_t)(st * Cfg::kSlotBytes) + 4u * R));
      const uint64_t b2 = f2_pack(bsc, bsc);
#pragma unroll
      for (int c = 0; c < Cfg::kCols / Cfg::kChunk; ++c) {
        uint32_t r[Cfg::kChunk];
        const uint32_t taddr = tmem_base + lane_base + (uint32_t)(buf * R + h * Cfg::kCols + c * Cfg::kChunk);
        if constexpr (Cfg::kChunk == 32)
          tmem_ld_32x32b_x32(taddr, r);
        else
          tmem_ld_32x32b_x16(taddr, r);
        tmem_ld_wait();
        tmem_regs_after_wait(r);
        // acc[m] += (a_s[m] * b_s) * P[m], two rows per fp32x2 operation
#pragma unroll
        for (int q = 0; q < Cfg::kChunk / 4; ++q) {
          float4 a4;
          asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                       : "=f"(a4.x), "=f"(a4.y), "=f"(a4.z), "=f"(a4.w)
                       : "r"(slot + 4u * (uint32_t)(c * Cfg::kChunk + 4 * q)));
          const int m = c * Cfg::kChunk + 4 * q;
          const uint64_t s01 = f2_mul(f2_pack(a4.x, a4.y), b2), s23 = f2_mul(f2_pack(a4.z, a4.w), b2);
          f2_unpack(f2_fma(s01, f2_pack(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1])),
                           f2_pack(acc[m], acc[m + 1])),
                    acc[m], acc[m + 1]);
          f2_unpack(f2_fma(s23, f2_pack(__uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3])),
                           f2_pack(acc[m + 2], acc[m + 3])),
                    acc[m + 2], acc[m + 3]);
        }
      }
      // the partial and the scales have been read: release the buffer and the slot
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(tempty_bar(buf));
        mbar_arrive(sempty_bar(st));
      }
    }
    if (splits == 1) {
      const int64_t n = n0 + nl;
      if (ok && n < p.N) {
#pragma unroll
        for (int m = 0; m < Cfg::kCols; ++m)
          if (h * Cfg::kCols + m < p.M)
            p.c[(int64_t)(h * Cfg::kCols + m) * p.ldc + n] = (uint16_t)(pack_bf16x2(acc[m], 0.0f) & 0xFFFFu);
      }
    } else if (ok) {
      // the K-loop is over (every MMA has completed, every copy has landed): the
      // partial sums go into the W stages
#pragma unroll
      for (int q = 0; q < Cfg::kCols / 4; ++q)
        asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(smallm_part_addr<R>(sW, nl, h * Cfg::kCols + 4 * q)),
                     "f"(acc[4 * q]),
                     "f"(acc[4 * q + 1]), "f"(acc[4 * q + 2]), "f"(acc[4 * q + 3])
                     : "memory");
    }
  } else if (XQ && warp >= 4 + PW) {
    // ------------------------------------------------------------ quantisers (XQ)
    const int qt = (int)threadIdx.x - (128 + 32 * PW);
    const int chunk = qt & 7;  // 16 columns of the K-block
    const int row16 = qt >> 3; // rows row16, row16 + 16, ..
    const uint32_t gmask = 0xFFu << (8 * (lane >> 3));  // the 8 lanes of this thread's row
    for (int j = 0; j < kbn; ++j) {
      const int st = j % ST;
      // raw x landed; the stage's codes and a_s were consumed by the MMA and the promotion of K-block j - ST
      const bool got = mbar_wait_bounded(rfull_bar(st), (j / ST) & 1, p.wait_limit_ns, abort_flag) &&
                       mbar_wait_bounded(empty_bar(st), ((j / ST) & 1) ^ 1, p.wait_limit_ns, abort_flag) &&
                       mbar_wait_bounded(sempty_bar(st), ((j / ST) & 1) ^ 1, p.wait_limit_ns, abort_flag);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) gemm_fail(kErrWaitFull, abort_flag);
        break;
      }
      const uint32_t raw = sRaw + (uint32_t)(st * Cfg::kRawBytes);
#pragma unroll
      for (int g = 0; g < R / 16; ++g) {
        const int row = row16 + 16 * g;
        // 16 bf16 values: 16-byte chunks 2*(chunk%4) and +1 of box chunk/4 (128-byte swizzle)
        const uint32_t rbase = raw + (uint32_t)((chunk >> 2) * (Cfg::kRawBytes / 2) + row * 128);
        const int c0 = 2 * (chunk & 3);
        uint4 v0, v1;
        asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(v0.x), "=r"(v0.y), "=r"(v0.z), "=r"(v0.w)
                     : "r"(rbase + (uint32_t)(((c0) ^ (row & 7)) << 4)));
        asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(v1.x), "=r"(v1.y), "=r"(v1.z), "=r"(v1.w)
                     : "r"(rbase + (uint32_t)(((c0 + 1) ^ (row & 7)) << 4)));
        uint32_t m = amax2(amax2(amax2(v0.x, v0.y), amax2(v0.z, v0.w)), amax2(amax2(v1.x, v1.y), amax2(v1.z, v1.w)));
        m = amax2(m, __shfl_xor_sync(gmask, m, 1));
        m = amax2(m, __shfl_xor_sync(gmask, m, 2));
        m = amax2(m, __shfl_xor_sync(gmask, m, 4));
        m = amax2(m, __byte_perm(m, 0, 0x1032));
        const float sc = scale_of(__uint_as_float(m & 0x7FFF0000u));
        const float ny = neg_rcp(sc);
        const uint64_t s2 = f2_pack(sc, sc), ny2 = f2_pack(ny, ny);
        const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        uint32_t q[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
          q[k] = __byte_perm(neg_codes2(w[2 * k], s2, ny2), neg_codes2(w[2 * k + 1], s2, ny2), 0x5410) ^ 0x80808080u;
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(sX + (uint32_t)(st * Cfg::kXBytes + row * 128) +
                                                                    (uint32_t)((chunk ^ (row & 7)) << 4)),
                     "r"(q[0]), "r"(q[1]), "r"(q[2]), "r"(q[3])
                     : "memory");
        if (chunk == 0)
          asm volatile("st.shared.f32 [%0], %1;" ::"r"(sSlot + (uint32_t)(st * Cfg::kSlotBytes) + 4u * (uint32_t)row),
                       "f"(sc)
                       : "memory");
      }
      fence_proxy_async_shared();  // the codes, for the MMA (async proxy)
      mbar_arrive(qfull_bar(st));
    }
  }

  __syncwarp();
  if (splits > 1) {
    // Every thread of every CTA of the cluster reaches both barriers (no role
    // leaves the kernel early, and every wait before them is bounded): the
    // first makes every CTA's partial sums visible, the second keeps each CTA
    // resident until no peer reads its shared memory any more.  A CTA whose
    // pipeline gave up has written no partial sums and flagged the error; the
    // sums stored from it are then not meaningful.
    cluster_sync_all();
    if (promo) {
      const int e = warp - 4;
      const int nl = 32 * (e % 4) + lane, h = e / 4;
      if (splits == 2) smallm_reduce_store<R, PW, 2>(sW, split, nl, h, n0, p);
      else if (splits == 4) smallm_reduce_store<R, PW, 4>(sW, split, nl, h, n0, p);
      else smallm_reduce_store<R, PW, 8>(sW, split, nl, h, n0, p);
    }
    __syncwarp();
    cluster_sync_all();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// Row-major [rows, inner] uint8 matrix with row stride ld bytes; box of
// 128 bytes x box_rows rows, 128-byte swizzle, out-of-range reads filled with 0.
static bool make_tma_u8(CUtensorMap* map, const void* base, int64_t inner, int64_t rows, int64_t ld,
                        int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld};
  cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
  cuuint32_t elem[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
                  elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

static bool make_tma_bf16(CUtensorMap* map, const void* base, int64_t inner, int64_t rows, int64_t ld_bytes,
                          int box_rows);

int gemm_pick_bn(int64_t M, int64_t N, bool col_scales, int num_sms) {
  // Problems whose 128-column tiles would occupy at most half the SMs (small
  // M: decoding, skinny layers) take narrow tiles with more tensor-memory
  // buffers: more CTAs streaming B, and MMAs that run ahead of the
  // promotion.  32 columns where those tiles still fit in one wave of SMs
  // (every CTA reads all of A through its own L2 port, so a CTA's bytes per
  // K-block, 16 KiB of A + BN x 128 of B, set its pace), else 64.
  // (1x128 x 128x128 modes only: the column-scale GEMM reduces over tokens
  // and is not small in both M and N.)
  if (!col_scales && cdiv(M, kBM) * cdiv(N, 32) <= num_sms) return 32;
  if (!col_scales && 2 * cdiv(M, kBM) * cdiv(N, 128) <= num_sms) return 64;
  if (N <= 128) return 128;
  const int64_t tiles256 = cdiv(M, kBM) * cdiv(N, 256);
  if (tiles256 < num_sms) return 128;
  // The 1x128 x 128x1 GEMM takes 224-column tiles where they fill the last
  // wave of SMs better: a tile's time taken as proportional to its width, 224
  // is chosen when its waves x width come out at least 5% below 256's (4096 x
  // 4096: 608 tiles = 4 whole waves of 152 against 3.37 of 256 columns).
  // (Measured: 4096 x 4096 x 8192 154 vs 164 us.  The 1x128 x 128x128 GEMMs
  // measured slower with them, 2048 x 4096 x 4096 43.6 vs 41.6 us.)
  if (!col_scales) return 256;
  const int64_t tiles224 = cdiv(M, kBM) * cdiv(N, 224);
  const int64_t cost256 = cdiv(tiles256, num_sms) * 256, cost224 = cdiv(tiles224, num_sms) * 224;
  return cost224 * 20 <= cost256 * 19 ? 224 : 256;
}

int64_t gemm_grid(int64_t M, int64_t N, int bn, int num_sms) {
  const int64_t tiles = cdiv(M, kBM) * cdiv(N, bn);
  return tiles < num_sms ? tiles : num_sms;
}

// Promotion warps per tile shape and mode (measured): 16 for the 256-column
// tiles and for the column-scale mode (more warps read tensor memory faster;
// the 2048x4096x4096 input gradient 43.0 -> 40.9 us, the 16384x14336x4096
// forward 818 -> 794 us), 8 for the 128- and 64-column tile-scale tiles
// (few-tile shapes: 16 measured slower there); and columns per tensor-memory
// load (one round trip per LDW columns of a warp's share, sized to the
// promotion warps' registers).
template <int MODE, int BN>
constexpr int gemm_ew() {
  return (MODE == kSbCol || BN >= 224) ? 16 : 8;  // = gemm_epi_warps(MODE == kSbCol, BN), which the host replay uses
}
template <int BN, int MODE, int EW>
constexpr int gemm_ldw() {
  return EW == 16 ? (BN >= 224 && MODE != kSbCol ? 32 : 16) : (MODE != kSbCol ? (BN >= 128 ? 64 : BN / 2) : 32);
}

template <int BN, int STAGES, int MODE, int GROUP = kGroupNone, int A_ROWS = 128, bool STG = false>
static cudaError_t run_gemm(const CUtensorMap& ma, const CUtensorMap& mb, const GemmParams& p, int64_t grid,
                            cudaStream_t st, const GemmGroupParams* gp = nullptr, const CUtensorMap* mc = nullptr) {
  constexpr int EW = gemm_ew<MODE, BN>(), LDW = gemm_ldw<BN, MODE, EW>();
  static_assert(GROUP == kGroupNone || A_ROWS == 128, "the grouped forms load 128-row A boxes");
  using Cfg = GemmCfg<BN, STAGES, EW, A_ROWS>;
  // grouped forms with the staged epilogue: the table for kStageGroups
  // experts, then (1024-aligned) the staging buffers
  constexpr int kStgSmem = (Cfg::kOffMisc + 16 + 2 * (kStageGroups + 1) * 4 + 1023) / 1024 * 1024 + EW * 4096 + 1024;
  constexpr int kSmem = GROUP != kGroupNone ? (STG ? kStgSmem : Cfg::kSmemBytes + Cfg::kGroupTabBytes)
                        : MODE != kSbCol    ? Cfg::kDenseSmemBytes
                                            : Cfg::kSmemBytes;
  static_assert(!STG || (GROUP != kGroupNone && Cfg::kEpiTma && kStgSmem <= 227 * 1024),
                "staged grouped epilogue: shared memory budget");
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    if constexpr (GROUP == kGroupNone)
      attr_err = cudaFuncSetAttribute(gemm_blockwise_kernel<BN, STAGES, MODE, LDW, EW, A_ROWS>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    else
      attr_err = cudaFuncSetAttribute(gemm_grouped_kernel<BN, STAGES, MODE, LDW, EW, GROUP, STG>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  });
  if (attr_err != cudaSuccess) return attr_err;
  if constexpr (GROUP == kGroupNone) {
    static_assert(Cfg::kDenseSmemBytes <= 227 * 1024, "shared memory budget (epilogue staging)");
    CUtensorMap none;  // (no C map: the kernel does not read it)
    if (!mc) memset(&none, 0, sizeof none);
    GemmParams q = p;
    q.pdl = pdl_for_gemm(p.M, p.N, p.K);
    return launch_kernel(q.pdl != 0, gemm_blockwise_kernel<BN, STAGES, MODE, LDW, EW, A_ROWS>, (unsigned)grid,
                         Cfg::kThreads, kSmem, st, ma, mb, mc ? *mc : none, q);
  }
  else {
    CUtensorMap none;  // (no C map: the kernel does not read it)
    if (!mc) memset(&none, 0, sizeof none);
    GemmParams q = p;
    q.pdl = pdl_for_gemm(p.M, p.N, p.K);
    return launch_kernel(q.pdl != 0, gemm_grouped_kernel<BN, STAGES, MODE, LDW, EW, GROUP, STG>, (unsigned)grid,
                         Cfg::kThreads, kSmem, st, ma, mb, mc ? *mc : none, q, *gp);
  }
}

// Parameters of the small-M kernel (Kb = -1 when a size is out of range).
static GemmParams smallm_params(const float* sa, int64_t ldsa, const float* sb, int64_t ldsb, void* c, int64_t ldc,
                                int64_t M, int64_t N, int64_t K, uint64_t wait_limit_ns, int debug_stall) {
  GemmParams p;
  p.sa = sa;
  p.ldsa = ldsa;
  p.sb = sb;
  p.ldsb = ldsb;
  p.c = reinterpret_cast<uint16_t*>(c);
  p.ldc = ldc;
  p.M = M;
  p.N = N;
  p.K = K;
  p.num_m = 1;
  p.num_n = (int)cdiv(N, kBM);
  p.num_tiles = p.num_n;
  const int64_t Kb = cdiv(K, kBK);
  p.Kb = (N >= (int64_t)1 << 31 || K >= (int64_t)1 << 31 || cdiv(N, kBM) * Kb >= (int64_t)1 << 31) ? -1 : (int)Kb;
  p.Nb = (int)cdiv(N, kBlock);
  p.c_vec = 0;
  p.sa_vec = sa && (ldsa % 4 == 0) && ((reinterpret_cast<uintptr_t>(sa) & 15u) == 0);
  p.sb_vec = 0;
  p.wait_limit_ns = wait_limit_ns;
  p.debug_stall = debug_stall;
  return p;
}

// The small-M kernel: T = ceil(N/128) tiles, each split over a cluster of S
// CTAs (S = 8, 4 or 2, at least four K-blocks each, S dividing the rows R),
// S the largest for which the T clusters are resident at once (one wave);
// S = 1 launches no cluster.
template <int MODE, bool XQ, int R>
static int smallm_splits(int tiles, int Kb, int num_sms) {
  using Cfg = SmallCfg<XQ, R>;
  static std::once_flag once;
  static int max_clusters[9] = {};
  std::call_once(once, [] {
    if (cudaFuncSetAttribute(gemm_smallm_kernel<MODE, XQ, R>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Cfg::kSmemBytes) != cudaSuccess)
      return;
    for (int s = 2; s <= 8; s *= 2) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)(s * 16));
      cfg.blockDim = dim3(Cfg::kThreads);
      cfg.dynamicSmemBytes = Cfg::kSmemBytes;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = (unsigned)s;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, gemm_smallm_kernel<MODE, XQ, R>, &cfg) == cudaSuccess)
        max_clusters[s] = n;
    }
    (void)cudaGetLastError();  // a size the device refuses leaves no error behind
  });
  // at least four K-blocks a CTA: below that the hand-over of the partial
  // sums costs more than the K-blocks it spreads (measured)
  for (int s = kSmallMaxSplits; s >= 2; s /= 2)
    if (s <= Kb / 4 && tiles * s <= num_sms && tiles <= max_clusters[s]) return s;
  return 1;
}

template <int MODE, bool XQ, int R>
static cudaError_t run_gemm_smallm(const CUtensorMap& mw, const CUtensorMap& mx, const GemmParams& p, int tiles,
                                   int num_sms, cudaStream_t st) {
  using Cfg = SmallCfg<XQ, R>;
  const int splits = smallm_splits<MODE, XQ, R>(tiles, p.Kb, num_sms);
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(gemm_smallm_kernel<MODE, XQ, R>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    Cfg::kSmemBytes);
  });
  if (attr_err != cudaSuccess) return attr_err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(tiles * splits));
  cfg.blockDim = dim3(Cfg::kThreads);
  cfg.dynamicSmemBytes = Cfg::kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = (unsigned)splits;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = splits > 1 ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, gemm_smallm_kernel<MODE, XQ, R>, mw, mx, p, splits);
}

template <int MODE, bool XQ>
static cudaError_t run_gemm_smallm_rows(int rows, const CUtensorMap& mw, const CUtensorMap& mx, const GemmParams& p,
                                        int tiles, int num_sms, cudaStream_t st) {
  return rows == 16 ? run_gemm_smallm<MODE, XQ, 16>(mw, mx, p, tiles, num_sms, st)
                    : run_gemm_smallm<MODE, XQ, 32>(mw, mx, p, tiles, num_sms, st);
}

cudaError_t launch_gemm(const GemmArgs& a, int num_sms, cudaStream_t st, const char** msg,
                        uint64_t wait_limit_ns, int debug_stall) {
  if (smallm_eligible(a.M, a.N, a.sb_mode == kSbCol, num_sms)) {
    // W (B^T, [N, K]) as the MMA's 128-row A; the rows of A as its 16-row B
    const int rows = smallm_rows(a.M);
    CUtensorMap mw, mx;
    if (!make_tma_u8(&mw, a.qb, a.K, a.N, a.ldb, kBM) || !make_tma_u8(&mx, a.qa, a.K, a.M, a.lda, rows)) {
      *msg = "cuTensorMapEncodeTiled failed for an operand (alignment, stride or size out of range)";
      return cudaErrorInvalidValue;
    }
    GemmParams p = smallm_params(a.sa, a.ldsa, a.sb, a.ldsb, a.c, a.ldc, a.M, a.N, a.K, wait_limit_ns, debug_stall);
    if (p.Kb < 0) {
      *msg = "GEMM too large: M, N, K and the number of (tile, K-block) units must stay below 2^31";
      return cudaErrorInvalidValue;
    }
    const int tiles = (int)cdiv(a.N, kBM);
    return a.sb_mode == kSbTile ? run_gemm_smallm_rows<kSbTile, false>(rows, mw, mx, p, tiles, num_sms, st)
                                : run_gemm_smallm_rows<kSbTileT, false>(rows, mw, mx, p, tiles, num_sms, st);
  }
  const int bn = gemm_pick_bn(a.M, a.N, a.sb_mode == kSbCol, num_sms);
  const int a_rows = gemm_a_rows(a.M, bn);
  CUtensorMap ma, mb;
  if (!make_tma_u8(&ma, a.qa, a.K, a.M, a.lda, a_rows) || !make_tma_u8(&mb, a.qb, a.K, a.N, a.ldb, bn)) {
    *msg = "cuTensorMapEncodeTiled failed for an operand (alignment, stride or size out of range)";
    return cudaErrorInvalidValue;
  }
  GemmParams p;
  p.sa = a.sa;
  p.ldsa = a.ldsa;
  p.sb = a.sb;
  p.ldsb = a.ldsb;
  p.c = reinterpret_cast<uint16_t*>(a.c);
  p.ldc = a.ldc;
  p.M = a.M;
  p.N = a.N;
  p.K = a.K;
  const int64_t num_m = cdiv(a.M, kBM), num_n = cdiv(a.N, bn), Kb = cdiv(a.K, kBK);
  if (a.M >= (int64_t)1 << 31 || a.N >= (int64_t)1 << 31 || a.K >= (int64_t)1 << 31 ||
      num_m * num_n * Kb >= (int64_t)1 << 31) {
    *msg = "GEMM too large: M, N, K and the number of (tile, K-block) units must stay below 2^31";
    return cudaErrorInvalidValue;
  }
  p.num_m = (int)num_m;
  p.num_n = (int)num_n;
  p.num_tiles = (int)(num_m * num_n);
  p.Kb = (int)Kb;
  p.Nb = (int)cdiv(a.N, kBlock);
  p.c_vec = (a.ldc % 8 == 0) && ((reinterpret_cast<uintptr_t>(a.c) & 15u) == 0);
  p.sa_vec = (a.ldsa % 4 == 0) && ((reinterpret_cast<uintptr_t>(a.sa) & 15u) == 0);
  p.sb_vec = (a.ldsb % 4 == 0) && ((reinterpret_cast<uintptr_t>(a.sb) & 15u) == 0);
  p.wait_limit_ns = wait_limit_ns;
  p.debug_stall = debug_stall;
  const int64_t grid = gemm_grid(a.M, a.N, bn, num_sms);
  // 32-column tiles (tile-scale modes): ten stages of 16 + 4 KiB, sixteen
  // tensor-memory buffers
  if (bn == 32)
    return a.sb_mode == kSbTile ? run_gemm<32, 10, kSbTile>(ma, mb, p, grid, st)
                                : run_gemm<32, 10, kSbTileT>(ma, mb, p, grid, st);
  // 64-column tiles (tile-scale modes): sixteen stages of 2 + 8 KiB with
  // 16-row A boxes, else eight of 16 + 8 KiB
  if (bn == 64) {
    const bool t = a.sb_mode == kSbTile;
    if (a_rows == 16)
      return t ? run_gemm<64, 16, kSbTile, kGroupNone, 16>(ma, mb, p, grid, st)
               : run_gemm<64, 16, kSbTileT, kGroupNone, 16>(ma, mb, p, grid, st);
    return t ? run_gemm<64, 8, kSbTile>(ma, mb, p, grid, st) : run_gemm<64, 8, kSbTileT>(ma, mb, p, grid, st);
  }
  // 224-column tiles (the 1x128 x 128x1 GEMM only): three stages of 44 KiB
  if (bn == 224) return run_gemm<224, 3, kSbCol>(ma, mb, p, grid, st);
  // 256-column tiles: three stages of 48 KiB (four measured no faster, and a
  // little slower for the weight gradient).  Their epilogue stores through a
  // tensor map of C (32-row x 64-column boxes) in the tile-scale modes, where
  // the map can clip at exactly N: 16-byte rows of C and N % 8 == 0; else
  // the warps store.
  if (bn == 256) {
    CUtensorMap mc;
    memset(&mc, 0, sizeof mc);
    p.c_tma = a.sb_mode != kSbCol && p.c_vec && a.N % 8 == 0 && make_tma_bf16(&mc, a.c, a.N, a.M, a.ldc * 2, 32);
    switch (a.sb_mode) {
      case kSbTile: return run_gemm<256, 3, kSbTile>(ma, mb, p, grid, st, nullptr, &mc);
      case kSbTileT: return run_gemm<256, 3, kSbTileT>(ma, mb, p, grid, st, nullptr, &mc);
      default: return run_gemm<256, 3, kSbCol>(ma, mb, p, grid, st, nullptr, &mc);
    }
  }
  switch (a.sb_mode) {
    case kSbTile: return run_gemm<128, 6, kSbTile>(ma, mb, p, grid, st);
    case kSbTileT: return run_gemm<128, 6, kSbTileT>(ma, mb, p, grid, st);
    default: return run_gemm<128, 6, kSbCol>(ma, mb, p, grid, st);
  }
}

cudaError_t launch_gemm_grouped(const GemmGroupArgs& ga, int num_sms, cudaStream_t st, const char** msg) {
  const GemmArgs& a = ga.g;
  const bool rows = ga.kind == kGroupRows;
  const int64_t E = ga.E;
  // kGroupRows: A is [M_total, K], B's map is [b_rows, b_inner]; kGroupRed: A is [M, T], B is [N, T]
  const int64_t a_rows = rows ? ga.M_total : a.M, a_inner = rows ? a.K : ga.M_total;
  const int64_t b_rows = rows ? (ga.b_row_step ? E * a.N : a.N) : a.N;
  const int64_t b_inner = rows ? (ga.b_k_step ? E * a.K : a.K) : ga.M_total;
  const int64_t num_n256 = cdiv(a.N, 256);
  const int64_t tiles256 = rows ? (cdiv(ga.M_total, kBM) + E) * num_n256 : E * cdiv(a.M, kBM) * num_n256;
  const int bn = (a.N <= 128 || tiles256 < num_sms) ? 128 : 256;
  // With an empty reduction no tile loads anything; the maps then only need
  // to be well formed.
  const bool empty_k = (rows ? a.K : ga.M_total) == 0;
  CUtensorMap ma, mb;
  if (!make_tma_u8(&ma, a.qa, empty_k ? 16 : a_inner, a_rows, empty_k ? 16 : a.lda, kBM) ||
      !make_tma_u8(&mb, a.qb, empty_k ? 16 : b_inner, b_rows, empty_k ? 16 : a.ldb, bn)) {
    *msg = "cuTensorMapEncodeTiled failed for an operand (alignment, stride or size out of range)";
    return cudaErrorInvalidValue;
  }
  const int64_t num_n = cdiv(a.N, bn);
  const int64_t num_m = rows ? 0 : cdiv(a.M, kBM);
  const int64_t Kb = rows ? cdiv(a.K, kBK) : 0;
  const int64_t tiles_max = rows ? (cdiv(ga.M_total, kBM) + E) * num_n : E * num_m * num_n;
  const int64_t kb_max = rows ? Kb : cdiv(ga.M_total, kBK);
  if (ga.M_total >= (int64_t)1 << 31 || a.M >= (int64_t)1 << 31 || a.N >= (int64_t)1 << 31 ||
      a.K >= (int64_t)1 << 31 || b_rows >= (int64_t)1 << 31 || b_inner >= (int64_t)1 << 31 ||
      tiles_max * kb_max >= (int64_t)1 << 31) {
    *msg = "grouped GEMM too large: sizes and the number of (tile, K-block) units must stay below 2^31";
    return cudaErrorInvalidValue;
  }
  GemmParams p;
  p.sa = a.sa;
  p.ldsa = a.ldsa;
  p.sb = a.sb;
  p.ldsb = a.ldsb;
  p.c = reinterpret_cast<uint16_t*>(a.c);
  p.ldc = a.ldc;
  p.M = rows ? ga.M_total : a.M;
  p.N = a.N;
  p.K = rows ? a.K : ga.M_total;
  p.num_m = (int)num_m;
  p.num_n = (int)num_n;
  p.num_tiles = rows ? 0 : (int)(E * num_m * num_n);
  p.Kb = (int)Kb;
  p.Nb = (int)cdiv(a.N, kBlock);
  p.c_vec = (a.ldc % 8 == 0) && (ga.c_step % 8 == 0) && ((reinterpret_cast<uintptr_t>(a.c) & 15u) == 0);
  p.sa_vec = (a.ldsa % 4 == 0) && ((reinterpret_cast<uintptr_t>(a.sa) & 15u) == 0);
  p.sb_vec = (a.ldsb % 4 == 0) && (ga.sb_step % 4 == 0) && ((reinterpret_cast<uintptr_t>(a.sb) & 15u) == 0);
  p.wait_limit_ns = kWaitLimitNs;
  p.debug_stall = 0;
  GemmGroupParams gp;
  gp.offs = ga.offs;
  gp.E = (int)E;
  gp.M_total = (int)ga.M_total;
  gp.b_row_step = (int)ga.b_row_step;
  gp.b_k_step = (int)ga.b_k_step;
  gp.sb_step = ga.sb_step;
  gp.c_step = ga.c_step;
  const int64_t grid = tiles_max < num_sms ? (tiles_max > 0 ? tiles_max : 1) : num_sms;
  // 256-column tiles of at most kStageGroups experts, with 16-byte rows of C,
  // N % 8 == 0 and (weight gradient) the experts' outputs whole rows apart:
  // the staged TMA-store epilogue, through one map over all experts' rows of C
  // (three stages, to make room for the staging buffers)
  CUtensorMap mc;
  memset(&mc, 0, sizeof mc);
  if (bn == 256 && E <= kStageGroups && p.c_vec && a.N % 8 == 0 &&
      (rows || (ga.c_step % a.ldc == 0 && ga.c_step / a.ldc >= a.M))) {
    const int64_t c_rows_total = rows ? ga.M_total : (E - 1) * (ga.c_step / a.ldc) + a.M;
    gp.c_rows = rows ? 0 : (int)(ga.c_step / a.ldc);
    p.c_tma = c_rows_total > 0 && c_rows_total < ((int64_t)1 << 31) &&
              make_tma_bf16(&mc, a.c, a.N, c_rows_total, a.ldc * 2, 32);
  }
  if (rows) {
    if (bn == 256) {
      if (p.c_tma)
        return a.sb_mode == kSbTile
                   ? run_gemm<256, 3, kSbTile, kGroupRows, 128, true>(ma, mb, p, grid, st, &gp, &mc)
                   : run_gemm<256, 3, kSbTileT, kGroupRows, 128, true>(ma, mb, p, grid, st, &gp, &mc);
      return a.sb_mode == kSbTile ? run_gemm<256, 4, kSbTile, kGroupRows>(ma, mb, p, grid, st, &gp)
                                  : run_gemm<256, 4, kSbTileT, kGroupRows>(ma, mb, p, grid, st, &gp);
    }
    return a.sb_mode == kSbTile ? run_gemm<128, 6, kSbTile, kGroupRows>(ma, mb, p, grid, st, &gp)
                                : run_gemm<128, 6, kSbTileT, kGroupRows>(ma, mb, p, grid, st, &gp);
  }
  if (bn == 256) {
    if (p.c_tma) return run_gemm<256, 3, kSbCol, kGroupRed, 128, true>(ma, mb, p, grid, st, &gp, &mc);
    return run_gemm<256, 3, kSbCol, kGroupRed>(ma, mb, p, grid, st, &gp);
  }
  return run_gemm<128, 6, kSbCol, kGroupRed>(ma, mb, p, grid, st, &gp);
}


// Row-major [rows, inner] bf16 matrix with row stride ld_bytes; 64-column x
// 128-row boxes, 128-byte swizzle, out-of-range reads filled with 0.
static bool make_tma_bf16(CUtensorMap* map, const void* base, int64_t inner, int64_t rows, int64_t ld_bytes,
                          int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld_bytes};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t elem[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, elem,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int RAW_ROWS, int BN>
static cudaError_t run_gemm_xq(const GemmXqArgs& a, int num_sms, cudaStream_t st, const char** msg) {
  constexpr int STAGES = RAW_ROWS == 16 ? (BN == 64 ? 12 : 8) : 4, LDW = 32;
  using Cfg = XqCfg<BN, STAGES, RAW_ROWS>;
  CUtensorMap mx, mb;
  if (!make_tma_bf16(&mx, a.x, a.K, a.M, a.ldx * 2, RAW_ROWS) || !make_tma_u8(&mb, a.qb, a.K, a.N, a.ldb, BN)) {
    *msg = "cuTensorMapEncodeTiled failed for an operand (alignment, stride or size out of range)";
    return cudaErrorInvalidValue;
  }
  const int64_t num_m = cdiv(a.M, kBM), num_n = cdiv(a.N, BN), Kb = cdiv(a.K, kBK);
  if (a.M >= (int64_t)1 << 31 || a.N >= (int64_t)1 << 31 || a.K >= (int64_t)1 << 31 ||
      num_m * num_n * Kb >= (int64_t)1 << 31) {
    *msg = "GEMM too large: M, N, K and the number of (tile, K-block) units must stay below 2^31";
    return cudaErrorInvalidValue;
  }
  GemmParams p;
  p.sa = nullptr;
  p.ldsa = 0;
  p.sb = a.sb;
  p.ldsb = a.ldsb;
  p.c = reinterpret_cast<uint16_t*>(a.c);
  p.ldc = a.ldc;
  p.M = a.M;
  p.N = a.N;
  p.K = a.K;
  p.num_m = (int)num_m;
  p.num_n = (int)num_n;
  p.num_tiles = (int)(num_m * num_n);
  p.Kb = (int)Kb;
  p.Nb = (int)cdiv(a.N, kBlock);
  p.c_vec = (a.ldc % 8 == 0) && ((reinterpret_cast<uintptr_t>(a.c) & 15u) == 0);
  p.sa_vec = 0;
  p.sb_vec = 0;
  p.wait_limit_ns = kWaitLimitNs;
  p.debug_stall = 0;
  const int64_t grid = p.num_tiles < num_sms ? p.num_tiles : num_sms;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(gemm_xq_kernel<BN, STAGES, LDW, RAW_ROWS>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
  });
  if (attr_err != cudaSuccess) return attr_err;
  return launch_pdl(gemm_xq_kernel<BN, STAGES, LDW, RAW_ROWS>, (unsigned)grid, Cfg::kThreads, Cfg::kSmemBytes, st, mx,
                    mb, p);
}

// x tiles of 16 rows (eight in flight) when every row of A fits in them,
// with the dense GEMM's 64-column tiles where 128-column ones would fill at
// most half the SMs; else x tiles of 128 rows and 128-column tiles.
cudaError_t launch_gemm_xq(const GemmXqArgs& a, int num_sms, cudaStream_t st, const char** msg) {
  if (smallm_eligible(a.M, a.N, false, num_sms)) {
    // the small-M kernel with x quantised in it (same splits as the plain GEMM, so the same bits)
    const int rows = smallm_rows(a.M);
    CUtensorMap mw, mx;
    if (!make_tma_u8(&mw, a.qb, a.K, a.N, a.ldb, kBM) || !make_tma_bf16(&mx, a.x, a.K, a.M, a.ldx * 2, rows)) {
      *msg = "cuTensorMapEncodeTiled failed for an operand (alignment, stride or size out of range)";
      return cudaErrorInvalidValue;
    }
    GemmParams p = smallm_params(nullptr, 0, a.sb, a.ldsb, a.c, a.ldc, a.M, a.N, a.K, kWaitLimitNs, 0);
    if (p.Kb < 0) {
      *msg = "GEMM too large: M, N, K and the number of (tile, K-block) units must stay below 2^31";
      return cudaErrorInvalidValue;
    }
    return run_gemm_smallm_rows<kSbTile, true>(rows, mw, mx, p, (int)cdiv(a.N, kBM), num_sms, st);
  }
  if (a.M <= 16)
    return gemm_pick_bn(a.M, a.N, false, num_sms) <= 64 ? run_gemm_xq<16, 64>(a, num_sms, st, msg)
                                                         : run_gemm_xq<16, 128>(a, num_sms, st, msg);
  return run_gemm_xq<128, 128>(a, num_sms, st, msg);
}

cudaError_t launch_gemm_wgrad_xq(const GemmWxqArgs& a, int num_sms, cudaStream_t st, const char** msg) {
  using Cfg = WxqCfg;
  CUtensorMap ma, mx;
  // X [K tokens, N features]: boxes of 64 features x 128 tokens
  if (!make_tma_u8(&ma, a.qa, a.K, a.M, a.lda, kBM) || !make_tma_bf16(&mx, a.x, a.N, a.K, a.ldx * 2, kBK)) {
    *msg = "cuTensorMapEncodeTiled failed for an operand (alignment, stride or size out of range)";
    return cudaErrorInvalidValue;
  }
  const int64_t num_m = cdiv(a.M, kBM), num_n = cdiv(a.N, Cfg::BN), Kb = cdiv(a.K, kBK);
  if (a.M >= (int64_t)1 << 31 || a.N >= (int64_t)1 << 31 || a.K >= (int64_t)1 << 31 ||
      num_m * num_n * Kb >= (int64_t)1 << 31) {
    *msg = "GEMM too large: M, N, K and the number of (tile, K-block) units must stay below 2^31";
    return cudaErrorInvalidValue;
  }
  GemmParams p;
  p.sa = a.sa;
  p.ldsa = a.ldsa;
  p.sb = nullptr;
  p.ldsb = 0;
  p.c = reinterpret_cast<uint16_t*>(a.c);
  p.ldc = a.ldc;
  p.M = a.M;
  p.N = a.N;
  p.K = a.K;
  p.num_m = (int)num_m;
  p.num_n = (int)num_n;
  p.num_tiles = (int)(num_m * num_n);
  p.Kb = (int)Kb;
  p.Nb = (int)cdiv(a.N, kBlock);
  p.c_vec = (a.ldc % 8 == 0) && ((reinterpret_cast<uintptr_t>(a.c) & 15u) == 0);
  p.sa_vec = (a.ldsa % 4 == 0) && ((reinterpret_cast<uintptr_t>(a.sa) & 15u) == 0);
  p.sb_vec = 0;
  p.wait_limit_ns = kWaitLimitNs;
  p.debug_stall = 0;
  const int64_t grid = p.num_tiles < num_sms ? p.num_tiles : num_sms;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(gemm_wgrad_xq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    Cfg::kSmemBytes);
  });
  if (attr_err != cudaSuccess) return attr_err;
  return launch_pdl(gemm_wgrad_xq_kernel, (unsigned)grid, Cfg::kThreads, Cfg::kSmemBytes, st, ma, mx, p);
}

cudaError_t gemm_read_errors(uint32_t* out) {
  uint32_t zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_gemm_error, sizeof(uint32_t));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_gemm_error, &zero, sizeof(uint32_t));
}

}  // namespace bfp8
