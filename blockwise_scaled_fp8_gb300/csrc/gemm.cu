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
//   warp 1      MMA issuer: 4 x tcgen05.mma.kind::f8f6f4 (K = 32 each) per
//               K-block into one of two tensor-memory partial buffers, then
//               tcgen05.commit to release the smem stage and publish the partial.
//   warps 2-3   idle (they complete the control warpgroup, which gives its
//               registers to the promotion warpgroups with setmaxnreg).
//   warps 4..19 promotion/epilogue, four per tensor-memory lane quarter, each
//               owning 32 rows x BN/4 columns of the tile: tcgen05.ld the
//               K-block's fp32 partial, release the tensor-memory buffer,
//               acc += (a_s*b_s) * partial in registers; at tile end round to
//               bf16 and store only rows m < M and columns n < N.
// The two tensor-memory buffers let the promotion of K-block kb overlap the
// MMAs of K-block kb+1.  A warp moves only about 30 bytes per cycle out of
// tensor memory, so sixteen warps are needed to read a 128 x 256 fp32 partial
// (128 KiB) in less time than the MMAs of the next K-block take (512 cycles).  Tails: TMA zero-fills rows/columns outside M, N, K;
// scale loads are predicated; the epilogue store is masked.
// Every mbarrier wait is bounded in time; a timeout records an error bit,
// lets every role leave its loop, waits for its own copies/MMAs in flight and
// frees tensor memory before the CTA exits.
#include <cudaTypedefs.h>

#include <string.h>

#include <mutex>

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
  int c_tma;   // C written by TMA stores through shared memory (same conditions)
  int sb_vec;  // 16-byte column-scale loads allowed (ldsb % 4 == 0, sb 16-byte aligned)
  uint64_t wait_limit_ns;
  int debug_stall;  // test hook: the promotion warps wait on a barrier nothing arrives on
};

template <int BN, int STAGES>
struct GemmCfg {
  static constexpr int kEpiWarps = kGemmEpiWarps;  // 16: four per tensor-memory lane quarter
  static constexpr int kCols = BN / 4;             // tile columns per promotion warp
  static constexpr int kThreads = 128 + 32 * kEpiWarps;
  // Register split: 640 threads launched at 96 registers each (61440); the
  // control warpgroup drops to 32 and the four promotion warpgroups rise to
  // 112: 128*32 + 512*112 = 61440.
  static constexpr int kCtrlRegs = 32;
  static constexpr int kEpiRegs = 112;
  static constexpr int kABytes = kBM * kBK;
  static constexpr int kBBytes = BN * kBK;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kTmemCols = 2 * BN;  // two fp32 partial buffers of BN columns
  static constexpr int kOffB = STAGES * kABytes;
  // per promotion warp: a 2 KiB buffer (32 rows x 32 bf16 columns, 64-byte
  // swizzled) that stages C for the TMA store at tile end, and holds the
  // K-block's column scales (128x1 mode) during the K loop
  static constexpr int kStageC = 32 * 32 * 2;
  static constexpr int kOffSb = kOffB + STAGES * kBBytes;
  static constexpr int kOffBar = kOffSb + kEpiWarps * kStageC;
  static constexpr int kNumBars = 2 * STAGES + 6;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + slack for 1024-byte alignment
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
  static_assert(kTmemCols >= 32 && kTmemCols <= 512 && (kTmemCols & (kTmemCols - 1)) == 0,
                "tensor-memory allocation must be a power of two in [32, 512]");
};

__device__ __forceinline__ void gemm_fail(uint32_t code, volatile int* abort_flag) {
  atomicOr(&g_gemm_error, code);
  *abort_flag = 1;
}

template <int BN, int STAGES, int SB_MODE, int LDW>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_blockwise_kernel(const __grid_constant__ CUtensorMap tma_a,
                          const __grid_constant__ CUtensorMap tma_b,
                          const __grid_constant__ CUtensorMap tma_c, const GemmParams p) {
  using Cfg = GemmCfg<BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sA = sbase;
  const uint32_t sB = sbase + Cfg::kOffB;
  uint8_t* cstage = smem + Cfg::kOffSb;
  const uint32_t bar0 = sbase + Cfg::kOffBar;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + Cfg::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::kOffMisc + 4);
  volatile int* never = reinterpret_cast<volatile int*>(smem + Cfg::kOffMisc + 8);

  // barrier addresses: full[S], empty[S], tfull[2], tempty[2], drain, stall
  auto full_bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  auto empty_bar = [&](int i) { return bar0 + 8u * (uint32_t)(STAGES + i); };
  auto tfull_bar = [&](int i) { return bar0 + 8u * (uint32_t)(2 * STAGES + i); };
  auto tempty_bar = [&](int i) { return bar0 + 8u * (uint32_t)(2 * STAGES + 2 + i); };
  const uint32_t drain_bar = bar0 + 8u * (uint32_t)(2 * STAGES + 4);
  const uint32_t stall_bar = bar0 + 8u * (uint32_t)(2 * STAGES + 5);  // never arrived on

  const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);
  const int lane = (int)(threadIdx.x & 31);

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(full_bar(i), 1);
      mbar_init(empty_bar(i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(tfull_bar(i), 1);
      mbar_init(tempty_bar(i), Cfg::kEpiWarps);
    }
    mbar_init(drain_bar, 1);
    mbar_init(stall_bar, 1);
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
    tma_prefetch_desc(&tma_b);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
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
          tma_load_2d(sA + (uint32_t)(st * Cfg::kABytes), &tma_a, full_bar(st), kb * kBK, g.m0);
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
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_e4m3_f32(kBM, BN);
      uint32_t it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
        for (int kb = 0; kb < p.Kb; ++kb, ++it) {
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
      // every MMA issued above completes before tensor memory is released
      mma_commit(drain_bar);
      if (!mbar_wait_bounded(drain_bar, 0, p.wait_limit_ns, never))
        gemm_fail(kErrWaitDrain, abort_flag);
    }
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(Cfg::kEpiRegs));
    // ------------------------------------------------------------ promotion + epilogue
    const int e = warp - 4;
    constexpr int kCols = Cfg::kCols;
    const int row = epi_row(e, lane);
    const int col0 = epi_col0(e, BN);
    const uint32_t lane_base = (uint32_t)(32 * (warp % 4)) << 16;
    uint8_t* cbuf = cstage + e * Cfg::kStageC;
    const uint32_t cbuf_s = smem_u32(cbuf);
    float* slot = reinterpret_cast<float*>(cbuf);
    uint32_t it = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
      const GemmTile g = gemm_tile(tile, p.num_m, p.num_n, BN);
      const int m = g.m0 + row;
      const bool m_ok = m < p.M;
      const int nb = (g.n0 + col0) / kBlock;  // B tile-scale block of this warp's columns
      const int ncol = g.n0 + col0 + 4 * lane;  // first of this lane's 4 column scales

      auto load_sa = [&](int kb) -> float { return m_ok ? __ldg(p.sa + (int64_t)kb * p.ldsa + m) : 0.0f; };
      auto load_sb_tile = [&](int kb) -> float {
        if (nb >= p.Nb) return 0.0f;
        return SB_MODE == kSbTile ? __ldg(p.sb + (int64_t)nb * p.ldsb + kb) : __ldg(p.sb + (int64_t)kb * p.ldsb + nb);
      };
      auto load_sb_col = [&](int kb) -> float4 {
        if (lane >= kCols / 4) return make_float4(0.f, 0.f, 0.f, 0.f);  // lanes beyond this warp's columns
        const float* src = p.sb + (int64_t)kb * p.ldsb + ncol;
        if (p.sb_vec && ncol + 4 <= p.N) return __ldg(reinterpret_cast<const float4*>(src));
        float4 r;
        r.x = (ncol + 0 < p.N) ? __ldg(src + 0) : 0.0f;
        r.y = (ncol + 1 < p.N) ? __ldg(src + 1) : 0.0f;
        r.z = (ncol + 2 < p.N) ? __ldg(src + 2) : 0.0f;
        r.w = (ncol + 3 < p.N) ? __ldg(src + 3) : 0.0f;
        return r;
      };

      float acc[kCols];
#pragma unroll
      for (int j = 0; j < kCols; ++j) acc[j] = 0.0f;
      if (SB_MODE == kSbCol && p.c_tma) {  // the staging buffer doubles as the scale slot
        if (lane == 0) bulk_wait_read_all();
        __syncwarp();
      }

      float sa_next = load_sa(0);
      float sb_next = 0.0f;
      float4 sbc_next = make_float4(0.f, 0.f, 0.f, 0.f);
      if (SB_MODE == kSbCol) sbc_next = load_sb_col(0);
      else sb_next = load_sb_tile(0);

      for (int kb = 0; kb < p.Kb; ++kb, ++it) {
        const float sa_cur = sa_next, sb_cur = sb_next;
        const float4 sbc_cur = sbc_next;
        if (kb + 1 < p.Kb) {  // prefetch the next K-block's scales (masked loads)
          sa_next = load_sa(kb + 1);
          if (SB_MODE == kSbCol) sbc_next = load_sb_col(kb + 1);
          else sb_next = load_sb_tile(kb + 1);
        }
        const int buf = (int)(it & 1u);
        const uint32_t tph = (it >> 1) & 1u;
        const bool got = mbar_wait_bounded(p.debug_stall ? stall_bar : tfull_bar(buf), tph, p.wait_limit_ns,
                                           abort_flag);
        if (!__all_sync(0xffffffffu, got)) {
          if (lane == 0) gemm_fail(kErrWaitTmemFull, abort_flag);
          ok = false;
          break;
        }
        tc_fence_after();
        if (SB_MODE == kSbCol) {
          __syncwarp();
          if (lane < kCols / 4) reinterpret_cast<float4*>(slot)[lane] = sbc_cur;
          __syncwarp();
        }
        const uint32_t taddr = tmem_base + lane_base + (uint32_t)(buf * BN + col0);
        const float scale = sa_cur * sb_cur;
        // LDW columns of the partial per tensor-memory load round trip (one wait)
#pragma unroll
        for (int c = 0; c < kCols / LDW; ++c) {
          uint32_t r[LDW];
          if constexpr (LDW == 32)
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
              const float4 sb4 = reinterpret_cast<const float4*>(slot)[LDW / 4 * c + j4];
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
            for (int j = 0; j < LDW; ++j) acc[LDW * c + j] = fmaf(scale, __uint_as_float(r[j]), acc[LDW * c + j]);
          }
        }
      }
      if (!ok) break;

      if (p.c_tma) {
        // 32x32 bf16 slices through the staging buffer (64-byte swizzle: the
        // 16-byte chunk k of row r sits at chunk k ^ ((r >> 1) & 3)), each
        // written by one TMA store (rows/columns outside [M, N] are dropped)
#pragma unroll
        for (int h = 0; h < kCols / 32; ++h) {
          if (lane == 0) bulk_wait_read_all();  // previous store has read the buffer
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t w[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
              w[q] = pack_bf16x2(acc[32 * h + 8 * j + 2 * q], acc[32 * h + 8 * j + 2 * q + 1]);
            const uint32_t addr = cbuf_s + (uint32_t)(lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4));
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[0]), "r"(w[1]), "r"(w[2]),
                         "r"(w[3])
                         : "memory");
          }
          fence_proxy_async_shared();
          __syncwarp();
          const int xs = g.n0 + col0 + 32 * h, ys = g.m0 + 32 * (warp % 4);
          if (lane == 0 && xs < p.N && ys < p.M) {  // a slice wholly outside C is not issued
            tma_store_2d(&tma_c, cbuf_s, xs, ys);
            bulk_commit();
          }
        }
      } else if (m_ok) {
        uint16_t* crow = p.c + (int64_t)m * p.ldc;
#pragma unroll
        for (int c8 = 0; c8 < kCols / 8; ++c8) {
          const int n = g.n0 + col0 + 8 * c8;
          if (n >= p.N) break;
          uint32_t w[4];
#pragma unroll
          for (int h = 0; h < 4; ++h) w[h] = pack_bf16x2(acc[8 * c8 + 2 * h], acc[8 * c8 + 2 * h + 1]);
          if (p.c_vec && n + 8 <= p.N) {
            *reinterpret_cast<uint4*>(crow + n) = make_uint4(w[0], w[1], w[2], w[3]);
          } else {
#pragma unroll
            for (int b = 0; b < 8; ++b)
              if (n + b < p.N) crow[n + b] = (uint16_t)(w[b >> 1] >> (16 * (b & 1)));
          }
        }
      }
    }
    if (p.c_tma && lane == 0) bulk_wait_all();  // stores complete before the CTA exits
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

// Row-major [rows, cols] bf16 output with row stride ld elements; box of
// 32 columns x 32 rows (one promotion warp's slice), 64-byte swizzle.
static bool make_tma_bf16_store(CUtensorMap* map, void* base, int64_t cols, int64_t rows, int64_t ld) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t elem[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int gemm_pick_bn(int64_t M, int64_t N, int num_sms) {
  if (N <= 128) return 128;
  const int64_t tiles256 = cdiv(M, kBM) * cdiv(N, 256);
  return tiles256 >= num_sms ? 256 : 128;
}

int64_t gemm_grid(int64_t M, int64_t N, int bn, int num_sms) {
  const int64_t tiles = cdiv(M, kBM) * cdiv(N, bn);
  return tiles < num_sms ? tiles : num_sms;
}

template <int BN, int STAGES, int MODE, int LDW = 16>
static cudaError_t run_gemm(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mc,
                            const GemmParams& p, int64_t grid, cudaStream_t st) {
  using Cfg = GemmCfg<BN, STAGES>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(gemm_blockwise_kernel<BN, STAGES, MODE, LDW>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
  });
  if (attr_err != cudaSuccess) return attr_err;
  gemm_blockwise_kernel<BN, STAGES, MODE, LDW><<<(unsigned)grid, Cfg::kThreads, Cfg::kSmemBytes, st>>>(ma, mb, mc, p);
  return cudaGetLastError();
}

cudaError_t launch_gemm(const GemmArgs& a, int num_sms, cudaStream_t st, const char** msg,
                        uint64_t wait_limit_ns, int debug_stall) {
  const int bn = gemm_pick_bn(a.M, a.N, num_sms);
  CUtensorMap ma, mb;
  if (!make_tma_u8(&ma, a.qa, a.K, a.M, a.lda, kBM) || !make_tma_u8(&mb, a.qb, a.K, a.N, a.ldb, bn)) {
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
  p.sb_vec = (a.ldsb % 4 == 0) && ((reinterpret_cast<uintptr_t>(a.sb) & 15u) == 0);
  CUtensorMap mc;
  // a TMA store clips the inner dimension in 16-byte units: only rows of whole
  // 16-byte units (N % 8 == 0) keep the padding past N untouched
  p.c_tma = p.c_vec && a.N % 8 == 0 && make_tma_bf16_store(&mc, a.c, a.N, a.M, a.ldc);
  if (!p.c_tma) memset(&mc, 0, sizeof(mc));
  p.wait_limit_ns = wait_limit_ns;
  p.debug_stall = debug_stall;
  const int64_t grid = gemm_grid(a.M, a.N, bn, num_sms);
  if (bn == 256) {
    switch (a.sb_mode) {
      case kSbTile: return run_gemm<256, 4, kSbTile, 32>(ma, mb, mc, p, grid, st);
      case kSbTileT: return run_gemm<256, 4, kSbTileT, 32>(ma, mb, mc, p, grid, st);
      default: return run_gemm<256, 4, kSbCol, 16>(ma, mb, mc, p, grid, st);
    }
  }
  switch (a.sb_mode) {
    case kSbTile: return run_gemm<128, 6, kSbTile>(ma, mb, mc, p, grid, st);
    case kSbTileT: return run_gemm<128, 6, kSbTileT>(ma, mb, mc, p, grid, st);
    default: return run_gemm<128, 6, kSbCol>(ma, mb, mc, p, grid, st);
  }
}

cudaError_t gemm_read_errors(uint32_t* out) {
  uint32_t zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_gemm_error, sizeof(uint32_t));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_gemm_error, &zero, sizeof(uint32_t));
}

}  // namespace bfp8
