// Shared device helpers: e4m3 rounding, bf16 unpacking, mbarrier / TMA /
// tcgen05 wrappers (inline PTX for sm_103a), bounded waits.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "index.cuh"

namespace bfp8 {

// ---------------------------------------------------------------------------
// Numerics of the method
// ---------------------------------------------------------------------------

// s = max(amax, 1e-12) / 448 — one IEEE division (the scale formula of the
// blockwise FP8 method; the floor keeps an all-zero group finite).
__device__ __forceinline__ float group_scale(float amax) {
  return __fdiv_rn(fmaxf(amax, kAmaxFloor), kE4m3Max);
}

// 1/s rounded to nearest even (once per group).
__device__ __forceinline__ float recip_rn(float s) { return __frcp_rn(s); }

// x / s rounded to nearest even, from y = RN(1/s), by Markstein's correction
// (P. Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Dev. 34(1), 1990): q0 = RN(x*y);
// r = x - s*q (exact with an FMA); q' = RN(q + r*y).  One correction makes q
// faithful, and from a faithful q the next correction returns RN(x/s) when no
// intermediate underflows.  Here s >= 1e-12/448 and |x| <= 448 s, so the
// remainders are normal whenever |x/s| >= 2^-11; smaller quotients can differ
// from the IEEE quotient by a few ulps but round to the same e4m3 code.  The
// corrections can turn a zero quotient's sign positive (-0 + +0 = +0), while
// x/s for s > 0 always has the sign of x, so the sign of x is copied back.
__device__ __forceinline__ float quotient(float x, float s, float y) {
  const float q0 = __fmul_rn(x, y);
  const float r0 = __fmaf_rn(-s, q0, x);
  const float q1 = __fmaf_rn(r0, y, q0);
  const float r1 = __fmaf_rn(-s, q1, x);
  return copysignf(__fmaf_rn(r1, y, q1), x);
}

// Two fp32 values -> two e4m3fn bytes, RNE, saturating to +-448 (the clamp of
// the method).  Result byte 0 = lo, byte 1 = hi.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two fp32 -> packed bf16x2 (RNE); lo in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Read-only 16-byte load that does not allocate in L1.
__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-suspending probe of a barrier phase (for latency-critical spins).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded spin on test_wait: same contract as mbar_wait_bounded, but the
// thread never suspends, so it sees the phase flip a few cycles after it.
__device__ __forceinline__ bool mbar_spin_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                                  const volatile int* abort) {
  if (mbar_test_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 256; ++i)
      if (mbar_test_wait(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// Bounded wait for the phase with parity `parity` of the barrier at `bar`.
// Gives up (returns false) after `limit_ns` of global time, or as soon as
// *abort becomes non-zero (another role of the CTA gave up first).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                                  const volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// ---------------------------------------------------------------------------
// Thread-block clusters: distributed shared memory and the cluster barrier
// ---------------------------------------------------------------------------

// The address in CTA `rank`'s shared memory of the variable at `addr` in this
// CTA's (a shared::cluster address).
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// 8 bytes from a shared::cluster address (another CTA's shared memory).
__device__ __forceinline__ float2 lds64_cluster(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
  return v;
}

// 16 bytes from a shared::cluster address (another CTA's shared memory).
__device__ __forceinline__ float4 lds128_cluster(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// Every thread of every CTA of the cluster: arrive (release) and wait
// (acquire) on the cluster barrier, all at one program point (aligned).  Used
// where every thread reaches it unconditionally; the CTAs of a cluster are
// resident together, so it completes.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Flags between CTAs of one launch (global memory, GPU scope)
// ---------------------------------------------------------------------------

__device__ __forceinline__ void st_release_gpu(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void st_relaxed_gpu(uint32_t* p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Bounded spin until *flag == 1 (written by another CTA of the same launch).
__device__ __forceinline__ bool spin_flag_bounded(const uint32_t* flag, uint64_t limit_ns,
                                                  const volatile int* abort) {
  if (ld_acquire_gpu(flag) == 1u) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (ld_acquire_gpu(flag) == 1u) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// ---------------------------------------------------------------------------
// TMA
// ---------------------------------------------------------------------------

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// 2-D tiled bulk tensor copy global -> shared, completion counted in bytes on `bar`.
// x = innermost coordinate (bytes for a uint8 map; multiple of 16), y = row.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// 2-D tiled bulk tensor copy shared -> global (bulk-group completion).
// Elements outside the tensor's bounds are not written.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(map), "r"(src),
               "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// wait until every committed bulk store of this thread has finished reading shared memory
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// wait until every committed bulk store of this thread is complete
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Asynchronous global -> shared copies (cp.async); bytes past src_bytes are
// zero-filled (src_bytes = 0 reads nothing).  16-byte form: both addresses 16-byte aligned.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
// Programmatic dependent launch.  A kernel of this library launched with it
// (launch_pdl, or launch_kernel with pdl set) may start (set up shared
// memory, barriers, tensor memory) while the kernel before it in the stream
// is still finishing; every kernel calls pdl_wait() before its first
// global-memory access, read or write, which returns once the previous grid
// has completed with its writes visible (at once when the kernel was launched
// without it).  pdl_launch_dependents() lets the next kernel start early; it
// is issued at kernel entry (the next kernel is only scheduled once every CTA
// of this grid has issued it, so it never takes a slot this grid still needs).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... P, typename... A>
inline cudaError_t launch_kernel(bool pdl, void (*kernel)(P...), unsigned grid, unsigned block, size_t smem,
                                 cudaStream_t st, A&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<A&&>(args)...);
}
template <typename... P, typename... A>
inline cudaError_t launch_pdl(void (*kernel)(P...), unsigned grid, unsigned block, size_t smem, cudaStream_t st,
                              A&&... args) {
  return launch_kernel(true, kernel, grid, block, smem, st, static_cast<A&&>(args)...);
}

// arrive on `bar` once every earlier cp.async of this thread has landed (the
// arrival is counted in the barrier's expected count: .noinc)
__device__ __forceinline__ void cp_async_mbar_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
// order this thread's generic-proxy shared-memory writes before later async-proxy reads
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// tcgen05 (5th-generation tensor cores, accumulators in tensor memory)
// ---------------------------------------------------------------------------

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile written by TMA
// with 128-byte swizzling: rows of 128 bytes, 8-row swizzle atoms of 1024
// bytes (stride-dimension offset), tile base 1024-byte aligned.
__device__ __forceinline__ uint64_t desc_kmajor_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);   // start address (16-byte units)
  d |= (uint64_t)(16u >> 4) << 16;            // leading-dimension offset (unused here)
  d |= (uint64_t)(1024u >> 4) << 32;          // stride-dimension offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;                     // descriptor version of tcgen05
  d |= (uint64_t)2 << 61;                     // 128-byte swizzle
  return d;
}

// Instruction descriptor: D fp32, A and B e4m3, both K-major, shape M x N.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int m, int n) {
  return (1u << 4)                          // D format: f32
         | (0u << 7) | (0u << 10)           // A, B format: e4m3
         | (0u << 15) | (0u << 16)          // A, B K-major
         | ((uint32_t)(n >> 3) << 17)       // N / 8
         | ((uint32_t)(m >> 4) << 24);      // M / 16
}

// D[tmem] (+)= A[smem] * B[smem]^T, one instruction of K = 32 e4m3 elements.
__device__ __forceinline__ void mma_e4m3(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive (once) on `bar` when all previously issued tcgen05 ops of this thread complete.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns of tensor memory -> 32 registers per thread.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
// 32 lanes x 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_32x32b_x8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 32 lanes x 64 consecutive columns in one instruction.  One instruction per
// batch keeps the whole batch in flight; several narrower loads before one
// wait may be issued one after another.
__device__ __forceinline__ void tmem_ld_32x32b_x64(uint32_t taddr, uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
        "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
        "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr));
}

// Registers filled by tcgen05.ld are only valid after tcgen05.wait::ld; this
// ties every later use of r to a point after the wait (no instructions).
template <int N>
__device__ __forceinline__ void tmem_regs_after_wait(uint32_t (&r)[N]) {
#pragma unroll
  for (int j = 0; j < N; ++j) asm volatile("" : "+r"(r[j]));
}

// Packed fp32x2 arithmetic (one instruction for two lanes of work).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
// copysign on both lanes: magnitude of q, sign of x
__device__ __forceinline__ uint64_t f2_copysign(uint64_t q, uint64_t x) {
  return (q & 0x7FFFFFFF7FFFFFFFull) | (x & 0x8000000080000000ull);
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// ---------------------------------------------------------------------------
// Blockwise quantisation arithmetic shared by the quantisation kernels and the
// GEMM that quantises its A operand itself (identical bytes by construction)
// ---------------------------------------------------------------------------

// Packed bf16 pair: per half, a value whose magnitude is max(|a|, |b|) (its
// sign bit is meaningless and is masked off where the maximum is used).
__device__ __forceinline__ uint32_t amax2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// s = RN(max(amax, 1e-12) / 448).  448 = 7 * 2^6 and a/448 stays a normal
// float for a >= 1e-12, so s = RN(a/7) * 2^-6 exactly.  RN(a/7) comes from
// y7 = RN(1/7) with one correction step of Markstein's method (P. Markstein,
// IBM J. Res. Dev. 34(1), 1990): q0 = RN(a*y7), r = a - 7*q0 (exact), RN(q0 + r*y7).
// For every bf16 amax this equals the IEEE quotient (checked exhaustively on
// the CPU; the GPU tests compare every scale bit for bit with the oracle).
__device__ __forceinline__ float scale_of(float amax) {
  constexpr float kRcp7 = 1.0f / 7.0f;
  const float a = fmaxf(amax, kAmaxFloor);
  const float q0 = __fmul_rn(a, kRcp7);
  const float r = __fmaf_rn(-7.0f, q0, a);
  return __fmul_rn(__fmaf_rn(r, kRcp7, q0), 0.015625f);
}

// -1/s to within one ulp (rcp.approx: at most 1 ulp of error over the whole
// range; s is normal, so flushing subnormals changes nothing).
__device__ __forceinline__ float neg_rcp(float s) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(-s));
  return y;
}

// The e4m3 codes of -(x/s) for the two bf16 values of `w`, given s2 = (s, s')
// and ny2 = (-1/s, -1/s') to within an ulp:
//   q0 = x*(-y), r = x - s*(x*y) (exact), q1 = q0 + r*(-y) = -RN(x/s).
// With bf16 x, |x| <= 448 s and any such y this one-step quotient rounds to
// the same e4m3 code as the IEEE quotient, including the sign of zero
// (checked exhaustively on the CPU over every pair of bf16 (amax, x)).  The
// caller flips the sign bits of the codes (XOR 0x80).
__device__ __forceinline__ uint32_t neg_codes2(uint32_t w, uint64_t s2, uint64_t ny2) {
  const uint64_t x2 = f2_pack(bf16_lo(w), bf16_hi(w));
  const uint64_t q0 = f2_mul(x2, ny2);
  const uint64_t r = f2_fma(s2, q0, x2);
  const uint64_t q1 = f2_fma(r, ny2, q0);
  return cvt_e4m3x2(__uint_as_float((uint32_t)q1), __uint_as_float((uint32_t)(q1 >> 32)));
}


}  // namespace bfp8
