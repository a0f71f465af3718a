/*
 * bfp8 — blockwise-scaled FP8 (e4m3) quantisation and GEMMs for GB300 (sm_103a).
 *
 * C ABI of the library libbfp8.so.  Every entry point is asynchronous on the
 * given CUDA stream, allocates nothing, and never synchronises (except
 * bfp8_check_device_errors).  The caller owns every buffer.  Pointers named
 * "device" must be device memory (or managed memory) of the current device.
 *
 * The method (pytorch/ao pull-request pages "Enable blockwise FP8 dense
 * training kernels on ROCm" and "Mask a_s/b_s scale loads in blockwise FP8
 * training GEMM kernels"):
 *   - a group of bf16 values (1x128 along the reduction dim, 128x1 along the
 *     reduction dim, or a 128x128 weight tile) has amax = max |x| over its
 *     in-range elements; s = max(amax, 1e-12) / 448 (fp32, one IEEE division);
 *     q = RNE_e4m3fn(clamp(x / s, -448, 448)) with x / s one IEEE division.
 *   - GEMM: C[m,n] = sum over 128-wide K-blocks kb of
 *     a_s[m,kb] * b_s(n,kb) * (sum_{k in kb} qA[m,k] * qB[k,n]), partial
 *     products in fp32 from the tensor cores, promoted per K-block into an
 *     fp32 running sum, stored as bf16 (round to nearest even) only where
 *     m < M and n < N; scale loads are masked the same way.
 *
 * Layout conventions.  Row-major everywhere; "ld" arguments are row strides
 * in ELEMENTS of the buffer's type.  e4m3 buffers are bytes.  Kb = ceil(K/128)
 * for the dimension that is grouped.  Bytes between the logical width and the
 * row stride (padding) are never read as data and never written.
 *
 * Errors.  Each call validates its arguments and returns BFP8_ERR_INVALID_ARG
 * (nothing launched) on a violation; BFP8_ERR_UNSUPPORTED when the current
 * device is not sm_103; BFP8_ERR_CUDA when a launch fails.  bfp8_last_error()
 * returns a message for the calling thread's last failed call.  A zero-sized
 * problem launches nothing and returns BFP8_OK (a GEMM with K == 0 and a
 * linear layer with an empty reduction write zeros into their outputs).
 * Inputs must be finite; results for Inf/NaN inputs are unspecified.
 */
#ifndef BFP8_H_
#define BFP8_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define BFP8_API __attribute__((visibility("default")))
#else
#define BFP8_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque CUDA stream (binary-compatible with cudaStream_t); NULL = legacy default stream. */
typedef struct CUstream_st *bfp8_stream_t;

typedef enum {
    BFP8_OK = 0,
    BFP8_ERR_INVALID_ARG = 1,
    BFP8_ERR_UNSUPPORTED = 2,
    BFP8_ERR_CUDA = 3,
    BFP8_ERR_TIMEOUT = 4
} bfp8_status;

/* Message describing the calling thread's most recent non-OK status. */
BFP8_API const char *bfp8_last_error(void);

/*
 * act_quant_lhs: 1x128 groups along K of A[M,K].
 * Source: "Enable blockwise FP8 dense training kernels on ROCm" — quantization
 * kernel correctness table (act_quant_lhs, block_size=128) and the root-cause
 * comment: the lhs kernel writes its scales into a column-major fp32 tensor and
 * the store must be masked to rows m < M.
 *   x            device bf16.  x_transposed == 0: A[m,k] = x[m*ldx + k]
 *                (x is [M,K], ldx >= K).  x_transposed == 1: A[m,k] =
 *                x[k*ldx + m] (x is [K,M], ldx >= M) — used to quantise dY^T
 *                along the token dimension for the weight-gradient GEMM.
 *   q            device e4m3 [M, ldq], ldq >= K, ldq % 16 == 0, 16-byte aligned.
 *   s            device fp32 column-major [M, Kb]: s[kb*lds + m], lds >= M.
 * Writes exactly q[m*ldq + k] (m < M, k < K) and s[kb*lds + m] (m < M, kb < Kb).
 */
BFP8_API bfp8_status bfp8_quant_lhs(const void *x, int64_t M, int64_t K, int64_t ldx, int x_transposed,
                           void *q, int64_t ldq, float *s, int64_t lds, bfp8_stream_t stream);

/*
 * act_quant_rhs: 128x1 groups along the reduction dimension K of X[K,N]
 * (one group = one column n and 128 consecutive rows k).
 * Source: "Enable blockwise FP8 dense training kernels on ROCm" — quantization
 * kernel correctness table (act_quant_rhs, block_size=128).
 *   x            device bf16 [K,N], ldx >= N.
 *   qT           device e4m3 [N, ldq] (the bytes written transposed, K
 *                contiguous, as the GEMM reads them), ldq >= K, ldq % 16 == 0,
 *                16-byte aligned.
 *   s            device fp32 row-major [Kb, N]: s[kb*lds + n], lds >= N.
 * Writes exactly qT[n*ldq + k] (n < N, k < K) and s[kb*lds + n].
 */
BFP8_API bfp8_status bfp8_quant_rhs(const void *x, int64_t K, int64_t N, int64_t ldx,
                           void *qT, int64_t ldq, float *s, int64_t lds, bfp8_stream_t stream);

/*
 * weight_quant_rhs: 128x128 tiles of W[N,K], one scale per tile.
 * Source: "Enable blockwise FP8 dense training kernels on ROCm" — quantization
 * kernel correctness table (weight_quant_rhs, block_size=128).
 *   w            device bf16 [N,K], ldw >= K.
 *   q            device e4m3 [N, ldq] or NULL (not written), ldq >= K,
 *                ldq % 16 == 0, 16-byte aligned.
 *   qt           device e4m3 [K, ldqt] or NULL: the same bytes transposed
 *                (qt[k*ldqt + n] = q[n*ldq + k]) for the input-gradient GEMM;
 *                ldqt >= N, ldqt % 16 == 0, 16-byte aligned.
 *   s            device fp32 row-major [Nb, Kb]: s[nb*lds + kb], lds >= Kb.
 * At least one of q, qt must be non-NULL.
 */
BFP8_API bfp8_status bfp8_quant_weight(const void *w, int64_t N, int64_t K, int64_t ldw,
                              void *q, int64_t ldq, void *qt, int64_t ldqt,
                              float *s, int64_t lds, bfp8_stream_t stream);

/*
 * Both 1x128 and 128x1 groups of one bf16 tensor X[T,C] from a single read:
 *   q_row[t*ldq_row + c], s_row[(c/128)*lds_row + t]   — as bfp8_quant_lhs(X)
 *   q_col[c*ldq_col + t], s_col[(t/128)*lds_col + c]   — as bfp8_quant_rhs(X),
 *                                                        = bfp8_quant_lhs(X^T)
 * Source: the same three quantisations of "Enable blockwise FP8 dense
 * training kernels on ROCm" (correctness table); fusing them is this
 * library's choice (a training step needs both forms of x and of dY).
 *   x  device bf16 [T,C], ldx >= C;  q_row, q_col 16-byte aligned, ld % 16 == 0,
 *   ldq_row >= C, ldq_col >= T, lds_row >= T, lds_col >= C.
 */
BFP8_API bfp8_status bfp8_quant_dual(const void *x, int64_t T, int64_t C, int64_t ldx,
                                     void *q_row, int64_t ldq_row, float *s_row, int64_t lds_row,
                                     void *q_col, int64_t ldq_col, float *s_col, int64_t lds_col,
                                     bfp8_stream_t stream);

/*
 * bfp8_quant_dual of x and bfp8_quant_weight of w (with both q and qt) in
 * one launch: a training step's forward needs both, and at small sizes one
 * persistent launch over both inputs' tiles beats two.  Same sources as the
 * two calls.  x device bf16 [T,C], w device bf16 [N,C] (C is the shared
 * reduction width); arguments and layouts as in bfp8_quant_dual (q_row, s_row,
 * q_col, s_col) and bfp8_quant_weight (qw = its q, qwt = its qt, sw = its s,
 * ldsw >= ceil(C/128)).  (x or w not 16-byte aligned, or ldx / ldw not
 * multiples of 8: the two calls are made instead.)
 */
BFP8_API bfp8_status bfp8_quant_dual_weight(const void *x, int64_t T, int64_t C, int64_t ldx,
                                     void *q_row, int64_t ldq_row, float *s_row, int64_t lds_row,
                                     void *q_col, int64_t ldq_col, float *s_col, int64_t lds_col,
                                     const void *w, int64_t N, int64_t ldw, void *qw, int64_t ldqw,
                                     void *qwt, int64_t ldqwt, float *sw, int64_t ldsw, bfp8_stream_t stream);

/*
 * MXFP8 casts of x [M,K] (bf16): E4M3 codes with one E8M0 exponent per block
 * of 32 elements.  Source: "Fixes accuracy error for mxfp8 linear" (the mxfp8
 * linear, its dim1 cast kernel, ScaleCalculationMode.FLOOR); the page does not
 * spell the format out, so the OCP Microscaling Formats v1.0 definition is
 * taken: e = floor(log2(amax)) - 8 clamped to [-127, 127] (-127 for an
 * all-zero block), stored biased (e + 127); q = RNE_e4m3(clamp(x * 2^-e, +-448)).
 *   dim0 (q0, e0 non-null): blocks of 32 along K; q0[m*ldq0 + k],
 *        e0[m*lde0 + k/32], ldq0 >= K, lde0 >= ceil(K/32).
 *   dim1 (q1, e1 non-null): blocks of 32 along M, written transposed;
 *        q1[k*ldq1 + m], e1[k*lde1 + m/32], ldq1 >= M, lde1 >= ceil(M/32).
 *   x and q0 / q1 16-byte aligned, ldx a multiple of 8, ldq0 / ldq1 multiples
 *   of 16 (BFP8_ERR_INVALID_ARG otherwise).  Either cast or both from one read.
 */
BFP8_API bfp8_status bfp8_mx_cast(const void *x, int64_t M, int64_t K, int64_t ldx,
                                 void *q0, int64_t ldq0, void *e0, int64_t lde0,
                                 void *q1, int64_t ldq1, void *e1, int64_t lde1, bfp8_stream_t stream);

/*
 * GEMM 1x128 x 128x128 (forward and input gradient).
 * Source: "Mask a_s/b_s scale loads in blockwise FP8 training GEMM kernels" —
 * Summary (triton_fp8_gemm_1x128_128x128_kernel, per-tile a_s/b_s) and Fix
 * (a_s load masked to offs_m < M, b_s load to offs_n < N, output store masked).
 * C[M,N] = A[M,K] B[K,N] with
 *   qa           device e4m3 [M, lda], lda >= K, lda % 16 == 0, 16-byte aligned.
 *   sa           device fp32 column-major 1x128 scales: sa[kb*ldsa + m], ldsa >= M.
 *   qb           device e4m3 B^T as [N, ldb] (K contiguous), ldb >= K,
 *                ldb % 16 == 0, 16-byte aligned.
 *   sb           device fp32 128x128 tile scales of B, nb = n/128:
 *                sb_transposed == 0: sb[nb*ldsb + kb], ldsb >= Kb
 *                  (the weight's own [Nb,Kb] scales: forward, y = x W^T);
 *                sb_transposed == 1: sb[kb*ldsb + nb], ldsb >= ceil(N/128)
 *                  (the weight's [Nb_out, Kb_in] scales read for dX = dY W).
 *   c            device bf16 [M, ldc], ldc >= N.  Only m < M, n < N written.
 */
BFP8_API bfp8_status bfp8_gemm_1x128_128x128(const void *qa, int64_t lda, const float *sa, int64_t ldsa,
                                    const void *qb, int64_t ldb, const float *sb, int64_t ldsb,
                                    int sb_transposed, void *c, int64_t ldc,
                                    int64_t M, int64_t N, int64_t K, bfp8_stream_t stream);

/*
 * GEMM 1x128 x 128x1 (weight gradient).
 * Source: "Mask a_s/b_s scale loads in blockwise FP8 training GEMM kernels" —
 * Summary (triton_fp8_gemm_1x128_128x1_kernel) and Fix.
 * As bfp8_gemm_1x128_128x128 except that B has one scale per column and
 * K-block: sb[kb*ldsb + n], ldsb >= N (the layout bfp8_quant_rhs writes).
 */
BFP8_API bfp8_status bfp8_gemm_1x128_128x1(const void *qa, int64_t lda, const float *sa, int64_t ldsa,
                                  const void *qb, int64_t ldb, const float *sb, int64_t ldsb,
                                  void *c, int64_t ldc,
                                  int64_t M, int64_t N, int64_t K, bfp8_stream_t stream);

/*
 * Grouped GEMM 1x128 x 128x128 for a mixture-of-experts layer (forward and
 * input gradient): token rows grouped by expert.
 * Source: "Enable blockwise FP8 dense training kernels on ROCm" — its
 * description names an MoE path beside the dense kernels; reading taken:
 * each expert's GEMM is exactly bfp8_gemm_1x128_128x128 on its tokens.
 *   offs   DEVICE int32 [E+1], 1 <= E <= 1024: expert e owns token rows
 *          offs[e] .. offs[e+1]; non-decreasing, 0 <= offs[e] <= M_total.
 *          Violations are clamped on the device and reported by
 *          bfp8_check_device_errors (BFP8_ERR_INVALID_ARG).
 *   qa, sa as bfp8_gemm_1x128_128x128 with M = M_total (sa[kb*ldsa + m], ldsa >= M_total).
 *   sb_transposed == 0 (forward, y_e = x_e W_e^T): qb = the experts' weight
 *          codes stacked [E*N, ldb], ldb >= K; sb = their tile scales stacked
 *          [E*ceil(N/128), ldsb], ldsb >= ceil(K/128).
 *   sb_transposed == 1 (input gradient, dx_e = dy_e W_e; here K = the
 *          experts' output features): qb = the transposed codes [N, ldb],
 *          ldb >= E*K, expert e in columns e*K .. (e+1)*K (what
 *          bfp8_quant_weight writes as qt for the stacked weight), K % 16 == 0
 *          when E > 1 (a TMA load starts on a 16-byte boundary); sb = the
 *          stacked weight's tile scales [E*ceil(K/128), ldsb], ldsb >= ceil(N/128).
 *   c      device bf16 [M_total, ldc], ldc >= N.  Rows outside
 *          [offs[0], offs[E]) and columns >= N are not written.
 */
BFP8_API bfp8_status bfp8_gemm_grouped_1x128_128x128(const void *qa, int64_t lda, const float *sa, int64_t ldsa,
                                    const void *qb, int64_t ldb, const float *sb, int64_t ldsb,
                                    int sb_transposed, const int32_t *offs, int64_t E,
                                    void *c, int64_t ldc, int64_t M_total, int64_t N, int64_t K,
                                    bfp8_stream_t stream);

/*
 * Grouped GEMM 1x128 x 128x1 for a mixture-of-experts layer (weight
 * gradient): dW_e = dY_e^T X_e, each expert reducing over its own tokens.
 * Source and reading as bfp8_gemm_grouped_1x128_128x128; the 128-token
 * groups along the token dim stay inside one expert only if every expert
 * starts on a 128-token boundary, so offs[e] % 128 == 0 is required for
 * e < E (offs[E] <= T may be ragged).
 *   qa     device e4m3 [M, lda], lda >= T (dY^T codes, 1x128 along tokens);
 *          sa[tb*ldsa + m], ldsa >= M.
 *   qb     device e4m3 [N, ldb], ldb >= T (X codes, 128x1 along tokens,
 *          transposed); sb[tb*ldsb + n], ldsb >= N.
 *   c      device bf16: expert e's [M, ldc] block at c + e*c_expert_stride
 *          elements, ldc >= N, c_expert_stride >= M*ldc.  An expert without
 *          tokens gets zeros.
 */
BFP8_API bfp8_status bfp8_gemm_grouped_1x128_128x1(const void *qa, int64_t lda, const float *sa, int64_t ldsa,
                                    const void *qb, int64_t ldb, const float *sb, int64_t ldsb,
                                    const int32_t *offs, int64_t E, void *c, int64_t ldc,
                                    int64_t c_expert_stride, int64_t M, int64_t N, int64_t T,
                                    bfp8_stream_t stream);

/*
 * Blockwise-FP8 linear layer (the Float8BlockwiseLinear computation of the
 * ROCm enablement page: quantise, then the blockwise GEMMs), y = x W^T.
 *   x  device bf16 [M,K] contiguous;  w  device bf16 [N,K] contiguous;
 *   y  device bf16 [M,N] contiguous.
 *   ws device workspace of at least bfp8_linear_workspace_size(M,N,K) bytes,
 *      256-byte aligned; its contents on return are the quantised operands
 *      (scratch for the caller).
 */
BFP8_API size_t bfp8_linear_workspace_size(int64_t M, int64_t N, int64_t K);
BFP8_API bfp8_status bfp8_linear_fwd(const void *x, const void *w, void *y, int64_t M, int64_t N, int64_t K,
                            void *ws, size_t ws_bytes, bfp8_stream_t stream);

/*
 * Backward of the linear layer: dx = dy W (GEMM 1x128 x 128x128 with dY
 * quantised 1x128 along N and W's tiles transposed) and dw = dy^T x (GEMM
 * 1x128 x 128x1 with dY^T quantised 1x128 along M and x quantised 128x1 along
 * M).  dy [M,N], x [M,K], w [N,K], dx [M,K], dw [N,K], all contiguous bf16.
 */
BFP8_API bfp8_status bfp8_linear_bwd(const void *dy, const void *x, const void *w, void *dx, void *dw,
                            int64_t M, int64_t N, int64_t K, void *ws, size_t ws_bytes,
                            bfp8_stream_t stream);

/*
 * Training form of the linear layer: the forward quantises x once into both
 * of its forms (1x128 along K for y = x W^T, 128x1 along M for dW) and W once
 * into its tiles as is and transposed, keeping them in `ws`; the backward
 * quantises dY once into both forms and runs dX = dY W and dW = dY^T x from
 * what the forward kept.  `ws` (>= bfp8_linear_train_workspace_size(M,N,K)
 * bytes, 256-byte aligned) must be the one the forward filled, unmodified,
 * with the same M, N, K.  All tensors contiguous bf16: x [M,K], w [N,K],
 * y [M,N], dy [M,N], dx [M,K], dw [N,K].
 */
BFP8_API size_t bfp8_linear_train_workspace_size(int64_t M, int64_t N, int64_t K);
BFP8_API bfp8_status bfp8_linear_fwd_train(const void *x, const void *w, void *y, int64_t M, int64_t N,
                                           int64_t K, void *ws, size_t ws_bytes, bfp8_stream_t stream);
BFP8_API bfp8_status bfp8_linear_bwd_saved(const void *dy, void *dx, void *dw, int64_t M, int64_t N,
                                           int64_t K, void *ws, size_t ws_bytes, bfp8_stream_t stream);

/*
 * One whole training step of the linear layer from HOST memory: copies x, W
 * and dY in, runs the training form (forward y = x W^T, input gradient
 * dX = dY W, weight gradient dW = dY^T x, each operand quantised once in the
 * method's groups — 1x128 for x / dY, 128x128 tiles for W, 128x1 along M
 * for the weight gradient's right operand; "Enable blockwise FP8 dense
 * training kernels on ROCm", the Float8BlockwiseLinear forward/backward) and
 * copies y, dX and dW out.  Results equal those of bfp8_linear_fwd_train +
 * bfp8_linear_bwd_saved on the same inputs.
 *
 * The copies overlap the kernels: W and dY travel in chunks of `chunk_n`
 * output features (0 = automatic: about N/8, at least 1024; otherwise a
 * multiple of 128, at most 64 chunks); chunk j's forward and weight-gradient
 * GEMMs run while chunk j+1 arrives, and its y and dW columns leave while
 * later chunks run; dX is computed in up to four row pieces at the end and
 * leaves piece by piece.  The copies run on two streams the library creates
 * per device (once, kept for the process); the caller's `stream` orders the
 * step: nothing starts before work already on it, and work enqueued on it
 * afterwards runs after every copy of the step.
 *
 *   x [M,K], w [N,K], dy [M,N] (inputs), y [M,N], dx [M,K], dw [N,K]
 *   (outputs): contiguous row-major bf16 in host memory.  Page-locked memory
 *   (cudaHostAlloc / cudaHostRegister) lets the copies run asynchronously;
 *   pageable memory works, with copies that block the host.  (Device
 *   pointers also work: copies use cudaMemcpyDefault.)  The buffers must stay
 *   valid and the inputs unmodified until the stream reaches the end of the
 *   step; the outputs are complete once it has.
 *   ws: device, >= bfp8_linear_step_host_workspace_size(M,N,K) bytes,
 *   256-byte aligned; holds the device copies and the quantised operands.
 *   Several host threads may call at once, each with its own workspace:
 *   their enqueues take turns on the device's copy streams.
 * Errors: BFP8_ERR_INVALID_ARG for bad sizes, pointers, chunk_n or workspace
 * (nothing enqueued); launch or copy failures return their status after the
 * caller's stream has been joined to the copy streams.
 */
BFP8_API size_t bfp8_linear_step_host_workspace_size(int64_t M, int64_t N, int64_t K);
BFP8_API bfp8_status bfp8_linear_step_host(const void *x, const void *w, const void *dy, void *y, void *dx,
                                           void *dw, int64_t M, int64_t N, int64_t K, int64_t chunk_n,
                                           void *ws, size_t ws_bytes, bfp8_stream_t stream);

/*
 * The mixture-of-experts layer's training step from HOST memory: tokens
 * sorted by expert, expert e owning token rows offs[e] .. offs[e+1] of x
 * [T,K], dy [T,N], y [T,N], dx [T,K] and the weight w[e] = w + e*N*K
 * ([N,K]), gradient dw[e] = dw + e*N*K.  Each expert with tokens runs as one
 * bfp8_linear_step_host step on its rows (the same per-expert quantisations
 * and GEMMs as the grouped path when the experts start on 128-token
 * boundaries; any boundaries work here), two experts' device buffers in turn
 * so that one expert's copies overlap another's kernels.  Experts without
 * tokens get dw[e] = 0; rows outside [offs[0], offs[E]) of y and dx are not
 * written.
 *   offs: HOST int32 [E+1], non-decreasing, within [0, T] (checked here);
 *   1 <= E <= 4096.  Other buffers, chunk_n, stream and errors as
 *   bfp8_linear_step_host.  ws: device, >= bfp8_moe_step_host_workspace_size(
 *   M_max, N, K) bytes (M_max = the largest expert's token count), 256-byte
 *   aligned.
 */
BFP8_API size_t bfp8_moe_step_host_workspace_size(int64_t M_max, int64_t N, int64_t K);
BFP8_API bfp8_status bfp8_moe_step_host(const void *x, const void *w, const void *dy, const int32_t *offs,
                                        int64_t E, void *y, void *dx, void *dw, int64_t T, int64_t N, int64_t K,
                                        int64_t chunk_n, void *ws, size_t ws_bytes, bfp8_stream_t stream);

/*
 * The forward GEMM 1x128 x 128x128 with its A operand quantised inside the
 * kernel: C = quant_lhs(x) . (the weight's 128x128-tile codes)^T, for an
 * activation x that has not been quantised yet and a weight that has (e.g.
 * cached between calls).  The method is that of bfp8_quant_lhs followed by
 * bfp8_gemm_1x128_128x128 ("Enable blockwise FP8 dense training kernels on
 * ROCm": act_quant_lhs, the 1x128 x 128x128 GEMM; "Mask a_s/b_s scale loads
 * in blockwise FP8 training GEMM kernels", Fix: masked loads and stores) and
 * the result is the same bits: each row's 1x128 group maximum, scale
 * s = amax/448 and codes RNE_e4m3(clamp(x/s, +-448)) are formed in shared
 * memory by a quantiser warpgroup with the quantisation kernels' arithmetic,
 * and never written to global memory.  One launch instead of two, without the
 * codes' HBM round trip: meant for small M (a few token rows), where the
 * separate quantisation launch is a large share of the forward.
 *   x  device bf16 [M, K] row-major, ldx >= K, ldx % 8 == 0, 16-byte aligned;
 *   qb device e4m3 [N, K] (bfp8_quant_weight's q), ldb >= K, ldb % 16 == 0,
 *      16-byte aligned; sb device fp32 [ceil(N/128), ceil(K/128)] tile scales,
 *      ldsb >= ceil(K/128);
 *   c  device bf16 [M, N], ldc >= N; only the logical [M, N] region is written.
 * K == 0 sets the [M, N] region of c to zero and reads nothing else.
 * Errors: BFP8_ERR_INVALID_ARG (sizes, strides, alignment, null pointers),
 * BFP8_ERR_UNSUPPORTED (not sm_103), BFP8_ERR_CUDA (launch); a bounded wait
 * that gave up is reported by bfp8_check_device_errors.
 */
BFP8_API bfp8_status bfp8_gemm_1x128_128x128_xq(const void *x, int64_t ldx, const void *qb, int64_t ldb,
                                                const float *sb, int64_t ldsb, void *c, int64_t ldc, int64_t M,
                                                int64_t N, int64_t K, bfp8_stream_t stream);

/*
 * Weight-gradient GEMM 1x128 x 128x1 with the rhs quantised inside the
 * kernel: C[M,N] = A[M,K] quant_rhs(X)[K,N], the optional fused quantisation
 * in the GEMM prologue for the weight gradient's rhs.  Source: "Enable
 * blockwise FP8 dense training kernels on ROCm" — quantization kernel
 * correctness table (act_quant_rhs, block_size=128) and the 1x128 x 128x1
 * GEMM; "Mask a_s/b_s scale loads in blockwise FP8 training GEMM kernels",
 * Summary (triton_fp8_gemm_1x128_128x1_kernel) and Fix (masked scale loads
 * and stores).  The result is the same bits as bfp8_quant_rhs followed by
 * bfp8_gemm_1x128_128x1: each 128-token block of each column of X gets its
 * group maximum, scale s = amax/448 and codes RNE_e4m3(clamp(x/s, +-448)),
 * formed in shared memory by a quantiser warpgroup with the quantisation
 * kernels' arithmetic and never written to global memory.  Every 128-row
 * tile of C quantises the columns of X it reads, so the quantisation work is
 * ceil(M/128)-fold: one launch and no HBM round trip of the codes, at the
 * cost of recomputation (the two-launch path is faster for large M).
 *   qa device e4m3 [M, lda] (K contiguous: dY^T for dW = dY^T X), lda >= K,
 *      lda % 16 == 0, 16-byte aligned; sa device fp32 1x128 scales
 *      sa[kb*ldsa + m], ldsa >= M (bfp8_quant_lhs's transposed form);
 *   x  device bf16 [K, N] row-major (K tokens, N features), ldx >= N,
 *      ldx % 8 == 0, 16-byte aligned;
 *   c  device bf16 [M, N], ldc >= N; only the logical [M, N] region is written.
 * K == 0 sets the [M, N] region of c to zero and reads nothing else.
 * Errors: BFP8_ERR_INVALID_ARG (sizes, strides, alignment, null pointers),
 * BFP8_ERR_UNSUPPORTED (not sm_103), BFP8_ERR_CUDA (launch); a bounded wait
 * that gave up is reported by bfp8_check_device_errors.
 */
BFP8_API bfp8_status bfp8_gemm_1x128_128x1_xq(const void *qa, int64_t lda, const float *sa, int64_t ldsa,
                                              const void *x, int64_t ldx, void *c, int64_t ldc, int64_t M,
                                              int64_t N, int64_t K, bfp8_stream_t stream);

/*
 * Linear forward without caller-provided scratch (no counterpart on the pages:
 * an addition for callers that cannot allocate device memory — plugins hosted
 * by a framework that owns every allocation and hands them no allocator, and
 * latency-critical code that must not enter the driver's allocator, where a
 * cudaMalloc can synchronise the device).  Same inputs, output and launches as
 * bfp8_linear_fwd, so the same result bits; the quantised x and W and their
 * scales live in one 32 MiB array that the library reserves on every GPU that
 * loads it, for the life of the process.  Problems needing more than 32 MiB
 * of quantised operands (about M*K + N*K bytes plus scales) return
 * BFP8_ERR_INVALID_ARG.  All calls share that array: calls whose work
 * overlaps on the GPU race, so order them (one stream, or events).  Nothing
 * in it needs clearing between calls.  The first call in each CUDA context
 * (normally once per device) looks the array's address up with that device
 * current and keeps it for that context.  A new context on the same device
 * (after cudaDeviceReset, or a driver-API context the caller made current) is
 * looked up again on its first call.  Allocates nothing.  Errors: BFP8_ERR_INVALID_ARG (sizes,
 * null pointers), BFP8_ERR_UNSUPPORTED (not sm_103), BFP8_ERR_CUDA (the
 * lookup or a launch failed).
 */
BFP8_API bfp8_status bfp8_linear_fwd_static(const void *x, const void *w, void *y, int64_t M, int64_t N,
                                            int64_t K, bfp8_stream_t stream);

/*
 * The method's rounding step on its own: q[i] = RNE_e4m3fn(x[i]) with
 * saturation to +-448 (the clamp).  x device fp32 [n], q device e4m3 [n].
 */
BFP8_API bfp8_status bfp8_cast_e4m3(const float *x, int64_t n, void *q, bfp8_stream_t stream);

/*
 * Synchronises `stream` and reports whether a GEMM kernel gave up on a
 * bounded wait since the last call (BFP8_ERR_TIMEOUT, with the failing wait
 * in the message); clears the flag.  Every wait inside the GEMM kernels is
 * bounded in time, so a broken pipeline ends the kernel with this flag set
 * instead of hanging the GPU.
 */
BFP8_API bfp8_status bfp8_check_device_errors(bfp8_stream_t stream);

/*
 * Test hook for failure detection (no counterpart on the pages): launches the
 * 1x128 x 128x128 GEMM with the arguments of bfp8_gemm_1x128_128x128
 * (sb not transposed) but makes its promotion warps wait on a barrier that
 * nothing arrives on, with every wait bounded by wait_limit_us (<= 2 s).  The
 * kernel must give up, record the timeout, release its resources and return;
 * bfp8_check_device_errors then reports BFP8_ERR_TIMEOUT and the context stays
 * usable.  C is left unwritten.
 */
BFP8_API bfp8_status bfp8_debug_gemm_stall(const void *qa, int64_t lda, const float *sa, int64_t ldsa,
                                           const void *qb, int64_t ldb, const float *sb, int64_t ldsb,
                                           void *c, int64_t ldc, int64_t M, int64_t N, int64_t K,
                                           int64_t wait_limit_us, bfp8_stream_t stream);

/*
 * Host-side replay of a kernel's index arithmetic (no GPU needed): counts how
 * many times each logical output element would be written by the kernel that
 * `kind` names, for the launch configuration the library would use on a
 * 152-SM GB300.  flag bit 0: x_transposed (kind 0); flag bit 1: replay the
 * untiled fallback kernels (used when the input is not 16-byte aligned or its
 * row stride is not a multiple of 8) instead of the TMA-staged tile kernel;
 * flag bit 3 (kind 3): the 1x128 x 128x1 GEMM (its epilogue has another
 * warp layout) instead of the 1x128 x 128x128 ones.
 *   kind 0: bfp8_quant_lhs q           (rows = M, cols = K), scales [Kb, M]
 *   kind 1: bfp8_quant_rhs qT          (rows = N, cols = K), scales [Kb, N]
 *   kind 2: bfp8_quant_weight q        (rows = N, cols = K), scales [Nb, Kb]
 *   kind 3: GEMM output C              (rows = M, cols = N)
 *   kind 4: bfp8_quant_weight qt       (rows = K, cols = N)
 *   kind 5: bfp8_quant_dual q_row      (rows = M, cols = K), scales [Kb, M]  (T = M, C = K)
 *   kind 6: bfp8_quant_dual q_col      (rows = K, cols = M), scales [Mb, K]
 * counts is host uint32 [rows*cols] (incremented); *oob receives the number
 * of writes that would land outside the logical tensor.  Scale writes are
 * counted in scale_counts (host uint32 [scale_rows*scale_cols], may be NULL).
 */
BFP8_API bfp8_status bfp8_debug_write_counts(int kind, int64_t M, int64_t N, int64_t K, int flag,
                                    uint32_t *counts, uint32_t *scale_counts, int64_t *oob);

/*
 * Host test hook: the output tile width (32, 64, 128, 224 or 256 columns) the
 * GEMM launcher picks for an M x N output on a GPU of num_sms SMs
 * (col_scales != 0: the 1x128 x 128x1 GEMM).  Pure host arithmetic; returns
 * the width, or 0 for a non-positive size.
 */
BFP8_API int bfp8_debug_gemm_pick_bn(int64_t M, int64_t N, int col_scales, int num_sms);

/*
 * Host test hook: whether a dense or grouped GEMM or a tiled quantisation of
 * this size is launched with programmatic dependent launch (its set-up
 * overlapping the end of the kernel before it; long kernels are launched
 * without it, and then do not let the next kernel start early either).
 * kind 0: a GEMM of a x b x c (M, N, K); kind 1: a quantisation reading a
 * bytes of bf16 (b, c unused).  Pure host arithmetic; returns 1 or 0, or -1
 * for an unknown kind or a negative size.
 */
BFP8_API int bfp8_debug_launch_pdl(int kind, int64_t a, int64_t b, int64_t c);

#ifdef __cplusplus
}
#endif
#endif /* BFP8_H_ */
