/*
 * gq.h -- GPTQ layer quantization, EoRA compensation and GPTQ-intrinsic LoRA on one
 * NVIDIA B300 (sm_103a).
 *
 * C ABI of libgq.so.  Every pointer argument is a CUDA DEVICE pointer unless its
 * comment says "host".  The caller owns every buffer; the library never
 * allocates or frees device memory: scratch space is the caller's workspace
 * `ws` of at least the size that the matching *_workspace_size() query returns,
 * 256-byte aligned.  All device work is enqueued on `stream` (a cudaStream_t;
 * NULL = the legacy default stream).  Matrices are row-major and dense.
 *
 * Shapes follow the linear layer y = x W^T: W is rows x cols = out x in, the
 * calibration activations X are n x cols (n tokens), H is cols x cols.
 *
 * Errors: argument errors are found on the host before anything is enqueued and
 * are returned as GQ_EINVAL / GQ_EUNSUPPORTED / GQ_EWORKSPACE.  A launch error is
 * returned as GQ_ECUDA.  Calls that factor H synchronize `stream` once, after the
 * factorization, to read the device status word; they return GQ_ENOTPD with
 * *info = the first input column whose pivot was not positive.  The same
 * synchronization reports an Inf or NaN in the inputs they read: GQ_ENONFINITE
 * with *info = 0 when it is in H (the diagonal and upper triangle, the part the
 * factor reads) and *info = 1 when it is in W (or EoRA's dW).  A non-finite
 * calibration token makes H non-finite, so it is reported as *info = 0 by the
 * first factoring call after gptq_hessian_accumulate; the asynchronous calls
 * (gptq_hessian_accumulate, gptq_sweep, the packed and Bid-Up calls) do not
 * check.  GQ_ENONFINITE takes precedence over GQ_ENOTPD.  On any non-OK
 * return the contents of the outputs are unspecified.
 *
 * Pages the operations follow (cited by title and section):
 *   [GPTQ-wiki]  "GPTQ", wikiprompt.org encyclopedia entry, "Enfoque Técnico".
 *   [LowBit]     "El balance de errores de la inferencia de pocos bits: escalas de
 *                cuantización, calibración y ahorro real de memoria", auturnal.com,
 *                sections 1 (format) and 2 (input covariance).
 *   [EoRA-blog]  "Aumento de la precisión de LLM de 2 bits con EoRA", 7minutos.es,
 *                "Bucear en el espacio propio en busca de un adaptador".
 *   [GPTQ-LoRA]  "Resumen Técnico: GPTQ-intrinsic LoRA", gist.science,
 *                "Metodología", item 2 "Algoritmo GPTQ-intrinsic LoRA".
 */
#ifndef GQ_H
#define GQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *gq_stream_t; /* identical to cudaStream_t */

typedef enum {
    GQ_OK = 0,
    GQ_EINVAL = -1,       /* null required pointer, bad shape, stride or size rule */
    GQ_ENOTPD = -2,       /* damped H not positive definite; *info = column */
    GQ_EUNSUPPORTED = -3, /* bits not in {2,3,4}, unknown dtype */
    GQ_ECUDA = -4,        /* CUDA runtime / launch error */
    GQ_ENONFINITE = -5,   /* Inf or NaN in an input; *info = 0 (H) or 1 (W / dW) */
    GQ_ETIMEOUT = -6,     /* a bounded device-side wait gave up */
    GQ_EWORKSPACE = -7    /* workspace missing, too small or not 256-byte aligned */
} gq_status;

typedef enum { GQ_F32 = 0, GQ_BF16 = 1 } gq_dtype;

/* Version of this ABI (bumped on any signature change). */
int gq_abi_version(void);

/* Number of kernel launches this library has enqueued since it was loaded,
 * all devices and streams (a monotonic host-side counter; for accounting). */
unsigned long long gq_kernel_launches(void);

/* Human-readable name of a status code (static string; never NULL). */
const char *gq_status_string(gq_status s);

/*
 * Synchronizes `stream`, then reports whether any bounded device-side wait of
 * the library's kernels gave up since the previous call (GQ_ETIMEOUT; the
 * affected outputs are then invalid) and clears that record.  GQ_OK otherwise.
 */
gq_status gq_check_device(gq_stream_t stream);

/*
 * Sets, on the current device, the budget in SM clock cycles of each bounded
 * wait in the pipelines of the tensor-core kernels (Hessian, 3xTF32 GEMM,
 * packed linear); cycles <= 0 restores the default of 4e9 cycles (about 2 s).
 * A wait that runs out records the failure for gq_check_device (GQ_ETIMEOUT)
 * and the kernel ends early: it still waits, with the default budget, for the
 * copies and MMAs it has issued, frees its tensor memory and returns.  For
 * tests of that failure path: a tiny budget makes ordinary waits run out.
 * Synchronous; call it with no library work in flight.
 */
gq_status gq_set_wait_budget(long long cycles);

/*
 * Per-kernel-class timing of this library's launches, for measurement.  After
 * gq_timing_begin, the launchers of the main kernels bracket every launch with
 * a pair of CUDA events on the launch's stream (all devices, all streams).
 * gq_timing_end stops recording, waits for the recorded events and writes,
 * for kernel class k < nkinds, into the host arrays: ms[k] the summed elapsed
 * time, flops[k] the summed useful floating-point operations the launches
 * declared, count[k] the number of launches.  Classes: 0 the Hessian kernel
 * (n cols (cols + 1) flops per call), 1 the 3xTF32 GEMM (2 M N K useful
 * float32 flops; only the outputs on and below the diagonal for the
 * triangular updates), 2 the sweep's block kernel (rows bw (bw - 1) flops of
 * the in-block updates), 3 the diagonal-block Cholesky + inverse (2 kb^3 / 3),
 * 4 the one-term TF32 GEMM of the subspace iterations (2 M N K).  Other kernels
 * are not bracketed.  Recording adds event records between launches: time a
 * workload without it and use this for the breakdown.
 */
gq_status gq_timing_begin(void);
gq_status gq_timing_end(double *ms, double *flops, unsigned long long *count, int nkinds);

/*
 * H += 2 X^T X.
 *
 * The second-order statistics of the layer inputs: the Hessian of the layer's
 * squared output error with respect to each weight row ([GPTQ-wiki] "Enfoque
 * Técnico"; [LowBit] section 2).  Both triangles of H are updated.
 *
 *   H     cols x cols float32, in/out (accumulated into; zero it for a fresh H).
 *   X     n x cols, element type xt (GQ_BF16 or GQ_F32), leading dimension ldx
 *         (elements, >= cols).  For GQ_BF16: X 16-byte aligned, ldx % 8 == 0.
 *   n     number of tokens; n == 0 is a no-op.
 * Accumulation is float32 (every bf16 x bf16 product is exact in float32).
 * Deterministic: the same inputs give bit-identical H.  Asynchronous.
 */
gq_status gptq_hessian_accumulate(float *H, int64_t cols, const void *X, gq_dtype xt, int64_t n,
                                  int64_t ldx, gq_stream_t stream);

/*
 * Factor of the damped Hessian.
 *
 * Dead inputs (H_ii == 0) get H_ii = 1; then H_d = H + damp * mean(diag H) * I.
 * Writes the upper-triangular F with H_d = F F^T (strictly-lower part set to 0),
 * obtained as the lower Cholesky factor of the index-reversed H_d.  Its inverse
 * U = F^-1 is the upper Cholesky factor of H_d^-1 (U^T U = H_d^-1), the matrix
 * whose rows drive GPTQ's error compensation ([GPTQ-wiki] "Enfoque Técnico");
 * the sweep uses F directly and never forms U.
 *
 *   H     cols x cols float32, read only (both triangles read; must be symmetric).
 *   F     cols x cols float32 output.
 *   dead  cols bytes output (1 = dead input), may be NULL.
 *   ws    >= gptq_factor_workspace_size(cols) bytes.
 *   info  host pointer, may be NULL; on GQ_ENOTPD receives the failing column.
 * Synchronizes `stream` once.
 */
size_t gptq_factor_workspace_size(int64_t cols);
gq_status gptq_factor(const float *H, int64_t cols, float damp, float *F, uint8_t *dead, void *ws,
                      size_t ws_bytes, gq_stream_t stream, int64_t *info);

/*
 * The GPTQ column sweep, given the factor F of gptq_factor.
 *
 * Columns are quantized in order, one group of `group` columns sharing a scale
 * and zero point per row ([LowBit] section 1; [GPTQ-wiki] "Enfoque Técnico":
 * per-group scale).  At a group's first column, from the weights as updated by
 * every earlier column: xmin = min(0, min w), xmax = max(0, max w) (both 0 ->
 * -1, +1), s = (xmax - xmin) / maxq, z = rint(-xmin / s), maxq = 2^bits - 1.
 * Each column: q = clamp(rint(w / s) + z, 0, maxq), ŵ = s (q - z), and the error
 * is propagated into the columns not yet quantized (closed-form OBQ update).
 * Blocks of `block` columns are swept in shared memory; the update of later
 * blocks is deferred and applied as GEMMs.  Decisions are float32 with IEEE
 * division and round-half-to-even.
 *
 *   W        rows x cols, type wt, read only (never modified), 16-byte aligned.
 *   F, dead  from gptq_factor (dead may be NULL = no dead inputs).
 *   bits     2, 3 or 4.  group % 32 == 0, cols % group == 0, block % group == 0,
 *            block <= 128, rows % 32 == 0, cols % 32 == 0.
 * Outputs (packing layout: little-endian bitstream of b-bit codes along the
 * packed axis, code k at bits [k*b, k*b+b) of the stream, cut into 32-bit words):
 *   qweight  [cols*bits/32][rows] int32: the codes of each output row packed
 *            along the input axis.
 *   scales   [cols/group][rows] float32, 16-byte aligned.
 *   qzeros   [cols/group][rows*bits/32] int32: zero points packed along rows.
 *   codes    rows x cols uint8, may be NULL (4-byte aligned).
 *   W_hat    rows x cols float32 dequantized weights, may be NULL (16-byte aligned).
 *   row_err  rows float32, may be NULL: sum over columns of e_j^2 with
 *            e_j = (w_j - ŵ_j) / U_jj, which equals ΔW_r H_d ΔW_r^T.
 *   ws       >= gptq_sweep_workspace_size(rows, cols, block) bytes.
 * Asynchronous.
 */
size_t gptq_sweep_workspace_size(int64_t rows, int64_t cols, int block);
gq_status gptq_sweep(const void *W, gq_dtype wt, int64_t rows, int64_t cols, const float *F,
                     const uint8_t *dead, int bits, int group, int block, int32_t *qweight,
                     float *scales, int32_t *qzeros, uint8_t *codes, float *W_hat, float *row_err,
                     void *ws, size_t ws_bytes, gq_stream_t stream);

/*
 * One layer: gptq_factor (into the workspace) followed by gptq_sweep.
 * Same arguments and rules as the two calls; H is read only.
 * Synchronizes `stream` once (after the factorization).
 */
size_t gptq_quantize_layer_workspace_size(int64_t rows, int64_t cols, int block);
gq_status gptq_quantize_layer(const void *W, gq_dtype wt, int64_t rows, int64_t cols, const float *H,
                              int bits, int group, int block, float damp, int32_t *qweight,
                              float *scales, int32_t *qzeros, uint8_t *codes, float *W_hat,
                              float *row_err, void *ws, size_t ws_bytes, gq_stream_t stream,
                              int64_t *info);

/*
 * The compression error that EoRA compensates, dW = W - Ŵ ([EoRA-blog]
 * "Bucear en el espacio propio en busca de un adaptador").
 *
 *   W      rows x cols, type wt (the original weights), read only.
 *   W_hat  rows x cols float32 (e.g. the W_hat output of gptq_quantize_layer).
 *   dW     rows x cols float32 output.
 * Asynchronous.
 */
gq_status gptq_weight_error(const void *W, gq_dtype wt, int64_t rows, int64_t cols, const float *W_hat, float *dW,
                            gq_stream_t stream);

/*
 * EoRA compensation of the quantization error ([EoRA-blog] "Bucear en el
 * espacio propio en busca de un adaptador").
 *
 * The error ΔW = W - Ŵ is projected into the eigenspace of the input
 * covariance, ΔW' = ΔW Q sqrt(Λ) with H = Q Λ Q^T, its SVD is truncated to
 * rank r, ΔW' ≈ U_r Σ_r V_r^T, and the result is projected back: B = U_r Σ_r,
 * A = V_r^T (Q sqrt(Λ))^-1, so that B A approximates ΔW and
 * 1/2 tr((ΔW - B A) H (ΔW - B A)^T) = 1/2 sum_{i>r} σ_i^2 (the layer loss left
 * after compensation) is minimal over all rank-r products.
 * Signs: the largest-magnitude entry of each column of B is positive (the
 * matching row of A carries the same sign).
 *
 *   dW     rows x cols float32, read only.
 *   H      cols x cols float32 (both triangles), used as passed (no damping);
 *          must be positive definite, else GQ_ENOTPD with *info = a column.
 *   r      1 <= r <= min(256, rows, cols); above 64 also cols >= r + 64.
 *   A      r x cols float32 output.   B  rows x r float32 output.
 *   sigma  r float32 output, may be NULL: the r largest singular values of the
 *          projected error ΔW', in descending order.
 *   ws     >= eora_compensate_workspace_size(rows, cols, r) bytes.
 * Computed in float32 with a block subspace iteration of width min(2r, 128,
 * cols) (30 iterations) and a Rayleigh-Ritz step.  Above r = 64 the singular
 * vectors come in chunks of 64: each chunk is found by a new iteration whose
 * block is kept orthogonal to the chunks before it (locking), and the r
 * values are sorted at the end.  When σ_r and σ_{r+1} are close,
 * the rank-r subspace is not unique and B A may differ from another exact
 * solution by directions of nearly equal σ; the compensated loss and σ do not.
 * Synchronizes `stream` once (after the factorization of H).
 */
size_t eora_compensate_workspace_size(int64_t rows, int64_t cols, int r);
gq_status eora_compensate(const float *dW, int64_t rows, int64_t cols, const float *H, int r, float *A, float *B,
                          float *sigma, void *ws, size_t ws_bytes, gq_stream_t stream, int64_t *info);

/*
 * The GPTQ-intrinsic LoRA basis ([GPTQ-LoRA] "Hessiano Aumentado"): L = V_r,
 * the r leading right singular vectors of the calibration matrix X, i.e. the r
 * leading eigenvectors of H = 2 X^T X.
 *
 *   H      cols x cols float32 (both triangles, symmetric positive
 *          semi-definite), read only.
 *   r      1 <= r <= min(64, cols).
 *   Lt     r x cols float32 output: row i is the i-th basis vector (L^T in the
 *          page's notation, which is also the adapter's A).  Rows are
 *          orthonormal; the largest-magnitude entry of each row is positive.
 *   lam    r float32 output, may be NULL: the Ritz values (eigenvalues of H,
 *          = 2 sigma_i(X)^2), descending.
 *   ws     >= gptq_lora_basis_workspace_size(cols, r) bytes.
 * Computed in float32 with a block subspace iteration of width min(2r, 128,
 * cols) (30 iterations) and a Rayleigh-Ritz step.  Where the eigenvalues
 * around the r-th are close the leading subspace is not unique; the Ritz
 * values and the captured sum tr(L^T H L) are.  Asynchronous.
 */
size_t gptq_lora_basis_workspace_size(int64_t cols, int r);
gq_status gptq_lora_basis(const float *H, int64_t cols, int r, float *Lt, float *lam, void *ws, size_t ws_bytes,
                          gq_stream_t stream);

/*
 * GPTQ-intrinsic LoRA of one layer ([GPTQ-LoRA] "Algoritmo GPTQ-intrinsic
 * LoRA"): W ≈ Q + R L^T with Q on the GPTQ grid and a rank-r correction whose
 * right factor is the given basis.
 *
 * Defined by the page's augmented problem: calibration X~ = [X, X L], Hessian
 * H~ = [[H, H L], [L^T H, L^T H L]] damped like GPTQ's (dead inputs, then
 * H~ + damp * mean(diag H~) * I over all cols + r diagonal entries), and the
 * GPTQ sweep over W~ = [W, 0] in which the first cols columns are quantized and
 * the last r, never quantized, absorb the quantization error; their final
 * values are R.  The library computes the same result by block elimination:
 * GPTQ on the Schur complement S = H_d - H L (L^T H L + delta I)^-1 L^T H (the
 * quantized block of the inverse of H~ is S^-1, so the codes are the augmented
 * sweep's), then R = (W - Ŵ) H L (L^T H L + delta I)^-1, the values the sweep
 * leaves in the free columns (the optimum of the augmented quadratic given Q).
 *
 *   W, wt, rows, cols, H, bits, group, block, qweight, scales, qzeros, codes,
 *   row_err   as for gptq_quantize_layer (row_err = sum_j e_j^2 over the
 *             quantized columns of the augmented sweep).
 *   Lt        r x cols float32 (rows orthonormal, e.g. from gptq_lora_basis), read only.
 *   r         1 <= r <= min(64, cols).
 *   damp      > 0 (H~ is singular: without damping it has no Cholesky factor).
 *   W_hat     rows x cols float32 output, required (R is formed from it), 16-byte aligned.
 *   R         rows x r float32 output: the adapter's B; its A is Lt.
 *   ws        >= gptq_intrinsic_lora_workspace_size(rows, cols, r, block) bytes.
 * Synchronizes `stream` once.  GQ_ENOTPD with *info = the failing column of
 * the augmented matrix: < cols for S, cols + i for row i of L^T H L + delta I.
 */
size_t gptq_intrinsic_lora_workspace_size(int64_t rows, int64_t cols, int r, int block);
gq_status gptq_intrinsic_lora(const void *W, gq_dtype wt, int64_t rows, int64_t cols, const float *H,
                              const float *Lt, int r, int bits, int group, int block, float damp, int32_t *qweight,
                              float *scales, int32_t *qzeros, uint8_t *codes, float *W_hat, float *row_err,
                              float *R, void *ws, size_t ws_bytes, gq_stream_t stream, int64_t *info);

/*
 * The quantized layer applied from its packed form ([LowBit] sections 1 and
 * 6: codes, per-group scale and zero point, dequantized inside the product;
 * [EoRA-blog] "Bucear en el espacio propio en busca de un adaptador": the
 * adapter B A added to the quantized weights, which also carries a
 * GPTQ-intrinsic LoRA with B = R, A = L^T):
 *
 *     Y = X Ŵ^T + (X A^T) B^T,    Ŵ[m, k] = scales[k / group][m] (q[m, k] - z[k / group][m])
 *
 * Ŵ is not rounded: each group's integer products are summed on the tensor
 * cores and scaled in float32, so Y is exact up to float32 summation.
 *
 *   X        n x cols bf16, row stride ldx (ldx >= cols, ldx % 8 == 0), 16-byte aligned.
 *   qweight, scales, qzeros   the layout gptq_quantize_layer writes for a layer of
 *            rows x cols at `bits` (2, 3, 4) and `group`; qweight and scales 16-byte aligned.
 *            Requires rows % 32 == 0, group % 64 == 0 (else GQ_EUNSUPPORTED), cols % group == 0.
 *   A, B     the adapter, r x cols and rows x r float32, or both NULL with r = 0; 0 <= r <= 64.
 *   Y        n x rows float32 output, row stride ldy (ldy >= rows, ldy % 4 == 0), 16-byte aligned.
 *   n        0 <= n <= 65535 * 128 tokens; n = 0 returns GQ_OK at once (X, Y may then be NULL).
 *   ws       >= gptq_packed_linear_workspace_size(n, rows, cols, group, r) bytes (X A^T, and for
 *            n <= 32 the partial sums of the decode path); may be NULL when that size is 0.
 * Up to 32 tokens (decode) the product runs on the SIMT pipes of every SM, split over K in
 * whole groups and reduced in a fixed order; above, on the tensor cores.  Asynchronous.
 */
size_t gptq_packed_linear_workspace_size(int64_t n, int64_t rows, int64_t cols, int group, int r);
gq_status gptq_packed_linear(const void *X, int64_t n, int64_t ldx, const int32_t *qweight, const float *scales,
                             const int32_t *qzeros, int64_t rows, int64_t cols, int bits, int group, const float *A,
                             const float *B, int r, float *Y, int64_t ldy, void *ws, size_t ws_bytes,
                             gq_stream_t stream);

/*
 * One Bid-Up sweep ([GPTQ-LoRA] "Metodología", item 4 "Refinamiento Bid-Up"):
 * the codes of a quantized layer are refined in place on their fixed grid
 * (each group's scale and zero point kept) against the target T = W - B A, the
 * layer minus its low-rank correction.  Column by column, in order, each code
 * moves to the grid point nearest ŵ_j + g_j / H_jj, where g = (T - Ŵ) H is kept
 * current after every move; each move minimizes 1/2 tr((T - Ŵ) H (T - Ŵ)^T)
 * over that one coordinate, so the objective never increases.  Alternated with
 * OLrC -- the optimal rank-r B A for fixed codes, which is eora_compensate on
 * W - Ŵ -- it gives the page's refinement cycle.
 *
 *   W        rows x cols, type wt, read only.   H  cols x cols float32 (undamped), 16-byte aligned.
 *   A, B     the correction, r x cols and rows x r float32, or both NULL with r = 0; 0 <= r <= 64.
 *   codes    rows x cols uint8, in/out (the layout gptq_quantize_layer writes).
 *   scales, qzeros   the grid, as gptq_quantize_layer writes them (read only).
 *   W_hat    rows x cols float32 output: s (q - z) of the refined codes.
 *   qweight  [cols*bits/32][rows] int32 output (the refined codes packed), may be NULL.
 *   changed  one device uint64, may be NULL: the number of codes that moved is ADDED to it.
 *   Requires rows % 32 == 0, cols % 32 == 0, group % 32 == 0, cols % group == 0.
 *   ws       >= gptq_bidup_workspace_size(rows, cols) bytes.
 * The integer decision rint(g_j / (H_jj s)) is taken in float32.  Asynchronous.
 */
size_t gptq_bidup_workspace_size(int64_t rows, int64_t cols);
gq_status gptq_bidup(const void *W, gq_dtype wt, int64_t rows, int64_t cols, const float *H, const float *A,
                     const float *B, int r, int bits, int group, uint8_t *codes, const float *scales,
                     const int32_t *qzeros, float *W_hat, int32_t *qweight, unsigned long long *changed, void *ws,
                     size_t ws_bytes, gq_stream_t stream);

/*
 * Round to nearest on the GPTQ grid, for low-precision low-rank factors
 * ([GPTQ-LoRA] "Resultados Clave": L and R quantized to 4 and 8 bits are often
 * lossless): per row and group of `group` consecutive columns, xmin = min(0,
 * min x), xmax = max(0, max x) ([-1, 1] when both are 0), s = (xmax - xmin) /
 * (2^bits - 1), z = rint(-xmin / s), q = clamp(rint(x / s) + z, 0, 2^bits - 1),
 * x̂ = s (q - z), every division IEEE float32 -- the grid of the GPTQ sweep
 * without its error propagation.
 *
 *   M       nrows x ncols float32, read only.   bits  2 .. 8.   ncols % group == 0.
 *   M_hat   nrows x ncols float32 output.   codes  nrows x ncols uint8 output, may be NULL.
 *   scales  [ncols/group][nrows] float32 output.   zeros  [ncols/group][nrows] uint8 output.
 * Asynchronous.
 */
gq_status gptq_quantize_rtn(const float *M, int64_t nrows, int64_t ncols, int bits, int group, float *M_hat,
                            uint8_t *codes, float *scales, uint8_t *zeros, gq_stream_t stream);

/*
 * gptq_quantize_layer without a caller-provided workspace, for callers that
 * cannot allocate device memory: code inside a host application that owns all
 * device memory through its own pool, a service that must not grow its device
 * footprint after start-up, a real-time loop where a synchronizing
 * cudaMalloc is not allowed.  The pages have no counterpart to this call; it
 * exists only because of how some callers manage memory.
 *
 * Same arguments, rules, outputs and status codes as gptq_quantize_layer,
 * without `ws` / `ws_bytes`.  The scratch is one fixed array of
 * GQ_NOALLOC_SCRATCH_BYTES (16 MiB) of device memory inside the library,
 * held by every GPU that loads the library until the process exits.  Nothing
 * is allocated or freed: no cudaMalloc, no cudaFree, no allocating library call.
 *
 *   Size limit: gptq_quantize_layer_workspace_size(rows, cols, block) must be
 *   <= GQ_NOALLOC_SCRATCH_BYTES (e.g. rows = cols = 768, block = 128 fits);
 *   larger layers are rejected with GQ_EWORKSPACE before anything is enqueued.
 *   Arguments are checked first, in gptq_quantize_layer's order, so a bad
 *   argument returns the status gptq_quantize_layer gives it at any size.
 *   All buffers must live on the current CUDA device, and `stream` must belong
 *   to it.  The first call on a device looks up the scratch's device address
 *   (cudaGetSymbolAddress); make that first call before any stream capture.
 *   Every call shares the one array and it keeps the last call's contents; the
 *   call clears what must start at zero itself.  Calls whose GPU work overlaps
 *   (other streams, other host threads) race on the array: serialize them.
 * Synchronizes `stream` once (after the factorization), like gptq_quantize_layer.
 */
#define GQ_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
gq_status gptq_quantize_layer_noalloc(const void *W, gq_dtype wt, int64_t rows, int64_t cols, const float *H,
                                      int bits, int group, int block, float damp, int32_t *qweight, float *scales,
                                      int32_t *qzeros, uint8_t *codes, float *W_hat, float *row_err,
                                      gq_stream_t stream, int64_t *info);

/*
 * The sweep's integer decision rule on its own, for verification: k[i] =
 * rint(w[i] / s[i]) with the quotient rounded as IEEE float32 division and ties
 * to even ([LowBit] section 1: the rounding rule is part of the format).  The
 * sweep forms the quotient from RN(1/s) with one FMA correction instead of a
 * division; this call lets a test compare the two on chosen inputs.
 *   w, s, k  n float32 each (device); s normal and nonzero.  Asynchronous.
 */
gq_status gptq_code_decisions(const float *w, const float *s, int64_t n, float *k, gq_stream_t stream);

/*
 * Standalone packing of codes (rows x cols uint8, each < 2^bits) into
 * qweight [cols*bits/32][rows] int32, and its inverse.  Same layout as
 * gptq_sweep.  rows % 32 == 0 is not required; cols*bits % 32 == 0 is.
 * Asynchronous.
 */
gq_status gptq_pack(const uint8_t *codes, int64_t rows, int64_t cols, int bits, int32_t *qweight,
                    gq_stream_t stream);
gq_status gptq_unpack(const int32_t *qweight, int64_t rows, int64_t cols, int bits, uint8_t *codes,
                      gq_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* GQ_H */
