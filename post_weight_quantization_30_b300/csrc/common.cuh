// Shared definitions of the libgq CUDA sources (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gq.h"

#define GQ_CUDA_TRY(expr)                                     \
    do {                                                      \
        cudaError_t err__ = (expr);                           \
        if (err__ != cudaSuccess) return GQ_ECUDA;            \
    } while (0)

#define GQ_LAUNCH_CHECK()                                     \
    do {                                                      \
        if (cudaGetLastError() != cudaSuccess) return GQ_ECUDA; \
    } while (0)

namespace gq {

// Counts one kernel launch enqueued by the library (host side).
void count_launch();

// Programmatic dependent launch.  The kernels of the long serial chains (the
// factor's panels, the sweep's blocks and their GEMMs) are launched with
// programmatic stream serialization: the next kernel may be scheduled while
// the previous one is still running, runs its prologue (barriers, TMEM,
// shared memory) on idle SMs, and calls pdl_wait() before its first access to
// global memory, which returns once the previous kernel has completed and its
// writes are visible.  Each of these kernels calls pdl_trigger() first, so
// that the next launch is not held back until it finishes.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Kernel classes of the optional per-launch timing (timing.cu; gq_timing_end
// reports them in this order).
enum TimedKind { TK_HESSIAN = 0, TK_GEMM3 = 1, TK_SWEEP = 2, TK_DIAG = 3, TK_GEMM_TF32 = 4, TK_COUNT = 5 };
// While recording is on, timing_begin records an event on `s` before a launch
// and returns a handle (-1 when off); timing_end records the closing event and
// the launch's useful floating-point operations.
int timing_begin(int kind, cudaStream_t s);
void timing_end(int handle, cudaStream_t s, double flops);

// Device status block kept in the workspace (set to all one bits before use).
// `bad_pivot` holds the first input column (in original index order) whose
// Cholesky pivot was not positive, or all ones when every pivot was fine.
// `finite` keeps all its bits while the inputs are finite: bit 0 is cleared
// when the part of H the factor reads holds an Inf or NaN, bit 1 when W (or
// EoRA's dW) does.
struct DeviceStatus {
    unsigned long long bad_pivot;
    double diag_sum;
    float delta;
    unsigned int finite;
};
constexpr unsigned int kNonFiniteH = 1u, kNonFiniteW = 2u;

static constexpr size_t kAlign = 256;

__host__ __device__ inline size_t align_up(size_t x, size_t a = kAlign) { return (x + a - 1) / a * a; }

// The quotient w / s rounded to nearest (IEEE), given y = RN(1/s): q0 = RN(w y),
// the exact residual r = w - s q0 (one FMA), q = RN(q0 + r y).  This is the
// FMA correction step of P. Markstein's division method ("IA-64 and Elementary
// Functions", Prentice Hall 2000, ch. 8): with y correctly rounded and q0
// within one ulp of w / s it yields the correctly rounded quotient for normal
// operands.  It was compared with the hardware IEEE division on 2.6e9 pairs
// (every significand of s against w within 3 ulps of half-integers, plus
// random pairs) without a difference; gptq_code_decisions exposes it to tests.
__device__ __forceinline__ float quotient_rn(float w, float s, float y) {
    const float q0 = w * y;
    const float r = fmaf(-s, q0, w);
    return fmaf(r, y, q0);
}

// The TF32 value nearest to x (ties away from zero); x - tf32_hi(x) is exact
// in float32, which is the split the 3xTF32 products use.
__device__ __forceinline__ float tf32_hi(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

template <typename T>
__device__ __forceinline__ float load_f32(const T *p);
template <>
__device__ __forceinline__ float load_f32<float>(const float *p) { return *p; }
template <>
__device__ __forceinline__ float load_f32<__nv_bfloat16>(const __nv_bfloat16 *p) { return __bfloat162float(*p); }

// ----------------------------------------------------------------------------
// Kernel launchers implemented in the .cu files (all enqueue on `s`).
// ----------------------------------------------------------------------------

// C[m, n] = beta * C[m, n] + alpha * sum_k A(m, k) B(k, n) in float32 on the SIMT
// pipes.  A(m, k) = a_t ? A[k * lda + m] : A[m * lda + k];
// B(k, n) = b_t ? B[n * ldb + k] : B[k * ldb + n].
// tri: 0 = full; 1 = only tiles that touch the lower triangle (m >= n);
//      2 = only tiles that touch the upper triangle, each off-diagonal tile
//      also written transposed (symmetric output).
template <typename TA>
cudaError_t sgemm(int64_t M, int64_t N, int64_t K, float alpha, const TA *A, int64_t lda, bool a_t,
                  const TA *B, int64_t ldb, bool b_t, float beta, float *C, int64_t ldc, int tri,
                  cudaStream_t s);

// C (M x N, row-major, ldc = N) = A B in float32, the K range split into
// `slices` parts computed by separate CTAs into `partials` (slices * M * N
// floats) and summed in a fixed order (deterministic).
cudaError_t sgemm_splitk(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda, bool a_t, const float *B,
                         int64_t ldb, bool b_t, float *C, float *partials, int slices, cudaStream_t s);

// C = beta C + alpha A B^T on the tensor cores with float32 accuracy (3xTF32):
// A (M x K) and B (N x K), K contiguous, each given as its TF32 split
// (hi, lo) with x = hi + lo.  tri = 1 skips the output tiles entirely above
// the diagonal; tri = 3 declares B lower triangular (B(k, n) = 0 for k > n,
// i.e. row n of the N x K operand is zero beyond column n), and the CTA-pair
// kernel then stops each tile's K loop after the tile's last column (the
// other kernels take the zero products).  Optional Chi / Clo (may be NULL) receive the split of the
// result (leading dimension ldcs).  Row strides must be multiples of 4
// elements and operand bases 16-byte aligned (gemm3_supported).
bool gemm3_supported(const void *p, int64_t ld);
// split_row0 / split_ncols restrict the split output to rows >= split_row0 and
// columns < split_ncols of C, written at row r - split_row0 (-1: all columns).
cudaError_t gemm3(int64_t M, int64_t N, int64_t K, float alpha, const float *Ahi, const float *Alo, int64_t lda,
                  const float *Bhi, const float *Blo, int64_t ldb, float beta, float *C, int64_t ldc, int tri,
                  float *Chi, float *Clo, int64_t ldcs, cudaStream_t s, int split_row0 = 0, int split_ncols = -1);
// C (M x N, row-major, ldc = N) = A B^T as gemm3, with K split into `slices`
// ranges computed by separate CTAs into `partials` (slices * M * N floats)
// and summed in a fixed order.  one_term: hi x hi only (TF32 accuracy, lo
// operands not read).
cudaError_t gemm3_splitk(int64_t M, int64_t N, int64_t K, const float *Ahi, const float *Alo, int64_t lda,
                         const float *Bhi, const float *Blo, int64_t ldb, float *C, float *partials, int slices,
                         cudaStream_t s, bool one_term = false);
// C[i] = sum over z < slices of partials[z * n + i] (fixed order).
cudaError_t sum_slices(const float *partials, int slices, int64_t n, float *C, cudaStream_t s);
// hi / lo TF32 split of the transpose of a rows x cols float32 matrix (cols x rows out).
cudaError_t split_transpose_tf32(const float *src, int64_t rows, int64_t cols, int64_t lds, float *hi, float *lo,
                                 int64_t ldd, cudaStream_t s);
// hi / lo TF32 split of a rows x cols float32 matrix (x = hi + lo exactly).
cudaError_t split_tf32(const float *src, int64_t rows, int64_t cols, int64_t lds, float *hi, float *lo, int64_t ldd,
                       cudaStream_t s);

// Hessian accumulation on the tensor cores (bf16 inputs, tcgen05 + TMA).
cudaError_t hessian_bf16_tc(float *H, int64_t cols, const __nv_bfloat16 *X, int64_t n, int64_t ldx,
                            cudaStream_t s);
bool hessian_bf16_tc_supported(int64_t cols, const void *X, int64_t ldx);
// Error bits recorded by bounded device-side waits since the last call (then
// cleared): the Hessian kernel's and the GEMM kernel's flags.  ~0u if the flag
// could not be read.
unsigned int read_and_clear_device_error();
unsigned int gemm_read_and_clear_error();
// Cycle budget of the bounded pipeline waits of the Hessian, GEMM and packed
// kernels (each source file holds its own copy), on the current device.
cudaError_t hessian_set_wait_budget(long long cycles);
cudaError_t gemm_set_wait_budget(long long cycles);
cudaError_t packed_set_wait_budget(long long cycles);

// Factor pieces.
// True when cholesky_lower_inplace can emit the sweep's block inverses.
inline bool factor_emits_uinv(int64_t cols, int block) { return block == 128 && cols % 128 == 0; }
cudaError_t factor_prepare(const float *H, int64_t cols, float damp, float *F, uint8_t *dead,
                           DeviceStatus *st, cudaStream_t s);
// scratch: cholesky_scratch_floats(cols) floats, 16-byte aligned; its first
// 128 x 128 floats hold the inverse of the last diagonal block on return.
size_t cholesky_scratch_floats(int64_t cols);
// Uinv (may be NULL): if non-NULL, block == 128 and cols % 128 == 0, receives the
// inverses of the diagonal blocks of F = J L J in sweep order (nblk x 128 x 128),
// (factor_emits_uinv tells when).
cudaError_t cholesky_lower_inplace(float *F, int64_t cols, DeviceStatus *st, float *scratch, cudaStream_t s,
                                   float *Uinv = nullptr, int block = 0);
cudaError_t factor_finalize(float *F, int64_t cols, cudaStream_t s);
size_t factor_scratch_bytes(int64_t cols);
// Clears `bit` of st->finite when any of the n values of X (float32 or bf16)
// is an Inf or NaN.
cudaError_t finite_check_launch(const void *X, bool bf16, int64_t n, DeviceStatus *st, unsigned int bit,
                                cudaStream_t s);

// Sweep pieces.
cudaError_t block_inverses(const float *F, int64_t cols, int block, float *Uinv, cudaStream_t s);
// VT[blk_b, rows above block b] = (F[..., blk_b] Uinv_b)^T for every block column
// b, written as its TF32 split (VThi, VTlo; cols x cols each, row-major).
cudaError_t premultiply_t(const float *F, int64_t cols, int block, const float *Uinv, float *VThi, float *VTlo,
                          cudaStream_t s);
// One block of the sweep, or with `pair` the two full 128-column blocks from
// c0 (Uinv_blk then points at the first of their two inverses) with the
// deferred update of the second by the first applied in the kernel, from V in
// VThi + VTlo.  On exit the blocks' columns of D hold the TF32 hi part of ΔW
// and those of DL the lo part.  `pair` needs sweep_pair_fits(rows): one CTA
// of 32 rows per SM.
cudaError_t sweep_block_launch(const void *W, bool w_bf16, int64_t rows, int64_t cols, int64_t c0,
                               int bw, const float *Uinv_blk, const float *F, const uint8_t *dead, int bits, int group,
                               float *D, float *DL, int32_t *qweight, float *scales, int32_t *qzeros,
                               uint8_t *codes, float *W_hat, float *row_err, const float *VThi, const float *VTlo,
                               bool pair, cudaStream_t s);
bool sweep_pair_fits(int64_t rows);

// Leading eigenpairs of a symmetric positive semi-definite G (subspace.cu).
constexpr int kSubspaceMaxK = 128;
struct SubspaceBufs {
    const float *G;               // cols x cols (SIMT path)
    const float *Ghi, *Glo;       // its TF32 split (tensor-core path)
    float *ZT, *ZT2;              // k x cols each
    float *Zhi, *Zlo;             // k x cols each (tensor-core path)
    float *Gm, *Wt;               // k x k each
    float *lam;                   // k
    float *part;                  // subspace_part_floats(k, cols, tc)
    float *Linv;                  // cholesky_scratch_floats(128)
    DeviceStatus *qst;            // status of the Cholesky-QR factorizations
    // Locked vectors (nl x cols, orthonormal rows) that every block is kept orthogonal
    // to, so that the iteration finds the next eigenpairs; nl = 0: none.
    const float *VL = nullptr;
    int nl = 0;
    float *Cp = nullptr;          // k x nl scratch of the projection
};
// k = min(2 r, 128, cols) vectors for r wanted eigenpairs.
int subspace_width(int64_t cols, int r);
// Floats of `part` that the projection against nl locked vectors needs (k-row blocks).
size_t subspace_projection_part_floats(int k, int nl);
size_t subspace_part_floats(int k, int64_t cols, bool tc);
// On return the rows of ZT are orthonormal, lam holds the k Ritz values in
// descending order and column i of Wt (k x k, row-major) the coefficients of
// Ritz vector i in those rows.
cudaError_t subspace_ritz(const SubspaceBufs &w, int k, int64_t cols, bool tc, cudaStream_t s);
// nvec vectors of length n, entry e of vector v at X[v * vs + e * es]: each
// negated unless its largest-magnitude entry (first on ties) is positive.
cudaError_t sign_normalize(float *X, int nvec, int64_t n, int64_t es, int64_t vs, cudaStream_t s);

// EoRA (eora.cu).  eora_run synchronizes `s` once, after the factorization of
// H, and reports a non-positive pivot through *bad_pivot_host (ULLONG_MAX = none,
// else the pivot index in reversed order) and non-finite H / dW through
// *finite_host (DeviceStatus::finite); nothing after that is launched then.
size_t eora_workspace_bytes(int64_t rows, int64_t cols, int r);
int eora_subspace_width(int64_t rows, int64_t cols, int r);
cudaError_t eora_run(const float *dW, int64_t rows, int64_t cols, const float *H, int r, float *A, float *B,
                     float *sigma, void *ws, cudaStream_t s, unsigned long long *bad_pivot_host,
                     unsigned int *finite_host);

// GPTQ-intrinsic LoRA (lora.cu).
size_t lora_basis_workspace_bytes(int64_t cols, int r);
// Lt (r x cols) = the r leading eigenvectors of H as rows; lam (may be NULL) their Ritz values.
cudaError_t lora_basis_run(const float *H, int64_t cols, int r, float *Lt, float *lam, void *ws, cudaStream_t s);
// dead[i] = (H_ii == 0); delta = damp * mean of the augmented diagonal (fix(H_ii), fix(C_ii)) into
// st->delta; C_ii <- fix(C_ii) + delta (C: r x r, ld r).
cudaError_t lora_damp_launch(const float *H, int64_t cols, float *C, int r, float damp, uint8_t *dead,
                             DeviceStatus *st, cudaStream_t s);
// S = H with diagonal fix(H_ii) + st->delta.
cudaError_t schur_init_launch(const float *H, int64_t cols, const DeviceStatus *st, float *S, cudaStream_t s);
// TF32 split of W - W_hat (dead inputs' weights taken as 0), rows x cols, ld cols.
cudaError_t dw_split_launch(const void *W, bool w_bf16, const float *W_hat, const uint8_t *dead, int64_t rows,
                            int64_t cols, float *hi, float *lo, cudaStream_t s);

// Packed quantized linear layer (packed_linear.cu): Y = X Ŵ^T (+ (X A^T) B^T when r > 0).
// Requirements checked by the caller (gq.h); ws holds packed_ws_bytes(...) bytes.
size_t packed_ws_bytes(int64_t n, int64_t rows, int64_t cols, int group, int r);
cudaError_t packed_forward(const __nv_bfloat16 *X, int64_t n, int64_t ldx, const int32_t *qweight,
                           const float *scales, const int32_t *qzeros, int64_t rows, int64_t cols, int bits,
                           int group, const float *A, const float *B, int r, float *Y, int64_t ldy, void *ws,
                           cudaStream_t s);
unsigned int packed_read_and_clear_error();
// Decode path for few tokens (n <= kPackedDecodeMaxTokens): SIMT product split over K
// into `slices` partial outputs (Ypart: slices x n x rows floats) and a fixed-order reduction.
constexpr int64_t kPackedDecodeMaxTokens = 32;
// The decode path holds a slice of X (16 tokens x whole groups) in 64 KB of shared memory.
inline bool packed_use_decode(int64_t n, int group) { return n <= kPackedDecodeMaxTokens && group <= 1024; }
void packed_gemv_split(int64_t rows, int64_t cols, int group, int64_t n, int *gps, int *slices);
cudaError_t packed_gemv_launch(const __nv_bfloat16 *X, int64_t n, int64_t ldx, const int32_t *qweight,
                               const float *scales, const int32_t *qzeros, int64_t rows, int64_t cols, int bits,
                               int group, const float *T, const float *B, int r, float *Ypart, float *Y, int64_t ldy,
                               cudaStream_t s);

// Bid-Up sweep (refine.cu): codes refined in place on their fixed grid against the target
// W - B A; W_hat written; qweight repacked when non-NULL; the number of moved codes added
// into *changed_out (device) when non-NULL.
size_t bidup_workspace_bytes(int64_t rows, int64_t cols);
cudaError_t bidup_run(const void *W, bool w_bf16, int64_t rows, int64_t cols, const float *H, const float *A,
                      const float *B, int r, int bits, int group, uint8_t *codes, const float *scales,
                      const int32_t *qzeros, float *W_hat, int32_t *qweight, unsigned long long *changed_out,
                      void *ws, cudaStream_t s);

// Round to nearest on the GPTQ grid per row and group (refine.cu).
cudaError_t rtn_launch(const float *M, int64_t nrows, int64_t ncols, int bits, int group, float *M_hat,
                       uint8_t *codes, float *scales, uint8_t *zeros, cudaStream_t s);

// dW = W - W_hat, n elements (W float32 or bf16).
cudaError_t weight_error_launch(const void *W, bool w_bf16, int64_t n, const float *W_hat, float *dW, cudaStream_t s);

// k[i] = rint(w[i] / s[i]) by the sweep's decision rule (quotient_rn).
cudaError_t code_decisions_launch(const float *w, const float *s, int64_t n, float *k, cudaStream_t st);

cudaError_t pack_launch(const uint8_t *codes, int64_t rows, int64_t cols, int bits, int32_t *qweight,
                        cudaStream_t s);
cudaError_t unpack_launch(const int32_t *qweight, int64_t rows, int64_t cols, int bits,
                          uint8_t *codes, cudaStream_t s);

}  // namespace gq
