// Factor of the damped Hessian: H_d = F F^T with F upper triangular.
//
// GPTQ drives its error compensation by the upper Cholesky factor U of H_d^-1
// ([GPTQ-wiki] "Enfoque Técnico": closed-form update from the inverse Hessian).
// With J the index reversal, J H_d J = L L^T (ordinary lower Cholesky) gives
// H_d = (J L J)(J L J)^T, so F = J L J is upper triangular and U = F^-1.  The
// sweep uses F and the inverses of its diagonal blocks only, so neither H_d^-1
// nor U is ever formed.
//
// Steps (all float32):
//   1. prepare: dead inputs (H_ii == 0 -> 1), damping delta = damp * mean(diag),
//      index reversal into F (lower triangle of J H_d J; the upper part zeroed);
//   2. blocked right-looking Cholesky of F in place, panel width 128: the
//      diagonal block is factored and inverted in shared memory by one CTA,
//      the panel below is multiplied by the transposed inverse, and the
//      trailing lower triangle is updated, both with the float32 SIMT GEMM;
//   3. finalize: F <- J L J in place (strictly-lower part zeroed).
#include "common.cuh"

namespace gq {
namespace {

constexpr int NB = 128;  // panel width

__global__ void diag_sum_kernel(const float *__restrict__ H, int64_t cols, float damp, DeviceStatus *st) {
    __shared__ double red[32];
    double acc = 0.0;
    for (int64_t i = threadIdx.x; i < cols; i += blockDim.x) {
        float d = H[i * cols + i];
        acc += (d == 0.f) ? 1.0 : (double)d;
    }
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x < 32) {
        acc = (threadIdx.x < blockDim.x / 32) ? red[threadIdx.x] : 0.0;
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (threadIdx.x == 0) {
            st->diag_sum = acc;
            st->delta = (float)((double)damp * (acc / (double)cols));
        }
    }
}

// F[p][q] = (J H_d J)[p][q] = H_d[C-1-p][C-1-q] for q <= p; 0 above the diagonal.
__global__ void reverse_damp_kernel(const float *__restrict__ H, int64_t cols, float *__restrict__ F,
                                    uint8_t *__restrict__ dead, const DeviceStatus *__restrict__ st) {
    const int64_t p = blockIdx.y;
    const float delta = st->delta;
    for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < cols; q += (int64_t)gridDim.x * blockDim.x) {
        float v = 0.f;
        if (q < p) {
            v = H[(cols - 1 - p) * cols + (cols - 1 - q)];
        } else if (q == p) {
            const int64_t i = cols - 1 - p;
            float d = H[i * cols + i];
            if (dead) dead[i] = (d == 0.f);
            v = ((d == 0.f) ? 1.f : d) + delta;
        }
        F[p * cols + q] = v;
    }
}

// Cholesky of the kb x kb diagonal block at (k0, k0) (kb <= NB) in shared
// memory, and the inverse of the factor (written to Linv, NB x NB row-major,
// zero above the diagonal).  Rows and columns from kb to NB are padded with
// the identity, which leaves the leading kb x kb part unchanged.
//
// The block is processed in four sub-panels of 32 columns.  For each:
//   1. warp 0 factors the 32 x 32 diagonal sub-block in registers (lane i
//      holds row i; the pivot row is broadcast by shuffles, so no CTA-wide
//      barrier is needed inside the 32 steps) and forms its inverse by
//      forward substitution (lane c holds column c of the inverse);
//   2. all warps solve the sub-panel below against it, X = A L_pp^-T, as a
//      product with the sub-block's inverse;
//   3. all warps update the trailing lower triangle, A -= X X^T, with 4 x 4
//      register tiles.
// Finally the off-diagonal 32 x 32 blocks of L^-1 are assembled block row by
// block row: Y_pq = -Y_pp sum_{q <= m < p} L_pm Y_mq.
constexpr int DIAG_THREADS = 256;
constexpr int SP = 32;           // sub-panel width
constexpr int LDA = NB + 4;      // shared-memory row stride (floats)
constexpr size_t DIAG_SMEM = (2 * NB * LDA + SP * LDA + 3 * SP * SP) * sizeof(float);

// Lane i holds row i of a 32 x 32 symmetric block (entries k <= i) and ends
// with row i of its lower Cholesky factor.  The pivot row is broadcast by
// shuffles, so the 32 elimination steps need no CTA-wide barrier.  The steps
// are unrolled by template recursion so that every index into `a` is a
// compile-time constant (the array stays in registers).
template <int J>
struct CholStep {
    static __device__ __forceinline__ void run(float (&a)[SP], int lane, int64_t gcol0, DeviceStatus *st) {
        const unsigned full = 0xffffffffu;
        const float d = __shfl_sync(full, a[J], J);
        if (lane == 0 && !(d > 0.f)) atomicMin(&st->bad_pivot, (unsigned long long)(gcol0 + J));
        const float l = sqrtf(d);
        const float r = 1.f / l;
        a[J] = (lane > J) ? a[J] * r : (lane == J ? l : a[J]);
#pragma unroll
        for (int k = J + 1; k < SP; ++k) {
            const float lkj = __shfl_sync(full, a[J], k);
            a[k] = (lane >= k) ? fmaf(-a[J], lkj, a[k]) : a[k];
        }
        CholStep<J + 1>::run(a, lane, gcol0, st);
    }
};
template <>
struct CholStep<SP> {
    static __device__ __forceinline__ void run(float (&)[SP], int, int64_t, DeviceStatus *) {}
};

__device__ __forceinline__ void warp_chol32(float (&a)[SP], int lane, int64_t gcol0, DeviceStatus *st) {
    CholStep<0>::run(a, lane, gcol0, st);
}

// Column `lane` of the inverse of the 32 x 32 lower factor stored at L (row
// stride LDA): y_i = (delta_i,lane - sum_{k<i} L_ik y_k) / L_ii.  L is read
// with shared-memory broadcasts; the result goes to Y (same stride).
__device__ __forceinline__ void warp_trinv32(const float *L, float *Y, int lane) {
    float y[SP];
#pragma unroll
    for (int i = 0; i < SP; ++i) {
        float s = (lane == i) ? 1.f : 0.f;
#pragma unroll
        for (int k = 0; k < i; ++k) s = fmaf(-L[i * LDA + k], y[k], s);
        y[i] = s / L[i * LDA + i];
        Y[i * LDA + lane] = y[i];
    }
}

__global__ void __launch_bounds__(DIAG_THREADS) potrf_diag_kernel(float *__restrict__ F, int64_t cols, int64_t k0,
                                                                  int kb, float *__restrict__ Linv,
                                                                  DeviceStatus *st) {
    extern __shared__ __align__(16) float sm[];
    float *A = sm;                 // [NB][LDA]: the block, lower triangle, becomes L
    float *Y = A + NB * LDA;       // [NB][LDA]: L^-1, lower triangle
    float *XT = Y + NB * LDA;      // [SP][LDA]: solved sub-panel, transposed (XT[k][i] = X_ik)
    float *T = XT + SP * LDA;      // [3][SP][SP]: partial sums of the inverse assembly
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;

    for (int idx = t; idx < NB * NB; idx += DIAG_THREADS) {
        const int i = idx / NB, j = idx % NB;
        float v;
        if (i < kb && j < kb) v = (j <= i) ? F[(k0 + i) * cols + (k0 + j)] : 0.f;
        else v = (i == j) ? 1.f : 0.f;
        A[i * LDA + j] = v;
        Y[i * LDA + j] = 0.f;
    }
    __syncthreads();

    for (int c0 = 0; c0 < NB; c0 += SP) {
        if (warp == 0) {
            float a[SP];
#pragma unroll
            for (int k = 0; k < SP; ++k) a[k] = (k <= lane) ? A[(c0 + lane) * LDA + c0 + k] : 0.f;
            warp_chol32(a, lane, k0 + c0, st);
#pragma unroll
            for (int k = 0; k < SP; ++k)
                if (k <= lane) A[(c0 + lane) * LDA + c0 + k] = a[k];
            __syncwarp();
            warp_trinv32(A + c0 * LDA + c0, Y + c0 * LDA + c0, lane);
        }
        __syncthreads();
        const int r0 = c0 + SP, R = NB - r0;  // rows below the diagonal sub-block
        if (R == 0) break;
        // X_ic = sum_{k <= c} A_ik Y_ck; TPR threads per row, interleaved columns.
        const int tpr = DIAG_THREADS / R >= 8 ? 8 : (DIAG_THREADS / R >= 4 ? 4 : 2);
        const int row = t / tpr, sub = t % tpr;
        float xo[SP / 2];
        if (row < R) {
            float ar[SP];
            const float *ap = A + (r0 + row) * LDA + c0;
#pragma unroll
            for (int k = 0; k < SP; k += 4) {
                const float4 v = *reinterpret_cast<const float4 *>(ap + k);
                ar[k] = v.x; ar[k + 1] = v.y; ar[k + 2] = v.z; ar[k + 3] = v.w;
            }
#pragma unroll
            for (int q = 0; q < SP / 2; ++q) {
                const int c = sub + q * tpr;
                float acc = 0.f;
                if (c < SP) {
                    const float *yp = Y + (c0 + c) * LDA + c0;
#pragma unroll
                    for (int k = 0; k < SP; ++k)
                        if (k <= c) acc = fmaf(ar[k], yp[k], acc);
                }
                xo[q] = acc;
            }
        }
        __syncthreads();
        if (row < R) {
#pragma unroll
            for (int q = 0; q < SP / 2; ++q) {
                const int c = sub + q * tpr;
                if (c < SP) {
                    A[(r0 + row) * LDA + c0 + c] = xo[q];
                    XT[c * LDA + r0 + row] = xo[q];
                }
            }
        }
        __syncthreads();
        // A_ij -= sum_k X_ik X_jk for r0 <= j <= i < NB, in 4 x 4 tiles.
        const int nt = R / 4, ntiles = nt * (nt + 1) / 2;
        for (int tile = t; tile < ntiles; tile += DIAG_THREADS) {
            int ti = (int)((sqrtf(8.f * (float)tile + 1.f) - 1.f) * 0.5f);
            while ((ti + 1) * (ti + 2) / 2 <= tile) ++ti;
            while (ti * (ti + 1) / 2 > tile) --ti;
            const int tj = tile - ti * (ti + 1) / 2;
            const int i0 = r0 + 4 * ti, j0 = r0 + 4 * tj;
            float acc[4][4] = {};
#pragma unroll 8
            for (int k = 0; k < SP; ++k) {
                const float4 xi = *reinterpret_cast<const float4 *>(XT + k * LDA + i0);
                const float4 xj = *reinterpret_cast<const float4 *>(XT + k * LDA + j0);
                const float vi[4] = {xi.x, xi.y, xi.z, xi.w}, vj[4] = {xj.x, xj.y, xj.z, xj.w};
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(vi[a], vj[b], acc[a][b]);
            }
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 4; ++b)
                    if (j0 + b <= i0 + a) A[(i0 + a) * LDA + j0 + b] -= acc[a][b];
        }
        __syncthreads();
    }

    // Off-diagonal blocks of Y = L^-1, one block row p at a time.
    for (int p = 1; p < NB / SP; ++p) {
        // T_q = sum_{m=q}^{p-1} L_pm Y_mq for q < p.
        for (int idx = t; idx < p * SP * SP; idx += DIAG_THREADS) {
            const int q = idx / (SP * SP), i = (idx / SP) % SP, c = idx % SP;
            const float *lp = A + (p * SP + i) * LDA;
            float acc = 0.f;
            for (int k = q * SP; k < p * SP; ++k) acc = fmaf(lp[k], Y[k * LDA + q * SP + c], acc);
            T[idx] = acc;
        }
        __syncthreads();
        // Y_pq = -Y_pp T_q.
        for (int idx = t; idx < p * SP * SP; idx += DIAG_THREADS) {
            const int q = idx / (SP * SP), i = (idx / SP) % SP, c = idx % SP;
            const float *yp = Y + (p * SP + i) * LDA + p * SP;
            const float *tq = T + q * SP * SP;
            float acc = 0.f;
            for (int k = 0; k <= i; ++k) acc = fmaf(yp[k], tq[k * SP + c], acc);
            Y[(p * SP + i) * LDA + q * SP + c] = -acc;
        }
        __syncthreads();
    }

    for (int idx = t; idx < NB * NB; idx += DIAG_THREADS) {
        const int i = idx / NB, j = idx % NB;
        const bool in = i < kb && j <= i;
        if (in) F[(k0 + i) * cols + (k0 + j)] = A[i * LDA + j];
        Linv[idx] = in ? Y[i * LDA + j] : 0.f;
    }
}

// F <- J F J restricted to the lower triangle -> upper triangle; lower zeroed.
__global__ void finalize_kernel(float *__restrict__ F, int64_t cols) {
    const int64_t p = blockIdx.y;
    for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q <= p; q += (int64_t)gridDim.x * blockDim.x) {
        if (q == p) {
            const int64_t p2 = cols - 1 - p;
            if (p < p2) {
                float a = F[p * cols + p], b = F[p2 * cols + p2];
                F[p * cols + p] = b;
                F[p2 * cols + p2] = a;
            }
        } else {
            const float v = F[p * cols + q];
            F[(cols - 1 - p) * cols + (cols - 1 - q)] = v;
            F[p * cols + q] = 0.f;
        }
    }
}

}  // namespace

cudaError_t factor_prepare(const float *H, int64_t cols, float damp, float *F, uint8_t *dead,
                           DeviceStatus *st, cudaStream_t s) {
    diag_sum_kernel<<<1, 1024, 0, s>>>(H, cols, damp, st);
    dim3 grid((unsigned)((cols + 255) / 256 < 8 ? (cols + 255) / 256 : 8), (unsigned)cols);
    reverse_damp_kernel<<<grid, 256, 0, s>>>(H, cols, F, dead, st);
    return cudaGetLastError();
}

cudaError_t cholesky_lower_inplace(float *F, int64_t cols, DeviceStatus *st, float *Linv, cudaStream_t s) {
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(potrf_diag_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)DIAG_SMEM);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    for (int64_t k0 = 0; k0 < cols; k0 += NB) {
        const int kb = (int)((cols - k0) < NB ? (cols - k0) : NB);
        potrf_diag_kernel<<<1, DIAG_THREADS, DIAG_SMEM, s>>>(F, cols, k0, kb, Linv, st);
        const int64_t k1 = k0 + kb;
        if (k1 < cols) {
            const int64_t rest = cols - k1;
            float *P = F + k1 * cols + k0;  // rest x kb panel below the diagonal block
            // P <- P L^-T in place: each 128-row tile reads its rows completely before writing them.
            cudaError_t e = sgemm<float>(rest, kb, kb, 1.f, P, cols, false, Linv, NB, true, 0.f, P, cols, 0, s);
            if (e != cudaSuccess) return e;
            e = sgemm<float>(rest, rest, kb, -1.f, P, cols, false, P, cols, true, 1.f, F + k1 * cols + k1, cols,
                             /*tri=*/1, s);
            if (e != cudaSuccess) return e;
        }
    }
    return cudaGetLastError();
}

cudaError_t factor_finalize(float *F, int64_t cols, cudaStream_t s) {
    dim3 grid((unsigned)((cols + 255) / 256 < 8 ? (cols + 255) / 256 : 8), (unsigned)cols);
    finalize_kernel<<<grid, 256, 0, s>>>(F, cols);
    return cudaGetLastError();
}

size_t factor_scratch_bytes() { return align_up(sizeof(DeviceStatus)) + align_up(NB * NB * sizeof(float)); }

}  // namespace gq
