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
//   2. blocked right-looking Cholesky of F in place, panel width 64: the
//      diagonal block is factored in shared memory by one CTA (which also
//      inverts it), the panel below is solved with that inverse, and the
//      trailing lower triangle is updated with the float32 SIMT GEMM;
//   3. finalize: F <- J L J in place (strictly-lower part zeroed).
#include <cfloat>

#include "common.cuh"

namespace gq {
namespace {

constexpr int NB = 64;

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

// Unblocked Cholesky of the kb x kb diagonal block at (k0, k0) in shared memory,
// followed by the inverse of the factor (written to Linv, kb x kb row-major).
__global__ void __launch_bounds__(256) potrf_diag_kernel(float *__restrict__ F, int64_t cols, int64_t k0,
                                                         int kb, float *__restrict__ Linv,
                                                         DeviceStatus *st) {
    __shared__ float A[NB][NB + 1];
    __shared__ float Y[NB][NB + 1];
    const int t = threadIdx.x;
    for (int idx = t; idx < NB * NB; idx += blockDim.x) {
        int i = idx / NB, j = idx % NB;
        A[i][j] = (i < kb && j <= i) ? F[(k0 + i) * cols + (k0 + j)] : 0.f;
    }
    __syncthreads();
    for (int j = 0; j < kb; ++j) {
        if (t == 0) {
            float d = A[j][j];
            if (!(d > 0.f)) {  // also catches NaN
                atomicMin(&st->bad_pivot, (unsigned long long)(k0 + j));
            }
            A[j][j] = sqrtf(d);
        }
        __syncthreads();
        const float l = A[j][j];
        for (int i = j + 1 + t; i < kb; i += blockDim.x) A[i][j] = A[i][j] / l;
        __syncthreads();
        const int m = kb - j - 1;  // trailing size
        for (int idx = t; idx < m * m; idx += blockDim.x) {
            int i = j + 1 + idx / m, k = j + 1 + idx % m;
            if (k <= i) A[i][k] = fmaf(-A[i][j], A[k][j], A[i][k]);
        }
        __syncthreads();
    }
    // Inverse of the lower factor, one column per thread (forward substitution).
    if (t < kb) {
        const int c = t;
        for (int i = 0; i < c; ++i) Y[i][c] = 0.f;
        Y[c][c] = 1.f / A[c][c];
        for (int i = c + 1; i < kb; ++i) {
            float acc = 0.f;
            for (int k = c; k < i; ++k) acc = fmaf(A[i][k], Y[k][c], acc);
            Y[i][c] = -acc / A[i][i];
        }
    }
    __syncthreads();
    for (int idx = t; idx < kb * kb; idx += blockDim.x) {
        int i = idx / kb, j = idx % kb;
        if (j <= i) F[(k0 + i) * cols + (k0 + j)] = A[i][j];
        Linv[i * NB + j] = (j <= i) ? Y[i][j] : 0.f;
    }
}

// Panel solve: rows r >= k0 + kb of columns [k0, k0 + kb): P <- P L^-T.
__global__ void __launch_bounds__(256) trsm_panel_kernel(float *__restrict__ F, int64_t cols, int64_t k0,
                                                         int kb, const float *__restrict__ Linv) {
    __shared__ float Li[NB][NB + 1];
    __shared__ float P[NB][NB + 1];
    const int t = threadIdx.x;
    const int64_t r0 = k0 + kb + (int64_t)blockIdx.x * NB;
    for (int idx = t; idx < NB * NB; idx += blockDim.x) {
        int i = idx / NB, j = idx % NB;
        Li[i][j] = (i < kb && j < kb) ? Linv[i * NB + j] : 0.f;
        int64_t r = r0 + i;
        P[i][j] = (r < cols && j < kb) ? F[r * cols + k0 + j] : 0.f;
    }
    __syncthreads();
    // X[r][c] = sum_{k <= c} P[r][k] * Linv[c][k]; thread -> row t/4, 16 columns.
    const int r = t / 4, cb = (t % 4) * 16;
    float out[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) out[c] = 0.f;
    for (int k = 0; k < kb; ++k) {
        const float pk = P[r][k];
#pragma unroll
        for (int c = 0; c < 16; ++c) out[c] = fmaf(pk, Li[cb + c][k], out[c]);
    }
    const int64_t gr = r0 + r;
    if (gr < cols) {
#pragma unroll
        for (int c = 0; c < 16; ++c)
            if (cb + c < kb) F[gr * cols + k0 + cb + c] = out[c];
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
    for (int64_t k0 = 0; k0 < cols; k0 += NB) {
        const int kb = (int)((cols - k0) < NB ? (cols - k0) : NB);
        potrf_diag_kernel<<<1, 256, 0, s>>>(F, cols, k0, kb, Linv, st);
        const int64_t k1 = k0 + kb;
        if (k1 < cols) {
            const int64_t rest = cols - k1;
            trsm_panel_kernel<<<(unsigned)((rest + NB - 1) / NB), 256, 0, s>>>(F, cols, k0, kb, Linv);
            cudaError_t e = sgemm<float>(rest, rest, kb, -1.f, F + k1 * cols + k0, cols, false,
                                         F + k1 * cols + k0, cols, true, 1.f, F + k1 * cols + k1, cols,
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
