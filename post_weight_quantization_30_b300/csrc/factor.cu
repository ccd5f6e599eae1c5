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
// memory, followed by the inverse of the factor (written to Linv, NB x NB
// row-major, zero above the diagonal).  Each thread owns a fixed set of
// lower-triangle elements.  Elimination step j subtracts a_ij a_kj / a_jj from
// every a_ik with j < k <= i, using column j as left by the earlier steps
// (unscaled), so a step needs one barrier; the factor is a_ij / sqrt(a_jj)
// afterwards.  The inverse is built the same way (right-looking, one barrier
// per step): R_ic -= (L_ik / L_kk) R_kc, then Y_ic = R_ic / L_ii.
constexpr int DIAG_THREADS = 512;
constexpr int TRI = NB * (NB + 1) / 2;
constexpr int DIAG_OWN = (TRI + DIAG_THREADS - 1) / DIAG_THREADS;
constexpr size_t DIAG_SMEM = 2 * NB * (NB + 1) * sizeof(float);

__global__ void __launch_bounds__(DIAG_THREADS) potrf_diag_kernel(float *__restrict__ F, int64_t cols, int64_t k0,
                                                                  int kb, float *__restrict__ Linv,
                                                                  DeviceStatus *st) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    float(*A)[NB + 1] = reinterpret_cast<float(*)[NB + 1]>(smem_raw);
    float(*Y)[NB + 1] = A + NB;
    const int t = threadIdx.x;
    int own[DIAG_OWN];
#pragma unroll
    for (int q = 0; q < DIAG_OWN; ++q) {
        const int e = t + q * DIAG_THREADS;
        int i = (int)((sqrtf(8.f * (float)e + 1.f) - 1.f) * 0.5f);
        while ((i + 1) * (i + 2) / 2 <= e) ++i;
        while (i * (i + 1) / 2 > e) --i;
        const int k = e - i * (i + 1) / 2;
        own[q] = (e < TRI && i < kb) ? ((i << 16) | k) : -1;
    }
    for (int idx = t; idx < NB * NB; idx += DIAG_THREADS) {
        const int i = idx / NB, j = idx % NB;
        A[i][j] = (i < kb && j <= i) ? F[(k0 + i) * cols + (k0 + j)] : 0.f;
    }
    __syncthreads();
    for (int j = 0; j < kb; ++j) {
        const float d = A[j][j];
        if (t == 0 && !(d > 0.f)) atomicMin(&st->bad_pivot, (unsigned long long)(k0 + j));
        const float rd = 1.f / d;
#pragma unroll
        for (int q = 0; q < DIAG_OWN; ++q) {
            if (own[q] < 0) continue;
            const int i = own[q] >> 16, k = own[q] & 0xffff;
            if (k > j) A[i][k] = fmaf(-A[i][j] * rd, A[k][j], A[i][k]);
        }
        __syncthreads();
    }
    // Scale to the Cholesky factor (L_ij = a_ij / sqrt(a_jj)); then Y starts as I.
#pragma unroll
    for (int q = 0; q < DIAG_OWN; ++q) {
        if (own[q] < 0) continue;
        const int i = own[q] >> 16, k = own[q] & 0xffff;
        const float l = sqrtf(A[k][k]);
        Y[i][k] = (i == k) ? l : A[i][k] / l;
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < DIAG_OWN; ++q) {
        if (own[q] < 0) continue;
        const int i = own[q] >> 16, k = own[q] & 0xffff;
        A[i][k] = Y[i][k];
        Y[i][k] = (i == k) ? 1.f : 0.f;
    }
    __syncthreads();
    for (int k = 0; k < kb; ++k) {
        const float rl = 1.f / A[k][k];
#pragma unroll
        for (int q = 0; q < DIAG_OWN; ++q) {
            if (own[q] < 0) continue;
            const int i = own[q] >> 16, c = own[q] & 0xffff;
            if (i > k && c <= k) Y[i][c] = fmaf(-A[i][k] * rl, Y[k][c], Y[i][c]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int q = 0; q < DIAG_OWN; ++q) {
        if (own[q] < 0) continue;
        const int i = own[q] >> 16, c = own[q] & 0xffff;
        Y[i][c] = Y[i][c] / A[i][i];
    }
    __syncthreads();
    for (int idx = t; idx < NB * NB; idx += DIAG_THREADS) {
        const int i = idx / NB, j = idx % NB;
        if (i < kb && j <= i) F[(k0 + i) * cols + (k0 + j)] = A[i][j];
        Linv[idx] = (i < kb && j <= i) ? Y[i][j] : 0.f;
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
