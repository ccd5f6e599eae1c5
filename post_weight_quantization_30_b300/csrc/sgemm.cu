// Float32 SIMT GEMM used where float32 accuracy is required: the trailing
// update of the blocked Cholesky and the deferred trailing update of the GPTQ
// sweep.  (A tensor-float32 product would flip too many codes: see the sweep's
// precision notes.)  128 x 128 output tile per CTA, 256 threads, 8 x 8 outputs
// per thread, BK = 16, register-staged double buffering.  C may alias A when
// N <= 128 (one column tile): every CTA reads all of its A rows before it
// writes the same rows of C.
#include "common.cuh"

namespace gq {
namespace {

constexpr int BM = 128, BN = 128, BK = 16, NT = 256;

template <typename TA, bool TRANS>
__device__ __forceinline__ void load_tile(const TA *__restrict__ P, int64_t ld, int64_t r0, int64_t k0,
                                          int64_t R, int64_t K, float (&reg)[8]) {
    // Tile element (k, r), k in [0, BK), r in [0, 128): P(r0 + r, k0 + k).
    // TRANS: P(r, k) = P[k * ld + r] (r contiguous); else P[r * ld + k] (k contiguous).
    const int t = threadIdx.x;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        int idx = t + NT * i;
        int k, r;
        if (TRANS) {
            k = idx / 128;
            r = idx % 128;
        } else {
            r = idx / BK;
            k = idx % BK;
        }
        int64_t gr = r0 + r, gk = k0 + k;
        float v = 0.f;
        if (gr < R && gk < K) v = TRANS ? load_f32(P + gk * ld + gr) : load_f32(P + gr * ld + gk);
        reg[i] = v;
    }
}

template <bool TRANS>
__device__ __forceinline__ void store_tile(float (*S)[BM + 4], const float (&reg)[8]) {
    const int t = threadIdx.x;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        int idx = t + NT * i;
        int k, r;
        if (TRANS) {
            k = idx / 128;
            r = idx % 128;
        } else {
            r = idx / BK;
            k = idx % BK;
        }
        S[k][r] = reg[i];
    }
}

template <typename TA, bool AT, bool BT>
__global__ void __launch_bounds__(NT) sgemm_kernel(int64_t M, int64_t N, int64_t K, float alpha,
                                                   const TA *A, int64_t lda,
                                                   const TA *__restrict__ B, int64_t ldb, float beta,
                                                   float *C, int64_t ldc, int tri, int64_t kslice,
                                                   int64_t c_zstride) {
    const int64_t m0 = (int64_t)blockIdx.y * BM, n0 = (int64_t)blockIdx.x * BN;
    if (gridDim.z > 1) {
        // Split K: slice z covers k in [z * kslice, min(K, (z + 1) * kslice)) and
        // writes its own partial product at C + z * c_zstride.
        const int64_t kz = (int64_t)blockIdx.z * kslice;
        A += AT ? kz * lda : kz;
        B += BT ? kz : kz * ldb;
        K = (K - kz) < kslice ? (K - kz) : kslice;
        C += (int64_t)blockIdx.z * c_zstride;
    }
    if (tri == 1 && n0 > m0 + BM - 1) return;  // tile entirely above the diagonal
    if (tri == 2 && m0 > n0 + BN - 1) return;  // tile entirely below the diagonal

    __shared__ __align__(16) float As[2][BK][BM + 4];
    __shared__ __align__(16) float Bs[2][BK][BN + 4];

    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

    float ra[8], rb[8];
    // A(m, k): AT -> A[k*lda + m] (m contiguous) == "TRANS" in load_tile.
    load_tile<TA, AT>(A, lda, m0, 0, M, K, ra);
    // B(k, n): BT -> B[n*ldb + k] (k contiguous) == not TRANS; else n contiguous.
    load_tile<TA, !BT>(B, ldb, n0, 0, N, K, rb);
    store_tile<AT>(As[0], ra);
    store_tile<!BT>(Bs[0], rb);
    __syncthreads();

    int buf = 0;
    for (int64_t k0 = 0; k0 < K; k0 += BK) {
        const bool more = k0 + BK < K;
        if (more) {
            load_tile<TA, AT>(A, lda, m0, k0 + BK, M, K, ra);
            load_tile<TA, !BT>(B, ldb, n0, k0 + BK, N, K, rb);
        }
#pragma unroll
        for (int k = 0; k < BK; ++k) {
            float a[8], b[8];
            float4 a0 = *reinterpret_cast<const float4 *>(&As[buf][k][ty * 4]);
            float4 a1 = *reinterpret_cast<const float4 *>(&As[buf][k][64 + ty * 4]);
            float4 b0 = *reinterpret_cast<const float4 *>(&Bs[buf][k][tx * 4]);
            float4 b1 = *reinterpret_cast<const float4 *>(&Bs[buf][k][64 + tx * 4]);
            a[0] = a0.x; a[1] = a0.y; a[2] = a0.z; a[3] = a0.w;
            a[4] = a1.x; a[5] = a1.y; a[6] = a1.z; a[7] = a1.w;
            b[0] = b0.x; b[1] = b0.y; b[2] = b0.z; b[3] = b0.w;
            b[4] = b1.x; b[5] = b1.y; b[6] = b1.z; b[7] = b1.w;
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        if (more) {
            store_tile<AT>(As[buf ^ 1], ra);
            store_tile<!BT>(Bs[buf ^ 1], rb);
        }
        __syncthreads();
        buf ^= 1;
    }

#pragma unroll
    for (int i = 0; i < 8; ++i) {
        int64_t m = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
        if (m >= M) continue;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            int64_t n = n0 + (j < 4 ? tx * 4 + j : 64 + tx * 4 + (j - 4));
            if (n >= N) continue;
            float v = alpha * acc[i][j];
            float *p = C + m * ldc + n;
            *p = (beta == 0.f) ? v : fmaf(beta, *p, v);
            if (tri == 2 && m0 != n0 && n != m) {
                float *q = C + n * ldc + m;
                *q = (beta == 0.f) ? v : fmaf(beta, *q, v);
            }
        }
    }
}

}  // namespace

template <typename TA>
cudaError_t sgemm(int64_t M, int64_t N, int64_t K, float alpha, const TA *A, int64_t lda, bool a_t,
                  const TA *B, int64_t ldb, bool b_t, float beta, float *C, int64_t ldc, int tri,
                  cudaStream_t s) {
    if (M <= 0 || N <= 0) return cudaSuccess;
    dim3 grid((unsigned)((N + BN - 1) / BN), (unsigned)((M + BM - 1) / BM));
    if (a_t && b_t)
        sgemm_kernel<TA, true, true><<<grid, NT, 0, s>>>(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, tri, K, 0);
    else if (a_t)
        sgemm_kernel<TA, true, false><<<grid, NT, 0, s>>>(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, tri, K, 0);
    else if (b_t)
        sgemm_kernel<TA, false, true><<<grid, NT, 0, s>>>(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, tri, K, 0);
    else
        sgemm_kernel<TA, false, false><<<grid, NT, 0, s>>>(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, tri, K, 0);
    count_launch();
    return cudaGetLastError();
}

namespace {
__global__ void sum_slices_kernel(const float *__restrict__ P, int slices, int64_t n, float *__restrict__ C) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        float acc = 0.f;
        for (int z = 0; z < slices; ++z) acc += P[z * n + i];
        C[i] = acc;
    }
}
}  // namespace

cudaError_t sum_slices(const float *partials, int slices, int64_t n, float *C, cudaStream_t s) {
    sum_slices_kernel<<<(unsigned)((n + 255) / 256 < 1184 ? (n + 255) / 256 : 1184), 256, 0, s>>>(partials, slices, n, C);
    count_launch();
    return cudaGetLastError();
}

cudaError_t sgemm_splitk(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda, bool a_t, const float *B,
                         int64_t ldb, bool b_t, float *C, float *partials, int slices, cudaStream_t s) {
    if (M <= 0 || N <= 0) return cudaSuccess;
    const int64_t kslice = ((K + slices - 1) / slices + BK - 1) / BK * BK;
    const int z = (int)((K + kslice - 1) / kslice);
    dim3 grid((unsigned)((N + BN - 1) / BN), (unsigned)((M + BM - 1) / BM), (unsigned)(z < 1 ? 1 : z));
    const int64_t cz = M * N;
    if (a_t && b_t)
        sgemm_kernel<float, true, true><<<grid, NT, 0, s>>>(M, N, K, 1.f, A, lda, B, ldb, 0.f, partials, N, 0, kslice, cz);
    else if (a_t)
        sgemm_kernel<float, true, false><<<grid, NT, 0, s>>>(M, N, K, 1.f, A, lda, B, ldb, 0.f, partials, N, 0, kslice, cz);
    else if (b_t)
        sgemm_kernel<float, false, true><<<grid, NT, 0, s>>>(M, N, K, 1.f, A, lda, B, ldb, 0.f, partials, N, 0, kslice, cz);
    else
        sgemm_kernel<float, false, false><<<grid, NT, 0, s>>>(M, N, K, 1.f, A, lda, B, ldb, 0.f, partials, N, 0, kslice, cz);
    count_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t n = M * N;
    sum_slices_kernel<<<(unsigned)((n + 255) / 256 < 1184 ? (n + 255) / 256 : 1184), 256, 0, s>>>(partials, z < 1 ? 1 : z, n, C);
    count_launch();
    return cudaGetLastError();
}

template cudaError_t sgemm<float>(int64_t, int64_t, int64_t, float, const float *, int64_t, bool,
                                  const float *, int64_t, bool, float, float *, int64_t, int,
                                  cudaStream_t);
template cudaError_t sgemm<__nv_bfloat16>(int64_t, int64_t, int64_t, float, const __nv_bfloat16 *,
                                          int64_t, bool, const __nv_bfloat16 *, int64_t, bool, float,
                                          float *, int64_t, int, cudaStream_t);

}  // namespace gq
