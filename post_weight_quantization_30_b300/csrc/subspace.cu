// Leading eigenpairs of a symmetric positive semi-definite matrix G (cols x
// cols): block subspace iteration, then Rayleigh-Ritz.  Used for the EoRA
// adapter (G = M^T M) and for the GPTQ-intrinsic LoRA basis (G = H, whose
// leading eigenvectors are the leading right singular vectors of X).
//
//   ZT  <- k x cols starting block (a fixed counter hash)
//   twice: ZT <- orth(ZT)                     shifted Cholesky-QR
//   ITERS times: ZT <- orth(ZT G)             one Cholesky-QR pass each
//   ZT  <- orth(ZT)                           once more before Rayleigh-Ritz
//   T = ZT G ZT^T (k x k), T = W diag(lam) W^T by cyclic Jacobi
//
// The Ritz vectors are the rows of W^T ZT; callers take the first r of them.
// On the tensor-core path the products with G run as 3xTF32 GEMMs from the
// split of G the caller provides.
#include <climits>

#include "common.cuh"

namespace gq {
namespace {

constexpr int ITERS = 30;   // subspace iterations
constexpr int SPLITK = 64;  // K slices of the thin Gram products
constexpr int ZSPLIT = 4;   // K slices of the block products on the tensor cores

// Starting block: k x cols values in [-1, 1) from a counter hash of (i, j).
__global__ void init_block_kernel(float *__restrict__ ZT, int k, int64_t cols) {
    const int64_t n = (int64_t)k * cols;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < n; idx += (int64_t)gridDim.x * blockDim.x) {
        uint64_t x = (uint64_t)idx * 0x9E3779B97F4A7C15ull + 0x632BE59BD9B4E019ull;
        x ^= x >> 30;
        x *= 0xBF58476D1CE4E5B9ull;
        x ^= x >> 27;
        x *= 0x94D049BB133111EBull;
        x ^= x >> 31;
        ZT[idx] = (float)(x >> 40) * (1.f / 8388608.f) - 1.f;
    }
}

// Each row of ZT (k x cols) scaled to unit norm (a zero row stays zero).  One
// CTA per row.  After this the Gram matrix of the block has a unit diagonal,
// so a fixed diagonal shift is relative to it whatever the spread of the
// eigenvalues the block was just multiplied by.
__global__ void normalize_rows_kernel(float *__restrict__ ZT, int64_t cols) {
    float *row = ZT + (int64_t)blockIdx.x * cols;
    __shared__ float red[32];
    float acc = 0.f;
    for (int64_t j = threadIdx.x; j < cols; j += blockDim.x) acc = fmaf(row[j], row[j], acc);
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x < 32) {
        acc = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (threadIdx.x == 0) red[0] = acc > 0.f ? 1.f / sqrtf(acc) : 0.f;
    }
    __syncthreads();
    const float sc = red[0];
    for (int64_t j = threadIdx.x; j < cols; j += blockDim.x) row[j] *= sc;
}

// Shift of the unit-diagonal Gram matrix, so that the Cholesky factorization of
// a (numerically) rank-deficient block still succeeds.
__global__ void shift_gram_kernel(float *__restrict__ Gm, int k) {
    for (int i = threadIdx.x; i < k; i += blockDim.x) Gm[i * k + i] += 1e-6f;
}

// Eigen-decomposition of the symmetric k x k matrix T (k <= 128) by the
// cyclic Jacobi method in one CTA, parallel over the k/2 disjoint (p, q) pairs
// of a round-robin ordering.  Outputs the eigenvalues in descending order and
// the matching eigenvectors as the columns of W (row-major k x k).
constexpr int JT = 512;
constexpr int JLD = kSubspaceMaxK + 1;
constexpr size_t JACOBI_SMEM = (2 * kSubspaceMaxK * JLD + 2 * (kSubspaceMaxK / 2 + 1)) * sizeof(float) +
                               (kSubspaceMaxK + 2 + 2 * (kSubspaceMaxK / 2 + 1)) * sizeof(int);

__global__ void __launch_bounds__(JT) jacobi_eig_kernel(const float *__restrict__ Tin, int k, float *__restrict__ lam,
                                                        float *__restrict__ W) {
    extern __shared__ __align__(16) float js[];
    float *T = js;                        // [k][JLD]
    float *V = T + kSubspaceMaxK * JLD;      // [k][JLD]
    float *cs = V + kSubspaceMaxK * JLD;     // [npairs] cosines
    float *sn = cs + kSubspaceMaxK / 2 + 1;  // [npairs] sines
    int *pos = (int *)(sn + kSubspaceMaxK / 2 + 1);  // [kk] round-robin positions
    int *pp = pos + kSubspaceMaxK + 2;       // [npairs]
    int *pq = pp + kSubspaceMaxK / 2 + 1;    // [npairs]
    __shared__ int rotated;
    const int t = threadIdx.x;
    const int kk = (k + 1) & ~1;  // even, with a dummy index k when k is odd
    const int np = kk / 2;

    for (int idx = t; idx < k * k; idx += JT) {
        const int i = idx / k, j = idx % k;
        T[i * JLD + j] = 0.5f * (Tin[i * k + j] + Tin[j * k + i]);
        V[i * JLD + j] = (i == j) ? 1.f : 0.f;
    }
    for (int i = t; i < kk; i += JT) pos[i] = i;
    for (int i = t; i < np; i += JT) sn[i] = 0.f;
    __shared__ float tol;
    __syncthreads();
    if (t == 0) {
        // Off-diagonal entries below 1e-7 of the largest diagonal entry are at the
        // float32 rounding level of T: they move no eigenvalue by more than that.
        float m = 0.f;
        for (int i = 0; i < k; ++i) m = fmaxf(m, fabsf(T[i * JLD + i]));
        tol = 1e-7f * m;
    }
    __syncthreads();

    for (int sweep = 0; sweep < 15; ++sweep) {
        if (t == 0) rotated = 0;
        __syncthreads();
        for (int round = 0; round < kk - 1; ++round) {
            if (t < np) {
                // The element the previous rotation of this slot annihilated is
                // set to exactly zero (it holds rounding residue only).
                if (round > 0 && sn[t] != 0.f) {
                    T[pp[t] * JLD + pq[t]] = 0.f;
                    T[pq[t] * JLD + pp[t]] = 0.f;
                }
                int p = pos[t], q = pos[kk - 1 - t];
                if (p > q) { const int x = p; p = q; q = x; }
                float c = 1.f, s = 0.f;
                if (q < k) {
                    const float apq = T[p * JLD + q];
                    const float app = T[p * JLD + p], aqq = T[q * JLD + q];
                    // Rotate unless a_pq is at the rounding level of T.
                    if (fabsf(apq) > tol) {
                        const float tau = (aqq - app) / (2.f * apq);
                        const float tt = (tau >= 0.f ? 1.f : -1.f) / (fabsf(tau) + sqrtf(1.f + tau * tau));
                        c = 1.f / sqrtf(1.f + tt * tt);
                        s = tt * c;
                        rotated = 1;
                    }
                }
                pp[t] = p;
                pq[t] = q;
                cs[t] = c;
                sn[t] = s;
            }
            __syncthreads();
            // Rows p, q of T  <- J^T T.
            for (int idx = t; idx < np * k; idx += JT) {
                const int pr = idx / k, j = idx % k;
                const int p = pp[pr], q = pq[pr];
                if (q >= k || sn[pr] == 0.f) continue;
                const float c = cs[pr], s = sn[pr];
                const float a = T[p * JLD + j], b = T[q * JLD + j];
                T[p * JLD + j] = c * a - s * b;
                T[q * JLD + j] = s * a + c * b;
            }
            __syncthreads();
            // Columns p, q of T and V  <- T J, V J.
            for (int idx = t; idx < np * k; idx += JT) {
                const int pr = idx / k, j = idx % k;
                const int p = pp[pr], q = pq[pr];
                if (q >= k || sn[pr] == 0.f) continue;
                const float c = cs[pr], s = sn[pr];
                const float a = T[j * JLD + p], b = T[j * JLD + q];
                T[j * JLD + p] = c * a - s * b;
                T[j * JLD + q] = s * a + c * b;
                const float va = V[j * JLD + p], vb = V[j * JLD + q];
                V[j * JLD + p] = c * va - s * vb;
                V[j * JLD + q] = s * va + c * vb;
            }
            __syncthreads();
            // Next round-robin arrangement: position 0 fixed, the others rotate.
            if (t == 0) {
                const int last = pos[kk - 1];
                for (int i = kk - 1; i > 1; --i) pos[i] = pos[i - 1];
                pos[1] = last;
            }
            __syncthreads();
        }
        if (t < np && sn[t] != 0.f) {
            T[pp[t] * JLD + pq[t]] = 0.f;
            T[pq[t] * JLD + pp[t]] = 0.f;
            sn[t] = 0.f;
        }
        __syncthreads();
        if (!rotated) break;
        __syncthreads();
    }
    // Sort by descending eigenvalue (ties by index).
    int *order = pos;
    __syncthreads();
    for (int i = t; i < k; i += JT) {
        const float li = T[i * JLD + i];
        int rank = 0;
        for (int j = 0; j < k; ++j) {
            const float lj = T[j * JLD + j];
            rank += (lj > li) || (lj == li && j < i);
        }
        order[rank] = i;
    }
    __syncthreads();
    for (int i = t; i < k; i += JT) lam[i] = T[order[i] * JLD + order[i]];
    for (int idx = t; idx < k * k; idx += JT) {
        const int row = idx / k, col = idx % k;
        W[idx] = V[row * JLD + order[col]];
    }
}
// Sign of each of nvec vectors of length n (entry e of vector v at
// X[v * vs + e * es]): the entry of largest magnitude (first on ties) is made
// positive; the vector is negated otherwise.  One CTA per vector.
__global__ void sign_normalize_kernel(float *__restrict__ X, int64_t n, int64_t es, int64_t vs) {
    float *x = X + (int64_t)blockIdx.x * vs;
    __shared__ float bv[32];
    __shared__ long long bi[32];
    __shared__ float flip;
    float best = -1.f;
    long long bidx = LLONG_MAX;
    for (int64_t m = threadIdx.x; m < n; m += blockDim.x) {
        const float v = fabsf(x[m * es]);
        if (v > best) {
            best = v;
            bidx = m;
        }
    }
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, best, o);
        const long long oi = __shfl_xor_sync(0xffffffffu, bidx, o);
        if (ov > best || (ov == best && oi < bidx)) {
            best = ov;
            bidx = oi;
        }
    }
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    if (l == 0) {
        bv[w] = best;
        bi[w] = bidx;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float b = -1.f;
        long long id = LLONG_MAX;
        for (int i = 0; i < (int)(blockDim.x >> 5); ++i)
            if (bv[i] > b || (bv[i] == b && bi[i] < id)) {
                b = bv[i];
                id = bi[i];
            }
        flip = (id != LLONG_MAX && x[id * es] < 0.f) ? -1.f : 1.f;
    }
    __syncthreads();
    if (flip < 0.f)
        for (int64_t m = threadIdx.x; m < n; m += blockDim.x) x[m * es] = -x[m * es];
}

unsigned grid1d(int64_t n) {
    const int64_t g = (n + 255) / 256;
    return (unsigned)(g < 1 ? 1 : (g > 148 * 8 ? 148 * 8 : g));
}

// One pass of shifted Cholesky-QR on the rows of src (k x cols): rows scaled
// to unit norm, src src^T + shift = L L^T, dst = L^-1 src.  src is scaled in place.
cudaError_t cholqr_pass(const SubspaceBufs &w, float *src, float *dst, int k, int64_t cols, cudaStream_t s) {
    normalize_rows_kernel<<<k, 256, 0, s>>>(src, cols);
    count_launch();
    cudaError_t e = sgemm_splitk(k, k, cols, src, cols, false, src, cols, true, w.Gm, w.part, SPLITK, s);
    if (e != cudaSuccess) return e;
    shift_gram_kernel<<<1, 128, 0, s>>>(w.Gm, k);
    count_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = cholesky_lower_inplace(w.Gm, k, w.qst, w.Linv, s)) != cudaSuccess) return e;
    return sgemm<float>(k, cols, k, 1.f, w.Linv, 128, false, src, cols, false, 0.f, dst, cols, 0, s);
}

// Y = the block ZT (k x cols) times the symmetric G.
cudaError_t block_times_g(const SubspaceBufs &w, const float *ZT, float *Y, int k, int64_t cols, bool tc,
                          cudaStream_t s) {
    if (!tc) return sgemm<float>(k, cols, cols, 1.f, ZT, cols, false, w.G, cols, false, 0.f, Y, cols, 0, s);
    cudaError_t e = split_tf32(ZT, k, cols, cols, w.Zhi, w.Zlo, cols, s);
    if (e != cudaSuccess) return e;
    return gemm3_splitk(k, cols, cols, w.Zhi, w.Zlo, cols, w.Ghi, w.Glo, cols, Y, w.part, ZSPLIT, s);
}

}  // namespace

int subspace_width(int64_t cols, int r) {
    int64_t k = 2 * (int64_t)r;
    if (k > kSubspaceMaxK) k = kSubspaceMaxK;
    if (k > cols) k = cols;
    return (int)k;
}

size_t subspace_part_floats(int k, int64_t cols, bool tc) {
    size_t part = (size_t)SPLITK * k * k;
    if (tc && (size_t)ZSPLIT * k * cols > part) part = (size_t)ZSPLIT * k * cols;
    return part;
}

cudaError_t subspace_ritz(const SubspaceBufs &w, int k, int64_t cols, bool tc, cudaStream_t s) {
    cudaError_t e;
    init_block_kernel<<<grid1d((int64_t)k * cols), 256, 0, s>>>(w.ZT2, k, cols);
    count_launch();
    if ((e = cholqr_pass(w, w.ZT2, w.ZT, k, cols, s)) != cudaSuccess) return e;
    if ((e = cholqr_pass(w, w.ZT, w.ZT2, k, cols, s)) != cudaSuccess) return e;
    if ((e = cudaMemcpyAsync(w.ZT, w.ZT2, (size_t)k * cols * sizeof(float), cudaMemcpyDeviceToDevice, s)) != cudaSuccess)
        return e;
    for (int it = 0; it < ITERS; ++it) {
        if ((e = block_times_g(w, w.ZT, w.ZT2, k, cols, tc, s)) != cudaSuccess) return e;
        if ((e = cholqr_pass(w, w.ZT2, w.ZT, k, cols, s)) != cudaSuccess) return e;
    }
    if ((e = cholqr_pass(w, w.ZT, w.ZT2, k, cols, s)) != cudaSuccess) return e;
    if ((e = cudaMemcpyAsync(w.ZT, w.ZT2, (size_t)k * cols * sizeof(float), cudaMemcpyDeviceToDevice, s)) != cudaSuccess)
        return e;

    // Rayleigh-Ritz: T = Z^T G Z (k x k), eigenpairs by Jacobi.
    if ((e = block_times_g(w, w.ZT, w.ZT2, k, cols, tc, s)) != cudaSuccess) return e;
    if ((e = sgemm_splitk(k, k, cols, w.ZT2, cols, false, w.ZT, cols, true, w.Gm, w.part, SPLITK, s)) != cudaSuccess)
        return e;
    static bool attr_set = false;
    if (!attr_set) {
        if ((e = cudaFuncSetAttribute(jacobi_eig_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)JACOBI_SMEM)) != cudaSuccess)
            return e;
        attr_set = true;
    }
    jacobi_eig_kernel<<<1, JT, JACOBI_SMEM, s>>>(w.Gm, k, w.lam, w.Wt);
    count_launch();
    return cudaGetLastError();
}

cudaError_t sign_normalize(float *X, int nvec, int64_t n, int64_t es, int64_t vs, cudaStream_t s) {
    if (nvec <= 0 || n <= 0) return cudaSuccess;
    sign_normalize_kernel<<<nvec, 256, 0, s>>>(X, n, es, vs);
    count_launch();
    return cudaGetLastError();
}

}  // namespace gq
