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
// With locked vectors VL (nl x cols, orthonormal) every block is projected
// onto their orthogonal complement after each product with G, so the
// iteration converges to the leading eigenpairs of (I - VL^T VL) G (I - VL^T VL):
// the next ones of G once VL spans leading eigenvectors.
// On the tensor-core path the products with G run on the tensor cores from the
// split of G the caller provides: one TF32 product per iteration, 3xTF32
// (float32 accuracy) for the last three iterations and the Rayleigh-Ritz step.
#include <climits>

#include "common.cuh"

namespace gq {
namespace {

constexpr int ITERS = 30;        // subspace iterations
constexpr int ACCURATE_TAIL = 3; // of which the last ones multiply with float32 accuracy
constexpr int SPLITK = 64;  // K slices of the thin Gram products
constexpr int ZSPLIT_MAX = 8;  // K slices of the block products on the tensor cores, at most

// K slices for a block product with ceil(cols / 128) x ceil(k / 128) output
// tiles: as many as keep every CTA in one wave on the 148 SMs (one CTA per SM).
int zsplit(int64_t cols, int k) {
    const int64_t tiles = ((cols + 127) / 128) * ((k + 127) / 128);
    int64_t z = 148 / tiles;
    if (z < 1) z = 1;
    if (z > ZSPLIT_MAX) z = ZSPLIT_MAX;
    return (int)z;
}

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
// cyclic Jacobi method in one CTA.  Each round applies the k/2 disjoint plane
// rotations of a round-robin pairing at once, T <- J^T T J, as independent
// 2 x 2 blocks J_i^T T[{p_i, q_i}, {p_j, q_j}] J_j over pairs of pairs (blocks
// i <= j, mirrored), so a round costs two barriers.  Outputs the eigenvalues in
// descending order and the matching eigenvectors as the columns of W
// (row-major k x k).
constexpr int JT = 1024;
constexpr int JNP = kSubspaceMaxK / 2;  // rotations per round, at most
constexpr int JLD = kSubspaceMaxK + 1;
constexpr int JNB = JNP * (JNP + 1) / 2;  // 2 x 2 blocks (i <= j) per round
constexpr size_t JACOBI_SMEM =
    (2 * kSubspaceMaxK * JLD + 2 * JNP) * sizeof(float) + (2 * JNP + kSubspaceMaxK + JNB) * sizeof(int);

__global__ void __launch_bounds__(JT) jacobi_eig_kernel(const float *__restrict__ Tin, int k, float *__restrict__ lam,
                                                        float *__restrict__ W) {
    extern __shared__ __align__(16) float js[];
    float *T = js;                        // [k][JLD]
    float *V = T + kSubspaceMaxK * JLD;   // [k][JLD]
    float *cs = V + kSubspaceMaxK * JLD;  // [np] cosines
    float *sn = cs + JNP;                 // [np] sines (0: no rotation this round)
    int *pp = (int *)(sn + JNP);          // [np] first index of each pair
    int *pq = pp + JNP;                   // [np] second index (k: the dummy of an odd k)
    int *order = pq + JNP;                // [k] sort order of the eigenvalues
    int *blk = order + kSubspaceMaxK;     // [np (np + 1) / 2] block (i, j), i <= j, as i << 16 | j
    __shared__ int rotated;
    __shared__ float tol;
    const int t = threadIdx.x;
    const int kk = (k + 1) & ~1;  // even, with a dummy index k when k is odd
    const int np = kk / 2;
    const int m = kk - 1;

    for (int idx = t; idx < k * k; idx += JT) {
        const int i = idx / k, j = idx % k;
        T[i * JLD + j] = 0.5f * (Tin[i * k + j] + Tin[j * k + i]);
        V[i * JLD + j] = (i == j) ? 1.f : 0.f;
    }
    for (int idx = t; idx < np * np; idx += JT) {
        const int i = idx / np, j = idx % np;
        // row i of the upper triangle starts at i * np - i (i - 1) / 2
        if (i <= j) blk[i * np - (i * (i - 1)) / 2 + (j - i)] = (i << 16) | j;
    }
    const int nblk = np * (np + 1) / 2;
    __syncthreads();
    if (t == 0) {
        // Off-diagonal entries below 1e-7 of the largest diagonal entry are at the
        // float32 rounding level of T: they move no eigenvalue by more than that.
        float mx = 0.f;
        for (int i = 0; i < k; ++i) mx = fmaxf(mx, fabsf(T[i * JLD + i]));
        tol = 1e-7f * mx;
    }

    for (int sweep = 0; sweep < 15; ++sweep) {
        if (t == 0) rotated = 0;
        __syncthreads();
        for (int round = 0; round < m; ++round) {
            if (t < np) {
                // Round-robin (circle) pairing: kk - 1 stays fixed and meets `round`;
                // slot t >= 1 pairs round + t with round - t (mod kk - 1).  Every pair
                // meets exactly once in kk - 1 rounds.
                int p = (t == 0) ? round : (round + t) % m;
                int q = (t == 0) ? m : (round - t + m) % m;
                if (p > q) { const int x = p; p = q; q = x; }
                float c = 1.f, sv = 0.f;
                if (q < k) {
                    const float apq = T[p * JLD + q];
                    // Rotate unless a_pq is at the rounding level of T.
                    if (fabsf(apq) > tol) {
                        const float app = T[p * JLD + p], aqq = T[q * JLD + q];
                        const float tau = (aqq - app) / (2.f * apq);
                        const float tt = (tau >= 0.f ? 1.f : -1.f) / (fabsf(tau) + sqrtf(1.f + tau * tau));
                        c = 1.f / sqrtf(1.f + tt * tt);
                        sv = tt * c;
                        rotated = 1;
                    }
                }
                pp[t] = p;
                pq[t] = q;
                cs[t] = c;
                sn[t] = sv;
            }
            __syncthreads();
            // T <- J^T T J by 2 x 2 blocks; rows: p' = c p - s q, q' = s p + c q;
            // columns likewise.  A diagonal block's off-diagonal pair is the
            // annihilated element: set to exactly zero.
            for (int b = t; b < nblk; b += JT) {
                const int i = blk[b] >> 16, j = blk[b] & 0xFFFF;
                const float si = sn[i], sj = sn[j];
                if (si == 0.f && sj == 0.f) continue;
                const float ci = cs[i], cj = cs[j];
                const int pi = pp[i], qi = pq[i], pj = pp[j], qj = pq[j];
                const bool vi = qi < k, vj = qj < k;
                const float a = T[pi * JLD + pj];
                const float bb = vj ? T[pi * JLD + qj] : 0.f;
                const float cc = vi ? T[qi * JLD + pj] : 0.f;
                const float d = (vi && vj) ? T[qi * JLD + qj] : 0.f;
                const float a1 = ci * a - si * cc, b1 = ci * bb - si * d;
                const float c1 = si * a + ci * cc, d1 = si * bb + ci * d;
                const float a2 = cj * a1 - sj * b1, d2 = sj * c1 + cj * d1;
                float b2 = sj * a1 + cj * b1, c2 = cj * c1 - sj * d1;
                if (i == j) {
                    b2 = 0.f;
                    c2 = 0.f;
                }
                T[pi * JLD + pj] = a2;
                if (vj) T[pi * JLD + qj] = b2;
                if (vi) T[qi * JLD + pj] = c2;
                if (vi && vj) T[qi * JLD + qj] = d2;
                if (i != j) {
                    T[pj * JLD + pi] = a2;
                    if (vj) T[qj * JLD + pi] = b2;
                    if (vi) T[pj * JLD + qi] = c2;
                    if (vi && vj) T[qj * JLD + qi] = d2;
                }
            }
            // V <- V J: columns p_i, q_i of every row (q_i < k whenever s_i != 0).
            // Thread t: pair i = t / 16 (+ 64 per pass), rows t % 16 + 16 m.
            for (int i = t >> 4; i < np; i += JT >> 4) {
                const float sv = sn[i];
                if (sv == 0.f) continue;
                const float c = cs[i];
                const int p = pp[i], q = pq[i];
                for (int r = t & 15; r < k; r += 16) {
                    const float va = V[r * JLD + p], vb = V[r * JLD + q];
                    V[r * JLD + p] = c * va - sv * vb;
                    V[r * JLD + q] = sv * va + c * vb;
                }
            }
            __syncthreads();
        }
        if (!rotated) break;
        __syncthreads();
    }
    // Sort by descending eigenvalue (ties by index).
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
    // dst = L^-1 src: one 128-row tile of outputs per 128 columns is fewer CTAs than SMs, so K (= k)
    // is split as the block products split theirs, the slices summed in a fixed order.
    const int z = zsplit(cols, k);
    if (z > 1) return sgemm_splitk(k, cols, k, w.Linv, 128, false, src, cols, false, dst, w.part, z, s);
    return sgemm<float>(k, cols, k, 1.f, w.Linv, 128, false, src, cols, false, 0.f, dst, cols, 0, s);
}

// Z <- Z - (Z VL^T) VL: the k rows of Z (k x cols) made orthogonal to the nl
// locked rows of VL.  Nothing to do when nl = 0.
cudaError_t project_out(const SubspaceBufs &w, float *Z, int k, int64_t cols, cudaStream_t s) {
    if (w.nl <= 0) return cudaSuccess;
    cudaError_t e = sgemm_splitk(k, w.nl, cols, Z, cols, false, w.VL, cols, true, w.Cp, w.part, SPLITK, s);
    if (e != cudaSuccess) return e;
    return sgemm<float>(k, cols, w.nl, -1.f, w.Cp, w.nl, false, w.VL, cols, false, 1.f, Z, cols, 0, s);
}

// Y = the block ZT (k x cols) times the symmetric G.  On the tensor cores
// either with float32 accuracy (3xTF32) or, when !accurate, as one TF32
// product that reads only the hi half of G's split (half the bytes; for
// cols <= 5120 that half fits in L2 across iterations).
cudaError_t block_times_g(const SubspaceBufs &w, const float *ZT, float *Y, int k, int64_t cols, bool tc,
                          bool accurate, cudaStream_t s) {
    if (!tc) return sgemm<float>(k, cols, cols, 1.f, ZT, cols, false, w.G, cols, false, 0.f, Y, cols, 0, s);
    cudaError_t e = split_tf32(ZT, k, cols, cols, w.Zhi, w.Zlo, cols, s);
    if (e != cudaSuccess) return e;
    return gemm3_splitk(k, cols, cols, w.Zhi, w.Zlo, cols, w.Ghi, w.Glo, cols, Y, w.part, zsplit(cols, k), s,
                        !accurate);
}

}  // namespace

int subspace_width(int64_t cols, int r) {
    int64_t k = 2 * (int64_t)r;
    if (k > kSubspaceMaxK) k = kSubspaceMaxK;
    if (k > cols) k = cols;
    return (int)k;
}

size_t subspace_projection_part_floats(int k, int nl) { return (size_t)SPLITK * k * nl; }

size_t subspace_part_floats(int k, int64_t cols, bool tc) {
    (void)tc;
    size_t part = (size_t)SPLITK * k * k;
    if ((size_t)zsplit(cols, k) * k * cols > part) part = (size_t)zsplit(cols, k) * k * cols;
    return part;
}

cudaError_t subspace_ritz(const SubspaceBufs &w, int k, int64_t cols, bool tc, cudaStream_t s) {
    cudaError_t e;
    init_block_kernel<<<grid1d((int64_t)k * cols), 256, 0, s>>>(w.ZT2, k, cols);
    count_launch();
    if ((e = project_out(w, w.ZT2, k, cols, s)) != cudaSuccess) return e;
    if ((e = cholqr_pass(w, w.ZT2, w.ZT, k, cols, s)) != cudaSuccess) return e;
    if ((e = cholqr_pass(w, w.ZT, w.ZT2, k, cols, s)) != cudaSuccess) return e;
    if ((e = cudaMemcpyAsync(w.ZT, w.ZT2, (size_t)k * cols * sizeof(float), cudaMemcpyDeviceToDevice, s)) != cudaSuccess)
        return e;
    for (int it = 0; it < ITERS; ++it) {
        // TF32 products while the block converges; the last ACCURATE_TAIL
        // iterations at float32 accuracy remove what TF32 rounding left in the
        // subspace (each shrinks it by lambda_{k+1} / lambda_i per direction).
        const bool accurate = it >= ITERS - ACCURATE_TAIL;
        if ((e = block_times_g(w, w.ZT, w.ZT2, k, cols, tc, accurate, s)) != cudaSuccess) return e;
        if ((e = project_out(w, w.ZT2, k, cols, s)) != cudaSuccess) return e;
        if ((e = cholqr_pass(w, w.ZT2, w.ZT, k, cols, s)) != cudaSuccess) return e;
    }
    if ((e = cholqr_pass(w, w.ZT, w.ZT2, k, cols, s)) != cudaSuccess) return e;
    if (w.nl > 0) {
        // With locked vectors the block can hold directions that the iteration drove down to
        // rounding level (when the complement has fewer large eigenvalues than k): the shifted
        // pass leaves them short of unit length, and rounding gives them components along the
        // locked vectors.  Two more passes, each after a projection, make the block orthonormal
        // and orthogonal to the locked vectors before the Rayleigh-Ritz step.
        if ((e = project_out(w, w.ZT2, k, cols, s)) != cudaSuccess) return e;
        if ((e = cholqr_pass(w, w.ZT2, w.ZT, k, cols, s)) != cudaSuccess) return e;
        if ((e = project_out(w, w.ZT, k, cols, s)) != cudaSuccess) return e;
        if ((e = cholqr_pass(w, w.ZT, w.ZT2, k, cols, s)) != cudaSuccess) return e;
    }
    if ((e = cudaMemcpyAsync(w.ZT, w.ZT2, (size_t)k * cols * sizeof(float), cudaMemcpyDeviceToDevice, s)) != cudaSuccess)
        return e;

    // Rayleigh-Ritz: T = Z^T G Z (k x k), eigenpairs by Jacobi.
    if ((e = block_times_g(w, w.ZT, w.ZT2, k, cols, tc, true, s)) != cudaSuccess) return e;
    if ((e = project_out(w, w.ZT2, k, cols, s)) != cudaSuccess) return e;
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
