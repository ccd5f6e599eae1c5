// EoRA: rank-r compensation of the quantization error in the eigenspace of
// the input covariance ("Aumento de la precisión de LLM de 2 bits con EoRA",
// 7minutos.es, "Bucear en el espacio propio en busca de un adaptador").
//
// The page projects the error ΔW = W - Ŵ with Q' = Q sqrt(Λ), where H = Q Λ Q^T,
// truncates the SVD of ΔW' = ΔW Q' and projects back.  Any S with S S^T = H
// gives the same adapter, because Q sqrt(Λ) = S O for an orthogonal O and the
// rotation only turns the right singular vectors.  The library takes S = F, the
// upper factor with H = F F^T that the GPTQ factorization already produces
// (without damping), so no eigendecomposition of H is needed:
//
//   M = ΔW F                          (rows x cols)
//   G = M^T M                         (cols x cols; its eigenvectors are M's
//                                      right singular vectors, eigenvalues σ²)
//   top-r eigenpairs of G             block subspace iteration with k = 2r
//                                      vectors (shifted Cholesky-QR after each
//                                      product), then Rayleigh-Ritz: Jacobi on
//                                      the k x k projected matrix
//   B = M V_r                         (= U_r Σ_r), sign-normalised so that the
//                                      largest-magnitude entry of each column is
//                                      positive
//   A = Σ_r^-2 B^T ΔW                 (= V_r^T F^-1: the projection back)
//
// so that B A = U_r U_r^T ΔW.
#include <climits>

#include "common.cuh"

namespace gq {
namespace {

constexpr int EORA_MAX_K = 128;   // subspace width limit (r <= 64)
constexpr int EORA_ITERS = 30;    // subspace iterations
constexpr int SPLITK = 64;        // K slices of the thin Gram products

// Marks a dead input (zero diagonal of H) as a failed pivot: EoRA needs a
// positive definite H.  Pivot columns are counted in reversed order.
__global__ void dead_to_pivot_kernel(const uint8_t *__restrict__ dead, int64_t cols, DeviceStatus *st) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < cols; i += (int64_t)gridDim.x * blockDim.x)
        if (dead[i]) atomicMin(&st->bad_pivot, (unsigned long long)(cols - 1 - i));
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
// cyclic Jacobi method in one CTA, parallel over the k/2 disjoint (p, q) pairs
// of a round-robin ordering.  Outputs the eigenvalues in descending order and
// the matching eigenvectors as the columns of W (row-major k x k).
constexpr int JT = 512;
constexpr int JLD = EORA_MAX_K + 1;
constexpr size_t JACOBI_SMEM = (2 * EORA_MAX_K * JLD + 2 * (EORA_MAX_K / 2 + 1)) * sizeof(float) +
                               (EORA_MAX_K + 2 + 2 * (EORA_MAX_K / 2 + 1)) * sizeof(int);

__global__ void __launch_bounds__(JT) jacobi_eig_kernel(const float *__restrict__ Tin, int k, float *__restrict__ lam,
                                                        float *__restrict__ W) {
    extern __shared__ __align__(16) float js[];
    float *T = js;                        // [k][JLD]
    float *V = T + EORA_MAX_K * JLD;      // [k][JLD]
    float *cs = V + EORA_MAX_K * JLD;     // [npairs] cosines
    float *sn = cs + EORA_MAX_K / 2 + 1;  // [npairs] sines
    int *pos = (int *)(sn + EORA_MAX_K / 2 + 1);  // [kk] round-robin positions
    int *pp = pos + EORA_MAX_K + 2;       // [npairs]
    int *pq = pp + EORA_MAX_K / 2 + 1;    // [npairs]
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

// Column signs of B (rows x r): the entry of largest magnitude (first on ties)
// is made positive; the column is negated otherwise.  One CTA per column.
__global__ void sign_normalize_kernel(float *__restrict__ B, int64_t rows, int r) {
    const int col = blockIdx.x;
    __shared__ float bv[32];
    __shared__ long long bi[32];
    __shared__ float flip;
    float best = -1.f;
    long long bidx = LLONG_MAX;
    for (int64_t m = threadIdx.x; m < rows; m += blockDim.x) {
        const float v = fabsf(B[m * r + col]);
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
        flip = (id != LLONG_MAX && B[id * r + col] < 0.f) ? -1.f : 1.f;
    }
    __syncthreads();
    if (flip < 0.f)
        for (int64_t m = threadIdx.x; m < rows; m += blockDim.x) B[m * r + col] = -B[m * r + col];
}

// sigma_i = sqrt(max(lam_i, 0)); row i of A scaled by 1 / sigma_i^2 (0 when
// sigma_i is not positive: that direction carries no error).
__global__ void finish_kernel(const float *__restrict__ lam, int r, float *__restrict__ sigma, float *__restrict__ A,
                              int64_t cols) {
    const int i = blockIdx.x;
    const float l = lam[i] > 0.f ? lam[i] : 0.f;
    if (threadIdx.x == 0 && sigma) sigma[i] = sqrtf(l);
    const float sc = l > 0.f ? 1.f / l : 0.f;
    for (int64_t j = threadIdx.x; j < cols; j += blockDim.x) A[i * cols + j] *= sc;
}

struct EoraWs {
    DeviceStatus *st;
    float *Linv, *F, *M, *G, *ZT, *ZT2, *Gm, *part, *lam, *Wt, *VrT;
    // tensor-core path only (null otherwise)
    float *FThi, *FTlo, *dWhi, *dWlo, *Mhi, *Mlo, *Mthi, *Mtlo, *Ghi, *Glo, *Zhi, *Zlo;
    uint8_t *dead;
};

constexpr int ZSPLIT = 4;   // K slices of the subspace products on the tensor cores
constexpr int ASPLIT = 8;   // K slices of A = B^T dW

int eora_k(int64_t rows, int64_t cols, int r) {
    (void)rows;
    int64_t k = 2 * (int64_t)r;
    if (k > EORA_MAX_K) k = EORA_MAX_K;
    if (k > cols) k = cols;
    return (int)k;
}

// The tensor-core path needs TMA-compatible row strides for M^T (rows) and H (cols).
bool eora_tc(int64_t rows, int64_t cols) { return rows % 4 == 0 && cols % 4 == 0; }

size_t eora_layout(int64_t rows, int64_t cols, int r, EoraWs *w, char *base) {
    const int k = eora_k(rows, cols, r);
    const bool tc = eora_tc(rows, cols);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        char *p = base ? base + off : nullptr;
        off += align_up(bytes);
        return p;
    };
    const size_t rc = (size_t)rows * cols * sizeof(float), cc = (size_t)cols * cols * sizeof(float);
    EoraWs t = {};
    t.st = (DeviceStatus *)take(sizeof(DeviceStatus));
    t.Linv = (float *)take(cholesky_scratch_floats(cols > 128 ? cols : 128) * sizeof(float));
    t.F = (float *)take(cc);
    t.dead = (uint8_t *)take((size_t)cols);
    t.M = (float *)take(rc);  // M = dW F (rows x cols)
    t.G = (float *)take(cc);
    t.ZT = (float *)take((size_t)k * cols * sizeof(float));
    t.ZT2 = (float *)take((size_t)k * cols * sizeof(float));
    t.Gm = (float *)take((size_t)k * k * sizeof(float));
    size_t part = (size_t)SPLITK * k * k;
    if ((size_t)ASPLIT * r * cols > part) part = (size_t)ASPLIT * r * cols;
    if (tc && (size_t)ZSPLIT * k * cols > part) part = (size_t)ZSPLIT * k * cols;
    t.part = (float *)take(part * sizeof(float));
    t.lam = (float *)take((size_t)k * sizeof(float));
    t.Wt = (float *)take((size_t)k * k * sizeof(float));
    t.VrT = (float *)take((size_t)r * cols * sizeof(float));
    if (tc) {
        t.FThi = (float *)take(cc);
        t.FTlo = (float *)take(cc);
        t.dWhi = (float *)take(rc);
        t.dWlo = (float *)take(rc);
        t.Mhi = (float *)take(rc);
        t.Mlo = (float *)take(rc);
        t.Mthi = (float *)take(rc);
        t.Mtlo = (float *)take(rc);
        t.Ghi = (float *)take(cc);
        t.Glo = (float *)take(cc);
        t.Zhi = (float *)take((size_t)k * cols * sizeof(float));
        t.Zlo = (float *)take((size_t)k * cols * sizeof(float));
    }
    if (w) *w = t;
    return off;
}

unsigned grid1d(int64_t n) {
    const int64_t g = (n + 255) / 256;
    return (unsigned)(g < 1 ? 1 : (g > 148 * 8 ? 148 * 8 : g));
}

// One pass of shifted Cholesky-QR on the rows of src (k x cols): rows scaled
// to unit norm, src src^T + shift = L L^T, dst = L^-1 src.  src is scaled in place.
cudaError_t cholqr_pass(const EoraWs &w, float *src, float *dst, int k, int64_t cols, DeviceStatus *qst,
                        cudaStream_t s) {
    normalize_rows_kernel<<<k, 256, 0, s>>>(src, cols);
    count_launch();
    cudaError_t e = sgemm_splitk(k, k, cols, src, cols, false, src, cols, true, w.Gm, w.part, SPLITK, s);
    if (e != cudaSuccess) return e;
    shift_gram_kernel<<<1, 128, 0, s>>>(w.Gm, k);
    count_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = cholesky_lower_inplace(w.Gm, k, qst, w.Linv, s)) != cudaSuccess) return e;
    return sgemm<float>(k, cols, k, 1.f, w.Linv, 128, false, src, cols, false, 0.f, dst, cols, 0, s);
}

// Y = Z^T-block times G: rows of ZT (k x cols) multiplied by the symmetric G.
cudaError_t block_times_g(const EoraWs &w, const float *ZT, float *Y, int k, int64_t cols, bool tc, cudaStream_t s) {
    if (!tc) return sgemm<float>(k, cols, cols, 1.f, ZT, cols, false, w.G, cols, false, 0.f, Y, cols, 0, s);
    cudaError_t e = split_tf32(ZT, k, cols, cols, w.Zhi, w.Zlo, cols, s);
    if (e != cudaSuccess) return e;
    return gemm3_splitk(k, cols, cols, w.Zhi, w.Zlo, cols, w.Ghi, w.Glo, cols, Y, w.part, ZSPLIT, s);
}

}  // namespace

size_t eora_workspace_bytes(int64_t rows, int64_t cols, int r) {
    // One extra DeviceStatus for the Cholesky-QR steps.
    return eora_layout(rows, cols, r, nullptr, nullptr) + align_up(sizeof(DeviceStatus));
}

cudaError_t eora_run(const float *dW, int64_t rows, int64_t cols, const float *H, int r, float *A, float *B,
                     float *sigma, void *ws, cudaStream_t s, unsigned long long *bad_pivot_host) {
    EoraWs w;
    const size_t main_bytes = eora_layout(rows, cols, r, &w, (char *)ws);
    DeviceStatus *qst = (DeviceStatus *)((char *)ws + main_bytes);
    const int k = eora_k(rows, cols, r);
    const bool tc = eora_tc(rows, cols);
    cudaError_t e;

    // H = F F^T (no damping); every input must be live.
    if ((e = cudaMemsetAsync(w.st, 0xFF, sizeof(DeviceStatus), s)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(qst, 0xFF, sizeof(DeviceStatus), s)) != cudaSuccess) return e;
    if ((e = factor_prepare(H, cols, 0.f, w.F, w.dead, w.st, s)) != cudaSuccess) return e;
    dead_to_pivot_kernel<<<grid1d(cols), 256, 0, s>>>(w.dead, cols, w.st);
    count_launch();
    if ((e = cholesky_lower_inplace(w.F, cols, w.st, w.Linv, s)) != cudaSuccess) return e;
    if ((e = factor_finalize(w.F, cols, s)) != cudaSuccess) return e;
    if ((e = cudaMemcpyAsync(bad_pivot_host, &w.st->bad_pivot, sizeof(unsigned long long), cudaMemcpyDeviceToHost,
                             s)) != cudaSuccess)
        return e;
    if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return e;
    if (*bad_pivot_host != ULLONG_MAX) return cudaSuccess;

    if (tc) {
        // M = dW F (rows x cols, also split), its transpose split, G = M^T M (cols x cols, also split).
        if ((e = split_transpose_tf32(w.F, cols, cols, cols, w.FThi, w.FTlo, cols, s)) != cudaSuccess) return e;
        if ((e = split_tf32(dW, rows, cols, cols, w.dWhi, w.dWlo, cols, s)) != cudaSuccess) return e;
        if ((e = gemm3(rows, cols, cols, 1.f, w.dWhi, w.dWlo, cols, w.FThi, w.FTlo, cols, 0.f, w.M, cols, 0, w.Mhi,
                       w.Mlo, cols, s)) != cudaSuccess)
            return e;
        if ((e = split_transpose_tf32(w.M, rows, cols, cols, w.Mthi, w.Mtlo, rows, s)) != cudaSuccess) return e;
        if ((e = gemm3(cols, cols, rows, 1.f, w.Mthi, w.Mtlo, rows, w.Mthi, w.Mtlo, rows, 0.f, w.G, cols, 0, w.Ghi,
                       w.Glo, cols, s)) != cudaSuccess)
            return e;
    } else {
        // M = dW F, G = M^T M (symmetric).
        if ((e = sgemm<float>(rows, cols, cols, 1.f, dW, cols, false, w.F, cols, false, 0.f, w.M, cols, 0, s)) !=
            cudaSuccess)
            return e;
        if ((e = sgemm<float>(cols, cols, rows, 1.f, w.M, cols, true, w.M, cols, false, 0.f, w.G, cols, 2, s)) !=
            cudaSuccess)
            return e;
    }

    // Block subspace iteration on G, the block kept as the rows of ZT (k x cols):
    // ZT <- orth(ZT G).  One Cholesky-QR pass per product, two at the start and
    // before the Rayleigh-Ritz step.
    init_block_kernel<<<grid1d((int64_t)k * cols), 256, 0, s>>>(w.ZT2, k, cols);
    count_launch();
    if ((e = cholqr_pass(w, w.ZT2, w.ZT, k, cols, qst, s)) != cudaSuccess) return e;
    if ((e = cholqr_pass(w, w.ZT, w.ZT2, k, cols, qst, s)) != cudaSuccess) return e;
    if ((e = cudaMemcpyAsync(w.ZT, w.ZT2, (size_t)k * cols * sizeof(float), cudaMemcpyDeviceToDevice, s)) != cudaSuccess)
        return e;
    for (int it = 0; it < EORA_ITERS; ++it) {
        if ((e = block_times_g(w, w.ZT, w.ZT2, k, cols, tc, s)) != cudaSuccess) return e;
        if ((e = cholqr_pass(w, w.ZT2, w.ZT, k, cols, qst, s)) != cudaSuccess) return e;
    }
    if ((e = cholqr_pass(w, w.ZT, w.ZT2, k, cols, qst, s)) != cudaSuccess) return e;
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
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // V_r^T = W[:, :r]^T Z^T  (r x cols)
    if ((e = sgemm<float>(r, cols, k, 1.f, w.Wt, k, true, w.ZT, cols, false, 0.f, w.VrT, cols, 0, s)) != cudaSuccess)
        return e;
    // B = M V_r (rows x r), signs normalised.
    if (tc) {
        if ((e = split_tf32(w.VrT, r, cols, cols, w.Zhi, w.Zlo, cols, s)) != cudaSuccess) return e;
        e = gemm3(rows, r, cols, 1.f, w.Mhi, w.Mlo, cols, w.Zhi, w.Zlo, cols, 0.f, B, r, 0, nullptr, nullptr, 0, s);
    } else {
        e = sgemm<float>(rows, r, cols, 1.f, w.M, cols, false, w.VrT, cols, true, 0.f, B, r, 0, s);
    }
    if (e != cudaSuccess) return e;
    sign_normalize_kernel<<<r, 256, 0, s>>>(B, rows, r);
    count_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // A = Σ^-2 B^T dW  (r x cols)
    if ((e = sgemm_splitk(r, cols, rows, B, r, true, dW, cols, false, A, w.part, ASPLIT, s)) != cudaSuccess) return e;
    finish_kernel<<<r, 256, 0, s>>>(w.lam, r, sigma, A, cols);
    count_launch();
    return cudaGetLastError();
}

int eora_subspace_width(int64_t rows, int64_t cols, int r) { return eora_k(rows, cols, r); }

}  // namespace gq
