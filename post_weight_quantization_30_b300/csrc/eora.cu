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
//                                      vectors, then Rayleigh-Ritz
//                                      (subspace.cu)
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

// Marks a dead input (zero diagonal of H) as a failed pivot: EoRA needs a
// positive definite H.  Pivot columns are counted in reversed order.
__global__ void dead_to_pivot_kernel(const uint8_t *__restrict__ dead, int64_t cols, DeviceStatus *st) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < cols; i += (int64_t)gridDim.x * blockDim.x)
        if (dead[i]) atomicMin(&st->bad_pivot, (unsigned long long)(cols - 1 - i));
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

// A[i][j] <- A[j][i] for i < j: the upper triangle of a symmetric n x n
// matrix from its lower one (row stride lda).  One 32 x 32 tile of the upper
// triangle per block (tiles below the diagonal return at once), read from
// the mirrored lower tile and transposed through shared memory, so that both
// the loads and the stores run along rows.
__global__ void mirror_lower_kernel(float *__restrict__ A, int64_t n, int64_t lda) {
    __shared__ float t[32][33];
    const int64_t ti = blockIdx.y, tj = blockIdx.x;  // destination tile (ti, tj), ti <= tj
    if (ti > tj) return;
    const int tx = threadIdx.x, ty = threadIdx.y;     // 32 x 8 threads
    for (int r = ty; r < 32; r += 8) {
        const int64_t gi = tj * 32 + r, gj = ti * 32 + tx;  // source: rows of tile column tj
        t[r][tx] = (gi < n && gj < n) ? A[gi * lda + gj] : 0.f;
    }
    __syncthreads();
    for (int r = ty; r < 32; r += 8) {
        const int64_t gi = ti * 32 + r, gj = tj * 32 + tx;
        if (gi < gj && gj < n) A[gi * lda + gj] = t[tx][r];
    }
}

cudaError_t mirror_lower(float *A, int64_t n, int64_t lda, cudaStream_t s) {
    const unsigned nt = (unsigned)((n + 31) / 32);
    mirror_lower_kernel<<<dim3(nt, nt), dim3(32, 8), 0, s>>>(A, n, lda);
    count_launch();
    return cudaGetLastError();
}

// perm[rank] = i, rank = the position of lam[i] in descending order (ties by index).
__global__ void rank_desc_kernel(const float *__restrict__ lam, int n, int *__restrict__ perm) {
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const float v = lam[i];
        int rank = 0;
        for (int j = 0; j < n; ++j) rank += (lam[j] > v || (lam[j] == v && j < i)) ? 1 : 0;
        perm[rank] = i;
    }
}

// Row j of dst (cols floats) = row perm[j] of src; lam_dst[j] = lam_src[perm[j]].
__global__ void gather_rows_kernel(const float *__restrict__ src, const int *__restrict__ perm, int64_t cols,
                                   float *__restrict__ dst, const float *__restrict__ lam_src,
                                   float *__restrict__ lam_dst) {
    const int j = blockIdx.x;
    const int i = perm[j];
    for (int64_t c = threadIdx.x; c < cols; c += blockDim.x) dst[j * cols + c] = src[i * cols + c];
    if (threadIdx.x == 0) lam_dst[j] = lam_src[i];
}

struct EoraWs {
    DeviceStatus *st;
    float *Linv, *F, *M, *G, *ZT, *ZT2, *Gm, *part, *lam, *Wt, *VrT;
    float *lamr, *lams, *Cp;  // the r eigenvalues (chunk order, then sorted); projection scratch (k x r)
    int *perm;                // r: the sort order
    // tensor-core path only (null otherwise)
    float *FThi, *FTlo, *dWhi, *dWlo, *Mhi, *Mlo, *Mthi, *Mtlo, *Ghi, *Glo, *Zhi, *Zlo;
    uint8_t *dead;
};

constexpr int ASPLIT = 8;   // K slices of A = B^T dW
constexpr int CHUNK = 64;   // eigenpairs found per subspace iteration (k = 2 CHUNK vectors)

// The tensor-core path needs TMA-compatible row strides for M^T (rows) and H (cols).
bool eora_tc(int64_t rows, int64_t cols) { return rows % 4 == 0 && cols % 4 == 0; }

size_t eora_layout(int64_t rows, int64_t cols, int r, EoraWs *w, char *base) {
    const int k = subspace_width(cols, r);
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
    size_t part = subspace_part_floats(k, cols, tc);
    if ((size_t)ASPLIT * r * cols > part) part = (size_t)ASPLIT * r * cols;
    if (subspace_projection_part_floats(k, r) > part) part = subspace_projection_part_floats(k, r);
    t.part = (float *)take(part * sizeof(float));
    t.lam = (float *)take((size_t)k * sizeof(float));
    t.Wt = (float *)take((size_t)k * k * sizeof(float));
    t.VrT = (float *)take((size_t)r * cols * sizeof(float));
    t.lamr = (float *)take((size_t)r * sizeof(float));
    t.lams = (float *)take((size_t)r * sizeof(float));
    t.Cp = (float *)take((size_t)k * r * sizeof(float));
    t.perm = (int *)take((size_t)r * sizeof(int));
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
        // The split of the k-row blocks, and at the end of V_r^T (r rows, r may exceed k).
        const size_t zr = (size_t)(k > r ? k : r);
        t.Zhi = (float *)take(zr * cols * sizeof(float));
        t.Zlo = (float *)take(zr * cols * sizeof(float));
    }
    if (w) *w = t;
    return off;
}

unsigned grid1d(int64_t n) {
    const int64_t g = (n + 255) / 256;
    return (unsigned)(g < 1 ? 1 : (g > 148 * 8 ? 148 * 8 : g));
}

}  // namespace

size_t eora_workspace_bytes(int64_t rows, int64_t cols, int r) {
    // One extra DeviceStatus for the Cholesky-QR steps.
    return eora_layout(rows, cols, r, nullptr, nullptr) + align_up(sizeof(DeviceStatus));
}

cudaError_t eora_run(const float *dW, int64_t rows, int64_t cols, const float *H, int r, float *A, float *B,
                     float *sigma, void *ws, cudaStream_t s, unsigned long long *bad_pivot_host,
                     unsigned int *finite_host) {
    EoraWs w;
    const size_t main_bytes = eora_layout(rows, cols, r, &w, (char *)ws);
    DeviceStatus *qst = (DeviceStatus *)((char *)ws + main_bytes);
    const int k = subspace_width(cols, r);
    const bool tc = eora_tc(rows, cols);
    cudaError_t e;

    // H = F F^T (no damping); every input must be live.
    if ((e = cudaMemsetAsync(w.st, 0xFF, sizeof(DeviceStatus), s)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(qst, 0xFF, sizeof(DeviceStatus), s)) != cudaSuccess) return e;
    if ((e = finite_check_launch(dW, false, rows * cols, w.st, kNonFiniteW, s)) != cudaSuccess) return e;
    if ((e = factor_prepare(H, cols, 0.f, w.F, w.dead, w.st, s)) != cudaSuccess) return e;
    dead_to_pivot_kernel<<<grid1d(cols), 256, 0, s>>>(w.dead, cols, w.st);
    count_launch();
    if ((e = cholesky_lower_inplace(w.F, cols, w.st, w.Linv, s)) != cudaSuccess) return e;
    if ((e = factor_finalize(w.F, cols, s)) != cudaSuccess) return e;
    DeviceStatus hst;
    if ((e = cudaMemcpyAsync(&hst, w.st, sizeof(hst), cudaMemcpyDeviceToHost, s)) != cudaSuccess) return e;
    if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return e;
    *bad_pivot_host = hst.bad_pivot;
    *finite_host = hst.finite;
    if (hst.finite != ~0u || hst.bad_pivot != ULLONG_MAX) return cudaSuccess;

    if (tc) {
        // M = dW F (rows x cols, also split), its transpose split, G = M^T M (cols x cols, also split).
        if ((e = split_transpose_tf32(w.F, cols, cols, cols, w.FThi, w.FTlo, cols, s)) != cudaSuccess) return e;
        if ((e = split_tf32(dW, rows, cols, cols, w.dWhi, w.dWlo, cols, s)) != cudaSuccess) return e;
        // F is upper triangular, so F^T (the B operand) is lower: tri = 3 skips its zero products.
        if ((e = gemm3(rows, cols, cols, 1.f, w.dWhi, w.dWlo, cols, w.FThi, w.FTlo, cols, 0.f, w.M, cols, 3, w.Mhi,
                       w.Mlo, cols, s)) != cudaSuccess)
            return e;
        if ((e = split_transpose_tf32(w.M, rows, cols, cols, w.Mthi, w.Mtlo, rows, s)) != cudaSuccess) return e;
        // G is symmetric: the tiles on and below the diagonal, then the upper triangle mirrored.
        if ((e = gemm3(cols, cols, rows, 1.f, w.Mthi, w.Mtlo, rows, w.Mthi, w.Mtlo, rows, 0.f, w.G, cols, 1, w.Ghi,
                       w.Glo, cols, s)) != cudaSuccess)
            return e;
        if ((e = mirror_lower(w.G, cols, cols, s)) != cudaSuccess) return e;
        if ((e = mirror_lower(w.Ghi, cols, cols, s)) != cudaSuccess) return e;
        if ((e = mirror_lower(w.Glo, cols, cols, s)) != cudaSuccess) return e;
    } else {
        // M = dW F, G = M^T M (symmetric).
        if ((e = sgemm<float>(rows, cols, cols, 1.f, dW, cols, false, w.F, cols, false, 0.f, w.M, cols, 0, s)) !=
            cudaSuccess)
            return e;
        if ((e = sgemm<float>(cols, cols, rows, 1.f, w.M, cols, true, w.M, cols, false, 0.f, w.G, cols, 2, s)) !=
            cudaSuccess)
            return e;
    }

    // Leading eigenpairs of G (block subspace iteration + Rayleigh-Ritz).
    // Up to CHUNK of them per subspace iteration of k vectors; beyond that the
    // ones found are locked and the next iteration runs orthogonal to them.
    SubspaceBufs sb;
    sb.G = w.G; sb.Ghi = w.Ghi; sb.Glo = w.Glo;
    sb.ZT = w.ZT; sb.ZT2 = w.ZT2; sb.Zhi = w.Zhi; sb.Zlo = w.Zlo;
    sb.Gm = w.Gm; sb.Wt = w.Wt; sb.lam = w.lam; sb.part = w.part; sb.Linv = w.Linv; sb.qst = qst;
    sb.VL = w.VrT; sb.Cp = w.Cp;
    for (int nl = 0; nl < r;) {
        const int take = (r - nl) < CHUNK ? (r - nl) : CHUNK;
        sb.nl = nl;
        if ((e = subspace_ritz(sb, k, cols, tc, s)) != cudaSuccess) return e;
        // Rows nl .. nl + take of V_r^T = W[:, :take]^T Z^T (take x cols), and their eigenvalues.
        if ((e = sgemm<float>(take, cols, k, 1.f, w.Wt, k, true, w.ZT, cols, false, 0.f, w.VrT + (int64_t)nl * cols,
                              cols, 0, s)) != cudaSuccess)
            return e;
        if ((e = cudaMemcpyAsync(w.lamr + nl, w.lam, (size_t)take * sizeof(float), cudaMemcpyDeviceToDevice, s)) !=
            cudaSuccess)
            return e;
        nl += take;
    }
    const float *lam_r = w.lamr;
    if (r > CHUNK) {
        // Chunks meet where eigenvalues are nearly equal: one descending order for all r.
        rank_desc_kernel<<<1, 256, 0, s>>>(w.lamr, r, w.perm);
        count_launch();
        gather_rows_kernel<<<r, 256, 0, s>>>(w.VrT, w.perm, cols, w.part, w.lamr, w.lams);
        count_launch();
        if ((e = cudaMemcpyAsync(w.VrT, w.part, (size_t)r * cols * sizeof(float), cudaMemcpyDeviceToDevice, s)) !=
            cudaSuccess)
            return e;
        lam_r = w.lams;
    }
    // B = M V_r (rows x r), signs normalised.
    if (tc) {
        if ((e = split_tf32(w.VrT, r, cols, cols, w.Zhi, w.Zlo, cols, s)) != cudaSuccess) return e;
        e = gemm3(rows, r, cols, 1.f, w.Mhi, w.Mlo, cols, w.Zhi, w.Zlo, cols, 0.f, B, r, 0, nullptr, nullptr, 0, s);
    } else {
        e = sgemm<float>(rows, r, cols, 1.f, w.M, cols, false, w.VrT, cols, true, 0.f, B, r, 0, s);
    }
    if (e != cudaSuccess) return e;
    if ((e = sign_normalize(B, r, rows, r, 1, s)) != cudaSuccess) return e;
    // A = Σ^-2 B^T dW  (r x cols)
    if ((e = sgemm_splitk(r, cols, rows, B, r, true, dW, cols, false, A, w.part, ASPLIT, s)) != cudaSuccess) return e;
    finish_kernel<<<r, 256, 0, s>>>(lam_r, r, sigma, A, cols);
    count_launch();
    return cudaGetLastError();
}

int eora_subspace_width(int64_t rows, int64_t cols, int r) {
    (void)rows;
    return subspace_width(cols, r);
}

}  // namespace gq