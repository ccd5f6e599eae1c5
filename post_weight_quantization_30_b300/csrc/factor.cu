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

__device__ __forceinline__ float tf32_round(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

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
// Every entry of H it reads (the upper triangle and the diagonal) is also
// checked: an Inf or NaN clears kNonFiniteH in st->finite.
__global__ void reverse_damp_kernel(const float *__restrict__ H, int64_t cols, float *__restrict__ F,
                                    uint8_t *__restrict__ dead, DeviceStatus *__restrict__ st) {
    const int64_t p = blockIdx.y;
    const float delta = st->delta;
    bool bad = false;
    for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < cols; q += (int64_t)gridDim.x * blockDim.x) {
        float v = 0.f;
        if (q < p) {
            v = H[(cols - 1 - p) * cols + (cols - 1 - q)];
            bad |= !isfinite(v);
        } else if (q == p) {
            const int64_t i = cols - 1 - p;
            float d = H[i * cols + i];
            bad |= !isfinite(d);
            if (dead) dead[i] = (d == 0.f);
            v = ((d == 0.f) ? 1.f : d) + delta;
        }
        F[p * cols + q] = v;
    }
    if (bad) atomicAnd(&st->finite, ~kNonFiniteH);
}

// The same for cols % 4 == 0 and 16-byte aligned H and F, four entries of a
// row of F per thread: F[p][q .. q + 3] come from one float4 of H's row
// C - 1 - p (columns C - 4 - q .. C - 1 - q, reversed), so every thread has
// its load in flight at once.  Only the entries with q <= p are taken (and
// checked); the rest of the float4 belongs to H's other triangle.
__global__ void reverse_damp4_kernel(const float *__restrict__ H, int64_t cols, float *__restrict__ F,
                                     uint8_t *__restrict__ dead, DeviceStatus *__restrict__ st) {
    const int64_t p = blockIdx.y;
    const float delta = st->delta;
    const float *hrow = H + (cols - 1 - p) * cols;
    bool bad = false;
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < cols / 4; v += (int64_t)gridDim.x * blockDim.x) {
        const int64_t q = 4 * v;
        float o[4] = {0.f, 0.f, 0.f, 0.f};
        if (q <= p) {
            const float4 h = *reinterpret_cast<const float4 *>(hrow + (cols - 4 - q));
            const float e[4] = {h.w, h.z, h.y, h.x};  // H[C-1-p][C-1-q-u]
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (q + u < p) {
                    o[u] = e[u];
                    bad |= !isfinite(e[u]);
                } else if (q + u == p) {
                    const int64_t i = cols - 1 - p;
                    bad |= !isfinite(e[u]);
                    if (dead) dead[i] = (e[u] == 0.f);
                    o[u] = ((e[u] == 0.f) ? 1.f : e[u]) + delta;
                }
            }
        }
        *reinterpret_cast<float4 *>(F + p * cols + q) = make_float4(o[0], o[1], o[2], o[3]);
    }
    if (bad) atomicAnd(&st->finite, ~kNonFiniteH);
}

// Clears `bit` of st->finite if an element of X is an Inf or NaN (all exponent
// bits set: 0x7F80 in bf16, 0x7F800000 in float32).  16-byte loads over the
// aligned middle of the buffer, element loads at both ends.
__global__ void finite_check_kernel(const unsigned char *__restrict__ X, int64_t nbytes, int esize,
                                    DeviceStatus *__restrict__ st, unsigned int bit) {
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t nth = (int64_t)gridDim.x * blockDim.x;
    const uint32_t m32 = esize == 2 ? 0x7F807F80u : 0x7F800000u;
    const int64_t head = (int64_t)((16 - ((uintptr_t)X & 15)) & 15) < nbytes ? (int64_t)((16 - ((uintptr_t)X & 15)) & 15)
                                                                            : nbytes;
    const int64_t nvec = (nbytes - head) / 16;
    const int64_t tail0 = head + nvec * 16;
    auto bad_elem = [&](int64_t off) {
        if (esize == 2) {
            const uint16_t u = *reinterpret_cast<const uint16_t *>(X + off);
            return (u & 0x7F80u) == 0x7F80u;
        }
        const uint32_t u = *reinterpret_cast<const uint32_t *>(X + off);
        return (u & 0x7F800000u) == 0x7F800000u;
    };
    auto bad_word = [&](uint32_t u) {
        if (esize == 2) return ((u & 0x7F80u) == 0x7F80u) || ((u & 0x7F800000u) == 0x7F800000u);
        return (u & m32) == m32;
    };
    bool bad = false;
    for (int64_t off = tid * esize; off < head; off += nth * esize) bad |= bad_elem(off);
    const uint4 *v = reinterpret_cast<const uint4 *>(X + head);
    for (int64_t i = tid; i < nvec; i += nth) {
        const uint4 w = __ldg(v + i);
        bad |= bad_word(w.x) | bad_word(w.y) | bad_word(w.z) | bad_word(w.w);
    }
    for (int64_t off = tail0 + tid * esize; off < nbytes; off += nth * esize) bad |= bad_elem(off);
    if (bad) atomicAnd(&st->finite, ~bit);
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
//      forward substitution (lane c produces column c of the inverse);
//   2. all warps solve the sub-panel below against it, X = A L_pp^-T, as a
//      product with the sub-block's inverse (4 x 4 register tiles);
//   3. all warps update the trailing lower triangle, A -= X X^T (4 x 4 tiles).
// The off-diagonal 32 x 32 blocks of L^-1 are assembled block row by block
// row, Y_pq = -Y_pp sum_{q <= m < p} L_pm Y_mq (4 x 4 tiles): rows 1 and 2 by
// six warps while warp 0 factors the sub-panel after them, row 3 at the end.
// The pivot reciprocal square root comes from rsqrtf; the factor is d * rsqrt(d).
constexpr int DIAG_THREADS = 256;
constexpr int SP = 32;           // sub-panel width
constexpr int LDA = NB + 4;      // shared-memory row stride (floats)
constexpr size_t DIAG_SMEM = (2 * NB * LDA + 2 * SP * LDA + 3 * SP * SP + 3 * SP) * sizeof(float);

// Lane i holds row i of a 32 x 32 symmetric block (entries k <= i) and ends
// with row i of its lower Cholesky factor; `rinv` of lane i ends as 1 / L_ii.
// Step J: the pivot comes by shuffle from lane J; the new column J of L is
// written once to a shared-memory buffer (two alternating buffers) and read
// back by every lane with float4 broadcast loads for the rank-1 update.  The
// steps are unrolled by template recursion so that every index into `a` is a
// compile-time constant (the array stays in registers).
template <int J>
struct CholStep {
    static __device__ __forceinline__ void run(float (&a)[SP], float &rinv, int lane, int64_t gcol0,
                                               DeviceStatus *st, float *colbuf) {
        const unsigned full = 0xffffffffu;
        const float d = __shfl_sync(full, a[J], J);
        if (lane == 0 && !(d > 0.f)) atomicMin(&st->bad_pivot, (unsigned long long)(gcol0 + J));
        const float r = rsqrtf(d);
        if (lane == J) rinv = r;
        // Lane J holds d, so d r = sqrt(d) there; below the diagonal a[J] r = L_iJ.
        // Entries above a lane's diagonal (k > lane) are never read, so every lane
        // updates all of its entries without a per-entry predicate.
        a[J] *= r;
        if (J + 1 < SP) {
            float *cb = colbuf + (J & 1) * SP;
            cb[lane] = a[J];
            __syncwarp();
#pragma unroll
            for (int k4 = ((J + 1) / 4) * 4; k4 < SP; k4 += 4) {
                const float4 c4 = *reinterpret_cast<const float4 *>(cb + k4);
                const float cv[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int k = k4 + u;
                    if (k > J) a[k] = fmaf(-a[J], cv[u], a[k]);
                }
            }
        }
        CholStep<J + 1>::run(a, rinv, lane, gcol0, st, colbuf);
    }
};
template <>
struct CholStep<SP> {
    static __device__ __forceinline__ void run(float (&)[SP], float &, int, int64_t, DeviceStatus *, float *) {}
};

// Column `lane` of the inverse of the 32 x 32 lower factor stored at L (row
// stride LDA, 16-byte aligned rows), dinv[i] = 1 / L_ii:
// y_i = (delta_i,lane - sum_{k<i} L_ik y_k) dinv_i, rows of L read as float4
// broadcasts.  Written transposed: YT[lane][i] = (L^-1)_{i,lane}.
__device__ __forceinline__ void warp_trinv32(const float *L, const float *dinv, float *YT, int lane) {
    float y[SP];
#pragma unroll
    for (int i = 0; i < SP; ++i) {
        float s0 = (lane == i) ? 1.f : 0.f, s1 = 0.f;
#pragma unroll
        for (int k4 = 0; k4 < i; k4 += 4) {
            const float4 l4 = *reinterpret_cast<const float4 *>(L + i * LDA + k4);
            if (k4 + 0 < i) s0 = fmaf(-l4.x, y[k4 + 0], s0);
            if (k4 + 1 < i) s1 = fmaf(-l4.y, y[k4 + 1], s1);
            if (k4 + 2 < i) s0 = fmaf(-l4.z, y[k4 + 2], s0);
            if (k4 + 3 < i) s1 = fmaf(-l4.w, y[k4 + 3], s1);
        }
        y[i] = (s0 + s1) * dinv[i];
    }
#pragma unroll
    for (int i = 0; i < SP; ++i) YT[lane * LDA + i] = y[i];
}

// Block row p >= 1 of Y = L^-1 off the diagonal, by threads tid = 0 .. nthr - 1
// in 4 x 4 tiles: T_q = sum_{m=q}^{p-1} L_pm Y_mq, then Y_pq = -Y_pp T_q, for
// q < p (32 x 32 blocks; L in A, T scratch [3][SP][SP]).  It reads L's block
// row p left of the diagonal, Y's block rows before p and Y_pp; `sync`
// separates the two products among the nthr threads.
template <typename Sync>
__device__ __forceinline__ void inverse_block_row(int p, int tid, int nthr, const float *A, float *Y, float *T,
                                                  Sync sync) {
    const int ntl = p * (SP / 4) * (SP / 4);
    for (int tl = tid; tl < ntl; tl += nthr) {
        const int q = tl / 64, i0 = ((tl / 8) % 8) * 4, c0 = (tl % 8) * 4;
        float acc[4][4] = {};
        for (int k = q * SP; k < p * SP; ++k) {
            const float4 yv = *reinterpret_cast<const float4 *>(Y + k * LDA + q * SP + c0);
            const float yb[4] = {yv.x, yv.y, yv.z, yv.w};
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const float lv = A[(p * SP + i0 + a) * LDA + k];
#pragma unroll
                for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(lv, yb[b], acc[a][b]);
            }
        }
#pragma unroll
        for (int a = 0; a < 4; ++a)
            *reinterpret_cast<float4 *>(T + q * SP * SP + (i0 + a) * SP + c0) =
                make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
    }
    sync();
    for (int tl = tid; tl < ntl; tl += nthr) {
        const int q = tl / 64, i0 = ((tl / 8) % 8) * 4, c0 = (tl % 8) * 4;
        const float *tq = T + q * SP * SP;
        float acc[4][4] = {};
        for (int k = 0; k < i0 + 4; ++k) {
            const float4 tv = *reinterpret_cast<const float4 *>(tq + k * SP + c0);
            const float tb[4] = {tv.x, tv.y, tv.z, tv.w};
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const float yv = Y[(p * SP + i0 + a) * LDA + p * SP + k];  // zero for k > i0 + a
#pragma unroll
                for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(yv, tb[b], acc[a][b]);
            }
        }
#pragma unroll
        for (int a = 0; a < 4; ++a)
            *reinterpret_cast<float4 *>(Y + (p * SP + i0 + a) * LDA + q * SP + c0) =
                make_float4(-acc[a][0], -acc[a][1], -acc[a][2], -acc[a][3]);
    }
}

// Outputs: Linv, the inverse (NB x NB), written only when Lhi is NULL; when
// Lhi / Llo are given they receive its TF32 split instead (the form the panel
// solve reads).  Optional (may be NULL): Urev, the index-reversed inverse Urev[i][j] = Linv[kb-1-i][kb-1-j] (kb x kb,
// row stride kb): the inverse of the matching diagonal block of F = J L J.
__global__ void __launch_bounds__(DIAG_THREADS, 1) potrf_diag_kernel(float *__restrict__ F, int64_t cols, int64_t k0,
                                                                  int kb, float *__restrict__ Linv,
                                                                  DeviceStatus *st, float *__restrict__ Lhi,
                                                                  float *__restrict__ Llo, float *__restrict__ Urev) {
    pdl_trigger();
    pdl_wait();  // the block was last updated by the previous kernel
    extern __shared__ __align__(16) float sm[];
    float *A = sm;                 // [NB][LDA]: the block, lower triangle, becomes L
    float *Y = A + NB * LDA;       // [NB][LDA]: L^-1, lower triangle
    float *XT = Y + NB * LDA;      // [SP][LDA]: solved sub-panel, transposed (XT[k][i] = X_ik)
    float *YT = XT + SP * LDA;     // [SP][LDA]: current diagonal inverse, transposed
    float *T = YT + SP * LDA;      // [3][SP][SP]: partial sums of the inverse assembly
    float *dinv = T + 3 * SP * SP; // [SP]
    float *colbuf = dinv + SP;     // [2][SP]: pivot column broadcast of the warp factorization
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;

    // Load: 16 float4 per thread, all issued before any shared-memory store.
    const bool vec = (cols % 4) == 0 && ((uintptr_t)F % 16) == 0;
    {
        float4 v[NB * NB / 4 / DIAG_THREADS];
#pragma unroll
        for (int u = 0; u < NB * NB / 4 / DIAG_THREADS; ++u) {
            const int idx = t + u * DIAG_THREADS;
            const int i = idx / (NB / 4), j = (idx % (NB / 4)) * 4;
            const float *src = F + (k0 + i) * cols + (k0 + j);
            if (vec && i < kb && j + 3 < kb) {
                v[u] = *reinterpret_cast<const float4 *>(src);
            } else {
                float e[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) e[c] = (i < kb && j + c < kb) ? src[c] : 0.f;
                v[u] = make_float4(e[0], e[1], e[2], e[3]);
            }
        }
#pragma unroll
        for (int u = 0; u < NB * NB / 4 / DIAG_THREADS; ++u) {
            const int idx = t + u * DIAG_THREADS;
            const int i = idx / (NB / 4), j = (idx % (NB / 4)) * 4;
            float e[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int jj = j + c;
                if (i >= kb || jj >= kb) e[c] = (i == jj) ? 1.f : 0.f;
                else if (jj > i) e[c] = 0.f;
            }
            *reinterpret_cast<float4 *>(A + i * LDA + j) = make_float4(e[0], e[1], e[2], e[3]);
            *reinterpret_cast<float4 *>(Y + i * LDA + j) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    __syncthreads();

    for (int c0 = 0; c0 < NB; c0 += SP) {
        if (warp == 0) {
            float a[SP], rinv = 0.f;
#pragma unroll
            for (int k = 0; k < SP; ++k) a[k] = (k <= lane) ? A[(c0 + lane) * LDA + c0 + k] : 0.f;
            CholStep<0>::run(a, rinv, lane, k0 + c0, st, colbuf);
#pragma unroll
            for (int k = 0; k < SP; ++k)
                if (k <= lane) A[(c0 + lane) * LDA + c0 + k] = a[k];
            dinv[lane] = rinv;
            __syncwarp();
            warp_trinv32(A + c0 * LDA + c0, dinv, YT, lane);
            __syncwarp();
            // Diagonal block of Y from its transposed copy.
#pragma unroll 4
            for (int i = 0; i < SP; ++i) Y[(c0 + i) * LDA + c0 + lane] = YT[lane * LDA + i];
        } else if (c0 >= 2 * SP && (warp & 3) != 0) {
            // While warp 0 factors this sub-panel, six other warps form the previous block
            // row of the inverse: everything it reads is final, and nothing the factorization
            // touches is written.  Warp 4 stays idle: it would share warp 0's scheduler.
            inverse_block_row(c0 / SP - 1, (warp - 1 - (warp >> 2)) * 32 + lane, 192, A, Y, T,
                              [] { asm volatile("bar.sync 1, 192;" ::: "memory"); });
        }
        __syncthreads();
        const int r0 = c0 + SP, R = NB - r0;  // rows below the diagonal sub-block
        if (R == 0) break;
        // X_ic = sum_{k <= c} A_ik Y_ck (Y_ck = YT[k][c]) in 4 x 4 tiles: rows i0.., columns cc..
        const int ntile = (R / 4) * (SP / 4);
        float xo[4][4];
        int ti0 = 0, tc0 = 0;
        const bool active = t < ntile;
        if (active) {
            ti0 = r0 + (t / (SP / 4)) * 4;
            tc0 = (t % (SP / 4)) * 4;
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 4; ++b) xo[a][b] = 0.f;
            for (int k = 0; k < tc0 + 4; ++k) {
                const float4 yv = *reinterpret_cast<const float4 *>(YT + k * LDA + tc0);
                const float yb[4] = {yv.x, yv.y, yv.z, yv.w};
#pragma unroll
                for (int a = 0; a < 4; ++a) {
                    const float av = A[(ti0 + a) * LDA + c0 + k];
#pragma unroll
                    for (int b = 0; b < 4; ++b) xo[a][b] = fmaf(av, yb[b], xo[a][b]);
                }
            }
        }
        __syncthreads();
        if (active) {
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                *reinterpret_cast<float4 *>(A + (ti0 + a) * LDA + c0 + tc0) =
                    make_float4(xo[a][0], xo[a][1], xo[a][2], xo[a][3]);
#pragma unroll
                for (int b = 0; b < 4; ++b) XT[(tc0 + b) * LDA + ti0 + a] = xo[a][b];
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

    // The last block row of Y = L^-1 (the earlier ones were formed during the
    // factorization of the sub-panel after them).
    inverse_block_row(NB / SP - 1, t, DIAG_THREADS, A, Y, T, [] { __syncthreads(); });
    __syncthreads();

    // Store: F gets the lower factor (its part above the diagonal is zero in A),
    // Linv the inverse or its split; padding rows / columns are not written to F.
#pragma unroll 4
    for (int u = 0; u < NB * NB / 4 / DIAG_THREADS; ++u) {
        const int idx = t + u * DIAG_THREADS;
        const int i = idx / (NB / 4), j = (idx % (NB / 4)) * 4;
        const float4 lv = *reinterpret_cast<const float4 *>(A + i * LDA + j);
        float4 yv = *reinterpret_cast<const float4 *>(Y + i * LDA + j);
        float *dst = F + (k0 + i) * cols + (k0 + j);
        if (vec && i < kb && j + 3 < kb) {
            *reinterpret_cast<float4 *>(dst) = lv;
        } else if (i < kb) {
            const float e[4] = {lv.x, lv.y, lv.z, lv.w};
#pragma unroll
            for (int c = 0; c < 4; ++c)
                if (j + c < kb) dst[c] = e[c];
        }
        if (i >= kb) yv = make_float4(0.f, 0.f, 0.f, 0.f);
        if (j + 0 >= kb) yv.x = 0.f;
        if (j + 1 >= kb) yv.y = 0.f;
        if (j + 2 >= kb) yv.z = 0.f;
        if (j + 3 >= kb) yv.w = 0.f;
        if (!Lhi) {
            *reinterpret_cast<float4 *>(Linv + idx * 4) = yv;
        } else {
            const float h[4] = {tf32_round(yv.x), tf32_round(yv.y), tf32_round(yv.z), tf32_round(yv.w)};
            *reinterpret_cast<float4 *>(Lhi + idx * 4) = make_float4(h[0], h[1], h[2], h[3]);
            *reinterpret_cast<float4 *>(Llo + idx * 4) =
                make_float4(yv.x - h[0], yv.y - h[1], yv.z - h[2], yv.w - h[3]);
        }
    }
    if (Urev && kb == NB) {
        // Four reversed columns at a time: Urev[i][j .. j + 3] = Y[ri][rj - 3 .. rj] backwards,
        // rj = NB - 1 - j (rj - 3 is a multiple of 4), zero where the column is above the diagonal.
        for (int idx = t; idx < NB * NB / 4; idx += DIAG_THREADS) {
            const int i = idx / (NB / 4), j = (idx % (NB / 4)) * 4;
            const int ri = NB - 1 - i, rj = NB - 1 - j;
            const float4 y = *reinterpret_cast<const float4 *>(Y + ri * LDA + rj - 3);
            const float4 o = make_float4(rj <= ri ? y.w : 0.f, rj - 1 <= ri ? y.z : 0.f, rj - 2 <= ri ? y.y : 0.f,
                                         rj - 3 <= ri ? y.x : 0.f);
            *reinterpret_cast<float4 *>(Urev + idx * 4) = o;
        }
    } else if (Urev) {
        for (int idx = t; idx < kb * kb; idx += DIAG_THREADS) {
            const int i = idx / kb, j = idx % kb;
            const int ri = kb - 1 - i, rj = kb - 1 - j;
            Urev[idx] = (rj <= ri) ? Y[ri * LDA + rj] : 0.f;
        }
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

// The same for cols % 4 == 0 and a 16-byte aligned F: the lower-triangle
// float4 F[p][q .. q + 3] with q + 3 < p goes reversed to F[C-1-p][C-4-q ..
// C-1-q] (upper triangle, written by this thread only) and is zeroed; the
// float4 that holds the diagonal entry is done element by element.
__global__ void finalize4_kernel(float *__restrict__ F, int64_t cols) {
    const int64_t p = blockIdx.y;
    const int64_t p2 = cols - 1 - p;
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; 4 * v <= p; v += (int64_t)gridDim.x * blockDim.x) {
        const int64_t q = 4 * v;
        if (q + 3 < p) {
            const float4 a = *reinterpret_cast<const float4 *>(F + p * cols + q);
            *reinterpret_cast<float4 *>(F + p2 * cols + (cols - 4 - q)) = make_float4(a.w, a.z, a.y, a.x);
            *reinterpret_cast<float4 *>(F + p * cols + q) = make_float4(0.f, 0.f, 0.f, 0.f);
        } else {
            for (int64_t qq = q; qq <= p; ++qq) {
                if (qq == p) {
                    if (p < p2) {
                        const float a = F[p * cols + p], b = F[p2 * cols + p2];
                        F[p * cols + p] = b;
                        F[p2 * cols + p2] = a;
                    }
                } else {
                    F[p2 * cols + (cols - 1 - qq)] = F[p * cols + qq];
                    F[p * cols + qq] = 0.f;
                }
            }
        }
    }
}

}  // namespace

cudaError_t factor_prepare(const float *H, int64_t cols, float damp, float *F, uint8_t *dead,
                           DeviceStatus *st, cudaStream_t s) {
    diag_sum_kernel<<<1, 1024, 0, s>>>(H, cols, damp, st);
    count_launch();
    if (cols % 4 == 0 && ((uintptr_t)H % 16) == 0 && ((uintptr_t)F % 16) == 0) {
        reverse_damp4_kernel<<<dim3((unsigned)((cols / 4 + 255) / 256), (unsigned)cols), 256, 0, s>>>(H, cols, F, dead,
                                                                                                     st);
    } else {
        dim3 grid((unsigned)((cols + 255) / 256 < 8 ? (cols + 255) / 256 : 8), (unsigned)cols);
        reverse_damp_kernel<<<grid, 256, 0, s>>>(H, cols, F, dead, st);
    }
    count_launch();
    return cudaGetLastError();
}

cudaError_t finite_check_launch(const void *X, bool bf16, int64_t n, DeviceStatus *st, unsigned int bit,
                                cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    const int esize = bf16 ? 2 : 4;
    const int64_t nbytes = n * esize;
    int64_t blocks = (nbytes / 16 + 255) / 256;
    if (blocks > 148 * 8) blocks = 148 * 8;
    if (blocks < 1) blocks = 1;
    finite_check_kernel<<<(unsigned)blocks, 256, 0, s>>>((const unsigned char *)X, nbytes, esize, st, bit);
    count_launch();
    return cudaGetLastError();
}

// Scratch of cholesky_lower_inplace: [Linv: NB x NB][Lhi, Llo: NB x NB][Phi, Plo: cols x NB]
// and, for the recursive path, [LThi, LTlo: cols x cols], the TF32 split of the
// solved panels (row stride cols).
constexpr int64_t REC_MIN = 1024;  // columns from which the recursive path is used
size_t cholesky_scratch_floats(int64_t cols) {
    size_t n = (size_t)3 * NB * NB + (size_t)2 * cols * NB;
    if (cols >= REC_MIN && cols % 4 == 0) n += (size_t)2 * cols * cols;
    return n;
}

namespace {

struct CholCtx {
    float *F;
    int64_t cols;
    DeviceStatus *st;
    float *Linv, *Lhi, *Llo, *Phi, *Plo, *LThi, *LTlo;
    float *Uinv;  // sweep block inverses (reversed), or null
    cudaStream_t s;
};

// One panel: diagonal block (factor + inverse), then the rows below solved,
// P <- P L^-T, written to F and, split, to (LThi, LTlo) or (Phi, Plo).
cudaError_t chol_panel(const CholCtx &c, int64_t k0, bool rec, bool p_split_ready = false) {
    const int64_t cols = c.cols;
    const int kb = (int)((cols - k0) < NB ? (cols - k0) : NB);
    const int64_t k1 = k0 + kb;
    const bool more = k1 < cols;
    const int64_t npanel = (cols + NB - 1) / NB;
    float *ur = c.Uinv ? c.Uinv + (npanel - 1 - k0 / NB) * NB * NB : nullptr;
    const int th = timing_begin(TK_DIAG, c.s);
    cudaError_t e = launch_pdl(potrf_diag_kernel, dim3(1), dim3(DIAG_THREADS), DIAG_SMEM, c.s, c.F, cols, k0, kb,
                               c.Linv, c.st, more ? c.Lhi : (float *)nullptr, c.Llo, ur);
    count_launch();
    timing_end(th, c.s, 2.0 * kb * kb * kb / 3.0);
    if (e != cudaSuccess || !more) return e;
    const int64_t rest = cols - k1;
    float *P = c.F + k1 * cols + k0;
    if (!p_split_ready && (e = split_tf32(P, rest, kb, cols, c.Phi, c.Plo, NB, c.s)) != cudaSuccess) return e;
    if (rec)
        return gemm3(rest, kb, kb, 1.f, c.Phi, c.Plo, NB, c.Lhi, c.Llo, NB, 0.f, P, cols, 0, c.LThi + k1 * cols + k0,
                     c.LTlo + k1 * cols + k0, cols, c.s);
    return gemm3(rest, kb, kb, 1.f, c.Phi, c.Plo, NB, c.Lhi, c.Llo, NB, 0.f, P, cols, 0, c.Phi, c.Plo, NB, c.s);
}

// Panels [a, b).  On entry the columns of these panels (rows from the first of
// them down) carry every update from the columns left of panel a.  The left
// half is factored, its whole contribution to the right half is applied as
// one GEMM (K = the left half's width), then the right half is factored.
// p_split_ready: the split of panel a's rows below its diagonal block is
// already in (Phi, Plo), written by the GEMM that last updated the panel.
cudaError_t chol_rec(const CholCtx &c, int64_t a, int64_t b, bool p_split_ready) {
    if (b - a == 1) return chol_panel(c, a * NB, true, p_split_ready);
    const int64_t m = (a + b) / 2;
    cudaError_t e = chol_rec(c, a, m, p_split_ready);
    if (e != cudaSuccess) return e;
    const int64_t c0 = a * NB, cm = m * NB, c1 = (b * NB < c.cols) ? b * NB : c.cols;
    // The update of panels [m, b) is the last one panel m receives (the next
    // launch factors it), so its epilogue also emits the split of panel m's rows
    // below the diagonal block: C rows >= NB, columns < NB.
    const bool emit = cm + NB < c.cols;
    e = gemm3(c.cols - cm, c1 - cm, cm - c0, -1.f, c.LThi + cm * c.cols + c0, c.LTlo + cm * c.cols + c0, c.cols,
              c.LThi + cm * c.cols + c0, c.LTlo + cm * c.cols + c0, c.cols, 1.f, c.F + cm * c.cols + cm, c.cols, 1,
              emit ? c.Phi : nullptr, emit ? c.Plo : nullptr, NB, c.s, NB, NB);
    if (e != cudaSuccess) return e;
    return chol_rec(c, m, b, emit);
}

}  // namespace

// Blocked Cholesky, panel width NB.  Per panel: the diagonal block and its
// inverse (one CTA) and the panel below, P <- P L_kk^-T.  The trailing updates
// A22 -= P P^T run on the tensor cores with float32 accuracy (3xTF32) when the
// row stride allows TMA (cols % 4 == 0): for cols >= REC_MIN in the recursive
// order above (few large GEMMs), else right-looking after every panel.
// Without TMA (cols % 4 != 0) both products run on the float32 SIMT GEMM.
cudaError_t cholesky_lower_inplace(float *F, int64_t cols, DeviceStatus *st, float *scratch, cudaStream_t s,
                                   float *Uinv, int block) {
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(potrf_diag_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)DIAG_SMEM);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    CholCtx c;
    c.F = F;
    c.cols = cols;
    c.st = st;
    c.Linv = scratch;
    c.Lhi = c.Linv + NB * NB;
    c.Llo = c.Lhi + NB * NB;
    c.Phi = c.Llo + NB * NB;
    c.Plo = c.Phi + cols * NB;
    c.LThi = c.Plo + cols * NB;
    c.LTlo = c.LThi + cols * cols;
    // Diagonal-block inverses for the sweep come out of the factorization when
    // its panels coincide with the sweep's blocks (reversed order).
    c.Uinv = (Uinv && block == NB && (cols % NB) == 0) ? Uinv : nullptr;
    c.s = s;
    const bool tc = (cols % 4) == 0;
    const int64_t npanel = (cols + NB - 1) / NB;
    if (tc && cols >= REC_MIN) {
        cudaError_t e = chol_rec(c, 0, npanel, false);
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
    for (int64_t k0 = 0; k0 < cols; k0 += NB) {
        const int kb = (int)((cols - k0) < NB ? (cols - k0) : NB);
        const int64_t k1 = k0 + kb;
        cudaError_t e;
        if (tc) {
            if ((e = chol_panel(c, k0, false)) != cudaSuccess) return e;
            if (k1 >= cols) break;
            // A22 -= P P^T (tiles touching the lower triangle).
            const int64_t rest = cols - k1;
            if ((e = gemm3(rest, rest, kb, -1.f, c.Phi, c.Plo, NB, c.Phi, c.Plo, NB, 1.f, F + k1 * cols + k1, cols, 1,
                           nullptr, nullptr, 0, s)) != cudaSuccess)
                return e;
        } else {
            float *ur = c.Uinv ? c.Uinv + (npanel - 1 - k0 / NB) * NB * NB : nullptr;
            const int th = timing_begin(TK_DIAG, s);
            potrf_diag_kernel<<<1, DIAG_THREADS, DIAG_SMEM, s>>>(F, cols, k0, kb, c.Linv, st, nullptr, nullptr, ur);
            count_launch();
            timing_end(th, s, 2.0 * kb * kb * kb / 3.0);
            if (k1 >= cols) break;
            const int64_t rest = cols - k1;
            float *P = F + k1 * cols + k0;  // rest x kb panel below the diagonal block
            // P <- P L^-T in place: each 128-row tile reads its rows completely before writing them.
            e = sgemm<float>(rest, kb, kb, 1.f, P, cols, false, c.Linv, NB, true, 0.f, P, cols, 0, s);
            if (e != cudaSuccess) return e;
            e = sgemm<float>(rest, rest, kb, -1.f, P, cols, false, P, cols, true, 1.f, F + k1 * cols + k1, cols,
                             /*tri=*/1, s);
            if (e != cudaSuccess) return e;
        }
    }
    return cudaGetLastError();
}

cudaError_t factor_finalize(float *F, int64_t cols, cudaStream_t s) {
    if (cols % 4 == 0 && ((uintptr_t)F % 16) == 0) {
        finalize4_kernel<<<dim3((unsigned)((cols / 4 + 255) / 256), (unsigned)cols), 256, 0, s>>>(F, cols);
        count_launch();
        return cudaGetLastError();
    }
    dim3 grid((unsigned)((cols + 255) / 256 < 8 ? (cols + 255) / 256 : 8), (unsigned)cols);
    finalize_kernel<<<grid, 256, 0, s>>>(F, cols);
    count_launch();
    return cudaGetLastError();
}

size_t factor_scratch_bytes(int64_t cols) {
    return align_up(sizeof(DeviceStatus)) + align_up(cholesky_scratch_floats(cols) * sizeof(float));
}

}  // namespace gq
