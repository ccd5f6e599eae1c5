// The GPTQ column sweep ([GPTQ-wiki] "Enfoque Técnico"; grid per [LowBit] section 1).
//
// Work split.  Columns are processed in blocks of `bw` <= 128 columns.  With F
// the upper factor of H_d = F F^T and U = F^-1 (upper triangular), the weights
// of block b as updated by every earlier column are
//     W_blk + ΔW[:, <s] F[<s, blk] Uinv_b,   Uinv_b = F[blk, blk]^-1 = U[blk, blk],
// with ΔW = W - Ŵ.  V = F blockdiag(Uinv_b) (rows above each diagonal block) is
// formed once, transposed and split into TF32 parts (VThi + VTlo), the operand
// layout of the tensor-core GEMM.  The buffer D (rows x cols float32, in the
// workspace) holds, for a block not yet swept, sum over earlier blocks of
// ΔW_prev V_prev,blk, accumulated by the deferred trailing GEMMs; once a block
// is swept its columns of D hold the TF32 hi part of ΔW and those of DL the lo
// part.  Inside the block the ordinary per-column update runs with Uinv_b.
//
// Kernel layout: see sweep_rows_kernel (four lanes per row, 8 rows per warp,
// 32 rows per CTA, every warp an independent chain over the block's columns).
#include "common.cuh"

namespace gq {
namespace {

constexpr int ROWS = 32;                   // rows per CTA (4 warps x 8 rows)
constexpr int SEG = 32;                    // block columns per lane (a quarter of the block)
constexpr int MAXB = 128;                  // max block width
constexpr int MAXG = MAXB / 32;            // max groups per block (group >= 32)

// Word w of the little-endian bitstream of BITS-bit values v[0..]: bits [32w, 32w + 32).
template <int BITS>
__device__ __forceinline__ uint32_t pack_word(const uint8_t *v, int w, int n) {
    uint32_t word = 0;
    const int k_lo = (32 * w) / BITS, k_hi = (32 * w + 31) / BITS;
    for (int k = k_lo; k <= k_hi && k < n; ++k) {
        const int pos = k * BITS - 32 * w;
        const uint32_t x = v[k];
        if (pos >= 0)
            word |= (pos < 32) ? (x << pos) : 0u;
        else
            word |= x >> (-pos);
    }
    return word;
}

template <typename TW>
__device__ __forceinline__ void load8(const TW *p, float (&o)[8]);
template <>
__device__ __forceinline__ void load8<float>(const float *p, float (&o)[8]) {
    const float4 a = *reinterpret_cast<const float4 *>(p), b = *reinterpret_cast<const float4 *>(p + 4);
    o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w; o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
}
template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16 *p, float (&o)[8]) {
    const uint4 v = *reinterpret_cast<const uint4 *>(p);
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        o[2 * i] = __uint_as_float(u[i] << 16);
        o[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
    }
}

template <typename TW>
__device__ __forceinline__ void load32(const TW *p, float (&o)[SEG]) {
#pragma unroll
    for (int c = 0; c < SEG; c += 8) {
        float t[8];
        load8<TW>(p + c, t);
#pragma unroll
        for (int i = 0; i < 8; ++i) o[c + i] = t[i];
    }
}

// rint(w / s) for the IEEE-rounded quotient w / s, without a division:
// inv_s = RN(1/s) and the FMA-corrected quotient (quotient_rn), then
// round-half-to-even.
__device__ __forceinline__ float rint_div(float w, float s, float inv_s) { return rintf(quotient_rn(w, s, inv_s)); }

__device__ __forceinline__ float tf32_hi(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

// The block sweep, four lanes per row.  A warp holds 8 rows; lane
// 4 r + q holds columns [32 q, 32 q + 32) of the block of row r in registers,
// so every warp of the CTA (4 warps, 32 rows) runs its own rows' column chain
// and no barrier is needed inside the block.  At column j = 32 qo + jj the
// lane of quarter qo quantizes its row's weight, the error goes to the row's
// other lanes by one shuffle, and every lane updates its 32 columns with row j
// of Uinv_b (shared memory; the quarters are 36 floats apart so the four
// quarter addresses of a warp's load fall in different banks).  Columns left
// of j meet zeros of the triangular Uinv_b and column j itself is no longer
// read, so the update needs no predicate.  At a group's first column its
// min / max is reduced over the row's lanes by two shuffles.  The epilogue
// recomputes ŵ from the codes and the lane's grid and writes ΔW = w0 - ŵ
// (split), the optional codes / Ŵ / row errors, the scales, the packed words of
// its own 32 columns (32 b bits = b words) and, through shared memory, the
// packed zero points of the CTA's 32 rows.
constexpr int QLD = 36;  // shared-memory floats per quarter row of Uinv_b

struct SweepRowsSmem {
    float U[MAXB][4 * QLD];   // Uinv_b, quarter-skewed; zero below the diagonal and beyond bw
    float fdiag[MAXB];        // F_jj = 1 / U_jj
    uint8_t zeros[MAXG][ROWS];
};

template <int BITS, typename TW>
__global__ void __launch_bounds__(128) sweep_rows_kernel(const TW *__restrict__ W, int64_t rows, int64_t cols,
                                                         int64_t c0, int bw, const float *__restrict__ Uinv,
                                                         const float *__restrict__ F, const uint8_t *__restrict__ dead,
                                                         int group, float *__restrict__ D, float *__restrict__ DL,
                                                         int32_t *__restrict__ qweight, float *__restrict__ scales,
                                                         int32_t *__restrict__ qzeros, uint8_t *__restrict__ codes,
                                                         float *__restrict__ W_hat, float *__restrict__ row_err) {
    pdl_trigger();
    pdl_wait();  // D was last updated by the previous kernel
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SweepRowsSmem &sm = *reinterpret_cast<SweepRowsSmem *>(smem_raw);
    constexpr float maxq = (float)((1 << BITS) - 1);
    const unsigned full = 0xffffffffu;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rr = warp * 8 + (lane >> 2);  // row within the CTA
    const int q = lane & 3;                 // quarter of the block this lane holds
    const int64_t row0 = (int64_t)blockIdx.x * ROWS;
    const int64_t row = row0 + rr;
    const bool row_on = row < rows;
    const int nq = bw / SEG;                // quarters in use
    const bool q_on = q < nq;
    const int gq = group / SEG;             // quarters per group

    // Uinv_b into shared memory (quarter-skewed rows) with 16-byte asynchronous copies.
    for (int idx = threadIdx.x; idx < MAXB * MAXB / 4; idx += 128) {
        const int i = idx / (MAXB / 4), j4 = (idx % (MAXB / 4)) * 4;
        float *dst = &sm.U[i][(j4 / SEG) * QLD + (j4 % SEG)];
        if (i < bw && j4 < bw) {
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                         "l"(Uinv + (int64_t)i * bw + j4)
                         : "memory");
        } else {
            *reinterpret_cast<float4 *>(dst) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    for (int i = threadIdx.x; i < MAXB; i += 128) sm.fdiag[i] = (i < bw) ? F[(c0 + i) * cols + c0 + i] : 1.f;

    // This lane's 32 columns: w0 (dead inputs zero) and w = w0 + D.
    float w[SEG];
    uint32_t dmask = 0;
#pragma unroll
    for (int c = 0; c < SEG; ++c) w[c] = 0.f;
    if (q_on && row_on) {
        float w0[SEG], t[SEG];
        load32<TW>(W + row * cols + c0 + q * SEG, w0);
        load32<float>(D + row * cols + c0 + q * SEG, t);
        if (dead) {
#pragma unroll
            for (int c = 0; c < SEG; ++c) dmask |= (dead[c0 + q * SEG + c] != 0 ? 1u : 0u) << c;
        }
#pragma unroll
        for (int c = 0; c < SEG; ++c) w[c] = (((dmask >> c) & 1u) ? 0.f : w0[c]) + t[c];
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncthreads();

    float my_s = 1.f, my_inv = 1.f, my_z = 0.f;  // the grid of this lane's quarter
    uint32_t cw[SEG / 4];                          // codes of this lane's columns, 8 bits each
#pragma unroll
    for (int k = 0; k < SEG / 4; ++k) cw[k] = 0u;
    float e2 = 0.f;
    const int src_base = lane & ~3;

    for (int qo = 0; qo < nq; ++qo) {
        if (qo % gq == 0) {
            // A group starts: min / max over its quarters of the row, as updated by every earlier column.
            const bool in_g = q >= qo && q < qo + gq && q_on;
            float lo = 3.402823466e38f, hi = -3.402823466e38f;
            if (in_g) {
#pragma unroll
                for (int c = 0; c < SEG; ++c) {
                    lo = fminf(lo, w[c]);
                    hi = fmaxf(hi, w[c]);
                }
            }
            lo = fminf(lo, __shfl_xor_sync(full, lo, 1));
            hi = fmaxf(hi, __shfl_xor_sync(full, hi, 1));
            lo = fminf(lo, __shfl_xor_sync(full, lo, 2));
            hi = fmaxf(hi, __shfl_xor_sync(full, hi, 2));
            float xmin = fminf(lo, 0.f), xmax = fmaxf(hi, 0.f);
            if (xmin == 0.f && xmax == 0.f) {
                xmin = -1.f;
                xmax = 1.f;
            }
            const float sc = __fdiv_rn(xmax - xmin, maxq);
            if (in_g) {
                my_s = sc;
                my_inv = __fdiv_rn(1.f, sc);
                my_z = rintf(__fdiv_rn(-xmin, sc));
            }
            if (q == qo) sm.zeros[(qo * SEG) / group][rr] = (uint8_t)rintf(__fdiv_rn(-xmin, sc));
        }
        const bool owner = (q == qo);
        const float *ub = &sm.U[qo * SEG][q * QLD];
#pragma unroll
        for (int jj = 0; jj < SEG; ++jj) {
            float e = 0.f;
            if (owner) {
                const float wv = w[jj];
                const float qv = fminf(fmaxf(rint_div(wv, my_s, my_inv) + my_z, 0.f), maxq);
                cw[jj / 4] |= ((uint32_t)qv) << (8 * (jj % 4));
                e = (wv - my_s * (qv - my_z)) * sm.fdiag[qo * SEG + jj];
                e2 = fmaf(e, e, e2);
            }
            e = __shfl_sync(full, e, src_base | qo);
            const float *ur = ub + jj * (4 * QLD);
#pragma unroll
            for (int c4 = 0; c4 < SEG; c4 += 4) {
                const float4 u = *reinterpret_cast<const float4 *>(ur + c4);
                w[c4 + 0] = fmaf(-e, u.x, w[c4 + 0]);
                w[c4 + 1] = fmaf(-e, u.y, w[c4 + 1]);
                w[c4 + 2] = fmaf(-e, u.z, w[c4 + 2]);
                w[c4 + 3] = fmaf(-e, u.w, w[c4 + 3]);
            }
        }
    }

    // Row errors: the owners' sums over the row's lanes.
    e2 += __shfl_xor_sync(full, e2, 1);
    e2 += __shfl_xor_sync(full, e2, 2);
    if (q == 0 && row_on && row_err) row_err[row] += e2;

    if (q_on && row_on) {
        // ΔW = w0 - ŵ (split), Ŵ, codes.
        float w0[SEG];
        load32<TW>(W + row * cols + c0 + q * SEG, w0);
        float *dp = D + row * cols + c0 + q * SEG;
        float *lp = DL + row * cols + c0 + q * SEG;
#pragma unroll
        for (int c = 0; c < SEG; c += 4) {
            float dh[4], dl[4], wq[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float qv = (float)((cw[(c + u) / 4] >> (8 * ((c + u) % 4))) & 0xffu);
                wq[u] = my_s * (qv - my_z);
                const float dw = (((dmask >> (c + u)) & 1u) ? 0.f : w0[c + u]) - wq[u];
                dh[u] = tf32_hi(dw);
                dl[u] = dw - dh[u];
            }
            *reinterpret_cast<float4 *>(dp + c) = make_float4(dh[0], dh[1], dh[2], dh[3]);
            *reinterpret_cast<float4 *>(lp + c) = make_float4(dl[0], dl[1], dl[2], dl[3]);
            if (W_hat)
                *reinterpret_cast<float4 *>(W_hat + row * cols + c0 + q * SEG + c) =
                    make_float4(wq[0], wq[1], wq[2], wq[3]);
        }
        if (codes) {
            uint8_t *dst = codes + row * cols + c0 + q * SEG;
            if (((uintptr_t)dst & 15) == 0) {
                reinterpret_cast<uint4 *>(dst)[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
                reinterpret_cast<uint4 *>(dst)[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
            } else {  // the library only requires 4-byte alignment of codes
#pragma unroll
                for (int i = 0; i < 8; ++i) reinterpret_cast<uint32_t *>(dst)[i] = cw[i];
            }
        }
        // The group's scale, written by the lane of its first quarter.
        if (q % gq == 0) scales[((c0 + q * SEG) / group) * rows + row] = my_s;
        // qweight: the lane's 32 codes are words [q BITS, q BITS + BITS) of the block's stream.
        uint32_t words[BITS];
#pragma unroll
        for (int k = 0; k < BITS; ++k) words[k] = 0u;
#pragma unroll
        for (int i = 0; i < SEG; ++i) {
            const uint32_t cv = (cw[i / 4] >> (8 * (i % 4))) & 0xffu;
            const int pos = i * BITS, wi = pos / 32, sh = pos % 32;
            words[wi] |= cv << sh;
            if (sh + BITS > 32) words[wi + 1] |= cv >> (32 - sh);
        }
        const int64_t w0i = c0 * BITS / 32 + q * BITS;
#pragma unroll
        for (int k = 0; k < BITS; ++k) qweight[(w0i + k) * rows + row] = (int32_t)words[k];
    }
    __syncthreads();
    // qzeros [cols/group][rows*BITS/32]: BITS words per group for these 32 rows.
    const int ng = bw / group;
    const int64_t zw = rows * BITS / 32;
    for (int idx = threadIdx.x; idx < ng * BITS; idx += 128) {
        const int g = idx / BITS, wi = idx % BITS;
        qzeros[((c0 / group) + g) * zw + row0 * BITS / 32 + wi] = (int32_t)pack_word<BITS>(sm.zeros[g], wi, ROWS);
    }
}

// VT[s0 + n][m] = sum_k Uinv_b[k][n] F[m][s0 + k] for m < s0: the transpose of
// V[:, blk_b] = F[:, blk_b] Uinv_b above each diagonal block b, so that the
// deferred update of block b from the earlier columns is ΔW_prev V_prev,b with
// V given K-contiguous, and written as its TF32 split.  One CTA per
// (128-column m-tile, block b), 256 threads, 8 x 8 outputs each; stores run
// along m (coalesced).
__global__ void __launch_bounds__(256) premultiply_t_kernel(const float *__restrict__ F, int64_t cols, int block,
                                                            const float *__restrict__ Uinv, float *__restrict__ VThi,
                                                            float *__restrict__ VTlo) {
    __shared__ __align__(16) float As[16][128 + 4];  // As[k][n] = Uinv_b[k][n]
    __shared__ __align__(16) float Bs[16][128 + 4];  // Bs[k][m] = F[m][s0 + k]
    const int b = blockIdx.y;
    const int64_t s0 = (int64_t)b * block;
    const int bw = (int)((cols - s0) < block ? (cols - s0) : block);
    const int64_t m0 = (int64_t)blockIdx.x * 128;
    if (m0 >= s0) return;  // only columns left of the diagonal block
    const float *Ub = Uinv + s0 * block;  // bw x bw, row stride bw
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
    for (int k0 = 0; k0 < bw; k0 += 16) {
        for (int idx = threadIdx.x; idx < 16 * 128; idx += 256) {
            const int kk = idx / 128, n = idx % 128;
            As[kk][n] = (k0 + kk < bw && n < bw) ? Ub[(int64_t)(k0 + kk) * bw + n] : 0.f;
            const int m = idx / 16, k = idx % 16;
            const int64_t gm = m0 + m;
            Bs[k][m] = (gm < s0 && k0 + k < bw) ? F[gm * cols + s0 + k0 + k] : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            float a[8], bb[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                a[i] = As[k][ty * 4 + i];
                a[4 + i] = As[k][64 + ty * 4 + i];
                bb[i] = Bs[k][tx * 4 + i];
                bb[4 + i] = Bs[k][64 + tx * 4 + i];
            }
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], bb[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int n = (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
        if (n >= bw) continue;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int64_t m = m0 + (j < 4 ? tx * 4 + j : 64 + tx * 4 + (j - 4));
            if (m >= s0) continue;
            const float v = acc[i][j];
            const float h = tf32_hi(v);
            VThi[(s0 + n) * cols + m] = h;
            VTlo[(s0 + n) * cols + m] = v - h;
        }
    }
}

// Inverse of each bw x bw diagonal block of the upper factor F (back substitution,
// one column per thread).  Out: Uinv[b][i][j], row-major bw x bw per block.
__global__ void __launch_bounds__(128) block_inverse_kernel(const float *__restrict__ F, int64_t cols,
                                                            int block, float *__restrict__ Uinv) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    float *T = reinterpret_cast<float *>(smem_raw);   // [MAXB][MAXB + 1]
    float *Y = T + MAXB * (MAXB + 1);                  // [MAXB][MAXB + 1]
    const int64_t s0 = (int64_t)blockIdx.x * block;
    const int bw = (int)((cols - s0) < block ? (cols - s0) : block);
    for (int idx = threadIdx.x; idx < bw * bw; idx += blockDim.x) {
        const int i = idx / bw, j = idx % bw;
        T[i * (MAXB + 1) + j] = (j >= i) ? F[(s0 + i) * cols + s0 + j] : 0.f;
    }
    __syncthreads();
    const int c = threadIdx.x;
    if (c < bw) {
        for (int i = bw - 1; i > c; --i) Y[i * (MAXB + 1) + c] = 0.f;
        Y[c * (MAXB + 1) + c] = 1.f / T[c * (MAXB + 1) + c];
        for (int i = c - 1; i >= 0; --i) {
            float acc = 0.f;
            for (int k = i + 1; k <= c; ++k) acc = fmaf(T[i * (MAXB + 1) + k], Y[k * (MAXB + 1) + c], acc);
            Y[i * (MAXB + 1) + c] = -acc / T[i * (MAXB + 1) + i];
        }
    }
    __syncthreads();
    float *out = Uinv + (int64_t)blockIdx.x * block * block;
    for (int idx = threadIdx.x; idx < bw * bw; idx += blockDim.x) {
        const int i = idx / bw, j = idx % bw;
        out[idx] = Y[i * (MAXB + 1) + j];
    }
}

template <int BITS, typename TW>
cudaError_t launch_sweep(const TW *W, int64_t rows, int64_t cols, int64_t c0, int bw, const float *Uinv,
                         const float *F, const uint8_t *dead, int group, float *D, float *DL, int32_t *qweight,
                         float *scales,
                         int32_t *qzeros, uint8_t *codes, float *W_hat, float *row_err, cudaStream_t s) {
    const size_t smem = sizeof(SweepRowsSmem);
    static bool attr_set = false;  // per template instance
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(sweep_rows_kernel<BITS, TW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const int th = timing_begin(TK_SWEEP, s);
    const cudaError_t e = launch_pdl(sweep_rows_kernel<BITS, TW>, dim3((unsigned)((rows + ROWS - 1) / ROWS)), dim3(128),
                                     smem, s, W, rows, cols, c0, bw, Uinv, F, dead, group, D, DL, qweight, scales,
                                     qzeros, codes, W_hat, row_err);
    count_launch();
    timing_end(th, s, (double)rows * bw * (bw - 1));
    return e;
}

}  // namespace

cudaError_t block_inverses(const float *F, int64_t cols, int block, float *Uinv, cudaStream_t s) {
    const size_t smem = 2 * MAXB * (MAXB + 1) * sizeof(float);
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(block_inverse_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const int64_t nblk = (cols + block - 1) / block;
    block_inverse_kernel<<<(unsigned)nblk, 128, smem, s>>>(F, cols, block, Uinv);
    count_launch();
    return cudaGetLastError();
}

cudaError_t premultiply_t(const float *F, int64_t cols, int block, const float *Uinv, float *VThi, float *VTlo,
                          cudaStream_t s) {
    const int64_t nblk = (cols + block - 1) / block;
    if (nblk < 2) return cudaSuccess;
    dim3 grid((unsigned)(((nblk - 1) * block + 127) / 128), (unsigned)nblk);
    premultiply_t_kernel<<<grid, 256, 0, s>>>(F, cols, block, Uinv, VThi, VTlo);
    count_launch();
    return cudaGetLastError();
}

cudaError_t sweep_block_launch(const void *W, bool w_bf16, int64_t rows, int64_t cols, int64_t c0, int bw,
                               const float *Uinv_blk, const float *F, const uint8_t *dead, int bits, int group,
                               float *D, float *DL, int32_t *qweight, float *scales, int32_t *qzeros, uint8_t *codes,
                               float *W_hat, float *row_err, cudaStream_t s) {
#define GQ_SWEEP_CASE(B)                                                                                         \
    if (bits == B) {                                                                                             \
        if (w_bf16)                                                                                              \
            return launch_sweep<B, __nv_bfloat16>((const __nv_bfloat16 *)W, rows, cols, c0, bw, Uinv_blk, F, dead, \
                                                  group, D, DL, qweight, scales, qzeros, codes, W_hat, row_err, s); \
        return launch_sweep<B, float>((const float *)W, rows, cols, c0, bw, Uinv_blk, F, dead, group, D, DL,       \
                                      qweight, scales, qzeros, codes, W_hat, row_err, s);                        \
    }
    GQ_SWEEP_CASE(2)
    GQ_SWEEP_CASE(3)
    GQ_SWEEP_CASE(4)
#undef GQ_SWEEP_CASE
    return cudaErrorInvalidValue;
}

}  // namespace gq
