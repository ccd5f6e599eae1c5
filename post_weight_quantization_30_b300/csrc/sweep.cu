// The GPTQ column sweep ([GPTQ-wiki] "Enfoque Técnico"; grid per [LowBit] section 1).
//
// Work split.  Columns are processed in blocks of `bw` <= 128 columns.  The
// buffer D (rows x cols float32, in the workspace) holds, for a block not yet
// swept, T = ΔW[:, <s] F[<s, blk] accumulated by the deferred trailing GEMMs
// (F = the upper factor of H_d = F F^T, ΔW = W - Ŵ); once a block is swept its
// columns of D hold ΔW.  Because U = F^-1 is upper triangular, the weights of
// the block as updated by every earlier column are
//     W_blk + T_blk Uinv_blk,   Uinv_blk = F[blk, blk]^-1 = U[blk, blk],
// and inside the block the ordinary per-column update runs with Uinv_blk.
//
// Kernel layout.  One CTA = 32 output rows x one block, 8 warps x 4 rows.  Lane
// l of a warp owns block columns 4l..4l+3 of its 4 rows, in registers.  Per
// column j: the owning lane quantizes (IEEE division, round-half-even), the
// scaled error e_j = (w_j - ŵ_j) / U_jj is broadcast by a warp shuffle, and
// every lane updates its columns with row j of Uinv_blk (shared memory,
// broadcast to all warps).  Group min/max are warp-shuffle butterflies.  The
// epilogue writes ΔW back to D, the optional codes / Ŵ / row errors, the
// scales, and packs codes and zero points into 32-bit words (coalesced
// word-rows of 32 output rows).
#include <cfloat>

#include "common.cuh"

namespace gq {
namespace {

constexpr int ROWS = 32;         // rows per CTA
constexpr int RPW = 4;           // rows per warp
constexpr int MAXB = 128;        // max block width
constexpr int MAXG = MAXB / 32;  // max groups per block (group >= 32)

struct SweepSmem {
    float U[MAXB][MAXB];                 // Uinv_blk, upper triangle (lower part zero)
    uint8_t codes[ROWS][MAXB + 4];       // staging for the qweight packing
    uint8_t zeros[MAXG][ROWS];           // staging for the qzeros packing
};

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
__device__ __forceinline__ void load4(const TW *p, float (&o)[4]);
template <>
__device__ __forceinline__ void load4<float>(const float *p, float (&o)[4]) {
    float4 v = *reinterpret_cast<const float4 *>(p);
    o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
}
template <>
__device__ __forceinline__ void load4<__nv_bfloat16>(const __nv_bfloat16 *p, float (&o)[4]) {
    uint2 v = *reinterpret_cast<const uint2 *>(p);
    o[0] = __uint_as_float(v.x << 16);
    o[1] = __uint_as_float(v.x & 0xffff0000u);
    o[2] = __uint_as_float(v.y << 16);
    o[3] = __uint_as_float(v.y & 0xffff0000u);
}

template <int BITS, typename TW>
__global__ void __launch_bounds__(256) sweep_kernel(const TW *__restrict__ W, int64_t rows, int64_t cols,
                                                    int64_t c0, int bw, const float *__restrict__ Uinv,
                                                    const uint8_t *__restrict__ dead, int group,
                                                    float *__restrict__ D, int32_t *__restrict__ qweight,
                                                    float *__restrict__ scales, int32_t *__restrict__ qzeros,
                                                    uint8_t *__restrict__ codes, float *__restrict__ W_hat,
                                                    float *__restrict__ row_err) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SweepSmem &sm = *reinterpret_cast<SweepSmem *>(smem_raw);
    constexpr float maxq = (float)((1 << BITS) - 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row0 = (int64_t)blockIdx.x * ROWS;
    const int64_t rbase = row0 + warp * RPW;
    const int cl = lane * 4;               // first block column owned by this lane
    const bool lane_on = cl < bw;

    // Uinv_blk -> shared memory (bw x bw, row stride MAXB).
    for (int idx = threadIdx.x; idx < MAXB * MAXB / 4; idx += blockDim.x) {
        const int i = idx / (MAXB / 4), j4 = (idx % (MAXB / 4)) * 4;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (i < bw && j4 < bw) v = *reinterpret_cast<const float4 *>(Uinv + (int64_t)i * bw + j4);
        *reinterpret_cast<float4 *>(&sm.U[i][j4]) = v;
    }

    // Weights of the block and the accumulated T = ΔW_{<s} F_{<s, blk}.
    float w[RPW][4], t[RPW][4];
    uint8_t dmask[4] = {0, 0, 0, 0};
    if (dead && lane_on) {
#pragma unroll
        for (int c = 0; c < 4; ++c) dmask[c] = dead[c0 + cl + c];
    }
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
        const int64_t row = rbase + r;
        if (lane_on && row < rows) {
            load4<TW>(W + row * cols + c0 + cl, w[r]);
            float4 tv = *reinterpret_cast<const float4 *>(D + row * cols + c0 + cl);
            t[r][0] = tv.x; t[r][1] = tv.y; t[r][2] = tv.z; t[r][3] = tv.w;
        } else {
#pragma unroll
            for (int c = 0; c < 4; ++c) w[r][c] = t[r][c] = 0.f;
        }
#pragma unroll
        for (int c = 0; c < 4; ++c)
            if (dmask[c]) w[r][c] = 0.f;
    }
    __syncthreads();

    // w += T Uinv_blk (row vector times upper-triangular block).
    for (int o = 0; o < bw / 4; ++o) {
#pragma unroll
        for (int ci = 0; ci < 4; ++ci) {
            const int i = o * 4 + ci;
            const float4 u = *reinterpret_cast<const float4 *>(&sm.U[i][cl]);
#pragma unroll
            for (int r = 0; r < RPW; ++r) {
                const float ti = __shfl_sync(0xffffffffu, t[r][ci], o);
                w[r][0] = fmaf(ti, u.x, w[r][0]);
                w[r][1] = fmaf(ti, u.y, w[r][1]);
                w[r][2] = fmaf(ti, u.z, w[r][2]);
                w[r][3] = fmaf(ti, u.w, w[r][3]);
            }
        }
    }

    float s[RPW], z[RPW], e2[RPW], wq[RPW][4];
    uint32_t q4[RPW];
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
        s[r] = 1.f; z[r] = 0.f; e2[r] = 0.f; q4[r] = 0u;
#pragma unroll
        for (int c = 0; c < 4; ++c) wq[r][c] = 0.f;
    }

    for (int o = 0; o < bw / 4; ++o) {
#pragma unroll
        for (int ci = 0; ci < 4; ++ci) {
            const int j = o * 4 + ci;
            if (ci == 0 && (j % group) == 0) {
                // Group parameters from the current weights of columns [j, j + group).
#pragma unroll
                for (int r = 0; r < RPW; ++r) {
                    float lo = FLT_MAX, hi = -FLT_MAX;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int col = cl + c;
                        if (col >= j && col < j + group && col < bw) {
                            lo = fminf(lo, w[r][c]);
                            hi = fmaxf(hi, w[r][c]);
                        }
                    }
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) {
                        lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, off));
                        hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, off));
                    }
                    float xmin = fminf(lo, 0.f), xmax = fmaxf(hi, 0.f);
                    if (xmin == 0.f && xmax == 0.f) {
                        xmin = -1.f;
                        xmax = 1.f;
                    }
                    s[r] = __fdiv_rn(xmax - xmin, maxq);
                    z[r] = rintf(__fdiv_rn(-xmin, s[r]));
                }
                const int g = j / group;
                if (lane == 0) {
                    const int64_t gi = (c0 + j) / group;
                    if (rbase < rows)
                        *reinterpret_cast<float4 *>(scales + gi * rows + rbase) = make_float4(s[0], s[1], s[2], s[3]);
#pragma unroll
                    for (int r = 0; r < RPW; ++r) sm.zeros[g][warp * RPW + r] = (uint8_t)z[r];
                }
            }
            const float udiag = sm.U[j][j];
            float e[RPW] = {0.f, 0.f, 0.f, 0.f};
            if (lane == o) {
#pragma unroll
                for (int r = 0; r < RPW; ++r) {
                    const float wv = w[r][ci];
                    const float q = fminf(fmaxf(rintf(__fdiv_rn(wv, s[r])) + z[r], 0.f), maxq);
                    const float dq = s[r] * (q - z[r]);
                    wq[r][ci] = dq;
                    q4[r] |= ((uint32_t)q) << (8 * ci);
                    e[r] = __fdiv_rn(wv - dq, udiag);
                    e2[r] = fmaf(e[r], e[r], e2[r]);
                }
            }
            const float4 u = *reinterpret_cast<const float4 *>(&sm.U[j][cl]);
#pragma unroll
            for (int r = 0; r < RPW; ++r) {
                const float eb = __shfl_sync(0xffffffffu, e[r], o);
                // Uinv is upper triangular: columns < j get zero updates; column j
                // itself is already quantized and its working value is unused.
                w[r][0] = fmaf(-eb, u.x, w[r][0]);
                w[r][1] = fmaf(-eb, u.y, w[r][1]);
                w[r][2] = fmaf(-eb, u.z, w[r][2]);
                w[r][3] = fmaf(-eb, u.w, w[r][3]);
            }
        }
    }

    // Epilogue: ΔW -> D, optional outputs, staging for packing.
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
        const int64_t row = rbase + r;
        float err = e2[r];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) err += __shfl_xor_sync(0xffffffffu, err, off);
        if (row >= rows) continue;
        if (lane == 0 && row_err) row_err[row] += err;
        if (!lane_on) continue;
        float w0[4];
        load4<TW>(W + row * cols + c0 + cl, w0);
#pragma unroll
        for (int c = 0; c < 4; ++c)
            if (dmask[c]) w0[c] = 0.f;
        *reinterpret_cast<float4 *>(D + row * cols + c0 + cl) =
            make_float4(w0[0] - wq[r][0], w0[1] - wq[r][1], w0[2] - wq[r][2], w0[3] - wq[r][3]);
        if (W_hat)
            *reinterpret_cast<float4 *>(W_hat + row * cols + c0 + cl) = make_float4(wq[r][0], wq[r][1], wq[r][2], wq[r][3]);
        if (codes) *reinterpret_cast<uint32_t *>(codes + row * cols + c0 + cl) = q4[r];
        *reinterpret_cast<uint32_t *>(&sm.codes[warp * RPW + r][cl]) = q4[r];
    }
    __syncthreads();

    // qweight [cols*BITS/32][rows]: words of this block, one word-row of 32 rows at a time.
    const int nw = bw * BITS / 32;
    const int64_t w0i = c0 * BITS / 32;
    for (int idx = threadIdx.x; idx < nw * ROWS; idx += blockDim.x) {
        const int wi = idx / ROWS, rr = idx % ROWS;
        if (row0 + rr < rows)
            qweight[(w0i + wi) * rows + row0 + rr] = (int32_t)pack_word<BITS>(sm.codes[rr], wi, bw);
    }
    // qzeros [cols/group][rows*BITS/32]: BITS words per group for these 32 rows.
    const int ng = bw / group;
    const int64_t zw = rows * BITS / 32;
    for (int idx = threadIdx.x; idx < ng * BITS; idx += blockDim.x) {
        const int g = idx / BITS, wi = idx % BITS;
        qzeros[((c0 / group) + g) * zw + row0 * BITS / 32 + wi] = (int32_t)pack_word<BITS>(sm.zeros[g], wi, ROWS);
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
                         const uint8_t *dead, int group, float *D, int32_t *qweight, float *scales,
                         int32_t *qzeros, uint8_t *codes, float *W_hat, float *row_err, cudaStream_t s) {
    const size_t smem = sizeof(SweepSmem);
    static bool attr_set = false;  // per template instance
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(sweep_kernel<BITS, TW>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    sweep_kernel<BITS, TW><<<(unsigned)((rows + ROWS - 1) / ROWS), 256, smem, s>>>(
        W, rows, cols, c0, bw, Uinv, dead, group, D, qweight, scales, qzeros, codes, W_hat, row_err);
    return cudaGetLastError();
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
    return cudaGetLastError();
}

cudaError_t sweep_block_launch(const void *W, bool w_bf16, int64_t rows, int64_t cols, int64_t c0, int bw,
                               const float *Uinv_blk, const uint8_t *dead, int bits, int group, float *D,
                               int32_t *qweight, float *scales, int32_t *qzeros, uint8_t *codes,
                               float *W_hat, float *row_err, cudaStream_t s) {
#define GQ_SWEEP_CASE(B)                                                                                       \
    if (bits == B) {                                                                                           \
        if (w_bf16)                                                                                            \
            return launch_sweep<B, __nv_bfloat16>((const __nv_bfloat16 *)W, rows, cols, c0, bw, Uinv_blk, dead, \
                                                  group, D, qweight, scales, qzeros, codes, W_hat, row_err, s); \
        return launch_sweep<B, float>((const float *)W, rows, cols, c0, bw, Uinv_blk, dead, group, D, qweight,   \
                                      scales, qzeros, codes, W_hat, row_err, s);                               \
    }
    GQ_SWEEP_CASE(2)
    GQ_SWEEP_CASE(3)
    GQ_SWEEP_CASE(4)
#undef GQ_SWEEP_CASE
    return cudaErrorInvalidValue;
}

}  // namespace gq
