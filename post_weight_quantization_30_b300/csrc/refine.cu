// Bid-Up: coordinate refinement of the codes on their fixed grid ("Resumen
// Técnico: GPTQ-intrinsic LoRA", "Refinamiento Bid-Up"), alternated with OLrC
// (the optimal low-rank compensation for fixed codes, which is the EoRA
// problem: eora.cu).
//
// With target T = W - B A (the layer minus its low-rank correction), residual
// r = T - Ŵ and gradient g = r H per row, moving ŵ_j by d changes r H r^T by
// -2 d g_j + d^2 H_jj: the best grid value for coordinate j alone is the grid
// point nearest ŵ_j + g_j / H_jj, i.e. q' = clamp(q + rint(g_j / (H_jj s))).
// One sweep takes the columns in order (Gauss-Seidel) and, after a move d_j,
// updates g_k -= d_j H_jk for every later k.
//
// Layout of the sweep (the same blocking as the GPTQ sweep):
//   G = (T - Ŵ) H                      3xTF32 GEMM
//   for each 128-column block:         bidup_block_kernel, one warp per 8 rows:
//                                      the block's g, codes and moves in shared
//                                      memory, the diagonal block of H too;
//                                      later columns of the block updated at once
//   later blocks                       G[:, right] -= D[:, left] H[left, right],
//                                      applied recursively as 3xTF32 GEMMs
#include "common.cuh"

namespace gq {
namespace {

constexpr int BU_B = 128;   // columns per block
constexpr int BU_R = 8;     // rows per CTA (one warp, four lanes per row)
constexpr int BU_LD = 9;    // row stride of the transposed tiles (column-major in shared memory)
constexpr size_t BU_SMEM = (size_t)BU_B * BU_B * 4 + 2 * (size_t)BU_B * BU_LD * 4 + (size_t)BU_B * BU_LD;

__device__ __forceinline__ uint32_t field_at(const int32_t *__restrict__ p, int64_t bit, int b) {
    const int64_t wi = bit >> 5;
    const int sh = (int)(bit & 31);
    uint32_t v = (uint32_t)p[wi] >> sh;
    if (sh + b > 32) v |= (uint32_t)p[wi + 1] << (32 - sh);
    return v & ((1u << b) - 1u);
}

// T = W (float32 copy; bf16 widened).
template <typename TW>
__global__ void widen_kernel(const TW *__restrict__ W, int64_t n, float *__restrict__ T) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        T[i] = load_f32<TW>(W + i);
}

// r = T - Ŵ with Ŵ = s (q - z) rounded to float32 (also written out), as its
// TF32 split for the GEMM G = r H.
__global__ void bidup_residual_kernel(const float *__restrict__ T, const uint8_t *__restrict__ codes,
                                      const float *__restrict__ scales, const int32_t *__restrict__ qzeros,
                                      int64_t rows, int64_t cols, int bits, int group, float *__restrict__ W_hat,
                                      float *__restrict__ rhi, float *__restrict__ rlo) {
    const int64_t n = rows * cols;
    const int64_t zwords = rows * bits / 32;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < n; idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i = idx / cols, j = idx - i * cols;
        const int64_t g = j / group;
        const float s = scales[g * rows + i];
        const float z = (float)field_at(qzeros + g * zwords, i * bits, bits);
        const float w = s * ((float)codes[idx] - z);
        W_hat[idx] = w;
        const float r = T[idx] - w;
        const float h = tf32_hi(r);
        rhi[idx] = h;
        rlo[idx] = r - h;
    }
}

// One 128-column block of the sweep for 8 rows: a warp, four lanes per row,
// lane part p owning the block's columns [32 p, 32 p + 32) of its row's gradient
// g (so a move updates at most 32 later columns per lane).  At column j the
// owning lane broadcasts g_j to the row's four lanes, which all take the same
// decision.  g, codes and moves are kept column-major in shared memory; the
// block's diagonal part of H is shared by all lanes (broadcast reads).  Writes
// back the codes, Ŵ and the TF32 split of the moves d for the block's columns
// (d = 0 where the code did not move).
__global__ void __launch_bounds__(32) bidup_block_kernel(const float *__restrict__ H, int64_t cols,
                                                         const float *__restrict__ G, uint8_t *__restrict__ codes,
                                                         const float *__restrict__ scales,
                                                         const int32_t *__restrict__ qzeros, int bits, int group,
                                                         int64_t rows, int64_t c0, int bw, float *__restrict__ W_hat,
                                                         float *__restrict__ Dhi, float *__restrict__ Dlo,
                                                         unsigned long long *__restrict__ changed) {
    extern __shared__ __align__(16) float bsm[];
    float *Hb = bsm;                          // [bw][BU_B]
    float *Gs = Hb + BU_B * BU_B;             // [bw][BU_LD]: column j, row rl at j * BU_LD + rl
    float *Ds = Gs + BU_B * BU_LD;            // [bw][BU_LD]
    uint8_t *Cs = (uint8_t *)(Ds + BU_B * BU_LD);  // [bw][BU_LD]
    const int lane = threadIdx.x;
    const int rl = lane >> 2, part = lane & 3;  // row within the CTA, column quarter
    const int64_t r0 = (int64_t)blockIdx.x * BU_R;
    const int64_t row = r0 + rl;
    const bool valid = row < rows;
    const int maxq = (1 << bits) - 1;
    const int64_t zwords = rows * bits / 32;

    // The diagonal block of H by asynchronous 16-byte copies, all in flight at once
    // (H is 16-byte aligned, cols and c0 multiples of 32; bw a multiple of 32).
    const int q4 = bw / 4;  // 16-byte chunks per row of the block
    for (int idx = lane; idx < bw * q4; idx += 32) {
        const int j = idx / q4, k4 = idx - j * q4;
        const float *src = H + (c0 + j) * cols + c0 + k4 * 4;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                         (uint32_t)__cvta_generic_to_shared(Hb + j * BU_B + k4 * 4)),
                     "l"(src)
                     : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    for (int idx = lane; idx < BU_R * bw; idx += 32) {  // coalesced along the row
        const int r = idx / bw, j = idx - r * bw;
        const bool v = r0 + r < rows;
        Gs[j * BU_LD + r] = v ? G[(r0 + r) * cols + c0 + j] : 0.f;
        Cs[j * BU_LD + r] = v ? codes[(r0 + r) * cols + c0 + j] : 0;
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncwarp();

    unsigned moved_count = 0;
    int64_t gcur = -1;
    float s = 1.f, zf = 0.f;
    const int k_lo = part * 32, k_hi = (k_lo + 32) < bw ? (k_lo + 32) : bw;
    for (int j = 0; j < bw; ++j) {
        const int64_t g = (c0 + j) / group;
        if (g != gcur) {
            gcur = g;
            s = valid ? scales[g * rows + row] : 1.f;
            zf = valid ? (float)field_at(qzeros + g * zwords, row * bits, bits) : 0.f;
        }
        const int owner = (rl << 2) | (j >> 5);
        const float gj = __shfl_sync(0xffffffffu, Gs[j * BU_LD + rl], owner);
        const int q = Cs[j * BU_LD + rl];
        const float hjj = Hb[j * BU_B + j];
        int qn = q;
        if (valid && hjj > 0.f) {
            float u = rintf(gj / (hjj * s));
            u = fminf(fmaxf(u, (float)-maxq), (float)maxq);  // finite and small before the integer step
            qn = q + (int)u;
            qn = qn < 0 ? 0 : (qn > maxq ? maxq : qn);
        }
        const bool moved = qn != q;
        const float d = moved ? s * ((float)qn - zf) - s * ((float)q - zf) : 0.f;
        __syncwarp();  // every lane has read Cs[j] before the owner rewrites it
        if (lane == owner) {
            Ds[j * BU_LD + rl] = d;
            Cs[j * BU_LD + rl] = (uint8_t)qn;
            moved_count += moved;
        }
        if (__any_sync(0xffffffffu, moved)) {
            const float *hr = Hb + j * BU_B;
            const int kb = (j + 1) > k_lo ? (j + 1) : k_lo;
#pragma unroll 8
            for (int k = kb; k < k_hi; ++k) Gs[k * BU_LD + rl] = fmaf(-d, hr[k], Gs[k * BU_LD + rl]);
        }
    }
    __syncwarp();
    for (int idx = lane; idx < BU_R * bw; idx += 32) {
        const int r = idx / bw, j = idx - r * bw;
        const int64_t rr = r0 + r;
        if (rr >= rows) continue;
        const int64_t o = rr * cols + c0 + j;
        const int64_t g = (c0 + j) / group;
        const uint8_t q = Cs[j * BU_LD + r];
        codes[o] = q;
        W_hat[o] = scales[g * rows + rr] * ((float)q - (float)field_at(qzeros + g * zwords, rr * bits, bits));
        const float d = Ds[j * BU_LD + r];
        const float h = tf32_hi(d);
        Dhi[o] = h;
        Dlo[o] = d - h;
    }
    for (int o = 16; o > 0; o >>= 1) moved_count += __shfl_xor_sync(0xffffffffu, moved_count, o);
    if (lane == 0 && moved_count && changed) atomicAdd(changed, (unsigned long long)moved_count);
}

unsigned grid_n(int64_t n) {
    int64_t g = (n + 255) / 256;
    if (g < 1) g = 1;
    if (g > 148 * 16) g = 148 * 16;
    return (unsigned)g;
}

struct BidupCtx {
    const float *H, *Hhi, *Hlo, *scales;
    const int32_t *qzeros;
    int64_t rows, cols;
    int bits, group;
    float *G, *Dhi, *Dlo, *W_hat;
    uint8_t *codes;
    unsigned long long *changed;
    cudaStream_t s;
};

// Blocks [a, b): the left half, its deferred update of the right half as one
// GEMM, the right half (the same sums as updating after every block).
cudaError_t bidup_range(const BidupCtx &c, int64_t a, int64_t b) {
    if (b - a == 1) {
        const int64_t c0 = a * BU_B;
        const int bw = (int)((c.cols - c0) < BU_B ? (c.cols - c0) : BU_B);
        bidup_block_kernel<<<(unsigned)((c.rows + BU_R - 1) / BU_R), 32, BU_SMEM, c.s>>>(
            c.H, c.cols, c.G, c.codes, c.scales, c.qzeros, c.bits, c.group, c.rows, c0, bw, c.W_hat, c.Dhi, c.Dlo,
            c.changed);
        count_launch();
        return cudaGetLastError();
    }
    const int64_t m = (a + b) / 2;
    cudaError_t e = bidup_range(c, a, m);
    if (e != cudaSuccess) return e;
    const int64_t k0 = a * BU_B, k1 = m * BU_B, n1 = (b * BU_B < c.cols) ? b * BU_B : c.cols;
    e = gemm3(c.rows, n1 - k1, k1 - k0, -1.f, c.Dhi + k0, c.Dlo + k0, c.cols, c.Hhi + k1 * c.cols + k0,
              c.Hlo + k1 * c.cols + k0, c.cols, 1.f, c.G + k1, c.cols, 0, nullptr, nullptr, 0, c.s);
    if (e != cudaSuccess) return e;
    return bidup_range(c, m, b);
}

struct BidupWs {
    float *T, *G, *Dhi, *Dlo, *Hhi, *Hlo;
    unsigned long long *changed;
};

size_t bidup_layout(int64_t rows, int64_t cols, BidupWs *w, char *base) {
    size_t off = 0;
    auto take = [&](size_t bytes) {
        char *p = base ? base + off : nullptr;
        off += align_up(bytes);
        return p;
    };
    const size_t rc = (size_t)rows * cols * sizeof(float), cc = (size_t)cols * cols * sizeof(float);
    BidupWs t;
    t.T = (float *)take(rc);
    t.G = (float *)take(rc);
    t.Dhi = (float *)take(rc);
    t.Dlo = (float *)take(rc);
    t.Hhi = (float *)take(cc);
    t.Hlo = (float *)take(cc);
    t.changed = (unsigned long long *)take(sizeof(unsigned long long));
    if (w) *w = t;
    return off;
}

}  // namespace

size_t bidup_workspace_bytes(int64_t rows, int64_t cols) { return bidup_layout(rows, cols, nullptr, nullptr); }

cudaError_t bidup_run(const void *W, bool w_bf16, int64_t rows, int64_t cols, const float *H, const float *A,
                      const float *B, int r, int bits, int group, uint8_t *codes, const float *scales,
                      const int32_t *qzeros, float *W_hat, int32_t *qweight, unsigned long long *changed_out,
                      void *ws, cudaStream_t s) {
    BidupWs w;
    bidup_layout(rows, cols, &w, (char *)ws);
    cudaError_t e;
    const int64_t n = rows * cols;
    // T = W - B A
    if (w_bf16)
        widen_kernel<__nv_bfloat16><<<grid_n(n), 256, 0, s>>>((const __nv_bfloat16 *)W, n, w.T);
    else
        widen_kernel<float><<<grid_n(n), 256, 0, s>>>((const float *)W, n, w.T);
    count_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (r > 0 && (e = sgemm<float>(rows, cols, r, -1.f, B, r, false, A, cols, false, 1.f, w.T, cols, 0, s)) !=
                     cudaSuccess)
        return e;
    // r = T - Ŵ (split), G = r H
    bidup_residual_kernel<<<grid_n(n), 256, 0, s>>>(w.T, codes, scales, qzeros, rows, cols, bits, group, W_hat,
                                                    w.Dhi, w.Dlo);
    count_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = split_tf32(H, cols, cols, cols, w.Hhi, w.Hlo, cols, s)) != cudaSuccess) return e;
    if ((e = gemm3(rows, cols, cols, 1.f, w.Dhi, w.Dlo, cols, w.Hhi, w.Hlo, cols, 0.f, w.G, cols, 0, nullptr, nullptr,
                   0, s)) != cudaSuccess)
        return e;
    if ((e = cudaMemsetAsync(w.changed, 0, sizeof(unsigned long long), s)) != cudaSuccess) return e;
    static bool attr_set = false;
    if (!attr_set) {
        if ((e = cudaFuncSetAttribute(bidup_block_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)BU_SMEM)) != cudaSuccess)
            return e;
        attr_set = true;
    }
    BidupCtx c;
    c.H = H; c.Hhi = w.Hhi; c.Hlo = w.Hlo; c.scales = scales; c.qzeros = qzeros;
    c.rows = rows; c.cols = cols; c.bits = bits; c.group = group;
    c.G = w.G; c.Dhi = w.Dhi; c.Dlo = w.Dlo; c.W_hat = W_hat; c.codes = codes; c.changed = w.changed; c.s = s;
    if ((e = bidup_range(c, 0, (cols + BU_B - 1) / BU_B)) != cudaSuccess) return e;
    if (qweight && (e = pack_launch(codes, rows, cols, bits, qweight, s)) != cudaSuccess) return e;
    if (changed_out)
        return cudaMemcpyAsync(changed_out, w.changed, sizeof(unsigned long long), cudaMemcpyDeviceToDevice, s);
    return cudaSuccess;
}

}  // namespace gq

// ---------------------------------------------------------------------------
// Round to nearest on the GPTQ grid, for the low-rank factors ("Resumen
// Técnico: GPTQ-intrinsic LoRA", "Resultados Clave": 4-bit L and 8-bit R).
// Per row and group of `group` columns: xmin = min(0, min x), xmax = max(0,
// max x) (both 0: [-1, 1]), s = (xmax - xmin) / maxq, z = rint(-xmin / s),
// q = clamp(rint(x / s) + z, 0, maxq), x̂ = s (q - z); every division IEEE.
// One warp per (row, group).
// ---------------------------------------------------------------------------
namespace gq {
namespace {

__global__ void rtn_kernel(const float *__restrict__ M, int64_t nrows, int64_t ncols, int bits, int group,
                           float *__restrict__ M_hat, uint8_t *__restrict__ codes, float *__restrict__ scales,
                           uint8_t *__restrict__ zeros) {
    const int64_t ngr = ncols / group;
    const int64_t wid = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (wid >= nrows * ngr) return;
    const int64_t row = wid / ngr, g = wid - row * ngr;
    const float *x = M + row * ncols + g * group;
    float mn = 0.f, mx = 0.f;
    for (int k = lane; k < group; k += 32) {
        mn = fminf(mn, x[k]);
        mx = fmaxf(mx, x[k]);
    }
    for (int o = 16; o > 0; o >>= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    if (mn == 0.f && mx == 0.f) {
        mn = -1.f;
        mx = 1.f;
    }
    const float maxq = (float)((1 << bits) - 1);
    const float s = __fdiv_rn(mx - mn, maxq);
    const float z = rintf(__fdiv_rn(-mn, s));
    if (lane == 0) {
        scales[g * nrows + row] = s;
        zeros[g * nrows + row] = (uint8_t)z;
    }
    for (int k = lane; k < group; k += 32) {
        const float q = fminf(fmaxf(rintf(__fdiv_rn(x[k], s)) + z, 0.f), maxq);
        const int64_t o = row * ncols + g * group + k;
        M_hat[o] = s * (q - z);
        if (codes) codes[o] = (uint8_t)q;
    }
}

}  // namespace

cudaError_t rtn_launch(const float *M, int64_t nrows, int64_t ncols, int bits, int group, float *M_hat,
                       uint8_t *codes, float *scales, uint8_t *zeros, cudaStream_t s) {
    const int64_t warps = nrows * (ncols / group);
    int64_t g = (warps * 32 + 255) / 256;
    if (g < 1) g = 1;
    rtn_kernel<<<(unsigned)g, 256, 0, s>>>(M, nrows, ncols, bits, group, M_hat, codes, scales, zeros);
    count_launch();
    return cudaGetLastError();
}

}  // namespace gq
