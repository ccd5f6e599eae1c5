// GPTQ-intrinsic LoRA ("Resumen Técnico: GPTQ-intrinsic LoRA", "Algoritmo
// GPTQ-intrinsic LoRA"): the basis L = V_r and the pieces of the block
// elimination that turn the page's augmented sweep into GPTQ on a Schur
// complement.
//
// Augmented Hessian (X~ = [X, X L]):  H~ = [[H, P], [P^T, C]],  P = H L,
// C = L^T H L, damped with delta = damp * mean(diag H~) over its cols + r
// diagonal entries (dead entries counted as 1).  With C_d = C + delta I = K K^T
// and Y = P K^-T:
//
//   S = H_d - Y Y^T               the Schur complement of the free block; the
//                                 quantized block of H~_d^-1 is S^-1, so GPTQ
//                                 on S gives the codes of the augmented sweep
//   R = (W - Ŵ) Y K^-1            the free columns at the end of the sweep:
//                                 argmin over R of the augmented quadratic
//                                 given Ŵ, C_d^-1 P^T (w - ŵ) per row
//
// The launches are ordered by the C ABI (api.cu); this file holds the kernels
// and the basis computation.
#include <climits>

#include "common.cuh"

namespace gq {
namespace {

__device__ __forceinline__ float fix_dead(float d) { return d == 0.f ? 1.f : d; }

// One CTA: dead inputs of H, delta = damp * (sum fix(H_ii) + sum fix(C_ii)) /
// (cols + r) (summed in float64), then C_ii = fix(C_ii) + delta.  delta is
// left in st->delta.
__global__ void __launch_bounds__(1024) lora_damp_kernel(const float *__restrict__ H, int64_t cols,
                                                         float *__restrict__ C, int r, float damp,
                                                         uint8_t *__restrict__ dead, DeviceStatus *st) {
    __shared__ double red[32];
    __shared__ float delta_s;
    double acc = 0.0;
    for (int64_t i = threadIdx.x; i < cols; i += blockDim.x) {
        const float d = H[i * cols + i];
        dead[i] = (d == 0.f);
        acc += (double)fix_dead(d);
    }
    for (int i = threadIdx.x; i < r; i += blockDim.x) acc += (double)fix_dead(C[i * r + i]);
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x < 32) {
        acc = (threadIdx.x < blockDim.x / 32) ? red[threadIdx.x] : 0.0;
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (threadIdx.x == 0) {
            delta_s = (float)((double)damp * (acc / (double)(cols + r)));
            st->diag_sum = acc;
            st->delta = delta_s;
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < r; i += blockDim.x) C[i * r + i] = fix_dead(C[i * r + i]) + delta_s;
}

// S = H with the diagonal replaced by fix(H_ii) + delta.
__global__ void schur_init_kernel(const float *__restrict__ H, int64_t cols, const DeviceStatus *__restrict__ st,
                                  float *__restrict__ S) {
    const float delta = st->delta;
    const int64_t n = cols * cols;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < n; idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i = idx / cols, j = idx - i * cols;
        const float h = H[idx];
        S[idx] = (i == j) ? fix_dead(h) + delta : h;
    }
}

// ΔW = W - Ŵ with the dead inputs' weights taken as 0, written as its TF32
// split (hi + lo = ΔW exactly).
template <typename T>
__global__ void dw_split_kernel(const T *__restrict__ W, const float *__restrict__ W_hat,
                                const uint8_t *__restrict__ dead, int64_t rows, int64_t cols, float *__restrict__ hi,
                                float *__restrict__ lo) {
    const int64_t n = rows * cols;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < n; idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t j = idx % cols;
        const float w = dead[j] ? 0.f : load_f32<T>(W + idx);
        const float d = w - W_hat[idx];
        const float h = tf32_hi(d);
        hi[idx] = h;
        lo[idx] = d - h;
    }
}

unsigned grid_for(int64_t n, int64_t cap) {
    int64_t g = (n + 255) / 256;
    if (g < 1) g = 1;
    if (g > cap) g = cap;
    return (unsigned)g;
}

// Basis workspace: [qst][Linv][Ghi][Glo][ZT][ZT2][Zhi][Zlo][Gm][Wt][lam][part]
// (Ghi, Glo, Zhi, Zlo only on the tensor-core path).
struct BasisWs {
    SubspaceBufs sb;
    float *Ghi, *Glo;
};

bool basis_tc(int64_t cols) { return cols % 4 == 0; }

size_t basis_layout(int64_t cols, int r, BasisWs *w, char *base) {
    const int k = subspace_width(cols, r);
    const bool tc = basis_tc(cols);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        char *p = base ? base + off : nullptr;
        off += align_up(bytes);
        return p;
    };
    BasisWs t = {};
    t.sb.qst = (DeviceStatus *)take(sizeof(DeviceStatus));
    t.sb.Linv = (float *)take(cholesky_scratch_floats(128) * sizeof(float));
    if (tc) {
        t.Ghi = (float *)take((size_t)cols * cols * sizeof(float));
        t.Glo = (float *)take((size_t)cols * cols * sizeof(float));
        t.sb.Zhi = (float *)take((size_t)k * cols * sizeof(float));
        t.sb.Zlo = (float *)take((size_t)k * cols * sizeof(float));
    }
    t.sb.ZT = (float *)take((size_t)k * cols * sizeof(float));
    t.sb.ZT2 = (float *)take((size_t)k * cols * sizeof(float));
    t.sb.Gm = (float *)take((size_t)k * k * sizeof(float));
    t.sb.Wt = (float *)take((size_t)k * k * sizeof(float));
    t.sb.lam = (float *)take((size_t)k * sizeof(float));
    t.sb.part = (float *)take(subspace_part_floats(k, cols, tc) * sizeof(float));
    t.sb.Ghi = t.Ghi;
    t.sb.Glo = t.Glo;
    if (w) *w = t;
    return off;
}

}  // namespace

size_t lora_basis_workspace_bytes(int64_t cols, int r) { return basis_layout(cols, r, nullptr, nullptr); }

cudaError_t lora_basis_run(const float *H, int64_t cols, int r, float *Lt, float *lam, void *ws, cudaStream_t s) {
    BasisWs w;
    basis_layout(cols, r, &w, (char *)ws);
    const int k = subspace_width(cols, r);
    const bool tc = basis_tc(cols);
    cudaError_t e;
    if ((e = cudaMemsetAsync(w.sb.qst, 0xFF, sizeof(DeviceStatus), s)) != cudaSuccess) return e;
    w.sb.G = H;
    if (tc && (e = split_tf32(H, cols, cols, cols, w.Ghi, w.Glo, cols, s)) != cudaSuccess) return e;
    if ((e = subspace_ritz(w.sb, k, cols, tc, s)) != cudaSuccess) return e;
    // L^T = W[:, :r]^T Z^T  (r x cols), each row's sign fixed.
    if ((e = sgemm<float>(r, cols, k, 1.f, w.sb.Wt, k, true, w.sb.ZT, cols, false, 0.f, Lt, cols, 0, s)) !=
        cudaSuccess)
        return e;
    if ((e = sign_normalize(Lt, r, cols, 1, cols, s)) != cudaSuccess) return e;
    if (lam)
        return cudaMemcpyAsync(lam, w.sb.lam, (size_t)r * sizeof(float), cudaMemcpyDeviceToDevice, s);
    return cudaSuccess;
}

cudaError_t lora_damp_launch(const float *H, int64_t cols, float *C, int r, float damp, uint8_t *dead,
                             DeviceStatus *st, cudaStream_t s) {
    lora_damp_kernel<<<1, 1024, 0, s>>>(H, cols, C, r, damp, dead, st);
    count_launch();
    return cudaGetLastError();
}

cudaError_t schur_init_launch(const float *H, int64_t cols, const DeviceStatus *st, float *S, cudaStream_t s) {
    schur_init_kernel<<<grid_for(cols * cols, 148 * 16), 256, 0, s>>>(H, cols, st, S);
    count_launch();
    return cudaGetLastError();
}

cudaError_t dw_split_launch(const void *W, bool w_bf16, const float *W_hat, const uint8_t *dead, int64_t rows,
                            int64_t cols, float *hi, float *lo, cudaStream_t s) {
    const unsigned g = grid_for(rows * cols, 148 * 16);
    if (w_bf16)
        dw_split_kernel<__nv_bfloat16><<<g, 256, 0, s>>>((const __nv_bfloat16 *)W, W_hat, dead, rows, cols, hi, lo);
    else
        dw_split_kernel<float><<<g, 256, 0, s>>>((const float *)W, W_hat, dead, rows, cols, hi, lo);
    count_launch();
    return cudaGetLastError();
}

}  // namespace gq
