// Standalone packing of b-bit codes into 32-bit words and its inverse.  Layout
// (this library's reading of the packing layout that [LowBit] section 1 says a
// format must fix): little-endian bitstream along the input axis, code k at
// bits [k*b, k*b + b), cut into 32-bit words; qweight is [cols*b/32][rows].
#include "common.cuh"

namespace gq {
namespace {

template <int BITS>
__global__ void pack_kernel(const uint8_t *__restrict__ codes, int64_t rows, int64_t cols,
                            int32_t *__restrict__ qweight) {
    const int64_t nw = cols * BITS / 32;
    const int64_t total = nw * rows;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t w = idx / rows, r = idx % rows;  // consecutive threads -> consecutive rows
        const uint8_t *v = codes + r * cols;
        uint32_t word = 0;
        const int64_t k_lo = (32 * w) / BITS, k_hi = (32 * w + 31) / BITS;
        for (int64_t k = k_lo; k <= k_hi && k < cols; ++k) {
            const int64_t pos = k * BITS - 32 * w;
            const uint32_t x = v[k] & ((1u << BITS) - 1u);
            if (pos >= 0)
                word |= (pos < 32) ? (x << pos) : 0u;
            else
                word |= x >> (-pos);
        }
        qweight[idx] = (int32_t)word;
    }
}

template <int BITS>
__global__ void unpack_kernel(const int32_t *__restrict__ qweight, int64_t rows, int64_t cols,
                              uint8_t *__restrict__ codes) {
    const int64_t total = rows * cols;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = idx / cols, k = idx % cols;
        const int64_t pos = k * BITS, w = pos / 32, sh = pos % 32;
        uint64_t v = (uint32_t)qweight[w * rows + r];
        if (sh + BITS > 32) v |= (uint64_t)(uint32_t)qweight[(w + 1) * rows + r] << 32;
        codes[idx] = (uint8_t)((v >> sh) & ((1u << BITS) - 1u));
    }
}

template <typename TW>
__global__ void weight_error_kernel(const TW *__restrict__ W, const float *__restrict__ W_hat, int64_t n,
                                    float *__restrict__ dW) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        dW[i] = load_f32(W + i) - W_hat[i];
}

__global__ void code_decisions_kernel(const float *__restrict__ w, const float *__restrict__ s, int64_t n,
                                      float *__restrict__ k) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const float sv = s[i];
        k[i] = rintf(quotient_rn(w[i], sv, __fdiv_rn(1.f, sv)));
    }
}

unsigned grid_for(int64_t total) {
    int64_t g = (total + 255) / 256;
    return (unsigned)(g < 148 * 16 ? (g < 1 ? 1 : g) : 148 * 16);
}

}  // namespace

cudaError_t weight_error_launch(const void *W, bool w_bf16, int64_t n, const float *W_hat, float *dW, cudaStream_t s) {
    if (w_bf16)
        weight_error_kernel<__nv_bfloat16><<<grid_for(n), 256, 0, s>>>((const __nv_bfloat16 *)W, W_hat, n, dW);
    else
        weight_error_kernel<float><<<grid_for(n), 256, 0, s>>>((const float *)W, W_hat, n, dW);
    count_launch();
    return cudaGetLastError();
}

cudaError_t code_decisions_launch(const float *w, const float *s, int64_t n, float *k, cudaStream_t st) {
    code_decisions_kernel<<<grid_for(n), 256, 0, st>>>(w, s, n, k);
    count_launch();
    return cudaGetLastError();
}

cudaError_t pack_launch(const uint8_t *codes, int64_t rows, int64_t cols, int bits, int32_t *qweight,
                        cudaStream_t s) {
    const unsigned g = grid_for(cols * bits / 32 * rows);
    if (bits == 2) pack_kernel<2><<<g, 256, 0, s>>>(codes, rows, cols, qweight);
    else if (bits == 3) pack_kernel<3><<<g, 256, 0, s>>>(codes, rows, cols, qweight);
    else if (bits == 4) pack_kernel<4><<<g, 256, 0, s>>>(codes, rows, cols, qweight);
    else return cudaErrorInvalidValue;
    count_launch();
    return cudaGetLastError();
}

cudaError_t unpack_launch(const int32_t *qweight, int64_t rows, int64_t cols, int bits, uint8_t *codes,
                          cudaStream_t s) {
    const unsigned g = grid_for(rows * cols);
    if (bits == 2) unpack_kernel<2><<<g, 256, 0, s>>>(qweight, rows, cols, codes);
    else if (bits == 3) unpack_kernel<3><<<g, 256, 0, s>>>(qweight, rows, cols, codes);
    else if (bits == 4) unpack_kernel<4><<<g, 256, 0, s>>>(qweight, rows, cols, codes);
    else return cudaErrorInvalidValue;
    count_launch();
    return cudaGetLastError();
}

}  // namespace gq
