// C ABI of libgq (declared in include/gq.h): argument validation, workspace
// layout and the order of the stream-ordered launches.
#include <atomic>
#include <climits>
#include <cmath>
#include <cstring>

#include "common.cuh"

using namespace gq;

namespace {
std::atomic<unsigned long long> g_launches{0};
}  // namespace

void gq::count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

namespace {

inline bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }
inline cudaStream_t cs(gq_stream_t s) { return (cudaStream_t)s; }

// Sweep workspace (float32, 256-byte aligned regions):
//   [Uinv: nblk x block x block][VThi: cols x cols][VTlo: cols x cols][D: rows x cols][DL: rows x cols].
size_t sweep_ws_bytes(int64_t rows, int64_t cols, int block) {
    const int64_t nblk = (cols + block - 1) / block;
    return align_up((size_t)nblk * block * block * sizeof(float)) + 2 * align_up((size_t)cols * cols * sizeof(float)) +
           2 * align_up((size_t)rows * cols * sizeof(float));
}

gq_status check_sweep_args(const void *W, gq_dtype wt, int64_t rows, int64_t cols, const float *F, int bits,
                           int group, int block, const int32_t *qweight, const float *scales,
                           const int32_t *qzeros, const uint8_t *codes, const float *W_hat, const float *row_err) {
    if (wt != GQ_F32 && wt != GQ_BF16) return GQ_EUNSUPPORTED;
    if (bits != 2 && bits != 3 && bits != 4) return GQ_EUNSUPPORTED;
    if (!W || !F || !qweight || !scales || !qzeros) return GQ_EINVAL;
    if (rows <= 0 || cols <= 0 || rows % 32 || cols % 32) return GQ_EINVAL;
    if (group <= 0 || group % 32 || cols % group) return GQ_EINVAL;
    if (block <= 0 || block > 128 || block % group) return GQ_EINVAL;
    if (!aligned(W, 16) || !aligned(scales, 16) || !aligned(qweight, 4) || !aligned(qzeros, 4))
        return GQ_EINVAL;
    if ((codes && !aligned(codes, 4)) || (W_hat && !aligned(W_hat, 16)) || (row_err && !aligned(row_err, 4)))
        return GQ_EINVAL;
    return GQ_OK;
}

// The float32 regions of the sweep workspace.
struct SweepRegions {
    float *Uinv, *VThi, *VTlo, *D, *DL;
};

SweepRegions sweep_regions(void *ws, int64_t rows, int64_t cols, int block) {
    const int64_t nblk = (cols + block - 1) / block;
    SweepRegions g;
    g.Uinv = (float *)ws;
    g.VThi = (float *)((char *)ws + align_up((size_t)nblk * block * block * sizeof(float)));
    g.VTlo = (float *)((char *)g.VThi + align_up((size_t)cols * cols * sizeof(float)));
    g.D = (float *)((char *)g.VTlo + align_up((size_t)cols * cols * sizeof(float)));
    g.DL = (float *)((char *)g.D + align_up((size_t)rows * cols * sizeof(float)));
    return g;
}

struct SweepCtx {
    const void *W;
    bool bf16;
    int64_t rows, cols;
    const float *F;
    const uint8_t *dead;
    int bits, group, block;
    int32_t *qweight;
    float *scales;
    int32_t *qzeros;
    uint8_t *codes;
    float *W_hat, *row_err;
    float *Uinv, *VThi, *VTlo, *D, *DL;
    cudaStream_t s;
};

// Blocks [a, b): sweep the left half, apply its deferred update to the right
// half as one GEMM, sweep the right half.  Same sums as updating after every
// block, in fewer and larger GEMMs.  The GEMM runs on the tensor cores with
// float32 accuracy (3xTF32): D[:, right] += ΔW[:, left] V[left, right].
cudaError_t sweep_range(const SweepCtx &c, int64_t a, int64_t b) {
    const int64_t B = c.block;
    if (b - a == 1) {
        const int64_t c0 = a * B;
        const int bw = (int)((c.cols - c0) < B ? (c.cols - c0) : B);
        return sweep_block_launch(c.W, c.bf16, c.rows, c.cols, c0, bw, c.Uinv + a * B * B, c.F, c.dead, c.bits, c.group,
                                  c.D, c.DL, c.qweight, c.scales, c.qzeros, c.codes, c.W_hat, c.row_err, c.VThi,
                                  c.VTlo, false, c.s);
    }
    // Two full 128-column blocks, when one wave of CTAs covers the rows: one launch sweeps both
    // and applies the first one's deferred update to the second itself (no GEMM between them).
    if (b - a == 2 && B == 128 && (b * B) <= c.cols && sweep_pair_fits(c.rows))
        return sweep_block_launch(c.W, c.bf16, c.rows, c.cols, a * B, (int)B, c.Uinv + a * B * B, c.F, c.dead, c.bits,
                                  c.group, c.D, c.DL, c.qweight, c.scales, c.qzeros, c.codes, c.W_hat, c.row_err,
                                  c.VThi, c.VTlo, true, c.s);
    const int64_t m = (a + b) / 2;
    cudaError_t e = sweep_range(c, a, m);
    if (e != cudaSuccess) return e;
    const int64_t k0 = a * B, k1 = m * B, n1 = (b * B < c.cols) ? b * B : c.cols;
    e = gemm3(c.rows, n1 - k1, k1 - k0, 1.f, c.D + k0, c.DL + k0, c.cols, c.VThi + k1 * c.cols + k0,
              c.VTlo + k1 * c.cols + k0, c.cols, 1.f, c.D + k1, c.cols, 0, nullptr, nullptr, 0, c.s);
    if (e != cudaSuccess) return e;
    return sweep_range(c, m, b);
}

// Dead inputs + damping, blocked Cholesky of the reversed matrix, reversal;
// one synchronization to read the status.  The part of H the factor reads is
// checked for Inf / NaN, and so are the `wn` values of Wchk (the layer's
// weights) when given: GQ_ENONFINITE with *info = 0 (H) or 1 (W).
gq_status factor_impl(const float *H, int64_t cols, float damp, float *F, uint8_t *dead, void *ws, cudaStream_t s,
                      int64_t *info, float *Uinv, int block, const void *Wchk = nullptr, bool w_bf16 = false,
                      int64_t wn = 0) {
    DeviceStatus *st = (DeviceStatus *)ws;
    float *scratch = (float *)((char *)ws + align_up(sizeof(DeviceStatus)));
    GQ_CUDA_TRY(cudaMemsetAsync(st, 0xFF, sizeof(DeviceStatus), s));
    if (Wchk) GQ_CUDA_TRY(finite_check_launch(Wchk, w_bf16, wn, st, kNonFiniteW, s));
    GQ_CUDA_TRY(factor_prepare(H, cols, damp, F, dead, st, s));
    GQ_CUDA_TRY(cholesky_lower_inplace(F, cols, st, scratch, s, Uinv, block));
    GQ_CUDA_TRY(factor_finalize(F, cols, s));
    DeviceStatus hst;
    GQ_CUDA_TRY(cudaMemcpyAsync(&hst, st, sizeof(hst), cudaMemcpyDeviceToHost, s));
    GQ_CUDA_TRY(cudaStreamSynchronize(s));
    if (hst.finite != ~0u) {
        if (info) *info = (hst.finite & kNonFiniteH) ? 1 : 0;
        return GQ_ENONFINITE;
    }
    if (hst.bad_pivot != ULLONG_MAX) {
        if (info) *info = cols - 1 - (int64_t)hst.bad_pivot;
        return GQ_ENOTPD;
    }
    if (info) *info = -1;
    return GQ_OK;
}

// The sweep on a checked workspace.  uinv_ready: the block-inverse region at
// the start of ws already holds F's diagonal-block inverses.
gq_status sweep_impl(const void *W, gq_dtype wt, int64_t rows, int64_t cols, const float *F, const uint8_t *dead,
                     int bits, int group, int block, int32_t *qweight, float *scales, int32_t *qzeros, uint8_t *codes,
                     float *W_hat, float *row_err, void *ws, cudaStream_t s, bool uinv_ready) {
    const int64_t nblk = (cols + block - 1) / block;
    SweepCtx c;
    c.W = W; c.bf16 = (wt == GQ_BF16); c.rows = rows; c.cols = cols; c.F = F; c.dead = dead;
    c.bits = bits; c.group = group; c.block = block;
    c.qweight = qweight; c.scales = scales; c.qzeros = qzeros; c.codes = codes; c.W_hat = W_hat; c.row_err = row_err;
    const SweepRegions g = sweep_regions(ws, rows, cols, block);
    c.Uinv = g.Uinv; c.VThi = g.VThi; c.VTlo = g.VTlo; c.D = g.D; c.DL = g.DL;
    c.s = s;
    GQ_CUDA_TRY(cudaMemsetAsync(c.D, 0, (size_t)rows * cols * sizeof(float), s));
    if (row_err) GQ_CUDA_TRY(cudaMemsetAsync(row_err, 0, (size_t)rows * sizeof(float), s));
    if (!uinv_ready) GQ_CUDA_TRY(block_inverses(F, cols, block, c.Uinv, s));
    GQ_CUDA_TRY(premultiply_t(F, cols, block, c.Uinv, c.VThi, c.VTlo, s));
    GQ_CUDA_TRY(sweep_range(c, 0, nblk));
    return GQ_OK;
}

// GPTQ-intrinsic LoRA workspace (float32 unless noted, 256-byte aligned regions):
//   [cst][deadH: cols bytes][deadS: cols bytes][Lthi, Ltlo, Pt, Yt, Ythi, Ytlo: r x cols each]
//   [Ppart: psplit x r x cols][C: r x r][Cpart: 64 x r x r][Kinv][Yhi, Ylo: cols x r4 each]
//   [Rtmp: rows x r][Rpart: rsplit x rows x r][F: cols x cols][factor scratch][sweep workspace]
// The split of H and then S live in the sweep workspace's VThi / VTlo regions, which
// the sweep itself only fills after the factorization of S has read them.
struct LoraLayout {
    DeviceStatus *cst;
    uint8_t *deadH, *deadS;
    float *Lthi, *Ltlo, *Pt, *Yt, *Ythi, *Ytlo, *Ppart, *C, *Cpart, *Kinv, *Yhi, *Ylo, *Rtmp, *Rpart, *F;
    void *fws, *sws;
};

constexpr int LORA_CSPLIT = 64;  // K slices of C = L^T P

// K slices that bring a GEMM of `tiles` 128 x 128 output tiles close to one CTA
// per SM without a second wave.
int splits_for(int64_t tiles) {
    int64_t z = 148 / tiles;
    if (z < 1) z = 1;
    if (z > 8) z = 8;
    return (int)z;
}

inline int64_t r4_of(int r) { return (r + 3) / 4 * 4; }

size_t lora_layout(int64_t rows, int64_t cols, int r, int block, LoraLayout *w, char *base) {
    size_t off = 0;
    auto take = [&](size_t bytes) {
        char *p = base ? base + off : nullptr;
        off += align_up(bytes);
        return p;
    };
    const size_t rc = (size_t)r * cols * sizeof(float);
    const int ps = splits_for((cols + 127) / 128), rs = splits_for((rows + 127) / 128);
    LoraLayout t = {};
    t.cst = (DeviceStatus *)take(sizeof(DeviceStatus));
    t.deadH = (uint8_t *)take((size_t)cols);
    t.deadS = (uint8_t *)take((size_t)cols);
    t.Lthi = (float *)take(rc);
    t.Ltlo = (float *)take(rc);
    t.Pt = (float *)take(rc);
    t.Yt = (float *)take(rc);
    t.Ythi = (float *)take(rc);
    t.Ytlo = (float *)take(rc);
    t.Ppart = (float *)take((size_t)ps * rc);
    t.C = (float *)take((size_t)r * r * sizeof(float));
    t.Cpart = (float *)take((size_t)LORA_CSPLIT * r * r * sizeof(float));
    t.Kinv = (float *)take(cholesky_scratch_floats(128) * sizeof(float));
    t.Yhi = (float *)take((size_t)cols * r4_of(r) * sizeof(float));
    t.Ylo = (float *)take((size_t)cols * r4_of(r) * sizeof(float));
    t.Rtmp = (float *)take((size_t)rows * r * sizeof(float));
    t.Rpart = (float *)take((size_t)rs * rows * r * sizeof(float));
    t.F = (float *)take((size_t)cols * cols * sizeof(float));
    t.fws = take(factor_scratch_bytes(cols));
    t.sws = take(sweep_ws_bytes(rows, cols, block));
    if (w) *w = t;
    return off;
}

// C = A B^T on the tensor cores (3xTF32), split over K when the output has few tiles.
cudaError_t gemm3_nt(int64_t M, int64_t N, int64_t K, const float *Ahi, const float *Alo, int64_t lda,
                     const float *Bhi, const float *Blo, int64_t ldb, float *C, float *part, int slices,
                     cudaStream_t s) {
    if (slices <= 1)
        return gemm3(M, N, K, 1.f, Ahi, Alo, lda, Bhi, Blo, ldb, 0.f, C, N, 0, nullptr, nullptr, 0, s);
    return gemm3_splitk(M, N, K, Ahi, Alo, lda, Bhi, Blo, ldb, C, part, slices, s);
}

gq_status intrinsic_impl(const void *W, gq_dtype wt, int64_t rows, int64_t cols, const float *H, const float *Lt,
                         int r, int bits, int group, int block, float damp, int32_t *qweight, float *scales,
                         int32_t *qzeros, uint8_t *codes, float *W_hat, float *row_err, float *R, void *ws,
                         cudaStream_t s, int64_t *info) {
    LoraLayout w;
    lora_layout(rows, cols, r, block, &w, (char *)ws);
    const SweepRegions g = sweep_regions(w.sws, rows, cols, block);
    const int ps = splits_for((cols + 127) / 128), rs = splits_for((rows + 127) / 128);
    const int64_t r4 = r4_of(r);
    float *S = g.VThi;
    GQ_CUDA_TRY(cudaMemsetAsync(w.cst, 0xFF, sizeof(DeviceStatus), s));
    // P^T = L^T H (H symmetric), C = L^T P.
    GQ_CUDA_TRY(split_tf32(Lt, r, cols, cols, w.Lthi, w.Ltlo, cols, s));
    GQ_CUDA_TRY(split_tf32(H, cols, cols, cols, g.VThi, g.VTlo, cols, s));
    GQ_CUDA_TRY(gemm3_nt(r, cols, cols, w.Lthi, w.Ltlo, cols, g.VThi, g.VTlo, cols, w.Pt, w.Ppart, ps, s));
    GQ_CUDA_TRY(sgemm_splitk(r, r, cols, Lt, cols, false, w.Pt, cols, true, w.C, w.Cpart, LORA_CSPLIT, s));
    // delta over the augmented diagonal; C_d = C + delta I = K K^T; Y^T = K^-1 P^T.
    GQ_CUDA_TRY(lora_damp_launch(H, cols, w.C, r, damp, w.deadH, w.cst, s));
    GQ_CUDA_TRY(cholesky_lower_inplace(w.C, r, w.cst, w.Kinv, s));
    GQ_CUDA_TRY(sgemm<float>(r, cols, r, 1.f, w.Kinv, 128, false, w.Pt, cols, false, 0.f, w.Yt, cols, 0, s));
    GQ_CUDA_TRY(split_tf32(w.Yt, r, cols, cols, w.Ythi, w.Ytlo, cols, s));
    GQ_CUDA_TRY(split_transpose_tf32(w.Yt, r, cols, cols, w.Yhi, w.Ylo, r4, s));
    // S = H_d - Y Y^T.
    GQ_CUDA_TRY(schur_init_launch(H, cols, w.cst, S, s));
    GQ_CUDA_TRY(gemm3(cols, cols, r, -1.f, w.Yhi, w.Ylo, r4, w.Yhi, w.Ylo, r4, 1.f, S, cols, 0, nullptr, nullptr, 0,
                      s));
    unsigned long long bad_c = 0;
    GQ_CUDA_TRY(cudaMemcpyAsync(&bad_c, &w.cst->bad_pivot, sizeof(bad_c), cudaMemcpyDeviceToHost, s));
    // GPTQ on S: the factorization synchronizes the stream, after which bad_c is valid.
    const bool uinv = factor_emits_uinv(cols, block);
    gq_status st = factor_impl(S, cols, 0.f, w.F, w.deadS, w.fws, s, info, uinv ? g.Uinv : nullptr, block, W,
                               wt == GQ_BF16, rows * cols);
    if (bad_c != ULLONG_MAX) {
        if (info) *info = cols + (int64_t)bad_c;
        return GQ_ENOTPD;
    }
    if (st != GQ_OK) return st;
    st = sweep_impl(W, wt, rows, cols, w.F, w.deadH, bits, group, block, qweight, scales, qzeros, codes, W_hat,
                    row_err, w.sws, s, uinv);
    if (st != GQ_OK) return st;
    // R = (W - Ŵ) Y K^-1.
    GQ_CUDA_TRY(dw_split_launch(W, wt == GQ_BF16, W_hat, w.deadH, rows, cols, g.D, g.DL, s));
    GQ_CUDA_TRY(gemm3_nt(rows, r, cols, g.D, g.DL, cols, w.Ythi, w.Ytlo, cols, w.Rtmp, w.Rpart, rs, s));
    GQ_CUDA_TRY(sgemm<float>(rows, r, r, 1.f, w.Rtmp, r, false, w.Kinv, 128, false, 0.f, R, r, 0, s));
    return GQ_OK;
}

}  // namespace

extern "C" {

int gq_abi_version(void) { return 1; }

unsigned long long gq_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

const char *gq_status_string(gq_status s) {
    switch (s) {
        case GQ_OK: return "GQ_OK";
        case GQ_EINVAL: return "GQ_EINVAL: invalid argument";
        case GQ_ENOTPD: return "GQ_ENOTPD: damped Hessian not positive definite";
        case GQ_EUNSUPPORTED: return "GQ_EUNSUPPORTED: unsupported bit width or dtype";
        case GQ_ECUDA: return "GQ_ECUDA: CUDA error";
        case GQ_ENONFINITE: return "GQ_ENONFINITE: non-finite input";
        case GQ_ETIMEOUT: return "GQ_ETIMEOUT: device wait gave up";
        case GQ_EWORKSPACE: return "GQ_EWORKSPACE: workspace too small or misaligned";
    }
    return "GQ_?: unknown status";
}

gq_status gq_check_device(gq_stream_t stream) {
    if (cudaStreamSynchronize(cs(stream)) != cudaSuccess) return GQ_ECUDA;
    const unsigned int e1 = read_and_clear_device_error();
    const unsigned int e2 = gemm_read_and_clear_error();
    const unsigned int e3 = packed_read_and_clear_error();
    if (e1 == ~0u || e2 == ~0u || e3 == ~0u) return GQ_ECUDA;
    return (e1 | e2 | e3) ? GQ_ETIMEOUT : GQ_OK;
}

gq_status gq_set_wait_budget(long long cycles) {
    const long long c = cycles > 0 ? cycles : 4000000000LL;
    if (hessian_set_wait_budget(c) != cudaSuccess || gemm_set_wait_budget(c) != cudaSuccess ||
        packed_set_wait_budget(c) != cudaSuccess)
        return GQ_ECUDA;
    return GQ_OK;
}

gq_status gptq_hessian_accumulate(float *H, int64_t cols, const void *X, gq_dtype xt, int64_t n, int64_t ldx,
                                  gq_stream_t stream) {
    if (xt != GQ_F32 && xt != GQ_BF16) return GQ_EUNSUPPORTED;
    if (cols <= 0 || n < 0 || ldx < cols) return GQ_EINVAL;
    if (n == 0) return GQ_OK;
    if (!H || !X) return GQ_EINVAL;
    cudaError_t e;
    if (xt == GQ_BF16) {
        if (hessian_bf16_tc_supported(cols, X, ldx))
            e = hessian_bf16_tc(H, cols, (const __nv_bfloat16 *)X, n, ldx, cs(stream));
        else
            e = sgemm<__nv_bfloat16>(cols, cols, n, 2.f, (const __nv_bfloat16 *)X, ldx, true, (const __nv_bfloat16 *)X,
                                     ldx, false, 1.f, H, cols, 2, cs(stream));
    } else {
        e = sgemm<float>(cols, cols, n, 2.f, (const float *)X, ldx, true, (const float *)X, ldx, false, 1.f, H, cols, 2,
                         cs(stream));
    }
    return e == cudaSuccess ? GQ_OK : GQ_ECUDA;
}

size_t gptq_factor_workspace_size(int64_t cols) {
    return factor_scratch_bytes(cols);
}

gq_status gptq_factor(const float *H, int64_t cols, float damp, float *F, uint8_t *dead, void *ws, size_t ws_bytes,
                      gq_stream_t stream, int64_t *info) {
    if (cols <= 0 || !H || !F) return GQ_EINVAL;
    if (!(damp >= 0.f)) return GQ_EINVAL;
    if (!ws || !aligned(ws, kAlign) || ws_bytes < gptq_factor_workspace_size(cols)) return GQ_EWORKSPACE;
    return factor_impl(H, cols, damp, F, dead, ws, cs(stream), info, nullptr, 0);
}

size_t gptq_sweep_workspace_size(int64_t rows, int64_t cols, int block) {
    if (rows <= 0 || cols <= 0 || block <= 0) return 0;
    return sweep_ws_bytes(rows, cols, block);
}

gq_status gptq_sweep(const void *W, gq_dtype wt, int64_t rows, int64_t cols, const float *F, const uint8_t *dead,
                     int bits, int group, int block, int32_t *qweight, float *scales, int32_t *qzeros, uint8_t *codes,
                     float *W_hat, float *row_err, void *ws, size_t ws_bytes, gq_stream_t stream) {
    gq_status st = check_sweep_args(W, wt, rows, cols, F, bits, group, block, qweight, scales, qzeros, codes, W_hat,
                                    row_err);
    if (st != GQ_OK) return st;
    if (!ws || !aligned(ws, kAlign) || ws_bytes < sweep_ws_bytes(rows, cols, block)) return GQ_EWORKSPACE;
    return sweep_impl(W, wt, rows, cols, F, dead, bits, group, block, qweight, scales, qzeros, codes, W_hat, row_err,
                      ws, cs(stream), false);
}

size_t gptq_quantize_layer_workspace_size(int64_t rows, int64_t cols, int block) {
    if (rows <= 0 || cols <= 0 || block <= 0) return 0;
    return align_up((size_t)cols * cols * sizeof(float)) + align_up((size_t)cols) + gptq_factor_workspace_size(cols) +
           sweep_ws_bytes(rows, cols, block);
}

gq_status gptq_quantize_layer(const void *W, gq_dtype wt, int64_t rows, int64_t cols, const float *H, int bits,
                              int group, int block, float damp, int32_t *qweight, float *scales, int32_t *qzeros,
                              uint8_t *codes, float *W_hat, float *row_err, void *ws, size_t ws_bytes,
                              gq_stream_t stream, int64_t *info) {
    if (!H) return GQ_EINVAL;
    gq_status st = check_sweep_args(W, wt, rows, cols, H, bits, group, block, qweight, scales, qzeros, codes, W_hat,
                                    row_err);
    if (st != GQ_OK) return st;
    if (!ws || !aligned(ws, kAlign) || ws_bytes < gptq_quantize_layer_workspace_size(rows, cols, block))
        return GQ_EWORKSPACE;
    char *p = (char *)ws;
    float *F = (float *)p;
    p += align_up((size_t)cols * cols * sizeof(float));
    uint8_t *dead = (uint8_t *)p;
    p += align_up((size_t)cols);
    void *fws = p;
    p += gptq_factor_workspace_size(cols);
    // The sweep workspace starts with its block-inverse region, which the
    // factorization fills directly when its panels coincide with the blocks.
    const bool uinv = factor_emits_uinv(cols, block);
    st = factor_impl(H, cols, damp, F, dead, fws, cs(stream), info, uinv ? (float *)p : nullptr, block, W,
                     wt == GQ_BF16, rows * cols);
    if (st != GQ_OK) return st;
    return sweep_impl(W, wt, rows, cols, F, dead, bits, group, block, qweight, scales, qzeros, codes, W_hat, row_err, p,
                      cs(stream), uinv);
}

size_t gptq_lora_basis_workspace_size(int64_t cols, int r) {
    if (cols <= 0 || r <= 0) return 0;
    return lora_basis_workspace_bytes(cols, r);
}

gq_status gptq_lora_basis(const float *H, int64_t cols, int r, float *Lt, float *lam, void *ws, size_t ws_bytes,
                          gq_stream_t stream) {
    if (!H || !Lt || cols <= 0) return GQ_EINVAL;
    if (r <= 0 || r > 64 || r > cols) return GQ_EINVAL;
    if (!ws || !aligned(ws, kAlign) || ws_bytes < lora_basis_workspace_bytes(cols, r)) return GQ_EWORKSPACE;
    return lora_basis_run(H, cols, r, Lt, lam, ws, cs(stream)) == cudaSuccess ? GQ_OK : GQ_ECUDA;
}

size_t gptq_intrinsic_lora_workspace_size(int64_t rows, int64_t cols, int r, int block) {
    if (rows <= 0 || cols <= 0 || r <= 0 || block <= 0) return 0;
    return lora_layout(rows, cols, r, block, nullptr, nullptr);
}

gq_status gptq_intrinsic_lora(const void *W, gq_dtype wt, int64_t rows, int64_t cols, const float *H,
                              const float *Lt, int r, int bits, int group, int block, float damp, int32_t *qweight,
                              float *scales, int32_t *qzeros, uint8_t *codes, float *W_hat, float *row_err,
                              float *R, void *ws, size_t ws_bytes, gq_stream_t stream, int64_t *info) {
    if (!H || !Lt || !R || !W_hat) return GQ_EINVAL;
    gq_status st = check_sweep_args(W, wt, rows, cols, H, bits, group, block, qweight, scales, qzeros, codes, W_hat,
                                    row_err);
    if (st != GQ_OK) return st;
    if (r <= 0 || r > 64 || r > cols) return GQ_EINVAL;
    if (!(damp > 0.f) || !(damp < INFINITY)) return GQ_EINVAL;
    if (!aligned(R, 4) || !aligned(Lt, 4)) return GQ_EINVAL;
    if (!ws || !aligned(ws, kAlign) || ws_bytes < gptq_intrinsic_lora_workspace_size(rows, cols, r, block))
        return GQ_EWORKSPACE;
    return intrinsic_impl(W, wt, rows, cols, H, Lt, r, bits, group, block, damp, qweight, scales, qzeros, codes,
                          W_hat, row_err, R, ws, cs(stream), info);
}

size_t gptq_packed_linear_workspace_size(int64_t n, int64_t rows, int64_t cols, int group, int r) {
    if (n <= 0 || rows <= 0 || cols <= 0 || group <= 0 || cols % group || r < 0 || r > 64) return 0;
    return packed_ws_bytes(n, rows, cols, group, r);
}

gq_status gptq_packed_linear(const void *X, int64_t n, int64_t ldx, const int32_t *qweight, const float *scales,
                             const int32_t *qzeros, int64_t rows, int64_t cols, int bits, int group, const float *A,
                             const float *B, int r, float *Y, int64_t ldy, void *ws, size_t ws_bytes,
                             gq_stream_t stream) {
    if (bits != 2 && bits != 3 && bits != 4) return GQ_EUNSUPPORTED;
    if (group <= 0 || group % 64) return GQ_EUNSUPPORTED;
    if (rows <= 0 || rows % 32 || rows > INT32_MAX || cols <= 0 || cols % group || cols > INT32_MAX) return GQ_EINVAL;
    if (n < 0 || n > (int64_t)65535 * 128 || r < 0 || r > 64) return GQ_EINVAL;
    if (n == 0) return GQ_OK;  // no token: nothing is read or written (X and Y may be NULL)
    if (!X || !qweight || !scales || !qzeros || !Y) return GQ_EINVAL;
    if (ldx < cols || ldx % 8 || !aligned(X, 16)) return GQ_EINVAL;
    if (ldy < rows || ldy % 4 || !aligned(Y, 16)) return GQ_EINVAL;
    if (!aligned(scales, 16) || !aligned(qweight, 16) || !aligned(qzeros, 4)) return GQ_EINVAL;
    if (r > 0 && (!A || !B || !aligned(A, 4) || !aligned(B, 4))) return GQ_EINVAL;
    const size_t need = gptq_packed_linear_workspace_size(n, rows, cols, group, r);
    if (need > 0 && (!ws || !aligned(ws, kAlign) || ws_bytes < need)) return GQ_EWORKSPACE;
    const cudaError_t e = packed_forward((const __nv_bfloat16 *)X, n, ldx, qweight, scales, qzeros, rows, cols, bits,
                                         group, r > 0 ? A : nullptr, r > 0 ? B : nullptr, r, Y, ldy, ws, cs(stream));
    return e == cudaSuccess ? GQ_OK : GQ_ECUDA;
}

size_t gptq_bidup_workspace_size(int64_t rows, int64_t cols) {
    if (rows <= 0 || cols <= 0) return 0;
    return bidup_workspace_bytes(rows, cols);
}

gq_status gptq_bidup(const void *W, gq_dtype wt, int64_t rows, int64_t cols, const float *H, const float *A,
                     const float *B, int r, int bits, int group, uint8_t *codes, const float *scales,
                     const int32_t *qzeros, float *W_hat, int32_t *qweight, unsigned long long *changed, void *ws,
                     size_t ws_bytes, gq_stream_t stream) {
    if (wt != GQ_F32 && wt != GQ_BF16) return GQ_EUNSUPPORTED;
    if (bits != 2 && bits != 3 && bits != 4) return GQ_EUNSUPPORTED;
    if (!W || !H || !codes || !scales || !qzeros || !W_hat) return GQ_EINVAL;
    if (rows <= 0 || cols <= 0 || rows % 32 || cols % 32) return GQ_EINVAL;
    if (group <= 0 || group % 32 || cols % group) return GQ_EINVAL;
    if (r < 0 || r > 64 || (r > 0 && (!A || !B))) return GQ_EINVAL;
    if (!aligned(H, 16) || !aligned(W_hat, 4) || !aligned(scales, 4) || !aligned(qzeros, 4)) return GQ_EINVAL;
    if ((qweight && !aligned(qweight, 4)) || (changed && !aligned(changed, 8))) return GQ_EINVAL;
    if (!ws || !aligned(ws, kAlign) || ws_bytes < bidup_workspace_bytes(rows, cols)) return GQ_EWORKSPACE;
    return bidup_run(W, wt == GQ_BF16, rows, cols, H, r > 0 ? A : nullptr, r > 0 ? B : nullptr, r, bits, group,
                     codes, scales, qzeros, W_hat, qweight, changed, ws, cs(stream)) == cudaSuccess
               ? GQ_OK
               : GQ_ECUDA;
}

gq_status gptq_quantize_rtn(const float *M, int64_t nrows, int64_t ncols, int bits, int group, float *M_hat,
                            uint8_t *codes, float *scales, uint8_t *zeros, gq_stream_t stream) {
    if (bits < 2 || bits > 8) return GQ_EUNSUPPORTED;
    if (!M || !M_hat || !scales || !zeros) return GQ_EINVAL;
    if (nrows <= 0 || ncols <= 0 || group <= 0 || ncols % group) return GQ_EINVAL;
    if (!aligned(M, 4) || !aligned(M_hat, 4) || !aligned(scales, 4)) return GQ_EINVAL;
    return rtn_launch(M, nrows, ncols, bits, group, M_hat, codes, scales, zeros, cs(stream)) == cudaSuccess
               ? GQ_OK
               : GQ_ECUDA;
}

gq_status gptq_weight_error(const void *W, gq_dtype wt, int64_t rows, int64_t cols, const float *W_hat, float *dW,
                            gq_stream_t stream) {
    if (wt != GQ_F32 && wt != GQ_BF16) return GQ_EUNSUPPORTED;
    if (!W || !W_hat || !dW || rows <= 0 || cols <= 0) return GQ_EINVAL;
    return weight_error_launch(W, wt == GQ_BF16, rows * cols, W_hat, dW, cs(stream)) == cudaSuccess ? GQ_OK : GQ_ECUDA;
}

size_t eora_compensate_workspace_size(int64_t rows, int64_t cols, int r) {
    if (rows <= 0 || cols <= 0 || r <= 0) return 0;
    return eora_workspace_bytes(rows, cols, r);
}

gq_status eora_compensate(const float *dW, int64_t rows, int64_t cols, const float *H, int r, float *A, float *B,
                          float *sigma, void *ws, size_t ws_bytes, gq_stream_t stream, int64_t *info) {
    if (!dW || !H || !A || !B || rows <= 0 || cols <= 0) return GQ_EINVAL;
    // Above 64 the eigenpairs come in locked chunks of 64, each from 128 vectors orthogonal to
    // the chunks before it, which needs cols >= r + 64.
    if (r <= 0 || r > 256 || r > rows || r > cols || (r > 64 && cols < (int64_t)r + 64)) return GQ_EINVAL;
    if (!ws || !aligned(ws, kAlign) || ws_bytes < eora_workspace_bytes(rows, cols, r)) return GQ_EWORKSPACE;
    unsigned long long bad = ULLONG_MAX;
    unsigned int finite = ~0u;
    if (eora_run(dW, rows, cols, H, r, A, B, sigma, ws, cs(stream), &bad, &finite) != cudaSuccess) return GQ_ECUDA;
    if (finite != ~0u) {
        if (info) *info = (finite & kNonFiniteH) ? 1 : 0;
        return GQ_ENONFINITE;
    }
    if (bad != ULLONG_MAX) {
        if (info) *info = cols - 1 - (int64_t)bad;
        return GQ_ENOTPD;
    }
    if (info) *info = -1;
    return GQ_OK;
}

gq_status gptq_code_decisions(const float *w, const float *s, int64_t n, float *k, gq_stream_t stream) {
    if (n < 0) return GQ_EINVAL;
    if (n == 0) return GQ_OK;
    if (!w || !s || !k) return GQ_EINVAL;
    return code_decisions_launch(w, s, n, k, cs(stream)) == cudaSuccess ? GQ_OK : GQ_ECUDA;
}

gq_status gptq_pack(const uint8_t *codes, int64_t rows, int64_t cols, int bits, int32_t *qweight, gq_stream_t stream) {
    if (bits != 2 && bits != 3 && bits != 4) return GQ_EUNSUPPORTED;
    if (!codes || !qweight || rows <= 0 || cols <= 0 || (cols * bits) % 32) return GQ_EINVAL;
    return pack_launch(codes, rows, cols, bits, qweight, cs(stream)) == cudaSuccess ? GQ_OK : GQ_ECUDA;
}

gq_status gptq_unpack(const int32_t *qweight, int64_t rows, int64_t cols, int bits, uint8_t *codes, gq_stream_t stream) {
    if (bits != 2 && bits != 3 && bits != 4) return GQ_EUNSUPPORTED;
    if (!codes || !qweight || rows <= 0 || cols <= 0 || (cols * bits) % 32) return GQ_EINVAL;
    return unpack_launch(qweight, rows, cols, bits, codes, cs(stream)) == cudaSuccess ? GQ_OK : GQ_ECUDA;
}

}  // extern "C"
