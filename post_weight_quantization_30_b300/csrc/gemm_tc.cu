// Float32-accurate GEMM on the fifth-generation tensor cores (sm_103a):
//     C = beta C + alpha A B^T      (A: M x K, B: N x K, both K contiguous)
// with every operand given as the pair (hi, lo) of a float32 value split into
// two tensor-float32 parts (x = hi + lo exactly; hi is x rounded to TF32,
// lo = x - hi).  Each product is formed as lo_A hi_B + hi_A lo_B + hi_A hi_B
// ("3xTF32"); the dropped lo_A lo_B term is below 2^-22 of |x y|.
//
// This is the GEMM of the deferred trailing update of the GPTQ sweep
// (W[:, later] -= E_blk U[blk, later], applied as an update of the pending
// deferred sums) and of the blocked Cholesky's trailing updates.
//
// Design:
// * One CTA per 128 x 128 output tile (tiles entirely above the diagonal can
//   be skipped).  Warp 0 / lane 0 issues TMA loads of the four operand tiles
//   (32 K-values = one 128-byte swizzle row each), three-stage mbarrier
//   pipeline, 64 KB per stage.  Warp 1 / lane 0 issues tcgen05.mma
//   (kind::tf32, M = 128, N = 128, K = 8), three per k-step.
// * The tensor core accumulates G_KF stages (256 K-values) into one of two
//   TMEM buffers; four epilogue warps add each partial into float32
//   registers with round-to-nearest while the next period fills the other
//   buffer.  Long in-TMEM accumulation is avoided because the tensor core's
//   own accumulation rounds less accurately than an IEEE add.
// * Every mbarrier wait is bounded; on expiry the CTA records the error flag
//   that gq_check_device reports, and exits without writing C.
#include "tc_common.cuh"

namespace gq {

// Bit 0: a bounded wait of this file's kernels gave up.  (Each translation
// unit has its own device flags: the library is built without relocatable
// device code.)
__device__ unsigned int g_gemm_error = 0;

namespace {
using namespace tc;

constexpr int GM = 128, GN = 128, GK = 32;
constexpr int G_STAGES = 3;
constexpr int TILE_A = GM * GK * 4;                  // 16 KB
constexpr int TILE_B = GN * GK * 4;                  // 16 KB
constexpr int G_STAGE = 2 * TILE_A + 2 * TILE_B;     // 64 KB
constexpr int G_SMEM = G_STAGES * G_STAGE + 1024;
constexpr uint32_t G_TMEM = GN;                      // columns per accumulator buffer
constexpr int G_KF = 8;                              // stages per TMEM period
constexpr int G_NWARPS = 6;                          // TMA, MMA, 4 epilogue warps

// Instruction descriptor, kind::tf32: D f32, A and B TF32 (format 2), both
// K-major, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_tf32(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_tf32_pair(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                              uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__global__ void __launch_bounds__(G_NWARPS * 32, 1)
    gemm3_kernel(const __grid_constant__ CUtensorMap ahi, const __grid_constant__ CUtensorMap alo,
                 const __grid_constant__ CUtensorMap bhi, const __grid_constant__ CUtensorMap blo, float *C,
                 int64_t ldc, int M, int N, int K, float alpha, float beta, int tri, float *Chi, float *Clo,
                 int64_t ldcs, int ktiles_per_z, int64_t c_zstride, int split_row0, int split_ncols, int one_term) {
    pdl_trigger();
    const int m0 = blockIdx.y * GM, n0 = blockIdx.x * GN;
    if (tri == 1 && n0 > m0 + GM - 1) return;  // tile entirely above the diagonal
    // Split K (gridDim.z > 1): slice z covers k-tiles [z * ktiles_per_z, ...) and
    // writes its partial product to C + z * c_zstride.
    const int kt_all = (K + GK - 1) / GK;
    const int kt0 = blockIdx.z * ktiles_per_z;
    const int kt1 = (kt0 + ktiles_per_z) < kt_all ? (kt0 + ktiles_per_z) : kt_all;
    C += (int64_t)blockIdx.z * c_zstride;

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[G_STAGES];
    __shared__ __align__(8) uint64_t empty_bar[G_STAGES];
    __shared__ __align__(8) uint64_t tfull[2];
    __shared__ __align__(8) uint64_t tempty[2];
    __shared__ __align__(8) uint64_t drain_bar;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    unsigned char *smem = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ktiles = kt1 > kt0 ? kt1 - kt0 : 0;
    const int periods = (ktiles + G_KF - 1) / G_KF;

    if (threadIdx.x == 0) {
        for (int s = 0; s < G_STAGES; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 4);
        }
        mbar_init(&drain_bar, 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_slot)),
                     "r"(2 * G_TMEM)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = tmem_slot;
    bool ok = true;
    pdl_wait();  // the operands and C come from earlier kernels

    if (warp == 0) {
        if (lane == 0) {
            int issued = 0;
            for (int kt = 0; kt < ktiles; ++kt, ++issued) {
                const int s = kt % G_STAGES;
                const uint32_t ph = (uint32_t)(kt / G_STAGES) & 1u;
                if (!mbar_wait(&empty_bar[s], ph ^ 1u) || *(volatile int *)&abort_flag) {
                    atomicOr(&g_gemm_error, 1u);
                    abort_flag = 1;
                    break;
                }
                unsigned char *st = smem + s * G_STAGE;
                mbar_arrive_expect_tx(&full_bar[s], one_term ? TILE_A + TILE_B : G_STAGE);
                const int x = (kt0 + kt) * GK;
                tma_load_2d(st, &ahi, x, m0, &full_bar[s]);
                tma_load_2d(st + 2 * TILE_A, &bhi, x, n0, &full_bar[s]);
                if (!one_term) {
                    tma_load_2d(st + TILE_A, &alo, x, m0, &full_bar[s]);
                    tma_load_2d(st + 2 * TILE_A + TILE_B, &blo, x, n0, &full_bar[s]);
                }
            }
            drain_loads<G_STAGES>(full_bar, issued);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_tf32(GM, GN);
            for (int p = 0; p < periods && ok; ++p) {
                const int b = p & 1;
                const uint32_t u = (uint32_t)(p >> 1) & 1u;
                if (!mbar_wait(&tempty[b], u ^ 1u)) {
                    ok = false;
                    break;
                }
                fence_after();
                const uint32_t acc = tmem + (uint32_t)(b * G_TMEM);
                const int k_end = (p + 1) * G_KF < ktiles ? (p + 1) * G_KF : ktiles;
                for (int kt = p * G_KF; kt < k_end; ++kt) {
                    const int s = kt % G_STAGES;
                    const uint32_t ph = (uint32_t)(kt / G_STAGES) & 1u;
                    if (!mbar_wait(&full_bar[s], ph)) {
                        ok = false;
                        break;
                    }
                    fence_after();
                    const uint32_t a_hi = smem_u32(smem + s * G_STAGE);
                    const uint32_t a_lo = a_hi + TILE_A;
                    const uint32_t b_hi = a_hi + 2 * TILE_A;
                    const uint32_t b_lo = b_hi + TILE_B;
#pragma unroll
                    for (int kk = 0; kk < GK / 8; ++kk) {
                        // K-major, 128-byte swizzle: 8-row groups 1024 B apart; a
                        // k-step of 8 TF32 values advances the start by 32 bytes.
                        const uint32_t off = kk * 32;
                        const uint64_t dah = smem_desc(a_hi + off, 16, 1024);
                        const uint64_t dal = smem_desc(a_lo + off, 16, 1024);
                        const uint64_t dbh = smem_desc(b_hi + off, 16, 1024);
                        const uint64_t dbl = smem_desc(b_lo + off, 16, 1024);
                        const uint32_t first = (kt == p * G_KF && kk == 0) ? 0u : 1u;
                        if (one_term) {
                            mma_tf32(acc, dah, dbh, idesc, first);
                        } else {
                            mma_tf32(acc, dal, dbh, idesc, first);
                            mma_tf32(acc, dah, dbl, idesc, 1u);
                            mma_tf32(acc, dah, dbh, idesc, 1u);
                        }
                    }
                    mma_commit(&empty_bar[s]);
                }
                mma_commit(&tfull[b]);
            }
            if (!ok) {
                atomicOr(&g_gemm_error, 1u);
                abort_flag = 1;
            }
            drain_mmas(&drain_bar);
        }
        __syncwarp();
    } else {
        // Epilogue warps: TMEM lane quarter = warp % 4; each thread owns one row x 128 columns.
        const int q = warp & 3;
        float master[GN];
#pragma unroll
        for (int i = 0; i < GN; ++i) master[i] = 0.f;
        for (int p = 0; p < periods; ++p) {
            const int b = p & 1;
            const uint32_t u = (uint32_t)(p >> 1) & 1u;
            if (!mbar_wait(&tfull[b], u)) {
                ok = false;
                break;
            }
            __syncwarp();
            fence_after();
            const uint32_t base = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * G_TMEM);
#pragma unroll
            for (int ch = 0; ch < GN / 32; ++ch) {
                float v[32];
                tmem_ld32(base + ch * 32, v);
#pragma unroll
                for (int i = 0; i < 32; ++i) master[ch * 32 + i] += v[i];
            }
            fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[b]);
        }
        if (!ok) {
            atomicOr(&g_gemm_error, 1u);
            abort_flag = 1;
        }
        __syncwarp();
        // Epilogue through shared memory (the pipeline stages are idle now): each
        // warp writes its 32 rows x 128 columns of partial sums there, then
        // reads C and writes the result one 512-byte row at a time, coalesced.
        // Row stride 132 floats keeps the float4 accesses free of bank conflicts.
        float *stage = reinterpret_cast<float *>(smem) + (size_t)q * 32 * (GN + 4);
        if (ok && periods > 0) {
#pragma unroll
            for (int j = 0; j < GN; j += 4)
                *reinterpret_cast<float4 *>(stage + lane * (GN + 4) + j) =
                    make_float4(master[j], master[j + 1], master[j + 2], master[j + 3]);
        }
        __syncwarp();
        const int c = n0 + lane * 4;  // this lane's 4 columns of every row
        const bool full4 = (c + 3 < N) && (ldc % 4) == 0 && ((uintptr_t)C % 16) == 0 &&
                           (!Chi || ((ldcs % 4) == 0 && ((uintptr_t)Chi % 16) == 0 && ((uintptr_t)Clo % 16) == 0));
        if (ok && periods > 0) {
            for (int rr0 = 0; rr0 < 32; rr0 += 8) {
                float4 old[8];
                if (beta != 0.f) {
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int r = m0 + q * 32 + rr0 + u;
                        old[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                        if (r < M) {
                            const float *cp = C + (int64_t)r * ldc + c;
                            if (full4) old[u] = *reinterpret_cast<const float4 *>(cp);
                            else {
                                if (c < N) old[u].x = cp[0];
                                if (c + 1 < N) old[u].y = cp[1];
                                if (c + 2 < N) old[u].z = cp[2];
                                if (c + 3 < N) old[u].w = cp[3];
                            }
                        }
                    }
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int rr = rr0 + u, r = m0 + q * 32 + rr;
                    if (r >= M || c >= N) continue;
                    const float4 a = *reinterpret_cast<const float4 *>(stage + rr * (GN + 4) + lane * 4);
                    float v[4] = {alpha * a.x, alpha * a.y, alpha * a.z, alpha * a.w};
                    if (beta != 0.f) {
                        v[0] = fmaf(beta, old[u].x, v[0]);
                        v[1] = fmaf(beta, old[u].y, v[1]);
                        v[2] = fmaf(beta, old[u].z, v[2]);
                        v[3] = fmaf(beta, old[u].w, v[3]);
                    }
                    float *cp = C + (int64_t)r * ldc + c;
                    float h[4], l[4];
                    // The split of the result goes to Chi / Clo for rows >= split_row0 and
                    // columns < split_ncols, at row r - split_row0.
                    const bool sp = Chi && r >= split_row0 && c < split_ncols;
                    const int64_t so = (int64_t)(r - split_row0) * ldcs + c;
                    if (sp) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            h[e] = tf32_hi(v[e]);
                            l[e] = v[e] - h[e];
                        }
                    }
                    if (full4 && (!sp || c + 3 < split_ncols)) {
                        *reinterpret_cast<float4 *>(cp) = make_float4(v[0], v[1], v[2], v[3]);
                        if (sp) {
                            *reinterpret_cast<float4 *>(Chi + so) = make_float4(h[0], h[1], h[2], h[3]);
                            *reinterpret_cast<float4 *>(Clo + so) = make_float4(l[0], l[1], l[2], l[3]);
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            if (c + e < N) {
                                cp[e] = v[e];
                                if (sp && c + e < split_ncols) {
                                    Chi[so + e] = h[e];
                                    Clo[so + e] = l[e];
                                }
                            }
                        }
                    }
                }
            }
        }
    }
    fence_before();
    __syncthreads();
    if (warp == 0) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(2 * G_TMEM) : "memory");
    }
}

// The product for one 128-column tile and a short K (the panel solves and the
// one-panel updates on the serial chains of the factor and the sweep), where a
// launch spends most of its time on C.  Two pipeline stages; eight epilogue
// warps (a 32-row lane quarter and 64 columns each); with beta != 0 the
// epilogue warps copy their part of C into shared memory (cp.async) while the
// MMAs run, so C is read from L2 once, overlapped, and the epilogue only adds,
// splits and stores.  No split-K.
namespace gsmall {
constexpr int STAGES = 2;
constexpr int NWARPS = 10;                     // TMA, MMA, 8 epilogue warps
constexpr int EPI = 8;
constexpr int SLD = 64 + 4;                    // staging row stride (floats)
constexpr int CBUF = EPI * 32 * SLD * 4;       // 32 rows x 64 columns per epilogue warp
constexpr int SMEM = STAGES * G_STAGE + CBUF + 1024;
constexpr int MAX_K = G_KF * GK;               // one TMEM period
}  // namespace gsmall

__global__ void __launch_bounds__(gsmall::NWARPS * 32, 1)
    gemm3_small_kernel(const __grid_constant__ CUtensorMap ahi, const __grid_constant__ CUtensorMap alo,
                       const __grid_constant__ CUtensorMap bhi, const __grid_constant__ CUtensorMap blo, float *C,
                       int64_t ldc, int M, int N, int K, float alpha, float beta, int tri, float *Chi, float *Clo,
                       int64_t ldcs, int split_row0, int split_ncols) {
    using namespace gsmall;
    pdl_trigger();
    const int m0 = blockIdx.y * GM, n0 = blockIdx.x * GN;
    if (tri == 1 && n0 > m0 + GM - 1) return;  // tile entirely above the diagonal

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[STAGES];
    __shared__ __align__(8) uint64_t empty_bar[STAGES];
    __shared__ __align__(8) uint64_t tfull;
    __shared__ __align__(8) uint64_t drain_bar;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    unsigned char *smem = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    float *cbuf = reinterpret_cast<float *>(smem + STAGES * G_STAGE);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ktiles = (K + GK - 1) / GK;  // <= G_KF: one TMEM period

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        mbar_init(&tfull, 1);
        mbar_init(&drain_bar, 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_slot)),
                     "r"(G_TMEM)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = tmem_slot;
    bool ok = true;
    pdl_wait();  // the operands and C come from earlier kernels

    if (warp == 0) {
        if (lane == 0) {
            int issued = 0;
            for (int kt = 0; kt < ktiles; ++kt, ++issued) {
                const int s = kt % STAGES;
                const uint32_t ph = (uint32_t)(kt / STAGES) & 1u;
                if (!mbar_wait(&empty_bar[s], ph ^ 1u) || *(volatile int *)&abort_flag) {
                    atomicOr(&g_gemm_error, 1u);
                    abort_flag = 1;
                    break;
                }
                unsigned char *st = smem + s * G_STAGE;
                mbar_arrive_expect_tx(&full_bar[s], G_STAGE);
                const int x = kt * GK;
                tma_load_2d(st, &ahi, x, m0, &full_bar[s]);
                tma_load_2d(st + TILE_A, &alo, x, m0, &full_bar[s]);
                tma_load_2d(st + 2 * TILE_A, &bhi, x, n0, &full_bar[s]);
                tma_load_2d(st + 2 * TILE_A + TILE_B, &blo, x, n0, &full_bar[s]);
            }
            drain_loads<STAGES>(full_bar, issued);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_tf32(GM, GN);
            for (int kt = 0; kt < ktiles; ++kt) {
                const int s = kt % STAGES;
                const uint32_t ph = (uint32_t)(kt / STAGES) & 1u;
                if (!mbar_wait(&full_bar[s], ph)) {
                    ok = false;
                    break;
                }
                fence_after();
                const uint32_t a_hi = smem_u32(smem + s * G_STAGE);
                const uint32_t a_lo = a_hi + TILE_A;
                const uint32_t b_hi = a_hi + 2 * TILE_A;
                const uint32_t b_lo = b_hi + TILE_B;
#pragma unroll
                for (int kk = 0; kk < GK / 8; ++kk) {
                    const uint32_t off = kk * 32;
                    const uint64_t dah = smem_desc(a_hi + off, 16, 1024);
                    const uint64_t dal = smem_desc(a_lo + off, 16, 1024);
                    const uint64_t dbh = smem_desc(b_hi + off, 16, 1024);
                    const uint64_t dbl = smem_desc(b_lo + off, 16, 1024);
                    const uint32_t first = (kt == 0 && kk == 0) ? 0u : 1u;
                    mma_tf32(tmem, dal, dbh, idesc, first);
                    mma_tf32(tmem, dah, dbl, idesc, 1u);
                    mma_tf32(tmem, dah, dbh, idesc, 1u);
                }
                mma_commit(&empty_bar[s]);
            }
            if (ok) mma_commit(&tfull);
            if (!ok) {
                atomicOr(&g_gemm_error, 1u);
                abort_flag = 1;
            }
            drain_mmas(&drain_bar);
        }
        __syncwarp();
    } else {
        // Epilogue warp: TMEM lane quarter q (rows q*32 + lane), columns h*64 .. h*64 + 63 of the tile.
        const int q = warp & 3, h = (warp - 2) >> 2;
        float *stage = cbuf + (size_t)(h * 4 + q) * 32 * SLD;
        const int r = m0 + q * 32 + lane;   // this thread's row (phase A)
        const int cl = n0 + h * 64;         // first column of this warp
        const bool vec = (ldc % 4) == 0 && ((uintptr_t)C % 16) == 0;
        // C of this thread's row into shared memory while the MMAs run.
        if (beta != 0.f) {
            if (r < M) {
                const float *cp = C + (int64_t)r * ldc + cl;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float *dst = stage + lane * SLD + 4 * i;
                    const int c = cl + 4 * i;
                    if (vec && c + 3 < N) {
                        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(cp + 4 * i)
                                     : "memory");
                    } else {
#pragma unroll
                        for (int e = 0; e < 4; ++e) dst[e] = (c + e < N) ? cp[4 * i + e] : 0.f;
                    }
                }
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
        }
        float acc[64];
        if (!mbar_wait(&tfull, 0u)) ok = false;
        __syncwarp();
        fence_after();
        if (ok) {
            const uint32_t base = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(h * 64);
            float v[32];
            tmem_ld32(base, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[i] = v[i];
            tmem_ld32(base + 32, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[32 + i] = v[i];
        }
        fence_before();
        if (beta != 0.f) asm volatile("cp.async.wait_group 0;" ::: "memory");
        __syncwarp();
        if (!ok) {
            atomicOr(&g_gemm_error, 1u);
            abort_flag = 1;
        }
        // Phase A (one row per thread): v = alpha acc + beta C, in place in the staging rows.
        if (ok && ktiles > 0) {
#pragma unroll
            for (int j = 0; j < 64; j += 4) {
                float4 *sp = reinterpret_cast<float4 *>(stage + lane * SLD + j);
                float4 o = make_float4(alpha * acc[j], alpha * acc[j + 1], alpha * acc[j + 2], alpha * acc[j + 3]);
                if (beta != 0.f) {
                    const float4 cv = *sp;
                    o.x = fmaf(beta, cv.x, o.x);
                    o.y = fmaf(beta, cv.y, o.y);
                    o.z = fmaf(beta, cv.z, o.z);
                    o.w = fmaf(beta, cv.w, o.w);
                }
                *sp = o;
            }
        }
        __syncwarp();
        // Phase B (coalesced): 16 lanes per row, 4 columns each, two rows per step.
        const int c = cl + (lane & 15) * 4;
        const bool full4 = vec && (c + 3 < N) &&
                           (!Chi || ((ldcs % 4) == 0 && ((uintptr_t)Chi % 16) == 0 && ((uintptr_t)Clo % 16) == 0));
        if (ok && ktiles > 0 && c < N) {
            for (int rr = lane >> 4; rr < 32; rr += 2) {
                const int row = m0 + q * 32 + rr;
                if (row >= M) break;
                const float4 a = *reinterpret_cast<const float4 *>(stage + rr * SLD + (lane & 15) * 4);
                const float vv[4] = {a.x, a.y, a.z, a.w};
                float *cp = C + (int64_t)row * ldc + c;
                const bool sp = Chi && row >= split_row0 && c < split_ncols;
                const int64_t so = (int64_t)(row - split_row0) * ldcs + c;
                float hh[4], ll[4];
                if (sp) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        hh[e] = tf32_hi(vv[e]);
                        ll[e] = vv[e] - hh[e];
                    }
                }
                if (full4 && (!sp || c + 3 < split_ncols)) {
                    *reinterpret_cast<float4 *>(cp) = a;
                    if (sp) {
                        *reinterpret_cast<float4 *>(Chi + so) = make_float4(hh[0], hh[1], hh[2], hh[3]);
                        *reinterpret_cast<float4 *>(Clo + so) = make_float4(ll[0], ll[1], ll[2], ll[3]);
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        if (c + e < N) {
                            cp[e] = vv[e];
                            if (sp && c + e < split_ncols) {
                                Chi[so + e] = hh[e];
                                Clo[so + e] = ll[e];
                            }
                        }
                    }
                }
            }
        }
    }
    fence_before();
    __syncthreads();
    if (warp == 0) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(G_TMEM) : "memory");
    }
}

// The same product on CTA pairs, for outputs wider than one tile: a cluster of
// two CTAs computes a 256 x 256 tile with tcgen05 cta_group::2 (M = 256 over
// the two CTAs' 128 rows, N = 256 over their halves of the 256 B rows), so each
// operand byte brought from L2 feeds twice the multiply-adds of the 128 x 128
// tile: 64 KB per CTA per 32 K-values carry 128 x 256 outputs instead of
// 128 x 128.  The pipeline is the Hessian pair kernel's: the even CTA's loads
// count on its full barrier and the odd CTA's directly on the even CTA's peer
// barrier, the even CTA's MMA thread commits to the barriers of both, the
// epilogue warps of both release an accumulator buffer on the even CTA's
// barrier, and the end is two cluster barriers around the even CTA's wait for
// every stage either CTA issued.  Eight epilogue warps per CTA (one row and 128 columns
// per thread) add the flushed partial sums and apply C = beta C + alpha A B^T
// through shared memory, as above.  tri = 1 skips the pair tiles entirely above
// the diagonal; tri = 3 (B lower triangular: B(k, n) = 0 for k > n) stops each
// tile's K loop after the tile's last column.  No split-K.
namespace gpair {
constexpr int PT = 256;                  // pair tile rows and columns
constexpr int TILE = 128 * GK * 4;       // 16 KB: 128 rows x 32 K-values
constexpr int STAGE = 4 * TILE;          // A hi, A lo, B hi, B lo (this CTA's halves)
constexpr int STAGES = 3;
constexpr int SMEM = STAGES * STAGE + 1024;
constexpr uint32_t TCOLS = 256;
constexpr int KF = 8;                    // stages per TMEM period (256 K-values)
constexpr int NWARPS = 10, EPI = 8;
constexpr int SLD = 128 + 4;             // staging row stride (floats)
}  // namespace gpair

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(gpair::NWARPS * 32, 1)
    gemm3_pair_kernel(const __grid_constant__ CUtensorMap ahi, const __grid_constant__ CUtensorMap alo,
                      const __grid_constant__ CUtensorMap bhi, const __grid_constant__ CUtensorMap blo, float *C,
                      int64_t ldc, int M, int N, int K, float alpha, float beta, int tri, float *Chi, float *Clo,
                      int64_t ldcs, int split_row0, int split_ncols) {
    using namespace gpair;
    pdl_trigger();
    const uint32_t rank = cluster_ctarank();
    const bool lead = rank == 0;
    const int pm0 = blockIdx.y * PT, n0 = (blockIdx.x >> 1) * PT;
    if (tri == 1 && n0 > pm0 + PT - 1) return;  // the whole pair tile is above the diagonal (both CTAs agree)
    const int m0 = pm0 + (int)rank * 128;       // this CTA's rows
    const int nb0 = n0 + (int)rank * 128;       // this CTA's B rows

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[STAGES];
    __shared__ __align__(8) uint64_t peer_bar[STAGES];
    __shared__ __align__(8) uint64_t empty_bar[STAGES];
    __shared__ __align__(8) uint64_t tfull[2];
    __shared__ __align__(8) uint64_t tempty[2];
    __shared__ __align__(8) uint64_t drain_bar;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    __shared__ int peer_issued;  // (even CTA) stages the odd CTA issued

    unsigned char *smem = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // tri = 3: B(k, n) = 0 for k > n, so this tile's columns n < n0 + PT need k < n0 + PT only.
    const int keff = (tri == 3 && n0 + PT < K) ? n0 + PT : K;
    const int ktiles = (keff + GK - 1) / GK;
    const int periods = (ktiles + KF - 1) / KF;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&peer_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 2 * EPI);
        }
        mbar_init(&drain_bar, 1);
        abort_flag = 0;
        peer_issued = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_slot)),
                     "r"(2 * TCOLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    fence_before();
    cluster_sync();
    fence_after();
    const uint32_t tmem = tmem_slot;
    bool ok = true;
    pdl_wait();  // the operands and C come from earlier kernels

    int issued = 0;  // (warp 0, lane 0) stages this CTA issued
    if (warp == 0) {
        if (lane == 0) {
            for (int kt = 0; kt < ktiles; ++kt, ++issued) {
                const int s = kt % STAGES;
                const uint32_t ph = (uint32_t)(kt / STAGES) & 1u;
                if (!mbar_wait(&empty_bar[s], ph ^ 1u) || *(volatile int *)&abort_flag) {
                    atomicOr(&g_gemm_error, 1u);
                    abort_flag = 1;
                    break;
                }
                unsigned char *st = smem + s * STAGE;
                const int x = kt * GK;
                if (lead) {
                    mbar_arrive_expect_tx(&full_bar[s], STAGE);
                    tma_load_2d(st, &ahi, x, m0, &full_bar[s]);
                    tma_load_2d(st + TILE, &alo, x, m0, &full_bar[s]);
                    tma_load_2d(st + 2 * TILE, &bhi, x, nb0, &full_bar[s]);
                    tma_load_2d(st + 3 * TILE, &blo, x, nb0, &full_bar[s]);
                } else {
                    const uint32_t pb = cluster_addr(smem_u32(&peer_bar[s]), 0);
                    mbar_arrive_expect_tx_cluster(pb, STAGE);
                    tma_load_2d_to_peer_bar(st, &ahi, x, m0, pb);
                    tma_load_2d_to_peer_bar(st + TILE, &alo, x, m0, pb);
                    tma_load_2d_to_peer_bar(st + 2 * TILE, &bhi, x, nb0, pb);
                    tma_load_2d_to_peer_bar(st + 3 * TILE, &blo, x, nb0, pb);
                }
            }
            if (!lead) {
                asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr(smem_u32(&peer_issued), 0)),
                             "r"(issued)
                             : "memory");
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0 && lead) {
            constexpr uint32_t idesc = idesc_tf32(PT, PT);
            for (int p = 0; p < periods && ok; ++p) {
                const int b = p & 1;
                const uint32_t u = (uint32_t)(p >> 1) & 1u;
                if (!mbar_wait(&tempty[b], u ^ 1u)) {
                    ok = false;
                    break;
                }
                fence_after();
                const uint32_t acc = tmem + (uint32_t)(b * TCOLS);
                const int k_end = (p + 1) * KF < ktiles ? (p + 1) * KF : ktiles;
                for (int kt = p * KF; kt < k_end; ++kt) {
                    const int s = kt % STAGES;
                    const uint32_t ph = (uint32_t)(kt / STAGES) & 1u;
                    if (!mbar_wait(&full_bar[s], ph) || !mbar_wait(&peer_bar[s], ph)) {
                        ok = false;
                        break;
                    }
                    fence_after();
                    const uint32_t a_hi = smem_u32(smem + s * STAGE);
                    const uint32_t a_lo = a_hi + TILE;
                    const uint32_t b_hi = a_hi + 2 * TILE;
                    const uint32_t b_lo = a_hi + 3 * TILE;
#pragma unroll
                    for (int kk = 0; kk < GK / 8; ++kk) {
                        const uint32_t off = kk * 32;
                        const uint64_t dah = smem_desc(a_hi + off, 16, 1024);
                        const uint64_t dal = smem_desc(a_lo + off, 16, 1024);
                        const uint64_t dbh = smem_desc(b_hi + off, 16, 1024);
                        const uint64_t dbl = smem_desc(b_lo + off, 16, 1024);
                        const uint32_t first = (kt == p * KF && kk == 0) ? 0u : 1u;
                        mma_tf32_pair(acc, dal, dbh, idesc, first);
                        mma_tf32_pair(acc, dah, dbl, idesc, 1u);
                        mma_tf32_pair(acc, dah, dbh, idesc, 1u);
                    }
                    mma_commit_pair(&empty_bar[s], 0x3);
                }
                if (!ok) break;
                mma_commit_pair(&tfull[b], 0x3);
            }
            if (!ok) {
                atomicOr(&g_gemm_error, 1u);
                abort_flag = 1;
            }
            mma_commit_pair(&drain_bar, 0x1);
            mbar_wait_for(&drain_bar, 0u, WAIT_BUDGET);
        }
        __syncwarp();
    } else {
        // Epilogue warps of both CTAs: TMEM lane quarter q = warp % 4, column half h.
        const int q = warp & 3, h = (warp - 2) >> 2;
        float master[128];
#pragma unroll
        for (int i = 0; i < 128; ++i) master[i] = 0.f;
        for (int p = 0; p < periods; ++p) {
            const int b = p & 1;
            const uint32_t u = (uint32_t)(p >> 1) & 1u;
            if (!mbar_wait(&tfull[b], u)) {
                ok = false;
                break;
            }
            __syncwarp();
            fence_after();
            const uint32_t base = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * TCOLS + h * 128);
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
                float v[32];
                tmem_ld32(base + ch * 32, v);
#pragma unroll
                for (int i = 0; i < 32; ++i) master[ch * 32 + i] += v[i];
            }
            fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(cluster_addr(smem_u32(&tempty[b]), 0));
        }
        if (!ok) {
            atomicOr(&g_gemm_error, 1u);
            abort_flag = 1;
        }
        __syncwarp();
        // Through shared memory (the pipeline stages are idle now): this warp's 32 rows x
        // 128 columns, then C read and written one 512-byte row segment at a time.
        float *stage = reinterpret_cast<float *>(smem) + (size_t)(h * 4 + q) * 32 * SLD;
        if (ok && periods > 0) {
#pragma unroll
            for (int j = 0; j < 128; j += 4)
                *reinterpret_cast<float4 *>(stage + lane * SLD + j) =
                    make_float4(master[j], master[j + 1], master[j + 2], master[j + 3]);
        }
        __syncwarp();
        const int c = n0 + h * 128 + lane * 4;  // this lane's 4 columns of every row
        const bool full4 = (c + 3 < N) && (ldc % 4) == 0 && ((uintptr_t)C % 16) == 0 &&
                           (!Chi || ((ldcs % 4) == 0 && ((uintptr_t)Chi % 16) == 0 && ((uintptr_t)Clo % 16) == 0));
        if (ok && periods > 0) {
            for (int rr0 = 0; rr0 < 32; rr0 += 8) {
                float4 old[8];
                if (beta != 0.f) {
#pragma unroll
                    for (int uu = 0; uu < 8; ++uu) {
                        const int r = m0 + q * 32 + rr0 + uu;
                        old[uu] = make_float4(0.f, 0.f, 0.f, 0.f);
                        if (r < M) {
                            const float *cp = C + (int64_t)r * ldc + c;
                            if (full4) old[uu] = *reinterpret_cast<const float4 *>(cp);
                            else {
                                if (c < N) old[uu].x = cp[0];
                                if (c + 1 < N) old[uu].y = cp[1];
                                if (c + 2 < N) old[uu].z = cp[2];
                                if (c + 3 < N) old[uu].w = cp[3];
                            }
                        }
                    }
                }
#pragma unroll
                for (int uu = 0; uu < 8; ++uu) {
                    const int rr = rr0 + uu, r = m0 + q * 32 + rr;
                    if (r >= M || c >= N) continue;
                    const float4 a = *reinterpret_cast<const float4 *>(stage + rr * SLD + lane * 4);
                    float v[4] = {alpha * a.x, alpha * a.y, alpha * a.z, alpha * a.w};
                    if (beta != 0.f) {
                        v[0] = fmaf(beta, old[uu].x, v[0]);
                        v[1] = fmaf(beta, old[uu].y, v[1]);
                        v[2] = fmaf(beta, old[uu].z, v[2]);
                        v[3] = fmaf(beta, old[uu].w, v[3]);
                    }
                    float *cp = C + (int64_t)r * ldc + c;
                    float hh[4], ll[4];
                    const bool sp = Chi && r >= split_row0 && c < split_ncols;
                    const int64_t so = (int64_t)(r - split_row0) * ldcs + c;
                    if (sp) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            hh[e] = tf32_hi(v[e]);
                            ll[e] = v[e] - hh[e];
                        }
                    }
                    if (full4 && (!sp || c + 3 < split_ncols)) {
                        *reinterpret_cast<float4 *>(cp) = make_float4(v[0], v[1], v[2], v[3]);
                        if (sp) {
                            *reinterpret_cast<float4 *>(Chi + so) = make_float4(hh[0], hh[1], hh[2], hh[3]);
                            *reinterpret_cast<float4 *>(Clo + so) = make_float4(ll[0], ll[1], ll[2], ll[3]);
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            if (c + e < N) {
                                cp[e] = v[e];
                                if (sp && c + e < split_ncols) {
                                    Chi[so + e] = hh[e];
                                    Clo[so + e] = ll[e];
                                }
                            }
                        }
                    }
                }
            }
        }
    }
    fence_before();
    cluster_sync();  // main loops done in both CTAs; the odd CTA's stage count is visible
    if (warp == 0 && lane == 0 && lead) {
        drain_loads<STAGES>(full_bar, issued);
        drain_loads<STAGES>(peer_bar, *(volatile int *)&peer_issued);
    }
    __syncwarp();
    cluster_sync();  // every load has landed; the even CTA's MMAs are done with both CTAs' memory
    if (warp == 0) {
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(2 * TCOLS) : "memory");
    }
}

__global__ void split_kernel(const float *__restrict__ src, int64_t rows, int64_t cols, int64_t lds,
                             float *__restrict__ hi, float *__restrict__ lo, int64_t ldd) {
    pdl_trigger();
    pdl_wait();
    const int64_t n = rows * cols;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / cols, c = i % cols;
        const float x = src[r * lds + c];
        const float h = tf32_hi(x);
        hi[r * ldd + c] = h;
        lo[r * ldd + c] = x - h;
    }
}

// dst = src^T split: hi[c][r] = tf32(src[r][c]), lo = src - hi.  32 x 32 tiles
// through shared memory so both the reads and the writes are coalesced.
__global__ void split_transpose_kernel(const float *__restrict__ src, int64_t rows, int64_t cols, int64_t lds,
                                       float *__restrict__ hi, float *__restrict__ lo, int64_t ldd) {
    __shared__ float tile[32][33];
    const int64_t r0 = (int64_t)blockIdx.y * 32, c0 = (int64_t)blockIdx.x * 32;
    for (int i = threadIdx.y; i < 32; i += blockDim.y) {
        const int64_t r = r0 + i, c = c0 + threadIdx.x;
        tile[i][threadIdx.x] = (r < rows && c < cols) ? src[r * lds + c] : 0.f;
    }
    __syncthreads();
    for (int i = threadIdx.y; i < 32; i += blockDim.y) {
        const int64_t c = c0 + i, r = r0 + threadIdx.x;
        if (c < cols && r < rows) {
            const float x = tile[threadIdx.x][i];
            const float h = tf32_hi(x);
            hi[c * ldd + r] = h;
            lo[c * ldd + r] = x - h;
        }
    }
}

bool make_map(CUtensorMap *map, const float *base, int64_t inner, int64_t outer, int64_t ld, int box_outer) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t gdim[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
    cuuint64_t gstride[1] = {(cuuint64_t)ld * 4};
    cuuint32_t box[2] = {(cuuint32_t)GK, (cuuint32_t)box_outer};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, (void *)base, gdim, gstride, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t gemm_set_wait_budget(long long cycles) { return tc::set_wait_budget_here(cycles); }

unsigned int gemm_read_and_clear_error() {
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_gemm_error, sizeof(v)) != cudaSuccess) return ~0u;
    const unsigned int zero = 0;
    if (v) cudaMemcpyToSymbol(g_gemm_error, &zero, sizeof(zero));
    return v;
}

bool gemm3_supported(const void *p, int64_t ld) { return ((uintptr_t)p % 16) == 0 && (ld % 4) == 0; }

cudaError_t gemm3(int64_t M, int64_t N, int64_t K, float alpha, const float *Ahi, const float *Alo, int64_t lda,
                  const float *Bhi, const float *Blo, int64_t ldb, float beta, float *C, int64_t ldc, int tri,
                  float *Chi, float *Clo, int64_t ldcs, cudaStream_t s, int split_row0, int split_ncols) {
    if (split_ncols < 0) split_ncols = (int)N;
    if (M <= 0 || N <= 0) return cudaSuccess;
    if (K <= 0 || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return cudaErrorInvalidValue;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(gemm3_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, G_SMEM);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(gemm3_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, gpair::SMEM);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    CUtensorMap mah, mal, mbh, mbl;
    if (!make_map(&mah, Ahi, K, M, lda, GM) || !make_map(&mal, Alo, K, M, lda, GM) ||
        !make_map(&mbh, Bhi, K, N, ldb, GN) || !make_map(&mbl, Blo, K, N, ldb, GN))
        return cudaErrorInvalidValue;
    // Useful products: all M x N outputs, or those on and below the diagonal for tri = 1;
    // for tri = 3 (B lower triangular) output column n takes min(K, n + 1) products.
    const double outs = tri == 1 ? (M >= N ? (double)M * N - (double)N * (N - 1) / 2 : (double)M * (M + 1) / 2)
                                 : (double)M * N;
    double prods = outs * (double)K;
    if (tri == 3)
        prods = (double)M * (N <= K ? (double)N * (N + 1) / 2 : (double)K * (K + 1) / 2 + (double)(N - K) * K);
    if (M > GM && N > GN) {
        // Wider than one tile both ways: 256 x 256 tiles on CTA pairs (the boxes stay 128 rows:
        // each CTA loads its 128 rows of A and its 128 of the pair's 256 rows of B).
        dim3 pgrid((unsigned)(2 * ((N + gpair::PT - 1) / gpair::PT)), (unsigned)((M + gpair::PT - 1) / gpair::PT));
        const int th = timing_begin(TK_GEMM3, s);
        const cudaError_t e = launch_pdl(gemm3_pair_kernel, pgrid, dim3(gpair::NWARPS * 32), gpair::SMEM, s, mah, mal,
                                         mbh, mbl, C, ldc, (int)M, (int)N, (int)K, alpha, beta, tri, Chi, Clo, ldcs,
                                         split_row0, split_ncols);
        count_launch();
        timing_end(th, s, 2.0 * prods);
        return e;
    }
    dim3 grid((unsigned)((N + GN - 1) / GN), (unsigned)((M + GM - 1) / GM));
    // The one-CTA kernels know tri = 0 and 1 only; with tri = 3 they also take the (zero) products k > n.
    const int tri1 = tri == 1 ? 1 : 0;
    if (N <= GN && K <= gsmall::MAX_K) {
        // One column tile, short K: the latency-bound shape of the serial chains.
        static bool small_attr = false;
        if (!small_attr) {
            cudaError_t e = cudaFuncSetAttribute(gemm3_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 gsmall::SMEM);
            if (e != cudaSuccess) return e;
            small_attr = true;
        }
        const int th = timing_begin(TK_GEMM3, s);
        const cudaError_t e = launch_pdl(gemm3_small_kernel, grid, dim3(gsmall::NWARPS * 32), gsmall::SMEM, s, mah,
                                         mal, mbh, mbl, C, ldc, (int)M, (int)N, (int)K, alpha, beta, tri1, Chi, Clo,
                                         ldcs, split_row0, split_ncols);
        count_launch();
        timing_end(th, s, 2.0 * prods);
        return e;
    }
    const int kt_all = (int)((K + GK - 1) / GK);
    const int th = timing_begin(TK_GEMM3, s);
    const cudaError_t e = launch_pdl(gemm3_kernel, grid, dim3(G_NWARPS * 32), G_SMEM, s, mah, mal, mbh, mbl, C, ldc,
                                     (int)M, (int)N, (int)K, alpha, beta, tri1, Chi, Clo, ldcs, kt_all, (int64_t)0,
                                     split_row0, split_ncols, 0);
    count_launch();
    timing_end(th, s, 2.0 * prods);
    return e;
}

cudaError_t gemm3_splitk(int64_t M, int64_t N, int64_t K, const float *Ahi, const float *Alo, int64_t lda,
                         const float *Bhi, const float *Blo, int64_t ldb, float *C, float *partials, int slices,
                         cudaStream_t s, bool one_term) {
    if (M <= 0 || N <= 0) return cudaSuccess;
    if (K <= 0 || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX || slices < 1) return cudaErrorInvalidValue;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(gemm3_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, G_SMEM);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    // One term: the lo operands are never read; their maps repeat the hi ones.
    if (one_term) {
        Alo = Ahi;
        Blo = Bhi;
    }
    CUtensorMap mah, mal, mbh, mbl;
    if (!make_map(&mah, Ahi, K, M, lda, GM) || !make_map(&mal, Alo, K, M, lda, GM) ||
        !make_map(&mbh, Bhi, K, N, ldb, GN) || !make_map(&mbl, Blo, K, N, ldb, GN))
        return cudaErrorInvalidValue;
    const int kt_all = (int)((K + GK - 1) / GK);
    const int per = (kt_all + slices - 1) / slices;
    const int z = (kt_all + per - 1) / per;
    dim3 grid((unsigned)((N + GN - 1) / GN), (unsigned)((M + GM - 1) / GM), (unsigned)z);
    const int th = timing_begin(one_term ? TK_GEMM_TF32 : TK_GEMM3, s);
    cudaError_t e = launch_pdl(gemm3_kernel, grid, dim3(G_NWARPS * 32), G_SMEM, s, mah, mal, mbh, mbl, partials,
                               (int64_t)N, (int)M, (int)N, (int)K, 1.f, 0.f, 0, (float *)nullptr, (float *)nullptr,
                               (int64_t)0, per, M * N, 0, 0, one_term ? 1 : 0);
    count_launch();
    timing_end(th, s, 2.0 * (double)M * (double)N * (double)K);
    if (e != cudaSuccess) return e;
    return sum_slices(partials, z, M * N, C, s);
}

cudaError_t split_transpose_tf32(const float *src, int64_t rows, int64_t cols, int64_t lds, float *hi, float *lo,
                                 int64_t ldd, cudaStream_t s) {
    if (rows <= 0 || cols <= 0) return cudaSuccess;
    dim3 grid((unsigned)((cols + 31) / 32), (unsigned)((rows + 31) / 32));
    split_transpose_kernel<<<grid, dim3(32, 8), 0, s>>>(src, rows, cols, lds, hi, lo, ldd);
    count_launch();
    return cudaGetLastError();
}

cudaError_t split_tf32(const float *src, int64_t rows, int64_t cols, int64_t lds, float *hi, float *lo, int64_t ldd,
                       cudaStream_t s) {
    const int64_t n = rows * cols;
    if (n <= 0) return cudaSuccess;
    int64_t g = (n + 255) / 256;
    if (g > 148 * 16) g = 148 * 16;
    const cudaError_t e = launch_pdl(split_kernel, dim3((unsigned)g), dim3(256), 0, s, src, rows, cols, lds, hi, lo, ldd);
    count_launch();
    return e;
}

}  // namespace gq
