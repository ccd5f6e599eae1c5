// Hessian accumulation H += 2 X^T X for bf16 X on the fifth-generation tensor
// cores: the second-order statistics of the layer inputs that GPTQ's updates
// are built from ([GPTQ-wiki] "Enfoque Técnico"; [LowBit] section 2).
//
// Design (sm_103a):
// * Tiles of 256 x 256 features, only those on or above the diagonal; each
//   element of H is written by exactly one CTA: the upper triangle (c >= r)
//   directly and the strict lower triangle as the mirror, so H stays bit-for-bit
//   symmetric and the result is deterministic.
// * A = X^T[i-tile, tokens] and B = X[tokens, j-tile] are both read straight
//   from the row-major X (features contiguous): MN-major operands, loaded by
//   TMA as 64-token x 64-feature boxes with 128-byte swizzle.
// * A cluster of two CTAs computes one tile with tcgen05 cta_group::2 (see the
//   kernel's comment); warp 0 / lane 0 of each CTA issues its TMA loads, warp 1
//   / lane 0 of the even CTA issues the MMAs (kind::f16, bf16 x bf16 -> f32,
//   M = 256, N = 256, K = 16).
// * Epilogue: eight warps per CTA read their TMEM lanes (one output row each,
//   half of the columns) with tcgen05.ld after every 1024 tokens, add the
//   partial sums into float32 registers and finally add 2 * sum into H.
// * Every wait on an mbarrier is bounded (clock64 budget); on expiry the CTA
//   records an error flag, waits (again bounded) until the TMA loads and MMAs
//   it issued have completed, frees TMEM and returns.
#include "tc_common.cuh"

namespace gq {

__device__ unsigned int g_device_error = 0;  // bit 0: a bounded wait gave up

namespace {
using namespace tc;

// ---------------------------------------------------------------------------
// The CTA-pair kernel.  A cluster of two CTAs computes a 256 x 256 tile of H
// with tcgen05 cta_group::2: each CTA loads its own 128 features of the A side
// and its half (128) of the B side's 256 features, and one MMA of M = 256,
// N = 256 reads both CTAs' shared memory, so every operand byte brought from
// L2 feeds twice the multiply-adds of the single-CTA 128 x 256 tile (32 KB per
// CTA per 64 tokens instead of 48 KB).  Each CTA's TMEM receives its 128 rows
// of the tile (two 256-column buffers).  The tensor core's own accumulation
// loses about half an ulp of the running sum per step, so each buffer sums KF
// k-tiles (1024 tokens) and the epilogue warps add it into float32 registers
// (round-to-nearest) while the MMAs fill the other buffer.  The error of H grows
// with the period (1.0e-6 relative at 512 tokens, 2.1e-6 at 1024, measured on
// 262144 tokens); the longer period halves the flushes and took 5 % off the
// kernel's time.
// * The even CTA's loads count on its full barrier; the odd CTA's loads count
//   directly on the even CTA's peer barrier of the stage (the odd CTA's
//   producer arrives there with the stage's byte count before it issues them).
//   The even CTA's MMA thread waits for both barriers before it issues.  The MMA
//   thread's commits arrive on the empty barriers and accumulator-full
//   barriers of both CTAs; the epilogue warps of both CTAs release an
//   accumulator buffer on the even CTA's barrier.
// * Tiles: the 256-aligned tiles on or above the diagonal, in groups of P_GROUP
//   tile-rows, column by column within a group.
// * Every wait is bounded.  At the end the even CTA waits for its MMAs, the odd
//   CTA publishes how many stages it issued, and after a cluster barrier the
//   even CTA waits until every stage either CTA issued has landed (both kinds
//   of barrier are its own); a second cluster barrier (the even CTA's MMAs read
//   the odd CTA's shared memory, and the odd CTA's loads count on the even
//   CTA's barriers) precedes the freeing of TMEM.
// Stage depth: three stages of 128 tokens (64 KB per CTA each).  Measured on a
// 65536-token x 11008-feature input: 1330 TFLOP/s, against 1119 with four
// stages of 64 tokens and 1028 with seven (the same 192-224 KB of shared memory
// in fewer, larger stages issues fewer barrier round trips per MMA).
namespace pair {
constexpr int PT = 256;                           // tile rows and columns (128 rows per CTA)
#ifndef GQ_HP_TK
#define GQ_HP_TK 128
#endif
#ifndef GQ_HP_STAGES
#define GQ_HP_STAGES 3
#endif
constexpr int TK = GQ_HP_TK;                      // tokens per stage (a multiple of 64)
constexpr int STAGES = GQ_HP_STAGES;
constexpr int BOX = 64 * 64 * 2;                  // one TMA box: 64 tokens x 64 features, bf16
constexpr int CH = TK * 64 * 2;                   // one 64-feature chunk of the stage: TK tokens
constexpr int A_BYTES = 2 * CH;                   // this CTA's 128 A features
constexpr int B_BYTES = 2 * CH;                   // this CTA's 128 of the 256 B features
constexpr int STAGE = A_BYTES + B_BYTES;          // 64 KB at 128 tokens
constexpr int SMEM = STAGES * STAGE + 1024;
constexpr uint32_t TCOLS = 256;                   // TMEM columns per accumulator buffer
constexpr int KF = 1024 / TK;                     // k-tiles per TMEM period (1024 tokens)
constexpr int P_GROUP = 8;                        // tile-rows per scheduling group
constexpr int NWARPS = 10, EPI = 8;
}  // namespace pair

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(pair::NWARPS * 32, 1)
    hessian_pair_kernel(const __grid_constant__ CUtensorMap xmap, float *__restrict__ H, int cols, int n) {
    using namespace pair;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[STAGES];   // this CTA's half of the stage landed
    __shared__ __align__(8) uint64_t peer_bar[STAGES];   // (even CTA) the odd CTA's half landed
    __shared__ __align__(8) uint64_t empty_bar[STAGES];
    __shared__ __align__(8) uint64_t tfull[2];
    __shared__ __align__(8) uint64_t tempty[2];
    __shared__ __align__(8) uint64_t drain_bar;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    __shared__ int peer_issued;  // (even CTA) stages the odd CTA issued

    unsigned char *smem = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool lead = rank == 0;

    // This pair's tile (bi, bj), bj >= bi, among nb x nb 256-aligned tiles.
    const int nb = (cols + PT - 1) / PT;
    int t = blockIdx.x >> 1, g0 = 0;
    for (; g0 < nb; g0 += P_GROUP) {
        const int g1 = (g0 + P_GROUP) < nb ? (g0 + P_GROUP) : nb;
        int cnt = 0;
        for (int i = g0; i < g1; ++i) cnt += nb - i;
        if (t < cnt) break;
        t -= cnt;
    }
    const int g1 = (g0 + P_GROUP) < nb ? (g0 + P_GROUP) : nb;
    int bi = g0, bj = g0;
    for (; bj < nb; ++bj) {
        const int valid = (bj + 1 < g1 ? bj + 1 : g1) - g0;  // tile-rows of the group that reach column bj
        if (t < valid) {
            bi = g0 + t;
            break;
        }
        t -= valid;
    }
    const int r0 = bi * PT + (int)rank * 128;   // this CTA's 128 rows of the tile
    const int c0 = bj * PT;                     // the tile's 256 columns
    const int cb = c0 + (int)rank * 128;        // this CTA's B half
    const int ktiles = (n + TK - 1) / TK;
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
    cluster_sync();  // barriers of both CTAs initialised, TMEM allocated in both
    fence_after();
    const uint32_t tmem = tmem_slot;

    int issued = 0;  // (warp 0, lane 0) stages this CTA issued
    if (warp == 0) {
        if (lane == 0) {
            for (int kt = 0; kt < ktiles; ++kt, ++issued) {
                const int s = kt % STAGES;
                const uint32_t ph = (uint32_t)(kt / STAGES) & 1u;
                if (!mbar_wait(&empty_bar[s], ph ^ 1u) || *(volatile int *)&abort_flag) {
                    atomicOr(&g_device_error, 1u);
                    abort_flag = 1;
                    break;
                }
                unsigned char *st = smem + s * STAGE;
                const int y = kt * TK;
                // Four 64-feature chunks (A: r0, r0 + 64; B: cb, cb + 64), each TK tokens as
                // TK / 64 boxes one after the other.
                const int xs[4] = {r0, r0 + 64, cb, cb + 64};
                if (lead) {
                    mbar_arrive_expect_tx(&full_bar[s], STAGE);
#pragma unroll
                    for (int c = 0; c < 4; ++c)
#pragma unroll
                        for (int tb = 0; tb < TK / 64; ++tb)
                            tma_load_2d(st + c * CH + tb * BOX, &xmap, xs[c], y + tb * 64, &full_bar[s]);
                } else {
                    const uint32_t pb = cluster_addr(smem_u32(&peer_bar[s]), 0);
                    mbar_arrive_expect_tx_cluster(pb, STAGE);
#pragma unroll
                    for (int c = 0; c < 4; ++c)
#pragma unroll
                        for (int tb = 0; tb < TK / 64; ++tb)
                            tma_load_2d_to_peer_bar(st + c * CH + tb * BOX, &xmap, xs[c], y + tb * 64, pb);
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
            constexpr uint32_t idesc = make_idesc(2 * 128, PT);
            bool ok = true;
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
                    const uint32_t a0 = smem_u32(smem + s * STAGE);
                    const uint32_t b0 = a0 + A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < TK / 16; ++kk) {
                        // 16 tokens = two 8-row core-matrix groups (SBO = 1024 B apart);
                        // 64-feature chunks are CH bytes apart (LBO).
                        const uint64_t ad = smem_desc(a0 + kk * 2048, CH, 1024);
                        const uint64_t bd = smem_desc(b0 + kk * 2048, CH, 1024);
                        mma_bf16_pair(acc, ad, bd, idesc, (kt > p * KF || kk > 0) ? 1u : 0u);
                    }
                    mma_commit_pair(&empty_bar[s], 0x3);
                }
                if (!ok) break;
                mma_commit_pair(&tfull[b], 0x3);
            }
            if (!ok) {
                atomicOr(&g_device_error, 1u);
                abort_flag = 1;
            }
            mma_commit_pair(&drain_bar, 0x1);
            mbar_wait_for(&drain_bar, 0u, WAIT_BUDGET);
        }
        __syncwarp();
    } else {
        // Accumulator warps of both CTAs: TMEM lane quarter = warp % 4, column half = (warp - 2) / 4.
        const int q = warp & 3, half = (warp - 2) >> 2;
        float master[128];
#pragma unroll
        for (int i = 0; i < 128; ++i) master[i] = 0.f;
        bool ok = true;
        for (int p = 0; p < periods; ++p) {
            const int b = p & 1;
            const uint32_t u = (uint32_t)(p >> 1) & 1u;
            if (!mbar_wait(&tfull[b], u)) {
                ok = false;
                break;
            }
            __syncwarp();
            fence_after();
            const uint32_t base = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * TCOLS + half * 128);
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
            atomicOr(&g_device_error, 1u);
            abort_flag = 1;
        }
        __syncwarp();
        // H += 2 * master: upper triangle directly, strict lower as the mirror.
        const int r = r0 + q * 32 + lane;
        const int cc = c0 + half * 128;
        if (ok && r < cols && periods > 0) {
#pragma unroll
            for (int j = 0; j < 128; ++j) {
                const int c = cc + j;
                if (c < cols && c >= r) {
                    const float add = 2.f * master[j];
                    H[(int64_t)r * cols + c] += add;
                    if (c > r) H[(int64_t)c * cols + r] += add;
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

}  // namespace

namespace tc {
EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (EncodeTiledFn)p;
    }
    return fn;
}
}  // namespace tc

unsigned int read_and_clear_device_error() {
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v)) != cudaSuccess) return ~0u;
    const unsigned int zero = 0;
    if (v) cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero));
    return v;
}

cudaError_t hessian_set_wait_budget(long long cycles) { return tc::set_wait_budget_here(cycles); }

bool hessian_bf16_tc_supported(int64_t cols, const void *X, int64_t ldx) {
    if (cols < 64 || cols > (1 << 20) || cols % 8) return false;
    if (((uintptr_t)X) % 16 || ldx % 8) return false;
    return encode_fn() != nullptr;
}

cudaError_t hessian_bf16_tc(float *H, int64_t cols, const __nv_bfloat16 *X, int64_t n, int64_t ldx, cudaStream_t s) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const int64_t max_chunk = (int64_t)1 << 30;  // token coordinates are 32-bit
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(hessian_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             pair::SMEM);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const int nb = (int)((cols + pair::PT - 1) / pair::PT);
    const int tiles = nb * (nb + 1) / 2;
    for (int64_t t0 = 0; t0 < n; t0 += max_chunk) {
        const int64_t nc = (n - t0) < max_chunk ? (n - t0) : max_chunk;
        CUtensorMap map;
        cuuint64_t gdim[2] = {(cuuint64_t)cols, (cuuint64_t)nc};
        cuuint64_t gstride[1] = {(cuuint64_t)ldx * 2};
        cuuint32_t box[2] = {64, 64};
        cuuint32_t estr[2] = {1, 1};
        CUresult r = enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (void *)(X + t0 * ldx), gdim, gstride, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
        const int th = timing_begin(TK_HESSIAN, s);
        hessian_pair_kernel<<<2 * tiles, pair::NWARPS * 32, pair::SMEM, s>>>(map, H, (int)cols, (int)nc);
        count_launch();
        timing_end(th, s, (double)nc * (double)cols * (double)(cols + 1));
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace gq
