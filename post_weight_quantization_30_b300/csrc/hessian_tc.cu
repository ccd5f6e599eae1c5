// Hessian accumulation H += 2 X^T X for bf16 X on the fifth-generation tensor
// cores: the second-order statistics of the layer inputs that GPTQ's updates
// are built from ([GPTQ-wiki] "Enfoque Técnico"; [LowBit] section 2).
//
// Design (sm_103a):
// * One CTA per output tile of 128 x 256 features, only for tiles that touch the
//   upper triangle; each element of H is written by exactly one CTA: the
//   upper triangle (c >= r) directly and the strict lower triangle as the
//   mirror, so H stays bit-for-bit symmetric and the result is deterministic.
// * A = X^T[i-tile, tokens] and B = X[tokens, j-tile] are both read straight
//   from the row-major X (features contiguous): MN-major operands, loaded by
//   TMA as 64-token x 64-feature boxes with 128-byte swizzle.  Four-stage
//   mbarrier pipeline, 48 KB per stage.
// * Warp 0 / lane 0 issues the TMA loads, warp 1 / lane 0 issues
//   tcgen05.mma (kind::f16, bf16 x bf16 -> f32, M = 128, N = 256, K = 16) into a
//   256-column TMEM accumulator; tcgen05.commit releases shared-memory stages
//   and finally signals the epilogue.
// * Epilogue: eight warps read their TMEM lanes (one output row each, half of
//   the columns) with tcgen05.ld after every 512 tokens, add the partial sums
//   into float32 registers and finally add 2 * sum into H.
// * Every wait on an mbarrier is bounded (clock64 budget); on expiry the CTA
//   records an error flag, waits (again bounded) until the TMA loads and MMAs
//   it issued have completed, frees TMEM and returns.
#include "tc_common.cuh"

namespace gq {

__device__ unsigned int g_device_error = 0;  // bit 0: a bounded wait gave up

namespace {
using namespace tc;

constexpr int TM = 128, TN = 256, TK = 64;  // tile rows, cols, tokens per stage
constexpr int STAGES = 4;
constexpr int BOX_BYTES = TK * 64 * 2;             // one 64-token x 64-feature bf16 box
constexpr int A_BYTES = 2 * BOX_BYTES;             // 128 features
constexpr int B_BYTES = 4 * BOX_BYTES;             // 256 features
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;     // 48 KB
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024;
constexpr uint32_t TMEM_COLS = 256;

// Warp roles: 0 = TMA producer, 1 = MMA issuer, 2..9 = accumulator warps.
// The tensor-core accumulator is summed over KF k-tiles (512 tokens) at a
// time in one of two TMEM buffers; the accumulator warps add each partial
// sum into float32 registers (round-to-nearest) while the MMAs fill the other
// buffer.  Long in-TMEM accumulation is avoided because each accumulate step
// of the tensor core loses about half an ulp of the running sum.
constexpr int KF = 8;
constexpr int GROUP = 16;  // tile-rows per scheduling group
constexpr int NWARPS = 10;
constexpr int EPI_WARPS = 8;

__global__ void __launch_bounds__(NWARPS * 32, 1)
    hessian_tc_kernel(const __grid_constant__ CUtensorMap xmap, float *__restrict__ H, int cols, int n) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[STAGES];
    __shared__ __align__(8) uint64_t empty_bar[STAGES];
    __shared__ __align__(8) uint64_t tfull[2];
    __shared__ __align__(8) uint64_t tempty[2];
    __shared__ __align__(8) uint64_t drain_bar;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    unsigned char *smem = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // Tile of this CTA among the tiles that touch the upper triangle (bj >=
    // bjmin(bi) = bi TM / TN), in groups of GROUP tile-rows; within a group
    // by column, then row.  CTAs that run at the same time then share a
    // compact set of features of X, which keeps the X stripes they stream in
    // L2 instead of re-reading all of X from HBM in every wave.
    const int nbi = (cols + TM - 1) / TM, nbj = (cols + TN - 1) / TN;
    int t = blockIdx.x, g0 = 0;
    for (; g0 < nbi; g0 += GROUP) {
        const int g1 = (g0 + GROUP) < nbi ? (g0 + GROUP) : nbi;
        int cnt = 0;
        for (int i = g0; i < g1; ++i) cnt += nbj - (i * TM) / TN;
        if (t < cnt) break;
        t -= cnt;
    }
    const int g1 = (g0 + GROUP) < nbi ? (g0 + GROUP) : nbi;
    int bi = g0, bj = (g0 * TM) / TN;
    for (; bj < nbj; ++bj) {
        int valid = 0;  // rows of the group that reach column bj: a prefix
        while (g0 + valid < g1 && ((g0 + valid) * TM) / TN <= bj) ++valid;
        if (t < valid) {
            bi = g0 + t;
            break;
        }
        t -= valid;
    }
    const int r0 = bi * TM, c0 = bj * TN;
    const int ktiles = (n + TK - 1) / TK;
    const int periods = (ktiles + KF - 1) / KF;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], EPI_WARPS);
        }
        mbar_init(&drain_bar, 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_slot)),
                     "r"(2 * TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            int issued = 0;
            for (int kt = 0; kt < ktiles; ++kt, ++issued) {
                const int s = kt % STAGES;
                const uint32_t ph = (uint32_t)(kt / STAGES) & 1u;
                if (!mbar_wait(&empty_bar[s], ph ^ 1u) || *(volatile int *)&abort_flag) {
                    atomicOr(&g_device_error, 1u);
                    abort_flag = 1;
                    break;
                }
                unsigned char *st = smem + s * STAGE_BYTES;
                mbar_arrive_expect_tx(&full_bar[s], STAGE_BYTES);
                const int y = kt * TK;
                tma_load_2d(st + 0 * BOX_BYTES, &xmap, r0, y, &full_bar[s]);
                tma_load_2d(st + 1 * BOX_BYTES, &xmap, r0 + 64, y, &full_bar[s]);
#pragma unroll
                for (int b = 0; b < 4; ++b)
                    tma_load_2d(st + A_BYTES + b * BOX_BYTES, &xmap, c0 + 64 * b, y, &full_bar[s]);
            }
            drain_loads<STAGES>(full_bar, issued);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = make_idesc(TM, TN);
            bool ok = true;
            for (int p = 0; p < periods && ok; ++p) {
                const int b = p & 1;
                const uint32_t u = (uint32_t)(p >> 1) & 1u;
                if (!mbar_wait(&tempty[b], u ^ 1u)) {
                    ok = false;
                    break;
                }
                fence_after();
                const uint32_t acc = tmem + (uint32_t)(b * TMEM_COLS);
                const int k_end = (p + 1) * KF < ktiles ? (p + 1) * KF : ktiles;
                for (int kt = p * KF; kt < k_end; ++kt) {
                    const int s = kt % STAGES;
                    const uint32_t ph = (uint32_t)(kt / STAGES) & 1u;
                    if (!mbar_wait(&full_bar[s], ph)) {
                        ok = false;
                        break;
                    }
                    fence_after();
                    const uint32_t a0 = smem_u32(smem + s * STAGE_BYTES);
                    const uint32_t b0 = a0 + A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < TK / 16; ++kk) {
                        // 16 tokens = two 8-row core-matrix groups (SBO = 1024 B apart);
                        // 64-feature chunks are whole boxes (LBO = box size apart).
                        const uint64_t ad = smem_desc(a0 + kk * 2048, BOX_BYTES, 1024);
                        const uint64_t bd = smem_desc(b0 + kk * 2048, BOX_BYTES, 1024);
                        mma_bf16(acc, ad, bd, idesc, (kt > p * KF || kk > 0) ? 1u : 0u);
                    }
                    mma_commit(&empty_bar[s]);
                }
                mma_commit(&tfull[b]);
            }
            if (!ok) {
                atomicOr(&g_device_error, 1u);
                abort_flag = 1;
            }
            drain_mmas(&drain_bar);
        }
        __syncwarp();
    } else {
        // Accumulator warps: TMEM lane quarter = warp % 4 (hardware rule), column
        // half = (warp - 2) / 4.  Each thread owns one row x 128 columns.
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
            const uint32_t base = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * TMEM_COLS + half * 128);
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
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
            atomicOr(&g_device_error, 1u);
            abort_flag = 1;
        }
        __syncwarp();
        // H += 2 * master: upper triangle directly, strict lower as the mirror.
        const int r = r0 + q * 32 + lane;
        const int cb = c0 + half * 128;
        if (ok && r < cols && periods > 0) {
#pragma unroll
            for (int j = 0; j < 128; ++j) {
                const int c = cb + j;
                if (c < cols && c >= r) {
                    const float add = 2.f * master[j];
                    H[(int64_t)r * cols + c] += add;
                    if (c > r) H[(int64_t)c * cols + r] += add;
                }
            }
        }
    }
    fence_before();
    __syncthreads();
    if (warp == 0) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(2 * TMEM_COLS)
                     : "memory");
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
        cudaError_t e = cudaFuncSetAttribute(hessian_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const int nbi = (int)((cols + TM - 1) / TM), nbj = (int)((cols + TN - 1) / TN);
    int tiles = 0;
    for (int bi = 0; bi < nbi; ++bi) tiles += nbj - (bi * TM) / TN;
    for (int64_t t0 = 0; t0 < n; t0 += max_chunk) {
        const int64_t nc = (n - t0) < max_chunk ? (n - t0) : max_chunk;
        CUtensorMap map;
        cuuint64_t gdim[2] = {(cuuint64_t)cols, (cuuint64_t)nc};
        cuuint64_t gstride[1] = {(cuuint64_t)ldx * 2};
        cuuint32_t box[2] = {64, TK};
        cuuint32_t estr[2] = {1, 1};
        CUresult r = enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (void *)(X + t0 * ldx), gdim, gstride, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
        const int th = timing_begin(TK_HESSIAN, s);
        hessian_tc_kernel<<<tiles, NWARPS * 32, SMEM_BYTES, s>>>(map, H, (int)cols, (int)nc);
        count_launch();
        timing_end(th, s, (double)nc * (double)cols * (double)(cols + 1));
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace gq
