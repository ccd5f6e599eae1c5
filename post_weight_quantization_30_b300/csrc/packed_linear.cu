// The quantized linear layer computed from its packed form, on the
// fifth-generation tensor cores (sm_103a):
//
//     Y = X Ŵ^T + (X A^T) B^T,      Ŵ[m, k] = s[k / g, m] (q[m, k] - z[k / g, m])
//
// ("El balance de errores de la inferencia de pocos bits", sections 1 and 6:
// codes, per-group scale and zero point, dequantized on the fly inside the
// product; "Aumento de la precisión de LLM de 2 bits con EoRA", the adapter
// B A added to the quantized weights.)
//
// Ŵ is never rounded.  Each code minus its zero point is a small integer
// (|q - z| < 16), exact in bf16, and a bf16 input times such an integer is
// exact in float32, so the tensor core accumulates exact products of one
// group's K range into TMEM; the epilogue adds s[g, m] times that partial into
// float32 registers.  The result is X Ŵ^T up to float32 summation.
//
// Design (one CTA per 128 tokens x 128 output columns = rows of W):
// * warp 0 / lane 0: TMA loads, per stage, of the X tile (128 tokens x 64 K,
//   bf16, K-major, 128-byte swizzle) and of the tile's packed words (64 K-values
//   x 128 rows of W as 2b word-rows of 128 int32): eight stages, deep enough to
//   cover the load latency;
// * the bf16 W operand tiles live in three separate buffers, written by the
//   dequantization warps just ahead of the MMA;
// * warps 2-5 (one thread per row of W): read the row's words from shared
//   memory, unpack the codes, subtract the group's zero point and write the
//   bf16 integers straight into the 128-byte-swizzled K-major operand tile,
//   then fence to the async proxy and arrive on the buffer's ready barrier;
// * warp 1 / lane 0: tcgen05.mma kind::f16 (M = N = 128, K = 16), one group's
//   k-tiles into one of two TMEM accumulators;
// * warps 6-21: per group, read the accumulator (TMEM lane quarter = warp % 4,
//   one quarter of the 128 columns per warp: one TMEM round trip per group),
//   scale by the group's per-row scales and add into registers; store Y
//   through shared memory, coalesced.
// * The adapter term T B^T (T = X A^T from lora_t2_kernel) is one more group
//   with scale 1: T and B as bf16 hi / lo pairs (x = hi + lo + O(2^-16 x)),
//   three pseudo k-tiles T_hi B_hi, T_hi B_lo, T_lo B_hi: T by TMA into the X
//   slot, B copied into a W buffer by the dequantization warps (K = r <= 64,
//   zero-padded to 64).
// Every mbarrier wait is bounded; on expiry the CTA records the error flag that
// gq_check_device reports and exits without writing Y.
#include "tc_common.cuh"

namespace gq {

// Bit 0: a bounded wait of this file's kernels gave up.
__device__ unsigned int g_packed_error = 0;

namespace {
using namespace tc;

constexpr int PM = 128, PN = 128, PK = 64;
constexpr int P_STAGES = 6;                      // TMA stages: X tile + packed words
constexpr int TILE_X = PM * PK * 2;              // 16 KB
constexpr int TILE_W = PN * PK * 2;              // 16 KB
constexpr int TILE_Q = PN * PK * 4 / 8;          // packed words of one stage, at most (4-bit): 4 KB
constexpr int P_STAGE = TILE_X + TILE_Q;         // 20 KB (X tiles 1024-byte aligned)
constexpr int W_BUFS = 5;                        // bf16 W operand tiles
constexpr int P_SMEM = P_STAGES * P_STAGE + W_BUFS * TILE_W + 1024;
constexpr uint32_t P_TMEM = PN;                  // columns per accumulator buffer
constexpr int P_DEQ = 8;                         // dequantization warps: 2 sets of 4, alternate k-tiles
constexpr int DEQ_SETS = 2;
constexpr int P_EPI = 16;                        // epilogue warps: 4 lane quarters x 4 column quarters
constexpr int P_NWARPS = 2 + P_DEQ + P_EPI;      // TMA, MMA, dequantization, epilogue
constexpr int P_COLS = PN / 4;                   // columns per epilogue thread
constexpr int P_STAGE_LD = PN + 4;               // epilogue staging row stride (floats)
constexpr int ADAPTER_MAX_R = 64;
constexpr int ADAPTER_TILES = 3;                 // T_hi B_hi, T_hi B_lo, T_lo B_hi
static_assert(4 * 32 * P_STAGE_LD * 4 <= P_STAGES * P_STAGE, "epilogue smem");
static_assert(P_SMEM <= 227 * 1024 - 4096, "shared memory");

// Instruction descriptor, kind::f16: D f32, A and B bf16, both K-major, N >> 3
// at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_bf16_kmajor(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// The b-bit field starting at bit `bit` of a little-endian stream of 32-bit
// words, word i at p[i * stride] (fields may straddle two words).
__device__ __forceinline__ uint32_t packed_field(const int32_t *__restrict__ p, int64_t stride, int64_t bit, int b) {
    const int64_t wi = bit >> 5;
    const int sh = (int)(bit & 31);
    uint32_t v = (uint32_t)p[wi * stride] >> sh;
    if (sh + b > 32) v |= (uint32_t)p[(wi + 1) * stride] << (32 - sh);
    return v & ((1u << b) - 1u);
}

// Eight 4-bit codes of one word (code i at bits [4i, 4i + 4)) as four bf16x2
// words holding (128 + q_2j, 128 + q_2j+1): a bf16 with biased exponent 134
// (0x43) has a unit step, so 0x4300 | q is 128 + q exactly for q < 128.
__device__ __forceinline__ void codes4_to_bf16(uint32_t w, uint32_t (&o)[4]) {
    const uint32_t t = w & 0x0F0F0F0Fu;          // codes 0, 2, 4, 6
    const uint32_t u = (w >> 4) & 0x0F0F0F0Fu;   // codes 1, 3, 5, 7
    const uint32_t m0 = __byte_perm(t, u, 0x5140);  // bytes c0 c1 c2 c3
    const uint32_t m1 = __byte_perm(t, u, 0x7362);  // bytes c4 c5 c6 c7
    o[0] = __byte_perm(m0, 0x43434343u, 0x4140);
    o[1] = __byte_perm(m0, 0x43434343u, 0x4342);
    o[2] = __byte_perm(m1, 0x43434343u, 0x4140);
    o[3] = __byte_perm(m1, 0x43434343u, 0x4342);
}

// Sixteen 2-bit codes of one word (code i at bits [2i, 2i + 2)) likewise, as
// eight bf16x2 words (128 + q_2j, 128 + q_2j+1).
__device__ __forceinline__ void codes2_to_bf16(uint32_t w, uint32_t (&o)[8]) {
    const uint32_t t0 = w & 0x03030303u;          // codes 0, 4, 8, 12
    const uint32_t t1 = (w >> 2) & 0x03030303u;   // codes 1, 5, 9, 13
    const uint32_t t2 = (w >> 4) & 0x03030303u;   // codes 2, 6, 10, 14
    const uint32_t t3 = (w >> 6) & 0x03030303u;   // codes 3, 7, 11, 15
    const uint32_t a0 = __byte_perm(t0, t1, 0x5140);  // c0 c1 c4 c5
    const uint32_t a1 = __byte_perm(t2, t3, 0x5140);  // c2 c3 c6 c7
    const uint32_t b0 = __byte_perm(t0, t1, 0x7362);  // c8 c9 c12 c13
    const uint32_t b1 = __byte_perm(t2, t3, 0x7362);  // c10 c11 c14 c15
    o[0] = __byte_perm(a0, 0x43434343u, 0x4140);  // c0 c1
    o[1] = __byte_perm(a1, 0x43434343u, 0x4140);  // c2 c3
    o[2] = __byte_perm(a0, 0x43434343u, 0x4342);  // c4 c5
    o[3] = __byte_perm(a1, 0x43434343u, 0x4342);  // c6 c7
    o[4] = __byte_perm(b0, 0x43434343u, 0x4140);  // c8 c9
    o[5] = __byte_perm(b1, 0x43434343u, 0x4140);  // c10 c11
    o[6] = __byte_perm(b0, 0x43434343u, 0x4342);  // c12 c13
    o[7] = __byte_perm(b1, 0x43434343u, 0x4342);  // c14 c15
}

__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
    const __nv_bfloat162 r = __hsub2(*reinterpret_cast<const __nv_bfloat162 *>(&a),
                                     *reinterpret_cast<const __nv_bfloat162 *>(&b));
    return *reinterpret_cast<const uint32_t *>(&r);
}

// NC consecutive values (q - z) of one row (NC a multiple of 32) as NC / 2
// bf16x2 words in K order.  Exact: every operand is an integer below 256.
template <int BITS, int NC>
__device__ __forceinline__ void dequant_row(const uint32_t (&w)[NC * BITS / 32], uint32_t zz, bool valid,
                                            float zf, uint32_t (&o)[NC / 2]) {
    if constexpr (BITS == 4) {
#pragma unroll
        for (int i = 0; i < NC / 8; ++i) {
            uint32_t t[4];
            codes4_to_bf16(w[i], t);
#pragma unroll
            for (int h = 0; h < 4; ++h) o[i * 4 + h] = bf16x2_sub(t[h], zz);
        }
    } else if constexpr (BITS == 2) {
#pragma unroll
        for (int i = 0; i < NC / 16; ++i) {
            uint32_t t[8];
            codes2_to_bf16(w[i], t);
#pragma unroll
            for (int h = 0; h < 8; ++h) o[i * 8 + h] = bf16x2_sub(t[h], zz);
        }
    } else {
        // 3-bit codes straddle words: extract each one.
#pragma unroll
        for (int h = 0; h < NC / 2; ++h) {
            float d[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int bit = (h * 2 + e) * BITS;
                const int wi = bit >> 5, sh = bit & 31;
                uint32_t v = w[wi] >> sh;
                if (sh + BITS > 32) v |= w[wi + 1] << (32 - sh);
                d[e] = (float)(v & ((1u << BITS) - 1u)) - zf;
            }
            const __nv_bfloat162 p2 = __floats2bfloat162_rn(d[0], d[1]);
            o[h] = *reinterpret_cast<const uint32_t *>(&p2);
        }
    }
    if (!valid) {
#pragma unroll
        for (int h = 0; h < NC / 2; ++h) o[h] = 0u;
    }
}

// Bounded wait that polls with the non-blocking test_wait instead of the
// suspending try_wait, for the waits on the critical path of the pipeline
// (producer hand-offs that usually complete within a few hundred cycles).
__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_spin(uint64_t *bar, uint32_t parity) {
    if (mbar_test(bar, parity)) return true;
    const long long budget = *(volatile long long *)&g_wait_budget;
    const long long t0 = clock64();
    while (!mbar_test(bar, parity)) {
        if (clock64() - t0 > budget) return false;
    }
    return true;
}

template <int BITS>
__global__ void __launch_bounds__(P_NWARPS * 32, 1)
    packed_linear_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap qmap,
                         const __grid_constant__ CUtensorMap thi, const __grid_constant__ CUtensorMap tlo,
                         const __nv_bfloat16 *__restrict__ Bhi, const __nv_bfloat16 *__restrict__ Blo,
                         const float *__restrict__ scales, const int32_t *__restrict__ qzeros, int n, int rows,
                         int cols, int group, int adapter, float *__restrict__ Y, int64_t ldy) {
    constexpr int NW = PK * BITS / 32;  // packed words per row per stage
    const int m0 = blockIdx.y * PM, n0 = blockIdx.x * PN;
    const int ktiles = cols / PK;
    const int ktg = group / PK;  // k-tiles per group
    const int ngroups = cols / group;
    const int kt_all = ktiles + (adapter ? ADAPTER_TILES : 0);  // with the adapter's pseudo k-tiles
    const int groups_all = ngroups + (adapter ? 1 : 0);

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[P_STAGES];   // X and packed words landed (TMA)
    __shared__ __align__(8) uint64_t empty_bar[P_STAGES];  // the MMA is done with the stage
    __shared__ __align__(8) uint64_t wready[W_BUFS];       // a bf16 W tile is written
    __shared__ __align__(8) uint64_t wempty[W_BUFS];       // the MMA is done with it
    __shared__ __align__(8) uint64_t tfull[2];
    __shared__ __align__(8) uint64_t tempty[2];
    __shared__ __align__(8) uint64_t drain_bar;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    // Scales of this tile's rows for groups gi (slot gi % 2) and gi + 1, staged by
    // the epilogue warps themselves (next group's loaded while this one drains).
    __shared__ __align__(16) float sc_ring[2][PN];
    __shared__ int epi_abort;

    unsigned char *smem = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < P_STAGES; ++s) {
            mbar_init(&full_bar[s], 1);   // the TMA thread's expect_tx
            mbar_init(&empty_bar[s], 1);
        }
        for (int d = 0; d < W_BUFS; ++d) {
            mbar_init(&wready[d], P_DEQ / DEQ_SETS);  // one arrival per warp of the set on this k-tile
            mbar_init(&wempty[d], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], P_EPI);
        }
        mbar_init(&drain_bar, 1);
        abort_flag = 0;
        epi_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_slot)),
                     "r"(2 * P_TMEM)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = tmem_slot;
    bool ok = true;

    if (warp == 0) {
        if (lane == 0) {
            int issued = 0;
            for (int kt = 0; kt < kt_all; ++kt, ++issued) {
                const int s = kt % P_STAGES;
                const uint32_t ph = (uint32_t)(kt / P_STAGES) & 1u;
                if (!mbar_wait(&empty_bar[s], ph ^ 1u) || *(volatile int *)&abort_flag) {
                    atomicOr(&g_packed_error, 1u);
                    abort_flag = 1;
                    break;
                }
                if (kt < ktiles) {
                    mbar_arrive_expect_tx(&full_bar[s], TILE_X + NW * PN * 4);
                    tma_load_2d(smem + s * P_STAGE, &xmap, kt * PK, m0, &full_bar[s]);
                    tma_load_2d(smem + s * P_STAGE + TILE_X, &qmap, n0, kt * NW, &full_bar[s]);
                } else {
                    // adapter pseudo k-tile a: T_hi, T_hi, T_lo (with B_hi, B_lo, B_hi)
                    const int a = kt - ktiles;
                    mbar_arrive_expect_tx(&full_bar[s], TILE_X);
                    tma_load_2d(smem + s * P_STAGE, a == 2 ? &tlo : &thi, 0, m0, &full_bar[s]);
                }
            }
            drain_loads<P_STAGES>(full_bar, issued);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_kmajor(PM, PN);
            const uint64_t dx0 = smem_desc(smem_u32(smem), 16, 1024);                       // stage 0, X
            const uint64_t dw0 = smem_desc(smem_u32(smem + P_STAGES * P_STAGE), 16, 1024);  // W buffer 0
            for (int gi = 0; gi < groups_all && ok; ++gi) {
                const int b = gi & 1;
                const uint32_t u = (uint32_t)(gi >> 1) & 1u;
                if (!mbar_wait(&tempty[b], u ^ 1u)) {
                    ok = false;
                    break;
                }
                fence_after();
                const uint32_t acc = tmem + (uint32_t)(b * P_TMEM);
                const int kb = gi * ktg, ke = gi < ngroups ? (gi + 1) * ktg : kt_all;
                for (int kt = kb; kt < ke; ++kt) {
                    const int s = kt % P_STAGES;
                    const uint32_t ph = (uint32_t)(kt / P_STAGES) & 1u;
                    const int d = kt % W_BUFS;
                    const uint32_t pd = (uint32_t)(kt / W_BUFS) & 1u;
                    // wready: the W tile is written -- by dequantization warps that first
                    // waited for the stage's TMA (X and packed words), so X has landed too;
                    // the adapter's W tiles are copied without that wait, so check full.
                    if ((kt >= ktiles && !mbar_spin(&full_bar[s], ph)) || !mbar_spin(&wready[d], pd)) {
                        ok = false;
                        break;
                    }
                    fence_after();
                    // K-major, 128-byte swizzle: 8-row groups 1024 B apart; a k-step of
                    // 16 bf16 values advances the start address (field in 16-byte units)
                    // by 32 bytes, i.e. the descriptor by 2.
                    const uint64_t da = dx0 + (uint64_t)(s * (P_STAGE >> 4));
                    const uint64_t dw = dw0 + (uint64_t)(d * (TILE_W >> 4));
#pragma unroll
                    for (int kk = 0; kk < PK / 16; ++kk)
                        mma_bf16(acc, da + 2 * kk, dw + 2 * kk, idesc, (kt == kb && kk == 0) ? 0u : 1u);
                    mma_commit(&empty_bar[s]);
                    mma_commit(&wempty[d]);
                }
                if (!ok) break;
                mma_commit(&tfull[b]);
            }
            if (!ok) {
                atomicOr(&g_packed_error, 1u);
                abort_flag = 1;
            }
            drain_mmas(&drain_bar);
        }
        __syncwarp();
    } else if (warp < 2 + P_DEQ) {
        // Dequantization: two sets of four warps take alternate k-tiles (the
        // per-k-tile chain of one warp -- words, unpacking, stores, proxy fence,
        // arrival -- is latency-bound); in a set thread t owns row n0 + t of W.
        // The packed words arrive with the stage (TMA); the zero point of the next
        // group is loaded one group ahead.
        const int t = (threadIdx.x - 64) & (PN - 1);
        const int set = (threadIdx.x - 64) >> 7;
        const int nrow = n0 + t;
        const bool valid = nrow < rows;
        const int64_t zwords = (int64_t)rows * BITS / 32;  // qzeros words per group
        auto zero_of = [&](int g) -> float {
            return valid ? (float)packed_field(qzeros + (int64_t)g * zwords, 1, (int64_t)nrow * BITS, BITS) : 0.f;
        };
        int zg = 0;
        float zf = zero_of(0);
        float znext = ngroups > 1 ? zero_of(1) : 0.f;
        uint32_t zz = 0u;
        {
            const __nv_bfloat162 z2 = __floats2bfloat162_rn(128.f + zf, 128.f + zf);
            zz = *reinterpret_cast<const uint32_t *>(&z2);
        }
        for (int kt = set; kt < kt_all; kt += DEQ_SETS) {
            const int s = kt % P_STAGES;
            const uint32_t ph = (uint32_t)(kt / P_STAGES) & 1u;
            const int d = kt % W_BUFS;
            const uint32_t pd = (uint32_t)(kt / W_BUFS) & 1u;
            unsigned char *dst = smem + P_STAGES * P_STAGE + d * TILE_W + t * 128;
            if (kt >= ktiles) {
                // adapter pseudo k-tile a: copy row t of B_hi (a = 0, 2) or B_lo (a = 1),
                // 64 bf16, into the swizzled W tile.
                const __nv_bfloat16 *bsrc = (kt - ktiles == 1 ? Blo : Bhi) + (int64_t)nrow * ADAPTER_MAX_R;
                uint4 v[8];
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    v[c] = valid ? __ldg(reinterpret_cast<const uint4 *>(bsrc) + c) : make_uint4(0u, 0u, 0u, 0u);
                if (!mbar_wait(&wempty[d], pd ^ 1u) || *(volatile int *)&abort_flag) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4 *>(dst + ((c ^ (t & 7)) << 4)) = v[c];
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(&wready[d]);
                continue;
            }
            const int g = kt / ktg;
            if (g != zg) {  // a new group
                zf = (g == zg + 1) ? znext : zero_of(g);
                zg = g;
                znext = g + 1 < ngroups ? zero_of(g + 1) : 0.f;
                const __nv_bfloat162 z2 = __floats2bfloat162_rn(128.f + zf, 128.f + zf);
                zz = *reinterpret_cast<const uint32_t *>(&z2);
            }
            if (!mbar_wait(&full_bar[s], ph) || *(volatile int *)&abort_flag) {
                ok = false;
                break;
            }
            const uint32_t *wq = reinterpret_cast<const uint32_t *>(smem + s * P_STAGE + TILE_X);
            uint32_t w[NW];
#pragma unroll
            for (int i = 0; i < NW; ++i) w[i] = wq[i * PN + t];
            uint32_t o[32];
            dequant_row<BITS, 64>(w, zz, valid, zf, o);
            if (!mbar_wait(&wempty[d], pd ^ 1u) || *(volatile int *)&abort_flag) {
                ok = false;
                break;
            }
#pragma unroll
            for (int c = 0; c < 8; ++c)
                *reinterpret_cast<uint4 *>(dst + ((c ^ (t & 7)) << 4)) =
                    make_uint4(o[c * 4], o[c * 4 + 1], o[c * 4 + 2], o[c * 4 + 3]);
            // Generic-proxy writes -> visible to the tensor core's async proxy.
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(&wready[d]);
        }
        if (!ok) {
            atomicOr(&g_packed_error, 1u);
            abort_flag = 1;
        }
        __syncwarp();
    } else {
        // Epilogue warps: TMEM lane quarter = warp % 4, column quarter cq; each
        // thread owns one token row x 32 columns.
        const int q = warp & 3, cq = (warp - 2 - P_DEQ) >> 2;
        const int cb = cq * P_COLS;  // first column of this warp's quarter
        float acc[P_COLS];
#pragma unroll
        for (int i = 0; i < P_COLS; ++i) acc[i] = 0.f;
        const int et = threadIdx.x - (2 + P_DEQ) * 32;  // 0..511 over the epilogue warps
        if (et < PN) sc_ring[0][et] = (n0 + et < rows) ? __ldg(scales + n0 + et) : 0.f;
        asm volatile("bar.sync 1, %0;" ::"n"(P_EPI * 32) : "memory");
        for (int gi = 0; gi < groups_all; ++gi) {
            // Next group's scale for one row, in flight while this group drains (the
            // adapter's group, last, has scale 1).
            float nxt = 0.f;
            if (et < PN && gi + 1 < groups_all && n0 + et < rows)
                nxt = (gi + 1 < ngroups) ? __ldg(scales + (int64_t)(gi + 1) * rows + n0 + et) : 1.f;
            const int b = gi & 1;
            const uint32_t u = (uint32_t)(gi >> 1) & 1u;
            if (!mbar_wait(&tfull[b], u)) {
                ok = false;
                epi_abort = 1;
            } else {
                __syncwarp();
                fence_after();
                const uint32_t base = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * P_TMEM + cb);
                const float *sg = &sc_ring[gi & 1][cb];
                float v[32];
                tmem_ld32(base, v);
#pragma unroll
                for (int i4 = 0; i4 < 8; ++i4) {
                    const float4 s4 = *(reinterpret_cast<const float4 *>(sg) + i4);
                    acc[i4 * 4 + 0] = fmaf(s4.x, v[i4 * 4 + 0], acc[i4 * 4 + 0]);
                    acc[i4 * 4 + 1] = fmaf(s4.y, v[i4 * 4 + 1], acc[i4 * 4 + 1]);
                    acc[i4 * 4 + 2] = fmaf(s4.z, v[i4 * 4 + 2], acc[i4 * 4 + 2]);
                    acc[i4 * 4 + 3] = fmaf(s4.w, v[i4 * 4 + 3], acc[i4 * 4 + 3]);
                }
                fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tempty[b]);
            }
            if (et < PN) sc_ring[(gi + 1) & 1][et] = nxt;
            // Every epilogue warp reaches this barrier once per group, failed or not,
            // and all leave the loop together on a failure.
            asm volatile("bar.sync 1, %0;" ::"n"(P_EPI * 32) : "memory");
            if (*(volatile int *)&epi_abort) break;
        }
        if (!ok) {
            atomicOr(&g_packed_error, 1u);
            abort_flag = 1;
        }
        // The pipeline stages are idle now (every stage was consumed before the
        // last group's accumulator completed): staging rows for the coalesced store.
        float *stage = reinterpret_cast<float *>(smem) + (size_t)q * 32 * P_STAGE_LD;
#pragma unroll
        for (int j = 0; j < P_COLS; j += 4)
            *reinterpret_cast<float4 *>(stage + lane * P_STAGE_LD + cb + j) =
                make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
        __syncwarp();
        // Store this warp's 32 rows x 32 columns: lanes 8 i .. 8 i + 7 one row,
        // 16 bytes per lane (128 contiguous bytes per row).
        const int c = n0 + cb + (lane & 7) * 4;  // rows % 4 == 0
        if (ok && c < rows) {
            for (int rr = lane >> 3; rr < 32; rr += 4) {
                const int mr = m0 + q * 32 + rr;
                if (mr >= n) break;
                const float4 v = *reinterpret_cast<const float4 *>(stage + rr * P_STAGE_LD + cb + (lane & 7) * 4);
                *reinterpret_cast<float4 *>(Y + (int64_t)mr * ldy + c) = v;
            }
        }
    }
    fence_before();
    __syncthreads();
    if (warp == 0) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(2 * P_TMEM) : "memory");
    }
}

// Partial sums of T = X A^T over K slices, Tpart[z] (n x r float32), X bf16
// (n x cols), A float32 (r x cols), r <= 64.  SIMT, register-tiled: a CTA owns
// 64 tokens x 64 adapter rows of one K slice; thread t computes tokens
// 4 (t / 8) .. + 3 and adapter rows 8 (t % 8) .. + 7 from float4 reads of the
// staged tiles (K-major in shared memory).
constexpr int LT_TOK = 64, LT_K = 32, LT_LD = 68;

__global__ void __launch_bounds__(128) lora_t2_kernel(const __nv_bfloat16 *__restrict__ X, int64_t ldx, int n,
                                                      int cols, const float *__restrict__ A, int r, int kslice,
                                                      float *__restrict__ Tpart) {
    __shared__ __align__(16) float Xs[LT_K][LT_LD];
    __shared__ __align__(16) float As[LT_K][LT_LD];
    const int t = threadIdx.x, tx = t & 7, ty = t >> 3;
    const int m0 = blockIdx.x * LT_TOK;
    const int kz0 = blockIdx.y * kslice;
    const int kz1 = (kz0 + kslice) < cols ? (kz0 + kslice) : cols;
    float acc[4][8];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
    for (int k0 = kz0; k0 < kz1; k0 += LT_K) {
        for (int idx = t; idx < LT_TOK * LT_K; idx += 128) {
            const int tok = idx / LT_K, kk = idx % LT_K, k = k0 + kk;
            Xs[kk][tok] = (m0 + tok < n && k < kz1) ? __bfloat162float(X[(int64_t)(m0 + tok) * ldx + k]) : 0.f;
        }
        for (int idx = t; idx < ADAPTER_MAX_R * LT_K; idx += 128) {
            const int i = idx / LT_K, kk = idx % LT_K, k = k0 + kk;
            As[kk][i] = (i < r && k < kz1) ? A[(int64_t)i * cols + k] : 0.f;
        }
        __syncthreads();
#pragma unroll 4
        for (int kk = 0; kk < LT_K; ++kk) {
            const float4 x4 = *reinterpret_cast<const float4 *>(&Xs[kk][ty * 4]);
            const float4 a0 = *reinterpret_cast<const float4 *>(&As[kk][tx * 8]);
            const float4 a1 = *reinterpret_cast<const float4 *>(&As[kk][tx * 8 + 4]);
            const float xv[4] = {x4.x, x4.y, x4.z, x4.w};
            const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(xv[i], av[j], acc[i][j]);
        }
        __syncthreads();
    }
    float *out = Tpart + (int64_t)blockIdx.y * n * r;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int m = m0 + ty * 4 + i;
        if (m < n)
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (tx * 8 + j < r) out[(int64_t)m * r + tx * 8 + j] = acc[i][j];
    }
}

// rowsxr float32 sum over `slices` stacked copies (fixed order) -> T (may be NULL),
// and its bf16 split hi + lo (lo = bf16(v - hi); NULL to skip) with row stride 64,
// columns r..63 zero.
__global__ void sum_split_kernel(const float *__restrict__ parts, int slices, int nrow, int r, float *__restrict__ T,
                                 __nv_bfloat16 *__restrict__ hi, __nv_bfloat16 *__restrict__ lo) {
    const int64_t total = (int64_t)nrow * ADAPTER_MAX_R;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int m = (int)(idx / ADAPTER_MAX_R), c = (int)(idx % ADAPTER_MAX_R);
        float v = 0.f;
        if (c < r) {
            for (int z = 0; z < slices; ++z) v += parts[(int64_t)z * nrow * r + (int64_t)m * r + c];
            if (T) T[(int64_t)m * r + c] = v;
        }
        if (hi) {
            const __nv_bfloat16 h = __float2bfloat16_rn(v);
            hi[idx] = h;
            lo[idx] = __float2bfloat16_rn(v - __bfloat162float(h));
        }
    }
}

// A bf16 operand of r <= 64 columns stored with row stride 64 (K-major, one
// 128-byte swizzle row per matrix row): dims {64, nrow}, box {64, 128}.
bool make_r_map(CUtensorMap *map, const __nv_bfloat16 *p, int64_t nrow) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t gdim[2] = {(cuuint64_t)ADAPTER_MAX_R, (cuuint64_t)nrow};
    cuuint64_t gstride[1] = {(cuuint64_t)ADAPTER_MAX_R * 2};
    cuuint32_t box[2] = {(cuuint32_t)PK, (cuuint32_t)PM};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (void *)p, gdim, gstride, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

unsigned grid_cap(int64_t total) {
    int64_t g = (total + 255) / 256;
    if (g < 1) g = 1;
    if (g > 148 * 8) g = 148 * 8;
    return (unsigned)g;
}

// K slices of lora_t2_kernel: about two CTAs per SM, slices a multiple of LT_K wide.
void lora_t_split(int64_t n, int64_t cols, int *kslice, int *slices) {
    const int64_t tiles = (n + LT_TOK - 1) / LT_TOK;
    int64_t z = (2 * 148 + tiles - 1) / tiles;
    if (z < 1) z = 1;
    if (z > cols / LT_K) z = cols / LT_K;
    if (z < 1) z = 1;
    int64_t ks = (cols + z - 1) / z;
    ks = (ks + LT_K - 1) / LT_K * LT_K;
    *kslice = (int)ks;
    *slices = (int)((cols + ks - 1) / ks);
}

bool make_x_map(CUtensorMap *map, const __nv_bfloat16 *X, int64_t n, int64_t cols, int64_t ldx) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t gdim[2] = {(cuuint64_t)cols, (cuuint64_t)n};
    cuuint64_t gstride[1] = {(cuuint64_t)ldx * 2};
    cuuint32_t box[2] = {(cuuint32_t)PK, (cuuint32_t)PM};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (void *)X, gdim, gstride, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The packed words as a 2-D int32 tensor: rows (contiguous) x cols * bits / 32
// word-rows; a stage's box is 128 rows x 2 bits word-rows.
bool make_q_map(CUtensorMap *map, const int32_t *qweight, int64_t rows, int64_t cols, int bits) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t gdim[2] = {(cuuint64_t)rows, (cuuint64_t)(cols * bits / 32)};
    cuuint64_t gstride[1] = {(cuuint64_t)rows * 4};
    cuuint32_t box[2] = {(cuuint32_t)PN, (cuuint32_t)(PK * bits / 32)};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, (void *)qweight, gdim, gstride, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BITS>
cudaError_t launch_bits(const CUtensorMap &xmap, const CUtensorMap &qmap, const CUtensorMap &thi,
                        const CUtensorMap &tlo, const __nv_bfloat16 *bhi, const __nv_bfloat16 *blo, const float *scales,
                        const int32_t *qzeros, int n, int rows, int cols, int group, int adapter, float *Y,
                        int64_t ldy, cudaStream_t s) {
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e =
            cudaFuncSetAttribute(packed_linear_kernel<BITS>, cudaFuncAttributeMaxDynamicSharedMemorySize, P_SMEM);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    dim3 grid((unsigned)((rows + PN - 1) / PN), (unsigned)((n + PM - 1) / PM));
    packed_linear_kernel<BITS><<<grid, P_NWARPS * 32, P_SMEM, s>>>(xmap, qmap, thi, tlo, bhi, blo, scales, qzeros, n,
                                                                   rows, cols, group, adapter, Y, ldy);
    count_launch();
    return cudaGetLastError();
}

// Workspace of packed_forward (256-byte aligned regions):
//   [Tpart: slices x n x r][T: n x r]                       when r > 0
//   [T_hi, T_lo: n x 64 bf16][B_hi, B_lo: rows x 64 bf16]   when r > 0 and the tensor-core path
//   [decode partials: slices x n x rows]                    on the decode path
struct PackedWs {
    float *Tpart, *T, *Ypart;
    __nv_bfloat16 *Thi, *Tlo, *Bhi, *Blo;
};

size_t packed_layout(int64_t n, int64_t rows, int64_t cols, int group, int r, PackedWs *w, char *base) {
    size_t off = 0;
    auto take = [&](size_t bytes) {
        char *p = base ? base + off : nullptr;
        off += align_up(bytes);
        return p;
    };
    PackedWs t = {};
    const bool decode = packed_use_decode(n, group);
    if (r > 0) {
        int ks, z;
        lora_t_split(n, cols, &ks, &z);
        t.Tpart = (float *)take((size_t)z * n * r * sizeof(float));
        t.T = (float *)take((size_t)n * r * sizeof(float));
        if (!decode) {
            t.Thi = (__nv_bfloat16 *)take((size_t)n * ADAPTER_MAX_R * 2);
            t.Tlo = (__nv_bfloat16 *)take((size_t)n * ADAPTER_MAX_R * 2);
            t.Bhi = (__nv_bfloat16 *)take((size_t)rows * ADAPTER_MAX_R * 2);
            t.Blo = (__nv_bfloat16 *)take((size_t)rows * ADAPTER_MAX_R * 2);
        }
    }
    if (decode) {
        int gps, slices;
        packed_gemv_split(rows, cols, group, n, &gps, &slices);
        t.Ypart = (float *)take((size_t)slices * n * rows * sizeof(float));
    }
    if (w) *w = t;
    return off;
}

}  // namespace

cudaError_t packed_set_wait_budget(long long cycles) { return tc::set_wait_budget_here(cycles); }

unsigned int packed_read_and_clear_error() {
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_packed_error, sizeof(v)) != cudaSuccess) return ~0u;
    const unsigned int zero = 0;
    if (v) cudaMemcpyToSymbol(g_packed_error, &zero, sizeof(zero));
    return v;
}

size_t packed_ws_bytes(int64_t n, int64_t rows, int64_t cols, int group, int r) {
    return packed_layout(n, rows, cols, group, r, nullptr, nullptr);
}

cudaError_t packed_forward(const __nv_bfloat16 *X, int64_t n, int64_t ldx, const int32_t *qweight,
                           const float *scales, const int32_t *qzeros, int64_t rows, int64_t cols, int bits,
                           int group, const float *A, const float *B, int r, float *Y, int64_t ldy, void *ws,
                           cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    PackedWs w;
    packed_layout(n, rows, cols, group, r, &w, (char *)ws);
    const bool decode = packed_use_decode(n, group);
    cudaError_t e;
    if (r > 0) {
        int ks, z;
        lora_t_split(n, cols, &ks, &z);
        dim3 g((unsigned)((n + LT_TOK - 1) / LT_TOK), (unsigned)z);
        lora_t2_kernel<<<g, 128, 0, s>>>(X, ldx, (int)n, (int)cols, A, r, ks, w.Tpart);
        count_launch();
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        sum_split_kernel<<<grid_cap(n * ADAPTER_MAX_R), 256, 0, s>>>(w.Tpart, z, (int)n, r, w.T, w.Thi, w.Tlo);
        count_launch();
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        if (!decode) {
            sum_split_kernel<<<grid_cap(rows * ADAPTER_MAX_R), 256, 0, s>>>(B, 1, (int)rows, r, nullptr, w.Bhi,
                                                                            w.Blo);
            count_launch();
            if ((e = cudaGetLastError()) != cudaSuccess) return e;
        }
    }
    if (decode)
        return packed_gemv_launch(X, n, ldx, qweight, scales, qzeros, rows, cols, bits, group, w.T, B, r, w.Ypart, Y,
                                  ldy, s);
    CUtensorMap xmap, qmap, thi, tlo;
    if (!make_x_map(&xmap, X, n, cols, ldx) || !make_q_map(&qmap, qweight, rows, cols, bits))
        return cudaErrorInvalidValue;
    if (r > 0) {
        if (!make_r_map(&thi, w.Thi, n) || !make_r_map(&tlo, w.Tlo, n)) return cudaErrorInvalidValue;
    } else {
        thi = tlo = xmap;  // never read without the adapter
    }
    const int ad = r > 0 ? 1 : 0;
    switch (bits) {
        case 2: return launch_bits<2>(xmap, qmap, thi, tlo, w.Bhi, w.Blo, scales, qzeros, (int)n, (int)rows, (int)cols, group, ad, Y, ldy, s);
        case 3: return launch_bits<3>(xmap, qmap, thi, tlo, w.Bhi, w.Blo, scales, qzeros, (int)n, (int)rows, (int)cols, group, ad, Y, ldy, s);
        case 4: return launch_bits<4>(xmap, qmap, thi, tlo, w.Bhi, w.Blo, scales, qzeros, (int)n, (int)rows, (int)cols, group, ad, Y, ldy, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gq

// ---------------------------------------------------------------------------
// Decode path (few tokens): the product is bound by reading the packed words,
// so it runs on the SIMT pipes across every SM.  One lane per row of W, 256
// rows per CTA; K split across CTAs in whole groups; the CTA's slice of X
// (NT tokens x its K range) is staged in shared memory as float32.  Per group,
// sum_k x[m, k] (q - z) is accumulated unscaled (exact integer weights) and
// then scaled in float32, as in the tensor-core path.  Partial sums per K slice
// go to a workspace and packed_reduce_kernel adds them in a fixed order
// (deterministic), with the adapter term.
// ---------------------------------------------------------------------------
namespace gq {
namespace {

constexpr int DV_ROWS = 256;            // rows of W per CTA (8 warps, lane = row)
constexpr int DV_SMEM_FLOATS = 16384;   // X slice in shared memory: NT x K-range floats (64 KB)

template <int BITS, int NT>
__global__ void __launch_bounds__(DV_ROWS) packed_gemv_kernel(const __nv_bfloat16 *__restrict__ X, int64_t ldx, int n,
                                                              const int32_t *__restrict__ qweight,
                                                              const float *__restrict__ scales,
                                                              const int32_t *__restrict__ qzeros, int rows, int cols,
                                                              int group, int gps, float *__restrict__ Ypart) {
    extern __shared__ __align__(16) float xs[];  // [kc][NT]: the NT tokens of one k are contiguous
    const int ngroups = cols / group;
    const int g0 = blockIdx.y * gps;
    const int g1 = (g0 + gps) < ngroups ? (g0 + gps) : ngroups;
    const int k0 = g0 * group, kc = (g1 - g0) * group;
    const int m0 = blockIdx.z * NT;
    for (int idx = threadIdx.x; idx < NT * kc; idx += DV_ROWS) {
        const int m = idx / kc, k = idx - m * kc;  // coalesced along k
        xs[k * NT + m] = (m0 + m < n) ? __bfloat162float(X[(int64_t)(m0 + m) * ldx + k0 + k]) : 0.f;
    }
    __syncthreads();
    const int nr = blockIdx.x * DV_ROWS + threadIdx.x;
    if (nr >= rows) return;
    const int64_t zwords = (int64_t)rows * BITS / 32;
    // The slice as chunks of 64 codes (2 BITS words per row, one word-row apart by
    // `rows`); the next chunk's words and the next group's zero point and scale are
    // loaded while the current chunk is summed.
    const int nch = kc / 64;
    const int cpg = group / 64;  // chunks per group
    const int32_t *src = qweight + (int64_t)k0 * BITS / 32 * rows + nr;
    auto load_chunk = [&](int ch, uint32_t (&w)[2 * BITS]) {
#pragma unroll
        for (int i = 0; i < 2 * BITS; ++i) w[i] = (uint32_t)__ldg(src + (int64_t)(ch * 2 * BITS + i) * rows);
    };
    auto zero_of = [&](int g) { return (float)packed_field(qzeros + (int64_t)g * zwords, 1, (int64_t)nr * BITS, BITS); };
    float acc[NT], accg[NT];
#pragma unroll
    for (int m = 0; m < NT; ++m) acc[m] = accg[m] = 0.f;
    uint32_t wcur[2 * BITS], wnxt[2 * BITS];
    load_chunk(0, wcur);
    float zf = zero_of(g0), sc = __ldg(scales + (int64_t)g0 * rows + nr);
    float zn = 0.f, sn = 0.f;
    if (g0 + 1 < g1) {
        zn = zero_of(g0 + 1);
        sn = __ldg(scales + (int64_t)(g0 + 1) * rows + nr);
    }
    for (int ch = 0; ch < nch; ++ch) {
        if (ch + 1 < nch) load_chunk(ch + 1, wnxt);
        if (ch > 0 && ch % cpg == 0) {  // a new group: scale and add the finished one
            const int g = g0 + ch / cpg;
#pragma unroll
            for (int m = 0; m < NT; ++m) {
                acc[m] = fmaf(sc, accg[m], acc[m]);
                accg[m] = 0.f;
            }
            zf = zn;
            sc = sn;
            if (g + 1 < g1) {
                zn = zero_of(g + 1);
                sn = __ldg(scales + (int64_t)(g + 1) * rows + nr);
            }
        }
        const float *xc = xs + (size_t)ch * 64 * NT;
#pragma unroll
        for (int j = 0; j < 64; ++j) {
            const int bit = j * BITS;
            const int wi = bit >> 5, sh = bit & 31;
            uint32_t v = wcur[wi] >> sh;
            if (sh + BITS > 32) v |= wcur[wi + 1] << (32 - sh);
            const float d = (float)(v & ((1u << BITS) - 1u)) - zf;
            const float *xk = xc + j * NT;  // same address in every lane: a broadcast
            if constexpr (NT % 4 == 0) {
#pragma unroll
                for (int m4 = 0; m4 < NT; m4 += 4) {
                    const float4 x4 = *reinterpret_cast<const float4 *>(xk + m4);
                    accg[m4] = fmaf(x4.x, d, accg[m4]);
                    accg[m4 + 1] = fmaf(x4.y, d, accg[m4 + 1]);
                    accg[m4 + 2] = fmaf(x4.z, d, accg[m4 + 2]);
                    accg[m4 + 3] = fmaf(x4.w, d, accg[m4 + 3]);
                }
            } else {
#pragma unroll
                for (int m = 0; m < NT; ++m) accg[m] = fmaf(xk[m], d, accg[m]);
            }
        }
#pragma unroll
        for (int i = 0; i < 2 * BITS; ++i) wcur[i] = wnxt[i];
    }
#pragma unroll
    for (int m = 0; m < NT; ++m) acc[m] = fmaf(sc, accg[m], acc[m]);
    float *yp = Ypart + (int64_t)blockIdx.y * n * rows;
#pragma unroll
    for (int m = 0; m < NT; ++m)
        if (m0 + m < n) yp[(int64_t)(m0 + m) * rows + nr] = acc[m];
}

// Y[m, c] = sum over slices of Ypart[z, m, c] (fixed order) + sum_i T[m, i] B[c, i].
__global__ void packed_reduce_kernel(const float *__restrict__ Ypart, int slices, int n, int rows,
                                     const float *__restrict__ T, const float *__restrict__ B, int r,
                                     float *__restrict__ Y, int64_t ldy) {
    const int64_t total = (int64_t)n * rows;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int m = (int)(idx / rows), c = (int)(idx - (int64_t)m * rows);
        float v = 0.f;
        for (int z = 0; z < slices; ++z) v += Ypart[(int64_t)z * total + idx];
        for (int i = 0; i < r; ++i) v = fmaf(T[(int64_t)m * r + i], B[(int64_t)c * r + i], v);
        Y[(int64_t)m * ldy + c] = v;
    }
}

template <int BITS, int NT>
cudaError_t gemv_launch(const __nv_bfloat16 *X, int64_t ldx, int n, const int32_t *qweight, const float *scales,
                        const int32_t *qzeros, int rows, int cols, int group, int gps, int slices, float *Ypart,
                        cudaStream_t s) {
    const size_t smem = (size_t)NT * gps * group * sizeof(float);
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(packed_gemv_kernel<BITS, NT>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             DV_SMEM_FLOATS * (int)sizeof(float));
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    dim3 grid((unsigned)((rows + DV_ROWS - 1) / DV_ROWS), (unsigned)slices, (unsigned)((n + NT - 1) / NT));
    packed_gemv_kernel<BITS, NT><<<grid, DV_ROWS, smem, s>>>(X, ldx, n, qweight, scales, qzeros, rows, cols, group,
                                                             gps, Ypart);
    count_launch();
    return cudaGetLastError();
}

template <int NT>
cudaError_t gemv_bits(int bits, const __nv_bfloat16 *X, int64_t ldx, int n, const int32_t *qweight,
                      const float *scales, const int32_t *qzeros, int rows, int cols, int group, int gps, int slices,
                      float *Ypart, cudaStream_t s) {
    switch (bits) {
        case 2: return gemv_launch<2, NT>(X, ldx, n, qweight, scales, qzeros, rows, cols, group, gps, slices, Ypart, s);
        case 3: return gemv_launch<3, NT>(X, ldx, n, qweight, scales, qzeros, rows, cols, group, gps, slices, Ypart, s);
        case 4: return gemv_launch<4, NT>(X, ldx, n, qweight, scales, qzeros, rows, cols, group, gps, slices, Ypart, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

// Groups per K slice of the decode path: enough slices for about two CTAs per SM,
// each slice's X (NT = 16 tokens) within DV_SMEM_FLOATS.
void packed_gemv_split(int64_t rows, int64_t cols, int group, int64_t n, int *gps_out, int *slices_out) {
    const int ngroups = (int)(cols / group);
    const int64_t rb = (rows + DV_ROWS - 1) / DV_ROWS, nt = (n + 15) / 16;
    int64_t want = (2 * 148 + rb * nt - 1) / (rb * nt);
    if (want < 1) want = 1;
    int gps = (int)((ngroups + want - 1) / want);
    const int gmax = DV_SMEM_FLOATS / (16 * group);
    if (gps > gmax) gps = gmax;
    if (gps < 1) gps = 1;
    *gps_out = gps;
    *slices_out = (ngroups + gps - 1) / gps;
}

cudaError_t packed_gemv_launch(const __nv_bfloat16 *X, int64_t n, int64_t ldx, const int32_t *qweight,
                               const float *scales, const int32_t *qzeros, int64_t rows, int64_t cols, int bits,
                               int group, const float *T, const float *B, int r, float *Ypart, float *Y, int64_t ldy,
                               cudaStream_t s) {
    int gps, slices;
    packed_gemv_split(rows, cols, group, n, &gps, &slices);
    cudaError_t e;
    if (n <= 1)
        e = gemv_bits<1>(bits, X, ldx, (int)n, qweight, scales, qzeros, (int)rows, (int)cols, group, gps, slices, Ypart, s);
    else if (n <= 4)
        e = gemv_bits<4>(bits, X, ldx, (int)n, qweight, scales, qzeros, (int)rows, (int)cols, group, gps, slices, Ypart, s);
    else
        e = gemv_bits<16>(bits, X, ldx, (int)n, qweight, scales, qzeros, (int)rows, (int)cols, group, gps, slices, Ypart, s);
    if (e != cudaSuccess) return e;
    const int64_t total = n * rows;
    int64_t gr = (total + 255) / 256;
    if (gr > 148 * 8) gr = 148 * 8;
    packed_reduce_kernel<<<(unsigned)gr, 256, 0, s>>>(Ypart, slices, (int)n, (int)rows, T, B, r, Y, ldy);
    count_launch();
    return cudaGetLastError();
}

}  // namespace gq
