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
// Kernel layout.  One CTA = 32 output rows x one block; lane = row, warp =
// one 32-column segment of the block (4 warps).  A warp sweeps its segment's
// columns one after the other: every lane quantizes its row's weight
// (round-half-even; the code decision equals the one from IEEE division
// w / s, see rint_div), forms the scaled error e_j = (w_j - ŵ_j) F_jj
// (= (w_j - ŵ_j) / U_jj) and updates the rest of the segment in registers
// with row j of Uinv_b (shared memory, read as broadcasts).  The segment's
// errors go through shared memory in chunks of 8 columns: after each chunk
// the sweeping warp arrives on a named barrier, and the warps of later
// segments wait on it and apply the chunk as a rank-8 update while the sweep
// of the next chunk runs, so that only the last chunk's update separates one
// segment's sweep from the next.  A group's min / max spans whole segments and
// is reduced through shared memory as well.  The epilogue writes ΔW (split) back
// to D / DL, the optional codes / Ŵ / row errors, the scales, and packs codes
// and zero points into 32-bit words (coalesced word-rows of 32 output rows).
// When all CTAs fit one wave, a launch can also sweep two adjacent blocks and
// apply the first one's deferred update to the second in the kernel (the
// two-block form below), which takes the first level of the recursive GEMMs
// off the serial chain.
#include "common.cuh"

namespace gq {
namespace {

constexpr int ROWS = 32;                   // rows per CTA: one per lane
constexpr int SEG = 32;                    // block columns per segment: one warp each
constexpr int MAXB = 128;                  // max block width
constexpr int NSEG = MAXB / SEG;           // segments (warps) per CTA
constexpr int NTHREADS = NSEG * 32;        // 128
constexpr int MAXG = MAXB / 32;            // max groups per block (group >= 32)
constexpr int ELD = SEG + 1;               // row stride of the error staging (conflict-free column reads)
constexpr int CH = 8;                      // columns per published chunk of errors
constexpr int NCH = SEG / CH;              // chunks per segment: named barriers 1 .. NCH

struct SweepSmem {
    float U[MAXB][MAXB];            // Uinv_b, upper triangle (lower part zero); read as broadcasts
    float fdiag[MAXB];              // F_jj = 1 / U_jj
    // Three stagings that are never live at the same time share one region, which
    // keeps the block under a third of the SM's shared memory (three CTAs per SM):
    union {
        float E[ROWS][ELD];         // scaled errors of the segment being swept, per row
        struct {
            float gmin[NSEG][ROWS]; // group min / max contributions of each segment (group start)
            float gmax[NSEG][ROWS];
        };
        float err[NSEG][ROWS];      // per-segment sums of e_j^2 (epilogue)
    };
    float gs[ROWS], ginv[ROWS], gz[ROWS];  // grid of the current group, per row
    uint8_t codes[ROWS][MAXB + 16]; // codes of the block (rows 16-byte aligned, for the packing epilogue)
    uint8_t zeros[MAXG][ROWS];      // staging for the qzeros packing
    float scales[MAXG][ROWS];       // staging for coalesced scale stores
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

// Named barriers (ids 1 .. NCH; 0 is __syncthreads): the sweeping warp
// arrives without waiting, the warps that consume its errors wait.  Both sides
// give the same thread count, 32 x (1 + consumers).
__device__ __forceinline__ void named_arrive(int id, int nthreads) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
__device__ __forceinline__ void named_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// The sweep of one block (columns c0 .. c0 + bw) for this CTA's 32 rows, from
// the block's Uinv_b (U) and F_jj (fdiag) in shared memory and w, the row
// segment as updated by every earlier column (w0: the original weights).
// Writes ΔW (split) to D / DL, Ŵ, the row errors and the packed outputs; with
// KEEP_DW, dwr receives this warp's segment of ΔW (rows inside the layer).
template <int BITS, bool KEEP_DW>
__device__ __forceinline__ void sweep_block(SweepSmem &sm, const float (*U)[MAXB], const float *fdiag, float (&w)[SEG],
                                            const float (&w0)[SEG], float (&dwr)[SEG], int64_t rows, int64_t cols,
                                            int64_t c0, int bw, int group, float *__restrict__ D,
                                            float *__restrict__ DL, int32_t *__restrict__ qweight,
                                            float *__restrict__ scales, int32_t *__restrict__ qzeros,
                                            uint8_t *__restrict__ codes, float *__restrict__ W_hat,
                                            float *__restrict__ row_err) {
    constexpr float maxq = (float)((1 << BITS) - 1);
    const int seg = threadIdx.x >> 5, r = threadIdx.x & 31;  // warp = segment, lane = row
    const int64_t row0 = (int64_t)blockIdx.x * ROWS;
    const int64_t row = row0 + r;
    const bool row_on = row < rows;
    const int nseg = bw / SEG;
    const int cl = seg * SEG;  // first block column of this warp
    const bool seg_on = seg < nseg;
    const int gseg = group / SEG;  // segments per group
    float e2 = 0.f;

    for (int s = 0; s < nseg; ++s) {
        if (s % gseg == 0) {
            // A group starts at segment s: min / max over its segments s .. s + gseg - 1,
            // whose weights carry every update from the columns before it.
            if (seg >= s && seg < s + gseg) {
                float lo = 3.402823466e38f, hi = -3.402823466e38f;
#pragma unroll
                for (int c = 0; c < SEG; ++c) {
                    lo = fminf(lo, w[c]);
                    hi = fmaxf(hi, w[c]);
                }
                sm.gmin[seg][r] = lo;
                sm.gmax[seg][r] = hi;
            }
            __syncthreads();
            if (seg == s) {
                float lo = sm.gmin[s][r], hi = sm.gmax[s][r];
                for (int k = 1; k < gseg; ++k) {
                    lo = fminf(lo, sm.gmin[s + k][r]);
                    hi = fmaxf(hi, sm.gmax[s + k][r]);
                }
                float xmin = fminf(lo, 0.f), xmax = fmaxf(hi, 0.f);
                if (xmin == 0.f && xmax == 0.f) {
                    xmin = -1.f;
                    xmax = 1.f;
                }
                const float sc = __fdiv_rn(xmax - xmin, maxq);
                sm.gs[r] = sc;
                sm.ginv[r] = __fdiv_rn(1.f, sc);
                sm.gz[r] = rintf(__fdiv_rn(-xmin, sc));
                sm.zeros[(s * SEG) / group][r] = (uint8_t)sm.gz[r];
                sm.scales[(s * SEG) / group][r] = sc;
            }
        }
        // Threads on the chunk barriers of segment s: its warp and the later live segments' warps.
        const int nbar = 32 * (nseg - s);
        if (seg == s) {
            // The segment's 32 columns, one after the other; every lane (row) quantizes
            // its own weight, and the error updates the rest of the segment in registers.
            __syncwarp();  // every lane has read the group's min / max before sm.E overwrites them
            const float sc = sm.gs[r], inv_s = sm.ginv[r], z = sm.gz[r];
            float wq[SEG];
            uint32_t cw[SEG / 4];
#pragma unroll
            for (int k = 0; k < SEG / 4; ++k) cw[k] = 0u;
#pragma unroll
            for (int ci = 0; ci < SEG; ++ci) {
                const int j = cl + ci;
                const float wv = w[ci];
                const float q = fminf(fmaxf(rint_div(wv, sc, inv_s) + z, 0.f), maxq);
                const float dq = sc * (q - z);
                wq[ci] = dq;
                cw[ci / 4] |= ((uint32_t)q) << (8 * (ci % 4));
                const float e = (wv - dq) * fdiag[j];
                sm.E[r][ci] = e;
                if (ci % CH == CH - 1 && nbar > 32) {
                    __threadfence_block();
                    named_arrive(1 + ci / CH, nbar);  // chunk ci / CH of the errors is in sm.E
                }
                e2 = fmaf(e, e, e2);
                // Uinv_b is upper triangular: only the later columns of the segment move here.
#pragma unroll
                for (int c4 = ((ci + 1) / 4) * 4; c4 < SEG; c4 += 4) {
                    const float4 u = *reinterpret_cast<const float4 *>(&U[j][cl + c4]);
                    if (c4 + 0 > ci) w[c4 + 0] = fmaf(-e, u.x, w[c4 + 0]);
                    if (c4 + 1 > ci) w[c4 + 1] = fmaf(-e, u.y, w[c4 + 1]);
                    if (c4 + 2 > ci) w[c4 + 2] = fmaf(-e, u.z, w[c4 + 2]);
                    if (c4 + 3 > ci) w[c4 + 3] = fmaf(-e, u.w, w[c4 + 3]);
                }
            }
            *reinterpret_cast<uint4 *>(&sm.codes[r][cl]) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
            *reinterpret_cast<uint4 *>(&sm.codes[r][cl + 16]) = make_uint4(cw[4], cw[5], cw[6], cw[7]);
            if (row_on) {
                float *dp = D + row * cols + c0 + cl;
                float *lp = DL + row * cols + c0 + cl;
#pragma unroll
                for (int c = 0; c < SEG; c += 4) {
                    // ΔW as its TF32 split: the operand of the deferred-update GEMMs.
                    float dw[4], dh[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        dw[u] = w0[c + u] - wq[c + u];
                        dh[u] = tf32_hi(dw[u]);
                        if (KEEP_DW) dwr[c + u] = dw[u];
                    }
                    *reinterpret_cast<float4 *>(dp + c) = make_float4(dh[0], dh[1], dh[2], dh[3]);
                    *reinterpret_cast<float4 *>(lp + c) =
                        make_float4(dw[0] - dh[0], dw[1] - dh[1], dw[2] - dh[2], dw[3] - dh[3]);
                    if (W_hat)
                        *reinterpret_cast<float4 *>(W_hat + row * cols + c0 + cl + c) =
                            make_float4(wq[c], wq[c + 1], wq[c + 2], wq[c + 3]);
                }
            }
        } else if (seg > s && seg_on) {
            // Update of this warp's segment by segment s, w -= E_s U[seg s, this segment],
            // one chunk of 8 columns as soon as it is published (the sums run in column order).
            for (int ch = 0; ch < NCH; ++ch) {
                named_sync(1 + ch, nbar);
#pragma unroll
                for (int ii = 0; ii < CH; ++ii) {
                    const int i = ch * CH + ii;
                    const float ei = sm.E[r][i];
                    const float *ur = &U[s * SEG + i][cl];
#pragma unroll
                    for (int c4 = 0; c4 < SEG; c4 += 4) {
                        const float4 u = *reinterpret_cast<const float4 *>(ur + c4);
                        w[c4 + 0] = fmaf(-ei, u.x, w[c4 + 0]);
                        w[c4 + 1] = fmaf(-ei, u.y, w[c4 + 1]);
                        w[c4 + 2] = fmaf(-ei, u.z, w[c4 + 2]);
                        w[c4 + 3] = fmaf(-ei, u.w, w[c4 + 3]);
                    }
                }
            }
        }
        __syncthreads();
    }

    // Epilogue: row errors, codes, scales, packed words.
    sm.err[seg][r] = e2;
    __syncthreads();
    if (seg == 0 && row_on && row_err) {
        float t = 0.f;
        for (int k = 0; k < nseg; ++k) t += sm.err[k][r];
        row_err[row] += t;
    }
    if (codes && row_on && seg_on) {
        const uint4 *src = reinterpret_cast<const uint4 *>(&sm.codes[r][cl]);
        uint8_t *dst = codes + row * cols + c0 + cl;
        if (((uintptr_t)dst & 15) == 0) {
            reinterpret_cast<uint4 *>(dst)[0] = src[0];
            reinterpret_cast<uint4 *>(dst)[1] = src[1];
        } else {  // the library only requires 4-byte alignment of codes
            const uint32_t *s32 = reinterpret_cast<const uint32_t *>(src);
#pragma unroll
            for (int i = 0; i < 8; ++i) reinterpret_cast<uint32_t *>(dst)[i] = s32[i];
        }
    }

    // scales [cols/group][rows]: 32 consecutive rows per group.
    const int ng = bw / group;
    for (int idx = threadIdx.x; idx < ng * ROWS; idx += NTHREADS) {
        const int g = idx / ROWS, rr = idx % ROWS;
        if (row0 + rr < rows) scales[((c0 / group) + g) * rows + row0 + rr] = sm.scales[g][rr];
    }
    // qweight [cols*BITS/32][rows]: words of this block, one word-row of 32 rows at a time.
    const int nw = bw * BITS / 32;
    const int64_t w0i = c0 * BITS / 32;
    for (int idx = threadIdx.x; idx < nw * ROWS; idx += NTHREADS) {
        const int wi = idx / ROWS, rr = idx % ROWS;
        if (row0 + rr < rows) qweight[(w0i + wi) * rows + row0 + rr] = (int32_t)pack_word<BITS>(sm.codes[rr], wi, bw);
    }
    // qzeros [cols/group][rows*BITS/32]: BITS words per group for these 32 rows.
    const int64_t zw = rows * BITS / 32;
    for (int idx = threadIdx.x; idx < ng * BITS; idx += NTHREADS) {
        const int g = idx / BITS, wi = idx % BITS;
        qzeros[((c0 / group) + g) * zw + row0 * BITS / 32 + wi] = (int32_t)pack_word<BITS>(sm.zeros[g], wi, ROWS);
    }
}

// Shared memory of the two-block kernel beyond SweepSmem: the second block's
// Uinv_b and F_jj, and V[blk a, blk a + 1] (row k, column n) for the
// first-level deferred update between the two.
struct PairSmem {
    float U1[MAXB][MAXB];
    float Vs[MAXB][MAXB];
    float fdiag1[MAXB];
};

// One launch sweeps one block (PAIR = false) or two adjacent full blocks a,
// a + 1 (PAIR = true).  With PAIR the deferred update of block a + 1 by block
// a, ΔW_a V[blk a, blk a + 1], is formed in registers (float32 FMA; lane =
// row, warp = its segment's 32 columns of block a + 1) from ΔW_a staged in
// shared memory, and added to block a + 1's weights as they are loaded:
// the first level of the recursive deferred update needs no GEMM launch.
template <int BITS, typename TW, bool PAIR>
__global__ void __launch_bounds__(NTHREADS) sweep_kernel(const TW *__restrict__ W, int64_t rows, int64_t cols,
                                                         int64_t c0, int bw, const float *__restrict__ Uinv,
                                                         const float *__restrict__ F, const uint8_t *__restrict__ dead,
                                                         int group, float *__restrict__ D, float *__restrict__ DL,
                                                         int32_t *__restrict__ qweight, float *__restrict__ scales,
                                                         int32_t *__restrict__ qzeros, uint8_t *__restrict__ codes,
                                                         float *__restrict__ W_hat, float *__restrict__ row_err,
                                                         const float *__restrict__ VThi,
                                                         const float *__restrict__ VTlo) {
    pdl_trigger();
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SweepSmem &sm = *reinterpret_cast<SweepSmem *>(smem_raw);
    PairSmem &ps = *reinterpret_cast<PairSmem *>(smem_raw + sizeof(SweepSmem));  // PAIR only

    const int seg = threadIdx.x >> 5, r = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * ROWS + r;
    const bool row_on = row < rows;
    const int cl = seg * SEG;
    const bool seg_on = seg < bw / SEG;

    // Uinv_b, F's diagonal, W, the dead mask and V were complete before the
    // first kernel of the sweep started, so they are read before waiting for
    // the previous kernel; D, which that kernel updates, is read after.
    // Uinv_b into shared memory with asynchronous 16-byte copies, all in flight
    // at once (the block's rows and columns beyond bw are zero-filled).
    auto load_uinv = [&](float (*Ud)[MAXB], const float *Us, int bwu) {
        for (int idx = threadIdx.x; idx < MAXB * MAXB / 4; idx += NTHREADS) {
            const int i = idx / (MAXB / 4), j4 = (idx % (MAXB / 4)) * 4;
            float *dst = &Ud[i][j4];
            if (i < bwu && j4 < bwu) {
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                             "l"(Us + (int64_t)i * bwu + j4)
                             : "memory");
            } else {
                *reinterpret_cast<float4 *>(dst) = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
    };
    load_uinv(sm.U, Uinv, bw);
    if (PAIR) load_uinv(ps.U1, Uinv + (int64_t)MAXB * MAXB, MAXB);
    asm volatile("cp.async.commit_group;" ::: "memory");
    for (int i = threadIdx.x; i < MAXB; i += NTHREADS) sm.fdiag[i] = (i < bw) ? F[(c0 + i) * cols + c0 + i] : 1.f;
    if (PAIR) {
        const int64_t c1 = c0 + MAXB;
        for (int i = threadIdx.x; i < MAXB; i += NTHREADS) ps.fdiag1[i] = F[(c1 + i) * cols + c1 + i];
        // Vs[k][n] = V[c0 + k][c1 + n] = VThi + VTlo at [c1 + n][c0 + k]: thread n reads row n of
        // the transposed split, four k at a time, and writes column n of Vs.
        const int n = threadIdx.x;  // NTHREADS == MAXB
        const float *hi = VThi + (c1 + n) * cols + c0, *lo = VTlo + (c1 + n) * cols + c0;
        for (int k = 0; k < MAXB; k += 4) {
            const float4 h = *reinterpret_cast<const float4 *>(hi + k), l = *reinterpret_cast<const float4 *>(lo + k);
            ps.Vs[k + 0][n] = h.x + l.x;
            ps.Vs[k + 1][n] = h.y + l.y;
            ps.Vs[k + 2][n] = h.z + l.z;
            ps.Vs[k + 3][n] = h.w + l.w;
        }
    }

    // This warp's segment of the row: the original weights w0 (dead inputs
    // zero) and the weights as updated by every earlier block, w = w0 + D.
    float w[SEG], w0[SEG], dwr[SEG];
    uint32_t dmask = 0;
#pragma unroll
    for (int c = 0; c < SEG; ++c) {
        w[c] = 0.f;
        w0[c] = 0.f;
        dwr[c] = 0.f;
    }
    if (seg_on && row_on) {
        load32<TW>(W + row * cols + c0 + cl, w0);
        if (dead) {
#pragma unroll
            for (int c = 0; c < SEG; ++c) dmask |= (dead[c0 + cl + c] != 0 ? 1u : 0u) << c;
        }
    }
    pdl_wait();  // D was last updated by the previous kernel
    if (seg_on && row_on) {
        float t[SEG];
        load32<float>(D + row * cols + c0 + cl, t);
#pragma unroll
        for (int c = 0; c < SEG; ++c) {
            w0[c] = ((dmask >> c) & 1u) ? 0.f : w0[c];
            w[c] = w0[c] + t[c];
        }
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncthreads();

    sweep_block<BITS, PAIR>(sm, sm.U, sm.fdiag, w, w0, dwr, rows, cols, c0, bw, group, D, DL, qweight, scales,
                            qzeros, codes, W_hat, row_err);
    if (PAIR) {
        const int64_t c1 = c0 + MAXB;
        // Every warp is done with block a's Uinv_b and staging; ΔW_a goes into the space of the former.
        __syncthreads();
        float (*dWs)[MAXB + 1] = reinterpret_cast<float (*)[MAXB + 1]>(&sm.U[0][0]);
#pragma unroll
        for (int c = 0; c < SEG; ++c) dWs[r][cl + c] = dwr[c];
        __syncthreads();
        // add = ΔW_a V[blk a, this warp's columns of blk a + 1] for this lane's row.
        float add[SEG];
#pragma unroll
        for (int c = 0; c < SEG; ++c) add[c] = 0.f;
#pragma unroll 4
        for (int k = 0; k < MAXB; ++k) {
            const float e = dWs[r][k];
#pragma unroll
            for (int c4 = 0; c4 < SEG; c4 += 4) {
                const float4 v = *reinterpret_cast<const float4 *>(&ps.Vs[k][cl + c4]);
                add[c4 + 0] = fmaf(e, v.x, add[c4 + 0]);
                add[c4 + 1] = fmaf(e, v.y, add[c4 + 1]);
                add[c4 + 2] = fmaf(e, v.z, add[c4 + 2]);
                add[c4 + 3] = fmaf(e, v.w, add[c4 + 3]);
            }
        }
        // Block a + 1: w = w0 + (D + ΔW_a V), D holding the updates from before block a.
        dmask = 0;
#pragma unroll
        for (int c = 0; c < SEG; ++c) {
            w[c] = 0.f;
            w0[c] = 0.f;
        }
        if (row_on) {
            float t[SEG];
            load32<TW>(W + row * cols + c1 + cl, w0);
            load32<float>(D + row * cols + c1 + cl, t);
            if (dead) {
#pragma unroll
                for (int c = 0; c < SEG; ++c) dmask |= (dead[c1 + cl + c] != 0 ? 1u : 0u) << c;
            }
#pragma unroll
            for (int c = 0; c < SEG; ++c) {
                w0[c] = ((dmask >> c) & 1u) ? 0.f : w0[c];
                w[c] = w0[c] + (t[c] + add[c]);
            }
        }
        sweep_block<BITS, false>(sm, ps.U1, ps.fdiag1, w, w0, dwr, rows, cols, c1, MAXB, group, D, DL, qweight,
                                 scales, qzeros, codes, W_hat, row_err);
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
            const float4 a0 = *reinterpret_cast<const float4 *>(&As[k][ty * 4]);
            const float4 a1 = *reinterpret_cast<const float4 *>(&As[k][64 + ty * 4]);
            const float4 b0 = *reinterpret_cast<const float4 *>(&Bs[k][tx * 4]);
            const float4 b1 = *reinterpret_cast<const float4 *>(&Bs[k][64 + tx * 4]);
            const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], bb[j], acc[i][j]);
        }
        __syncthreads();
    }
    // Each thread stores its four consecutive m of a row as one float4 when cols % 4 == 0 (a
    // warp's stores cover 256 contiguous bytes of a row of VT); s0 is a multiple of the block
    // width, itself a multiple of 32, so a group of four never straddles s0.
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int n = (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
        if (n >= bw) continue;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int64_t m = m0 + half * 64 + tx * 4;
            if (m >= s0) continue;
            float h[4], l[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float v = acc[i][half * 4 + j];
                h[j] = tf32_hi(v);
                l[j] = v - h[j];
            }
            if ((cols & 3) == 0) {
                *reinterpret_cast<float4 *>(VThi + (s0 + n) * cols + m) = make_float4(h[0], h[1], h[2], h[3]);
                *reinterpret_cast<float4 *>(VTlo + (s0 + n) * cols + m) = make_float4(l[0], l[1], l[2], l[3]);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    VThi[(s0 + n) * cols + m + j] = h[j];
                    VTlo[(s0 + n) * cols + m + j] = l[j];
                }
            }
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

template <int BITS, typename TW, bool PAIR>
cudaError_t launch_sweep(const TW *W, int64_t rows, int64_t cols, int64_t c0, int bw, const float *Uinv,
                         const float *F, const uint8_t *dead, int group, float *D, float *DL, int32_t *qweight,
                         float *scales, int32_t *qzeros, uint8_t *codes, float *W_hat, float *row_err,
                         const float *VThi, const float *VTlo, cudaStream_t s) {
    const size_t smem = sizeof(SweepSmem) + (PAIR ? sizeof(PairSmem) : 0);
    static bool attr_set = false;  // per template instance
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(sweep_kernel<BITS, TW, PAIR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
        // All of the unified L1 as shared memory, so that three one-block CTAs fit on an SM.
        e = cudaFuncSetAttribute(sweep_kernel<BITS, TW, PAIR>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const int th = timing_begin(TK_SWEEP, s);
    const cudaError_t e = launch_pdl(sweep_kernel<BITS, TW, PAIR>, dim3((unsigned)((rows + ROWS - 1) / ROWS)),
                                     dim3(NTHREADS), smem, s, W, rows, cols, c0, bw, Uinv, F, dead, group, D, DL,
                                     qweight, scales, qzeros, codes, W_hat, row_err, VThi, VTlo);
    count_launch();
    // Column-step work of the block(s), and for two blocks the 2 rows x 128 x 128 flops between them.
    timing_end(th, s, PAIR ? 2.0 * rows * MAXB * (MAXB - 1) + 2.0 * rows * MAXB * MAXB : (double)rows * bw * (bw - 1));
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
                               float *W_hat, float *row_err, const float *VThi, const float *VTlo, bool pair,
                               cudaStream_t s) {
#define GQ_SWEEP_CALL(B, T, P)                                                                                      \
    return launch_sweep<B, T, P>((const T *)W, rows, cols, c0, bw, Uinv_blk, F, dead, group, D, DL, qweight, scales, \
                                 qzeros, codes, W_hat, row_err, VThi, VTlo, s)
#define GQ_SWEEP_CASE(B)                                      \
    if (bits == B) {                                          \
        if (w_bf16) {                                         \
            if (pair) GQ_SWEEP_CALL(B, __nv_bfloat16, true);  \
            GQ_SWEEP_CALL(B, __nv_bfloat16, false);           \
        }                                                     \
        if (pair) GQ_SWEEP_CALL(B, float, true);              \
        GQ_SWEEP_CALL(B, float, false);                       \
    }
    GQ_SWEEP_CASE(2)
    GQ_SWEEP_CASE(3)
    GQ_SWEEP_CASE(4)
#undef GQ_SWEEP_CASE
#undef GQ_SWEEP_CALL
    return cudaErrorInvalidValue;
}

bool sweep_pair_fits(int64_t rows) { return (rows + ROWS - 1) / ROWS <= 148; }

}  // namespace gq
