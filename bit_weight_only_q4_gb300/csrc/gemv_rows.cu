// Weight-streaming kernels for sm_103a that own whole rows: the decode GEMV of
// both 4-bit layouts for one to four tokens, and the restricted BF16 head.
//
// Arithmetic: x staged per 32-column chunk with a power-of-two prescale
// (stream_common.cuh); NVFP4 decoded by cvt.rn.f16x2.e2m1x2 and summed per half
// group in packed fp16 FMAs, the half sums meeting the group scales in
// mixed-precision FMAs; int4 summed exactly with dp2a on int16-staged x, scale
// and min applied to the integer sums in fp32.  Data movement is chosen for
// short, dependent calls:
//
//   * Each CTA owns a contiguous range of output rows with their full K.  Warp w
//     owns one k-step ks = w % S (W x 1024 4-bit or 256 bf16 columns, W = 1 or
//     2 slices per lane) of the rows g, g + G, g + 2G, ... of its CTA (g = w / S,
//     G = warps / S).  S is a template parameter, so the warp geometry costs no
//     divisions.  No row is split between CTAs: no workspace, deterministic
//     results.
//   * Weights do not depend on the previous kernel, so they are requested
//     before griddepcontrol.wait.  For one token a call runs one CTA per SM on
//     half of the SM's registers and shared memory (16 warps with one slice per
//     lane, or 8 warps with two for the 4-bit layouts at K <= 2048), so the next
//     call's CTA is resident beside it (programmatic dependent launch) and
//     streams its weights while this call computes.
//   * After the wait the CTA stages x once in shared memory (prescaled fp16);
//     every warp keeps its k-step's slice in registers, decodes and multiplies
//     its rows, reduces each row across lanes (transposing butterfly) and parks
//     the partial per k-step in shared memory.  A final pass sums each row's S
//     partials in k order and stores bf16 (or, in the DS variant, with one
//     k-step and few rows per warp, the reduction stores each row at once).
//
// Bringing the weights in: for one token the first RB rows of every warp come
// straight into registers with 128-bit loads; every later row comes through a
// per-thread ring of NB * RB shared-memory slots filled with cp.async (each lane
// copies its own 16-byte slice, so no barrier is needed; the group scales come
// with plain loads into a matching register ring).  Both are issued before
// griddepcontrol.wait.  (Measured on the NVFP4 16384 x 2048 GEMV chain: a TMA
// bulk-copy stage ring was slower, 6.9 against 5.2 us per call, and a deeper
// cp.async ring did not help: 16 warps of cp.async per SM are throttled near
// 34 GB/s, so fewer requests in flight let the first rows land sooner.)
//
// Eligibility: S = ceil(K / kstep) rounded up to a power of two, at most 8 (16
// for int8 at one token); 16-byte aligned rows (int4 always, NVFP4 K % 32 == 0,
// bf16 H % 8 == 0).  Other shapes use gemv.cu.
#include "q4_device.cuh"
#include "q4_internal.h"
#include "stream_common.cuh"

namespace q4 {

// Ring bytes of a CTA of NW warps holding NB batches of RB rows per thread,
// each row W 16-byte slices.
__host__ __device__ constexpr size_t rows_ring_bytes(int NW, int NB, int RB, int W)
{
    return (size_t)NB * RB * W * NW * 32 * 16;
}

// One token (MT = 1): one CTA per SM per call on half of the SM's registers, so
// the CTA of the next call fits beside it -- 16 warps at 64 registers with one
// 32-column slice per lane (W = 1), or 8 warps at 128 registers with two (W = 2).
// Several tokens: 8-warp CTAs, two per SM.
template <int MT, int W>
struct RowsShape {
    static constexpr int NW = (MT == 1 && W == 1) ? 16 : 8;
    static constexpr int MIN_CTAS = 2;
};

// x slice of one lane in registers (XV words per token) and its per-chunk data.
template <int WK, int MT, int XV>
__device__ __forceinline__ void rows_load_x(const uint16_t *xs, const float *cf, int Kpad,
                                            int ks, int lane, int col0, float gsc,
                                            uint32_t (&xr)[MT][XV], float4 (&cd)[MT])
{
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        if constexpr (WK == W_BF16) {
            const uint4 t = *reinterpret_cast<const uint4 *>(xs + (size_t)m * Kpad + col0);
            xr[m][0] = t.x; xr[m][1] = t.y; xr[m][2] = t.z; xr[m][3] = t.w;
            cd[m] = make_float4(1.f, 0.f, 0.f, 0.f);
        } else if constexpr (WK == W_INT8) {
            const uint4 *src = reinterpret_cast<const uint4 *>(xs + (size_t)m * Kpad) + ks * 64;
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const uint4 t = src[i * 32 + lane];
                xr[m][4 * i + 0] = t.x; xr[m][4 * i + 1] = t.y;
                xr[m][4 * i + 2] = t.z; xr[m][4 * i + 3] = t.w;
            }
            const float4 c4 = reinterpret_cast<const float4 *>(cf)[(size_t)m * (Kpad / 32) + col0 / 32];
            // x' sum over this lane's 16 columns (first or second half of the chunk)
            cd[m] = make_float4(c4.x, (lane & 1) ? c4.z : c4.y, 0.f, 0.f);
        } else {
            const uint4 *src = reinterpret_cast<const uint4 *>(xs + (size_t)m * Kpad) + ks * 128;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint4 t = src[i * 32 + lane];
                xr[m][4 * i + 0] = t.x; xr[m][4 * i + 1] = t.y;
                xr[m][4 * i + 2] = t.z; xr[m][4 * i + 3] = t.w;
            }
            if constexpr (WK == W_INT4)
                cd[m] = reinterpret_cast<const float4 *>(cf)[(size_t)m * (Kpad / 32) + col0 / 32];
            else
                cd[m] = make_float4(cf[(size_t)m * (Kpad / 32) + col0 / 32] * gsc, 0.f, 0.f, 0.f);
        }
    }
}

// One lane's share of one row: 16 weight bytes (w4) and its scale words (int4:
// fp16 scale in swr, fp16 min in swm; NVFP4: two e4m3 group scales in swr; int8:
// the fp16 row scale) against MT tokens.
template <int WK, int MT, int XV>
__device__ __forceinline__ void rows_dot(const uint4 qv, uint32_t swr, uint32_t swm,
                                         const uint32_t (&xr)[MT][XV], const float4 (&cd)[MT],
                                         float *out)
{
    const uint32_t w4[4] = {qv.x, qv.y, qv.z, qv.w};
    if constexpr (WK == W_BF16) {
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            float t = 0.f;
#pragma unroll
            for (int jj = 0; jj < 4; ++jj)
                t = fma2_bf16(t, w4[jj], xr[m][jj]);
            out[m] = t;
        }
    } else if constexpr (WK == W_INT8) {
        // 16 signed codes: (q ^ 0x80) = q + 128 in the low byte of the fp16 magic
        // 1024, i.e. 1152 + q, two per register; sum_k (1152 + q) x' - 1152 X = sum_k q x'
        float A[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m)
            A[m] = 0.f;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const uint32_t v = w4[jj] ^ 0x80808080u;
            uint32_t pa, pb;
            asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(pa) : "r"(v), "r"(0x64646464u));   // cols 0, 1
            asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(pb) : "r"(v), "r"(0x64646464u));   // cols 2, 3
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                A[m] = fma2_f16(A[m], pa, xr[m][2 * jj + 0]);
                A[m] = fma2_f16(A[m], pb, xr[m][2 * jj + 1]);
            }
        }
        const float sc = f16lo_unpack_f32(swr);
#pragma unroll
        for (int m = 0; m < MT; ++m)
            out[m] = fmaf(-1152.f, cd[m].y, A[m]) * cd[m].x * sc;
    } else if constexpr (WK == W_INT4) {
        // Exact integer sums: x' is int16 (the int16 staging path, |x'| < 2^15)
        // and the codes become bytes -- w & 0x0F0F0F0F holds the even
        // columns' codes, (w >> 4) & 0x0F0F0F0F the odd columns' -- so each
        // dp2a adds two exact products to an int32.  Over the lane's 32
        // columns |C| <= 32 * 15 * 32767 < 2^24, so C converts to fp32
        // exactly; then sum_k (c s + m) x' = s C + m X in fp32, with X the
        // chunk's sum of x' from staging.
        int A[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m)
            A[m] = 0;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const uint32_t ce = w4[jj] & 0x0F0F0F0Fu;          // c of columns 0, 2, 4, 6
            const uint32_t co = (w4[jj] >> 4) & 0x0F0F0F0Fu;   // c of columns 1, 3, 5, 7
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                A[m] = dp2a_lo_su(xr[m][4 * jj + 0], ce, A[m]);
                A[m] = dp2a_hi_su(xr[m][4 * jj + 1], ce, A[m]);
                A[m] = dp2a_lo_su(xr[m][4 * jj + 2], co, A[m]);
                A[m] = dp2a_hi_su(xr[m][4 * jj + 3], co, A[m]);
            }
        }
        const float sc = f16lo_unpack_f32(swr);
        const float mn = f16lo_unpack_f32(swm);
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            const float C = (float)A[m];
            out[m] = fmaf(sc, C, mn * cd[m].y) * cd[m].x;
        }
    } else {
        // NVFP4: each 16-column group (two words) is summed in fp16 -- eight exact
        // products (E2M1 x prescaled x, at most 10 significant bits) per half, one
        // rounding per add, magnitude below 2^16 by the prescale -- then each half
        // meets the group scale in an fp32 accumulator.  Packed fp16 FMAs take one
        // instruction per two weights where fp32 accumulation of fp16 products
        // takes two per weight.
        uint32_t Ha[MT], Hb[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            Ha[m] = 0u;
            Hb[m] = 0u;
        }
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            uint32_t hh[4];
            e2m1x8_to_f16x2x4(w4[jj], hh);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    if (jj < 2)
                        Ha[m] = hfma2_rn(hh[q], xr[m][4 * jj + q], Ha[m]);
                    else
                        Hb[m] = hfma2_rn(hh[q], xr[m][4 * jj + q], Hb[m]);
                }
            }
        }
        // the two e4m3 group scales are exact in fp16; half sums meet them in
        // mixed-precision FMAs
        const uint32_t s2 = e4m3x2lo_to_f16x2(swr);
#pragma unroll
        for (int m = 0; m < MT; ++m)
            out[m] = f16_group_pair_f32(Ha[m], Hb[m], s2) * cd[m].x;
    }
}

// Sum RB x MT partials across the warp and park each row's total for k-step ks;
// with DS (one k-step) the total is the row's result and goes to y as bf16.
template <int RB, int MT, int S, bool DS>
__device__ __forceinline__ void rows_park(const GemvParams &p, int n0, float (&part)[RB * MT],
                                          int lane, int ks, int row0, int G, int nvalid,
                                          float *red)
{
    int idx = 0;
    const float tot = warp_sum_transpose<RB * MT>(part, lane, idx);
    const int r = idx / MT, m = idx - (idx / MT) * MT;
    if ((lane & (32 / (RB * MT) - 1)) == 0 && r < nvalid) {
        const int row = row0 + G * r;
        if constexpr (DS) {
            static_assert(S == 1, "direct stores need one k-step");
            (void)ks;
            (void)red;
            if (m < p.mcount)
                p.y[(int64_t)(p.m0 + m) * p.ldy + n0 + row] = f32_to_bf16_bits(tot);
        } else {
            (void)p;
            (void)n0;
            red[((size_t)row * S + ks) * MT + m] = tot;
        }
    }
}

// Final pass: each row's S partials summed in k order, stored as bf16.
template <int MT, int S>
__device__ __forceinline__ void rows_store(const GemvParams &p, const float *red, int n0,
                                           int rows_cta, int nthreads)
{
    for (int e = (int)threadIdx.x; e < rows_cta * MT; e += nthreads) {
        const int row = e / MT, m = e - (e / MT) * MT;
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < S; ++k)
            s += red[((size_t)row * S + k) * MT + m];
        if (m < p.mcount)
            p.y[(int64_t)(p.m0 + m) * p.ldy + n0 + row] = f32_to_bf16_bits(s);
    }
}

// Physical weight row of logical row n.
__device__ __forceinline__ int64_t rows_phys(const GemvParams &p, int64_t n)
{
    return n < p.n_rows ? (int64_t)p.row_begin + n : (int64_t)p.extra_row;
}

// Scale word of physical row prow for the lane whose columns start at col0.
template <int WK>
__device__ __forceinline__ uint32_t rows_scale_global(const GemvParams &p, int64_t prow, int col0)
{
    if constexpr (WK == W_INT4) {
        return ld_nc_u16(static_cast<const uint16_t *>(p.scale) + prow * (p.K / 128) + col0 / 128);
    } else if constexpr (WK == W_NVFP4_A16) {
        return ld_nc_u16(static_cast<const uint8_t *>(p.scale) + prow * (p.K / 16) + col0 / 16);
    } else if constexpr (WK == W_INT8) {
        (void)col0;
        return ld_nc_u16(static_cast<const uint16_t *>(p.scale) + prow);
    } else {
        return 0u;
    }
}

// int4: the min word of physical row prow for the lane (loaded apart from the
// scale and combined only where it is used).
template <int WK>
__device__ __forceinline__ uint32_t rows_min_global(const GemvParams &p, int64_t prow, int col0)
{
    if constexpr (WK == W_INT4)
        return ld_nc_u16(p.minv + prow * (p.K / 128) + col0 / 128);
    else
        return 0u;
}

// ------------------------------------------------------------ cp.async ring
// A lane holds W slices of 32 columns (16 weight bytes) of each of its rows:
// slice h of wide k-step ks is the lane's slice of 1024-column k-step W ks + h,
// so the x image, the per-chunk data and the slice arithmetic are those of the
// one-slice kernel, and every warp-wide request covers 512 contiguous bytes.
template <int WK, int MT, int RB, int S, int NB, int REG, int W, bool DS>
__global__ void __launch_bounds__(RowsShape<MT, W>::NW * 32, RowsShape<MT, W>::MIN_CTAS)
q4_rows_kernel(GemvParams p)
{
    constexpr int RK_WARPS = RowsShape<MT, W>::NW;
    constexpr int RK_THREADS = RK_WARPS * 32;
    extern __shared__ __align__(16) unsigned char smem[];
    constexpr int KSTEP = Kind<WK>::KSTEP;
    constexpr int COLS = Kind<WK>::COLS;
    constexpr int CH = Kind<WK>::CH;
    constexpr int XV = (WK == W_BF16) ? 4 : ((WK == W_INT8) ? 8 : 16);   // x registers per token
    constexpr int G = RK_WARPS / S;
    constexpr int NSLOT = NB * RB;
    constexpr int Kpad = S * W * KSTEP;
    // bytes between a lane's slices in a weight row, and in its scale row
    constexpr int HB = 512;
    constexpr int SB = (WK == W_INT4) ? (KSTEP / 128) * 2 : (WK == W_NVFP4_A16 ? KSTEP / 16 : 0);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int ks = warp % S;
    const int g = warp / S;
    int col0[W];
    bool colok[W];
#pragma unroll
    for (int h = 0; h < W; ++h) {
        col0[h] = (W * ks + h) * KSTEP + lane * COLS;
        colok[h] = col0[h] < p.K;
    }
    const uint32_t ring = smem_u32(smem) + threadIdx.x * 16;   // slice i at + i * 16 * threads
    const uint4 *ring_ld = reinterpret_cast<const uint4 *>(smem) + threadIdx.x;
    constexpr size_t RING = rows_ring_bytes(RK_WARPS, NB, RB, W);
    uint16_t *xs = reinterpret_cast<uint16_t *>(smem + RING);
    float *cf = reinterpret_cast<float *>(smem + RING + (size_t)MT * Kpad * 2);
    float *red = cf + (size_t)MT * (Kpad / 32) * CH;        // [row][ks][m] partials
    const int b = blockIdx.x;
    const int n0 = b * p.rows_q + (b < p.rows_r ? b : p.rows_r);
    const int rows_cta = p.rows_q + (b < p.rows_r ? 1 : 0);
    const int my_rows = rows_cta > g ? (rows_cta - g + G - 1) / G : 0;   // rows g + G*j
    const int my_ring = my_rows > REG ? my_rows - REG : 0;    // rows j >= REG use the ring
    const int64_t colbyte = (WK == W_BF16) ? (int64_t)col0[0] * 2
                            : (WK == W_INT8) ? (int64_t)col0[0] : (int64_t)(col0[0] / 2);

    // Ring rows are requested strictly in order (jr = 0, 1, 2, ...).  The linear
    // layers map logical row n to physical row n, so their weight and scale
    // pointers simply advance by G rows per request (two 64-bit adds) instead of
    // being recomputed from the row index; the head keeps the row mapping.
    constexpr bool kStep = WK != W_BF16;
    const uint8_t *wnext = p.w;                   // weights of the next ring row
    const uint8_t *snext = nullptr;               // its scale bytes (int4: scale, min)
    int64_t wstep = 0, sstep = 0, mdiff = 0;
    if constexpr (kStep) {
        const int64_t prow = (int64_t)p.row_begin + n0 + g + G * REG;
        wnext = p.w + prow * p.w_row_bytes + colbyte;
        wstep = (int64_t)G * p.w_row_bytes;
        if constexpr (WK == W_INT4) {
            const int64_t gi = prow * (p.K >> 7) + (col0[0] >> 7);
            snext = reinterpret_cast<const uint8_t *>(static_cast<const uint16_t *>(p.scale) + gi);
            mdiff = reinterpret_cast<const uint8_t *>(p.minv) -
                    reinterpret_cast<const uint8_t *>(p.scale);
            sstep = (int64_t)G * (p.K >> 7) * 2;
        } else if constexpr (WK == W_NVFP4_A16) {
            snext = static_cast<const uint8_t *>(p.scale) + prow * (p.K >> 4) + (col0[0] >> 4);
            sstep = (int64_t)G * (p.K >> 4);
        } else {
            snext = reinterpret_cast<const uint8_t *>(static_cast<const uint16_t *>(p.scale) + prow);
            sstep = (int64_t)G * 2;
        }
    }

    // Request ring row jr (row j = REG + jr of this warp) into ring slot `slot`
    // (one commit group per call, empty past the last row, so wait_group counts
    // stay uniform).
    uint32_t sw[NSLOT][W], swm[NSLOT][W];
    auto issue = [&](int jr, int slot) {
        uint32_t sv[W], mv[W];
#pragma unroll
        for (int h = 0; h < W; ++h) {
            sv[h] = 0u;
            mv[h] = 0u;
        }
        if (jr < my_ring) {
#pragma unroll
            for (int h = 0; h < W; ++h) {
                const uint8_t *src = p.w;
                if (colok[h]) {
                    if constexpr (kStep) {
                        src = wnext + h * HB;
                        sv[h] = ld_nc_u16(snext + h * SB);
                        if constexpr (WK == W_INT4)
                            mv[h] = ld_nc_u16(snext + h * SB + mdiff);
                    } else {
                        const int64_t prow = rows_phys(p, n0 + g + G * (REG + jr));
                        src = p.w + prow * p.w_row_bytes + colbyte + h * HB;
                        sv[h] = rows_scale_global<WK>(p, prow, col0[h]);
                        mv[h] = rows_min_global<WK>(p, prow, col0[h]);
                    }
                }
                cp_async_16(ring + (uint32_t)(slot * W + h) * (RK_THREADS * 16), src,
                            colok[h] ? 16u : 0u);
            }
            if constexpr (kStep) {
                wnext += wstep;
                snext += sstep;
            }
        }
#pragma unroll
        for (int h = 0; h < W; ++h) {
            sw[slot][h] = sv[h];
            swm[slot][h] = mv[h];
        }
        cp_async_commit();
    };

    // the first REG rows of the warp: 128-bit loads straight into registers
    constexpr int NREG = REG > 0 ? REG : 1;
    uint4 q[NREG][W];
    uint32_t sq[NREG][W], sqm[NREG][W];
#pragma unroll
    for (int r = 0; r < NREG; ++r) {
#pragma unroll
        for (int h = 0; h < W; ++h) {
            q[r][h] = make_uint4(0u, 0u, 0u, 0u);
            sq[r][h] = 0u;
            sqm[r][h] = 0u;
        }
        if (r < REG && r < my_rows) {
            const int64_t prow = rows_phys(p, n0 + g + G * r);
#pragma unroll
            for (int h = 0; h < W; ++h) {
                if (colok[h]) {
                    q[r][h] = ld_stream_v4(p.w + prow * p.w_row_bytes + colbyte + h * HB);
                    sq[r][h] = rows_scale_global<WK>(p, prow, col0[h]);
                    sqm[r][h] = rows_min_global<WK>(p, prow, col0[h]);
                }
            }
        }
    }
    if (REG > 0 && p.ring_defer_ns)
        __nanosleep(p.ring_defer_ns);
#pragma unroll
    for (int i = 0; i < NSLOT; ++i)
        issue(i, i);
    float gsc = 1.f;
    if constexpr (WK == W_NVFP4_A16)
        gsc = __ldg(p.gscale);
    pdl_launch_dependents();
    // x comes from the previous kernel.  One warp waits for it; the others wait
    // at the barrier, which issues nothing (all warps polling the dependency
    // would take issue slots from the running call's CTA beside this one).
    if (threadIdx.x < 32)
        pdl_wait();
    __syncthreads();
    stage_x<WK, MT, WK == W_INT4>(p, Kpad, xs, cf, (int)threadIdx.x, RK_THREADS);
    __syncthreads();

    uint32_t xr[W][MT][XV];
    float4 cd[W][MT];        // int4: (2^-p, X, -, -); NVFP4: (2^-p * g, ...)
#pragma unroll
    for (int h = 0; h < W; ++h)
        rows_load_x<WK, MT, XV>(xs, cf, Kpad, W * ks + h, lane, col0[h], gsc, xr[h], cd[h]);

    // one row's partial: the slices' dot products, summed in slice order
    auto row_dot = [&](const uint4 (&qv)[W], const uint32_t (&s0)[W], const uint32_t (&s1)[W],
                       float *out) {
        rows_dot<WK, MT, XV>(qv[0], s0[0], s1[0], xr[0], cd[0], out);
#pragma unroll
        for (int h = 1; h < W; ++h) {
            float t[MT];
            rows_dot<WK, MT, XV>(qv[h], s0[h], s1[h], xr[h], cd[h], t);
#pragma unroll
            for (int m = 0; m < MT; ++m)
                out[m] += t[m];
        }
    };

    if constexpr (REG > 0) {
        static_assert(REG == RB, "the register batch is one row batch");
        float part[RB * MT];
#pragma unroll
        for (int r = 0; r < RB; ++r)
            row_dot(q[r], sq[r], sqm[r], part + r * MT);
        rows_park<RB, MT, S, DS>(p, n0, part, lane, ks, g, G, my_rows, red);
    }

    for (int j0 = 0; j0 < my_ring; j0 += NSLOT) {
#pragma unroll
        for (int hb = 0; hb < NB; ++hb) {
            const int jb = j0 + hb * RB;
            if (jb >= my_ring)
                break;
            cp_async_wait<(NB - 1) * RB>();       // this batch's RB groups have landed
            float part[RB * MT];
#pragma unroll
            for (int r = 0; r < RB; ++r) {
                uint4 qv[W];
#pragma unroll
                for (int h = 0; h < W; ++h)
                    qv[h] = ring_ld[((hb * RB + r) * W + h) * RK_THREADS];
                row_dot(qv, sw[hb * RB + r], swm[hb * RB + r], part + r * MT);
            }
            // the slots' contents are in registers now: refill them NB * RB rows ahead
#pragma unroll
            for (int r = 0; r < RB; ++r)
                issue(jb + NSLOT + r, hb * RB + r);
            rows_park<RB, MT, S, DS>(p, n0, part, lane, ks, g + G * (REG + jb), G, my_ring - jb,
                                     red);
        }
    }
    cp_async_wait<0>();                           // nothing left in flight at exit
    if constexpr (!DS) {
        __syncthreads();
        rows_store<MT, S>(p, red, n0, rows_cta, RK_THREADS);
    }
}

// ------------------------------------------------------------------ host side
template <int WK, int MT, int RB, int NB, int W>
static const void *rows_select_s(int S, bool direct)
{
    constexpr int REG = MT == 1 ? RB : 0;       // one token: first batch in registers
    if constexpr (W == 2) {
        if (S == 1 && direct) return reinterpret_cast<const void *>(&q4_rows_kernel<WK, MT, RB, 1, NB, REG, W, true>);
    }
    if (S == 1) return reinterpret_cast<const void *>(&q4_rows_kernel<WK, MT, RB, 1, NB, REG, W, false>);
    if constexpr (W == 1) {
        if (S == 2) return reinterpret_cast<const void *>(&q4_rows_kernel<WK, MT, RB, 2, NB, REG, W, false>);
        if (S == 4) return reinterpret_cast<const void *>(&q4_rows_kernel<WK, MT, RB, 4, NB, REG, W, false>);
        if (S == 8) return reinterpret_cast<const void *>(&q4_rows_kernel<WK, MT, RB, 8, NB, REG, W, false>);
        if constexpr (WK == W_INT8 && MT == 1) {    // K up to 8192 int8 columns: 16 k-steps
            if (S == 16) return reinterpret_cast<const void *>(&q4_rows_kernel<WK, MT, RB, 16, NB, REG, W, false>);
        }
    }
    return nullptr;
}

// (MT, RB, NB, W) variants: one token (1, 4, 2, 1 or 2), two (2, 4, 2, 1), four
// (4, 2, 2, 1).  Two slices per lane only for one token of the 4-bit kinds with
// K <= 2048 (one wide k-step).
template <int WK>
static const void *rows_select_kind(int mt, int w, int S, bool direct)
{
    if constexpr (WK == W_INT4 || WK == W_NVFP4_A16) {
        if (mt == 1 && w == 2) return rows_select_s<WK, 1, 4, 2, 2>(S, direct);
    }
    if (w != 1) return nullptr;
    if (mt == 1) return rows_select_s<WK, 1, 4, 2, 1>(S, false);
    if (mt == 2) return rows_select_s<WK, 2, 4, 2, 1>(S, false);
    if (mt == 4) return rows_select_s<WK, 4, 2, 2, 1>(S, false);
    return nullptr;
}

static const void *rows_select(const RowsPlan &pl)
{
    if (pl.kind == W_INT4) return rows_select_kind<W_INT4>(pl.mt, pl.w, pl.S, pl.direct);
    if (pl.kind == W_NVFP4_A16) return rows_select_kind<W_NVFP4_A16>(pl.mt, pl.w, pl.S, pl.direct);
    if (pl.kind == W_BF16) return rows_select_kind<W_BF16>(pl.mt, pl.w, pl.S, pl.direct);
    if (pl.kind == W_INT8) return rows_select_kind<W_INT8>(pl.mt, pl.w, pl.S, pl.direct);
    return nullptr;
}

static int rows_warps(const RowsPlan &pl)
{
    if (pl.mt == 1)
        return pl.w == 2 ? RowsShape<1, 2>::NW : RowsShape<1, 1>::NW;
    return RowsShape<2, 1>::NW;
}

// Slices per lane of the one-token 4-bit kernels (1 or 2).
constexpr int kOneTokenSlices = 2;

static int rows_kstep(int kind)
{
    return kind == W_BF16 ? 256 : (kind == W_INT8 ? 512 : 1024);
}

// k-steps of a row: ceil(K / kstep) rounded up to a power of two, so that the
// warps of a CTA split evenly into row groups (the k-steps past K read nothing
// and add zeros).
static int rows_ksteps(int kind, int K, int w = 1)
{
    const int kstep = rows_kstep(kind) * w;
    const int s = (K + kstep - 1) / kstep;
    int S = 1;
    while (S < s)
        S *= 2;
    return S;
}

bool rows_eligible(int kind, int K)
{
    const int S = rows_ksteps(kind, K);
    if (S > 8 && !(kind == W_INT8 && S == 16))
        return false;
    if (kind == W_INT8) return K % 16 == 0;
    if (kind == W_INT4) return K % 128 == 0;
    if (kind == W_NVFP4_A16) return K % 32 == 0;
    if (kind == W_BF16) return K % 8 == 0;
    return false;
}

q4_status rows_plan(const DeviceInfo &dev, int kind, int M, int N, int K, RowsPlan &plan)
{
    plan = RowsPlan{};
    plan.kind = kind;
    const int ch = (kind == W_INT4 || kind == W_INT8) ? 4 : (kind == W_BF16 ? 0 : 1);
    // one launch per 1, 2 or 4 tokens; three tokens take the 4-token kernel once
    // (weights read once: 17.7 against 20.6 us per NVFP4 batched-decode step as
    // a 2-token plus a 1-token launch)
    plan.mt = M >= 3 ? 4 : (M >= 2 ? 2 : 1);
    if (rows_ksteps(kind, K) > 8)
        plan.mt = 1;                 // 16 k-steps need the 16-warp one-token CTA
    // One token of a 4-bit kind with K <= 2048: two 32-column slices per lane,
    // 8 warps (fewer instructions per weight byte: 2.94M against 3.66M for the
    // NVFP4 16384 x 2048 GEMV; 4.68 against 4.75 us per chained call).  Longer
    // rows keep 16 warps: with under seven rows per warp the call is bound by
    // latency, not issue (int4 2048 x 8192: 4.13 against 3.92 us).
    plan.w = (plan.mt == 1 && (kind == W_INT4 || kind == W_NVFP4_A16) &&
              rows_ksteps(kind, K) <= 2) ? kOneTokenSlices : 1;
    const int kstep = rows_kstep(kind) * plan.w;
    plan.S = rows_ksteps(kind, K, plan.w);
    plan.rb = plan.mt == 4 ? 2 : 4;
    const int nw = rows_warps(plan);
    const int G = nw / plan.S;
    const size_t Kpad = (size_t)plan.S * kstep;
    // Grid: one 16-warp CTA per SM per call for one token, two 8-warp CTAs for
    // several (at least one row per warp group); per-row partials capped at
    // 24 KB per CTA.
    int64_t grid = (int64_t)dev.sms * (plan.mt == 1 ? 1 : 2);
    const int64_t want = ((int64_t)N + G - 1) / G;
    if (want < grid)
        grid = want;
    const int64_t rows_limit = (24 * 1024) / ((int64_t)plan.S * plan.mt * 4);
    const int64_t need = ((int64_t)N + rows_limit - 1) / rows_limit;
    if (need > grid)
        grid = need;
    if (grid < 1)
        grid = 1;
    if (grid > 0x7fffffff)
        return fail(Q4_ERR_SHAPE, "N=%d too large", N);
    plan.grid = (int)grid;
    const int64_t rows_cap = ((int64_t)N + grid - 1) / grid;
    const size_t rest = (size_t)plan.mt * Kpad * 2 + (size_t)plan.mt * (Kpad / 32) * ch * 4 +
                        (size_t)rows_cap * plan.S * plan.mt * 4;
    // Two row batches in flight per thread (measured: a deeper ring only delays
    // the first batches, since 16 warps' cp.async traffic per SM is throttled).
    plan.nb = 2;
    // Two-slice kernels whose warps own no more rows than they request before
    // the dependency wait (4 register rows + an 8-row ring) store each row from
    // the cross-lane reduction; longer row lists keep the final store pass,
    // since their stores would meet their own later ring refills (NVFP4 16384 x
    // 2048: 4.48 against 4.43 us per chained call with direct stores).
    if (plan.w == 2 && plan.S == 1) {
        const int64_t rows_cta = ((int64_t)N + grid - 1) / grid;
        const int64_t per_warp = (rows_cta + (nw / plan.S) - 1) / (nw / plan.S);
        plan.direct = per_warp <= (int64_t)plan.rb * (1 + plan.nb);
    }
    plan.smem = rows_ring_bytes(nw, plan.nb, plan.rb, plan.w) + rest;
    if (plan.smem > dev.smem_optin)
        return fail(Q4_ERR_SHAPE, "K=%d too large for the whole-row kernels", K);
    const void *k = rows_select(plan);
    if (!k)
        return fail(Q4_ERR_ARG, "no whole-row kernel for kind %d, S=%d", kind, plan.S);
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)plan.smem);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaFuncSetAttribute(whole-row kernel)");
    return Q4_OK;
}

q4_status rows_launch(const RowsPlan &plan, GemvParams p, int M, cudaStream_t stream, bool pdl)
{
    const void *k = rows_select(plan);
    p.S = plan.S;
    p.grid = plan.grid;
    p.rows_q = p.N / plan.grid;
    p.rows_r = p.N % plan.grid;
    // A chained one-token NVFP4 call whose warps own more rows than their
    // registers and ring request before the wait (the rest are requested while
    // the call computes) holds its ring requests back by 300 ns: the register
    // rows go out at once, and the ring burst no longer lands on the running
    // call's x staging and refills.  Measured on 16384 x 2048: 4.80 against
    // 5.19 us per chained call.  int4 at that shape is 1.3-1.8% faster without
    // it (4.83 against 4.89-4.92 us), and shapes whose rows all fit the
    // pre-wait requests lose 3-14% with any delay; neither uses it.
    p.ring_defer_ns = 0;
    if (pdl && plan.mt == 1 && plan.kind == W_NVFP4_A16) {
        const int G = rows_warps(plan) / plan.S;
        const int64_t per_warp = ((int64_t)(p.rows_q + (p.rows_r ? 1 : 0)) + G - 1) / G;
        if (per_warp > (int64_t)plan.rb * (1 + plan.nb))
            p.ring_defer_ns = 300;
    }
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    for (int m0 = 0; m0 < M; m0 += plan.mt) {
        p.m0 = m0;
        p.mcount = (M - m0) < plan.mt ? (M - m0) : plan.mt;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)plan.grid);
        cfg.blockDim = dim3(rows_warps(plan) * 32);
        cfg.dynamicSmemBytes = plan.smem;
        cfg.stream = stream;
        cfg.attrs = pdl ? attr : nullptr;
        cfg.numAttrs = pdl ? 1 : 0;
        void *args[] = {&p};
        cudaError_t e = cudaLaunchKernelExC(&cfg, k, args);
        if (e != cudaSuccess)
            return cuda_fail(e, "launch of a whole-row kernel");
    }
    return Q4_OK;
}

}  // namespace q4
