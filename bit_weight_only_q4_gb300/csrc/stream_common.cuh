// Pieces shared by the CUDA-core weight-streaming kernels (whole-row kernel in
// gemv_rows.cu, split-K register path in gemv.cu): the unit geometry, the
// staging of x in shared memory and the in-register decode + dot product of one
// unit.
//
// Arithmetic (both 4-bit layouts): x is staged as fp16 values x' = x * 2^p with
// one power-of-two p per 32-column chunk, chosen so the chunk's largest |x'| lies
// in [2^14, 2^15): every bf16 value converts without overflow, and exactly down
// to 2^-22 of the chunk maximum.  Codes are decoded to exact fp16 operands and
// every product is accumulated in fp32 by one mixed-precision FMA
// (fma.rn.f32.f16); the chunk's partial sums are scaled back by 2^-p, the group
// scale (and min) in fp32.
//   NVFP4: E2M1 pairs -> f16x2 by cvt.rn.f16x2.e2m1x2 on bytes unpacked from the
//     packed word (no shifts); per group of 16 columns: sum_k e2m1(c) x'.
//   int4: nibble pairs -> f16x2 (1024 + c) or (1024 + 16 c) by one LOP3 each
//     ("magic number" decode); per chunk the two partial sums
//       A1 = sum_{even k} (1024 + c) x'   and   A2 = sum_{odd k} (1024 + 16 c) x'
//     give  sum_k (c s + m) x' = s A1 + (s/16) A2 + (m - 1024 s) X1 + (m - 64 s) X2
//     with X1, X2 the sums of x' over the chunk's even and odd columns (the
//     split-K kernel; the whole-row kernel stages int4 x as
//     int16 and sums c x' exactly with integer dot products, see stage_x).
#pragma once

#include "q4_device.cuh"
#include "q4_internal.h"

namespace q4 {

template <int WK>
struct Kind {
    // columns held by one lane's 16 weight bytes
    static constexpr int COLS = (WK == W_BF16) ? 8 : ((WK == W_INT8) ? 16 : 32);
    static constexpr int KSTEP = 32 * COLS;
    // floats of per-chunk data in shared memory: int4 (2^-p, X1, X2, 0), or
    // (2^-p, X, 0, 0) with int16 staging; NVFP4 (2^-p), bf16 none
    // INT8: (2^-p, sum of x' over the chunk's first 16 columns, over its last 16, 0)
    static constexpr int CH = (WK == W_INT4 || WK == W_INT8) ? 4 : ((WK == W_BF16) ? 0 : 1);
};

template <int RW>
struct UnitRegs {
    uint4 q[RW];
    uint32_t s[RW];
};

// Shared-memory image of x for one launch: MT rows of Kpad operand values
// (f16 bits of x' for the 4-bit kinds, bf16 bits for bf16 weights), then
// MT x (Kpad/32) x CH floats of per-chunk data.  For the 4-bit kinds every k-step
// of 1024 columns is stored lane-interleaved: the i-th 16-byte vector of lane l
// (columns 32 l + 8 i .. + 7) sits at vector index i * 32 + l, so the four
// vector loads a lane issues per k-step are each conflict-free across the warp.
// For int4 each vector holds the pairs (x'[8j+t], x'[8j+t+4]), t = 0..3 -- the
// order the nibble decoder produces codes in.
// INT8 (16 columns per lane, k-steps of 512): vector i of lane l (columns
// 16 l + 8 i .. + 7) at index ks * 64 + i * 32 + l.
template <int WK>
__device__ __forceinline__ int xs_vec_index_kind(int k0)
{
    if constexpr (WK == W_INT8) {
        const int ks = k0 >> 9, kk = k0 & 511;
        return ks * 64 + ((kk & 15) >> 3) * 32 + (kk >> 4);
    } else {
        const int ks = k0 >> 10, kk = k0 & 1023;
        return ks * 128 + ((kk & 31) >> 3) * 32 + (kk >> 5);
    }
}

__device__ __forceinline__ int xs_vec_index(int k0)
{
    const int ks = k0 >> 10, kk = k0 & 1023;
    return ks * 128 + ((kk & 31) >> 3) * 32 + (kk >> 5);
}

__device__ __forceinline__ float pow2f(int e)  // 2^e for -126 <= e <= 127
{
    return __uint_as_float((uint32_t)(e + 127) << 23);
}

// XI16 (int4 whole-row kernel): x' is an int16 fixed-point value instead, chunk
// maximum in [2^14, 2^15), stored as signed 16-bit pairs in the order the integer
// dot products take them -- (x0, x2), (x4, x6), (x1, x3), (x5, x7) for each 8
// columns -- with chunk data (2^-p, sum of x', -, -); a chunk holding a
// non-finite value gets a NaN sum, so its rows come out NaN.
template <int WK, int MT, bool XI16 = false>
__device__ void stage_x(const GemvParams &p, int Kpad, uint16_t *xs, float *cf, int tid,
                        int nthreads)
{
    static_assert(!XI16 || WK == W_INT4, "int16 staging is for int4 weights");
    constexpr int CH = Kind<WK>::CH;
    const int blocks_per_row = Kpad / 8;
    const int total = MT * blocks_per_row;
    // total is a multiple of 4 and every 4 consecutive blocks form one 32-column
    // chunk handled by 4 consecutive lanes of one warp.  A thread requests up to
    // XU blocks before converting any, so that long rows cost one round trip.
    constexpr int XU = 2;
    for (int b00 = 0; b00 < total; b00 += XU * nthreads) {
        uint4 vv[XU];
#pragma unroll
        for (int u = 0; u < XU; ++u) {
            const int b = b00 + u * nthreads + tid;
            const int m = b < total ? b / blocks_per_row : 0;
            const int k0 = b < total ? (b - m * blocks_per_row) * 8 : 0;
            vv[u] = make_uint4(0u, 0u, 0u, 0u);
            if (b < total && m < p.mcount && k0 < p.K)
                vv[u] = *reinterpret_cast<const uint4 *>(p.x + (int64_t)(p.m0 + m) * p.K + k0);
        }
#pragma unroll
        for (int u = 0; u < XU; ++u) {
            const int b0 = b00 + u * nthreads;
            if (b0 >= total)          // uniform across the block
                break;
            const int b = b0 + tid;
            const bool active = b < total;
            const int m = active ? b / blocks_per_row : 0;
            const int k0 = active ? (b - m * blocks_per_row) * 8 : 0;
            const uint4 v = vv[u];
            if constexpr (WK == W_BF16) {
                if (active)
                    *reinterpret_cast<uint4 *>(xs + (size_t)m * Kpad + k0) = v;
            } else {
                const uint32_t e[4] = {v.x, v.y, v.z, v.w};
                float f[8];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    f[2 * i] = bf16_bits_to_f32(e[i] & 0xffffu);
                    f[2 * i + 1] = bf16_bits_to_f32(e[i] >> 16);
                }
                float amax = 0.f;
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    amax = fmaxf(amax, fabsf(f[i]));
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
                // exponent ex with amax = f * 2^ex, f in [0.5, 1)
                int ex = 0;
                if (amax > 0.f && !isinf(amax)) {
                    const int be = (int)((__float_as_uint(amax) >> 23) & 0xff);
                    if (be > 0)
                        ex = be - 126;
                    else
                        frexpf(amax, &ex);
                }
                // chunk maximum in [2^14, 2^15); NVFP4 in [2^9, 2^10) and int4 in
                // [2^8, 2^9), so that a sum of eight products (|E2M1| <= 6,
                // |c - 8| <= 8) stays below 2^16 when a kernel accumulates it in
                // fp16; int16 staging in [2^14, 2^15)
                int pw = (XI16 ? 15 : (WK == W_NVFP4_A16 ? 10 : (WK == W_INT4 ? 9 : 15))) - ex;
                // |pw| <= 126 keeps 2^pw and 2^-pw normal fp32 numbers; the top of the
                // bf16 range (amax < 2^128) needs pw >= 15 - 128 = -113, so no finite
                // chunk is clamped at the top and every one lands in its target range
                pw = pw > 126 ? 126 : (pw < -126 ? -126 : pw);
                const float up = pow2f(pw);
                if constexpr (XI16) {
                    // x * 2^p is exact in fp32 and below 2^15 in magnitude; rounding
                    // to the nearest integer is exact for values within 2^7 of the
                    // chunk maximum (BF16 has 8 significant bits)
                    int xi[8];
                    bool bad = false;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        bad |= !(fabsf(f[i]) <= 3.402823466e38f);
                        xi[i] = __float2int_rn(f[i] * up);
                    }
                    auto pack = [](int lo, int hi) {
                        return ((uint32_t)lo & 0xffffu) | ((uint32_t)hi << 16);
                    };
                    if (active)
                        reinterpret_cast<uint4 *>(xs + (size_t)m * Kpad)[xs_vec_index_kind<WK>(k0)] =
                            make_uint4(pack(xi[0], xi[2]), pack(xi[4], xi[6]), pack(xi[1], xi[3]),
                                       pack(xi[5], xi[7]));
                    float sx = (float)(((xi[0] + xi[1]) + (xi[2] + xi[3])) + ((xi[4] + xi[5]) + (xi[6] + xi[7])));
                    if (bad)
                        sx = __int_as_float(0x7fc00000);
                    sx += __shfl_xor_sync(0xffffffffu, sx, 1);
                    sx += __shfl_xor_sync(0xffffffffu, sx, 2);
                    if (active && (k0 % 32) == 0)
                        reinterpret_cast<float4 *>(cf)[(size_t)m * (Kpad / 32) + k0 / 32] =
                            make_float4(pow2f(-pw), sx, 0.f, 0.f);
                } else {
                    float xq[8];
                    uint32_t h[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        __half2 hh;
                        if constexpr (WK == W_INT4)   // pairs (x'[t], x'[t+4])
                            hh = __floats2half2_rn(f[i] * up, f[i + 4] * up);
                        else                          // natural order
                            hh = __floats2half2_rn(f[2 * i] * up, f[2 * i + 1] * up);
                        h[i] = *reinterpret_cast<uint32_t *>(&hh);
                        xq[2 * i] = __low2float(hh);
                        xq[2 * i + 1] = __high2float(hh);
                    }
                    if (active)
                        reinterpret_cast<uint4 *>(xs + (size_t)m * Kpad)[xs_vec_index_kind<WK>(k0)] =
                            make_uint4(h[0], h[1], h[2], h[3]);
                    if constexpr (WK == W_INT4) {
                        // h[i] holds columns (i, i+4): even columns are i = 0, 2
                        float s_even = (xq[0] + xq[1]) + (xq[4] + xq[5]);
                        float s_odd = (xq[2] + xq[3]) + (xq[6] + xq[7]);
                        s_even += __shfl_xor_sync(0xffffffffu, s_even, 1);
                        s_even += __shfl_xor_sync(0xffffffffu, s_even, 2);
                        s_odd += __shfl_xor_sync(0xffffffffu, s_odd, 1);
                        s_odd += __shfl_xor_sync(0xffffffffu, s_odd, 2);
                        if (active && (k0 % 32) == 0)
                            reinterpret_cast<float4 *>(cf)[(size_t)m * (Kpad / 32) + k0 / 32] =
                                make_float4(pow2f(-pw), s_even, s_odd, 0.f);
                    } else if constexpr (WK == W_INT8) {
                        // sums of x' over the chunk's first and last 16 columns (the two
                        // lanes of the chunk): blocks t = 0, 1 and t = 2, 3
                        float sh = 0.f;
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            sh += xq[i];
                        sh += __shfl_xor_sync(0xffffffffu, sh, 1);
                        const float other = __shfl_xor_sync(0xffffffffu, sh, 2);
                        if (active && (k0 % 32) == 0)
                            reinterpret_cast<float4 *>(cf)[(size_t)m * (Kpad / 32) + k0 / 32] =
                                make_float4(pow2f(-pw), sh, other, 0.f);
                    } else {
                        if (active && (k0 % 32) == 0)
                            cf[(size_t)m * (Kpad / 32) + k0 / 32] = pow2f(-pw);
                    }
                }
                (void)CH;
            }
        }
    }
}

template <int WK, int MT, int RW>
__device__ __forceinline__ void compute_unit(const GemvParams &p, const UnitRegs<RW> &R,
                                             int ks, int lane, int Kpad, const uint16_t *xs,
                                             const float *cf, float gsc,
                                             float (&acc)[RW][MT])
{
    constexpr int COLS = Kind<WK>::COLS;
    const int col0 = ks * Kind<WK>::KSTEP + lane * COLS;
    if constexpr (WK == W_BF16) {
        uint32_t xr[MT][4];
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            uint4 t = *reinterpret_cast<const uint4 *>(xs + (size_t)m * Kpad + col0);
            xr[m][0] = t.x; xr[m][1] = t.y; xr[m][2] = t.z; xr[m][3] = t.w;
        }
#pragma unroll
        for (int r = 0; r < RW; ++r) {
            const uint32_t q[4] = {R.q[r].x, R.q[r].y, R.q[r].z, R.q[r].w};
#pragma unroll
            for (int m = 0; m < MT; ++m) {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    acc[r][m] = fma2_bf16(acc[r][m], q[j], xr[m][j]);
            }
        }
    } else {
        uint32_t xr[MT][16];
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            const uint4 *src = reinterpret_cast<const uint4 *>(xs + (size_t)m * Kpad) + ks * 128;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint4 t = src[i * 32 + lane];
                xr[m][4 * i + 0] = t.x; xr[m][4 * i + 1] = t.y;
                xr[m][4 * i + 2] = t.z; xr[m][4 * i + 3] = t.w;
            }
        }
        const int chunk = col0 / 32;
        if constexpr (WK == W_INT4) {
            float4 cd[MT];
#pragma unroll
            for (int m = 0; m < MT; ++m)
                cd[m] = reinterpret_cast<const float4 *>(cf)[(size_t)m * (Kpad / 32) + chunk];
#pragma unroll
            for (int r = 0; r < RW; ++r) {
                const uint32_t q[4] = {R.q[r].x, R.q[r].y, R.q[r].z, R.q[r].w};
                float A1[MT], A2[MT];
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    A1[m] = 0.f;
                    A2[m] = 0.f;
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t w8 = q[j] >> 8;
                    const uint32_t pa = int4_pair_f16_biased<0x000F000Fu>(q[j]);   // cols 0, 4
                    const uint32_t pb = int4_pair_f16_biased<0x00F000F0u>(q[j]);   // cols 1, 5
                    const uint32_t pc = int4_pair_f16_biased<0x000F000Fu>(w8);     // cols 2, 6
                    const uint32_t pd = int4_pair_f16_biased<0x00F000F0u>(w8);     // cols 3, 7
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        A1[m] = fma2_f16(A1[m], pa, xr[m][4 * j + 0]);
                        A2[m] = fma2_f16(A2[m], pb, xr[m][4 * j + 1]);
                        A1[m] = fma2_f16(A1[m], pc, xr[m][4 * j + 2]);
                        A2[m] = fma2_f16(A2[m], pd, xr[m][4 * j + 3]);
                    }
                }
                const float s = f16lo_to_f32(R.s[r]);
                const float mn = f16hi_to_f32(R.s[r]);
                const float c1 = fmaf(-1024.f, s, mn);
                const float c2 = fmaf(-64.f, s, mn);
                const float s16 = s * 0.0625f;
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    float t = s * A1[m];
                    t = fmaf(s16, A2[m], t);
                    t = fmaf(c1, cd[m].y, t);
                    t = fmaf(c2, cd[m].z, t);
                    acc[r][m] = fmaf(t, cd[m].x, acc[r][m]);
                }
            }
        } else {
            float cc[MT];
#pragma unroll
            for (int m = 0; m < MT; ++m)
                cc[m] = cf[(size_t)m * (Kpad / 32) + chunk] * gsc;
#pragma unroll
            for (int r = 0; r < RW; ++r) {
                const uint32_t q[4] = {R.q[r].x, R.q[r].y, R.q[r].z, R.q[r].w};
                float Ta[MT], Tb[MT];
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    Ta[m] = 0.f;
                    Tb[m] = 0.f;
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t h[4];
                    e2m1x8_to_f16x2x4(q[j], h);
#pragma unroll
                    for (int b = 0; b < 4; ++b) {
#pragma unroll
                        for (int m = 0; m < MT; ++m) {
                            if (j < 2)
                                Ta[m] = fma2_f16(Ta[m], h[b], xr[m][4 * j + b]);
                            else
                                Tb[m] = fma2_f16(Tb[m], h[b], xr[m][4 * j + b]);
                        }
                    }
                }
                const uint32_t sc = e4m3x2_to_f16x2(R.s[r]);
                const float sa = f16lo_to_f32(sc);
                const float sb = f16hi_to_f32(sc);
#pragma unroll
                for (int m = 0; m < MT; ++m)
                    acc[r][m] = fmaf(fmaf(Ta[m], sa, Tb[m] * sb), cc[m], acc[r][m]);
            }
        }
    }
}

}  // namespace q4
