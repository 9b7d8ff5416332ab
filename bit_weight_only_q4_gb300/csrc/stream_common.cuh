// Pieces shared by the two CUDA-core weight-streaming kernels (register path in
// gemv.cu, bulk-copy path in gemv_bulk.cu): the unit geometry, the staging of x
// in shared memory and the in-register decode + dot product of one unit.
#pragma once

#include "q4_device.cuh"
#include "q4_internal.h"

namespace q4 {

template <int WK>
struct Kind {
    // columns held by one lane's 16 weight bytes
    static constexpr int COLS = (WK == W_BF16) ? 8 : 32;
    static constexpr int KSTEP = 32 * COLS;
};

template <int RW>
struct UnitRegs {
    uint4 q[RW];
    uint32_t s[RW];
};

// Shared-memory image of x for one launch: MT rows of Kpad operand values
// (bf16 bits for int4 and bf16 weights, f16 bits for NVFP4), then MT x Kpad/COLS
// floats of per-chunk data (int4: chunk sum of x; NVFP4: 2^-p of the chunk's
// power-of-two prescale).  For the 4-bit kinds every k-step of 1024 columns is
// stored lane-interleaved: the i-th 16-byte vector of lane l (columns
// 32 l + 8 i .. + 7) sits at vector index i * 32 + l, so the four vector loads a
// lane issues per k-step are each conflict-free across the warp.
__device__ __forceinline__ int xs_vec_index(int k0)
{
    const int ks = k0 >> 10, kk = k0 & 1023;
    return ks * 128 + ((kk & 31) >> 3) * 32 + (kk >> 5);
}

template <int WK, int MT>
__device__ void stage_x(const GemvParams &p, int Kpad, uint16_t *xs, float *cf, int tid,
                        int nthreads)
{
    constexpr int COLS = Kind<WK>::COLS;
    const int blocks_per_row = Kpad / 8;
    const int total = MT * blocks_per_row;
    // total is a multiple of 4 and every 4 consecutive blocks form one 32-column
    // chunk handled by 4 consecutive lanes of one warp.
    for (int b0 = 0; b0 < total; b0 += nthreads) {
        const int b = b0 + tid;
        const bool active = b < total;
        const int m = active ? b / blocks_per_row : 0;
        const int k0 = active ? (b - m * blocks_per_row) * 8 : 0;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (active && m < p.mcount && k0 < p.K)
            v = *reinterpret_cast<const uint4 *>(p.x + (int64_t)(p.m0 + m) * p.K + k0);
        uint32_t e[4] = {v.x, v.y, v.z, v.w};
        if constexpr (WK == W_INT4) {
            // pair (x[8j+t], x[8j+t+4]) -- the order int4_pair_bf16_biased(w >> 4t)
            // produces codes in
            uint4 o;
            o.x = __byte_perm(e[0], e[2], 0x5410);
            o.y = __byte_perm(e[0], e[2], 0x7632);
            o.z = __byte_perm(e[1], e[3], 0x5410);
            o.w = __byte_perm(e[1], e[3], 0x7632);
            float s = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i)
                s += bf16_bits_to_f32(e[i] & 0xffffu) + bf16_bits_to_f32(e[i] >> 16);
            s += __shfl_xor_sync(0xffffffffu, s, 1);
            s += __shfl_xor_sync(0xffffffffu, s, 2);
            if (active) {
                reinterpret_cast<uint4 *>(xs + (size_t)m * Kpad)[xs_vec_index(k0)] = o;
                if ((k0 % 32) == 0)
                    cf[(size_t)m * (Kpad / COLS) + k0 / 32] = s;
            }
        } else if constexpr (WK == W_NVFP4_A16 || WK == W_NVFP4_A8) {
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
            // power-of-two prescale putting the chunk's largest |x| in [2^14, 2^15)
            // so every bf16 value of the chunk converts to fp16 without overflow
            // and, down to 2^-16 of the maximum, without rounding
            int ex = 0;
            if (amax > 0.f && !isinf(amax))
                frexpf(amax, &ex);
            int pw = 15 - ex;
            pw = pw > 100 ? 100 : (pw < -100 ? -100 : pw);
            uint32_t h[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                __half2 hh = __floats2half2_rn(ldexpf(f[2 * i], pw), ldexpf(f[2 * i + 1], pw));
                h[i] = *reinterpret_cast<uint32_t *>(&hh);
            }
            if (active) {
                reinterpret_cast<uint4 *>(xs + (size_t)m * Kpad)[xs_vec_index(k0)] =
                    make_uint4(h[0], h[1], h[2], h[3]);
                if ((k0 % 32) == 0)
                    cf[(size_t)m * (Kpad / COLS) + k0 / 32] = ldexpf(1.f, -pw);
            }
        } else {
            if (active)
                *reinterpret_cast<uint4 *>(xs + (size_t)m * Kpad + k0) = v;
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
        float cc[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            const uint4 *src = reinterpret_cast<const uint4 *>(xs + (size_t)m * Kpad) + ks * 128;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint4 t = src[i * 32 + lane];
                xr[m][4 * i + 0] = t.x; xr[m][4 * i + 1] = t.y;
                xr[m][4 * i + 2] = t.z; xr[m][4 * i + 3] = t.w;
            }
            cc[m] = cf[(size_t)m * (Kpad / COLS) + col0 / 32];
        }
#pragma unroll
        for (int r = 0; r < RW; ++r) {
            const uint32_t q[4] = {R.q[r].x, R.q[r].y, R.q[r].z, R.q[r].w};
            if constexpr (WK == W_INT4) {
                float T[MT];
#pragma unroll
                for (int m = 0; m < MT; ++m)
                    T[m] = 0.f;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const uint32_t pr = int4_pair_bf16_biased(q[j] >> (4 * t));
#pragma unroll
                        for (int m = 0; m < MT; ++m)
                            T[m] = fma2_bf16(T[m], pr, xr[m][4 * j + t]);
                    }
                }
                // sum_k (128 + c) x = 128 X + sum_k c x, so
                // s * sum c x + min * X = s * T + (min - 128 s) * X
                const float s = f16lo_to_f32(R.s[r]);
                const float mn = f16hi_to_f32(R.s[r]);
                const float mb = fmaf(-128.f, s, mn);
#pragma unroll
                for (int m = 0; m < MT; ++m)
                    acc[r][m] = fmaf(mb, cc[m], fmaf(s, T[m], acc[r][m]));
            } else {
                float Ta[MT], Tb[MT];
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    Ta[m] = 0.f;
                    Tb[m] = 0.f;
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
#pragma unroll
                    for (int b = 0; b < 4; ++b) {
                        const uint32_t h = e2m1x2_to_f16x2(q[j] >> (8 * b));
#pragma unroll
                        for (int m = 0; m < MT; ++m) {
                            if (j < 2)
                                Ta[m] = fma2_f16(Ta[m], h, xr[m][4 * j + b]);
                            else
                                Tb[m] = fma2_f16(Tb[m], h, xr[m][4 * j + b]);
                        }
                    }
                }
                const uint32_t sc = e4m3x2_to_f16x2(R.s[r]);
                const float sa = f16lo_to_f32(sc) * gsc;
                const float sb = f16hi_to_f32(sc) * gsc;
#pragma unroll
                for (int m = 0; m < MT; ++m)
                    acc[r][m] = fmaf(fmaf(Ta[m], sa, Tb[m] * sb), cc[m], acc[r][m]);
            }
        }
    }
}

}  // namespace q4
