// Whole-matrix decoders to fp32 (test helpers).  They run the same in-register
// decoders as the linear kernels -- the bf16 (128 + c) trick for int4 codes, the
// E2M1 and e4m3 conversions for NVFP4 -- so that a bit-exact comparison of their
// output with the CPU oracle checks those decoders and the nibble order.
//   int4-g128-minmax ("rumik-oss-1-int4", "Format"): w = c * scale + min; c*scale
//     is exact in fp32, so fmaf gives the exact value rounded once.
//   NVFP4 ("VoxCPM2 NVFP4 (GPTQ)", "NVFP4 settings"): w = E2M1 * e4m3 * g;
//     E2M1 * e4m3 is exact in fp32, so one multiply by g rounds once.
#include "q4_device.cuh"
#include "q4_internal.h"

namespace q4 {

// One thread per 4 packed bytes (8 weights).  K % 8 == 0 for both layouts.
__global__ void dequant_int4_kernel(const uint8_t *__restrict__ q,
                                    const uint16_t *__restrict__ sc,
                                    const uint16_t *__restrict__ mn, float *__restrict__ w,
                                    int N, int K)
{
    const int64_t words_per_row = K / 8;
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= (int64_t)N * words_per_row)
        return;
    const int64_t n = t / words_per_row;
    const int k0 = (int)(t - n * words_per_row) * 8;
    const uint32_t word = *reinterpret_cast<const uint32_t *>(q + n * (K / 2) + k0 / 2);
    const int64_t gi = n * (K / 128) + k0 / 128;
    const float s = __half2float(__ushort_as_half(sc[gi]));
    const float m = __half2float(__ushort_as_half(mn[gi]));
    float out[8];
#pragma unroll
    for (int t4 = 0; t4 < 4; ++t4) {
        // columns k0 + t4 (low half) and k0 + t4 + 4 (high half)
        const uint32_t pr = int4_pair_bf16_biased(word >> (4 * t4));
        const float clo = bf16_bits_to_f32(pr & 0xffffu) - 128.f;
        const float chi = bf16_bits_to_f32(pr >> 16) - 128.f;
        out[t4] = fmaf(clo, s, m);
        out[t4 + 4] = fmaf(chi, s, m);
    }
    float4 *dst = reinterpret_cast<float4 *>(w + n * K + k0);
    dst[0] = make_float4(out[0], out[1], out[2], out[3]);
    dst[1] = make_float4(out[4], out[5], out[6], out[7]);
}

__global__ void dequant_nvfp4_kernel(const uint8_t *__restrict__ q,
                                     const uint8_t *__restrict__ sc,
                                     const float *__restrict__ gscale, float *__restrict__ w,
                                     int N, int K)
{
    const int64_t words_per_row = K / 8;
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= (int64_t)N * words_per_row)
        return;
    const int64_t n = t / words_per_row;
    const int k0 = (int)(t - n * words_per_row) * 8;
    const uint32_t word = *reinterpret_cast<const uint32_t *>(q + n * (K / 2) + k0 / 2);
    const uint32_t s2 = e4m3x2_to_f16x2(sc[n * (K / 16) + k0 / 16]);
    const float s = f16lo_to_f32(s2);
    const float g = *gscale;
    float out[8];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        const uint32_t h = e2m1x2_to_f16x2(word >> (8 * b));
        out[2 * b] = (f16lo_to_f32(h) * s) * g;
        out[2 * b + 1] = (f16hi_to_f32(h) * s) * g;
    }
    float4 *dst = reinterpret_cast<float4 *>(w + n * K + k0);
    dst[0] = make_float4(out[0], out[1], out[2], out[3]);
    dst[1] = make_float4(out[4], out[5], out[6], out[7]);
}

static unsigned blocks_for(int64_t threads, int per_block)
{
    return (unsigned)((threads + per_block - 1) / per_block);
}

q4_status launch_dequant_int4(const uint8_t *q, const uint16_t *s, const uint16_t *m, float *w,
                              int N, int K, cudaStream_t st)
{
    const int64_t threads = (int64_t)N * (K / 8);
    dequant_int4_kernel<<<blocks_for(threads, 256), 256, 0, st>>>(q, s, m, w, N, K);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? Q4_OK : cuda_fail(e, "launch of dequant_int4_kernel");
}

q4_status launch_dequant_nvfp4(const uint8_t *q, const uint8_t *s, const float *g, float *w,
                               int N, int K, cudaStream_t st)
{
    const int64_t threads = (int64_t)N * (K / 8);
    dequant_nvfp4_kernel<<<blocks_for(threads, 256), 256, 0, st>>>(q, s, g, w, N, K);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? Q4_OK : cuda_fail(e, "launch of dequant_nvfp4_kernel");
}

}  // namespace q4
