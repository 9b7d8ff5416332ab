// Round-to-nearest quantisers from BF16 weights to the two 4-bit layouts (run
// once, when a checkpoint is packed; not on the decode path).
//
//   int4-g128-minmax ("rumik-oss-1-int4", "Format (rumik-int4-g128-minmax-v1)"):
//     per group of 128 columns lo = min, hi = max; scale = fp16((hi - lo) / 15),
//     min = fp16(lo); code = clamp(rint((w - min) / scale), 0, 15), 0 when the
//     fp16 scale is 0; two codes per byte, low nibble = even column.
//   NVFP4 ("VoxCPM2 NVFP4 (GPTQ)", "NVFP4 settings": E2M1 codes, group 16, e4m3
//     group scales, one global scale per matrix): G = amax(W) / (6 * 448) (1 when
//     the matrix is 0), per group s = e4m3((amax_g / 6) / G) (nearest even,
//     saturating), S = e4m3(s) * G, code = E2M1(w / S) (nearest even, saturating
//     at 6, magnitude 0 stored as +0).  The global scale multiplies on decode.
//
// Every arithmetic step is a single IEEE fp32 operation rounded to nearest even
// (explicit __f*_rn intrinsics, so nothing is contracted into a fused
// multiply-add); the conversions use the hardware's round-to-nearest-even
// converters (cvt.rn.f16.f32, cvt.rn.satfinite.e4m3x2.f32,
// cvt.rn.satfinite.e2m1x2.f32).
#include "q4_device.cuh"
#include "q4_internal.h"

namespace q4 {

__device__ __forceinline__ uint32_t e4m3_of(float v)      // one e4m3 byte
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.f), "f"(v));
    return r & 0xffu;                                      // b converts to the low byte
}

__device__ __forceinline__ uint32_t e2m1_pair(float even, float odd)   // two nibbles
{
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
        "cvt.u32.u8 %0, t;\n\t}"
        : "=r"(r) : "f"(odd), "f"(even));                 // a -> high nibble, b -> low
    // a magnitude-0 result is stored as +0
    if ((r & 0x7u) == 0u) r &= 0xf0u;
    if ((r & 0x70u) == 0u) r &= 0x0fu;
    return r;
}

// ------------------------------------------------------------------ int4-g128
// One warp per group of 128 columns: lane l holds columns 4l .. 4l + 3.
__global__ void __launch_bounds__(256) quantize_int4_kernel(const uint16_t *__restrict__ w,
                                                            uint8_t *__restrict__ q,
                                                            uint16_t *__restrict__ sc,
                                                            uint16_t *__restrict__ mn,
                                                            int N, int K)
{
    const int groups = K / 128;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (warp >= (int64_t)N * groups)
        return;
    const int64_t n = warp / groups;
    const int g = (int)(warp - n * groups);
    const uint2 raw = *reinterpret_cast<const uint2 *>(w + n * K + g * 128 + lane * 4);
    const float v[4] = {bf16_bits_to_f32(raw.x & 0xffffu), bf16_bits_to_f32(raw.x >> 16),
                        bf16_bits_to_f32(raw.y & 0xffffu), bf16_bits_to_f32(raw.y >> 16)};
    float lo = fminf(fminf(v[0], v[1]), fminf(v[2], v[3]));
    float hi = fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3]));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
        hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    const __half s16 = __float2half_rn(__fdiv_rn(__fsub_rn(hi, lo), 15.f));
    const __half m16 = __float2half_rn(lo);
    const float s = __half2float(s16);
    const float m = __half2float(m16);
    uint32_t c[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        int ci = 0;
        if (s > 0.f) {
            ci = __float2int_rn(__fdiv_rn(__fsub_rn(v[i], m), s));
            ci = ci < 0 ? 0 : (ci > 15 ? 15 : ci);
        }
        c[i] = (uint32_t)ci;
    }
    const uint16_t packed = (uint16_t)(c[0] | (c[1] << 4) | (c[2] << 8) | (c[3] << 12));
    *reinterpret_cast<uint16_t *>(q + n * (K / 2) + g * 64 + lane * 2) = packed;
    if (lane == 0) {
        sc[n * groups + g] = __half_as_ushort(s16);
        mn[n * groups + g] = __half_as_ushort(m16);
    }
}

// ---------------------------------------------------------------------- NVFP4
// Pass 1: amax of the whole matrix, as the bits of a non-negative float (which
// order like unsigned integers), into *amax_bits (zeroed before the launch).
__global__ void __launch_bounds__(256) amax_kernel(const uint4 *__restrict__ w, int64_t n8,
                                                   unsigned *amax_bits)
{
    float a = 0.f;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8;
         i += (int64_t)gridDim.x * blockDim.x) {
        const uint4 t = w[i];
        const uint32_t e[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            a = fmaxf(a, fabsf(bf16_bits_to_f32(e[j] & 0xffffu)));
            a = fmaxf(a, fabsf(bf16_bits_to_f32(e[j] >> 16)));
        }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1)
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    __shared__ float wmax[8];
    if ((threadIdx.x & 31) == 0)
        wmax[threadIdx.x >> 5] = a;
    __syncthreads();
    if (threadIdx.x == 0) {
        float b = 0.f;
        for (int i = 0; i < (int)(blockDim.x >> 5); ++i)
            b = fmaxf(b, wmax[i]);
        atomicMax(amax_bits, __float_as_uint(b));
    }
}

__device__ __forceinline__ float global_scale_of(unsigned amax_bits)
{
    const float amax = __uint_as_float(amax_bits);
    return amax > 0.f ? __fdiv_rn(amax, 2688.f) : 1.f;    // 2688 = 6 * 448
}

// Pass 2: one thread per group of 16 columns.
__global__ void __launch_bounds__(256) quantize_nvfp4_kernel(const uint16_t *__restrict__ w,
                                                             uint8_t *__restrict__ q,
                                                             uint8_t *__restrict__ sc,
                                                             const unsigned *amax_bits,
                                                             int N, int K)
{
    const int groups = K / 16;
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= (int64_t)N * groups)
        return;
    const int64_t n = t / groups;
    const int g = (int)(t - n * groups);
    const uint4 *src = reinterpret_cast<const uint4 *>(w + n * K + g * 16);
    const uint4 r0 = src[0], r1 = src[1];
    const uint32_t e[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
    float v[16];
    float ag = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        v[2 * j] = bf16_bits_to_f32(e[j] & 0xffffu);
        v[2 * j + 1] = bf16_bits_to_f32(e[j] >> 16);
        ag = fmaxf(ag, fmaxf(fabsf(v[2 * j]), fabsf(v[2 * j + 1])));
    }
    const float G = global_scale_of(*amax_bits);
    const uint32_t s8 = e4m3_of(__fdiv_rn(__fdiv_rn(ag, 6.f), G));
    const float S = __fmul_rn(__half2float(__ushort_as_half(
                                  (uint16_t)(e4m3x2_to_f16x2(s8) & 0xffffu))), G);
    uint32_t packed[2] = {0u, 0u};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        uint32_t byte = 0u;
        if (S > 0.f)
            byte = e2m1_pair(__fdiv_rn(v[2 * j], S), __fdiv_rn(v[2 * j + 1], S));
        packed[j / 4] |= byte << (8 * (j % 4));
    }
    *reinterpret_cast<uint2 *>(q + n * (K / 2) + g * 8) = make_uint2(packed[0], packed[1]);
    sc[n * groups + g] = (uint8_t)s8;
}

// Pass 3: the amax word becomes the global scale.
__global__ void global_scale_kernel(float *gscale)
{
    *gscale = global_scale_of(__float_as_uint(*gscale));
}

static unsigned blocks_of(int64_t threads)
{
    return (unsigned)((threads + 255) / 256);
}

q4_status launch_quantize_int4(const uint16_t *w, uint8_t *q, uint16_t *s, uint16_t *m, int N,
                               int K, cudaStream_t st)
{
    const int64_t threads = (int64_t)N * (K / 128) * 32;
    quantize_int4_kernel<<<blocks_of(threads), 256, 0, st>>>(w, q, s, m, N, K);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? Q4_OK : cuda_fail(e, "launch of quantize_int4_kernel");
}

q4_status launch_quantize_nvfp4(const uint16_t *w, uint8_t *q, uint8_t *s, float *gscale, int N,
                                int K, cudaStream_t st)
{
    // the global-scale word holds the amax bits until pass 3 converts it
    cudaError_t e = cudaMemsetAsync(gscale, 0, sizeof(float), st);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaMemsetAsync(global scale)");
    const int64_t n8 = (int64_t)N * K / 8;
    int64_t blocks = blocks_of(n8);
    if (blocks > 4096)
        blocks = 4096;
    amax_kernel<<<(unsigned)blocks, 256, 0, st>>>(reinterpret_cast<const uint4 *>(w), n8,
                                                   reinterpret_cast<unsigned *>(gscale));
    quantize_nvfp4_kernel<<<blocks_of((int64_t)N * (K / 16)), 256, 0, st>>>(
        w, q, s, reinterpret_cast<const unsigned *>(gscale), N, K);
    global_scale_kernel<<<1, 1, 0, st>>>(gscale);
    e = cudaGetLastError();
    return e == cudaSuccess ? Q4_OK : cuda_fail(e, "launch of the NVFP4 quantiser");
}

}  // namespace q4
