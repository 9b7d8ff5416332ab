// Token-embedding gather with int8 dequantisation ("rumik-oss-1-int4", "Format":
// embed_tokens.qweight int8 [V, 2048], scale fp16 [V]).  Reading: signed codes,
// one symmetric scale per row, e[t, k] = q[t, k] * scale[t]; the product of an
// 8-bit integer and an fp16 value is exact in fp32, so the bf16 output is that
// exact value rounded once (nearest even).
//
// One thread writes 16 columns of one token (16 code bytes in, 32 bytes of bf16
// out).  The token ids come from the previous kernel (the sampler), so they are
// read after griddepcontrol.wait; an id outside 0 .. V-1 writes a row of zeros and
// sets Q4_DEVERR_INDEX instead of reading outside the table.
#include "q4_device.cuh"
#include "q4_internal.h"

namespace q4 {

constexpr unsigned kErrIndex = 4u;

__global__ void __launch_bounds__(256) embedding_int8_kernel(const int32_t *__restrict__ ids,
                                                             const int8_t *__restrict__ q,
                                                             const uint16_t *__restrict__ sc,
                                                             uint16_t *__restrict__ out, int V,
                                                             int H, unsigned *err)
{
    pdl_launch_dependents();
    pdl_wait();
    const int m = blockIdx.y;
    const int j = blockIdx.x * blockDim.x + threadIdx.x;     // 16-column block
    if (j * 16 >= H)
        return;
    const int t = ids[m];
    uint4 o0 = make_uint4(0u, 0u, 0u, 0u), o1 = o0;
    if (t >= 0 && t < V) {
        const uint4 c = *reinterpret_cast<const uint4 *>(q + (int64_t)t * H + j * 16);
        const float s = __half2float(__ushort_as_half(sc[t]));
        const uint32_t w[4] = {c.x, c.y, c.z, c.w};
        uint32_t r[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                const float lo = __fmul_rn((float)(int8_t)(w[i] >> (16 * b)), s);
                const float hi = __fmul_rn((float)(int8_t)(w[i] >> (16 * b + 8)), s);
                r[2 * i + b] = (uint32_t)f32_to_bf16_bits(lo) | ((uint32_t)f32_to_bf16_bits(hi) << 16);
            }
        }
        o0 = make_uint4(r[0], r[1], r[2], r[3]);
        o1 = make_uint4(r[4], r[5], r[6], r[7]);
    } else if (j == 0 && err) {
        atomicOr(err, kErrIndex);
    }
    uint4 *dst = reinterpret_cast<uint4 *>(out + (int64_t)m * H + j * 16);
    dst[0] = o0;
    dst[1] = o1;
}

q4_status launch_embedding_int8(const int32_t *ids, const int8_t *q, const uint16_t *sc,
                                uint16_t *out, int M, int V, int H, cudaStream_t st, bool pdl)
{
    const int blocks16 = H / 16;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((blocks16 + 255) / 256), (unsigned)M);
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = pdl ? attr : nullptr;
    cfg.numAttrs = pdl ? 1 : 0;
    unsigned *err = device_error_flags();
    cudaError_t e = cudaLaunchKernelEx(&cfg, embedding_int8_kernel, ids, q, sc, out, V, H, err);
    return e == cudaSuccess ? Q4_OK : cuda_fail(e, "launch of embedding_int8_kernel");
}

}  // namespace q4
