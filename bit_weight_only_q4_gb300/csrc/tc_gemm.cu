// Tensor-core (tcgen05) weight-only GEMM for sm_103a: y[M,N] = x[M,K] W^T with W in
// either 4-bit layout, for batched decode (a few dozen tokens) and prefill.
//
// What it computes: the same dequantise-and-multiply as the CUDA-core kernels
// ("rumik-oss-1-int4", "Format": w = code * scale + min; "VoxCPM2 NVFP4 (GPTQ)",
// "NVFP4 settings": w = E2M1 * e4m3 * g), with the products accumulated in fp32
// by the tensor cores and the output rounded to bf16.
//
// Design (swap-AB: weights are the MMA's M dimension, tokens its N dimension):
//   * One CTA computes a tile of 128 weight rows x TN tokens over a range of
//     64-column K chunks (split-K across CTAs when the grid would be too small).
//   * Warp 0 (one thread) streams, per chunk, the token tile of x (bf16, TMA
//     tensor load with 128-byte swizzle) and the 128 rows x 32 bytes of packed
//     codes (TMA tensor load) into a ring of shared-memory stages.
//   * Sixteen worker warps in two groups of eight take the stages in turn and
//     dequantise them into the A operand tiles (16-bit, K-major, 128-byte
//     swizzle): a thread takes 16 weights of one row per step, and a warp's code
//     reads are 256 contiguous bytes (no bank conflicts).
//   * NVFP4: bf16 operands.  x goes to the MMA as stored, and the weights are
//     E2M1 * e4m3 * 2^eg in bf16, exact (2^eg a power-of-two share of the global
//     scale; the epilogue applies the rest).
//   * int4: fp16 operands, w = fp16(c * s + m) (one fused multiply-add, single
//     rounding).  The workers also convert the chunk's x tile in place from bf16
//     to fp16, each token scaled by a power of two that puts its largest |x| in
//     [2^14, 2^15) (for large M a small kernel converts x once per call
//     instead); the epilogue undoes the scale, so every bf16 activation is in
//     range.
//   * Warp 1 allocates the TMEM accumulator (128 lanes x TN fp32 columns) and one
//     thread issues tcgen05.mma (kind::f16, M=128, N=TN, K=16) four times per
//     chunk, then tcgen05.commit frees the stage.
//   * The worker warps read the accumulator back with tcgen05.ld (each warp its
//     32-lane quadrant), apply the global scale and store bf16 -- or, under
//     split-K, write fp32 partials and the last CTA to arrive sums them in k
//     order (deterministic, no CTA waits for another).
// Every mbarrier wait is bounded and reports a timeout in the device error word;
// the TMEM allocation is released on every path.
#include <cuda.h>
#include <mutex>

#include "q4_device.cuh"
#include "q4_internal.h"

namespace q4 {

constexpr int TC_ROWS = 128;           // weight rows per tile (MMA M)
constexpr int TC_KC = 64;              // K columns per chunk (128 bytes of fp16)
constexpr int TC_GROUPS = 4;           // epilogue: four warps share a TMEM lane quadrant
constexpr int TC_WORKERS = 4 * TC_GROUPS;   // dequant / epilogue warps
constexpr int TC_THREADS = (2 + TC_WORKERS) * 32;

struct TcParams {
    const uint16_t *x;         // bf16 [M, K]
    const uint8_t *codes;      // [N, K/2]
    const void *scale;         // int4: fp16 [N, K/128]; NVFP4: e4m3 [N, K/16]
    const uint16_t *minv;      // int4: fp16 [N, K/128]
    const float *gscale;       // NVFP4: device fp32 scalar
    uint16_t *y;               // bf16 [M, N]
    float *ws;                 // split-K partials [tile][ks][TN][128]
    unsigned *tickets;         // [tile]
    unsigned *err;
    int M, N, K;
    int TN;                    // tokens per tile (multiple of 16, <= 256)
    int tiles_m;               // ceil(M / TN)
    int KS;                    // split-K factor
    int chunks;                // K / 64
    int ns;                    // ring stages (super-chunks)
    int tmem_cols;             // power of two >= max(32, TN)
    int tmem_a0;               // A in tensor memory: first column of the A sub-tiles
    int x_f16;                 // x already converted to prescaled fp16 (large M)
    const float *xdn;          // with x_f16: 2^-e_m per token [M]
};


// ------------------------------------------------------------ PTX helpers
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            uint32_t bar)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%2, %3}], [%4];"
                 ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
                 : "memory");
}


__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major operand in the canonical 128-byte
// swizzle layout (rows of 128 bytes, 8-row atoms of 1024 bytes).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr)
{
    uint64_t d = 0;
    d |= (uint64_t)((addr & 0x3FFFFu) >> 4);          // start address
    d |= (uint64_t)1 << 16;                            // leading byte offset (unused)
    d |= (uint64_t)(1024 >> 4) << 32;                  // stride byte offset: 8 rows
    d |= (uint64_t)1 << 46;                            // descriptor version
    d |= (uint64_t)2 << 61;                            // 128-byte swizzle
    return d;
}

// Instruction descriptor of tcgen05.mma kind::f16: fp16 A and B (K-major),
// fp32 accumulator, M = 128, N = n.
__device__ __forceinline__ uint32_t idesc_f16(int n, bool bf16 = false)
{
    const uint32_t ab = bf16 ? 1u : 0u;        // operand format: 0 f16, 1 bf16
    return (1u << 4)                    // D format: f32
         | (ab << 7) | (ab << 10)       // A, B format
         | ((uint32_t)(n >> 3) << 17)   // N / 8
         | ((uint32_t)(TC_ROWS >> 4) << 24);   // M / 16
}

// tcgen05.mma kind::f16 (M = 128) with both descriptors passed as 32-bit halves,
// so that the issuing loop only steps the start-address fields (low halves: +2 per
// 32 bytes).  One thread issues every MMA of a CTA; rebuilding two 64-bit
// descriptors per MMA costs that thread more than the MMA costs the tensor core.
__device__ __forceinline__ void mma_f16_2(uint32_t tmem_d, uint32_t a_lo, uint32_t a_hi, uint32_t b_lo,
                                          uint32_t b_hi, uint32_t idesc, uint32_t accumulate)
{
    asm volatile("{\n\t.reg .b64 ad, bd;\n\t.reg .pred p;\n\t"
                 "setp.ne.u32 p, %6, 0;\n\t"
                 "mov.b64 ad, {%1, %2};\n\t"
                 "mov.b64 bd, {%3, %4};\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %5, p;\n\t}"
                 ::"r"(tmem_d), "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate)
                 : "memory");
}

// The same MMA with the A operand in tensor memory (row i of A in lane i, its K
// values packed two per 32-bit column, K = 16 in eight columns).
__device__ __forceinline__ void mma_f16_tmem_a(uint32_t tmem_d, uint32_t tmem_a, uint32_t b_lo,
                                               uint32_t b_hi, uint32_t idesc, uint32_t accumulate)
{
    asm volatile("{\n\t.reg .b64 bd;\n\t.reg .pred p;\n\t"
                 "setp.ne.u32 p, %5, 0;\n\t"
                 "mov.b64 bd, {%2, %3};\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], bd, %4, p;\n\t}"
                 ::"r"(tmem_d), "r"(tmem_a), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate)
                 : "memory");
}

// A warp writes 16 consecutive 32-bit columns of its 32 TMEM lanes.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
                 "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};"
                 ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]),
                   "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]),
                   "r"(v[13]), "r"(v[14]), "r"(v[15])
                 : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 "
                 "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]),
                   "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]),
                   "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t r;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
    return r;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// 2^e for -126 <= e <= 127 (a normal fp32 number, built from its exponent field)
__device__ __forceinline__ float pow2f_tc(int e)
{
    return __uint_as_float((uint32_t)(e + 127) << 23);
}

// 32-bit load through the non-coherent path (p 4-byte aligned)
__device__ __forceinline__ uint32_t ld_nc_u32(const void *p)
{
    uint32_t r;
    asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(r) : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t bmul2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// An fp16 pair whose values have at most 7 significant bits and no bits below
// the mantissa's third (every E2M1 value qualifies) -> the bf16 pair of the same
// values times 2^-112: the exponent and mantissa fields move down by 3 bits (f16
// bias 15, bf16 bias 127), the sign stays; zero stays zero.
__device__ __forceinline__ uint32_t f16x2_to_bf16x2_scaled(uint32_t h)
{
    return ((h & 0x7fff7fffu) >> 3) | (h & 0x80008000u);
}

// NVFP4 with bf16 operands: the power of two 2^eg nearest below the global scale g
// (clamped so that every E2M1 * e4m3 * 2^eg is a normal bf16 number and every
// e4m3 * 2^(112 + eg) is finite in bf16) -- the weights are dequantised as
// E2M1 * e4m3 * 2^eg, exactly, and the epilogue multiplies by g * 2^-eg.
__device__ __forceinline__ int nvfp4_bf16_exponent(float g)
{
    const int eb = (int)((__float_as_uint(g) >> 23) & 0xffu);
    if (eb == 0xff)
        return 0;
    const int e = eb - 127;
    return e < -100 ? -100 : (e > 6 ? 6 : e);
}

// e4m3 scale byte -> bf16 pair (splatted) of scale * 2^(112 + eg), exact (4
// significant bits, magnitude between 2^3 and 2^127).
__device__ __forceinline__ uint32_t e4m3_to_bf16x2_scaled(uint32_t byte, float up)
{
    float lo, hi;
    f16x2_to_f32x2(e4m3x2_to_f16x2(byte & 0xffu), lo, hi);
    (void)hi;
    const float s = lo * up;
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %1;" : "=r"(r) : "f"(s));
    return r;
}

// Per-token power-of-two prescale of x for the fp16 MMA operand.  The MMA reads
// x as fp16, whose range ends at 65504, while bf16 activations reach 3.4e38.  So
// each token m is multiplied by 2^e_m before the conversion, with e_m chosen
// from the token's largest |x| over the K range in question so that this
// maximum lands in [2^14, 2^15); the accumulator of that token is multiplied by
// 2^-e_m afterwards.  Both multiplications are exact, and the conversion is
// exact for every value within 2^28 of the token's maximum (the fp16 normal
// range); smaller values round to fp16 subnormals, an absolute error of at most
// 2^-39 of that maximum.
//   maxbits: the largest (bf16 bits & 0x7fff) of the token -- magnitudes of
//   non-NaN bf16 values order like their bit patterns, so an integer maximum
//   finds the largest |x| (inf 0x7f80 and NaN above every finite value).  A
//   token holding inf or NaN keeps e = 0: its outputs are non-finite anyway.
__device__ __forceinline__ int x_prescale_exponent(uint32_t maxbits)
{
    if (maxbits >= 0x7f80u)
        return 0;
    const int e = 141 - (int)(maxbits >> 7);   // biased exponent b: max in [2^(b-127), 2^(b-126))
    return e > 126 ? 126 : e;                   // >= 141 - 254 = -113 for every finite value
}

// Largest |x| bit pattern (see x_prescale_exponent) of the 8 bf16 values of v,
// folded into acc.
__device__ __forceinline__ uint32_t bf16x8_absmax_bits(uint4 v, uint32_t acc)
{
    const uint32_t a = __vmaxu2(__vmaxu2(v.x & 0x7fff7fffu, v.y & 0x7fff7fffu),
                                __vmaxu2(v.z & 0x7fff7fffu, v.w & 0x7fff7fffu));
    const uint32_t b = (a & 0xffffu) > (a >> 16) ? (a & 0xffffu) : (a >> 16);
    return b > acc ? b : acc;
}

__device__ __forceinline__ uint32_t f16x2_splat(uint32_t h16)
{
    return (h16 & 0xffffu) | (h16 << 16);
}

// One packed code word (8 consecutive columns of a row, low nibble = even column)
// -> 4 f16 pairs of weights in column order.  int4: w = c * s + min (s2, m2 the
// splatted fp16 scale and min; one rounding); NVFP4: w = E2M1 * e4m3 scale (sg
// splatted; exact in fp16, the global scale is applied in the epilogue), or with
// XB the bf16 pairs of E2M1 * e4m3 * 2^eg (exact).
template <int LAYOUT, bool XB>
__device__ __forceinline__ void tc_dequant_word(uint32_t word, uint32_t s2, uint32_t m2,
                                                uint32_t (&o)[4])
{
    if constexpr (LAYOUT == 0) {
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            // byte b -> (1024 + c_lo, 1024 + 16 c_hi) -> (c_lo, c_hi)
            const uint32_t t = prmt(word, 0u, (uint32_t)(b | (4 << 4) | (b << 8) | (4 << 12)));
            uint32_t v2;
            asm("lop3.b32 %0, %1, 0x00F0000F, 0x64006400, 0xEA;" : "=r"(v2) : "r"(t));
            v2 = hfma2(v2, 0x2C003C00u, 0xD400E400u);   // * (1, 1/16) + (-1024, -64)
            o[b] = hfma2(v2, s2, m2);                   // c * s + min, one rounding
        }
    } else if constexpr (XB) {
        (void)m2;
        uint32_t h[4];
        e2m1x8_to_f16x2x4(word, h);
#pragma unroll
        for (int b = 0; b < 4; ++b)                     // exact in bf16 (s2: see
            o[b] = bmul2(f16x2_to_bf16x2_scaled(h[b]), s2);   // e4m3_to_bf16x2_scaled)
    } else {
        (void)m2;
        uint32_t h[4];
        e2m1x8_to_f16x2x4(word, h);
#pragma unroll
        for (int b = 0; b < 4; ++b)
            o[b] = hmul2(h[b], s2);                     // exact in fp16
    }
}

// Split-K sum of one tile by its last-arriving CTA: y[m0 + c][n0 + 4q .. + 3] is
// the sum over k of the KS partials (k < KS <= KSM), added in k order, so the
// result does not depend on timing.  Work unit g4 = 32 c + q (four rows of one
// token column); a thread takes 16 / KSM units per round and requests all their
// partials (16-byte loads) before any add, so one round trip covers them.
template <int KSM>
__device__ __forceinline__ void tc_splitk_sum(const TcParams &p, const float4 *part, int n0, int m0,
                                              int t0, int nthreads)
{
    constexpr int GU = 16 / KSM;
    const int TN = p.TN, KS = p.KS;
    const int total = TN * (TC_ROWS / 4);
    const size_t kstride4 = (size_t)TN * TC_ROWS / 4;
    for (int base = t0; base < total; base += GU * nthreads) {
        float4 v[GU][KSM];
#pragma unroll
        for (int g = 0; g < GU; ++g) {
            const int g4 = base + g * nthreads;
#pragma unroll
            for (int k = 0; k < KSM; ++k)
                v[g][k] = (g4 < total && k < KS) ? __ldcg(part + k * kstride4 + g4)
                                                 : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int g = 0; g < GU; ++g) {
            const int g4 = base + g * nthreads;
            if (g4 >= total)
                continue;
            float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int k = 0; k < KSM; ++k)
                if (k < KS) {
                    sum.x += v[g][k].x; sum.y += v[g][k].y;
                    sum.z += v[g][k].z; sum.w += v[g][k].w;
                }
            const int c = g4 / (TC_ROWS / 4), q = g4 % (TC_ROWS / 4);
            const int m = m0 + c;
            const int nb = n0 + 4 * q;
            if (m < p.M) {
                uint16_t *yr = p.y + (int64_t)m * p.N;
                const float o[4] = {sum.x, sum.y, sum.z, sum.w};
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (nb + i < p.N)
                        yr[nb + i] = f32_to_bf16_bits(o[i]);
            }
        }
    }
}

// Epilogue of both tensor-core kernels, run by the 16 worker warps (w = 0..15)
// once the final MMA commit has been seen (ok): read the accumulator back from
// TMEM (warp w reads lane quadrant (w + 2) % 4, a quarter of its columns),
// release warp 1 to free TMEM after the last read, then store bf16 y -- or, under
// split-K, fp32 partials that the last CTA of the tile to arrive sums in k order.
template <int LAYOUT, bool SPLITK>
__device__ __forceinline__ void tc_epilogue(const TcParams &p, uint32_t tmem_base, bool ok, int w,
                                            int lane, int n0, int m0, int tile, int ks,
                                            const float *xdn, unsigned *last_flag, bool free_tmem,
                                            float gmul)
{
    const int TN = p.TN;
    const int quad = (w + 2) & 3;            // TMEM lane quadrant of this warp
    const int grp = w >> 2;                  // column share of the quadrant
    const int r = quad * 32 + lane;          // TMEM lane = weight row within the tile
    const int n = n0 + r;
    const bool nok = n < p.N;
    float gsc = 1.f;
    if constexpr (LAYOUT == 1)
        gsc = __ldg(p.gscale) * gmul;      // gmul: a power of two, exact
    const int ncb = (TN + 16 * TC_GROUPS - 1) / (16 * TC_GROUPS);   // same for every worker
    for (int it = 0; it < ncb; ++it) {
        const int cb = grp * 16 + it * 16 * TC_GROUPS;
        uint32_t v[16];
        if (cb < TN)
            tmem_ld16(tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)cb, v);
        if (free_tmem && it == ncb - 1) {
            // last TMEM read done: let warp 1 free the accumulator now
            tc_fence_before();
            asm volatile("bar.arrive 3, %0;" ::"r"((TC_WORKERS + 1) * 32) : "memory");
        }
        if (!ok || cb >= TN)
            continue;
        // token m's sums times the global scale, then 2^-e_m (exact), undoing the
        // prescale of its x.  In this order an intermediate overflows only where
        // the result itself does (2^-e_m reaches 2^113 for the largest tokens).
        if (!SPLITK || p.KS == 1) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int m = m0 + cb + j;
                if (nok && m < p.M)
                    p.y[(int64_t)m * p.N + n] =
                        f32_to_bf16_bits((__uint_as_float(v[j]) * gsc) * xdn[cb + j]);
            }
        } else {
            float *dst = p.ws + ((size_t)(tile * p.KS + ks) * TN + cb) * TC_ROWS + r;
#pragma unroll
            for (int j = 0; j < 16; ++j)
                dst[(size_t)j * TC_ROWS] = (__uint_as_float(v[j]) * gsc) * xdn[cb + j];
        }
    }
    if (SPLITK && p.KS > 1) {
        // split-K: the last CTA of this tile to arrive sums the partials (every
        // worker reaches both barriers, whatever happened before).  Every CTA
        // takes its ticket, also one whose wait timed out, so the counter always
        // reaches KS and the last arriver resets it for the next call; a CTA
        // without a valid partial adds a failure mark (bit 16 up), and then the
        // last arriver stores nothing (the timeout bit of the error word is set).
        __threadfence();
        asm volatile("bar.sync 2, %0;" ::"r"(TC_WORKERS * 32) : "memory");
        if (w == 0 && lane == 0) {
            const unsigned old = atomicAdd(&p.tickets[tile], ok ? 1u : 0x10001u);
            const bool last = (old & 0xffffu) == (unsigned)(p.KS - 1);
            const bool failed = !ok || (old >> 16) != 0u;
            *last_flag = last ? (failed ? 2u : 1u) : 0u;
        }
        asm volatile("bar.sync 2, %0;" ::"r"(TC_WORKERS * 32) : "memory");
        if (*last_flag == 1u) {
            __threadfence();
            const float4 *part = reinterpret_cast<const float4 *>(
                p.ws + (size_t)tile * p.KS * TN * TC_ROWS);
            if (p.KS <= 2)
                tc_splitk_sum<2>(p, part, n0, m0, w * 32 + lane, TC_WORKERS * 32);
            else if (p.KS <= 4)
                tc_splitk_sum<4>(p, part, n0, m0, w * 32 + lane, TC_WORKERS * 32);
            else
                tc_splitk_sum<8>(p, part, n0, m0, w * 32 + lane, TC_WORKERS * 32);
        }
        if (*last_flag != 0u && w == 0 && lane == 0)
            p.tickets[tile] = 0u;
    }
}

// ------------------------------------------------------------------ kernel
// One ring stage holds SC consecutive 64-column chunks ("super-chunk"): the packed
// codes of the tile's 128 rows (one TMA box, SC * 32 bytes per row), the SC x
// sub-tiles (TN x 64, 128-byte swizzle) and the SC A sub-tiles (128 x 64 fp16,
// 128-byte swizzle).  One barrier says the stage's copies landed, one that all
// sixteen worker warps wrote its A tiles, one that the MMAs reading it finished.
template <int SC>
struct TcStage {
    static constexpr uint32_t A = SC * 16384u;          // A sub-tiles
    static constexpr uint32_t CODE = SC * 4096u;        // 128 rows x SC * 32 bytes
};

// ATM (tiles of more than 64 tokens, one chunk per stage; NVFP4 tiles of at most
// 64 tokens, two): the dequantised A sub-tiles go to tensor memory instead of
// shared memory.  A stage then holds only the x sub-tiles and the codes, so more
// stages fit (more copies in flight), the A tiles cost no shared-memory
// bandwidth, and an MMA reading A from TMEM is shorter at N = 256 (138 against
// 171 cycles, measured alone).  TMEM: accumulator in columns 0 .. TN - 1, chunk c
// of ring stage s in columns a0 + 32 (SC s + c) .. + 31 (a0 = p.tmem_a0, TN
// rounded up to 32).
//
// RT = 2 (prefill tiles of 256 tokens): a CTA owns two 128-row weight tiles and
// issues both tiles' MMAs against each x sub-tile it loads, into two TMEM
// accumulators (columns 0 .. 255 and 256 .. 511), so each token tile is read from
// L2 half as often; the stage then holds both A sub-tiles and a 256-row code box.
//
// XB (NVFP4): the MMA takes bf16 operands.  x then goes to the tensor cores
// exactly as the caller stored it (no scan, no conversion, no prescale), and the
// weights are dequantised to bf16 as E2M1 * e4m3 * 2^eg, which is exact (at most
// 6 significant bits; see nvfp4_bf16_exponent).
template <int LAYOUT, int SC, int G, bool ATM, int RT, bool XB = false>   // LAYOUT 0 int4-g128, 1 NVFP4; G worker groups
__global__ void __launch_bounds__(TC_THREADS, 1)
q4_tc_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap,
             TcParams p)
{
    static_assert(!ATM || SC <= 4, "A in tensor memory: one, two or four chunks per stage");
    static_assert(RT == 1 || (RT == 2 && SC == 1 && !ATM), "two row tiles: one chunk per stage, A in shared memory");
    static_assert(!XB || LAYOUT == 1, "bf16 operands: NVFP4 only");
    constexpr uint32_t A_BYTES = (uint32_t)RT * TcStage<SC>::A;
    constexpr uint32_t CODE_BYTES = (uint32_t)RT * TcStage<SC>::CODE;
    constexpr uint32_t OFF_X = ATM ? 0u : A_BYTES;          // x sub-tiles in a stage
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ float s_xup[256], s_xdn[256];    // per-token 2^e_m and 2^-e_m (TN <= 256)
    const int TN = p.TN;
    const int NS = p.ns;
    const uint32_t x_bytes = (uint32_t)TN * 128;
    const uint32_t x_stride = (x_bytes + 1023) & ~1023u;
    const uint32_t stage_bytes = OFF_X + (uint32_t)SC * x_stride + CODE_BYTES;
    // stage u: [A sub-tiles][x sub-tiles][codes]; barriers after the stages
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (size_t)NS * stage_bytes);
    // bars: full[NS], afull[NS], empty[NS], done
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 3 * NS + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int tiles_mk = p.tiles_m * p.KS;
    const int tile_n = blockIdx.x / tiles_mk;
    const int rem = blockIdx.x - tile_n * tiles_mk;
    const int tile_m = rem / p.KS;
    const int ks = rem - tile_m * p.KS;
    const int n0 = tile_n * TC_ROWS * RT;
    const int m0 = tile_m * TN;
    // split-K on super-chunk boundaries
    const int sup_total = (p.chunks + SC - 1) / SC;
    const int u0 = (int)((int64_t)ks * sup_total / p.KS);
    const int u1 = (int)((int64_t)(ks + 1) * sup_total / p.KS);
    const int nsup = u1 - u0;
    const int c0 = u0 * SC;
    const int c1 = (u1 * SC) < p.chunks ? u1 * SC : p.chunks;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(smem_u32(&bars[i]), 1);                  // TMA arrive + bytes
            mbar_init(smem_u32(&bars[NS + i]), TC_WORKERS / G);   // the stage's worker group
            mbar_init(smem_u32(&bars[2 * NS + i]), 1);         // MMA commit
        }
        mbar_init(smem_u32(&bars[3 * NS]), 1);                 // final commit
        mbar_init_fence();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(tmem_slot)), "r"(p.tmem_cols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        pdl_launch_dependents();
        if (lane == 0) {
            int issued = 0;
            for (int u = 0; u < nsup; ++u) {
                const int s = u % NS, use = u / NS;
                if (use > 0 && !mbar_wait(smem_u32(&bars[2 * NS + s]), (use - 1) & 1, p.err))
                    break;
                const int kc = c0 + u * SC;
                const int nv = (c1 - kc) < SC ? (c1 - kc) : SC;
                unsigned char *st = smem + (size_t)s * stage_bytes;
                const uint32_t full = smem_u32(&bars[s]);
                mbar_arrive_expect_tx(full, CODE_BYTES + (uint32_t)nv * x_bytes);
                // codes of the super-chunk: 128 RT rows x SC * 32 bytes in one copy
                tma_load_2d(smem_u32(st + OFF_X + SC * x_stride), &wmap, kc * (TC_KC / 2),
                            n0, full);
                if (u == 0)
                    pdl_wait();                // x comes from the previous kernel
                for (int c = 0; c < nv; ++c)
                    tma_load_2d(smem_u32(st + OFF_X + c * x_stride), &xmap, (kc + c) * TC_KC,
                                m0, full);
                issued = u + 1;
            }
            // drain: every issued copy has landed before the CTA can exit
            for (int u = issued - NS > 0 ? issued - NS : 0; u < issued; ++u)
                mbar_wait(smem_u32(&bars[u % NS]), (u / NS) & 1, p.err);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------- MMA issue
        if (lane == 0) {
            const uint32_t idesc = idesc_f16(TN, XB);
            for (int u = 0; u < nsup; ++u) {
                const int s = u % NS, use = u / NS;
                if (!mbar_wait(smem_u32(&bars[NS + s]), use & 1, p.err))
                    break;
                tc_fence_after();
                const int kc = c0 + u * SC;
                const int nv = (c1 - kc) < SC ? (c1 - kc) : SC;
                const uint32_t st = smem_u32(smem + (size_t)s * stage_bytes);
                const uint64_t ad = smem_desc_sw128(st);
                const uint64_t bd = smem_desc_sw128(st + OFF_X);
                const uint32_t alo = (uint32_t)ad, ahi = (uint32_t)(ad >> 32);
                const uint32_t blo = (uint32_t)bd, bhi = (uint32_t)(bd >> 32);
                if constexpr (ATM) {
                    (void)alo;
                    (void)ahi;
                    // chunk c of stage s: A in columns a0 + 32 (SC s + c) .. + 31
                    const uint32_t a = tmem_base + (uint32_t)p.tmem_a0 + 32u * (uint32_t)(SC * s);
#pragma unroll
                    for (int c = 0; c < SC; ++c) {
                        if (c >= nv)
                            break;
#pragma unroll
                        for (int kk = 0; kk < TC_KC / 16; ++kk)
                            mma_f16_tmem_a(tmem_base, a + 32u * (uint32_t)c + 8u * kk,
                                           blo + (uint32_t)c * (x_stride >> 4) + 2u * kk, bhi, idesc,
                                           (u > 0 || c > 0 || kk > 0) ? 1u : 0u);
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < SC; ++c) {
                        if (c >= nv)
                            break;
#pragma unroll
                        for (int kk = 0; kk < TC_KC / 16; ++kk)
#pragma unroll
                            for (int rt = 0; rt < RT; ++rt)     // row tile rt: A at + 16 KB rt
                                mma_f16_2(tmem_base + 256u * (uint32_t)rt,
                                          alo + (uint32_t)(c * RT + rt) * 1024u + 2u * kk, ahi,
                                          blo + (uint32_t)c * (x_stride >> 4) + 2u * kk, bhi, idesc,
                                          (u > 0 || c > 0 || kk > 0) ? 1u : 0u);
                    }
                }
                mma_commit(smem_u32(&bars[2 * NS + s]));
            }
            mma_commit(smem_u32(&bars[3 * NS]));
        }
        // free the accumulator as soon as every worker has read it back
        __syncwarp();
        asm volatile("bar.sync 3, %0;" ::"r"((TC_WORKERS + 1) * 32) : "memory");
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                     ::"r"(tmem_base), "r"(p.tmem_cols) : "memory");
    } else {
        // ------------------------------------------------------------- workers
        const int w = warp - 2;                  // 0..15
        // Per-token prescale of x (see x_prescale_exponent): tiles converted here
        // take 2^e_m from the largest |x| of token m over this CTA's K range (one
        // warp per token reads that range from global memory while the first
        // stage's copies are in flight); x converted by the pre-pass brings its
        // 2^-e_m along.  The epilogue multiplies token m's sums by 2^-e_m.
        auto prescale = [&]() {
            if constexpr (XB) {
                // bf16 x goes to the MMA unscaled; the workers never read x
                for (int t = w * 32 + lane; t < TN; t += TC_WORKERS * 32)
                    s_xdn[t] = 1.f;
                asm volatile("bar.sync 2, %0;" ::"r"(TC_WORKERS * 32) : "memory");
                return;
            }
            pdl_wait();                              // x comes from the previous kernel
            if (!p.x_f16) {
                // eight consecutive threads per token (TN <= 64 here), four 16-byte
                // loads in flight each (the scale registers above are live), then a
                // max over the eight
                const int nvec = (c1 - c0) * (TC_KC / 8);
                const int t = (w * 32 + lane) >> 3;
                uint32_t mb = 0u;
                if (t < TN && m0 + t < p.M) {
                    const uint4 *row = reinterpret_cast<const uint4 *>(
                        p.x + (int64_t)(m0 + t) * p.K + (int64_t)c0 * TC_KC);
                    int j = lane & 7;
                    for (; j + 24 < nvec; j += 32) {
                        uint4 v[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            v[u] = __ldcg(row + j + 8 * u);
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            mb = bf16x8_absmax_bits(v[u], mb);
                    }
                    for (; j < nvec; j += 8)
                        mb = bf16x8_absmax_bits(__ldcg(row + j), mb);
                }
#pragma unroll
                for (int o = 4; o >= 1; o >>= 1) {
                    const uint32_t u2 = __shfl_xor_sync(0xffffffffu, mb, o);
                    mb = u2 > mb ? u2 : mb;
                }
                if ((lane & 7) == 0 && t < TN) {
                    const int e = x_prescale_exponent(mb);
                    s_xup[t] = pow2f_tc(e);
                    s_xdn[t] = pow2f_tc(-e);
                }
            } else {
                for (int t = w * 32 + lane; t < TN; t += TC_WORKERS * 32)
                    s_xdn[t] = m0 + t < p.M ? p.xdn[m0 + t] : 1.f;
            }
            asm volatile("bar.sync 2, %0;" ::"r"(TC_WORKERS * 32) : "memory");
        };
        if constexpr (ATM) {
            // G groups of WG = 16 / G warps take the stages in turn.  A warp may
            // write only TMEM lane quadrant warp % 4, so it owns rows 32 (warp % 4) +
            // lane; the WG / 4 warps of a group in one quadrant split the stage's
            // 64 SC columns (h = 0, 1: CPT = 32 SC columns from CPT h, i.e. half a
            // chunk for SC = 1 and chunk h for SC = 2).  A thread reads its row's
            // 16 SC code bytes, dequantises CPT weights and writes them as 16 SC
            // packed columns of its lane.
            static_assert(TC_WORKERS / G == 8, "two warps per quadrant and group");
            constexpr int SA = 4;                    // stages of scales loaded ahead
            constexpr int CPT = 32 * SC;             // columns per thread and stage
            const int gi = w / 8;
            const int h = (w % 8) / 4;
            const int quad = warp & 3;
            const int row = quad * 32 + lane;
            const int64_t n = n0 + row;
            const bool rok = n < p.N;
            const uint32_t t_lane = (uint32_t)(quad * 32) << 16;
            // int4: scale | min << 16 of the row's group; NVFP4: the e4m3 scales of
            // the thread's 2 SC 16-column groups (low byte first)
            auto load_scale = [&](int u) -> uint64_t {
                const int col = (c0 + u * SC) * TC_KC + CPT * h;   // first column
                if (u >= nsup || !rok || col / TC_KC >= c1)
                    return 0u;
                if constexpr (LAYOUT == 0) {
                    const int64_t g2 = n * (p.K / 128) + col / 128;
                    return ld_nc_u16(static_cast<const uint16_t *>(p.scale) + g2) |
                           (ld_nc_u16(p.minv + g2) << 16);
                } else {
                    const uint8_t *sp = static_cast<const uint8_t *>(p.scale) + n * (p.K / 16) + col / 16;
                    if constexpr (SC == 1)
                        return ld_nc_u16(sp);
                    else if constexpr (SC == 2)
                        return ld_nc_u32(sp);
                    else {                             // 4-byte aligned only
                        const uint64_t lo = ld_nc_u32(sp);
                        // the second chunk of the pair may lie past the row's end
                        return (col / TC_KC + 1 < c1) ? lo | ((uint64_t)ld_nc_u32(sp + 4) << 32) : lo;
                    }
                }
            };
            float bf16_up = 1.f;               // XB: see e4m3_to_bf16x2_scaled
            if constexpr (XB)
                bf16_up = pow2f_tc(112 + nvfp4_bf16_exponent(__ldg(p.gscale)));
            uint64_t scq[SA];
#pragma unroll
            for (int j = 0; j < SA; ++j)
                scq[j] = load_scale(gi + j * G);
            prescale();
            auto stage = [&](int u, uint64_t sc) -> bool {
                const int st_i = u % NS, use = u / NS;
                const unsigned char *st = smem + (size_t)st_i * stage_bytes;
                if (!mbar_wait_warp(smem_u32(&bars[st_i]), use & 1, p.err))
                    return false;
                // The slot's previous A was read by MMAs whose commit the producer
                // waited for before requesting this use's copies.
                tc_fence_after();
                const unsigned char *crow = st + SC * x_stride + row * (32 * SC) + h * (16 * SC);
                uint32_t m2 = 0u;
                if constexpr (LAYOUT == 0)
                    m2 = f16x2_splat((uint32_t)(sc >> 16) & 0xffffu);
#pragma unroll
                for (int i = 0; i < SC; ++i) {         // 32 columns: 16 packed TMEM columns
                    const uint4 cw = *reinterpret_cast<const uint4 *>(crow + 16 * i);
                    const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
                    uint32_t v[16];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint32_t s2;
                        if constexpr (LAYOUT == 0) {
                            s2 = f16x2_splat((uint32_t)sc & 0xffffu);
                        } else {
                            // 16-column group (2 i + j / 2) of the thread's columns
                            const uint32_t b = (uint32_t)(sc >> (8 * (2 * i + j / 2))) & 0xffu;
                            s2 = XB ? e4m3_to_bf16x2_scaled(b, bf16_up)
                                    : f16x2_splat(e4m3x2_to_f16x2(b) & 0xffffu);
                        }
                        uint32_t o[4];
                        tc_dequant_word<LAYOUT, XB>(words[j], s2, m2, o);
#pragma unroll
                        for (int b = 0; b < 4; ++b)
                            v[4 * j + b] = o[b];
                    }
                    tmem_st16(tmem_base + t_lane + (uint32_t)p.tmem_a0 + (uint32_t)(32 * SC) * (uint32_t)st_i +
                                  (uint32_t)(16 * SC) * (uint32_t)h + 16u * (uint32_t)i,
                              v);
                }
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(smem_u32(&bars[NS + st_i]));
                return true;
            };
            bool alive = true;
            for (int u0 = gi; u0 < nsup && alive; u0 += SA * G) {
#pragma unroll
                for (int j = 0; j < SA; ++j) {
                    const int u = u0 + j * G;
                    if (alive && u < nsup)
                        alive = stage(u, scq[j]);
                    scq[j] = load_scale(u + SA * G);
                }
            }
        } else {
            // G groups of WG = 16 / G warps take the stages in turn (group gi the
            // stages gi, gi + G, ...), so G stages are dequantised at once.
            // Dequant mapping inside a group: a warp reads 256 contiguous code bytes
            // per step (no bank conflicts): L = 4 SC lanes per code row, 32 / L rows per
            // step, STEPS = SC * G * RT steps.  In step k a lane takes 16 weights: row
            // (128 RT / WG) wg + (32 / L) k + lane / L, chunk c = (lane % L) / 4,
            // columns 16 (lane % 4) .. + 15 of that chunk (rows 128 .. 255 are the
            // second row tile, whose A sub-tile follows the first's).
            constexpr int WG = TC_WORKERS / G;
            constexpr int L = 4 * SC;
            constexpr int RPS = 32 / L;
            constexpr int STEPS = SC * G * RT;
            constexpr int SA = 4;                    // stages of scales loaded ahead
            const int gi = w / WG;                   // worker group
            const int wg = w % WG;                   // warp within the group
            const int wt = wg * 32 + lane;           // thread within the group
            const int cl = lane % L;
            const int c = cl >> 2;
            const int qd = cl & 3;
            int rowk[STEPS];
            bool rok[STEPS];
#pragma unroll
            for (int k = 0; k < STEPS; ++k) {
                rowk[k] = (128 * RT / WG) * wg + RPS * k + lane / L;
                rok[k] = n0 + rowk[k] < p.N;
            }
            // Group scales (int4: fp16 scale and min, loaded apart and combined only
            // where used; NVFP4: the e4m3 byte) run SA stages ahead in SA register
            // sets, each refilled right after its stage: no register moves, so no
            // wait on a load still in flight.
            auto load_scale = [&](int u, int k, const void *base) -> uint32_t {
                const int kc = c0 + u * SC + c;
                if (u >= nsup || !rok[k] || kc >= c1)
                    return 0u;
                const int64_t n = n0 + rowk[k];
                if constexpr (LAYOUT == 0)
                    return ld_nc_u16(static_cast<const uint16_t *>(base) + n * (p.K / 128) + (kc * TC_KC) / 128);
                else
                    return ld_nc_u8(static_cast<const uint8_t *>(base) + n * (p.K / 16) + kc * 4 + qd);
            };
            // XB: e4m3 scales become bf16 scale * 2^(112 + eg) (see e4m3_to_bf16x2_scaled)
            float bf16_up = 1.f;
            if constexpr (XB)
                bf16_up = pow2f_tc(112 + nvfp4_bf16_exponent(__ldg(p.gscale)));
            uint32_t scq[SA][STEPS], mnq[SA][STEPS];
#pragma unroll
            for (int j = 0; j < SA; ++j)
#pragma unroll
                for (int k = 0; k < STEPS; ++k) {
                    scq[j][k] = load_scale(gi + j * G, k, p.scale);
                    mnq[j][k] = LAYOUT == 0 ? load_scale(gi + j * G, k, p.minv) : 0u;
                }
            prescale();
            // one stage; false when a wait timed out
            auto stage = [&](int u, const uint32_t (&scs)[STEPS], const uint32_t (&mns)[STEPS]) -> bool {
                const int st_i = u % NS, use = u / NS;
                const int kc = c0 + u * SC;
                const int nv = (c1 - kc) < SC ? (c1 - kc) : SC;
                unsigned char *st = smem + (size_t)st_i * stage_bytes;
                if (!mbar_wait_warp(smem_u32(&bars[st_i]), use & 1, p.err))
                    return false;
                // x sub-tiles: bf16 -> prescaled fp16 in place (element-wise; a
                // 16-byte vector v holds 8 columns of token v / 8, whatever the
                // swizzle).  Only tiles of at most 64 tokens are converted here
                // (larger M arrive in fp16), so a thread has at most SC * G vectors:
                // the loop is unrolled and interleaves with the code loads below.
                if (!XB && !p.x_f16) {
                    const int per = TN * 8;                  // vectors per sub-tile
#pragma unroll
                    for (int j = 0; j < SC * G; ++j) {
                        const int v = wt + j * WG * 32;
                        if (v < nv * per) {
                            const int sub = (v >= per) + (v >= 2 * per) + (v >= 3 * per);
                            const int vv = v - sub * per;
                            uint4 *xv = reinterpret_cast<uint4 *>(st + OFF_X + sub * x_stride) + vv;
                            const float up = s_xup[vv >> 3];
                            const uint4 t = *xv;
                            const uint32_t e[4] = {t.x, t.y, t.z, t.w};
                            uint32_t o[4];
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                __half2 h = __floats2half2_rn(bf16_bits_to_f32(e[q] & 0xffffu) * up,
                                                              bf16_bits_to_f32(e[q] >> 16) * up);
                                o[q] = *reinterpret_cast<uint32_t *>(&h);
                            }
                            *xv = make_uint4(o[0], o[1], o[2], o[3]);
                        }
                    }
                }
                const unsigned char *codes = st + OFF_X + SC * x_stride;
#pragma unroll
                for (int k = 0; k < STEPS; ++k) {
                    const int rd = rowk[k];
                    const uint2 cw = *reinterpret_cast<const uint2 *>(codes + rd * (SC * 32) + cl * 8);
                    const uint32_t words[2] = {cw.x, cw.y};
                    unsigned char *arow = st + c * 16384 + rd * 128;
                    uint32_t sg = 0u;
                    if constexpr (XB)
                        sg = e4m3_to_bf16x2_scaled(scs[k], bf16_up);
                    else if constexpr (LAYOUT == 1)
                        sg = f16x2_splat(e4m3x2_to_f16x2(scs[k] & 0xffu) & 0xffffu);
#pragma unroll
                    for (int j = 0; j < 2; ++j) {           // 8 K columns per 16-byte chunk
                        uint32_t o[4];
                        if constexpr (LAYOUT == 0) {
                            const uint32_t s2 = f16x2_splat(scs[k]);
                            const uint32_t m2 = f16x2_splat(mns[k]);
#pragma unroll
                            for (int b = 0; b < 4; ++b) {
                                // byte b -> (1024 + c_lo, 1024 + 16 c_hi) -> (c_lo, c_hi)
                                const uint32_t t = prmt(words[j], 0u, (uint32_t)(b | (4 << 4) | (b << 8) | (4 << 12)));
                                uint32_t v2;
                                asm("lop3.b32 %0, %1, 0x00F0000F, 0x64006400, 0xEA;" : "=r"(v2) : "r"(t));
                                v2 = hfma2(v2, 0x2C003C00u, 0xD400E400u);   // * (1, 1/16) + (-1024, -64)
                                o[b] = hfma2(v2, s2, m2);                   // c * s + min, one rounding
                            }
                        } else if constexpr (XB) {
                            uint32_t h[4];
                            e2m1x8_to_f16x2x4(words[j], h);
#pragma unroll
                            for (int b = 0; b < 4; ++b)                    // exact in bf16
                                o[b] = bmul2(f16x2_to_bf16x2_scaled(h[b]), sg);
                        } else {
                            uint32_t h[4];
                            e2m1x8_to_f16x2x4(words[j], h);
#pragma unroll
                            for (int b = 0; b < 4; ++b)
                                o[b] = hmul2(h[b], sg);                    // exact in fp16
                        }
                        const int seg = 2 * qd + j;
                        *reinterpret_cast<uint4 *>(arow + ((seg ^ (rd & 7)) << 4)) =
                            make_uint4(o[0], o[1], o[2], o[3]);
                    }
                }
                fence_proxy_async();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(smem_u32(&bars[NS + st_i]));
                return true;
            };
            bool alive = true;
            for (int u0 = gi; u0 < nsup && alive; u0 += SA * G) {
#pragma unroll
                for (int j = 0; j < SA; ++j) {
                    const int u = u0 + j * G;
                    if (alive && u < nsup)
                        alive = stage(u, scq[j], mnq[j]);
#pragma unroll
                    for (int k = 0; k < STEPS; ++k) {
                        scq[j][k] = load_scale(u + SA * G, k, p.scale);
                        if constexpr (LAYOUT == 0)
                            mnq[j][k] = load_scale(u + SA * G, k, p.minv);
                    }
                }
            }
        }

        // ------------------------------------------------------------ epilogue
        const bool ok = nsup > 0 && mbar_wait_warp(smem_u32(&bars[3 * NS]), 0, p.err);
        tc_fence_after();
        __shared__ unsigned last_flag;
        float gmul = 1.f;
        if constexpr (XB)
            gmul = pow2f_tc(-nvfp4_bf16_exponent(__ldg(p.gscale)));
#pragma unroll
        for (int rt = 0; rt < RT; ++rt)
            tc_epilogue<LAYOUT, RT == 1>(p, tmem_base + 256u * (uint32_t)rt, ok, w, lane, n0 + TC_ROWS * rt, m0,
                                (tile_n * RT + rt) * p.tiles_m + tile_m, ks, s_xdn, &last_flag,
                                rt == RT - 1, gmul);
    }

    __syncthreads();
}

// x (bf16) -> prescaled fp16 once per call for large M, so that the GEMM's CTAs
// do not each convert the same token tiles: one 256-thread block per token holds
// the row in registers (up to XP_V 16-byte vectors per thread, K <= 16384; longer
// rows are read a second time), reduces its maximum through shared memory, then
// converts and writes the row and 2^-e_m to xdn[m] for the GEMM's epilogue.
constexpr int XP_THREADS = 256;
constexpr int XP_V = 8;

__global__ void __launch_bounds__(XP_THREADS) q4_x_to_f16_kernel(const uint16_t *__restrict__ x,
                                                                 uint16_t *__restrict__ out,
                                                                 float *__restrict__ xdn, int M, int K)
{
    __shared__ uint32_t s_max[XP_THREADS / 32];
    pdl_launch_dependents();
    pdl_wait();
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int nvec = K / 8;
    for (int m = blockIdx.x; m < M; m += gridDim.x) {
        const uint4 *row = reinterpret_cast<const uint4 *>(x + (int64_t)m * K);
        uint4 v[XP_V];
        uint32_t mb = 0u;
#pragma unroll
        for (int u = 0; u < XP_V; ++u) {
            const int i = t + u * XP_THREADS;
            v[u] = i < nvec ? __ldcg(row + i) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < XP_V; ++u)
            mb = bf16x8_absmax_bits(v[u], mb);
        for (int i = t + XP_V * XP_THREADS; i < nvec; i += XP_THREADS)
            mb = bf16x8_absmax_bits(__ldcg(row + i), mb);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            const uint32_t u2 = __shfl_xor_sync(0xffffffffu, mb, o);
            mb = u2 > mb ? u2 : mb;
        }
        if (lane == 0)
            s_max[warp] = mb;
        __syncthreads();
        mb = 0u;
#pragma unroll
        for (int w = 0; w < XP_THREADS / 32; ++w)
            mb = s_max[w] > mb ? s_max[w] : mb;
        __syncthreads();                        // s_max is rewritten for the next row
        const int e = x_prescale_exponent(mb);
        const float up = pow2f_tc(e);
        auto conv = [up](uint4 q) {
            const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
            uint32_t o[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                __half2 h = __floats2half2_rn(bf16_bits_to_f32(w4[j] & 0xffffu) * up,
                                              bf16_bits_to_f32(w4[j] >> 16) * up);
                o[j] = *reinterpret_cast<uint32_t *>(&h);
            }
            return make_uint4(o[0], o[1], o[2], o[3]);
        };
        uint4 *dst = reinterpret_cast<uint4 *>(out + (int64_t)m * K);
#pragma unroll
        for (int u = 0; u < XP_V; ++u) {
            const int i = t + u * XP_THREADS;
            if (i < nvec)
                dst[i] = conv(v[u]);
        }
        for (int i = t + XP_V * XP_THREADS; i < nvec; i += XP_THREADS)
            dst[i] = conv(__ldcg(row + i));
        if (t == 0)
            xdn[m] = pow2f_tc(-e);
    }
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

bool tc_eligible(int kind, int M, int N, int K)
{
    (void)M;
    (void)N;
    if (K % TC_KC)
        return false;
    return kind == W_INT4 || kind == W_NVFP4_A16;
}

// Tiles of more than 64 tokens: int4 x is converted by a separate pass (up to 64
// tokens, inside the GEMM: at most SC vectors per thread), and the dequantised A
// sub-tiles live in tensor memory, except in CTAs that own two weight-row tiles
// (two accumulators fill the tensor memory).
static bool tc_preconvert(int M) { return M > 64; }

// Chunks per stage of the NVFP4 tiles of at most 64 tokens (A in tensor memory).
constexpr int kTcSkinnySc = 4;

// CTA tile: TN tokens (MMA N) x RT weight-row tiles of 128.  Each x sub-tile a
// CTA loads feeds RT tiles' MMAs, so for prefill (more than 256 tokens) the CTA
// takes two row tiles where that still gives over half a wave of CTAs without
// split-K.  Measured at M = 2048 (int4): 2048 -> 8192 72 against 94 us with one
// row tile and A in shared memory, 70 against 77 with one row tile and A in
// tensor memory; 8192 -> 2048 (64 CTAs of two row tiles) 95 with two-way split-K
// and 105 with 128-token tiles, against 77-79 with one row tile (59 with
// two-chunk tensor-memory stages).  Otherwise one row tile and TN = M rounded up
// to 16 (at most 256); long token ranges then refit TN to whole waves.
struct TcShape {
    int TN, RT;
};

// Long token ranges (M >= 1024) take the token-tile width from 256 down to 192
// that needs the fewest waves of CTAs per token of a tile (each CTA's time grows
// with its width): at M = 2048, 240-token tiles give 144 one-row-tile CTAs
// (8192 -> 2048) where 256 give 128, or 288 two-row-tile CTAs (2048 -> 8192), two
// full waves of 152 SMs, where 256 give 1.7.
static int tc_long_tn(int M, int64_t row_units, int sms)
{
    if (M < 1024)
        return 256;
    int best = 256;
    int64_t best_cost = -1;
    for (int tn = 256; tn >= 192; tn -= 16) {
        const int64_t ctas = row_units * ((M + tn - 1) / tn);
        const int64_t cost = (ctas + sms - 1) / sms * tn;
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = tn;
        }
    }
    return best;
}

static TcShape tc_shape(int M, int N, int sms)
{
    const int tn = M > 256 ? 256 : ((M + 15) / 16 * 16 < 16 ? 16 : (M + 15) / 16 * 16);
    const int64_t rows1 = (N + TC_ROWS - 1) / TC_ROWS;
    if (!tc_preconvert(M) || M < 256)
        return {M > 256 ? tc_long_tn(M, rows1, sms) : tn, 1};
    const int64_t pairs = (N + 2 * TC_ROWS - 1) / (2 * TC_ROWS);
    if (pairs * ((M + 255) / 256) * 2 > sms)
        return {tc_long_tn(M, pairs, sms), 2};
    return {tc_long_tn(M, rows1, sms), 1};
}

// Tiles of 128 weight rows x TN tokens (a CTA owns RT of them).
static int64_t tc_tiles(int M, int N, int sms)
{
    const TcShape sh = tc_shape(M, N, sms);
    return (int64_t)((N + TC_ROWS * sh.RT - 1) / (TC_ROWS * sh.RT)) * sh.RT * ((M + sh.TN - 1) / sh.TN);
}

// Split-K factor: as many CTAs as fit in one wave (one CTA per SM) when the tile
// grid is small, keeping at least four K chunks per CTA and at most eight
// partials per tile (the last CTA of a tile sums them; more would lengthen that
// tail more than the extra CTAs shorten the main loop).
static int tc_ks(const DeviceInfo &dev, int M, int N, int K)
{
    const int64_t tiles = tc_tiles(M, N, dev.sms) / tc_shape(M, N, dev.sms).RT;   // CTAs per K slice
    const int chunks = K / TC_KC;
    if (tiles * 2 > dev.sms)
        return 1;
    int ks = (int)(dev.sms / tiles);
    if (ks > chunks / 4)
        ks = chunks / 4;
    if (ks > 8)
        ks = 8;
    return ks < 1 ? 1 : ks;
}

// [fp16 x, prescaled per token][per-token 2^-e_m, fp32]
static size_t tc_xf16_data_bytes(int M, int K) { return ((size_t)M * K * 2 + 255) / 256 * 256; }

// NVFP4 calls take bf16 operands (exact dequantised weights, x as stored): no
// copy of x.
static bool tc_bf16_operands(int kind) { return kind == W_NVFP4_A16; }

static size_t tc_xf16_bytes(int kind, int M, int K)
{
    return tc_preconvert(M) && !tc_bf16_operands(kind)
               ? tc_xf16_data_bytes(M, K) + ((size_t)M * 4 + 255) / 256 * 256 : 0;
}

static size_t tc_split_bytes(int M, int N, int K, int sms)
{
    DeviceInfo d;
    d.sms = sms;
    const int ks = tc_ks(d, M, N, K);
    if (ks == 1)
        return 0;
    const int TN = tc_shape(M, N, sms).TN;
    const size_t tiles = (size_t)tc_tiles(M, N, sms);
    return (tiles * 4 + 255) / 256 * 256 + tiles * ks * TN * TC_ROWS * 4;
}

// Workspace layout: [fp16 copy of x and its per-token scales (large M)][split-K
// counters][partials].
size_t tc_workspace_bytes(int kind, int M, int N, int K, int sms)
{
    if (K % TC_KC || M < 1 || N < 1)
        return 0;
    return tc_xf16_bytes(kind, M, K) + tc_split_bytes(M, N, K, sms);
}

static CUresult tc_encode_maps(EncodeTiledFn enc, CUtensorMap &xmap, CUtensorMap &wmap,
                               const void *xsrc, bool x_f16, const uint8_t *codes, int M, int N,
                               int K, int TN, int code_box_bytes, int code_box_rows,
                               bool code_swizzle)
{
    cuuint64_t xd[2] = {(cuuint64_t)K, (cuuint64_t)M};
    cuuint64_t xstr[1] = {(cuuint64_t)K * 2};
    cuuint32_t xbox[2] = {TC_KC, (cuuint32_t)TN};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(&xmap, x_f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                     2, const_cast<void *>(xsrc), xd, xstr, xbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return r;
    cuuint64_t wd[2] = {(cuuint64_t)K / 2, (cuuint64_t)N};
    cuuint64_t wstr[1] = {(cuuint64_t)K / 2};
    cuuint32_t wbox[2] = {(cuuint32_t)code_box_bytes, (cuuint32_t)code_box_rows};
    return enc(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(codes), wd, wstr, wbox,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               code_swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

template <int LAYOUT>
static const void *tc_select_layout(int sc, bool atm, int rt, bool xb)
{
    if constexpr (LAYOUT == 1) {
        if (xb) {
            if (rt == 2)
                return reinterpret_cast<const void *>(&q4_tc_kernel<1, 1, 2, false, 2, true>);
            if (atm)
                return sc == 4 ? reinterpret_cast<const void *>(&q4_tc_kernel<1, 4, 2, true, 1, true>)
                     : sc == 2 ? reinterpret_cast<const void *>(&q4_tc_kernel<1, 2, 2, true, 1, true>)
                               : reinterpret_cast<const void *>(&q4_tc_kernel<1, 1, 2, true, 1, true>);
            return sc == 4 ? reinterpret_cast<const void *>(&q4_tc_kernel<1, 4, 2, false, 1, true>)
                 : sc == 2 ? reinterpret_cast<const void *>(&q4_tc_kernel<1, 2, 2, false, 1, true>)
                           : reinterpret_cast<const void *>(&q4_tc_kernel<1, 1, 2, false, 1, true>);
        }
    }
    if (rt == 2)
        return reinterpret_cast<const void *>(&q4_tc_kernel<LAYOUT, 1, 2, false, 2>);
    if (atm)
        return sc == 2 ? reinterpret_cast<const void *>(&q4_tc_kernel<LAYOUT, 2, 2, true, 1>)
                       : reinterpret_cast<const void *>(&q4_tc_kernel<LAYOUT, 1, 2, true, 1>);
    return sc == 4 ? reinterpret_cast<const void *>(&q4_tc_kernel<LAYOUT, 4, 2, false, 1>)
         : sc == 2 ? reinterpret_cast<const void *>(&q4_tc_kernel<LAYOUT, 2, 2, false, 1>)
                   : reinterpret_cast<const void *>(&q4_tc_kernel<LAYOUT, 1, 2, false, 1>);
}

static const void *tc_select(int kind, int sc, bool atm, int rt, bool xb)
{
    return kind == W_INT4 ? tc_select_layout<0>(sc, atm, rt, false)
                          : tc_select_layout<1>(sc, atm, rt, xb);
}

q4_status tc_launch(int kind, const void *x, const uint8_t *codes, const void *scale,
                    const void *minv, const float *gscale, void *y, int M, int N, int K,
                    void *ws, size_t ws_bytes, cudaStream_t stream, bool pdl)
{
    DeviceInfo dev;
    q4_status s = current_device(dev);
    if (s != Q4_OK)
        return s;
    EncodeTiledFn enc = encode_fn();
    if (!enc)
        return fail(Q4_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    TcParams p = {};
    p.x = static_cast<const uint16_t *>(x);
    p.codes = codes;
    p.scale = scale;
    p.minv = static_cast<const uint16_t *>(minv);
    p.gscale = gscale;
    p.y = static_cast<uint16_t *>(y);
    p.err = device_error_flags();
    p.M = M;
    p.N = N;
    p.K = K;
    const TcShape shape = tc_shape(M, N, dev.sms);
    p.TN = shape.TN;
    p.tiles_m = (M + p.TN - 1) / p.TN;
    p.KS = tc_ks(dev, M, N, K);
    p.chunks = K / TC_KC;
    int cols = 32;
    while (cols < p.TN)
        cols *= 2;
    p.tmem_cols = cols;
    const size_t need = tc_workspace_bytes(kind, M, N, K, dev.sms);
    if (need > ws_bytes)
        return fail(Q4_ERR_WORKSPACE, "tensor-core path needs %zu bytes of workspace", need);
    const int rt = shape.RT;
    if (rt == 2 && p.KS != 1)          // two-tile CTAs are only planned without split-K
        return fail(Q4_ERR_SHAPE, "tensor-core plan: split-K with two row tiles");
    const size_t tiles = (size_t)tc_tiles(M, N, dev.sms);     // 128-row tiles
    unsigned char *wsb = static_cast<unsigned char *>(ws);
    const size_t xf16 = tc_xf16_bytes(kind, M, K);
    if (p.KS > 1) {
        unsigned char *b = wsb + xf16;
        p.tickets = reinterpret_cast<unsigned *>(b);
        p.ws = reinterpret_cast<float *>(b + (tiles * 4 + 255) / 256 * 256);
    }
    const void *xsrc = x;
    p.x_f16 = 0;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    if (xf16 > 0) {
        int64_t blocks = M;                                   // one block per token
        if (blocks > (int64_t)dev.sms * 8)
            blocks = (int64_t)dev.sms * 8;
        cudaLaunchConfig_t pc = {};
        pc.gridDim = dim3((unsigned)blocks);
        pc.blockDim = dim3(XP_THREADS);
        pc.stream = stream;
        pc.attrs = pdl ? attr : nullptr;
        pc.numAttrs = pdl ? 1 : 0;
        const uint16_t *xin = static_cast<const uint16_t *>(x);
        uint16_t *xo = reinterpret_cast<uint16_t *>(wsb);
        float *xdn = reinterpret_cast<float *>(wsb + tc_xf16_data_bytes(M, K));
        int Mi = M, Ki = K;
        void *pargs[] = {&xin, &xo, &xdn, &Mi, &Ki};
        cudaError_t e0 = cudaLaunchKernelExC(&pc, reinterpret_cast<const void *>(&q4_x_to_f16_kernel),
                                             pargs);
        if (e0 != cudaSuccess)
            return cuda_fail(e0, "launch of the x conversion kernel");
        xsrc = wsb;
        p.x_f16 = 1;
        p.xdn = xdn;
    }
    // Stage = SC chunks (A sub-tiles, x sub-tiles, codes).  The largest SC that
    // still leaves four stages in flight (three, two) amortises each hand-off
    // over more weights without starving the copies.  One-row-tile CTAs of more
    // than 64 tokens, and NVFP4 CTAs of at most 64, keep the A sub-tiles in
    // tensor memory instead, with two chunks per stage where three stages fit
    // (each hand-off costs about as much as a stage's MMAs at 256 tokens: at
    // M = 2048, K = 8192 -> N = 2048, 59 / 49 us int4 / NVFP4 against 77 / 65
    // with one chunk per stage and six stages).
    const size_t x_stride = ((size_t)p.TN * 128 + 1023) / 1024 * 1024;
    const size_t budget = dev.smem_optin - 1024 /* alignment */ - 3072 /* static */ - 256;
    const bool xb = tc_bf16_operands(kind);
    // (A in tensor memory for int4 tiles of at most 64 tokens, whose x is
    // converted in the kernel, was slower: M = 48 step 31.4 against 27.9 us)
    const bool atm_skinny = xb && !tc_preconvert(M);
    const bool atm = rt == 1 && (tc_preconvert(M) || atm_skinny);
    // A in tensor memory: the A sub-tiles after the accumulator, SC 32-column
    // slots per stage
    p.tmem_a0 = (p.TN + 31) / 32 * 32;
    const size_t a_bytes = atm ? 0 : 16384 * (size_t)rt;
    const size_t code_bytes = 4096 * (size_t)rt;
    const int sc_max = atm ? (atm_skinny ? kTcSkinnySc : 2) : (rt == 2 ? 1 : 4);
    int sc = 1, ns = 0;
    for (int need_ns = atm ? 3 : 4; need_ns >= 2 && ns == 0; --need_ns)
        for (int cand = sc_max; cand >= 1; cand /= 2) {
            const size_t stage = (size_t)cand * (a_bytes + x_stride + code_bytes);
            const int fit = (int)(budget / stage);
            const int ns_cap = atm ? (512 - p.tmem_a0) / (32 * cand) : 8;
            if (fit >= need_ns && ns_cap >= need_ns) {
                sc = cand;
                ns = fit > ns_cap ? ns_cap : fit;
                break;
            }
        }
    if (ns < 2)
        return fail(Q4_ERR_SHAPE, "tensor-core tile does not fit in shared memory");
    p.ns = ns;
    if (atm || rt == 2)
        p.tmem_cols = 512;
    const size_t stage = (size_t)sc * (a_bytes + x_stride + code_bytes);
    const size_t smem = 1024 + (size_t)ns * stage + (3 * ns + 1) * 8 + 16;

    CUtensorMap xmap, wmap;
    {
        const CUresult r = tc_encode_maps(enc, xmap, wmap, xsrc, p.x_f16 != 0, codes, M, N, K, p.TN,
                                          sc * TC_KC / 2, TC_ROWS * rt, false);
        if (r != CUDA_SUCCESS)
            return fail(Q4_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    }
    // two worker groups, two stages dequantised at once (measured: prefill
    // GEMMs 5-22% faster than one group of 16 warps; batched decode unchanged)
    const void *k = tc_select(kind, sc, atm, rt, xb);
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaFuncSetAttribute(tensor-core kernel)");
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(tiles / rt * p.KS));
    cfg.blockDim = dim3(TC_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = pdl ? attr : nullptr;
    cfg.numAttrs = pdl ? 1 : 0;
    void *args[] = {&xmap, &wmap, &p};
    e = cudaLaunchKernelExC(&cfg, k, args);
    if (e != cudaSuccess)
        return cuda_fail(e, "launch of the tensor-core kernel");
    return Q4_OK;
}

}  // namespace q4
