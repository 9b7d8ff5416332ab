// One-token decode GEMV for sm_103a with bulk-copy weight stages: y[N] = x[K] W^T
// for both 4-bit layouts when K is a multiple of 2048 (every decode projection of
// the pages' 3B-class stack: q|k|v, o, gate|up with K = 2048, down with K = 8192).
//
// What it computes is the whole-row kernel's arithmetic (stream_common.cuh):
// "rumik-oss-1-int4", "Format": w = code * scale + min, summed exactly as
// integers c * x' against x staged as int16 fixed point, scale and min applied
// per lane in fp32; "VoxCPM2 NVFP4 (GPTQ)", "NVFP4 settings": w = E2M1 * e4m3 * g,
// E2M1 decoded by cvt.rn.f16x2.e2m1x2 and summed in fp16 eight products per half
// group against x prescaled per 32 columns, group scale and g in fp32.
//
// Data movement, built for chains of dependent calls (programmatic dependent
// launch, one CTA per SM and call, the next call's CTA resident beside it):
//   * A unit is 2048 columns of one row (1024 code bytes + its scales).  A stage
//     is 16 units = 16 / S whole rows (S = K / 2048): their codes and scales are
//     contiguous in memory, so one thread fills a stage with two or three
//     cp.async.bulk copies completing on one mbarrier.
//   * The CTA's rows are one contiguous block.  Weights do not depend on the
//     previous kernel, so the producer requests the first NS stages (about 108 KB,
//     most of a CTA's share of a 16384 x 2048 matrix) before griddepcontrol.wait
//     and the rest as consumers free stages.
//   * After the wait the 16 consumer warps stage x once in shared memory
//     (prescaled fp16 for NVFP4, int16 fixed point for int4, with per-chunk
//     factors), then each keeps its 64 columns per lane in 32 registers.  Warp w
//     takes unit w of every stage; a lane reads two 16-byte code vectors (columns
//     32l .. 32l + 31 and 1024 + 32l .. + 31 of the unit, conflict-free) and its
//     scale words.  A row is reduced across lanes (transposing butterfly over four
//     stages' rows at once) and, with S = 1, stored as bf16 by the warp itself;
//     with S > 1 the warp parks its partial and the last of the row's S warps to
//     arrive sums them in k order.  Results do not depend on timing.
// Every wait is bounded (mbar_wait): a timeout sets Q4_DEVERR_TIMEOUT and the
// kernel drains the copies it issued before leaving.
#include "q4_device.cuh"
#include "q4_internal.h"
#include "stream_common.cuh"

namespace q4 {

constexpr int GS_CWARPS = 16;                       // consumer warps = units per stage
constexpr int GS_THREADS = (GS_CWARPS + 1) * 32;    // + one producer warp
constexpr int GS_KSEG = 2048;                       // columns per unit
constexpr int GS_CODE = GS_KSEG / 2;                // code bytes per unit
constexpr int GS_RB = 4;                            // stages per cross-lane reduction

template <int WK>
struct GsUnit {
    // scale bytes per unit: NVFP4 e4m3 per 16 columns; int4 fp16 scale per 128
    // columns, and as many min bytes after them
    static constexpr int SC = WK == W_NVFP4_A16 ? GS_KSEG / 16 : (GS_KSEG / 128) * 2;
    static constexpr int MN = WK == W_INT4 ? (GS_KSEG / 128) * 2 : 0;
    static constexpr uint32_t STAGE = GS_CWARPS * (GS_CODE + SC + MN);
};

struct GsParams {
    const uint16_t *x;      // bf16 [K]
    const uint8_t *codes;   // [N, K/2]
    const uint8_t *scale;   // NVFP4 e4m3 [N, K/16]; int4 fp16 [N, K/128]
    const uint8_t *minv;    // int4 fp16 [N, K/128]
    const float *gscale;    // NVFP4 global scale (device)
    uint16_t *y;            // bf16 [N]
    unsigned *err;
    int N, K, S;
    int rows_q, rows_r;     // CTA b owns rows_q (+1 if b < rows_r) rows
    int ns;                 // ring stages
    int rows_max;           // ceil(N / grid): partial-sum slots per CTA (S > 1)
};

// Shared memory (after the stage ring): x' image [K / 8 vectors of 16 bytes], chunk
// factors [K / 32] (NVFP4: 2^-p * g; int4: 2^-p and the chunk's sum of x' as a
// float2), then for S > 1 the row partials [rows_max][S] and arrival counters
// [rows_max], and the barriers full[ns], empty[ns].
template <int WK>
__host__ __device__ constexpr uint32_t gs_cf_bytes(int K)
{
    return (uint32_t)(K / 32) * (WK == W_INT4 ? 8u : 4u);
}

// x' vector i (0..3) of half h (0, 1) of lane l in k-segment k: index in the image.
__device__ __forceinline__ int gs_xvec(int k, int h, int i, int l)
{
    return ((k * 2 + h) * 4 + i) * 32 + l;
}

// Stage x: thread t converts 8 columns (block b = t, t + nthreads, ...); 4
// consecutive blocks form a 32-column chunk (4 consecutive lanes).  The prescale
// exponent p puts the chunk maximum in [2^9, 2^10) (NVFP4 fp16 sums) or [2^14,
// 2^15) (int4 int16 fixed point), clamped to +-126.
template <int WK>
__device__ __forceinline__ void gs_stage_x(const GsParams &p, uint4 *xs, float *cf, float gsc,
                                           int t, int nthreads)
{
    const int nblk = p.K / 8;
    for (int b0 = 0; b0 < nblk; b0 += nthreads) {
        const int b = b0 + t;
        const bool active = b < nblk;                 // nblk is a multiple of 32
        const int k0 = active ? 8 * b : 0;
        const uint4 v = active ? __ldcg(reinterpret_cast<const uint4 *>(p.x + k0)) : make_uint4(0, 0, 0, 0);
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
        int ex = 0;
        if (amax > 0.f && !isinf(amax)) {
            const int be = (int)((__float_as_uint(amax) >> 23) & 0xff);
            if (be > 0)
                ex = be - 126;
            else
                frexpf(amax, &ex);
        }
        int pw = (WK == W_INT4 ? 15 : 10) - ex;
        pw = pw > 126 ? 126 : (pw < -126 ? -126 : pw);
        const float up = pow2f(pw);
        const int ks = k0 / GS_KSEG, kk = k0 % GS_KSEG;
        const int h = kk / 1024, l = (kk % 1024) / 32, i = (kk % 32) / 8;
        if constexpr (WK == W_INT4) {
            int xi[8];
            bool bad = false;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                bad |= !(fabsf(f[j]) <= 3.402823466e38f);
                xi[j] = __float2int_rn(f[j] * up);
            }
            auto pack = [](int lo, int hi) { return ((uint32_t)lo & 0xffffu) | ((uint32_t)hi << 16); };
            if (active)
                xs[gs_xvec(ks, h, i, l)] = make_uint4(pack(xi[0], xi[2]), pack(xi[4], xi[6]),
                                                      pack(xi[1], xi[3]), pack(xi[5], xi[7]));
            float sx = (float)(((xi[0] + xi[1]) + (xi[2] + xi[3])) + ((xi[4] + xi[5]) + (xi[6] + xi[7])));
            if (bad)
                sx = __int_as_float(0x7fc00000);
            sx += __shfl_xor_sync(0xffffffffu, sx, 1);
            sx += __shfl_xor_sync(0xffffffffu, sx, 2);
            if (active && (k0 % 32) == 0)
                reinterpret_cast<float2 *>(cf)[k0 / 32] = make_float2(pow2f(-pw), sx);
        } else {
            uint32_t hq[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                __half2 hh = __floats2half2_rn(f[2 * j] * up, f[2 * j + 1] * up);
                hq[j] = *reinterpret_cast<uint32_t *>(&hh);
            }
            if (active)
                xs[gs_xvec(ks, h, i, l)] = make_uint4(hq[0], hq[1], hq[2], hq[3]);
            if (active && (k0 % 32) == 0)
                cf[k0 / 32] = pow2f(-pw) * gsc;
        }
    }
}

// One lane's 32 columns of a row: 16 code bytes q, its scale word sw (NVFP4: two
// e4m3 bytes; int4: fp16 scale) and min word mw (int4 fp16 min), against its x'
// registers xr and chunk data (NVFP4 factor; int4 factor and sum of x').
template <int WK>
__device__ __forceinline__ float gs_dot32(const uint4 q, uint32_t sw, uint32_t mw,
                                          const uint32_t (&xr)[16], float2 cd)
{
    const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
    if constexpr (WK == W_INT4) {
        int A = 0;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const uint32_t ce = w4[jj] & 0x0F0F0F0Fu;          // c of columns 0, 2, 4, 6
            const uint32_t co = (w4[jj] >> 4) & 0x0F0F0F0Fu;   // c of columns 1, 3, 5, 7
            A = dp2a_lo_su(xr[4 * jj + 0], ce, A);
            A = dp2a_hi_su(xr[4 * jj + 1], ce, A);
            A = dp2a_lo_su(xr[4 * jj + 2], co, A);
            A = dp2a_hi_su(xr[4 * jj + 3], co, A);
        }
        // |A| <= 32 * 15 * 32767 < 2^24: exact in fp32
        return fmaf(f16lo_to_f32(sw), (float)A, f16lo_to_f32(mw) * cd.y) * cd.x;
    } else {
        uint32_t Ha = 0u, Hb = 0u;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            uint32_t hh[4];
            e2m1x8_to_f16x2x4(w4[jj], hh);
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
                if (jj < 2)
                    Ha = hfma2_rn(hh[qq], xr[4 * jj + qq], Ha);
                else
                    Hb = hfma2_rn(hh[qq], xr[4 * jj + qq], Hb);
            }
        }
        const uint32_t s2 = e4m3x2_to_f16x2(sw);
        const float ta = f16lo_to_f32(Ha) + f16hi_to_f32(Ha);
        const float tb = f16lo_to_f32(Hb) + f16hi_to_f32(Hb);
        return fmaf(ta, f16lo_to_f32(s2), tb * f16hi_to_f32(s2)) * cd.x;
    }
}

template <int WK>
__global__ void __launch_bounds__(GS_THREADS, 2) q4_gemv_stage_kernel(GsParams p)
{
    extern __shared__ __align__(128) unsigned char smem[];
    constexpr uint32_t STAGE = GsUnit<WK>::STAGE;
    constexpr int SC = GsUnit<WK>::SC;
    constexpr int MN = GsUnit<WK>::MN;
    const int NS = p.ns;
    const int S = p.S;
    const int RS = GS_CWARPS / S;                    // rows per stage
    uint4 *xs = reinterpret_cast<uint4 *>(smem + (size_t)NS * STAGE);
    float *cf = reinterpret_cast<float *>(smem + (size_t)NS * STAGE + (size_t)p.K * 2);
    float *part = reinterpret_cast<float *>(reinterpret_cast<unsigned char *>(cf) + gs_cf_bytes<WK>(p.K));
    unsigned *cnt = reinterpret_cast<unsigned *>(part + (size_t)p.rows_max * S);
    uint64_t *bars = reinterpret_cast<uint64_t *>(
        (reinterpret_cast<uintptr_t>(cnt + p.rows_max) + 7) & ~(uintptr_t)7);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.x;
    const int n0 = b * p.rows_q + (b < p.rows_r ? b : p.rows_r);
    const int rows = p.rows_q + (b < p.rows_r ? 1 : 0);
    const int nst = (rows + RS - 1) / RS;
    const int64_t row_bytes = (int64_t)p.K / 2;
    const int64_t srow = WK == W_NVFP4_A16 ? p.K / 16 : (p.K / 128) * 2;   // scale bytes per row

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(smem_u32(&bars[i]), 1);
            mbar_init(smem_u32(&bars[NS + i]), GS_CWARPS);
        }
        mbar_init_fence();
    }
    for (int i = threadIdx.x; i < p.rows_max; i += GS_THREADS)
        cnt[i] = 0u;
    __syncthreads();
    pdl_launch_dependents();

    if (warp == GS_CWARPS) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            auto issue = [&](int s) {
                unsigned char *st = smem + (size_t)(s % NS) * STAGE;
                const int r0 = s * RS;
                const int nr = rows - r0 < RS ? rows - r0 : RS;
                const uint32_t cb = (uint32_t)(nr * row_bytes), sb = (uint32_t)(nr * srow);
                const uint32_t full = smem_u32(&bars[s % NS]);
                mbar_arrive_expect_tx(full, cb + sb * (MN ? 2u : 1u));
                bulk_copy_g2s(smem_u32(st), p.codes + (int64_t)(n0 + r0) * row_bytes, cb, full);
                bulk_copy_g2s(smem_u32(st + GS_CWARPS * GS_CODE),
                              p.scale + (int64_t)(n0 + r0) * srow, sb, full);
                if constexpr (MN > 0)
                    bulk_copy_g2s(smem_u32(st + GS_CWARPS * (GS_CODE + SC)),
                                  p.minv + (int64_t)(n0 + r0) * srow, sb, full);
            };
            int issued = 0;
            for (; issued < nst && issued < NS; ++issued)
                issue(issued);
            bool alive = true;
            for (; issued < nst; ++issued) {
                const int s = issued;
                if (!mbar_wait(smem_u32(&bars[NS + s % NS]), ((s / NS) - 1) & 1, p.err)) {
                    alive = false;
                    break;
                }
                issue(s);
            }
            // every issued copy has landed before the CTA may leave
            for (int s = issued - NS > 0 ? issued - NS : 0; s < issued; ++s)
                mbar_wait(smem_u32(&bars[s % NS]), (s / NS) & 1, p.err);
            (void)alive;
        }
        return;
    }

    // ------------------------------------------------------------ consumers
    float gsc = 1.f;
    if constexpr (WK == W_NVFP4_A16)
        gsc = __ldg(p.gscale);
    pdl_wait();                                     // x comes from the previous kernel
    gs_stage_x<WK>(p, xs, cf, gsc, (int)threadIdx.x, GS_CWARPS * 32);
    asm volatile("bar.sync 1, %0;" ::"r"(GS_CWARPS * 32) : "memory");

    const int k = warp % S;                         // this warp's k-segment
    const int rw = warp / S;                        // its row within a stage
    uint32_t xr[2][16];
    float2 cd[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 t = xs[gs_xvec(k, h, i, lane)];
            xr[h][4 * i + 0] = t.x; xr[h][4 * i + 1] = t.y;
            xr[h][4 * i + 2] = t.z; xr[h][4 * i + 3] = t.w;
        }
        const int chunk = (k * GS_KSEG + h * 1024 + 32 * lane) / 32;
        if constexpr (WK == W_INT4)
            cd[h] = reinterpret_cast<const float2 *>(cf)[chunk];
        else
            cd[h] = make_float2(cf[chunk], 0.f);
    }

    // offsets of this lane's data inside a stage
    const uint32_t code_off = (uint32_t)warp * GS_CODE + 16u * lane;
    uint32_t sc_off[2], mn_off[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int col = h * 1024 + 32 * lane;       // column within the unit
        if constexpr (WK == W_INT4) {
            sc_off[h] = GS_CWARPS * GS_CODE + warp * SC + (col / 128) * 2;
            mn_off[h] = GS_CWARPS * (GS_CODE + SC) + warp * SC + (col / 128) * 2;
        } else {
            sc_off[h] = GS_CWARPS * GS_CODE + warp * SC + col / 16;
            mn_off[h] = 0;
        }
    }

    bool alive = true;
    for (int s0 = 0; s0 < nst; s0 += GS_RB) {
        float v[GS_RB];
#pragma unroll
        for (int j = 0; j < GS_RB; ++j) {
            const int s = s0 + j;
            v[j] = 0.f;
            if (s >= nst || !alive)
                continue;
            const unsigned char *st = smem + (size_t)(s % NS) * STAGE;
            if (!mbar_wait_warp(smem_u32(&bars[s % NS]), (s / NS) & 1, p.err)) {
                alive = false;
                continue;
            }
            const bool ok = s * RS + rw < rows;
            uint4 q0 = make_uint4(0, 0, 0, 0), q1 = q0;
            uint32_t s0w = 0, s1w = 0, m0w = 0, m1w = 0;
            if (ok) {
                q0 = *reinterpret_cast<const uint4 *>(st + code_off);
                q1 = *reinterpret_cast<const uint4 *>(st + code_off + 512);
                s0w = *reinterpret_cast<const uint16_t *>(st + sc_off[0]);
                s1w = *reinterpret_cast<const uint16_t *>(st + sc_off[1]);
                if constexpr (WK == W_INT4) {
                    m0w = *reinterpret_cast<const uint16_t *>(st + mn_off[0]);
                    m1w = *reinterpret_cast<const uint16_t *>(st + mn_off[1]);
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_u32(&bars[NS + s % NS]));   // slot free for the producer
            if (ok)
                v[j] = gs_dot32<WK>(q0, s0w, m0w, xr[0], cd[0]) + gs_dot32<WK>(q1, s1w, m1w, xr[1], cd[1]);
        }
        int idx = 0;
        const float tot = warp_sum_transpose<GS_RB>(v, lane, idx);
        const int s = s0 + idx;
        const int r = s * RS + rw;                  // row within the CTA
        if ((lane & (32 / GS_RB - 1)) == 0 && s < nst && r < rows && alive) {
            if (S == 1) {
                p.y[n0 + r] = f32_to_bf16_bits(tot);
            } else {
                part[r * S + k] = tot;
                __threadfence_block();
                if (atomicAdd(&cnt[r], 1u) == (unsigned)(S - 1)) {
                    __threadfence_block();
                    float sum = 0.f;
                    for (int kk = 0; kk < S; ++kk)
                        sum += *reinterpret_cast<volatile float *>(&part[r * S + kk]);
                    p.y[n0 + r] = f32_to_bf16_bits(sum);
                }
            }
        }
    }
}

// ------------------------------------------------------------------ host side
static size_t stage_smem(int kind, int K, int rows_max, int ns)
{
    const uint32_t stage = kind == W_INT4 ? GsUnit<W_INT4>::STAGE : GsUnit<W_NVFP4_A16>::STAGE;
    const uint32_t cfb = kind == W_INT4 ? gs_cf_bytes<W_INT4>(K) : gs_cf_bytes<W_NVFP4_A16>(K);
    const int S = K / GS_KSEG;
    size_t b = (size_t)ns * stage + (size_t)K * 2 + cfb;
    b += (size_t)rows_max * S * 4 + (size_t)rows_max * 4;
    b = (b + 7) / 8 * 8 + (size_t)ns * 2 * 8;
    return b;
}

bool stage_plan(const DeviceInfo &dev, int kind, int M, int N, int K, const void *x,
                const void *codes, const void *scale, const void *minv, const void *y,
                StagePlan &plan)
{
    plan = StagePlan{};
    const int S = K / GS_KSEG;
    if (M != 1 || K % GS_KSEG || (S != 1 && S != 2 && S != 4 && S != 8))
        return false;
    if (kind != W_INT4 && kind != W_NVFP4_A16)
        return false;
    auto a16 = [](const void *q) { return ((uintptr_t)q % 16) == 0; };
    if (!a16(x) || !a16(codes) || !a16(scale) || !a16(y) || (kind == W_INT4 && !a16(minv)))
        return false;
    plan.kind = kind;
    plan.grid = dev.sms < N ? dev.sms : N;
    // row partials and counters only when a row spans several units
    plan.rows_max = S > 1 ? (N + plan.grid - 1) / plan.grid : 0;
    // Half of the SM's shared memory, so that the next call's CTA fits beside this
    // one: as many stages as that leaves room for, between two and eight.
    const size_t half = dev.smem_optin / 2 > 1024 ? dev.smem_optin / 2 - 1024 : 0;
    int ns = 8;
    while (ns > 2 && stage_smem(kind, K, plan.rows_max, ns) > half)
        --ns;
    plan.ns = ns;
    plan.smem = stage_smem(kind, K, plan.rows_max, ns);
    return plan.smem <= half;
}

q4_status stage_launch(const StagePlan &plan, const void *x, const uint8_t *codes,
                       const void *scale, const void *minv, const float *gscale, void *y, int N,
                       int K, cudaStream_t stream, bool pdl)
{
    GsParams p = {};
    p.x = static_cast<const uint16_t *>(x);
    p.codes = codes;
    p.scale = static_cast<const uint8_t *>(scale);
    p.minv = static_cast<const uint8_t *>(minv);
    p.gscale = gscale;
    p.y = static_cast<uint16_t *>(y);
    p.err = device_error_flags();
    p.N = N;
    p.K = K;
    p.S = K / GS_KSEG;
    p.rows_q = N / plan.grid;
    p.rows_r = N % plan.grid;
    p.rows_max = plan.rows_max;
    p.ns = plan.ns;
    const void *k = plan.kind == W_INT4
                        ? reinterpret_cast<const void *>(&q4_gemv_stage_kernel<W_INT4>)
                        : reinterpret_cast<const void *>(&q4_gemv_stage_kernel<W_NVFP4_A16>);
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)plan.smem);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaFuncSetAttribute(staged GEMV)");
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)plan.grid);
    cfg.blockDim = dim3(GS_THREADS);
    cfg.dynamicSmemBytes = plan.smem;
    cfg.stream = stream;
    cfg.attrs = pdl ? attr : nullptr;
    cfg.numAttrs = pdl ? 1 : 0;
    void *args[] = {&p};
    e = cudaLaunchKernelExC(&cfg, k, args);
    if (e != cudaSuccess)
        return cuda_fail(e, "launch of the staged GEMV");
    return Q4_OK;
}

}  // namespace q4
