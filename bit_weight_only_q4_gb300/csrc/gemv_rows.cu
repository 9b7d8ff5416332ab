// Register-prefetch weight-streaming kernel for sm_103a: the decode GEMV of both
// 4-bit layouts for one to four tokens, and the restricted BF16 head.
//
// Same arithmetic as the other streaming kernels (stream_common.cuh: prescaled
// fp16 x, shift-free E2M1 / fp16-magic int4 decode, fp32 accumulation by
// mixed-precision FMAs).  Data movement is chosen for short, dependent calls:
//
//   * Small CTAs (8 warps) each own a contiguous range of output rows with their
//     full K.  Warp w owns one k-step ks = w % S (1024 4-bit or 256 bf16
//     columns) of the rows g, g + G, g + 2G, ... of its CTA (g = w / S, G = 8/S).
//   * Before griddepcontrol.wait every lane issues the 128-bit loads of its
//     first RB rows (codes and scales): weights do not depend on the previous
//     kernel, so they stream while that kernel finishes.  With up to four CTAs
//     per SM, a CTA of the next call starts loading as soon as any CTA of this
//     call exits.  (A TMA bulk-copy ring was measured slower here: the per-SM
//     copy engine sustained ~26 GB/s in this short-burst pattern, below the
//     ~44 GB/s per SM that HBM delivers.)
//   * After the wait the CTA stages x once in shared memory; every warp keeps
//     its k-step's slice in registers, decodes and multiplies its rows, reduces
//     each row across lanes (transposing butterfly) and parks the partial per
//     k-step in shared memory; later row batches are loaded after the first.
//   * A final pass sums each row's S partials in k order and stores bf16.  No
//     row is split between CTAs: no workspace, deterministic results.
//
// Eligibility: S = ceil(K / kstep) in {1, 2, 4, 8}; 16-byte aligned rows (int4
// always, NVFP4 K % 32 == 0, bf16 H % 8 == 0).  Other shapes use gemv.cu.
#include "q4_device.cuh"
#include "q4_internal.h"
#include "stream_common.cuh"

namespace q4 {

constexpr int RK_WARPS = 8;
constexpr int RK_THREADS = RK_WARPS * 32;

template <int WK, int MT, int RB>
__global__ void __launch_bounds__(RK_THREADS, (MT == 1 ? 4 : 2)) q4_rows_kernel(GemvParams p)
{
    extern __shared__ __align__(16) unsigned char smem[];
    constexpr int KSTEP = Kind<WK>::KSTEP;
    constexpr int COLS = Kind<WK>::COLS;
    constexpr int CH = Kind<WK>::CH;
    constexpr int XV = (WK == W_BF16) ? 4 : 16;      // x registers per token
    const int S = p.S;
    const int G = RK_WARPS / S;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int ks = warp % S;
    const int g = warp / S;
    const int col0 = ks * KSTEP + lane * COLS;
    const bool colok = col0 < p.K;
    const int Kpad = S * KSTEP;
    uint16_t *xs = reinterpret_cast<uint16_t *>(smem);
    float *cf = reinterpret_cast<float *>(smem + (size_t)MT * Kpad * 2);
    float *red = cf + (size_t)MT * (Kpad / 32) * CH;        // [row][ks][m] partials
    const int64_t n0 = (int64_t)blockIdx.x * p.N / p.grid;
    const int64_t n1 = ((int64_t)blockIdx.x + 1) * p.N / p.grid;
    const int rows_cta = (int)(n1 - n0);
    const int my_rows = rows_cta > g ? (rows_cta - g + G - 1) / G : 0;   // rows g + G*j

    uint4 q[RB];
    uint32_t sw[RB];
    auto load_batch = [&](int j0) {
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            q[r] = make_uint4(0u, 0u, 0u, 0u);
            sw[r] = 0u;
            const int j = j0 + r;
            if (j < my_rows && colok) {
                const int64_t n = n0 + g + (int64_t)G * j;
                const int64_t prow = n < p.n_rows ? (int64_t)p.row_begin + n : (int64_t)p.extra_row;
                if constexpr (WK == W_BF16) {
                    q[r] = ld_stream_v4(p.w + prow * p.w_row_bytes + (int64_t)col0 * 2);
                } else {
                    q[r] = ld_stream_v4(p.w + prow * p.w_row_bytes + col0 / 2);
                    if constexpr (WK == W_INT4) {
                        const int64_t gi = prow * (p.K / 128) + col0 / 128;
                        sw[r] = ld_nc_u16(static_cast<const uint16_t *>(p.scale) + gi) |
                                (ld_nc_u16(p.minv + gi) << 16);
                    } else {
                        sw[r] = ld_nc_u16(static_cast<const uint8_t *>(p.scale) +
                                          prow * (p.K / 16) + col0 / 16);
                    }
                }
            }
        }
    };

    // weights (and the global scale) do not depend on the previous kernel
    load_batch(0);
    float gsc = 1.f;
    if constexpr (WK == W_NVFP4_A16)
        gsc = __ldg(p.gscale);
    pdl_launch_dependents();
    pdl_wait();                                   // x comes from the previous kernel
    stage_x<WK, MT>(p, Kpad, xs, cf, (int)threadIdx.x, RK_THREADS);
    __syncthreads();

    uint32_t xr[MT][XV];
    float4 cd[MT];           // int4: (2^-p, X1, X2, -); NVFP4: (2^-p * g, ...)
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        if constexpr (WK == W_BF16) {
            const uint4 t = *reinterpret_cast<const uint4 *>(xs + (size_t)m * Kpad + col0);
            xr[m][0] = t.x; xr[m][1] = t.y; xr[m][2] = t.z; xr[m][3] = t.w;
            cd[m] = make_float4(1.f, 0.f, 0.f, 0.f);
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

    for (int j0 = 0; j0 < my_rows; j0 += RB) {
        if (j0 > 0)
            load_batch(j0);
        float part[RB * MT];
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            const uint32_t w4[4] = {q[r].x, q[r].y, q[r].z, q[r].w};
            if constexpr (WK == W_BF16) {
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    float t = 0.f;
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj)
                        t = fma2_bf16(t, w4[jj], xr[m][jj]);
                    part[r * MT + m] = t;
                }
            } else if constexpr (WK == W_INT4) {
                float A1[MT], A2[MT];
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    A1[m] = 0.f;
                    A2[m] = 0.f;
                }
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const uint32_t w8 = w4[jj] >> 8;
                    const uint32_t pa = int4_pair_f16_biased<0x000F000Fu>(w4[jj]);  // cols 0, 4
                    const uint32_t pb = int4_pair_f16_biased<0x00F000F0u>(w4[jj]);  // cols 1, 5
                    const uint32_t pc = int4_pair_f16_biased<0x000F000Fu>(w8);      // cols 2, 6
                    const uint32_t pd = int4_pair_f16_biased<0x00F000F0u>(w8);      // cols 3, 7
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        A1[m] = fma2_f16(A1[m], pa, xr[m][4 * jj + 0]);
                        A2[m] = fma2_f16(A2[m], pb, xr[m][4 * jj + 1]);
                        A1[m] = fma2_f16(A1[m], pc, xr[m][4 * jj + 2]);
                        A2[m] = fma2_f16(A2[m], pd, xr[m][4 * jj + 3]);
                    }
                }
                const float sc = f16lo_to_f32(sw[r]);
                const float mn = f16hi_to_f32(sw[r]);
                const float c1 = fmaf(-1024.f, sc, mn);
                const float c2 = fmaf(-64.f, sc, mn);
                const float s16 = sc * 0.0625f;
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    float t = sc * A1[m];
                    t = fmaf(s16, A2[m], t);
                    t = fmaf(c1, cd[m].y, t);
                    t = fmaf(c2, cd[m].z, t);
                    part[r * MT + m] = t * cd[m].x;
                }
            } else {
                float Ta[MT], Tb[MT];
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    Ta[m] = 0.f;
                    Tb[m] = 0.f;
                }
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    uint32_t h[4];
                    e2m1x8_to_f16x2x4(w4[jj], h);
#pragma unroll
                    for (int b = 0; b < 4; ++b) {
#pragma unroll
                        for (int m = 0; m < MT; ++m) {
                            if (jj < 2)
                                Ta[m] = fma2_f16(Ta[m], h[b], xr[m][4 * jj + b]);
                            else
                                Tb[m] = fma2_f16(Tb[m], h[b], xr[m][4 * jj + b]);
                        }
                    }
                }
                const uint32_t s2 = e4m3x2_to_f16x2(sw[r]);
                const float sa = f16lo_to_f32(s2);
                const float sb = f16hi_to_f32(s2);
#pragma unroll
                for (int m = 0; m < MT; ++m)
                    part[r * MT + m] = fmaf(Ta[m], sa, Tb[m] * sb) * cd[m].x;
            }
        }
        int idx = 0;
        const float tot = warp_sum_transpose<RB * MT>(part, lane, idx);
        const int r = idx / MT, m = idx - (idx / MT) * MT;
        const int j = j0 + r;
        if ((lane & (32 / (RB * MT) - 1)) == 0 && j < my_rows) {
            const int row = g + G * j;
            red[((size_t)row * S + ks) * MT + m] = tot;
        }
    }

    __syncthreads();
    for (int e = (int)threadIdx.x; e < rows_cta * MT; e += RK_THREADS) {
        const int row = e / MT, m = e - (e / MT) * MT;
        float s = 0.f;
        for (int k = 0; k < S; ++k)
            s += red[((size_t)row * S + k) * MT + m];
        if (m < p.mcount)
            p.y[(int64_t)(p.m0 + m) * p.ldy + n0 + row] = f32_to_bf16_bits(s);
    }
}

// ------------------------------------------------------------------ host side
template <int WK, int MT, int RB>
static const void *rows_ptr()
{
    return reinterpret_cast<const void *>(&q4_rows_kernel<WK, MT, RB>);
}

template <int WK>
static const void *rows_select_kind(int mt, int rb)
{
#define Q4_R(MT_, RB_) if (mt == MT_ && rb == RB_) return rows_ptr<WK, MT_, RB_>();
    Q4_R(1, 4) Q4_R(1, 8) Q4_R(2, 2) Q4_R(2, 4) Q4_R(4, 1) Q4_R(4, 2)
#undef Q4_R
    return nullptr;
}

static const void *rows_select(int kind, int mt, int rb)
{
    if (kind == W_INT4) return rows_select_kind<W_INT4>(mt, rb);
    if (kind == W_NVFP4_A16) return rows_select_kind<W_NVFP4_A16>(mt, rb);
    if (kind == W_BF16) return rows_select_kind<W_BF16>(mt, rb);
    return nullptr;
}

#ifndef Q4_ROWS_RB
#define Q4_ROWS_RB 0          // rows per warp batch for M = 1; 0 = planner
#endif
#ifndef Q4_ROWS_CTAS_PER_SM
#define Q4_ROWS_CTAS_PER_SM 4
#endif

bool rows_eligible(int kind, int K)
{
    const int kstep = kind == W_BF16 ? 256 : 1024;
    const int S = (K + kstep - 1) / kstep;
    if (S != 1 && S != 2 && S != 4 && S != 8)
        return false;
    if (kind == W_INT4) return K % 128 == 0;
    if (kind == W_NVFP4_A16) return K % 32 == 0;
    if (kind == W_BF16) return K % 8 == 0;
    return false;
}

q4_status rows_plan(const DeviceInfo &dev, int kind, int M, int N, int K, RowsPlan &plan)
{
    plan = RowsPlan{};
    plan.kind = kind;
    const int kstep = kind == W_BF16 ? 256 : 1024;
    const int ch = kind == W_INT4 ? 4 : (kind == W_BF16 ? 0 : 1);
    plan.S = (K + kstep - 1) / kstep;
    const int G = RK_WARPS / plan.S;
    const size_t Kpad = (size_t)plan.S * kstep;
    plan.mt = M >= 4 ? 4 : (M >= 2 ? 2 : 1);
    plan.rb = plan.mt == 4 ? 2 : (plan.mt == 2 ? 4 : 4);
    if (plan.mt == 1 && Q4_ROWS_RB > 0)
        plan.rb = Q4_ROWS_RB;
    // about four CTAs per SM (one batch of RB rows per warp when the matrix is
    // small enough), each with a contiguous row range
    int64_t grid = (int64_t)dev.sms * Q4_ROWS_CTAS_PER_SM;
    const int64_t rows_one_batch = (int64_t)G * plan.rb;
    const int64_t want = ((int64_t)N + rows_one_batch - 1) / rows_one_batch;
    if (want < grid)
        grid = want;
    if (grid < 1)
        grid = 1;
    // per-row partials must fit: cap rows per CTA at 24 KB of partials
    const int64_t rows_limit = (24 * 1024) / ((int64_t)plan.S * plan.mt * 4);
    const int64_t need = ((int64_t)N + rows_limit - 1) / rows_limit;
    if (need > grid)
        grid = need;
    if (grid > 0x7fffffff)
        return fail(Q4_ERR_SHAPE, "N=%d too large", N);
    plan.grid = (int)grid;
    const int64_t rows_cap = ((int64_t)N + grid - 1) / grid;
    plan.smem = (size_t)plan.mt * Kpad * 2 + (size_t)plan.mt * (Kpad / 32) * ch * 4 +
                (size_t)rows_cap * plan.S * plan.mt * 4;
    if (plan.smem > dev.smem_optin)
        return fail(Q4_ERR_SHAPE, "K=%d too large for the register-prefetch kernel", K);
    const void *k = rows_select(kind, plan.mt, plan.rb);
    if (!k)
        return fail(Q4_ERR_ARG, "no register-prefetch kernel for kind %d", kind);
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)plan.smem);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaFuncSetAttribute(register-prefetch kernel)");
    return Q4_OK;
}

q4_status rows_launch(const RowsPlan &plan, GemvParams p, int M, cudaStream_t stream, bool pdl)
{
    const void *k = rows_select(plan.kind, plan.mt, plan.rb);
    p.S = plan.S;
    p.grid = plan.grid;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    for (int m0 = 0; m0 < M; m0 += plan.mt) {
        p.m0 = m0;
        p.mcount = (M - m0) < plan.mt ? (M - m0) : plan.mt;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)plan.grid);
        cfg.blockDim = dim3(RK_THREADS);
        cfg.dynamicSmemBytes = plan.smem;
        cfg.stream = stream;
        cfg.attrs = pdl ? attr : nullptr;
        cfg.numAttrs = pdl ? 1 : 0;
        void *args[] = {&p};
        cudaError_t e = cudaLaunchKernelExC(&cfg, k, args);
        if (e != cudaSuccess)
            return cuda_fail(e, "launch of the register-prefetch kernel");
    }
    return Q4_OK;
}

}  // namespace q4
