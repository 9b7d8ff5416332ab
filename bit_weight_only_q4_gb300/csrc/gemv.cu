// CUDA-core weight-streaming kernel for sm_103a: the decode GEMV (one to a few
// tokens) of both 4-bit layouts and the restricted BF16 head.
//
// What it computes:
//   int4-g128-minmax ("rumik-oss-1-int4", "Format"): y[m,n] = sum_k x[m,k] w[n,k]
//     with w = code * scale + min.  Per group of 128 columns the min factors out:
//     sum_k x w = s * sum_k c x + m * sum_k x; the per-chunk sums of x are shared
//     by every row and computed once per CTA.
//   NVFP4 weight-only ("VoxCPM2 NVFP4 (GPTQ)", "NVFP4 settings"):
//     w = E2M1(code) * e4m3(scale) * g; per group of 16 columns the scale and the
//     global factor are applied to the group's partial dot product.
//   Restricted head ("Rumik TTS Fast Inference", "What Made It Faster", Fig. 3):
//     bf16 weights, logical row n read from row (row_begin + n) or extra_row.
//
// How (HBM-bound design):
//   * Work is cut into units of RW rows x one k-step (32 lanes x 16 bytes of
//     weights per row = 1024 4-bit columns or 256 bf16 columns).  Units are laid
//     out row-group-major and every warp of the grid takes one contiguous range
//     of them ("stream-K"), so all warps stream the same number of bytes +-1 unit
//     whatever N and K are.
//   * Each lane streams 128-bit weight loads (L1 no-allocate), one unit ahead of
//     the one it decodes; decode is in registers: int4 nibbles become bf16
//     (128 + c) by one LOP3 per pair, E2M1 pairs become f16x2 by one cvt.
//   * Products accumulate in fp32 with mixed-precision FMAs (bf16 or f16
//     operands, fp32 accumulator).  x is staged once per CTA in shared memory,
//     already in the operand format and order the decoder produces.
//   * A warp that covers a whole row group reduces across lanes (transposing
//     butterfly) and stores bf16.  Row groups split between warps write fp32
//     partials; the last warp to arrive (atomic ticket) sums them in k order --
//     deterministic, and no warp ever waits for another.
//   * Weights are read before griddepcontrol.wait, so under programmatic
//     dependent launch the first loads overlap the previous kernel's tail.
#include <cstdio>

#include "q4_device.cuh"
#include "q4_internal.h"
#include "stream_common.cuh"

namespace q4 {

constexpr int GEMV_WARPS = 8;
constexpr int GEMV_THREADS = GEMV_WARPS * 32;

// Warp w of TW takes units [unit_start(w), unit_start(w + 1)).  Ranges are
// multiples of p.gran units: gran == 1 splits row groups between warps
// (stream-K, partial sums in the workspace); gran == S keeps every row group in
// one warp (no workspace).
__device__ __forceinline__ int64_t unit_start(const GemvParams &p, int64_t w)
{
    const int64_t Uq = p.U / p.gran;
    return (w * Uq / p.TW) * p.gran;
}

// The warp whose range contains unit u.
__device__ __forceinline__ int64_t warp_of_unit(const GemvParams &p, int64_t u)
{
    const int64_t Uq = p.U / p.gran;
    const int64_t v = u / p.gran;
    return ((v + 1) * p.TW + Uq - 1) / Uq - 1;
}

__device__ __forceinline__ int64_t physical_row(const GemvParams &p, int n)
{
    return n < p.n_rows ? (int64_t)p.row_begin + n : (int64_t)p.extra_row;
}

template <int WK, int RW>
__device__ __forceinline__ void load_unit(const GemvParams &p, int64_t u, int lane,
                                          UnitRegs<RW> &R)
{
    constexpr int COLS = Kind<WK>::COLS;
    const int g = (int)(u / p.S);
    const int ks = (int)(u - (int64_t)g * p.S);
    const int col0 = ks * Kind<WK>::KSTEP + lane * COLS;
    const bool colok = col0 < p.K;
#pragma unroll
    for (int r = 0; r < RW; ++r) {
        const int n = g * RW + r;
        R.q[r] = make_uint4(0u, 0u, 0u, 0u);
        R.s[r] = 0u;
        if (colok && n < p.N) {
            const int64_t prow = physical_row(p, n);
            if constexpr (WK == W_BF16) {
                R.q[r] = ld_stream_v4(p.w + prow * p.w_row_bytes + (int64_t)col0 * 2);
            } else {
                const uint8_t *src = p.w + prow * p.w_row_bytes + col0 / 2;
                if constexpr (WK == W_NVFP4_A8) {
                    // rows are only 8-byte aligned (K % 32 == 16); the last chunk
                    // of a row may hold 16 columns only
                    uint2 lo = ld_stream_v2(src);
                    uint2 hi = (col0 + 16 < p.K) ? ld_stream_v2(src + 8) : make_uint2(0u, 0u);
                    R.q[r] = make_uint4(lo.x, lo.y, hi.x, hi.y);
                } else {
                    R.q[r] = ld_stream_v4(src);
                }
            }
            if constexpr (WK == W_INT4) {
                const int64_t gi = prow * (p.K / 128) + col0 / 128;
                const uint16_t *sc = static_cast<const uint16_t *>(p.scale);
                R.s[r] = ld_nc_u16(sc + gi) | (ld_nc_u16(p.minv + gi) << 16);
            } else if constexpr (WK == W_NVFP4_A16) {
                const uint8_t *sc = static_cast<const uint8_t *>(p.scale);
                R.s[r] = ld_nc_u16(sc + prow * (p.K / 16) + col0 / 16);
            } else if constexpr (WK == W_NVFP4_A8) {
                const uint8_t *sc = static_cast<const uint8_t *>(p.scale) + prow * (p.K / 16) +
                                    col0 / 16;
                R.s[r] = ld_nc_u8(sc) | ((col0 + 16 < p.K) ? (ld_nc_u8(sc + 1) << 8) : 0u);
            }
        }
    }
}

template <int MT, int RW>
__device__ __forceinline__ void finish_row_group(const GemvParams &p, int64_t g, int ks_first,
                                                 int ks_last, int64_t my_warp, int lane,
                                                 float (&acc)[RW][MT])
{
    constexpr int V = RW * MT;
    static_assert(V <= 32, "RW * MT must not exceed 32");
    float v[V];
#pragma unroll
    for (int r = 0; r < RW; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m)
            v[r * MT + m] = acc[r][m];
    int idx = 0;
    const float tot = warp_sum_transpose<V>(v, lane, idx);
    const bool writer = (lane & (32 / V - 1)) == 0;
    const int r = idx / MT, m = idx - (idx / MT) * MT;
    const int n = (int)g * RW + r;
    const bool valid = writer && n < p.N && m < p.mcount;
    if (ks_first == 0 && ks_last == p.S - 1) {
        if (valid)
            p.y[(int64_t)(p.m0 + m) * p.ldy + n] = f32_to_bf16_bits(tot);
        return;
    }
    // part of a row group: publish the partial, the last arriving warp sums
    const int64_t base = g * p.S;
    if (writer)
        p.ws[(base + ks_first) * V + idx] = tot;
    __threadfence();
    __syncwarp();
    unsigned old = 0;
    if (lane == 0)
        old = atomicAdd(&p.tickets[g], 1u);
    old = __shfl_sync(0xffffffffu, old, 0);
    // contributors: the non-empty warp ranges that meet [base, base + S), walked in
    // k order (a warp with an empty range owns no unit and never arrives)
    unsigned contributors = 0;
    for (int64_t pos = base; pos < base + p.S; pos = unit_start(p, warp_of_unit(p, pos) + 1))
        ++contributors;
    if (old == contributors - 1) {
        __threadfence();
        if (writer) {
            float s = 0.f;
            for (int64_t pos = base; pos < base + p.S;
                 pos = unit_start(p, warp_of_unit(p, pos) + 1))
                s += __ldcg(&p.ws[pos * V + idx]);
            if (valid)
                p.y[(int64_t)(p.m0 + m) * p.ldy + n] = f32_to_bf16_bits(s);
        }
        if (lane == 0)
            p.tickets[g] = 0u;
    }
    (void)my_warp;
}

template <int WK, int MT, int RW>
__global__ void __launch_bounds__(GEMV_THREADS) q4_stream_kernel(GemvParams p)
{
    extern __shared__ __align__(16) unsigned char smem[];
    constexpr int COLS = Kind<WK>::COLS;
    const int lane = threadIdx.x & 31;
    const int64_t gw = (int64_t)blockIdx.x * GEMV_WARPS + (threadIdx.x >> 5);
    const int64_t u0 = unit_start(p, gw);
    const int64_t u1 = unit_start(p, gw + 1);
    const int Kpad = p.S * Kind<WK>::KSTEP;
    uint16_t *xs = reinterpret_cast<uint16_t *>(smem);
    float *cf = reinterpret_cast<float *>(smem + (size_t)MT * Kpad * 2);  // 16-byte aligned

    UnitRegs<RW> A, B;
    if (u0 < u1)
        load_unit<WK, RW>(p, u0, lane, A);          // weights do not depend on the
    float gsc = 1.f;                                 // previous kernel
    if constexpr (WK == W_NVFP4_A16 || WK == W_NVFP4_A8)
        gsc = __ldg(p.gscale);
    pdl_launch_dependents();
    pdl_wait();
    stage_x<WK, MT>(p, Kpad, xs, cf, (int)threadIdx.x, GEMV_THREADS);
    __syncthreads();
    (void)COLS;

    float acc[RW][MT];
#pragma unroll
    for (int r = 0; r < RW; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m)
            acc[r][m] = 0.f;
    int64_t seg_first = u0;

    auto step = [&](const UnitRegs<RW> &R, int64_t u) {
        const int64_t g = u / p.S;
        const int ks = (int)(u - g * p.S);
        compute_unit<WK, MT, RW>(p, R, ks, lane, Kpad, xs, cf, gsc, acc);
        if (ks == p.S - 1 || u + 1 == u1) {
            const int ksf = (int)(seg_first - g * p.S);
            finish_row_group<MT, RW>(p, g, ksf, ks, gw, lane, acc);
#pragma unroll
            for (int r = 0; r < RW; ++r)
#pragma unroll
                for (int m = 0; m < MT; ++m)
                    acc[r][m] = 0.f;
            seg_first = u + 1;
        }
    };

    for (int64_t u = u0; u < u1; u += 2) {
        if (u + 1 < u1)
            load_unit<WK, RW>(p, u + 1, lane, B);
        step(A, u);
        if (u + 1 >= u1)
            break;
        if (u + 2 < u1)
            load_unit<WK, RW>(p, u + 2, lane, A);
        step(B, u + 1);
    }
}

// ------------------------------------------------------------------ host side
template <int WK, int MT, int RW>
static const void *kernel_ptr()
{
    return reinterpret_cast<const void *>(&q4_stream_kernel<WK, MT, RW>);
}

static const void *select_kernel(int kind, int mt, int rw)
{
#define Q4_K(WK)                                                         \
    if (kind == WK) {                                                    \
        if (mt == 1 && rw == 4) return kernel_ptr<WK, 1, 4>();           \
        if (mt == 1 && rw == 8) return kernel_ptr<WK, 1, 8>();           \
        if (mt == 2 && rw == 4) return kernel_ptr<WK, 2, 4>();           \
        if (mt == 2 && rw == 8) return kernel_ptr<WK, 2, 8>();           \
        if (mt == 4 && rw == 4) return kernel_ptr<WK, 4, 4>();           \
        if (mt == 4 && rw == 8) return kernel_ptr<WK, 4, 8>();           \
    }
    Q4_K(W_INT4)
    Q4_K(W_NVFP4_A16)
    Q4_K(W_NVFP4_A8)
    Q4_K(W_BF16)
#undef Q4_K
    if (kind == W_BF16) {
        if (mt == 1 && rw == 1) return kernel_ptr<W_BF16, 1, 1>();
        if (mt == 1 && rw == 2) return kernel_ptr<W_BF16, 1, 2>();
        if (mt == 2 && rw == 1) return kernel_ptr<W_BF16, 2, 1>();
        if (mt == 2 && rw == 2) return kernel_ptr<W_BF16, 2, 2>();
        if (mt == 4 && rw == 1) return kernel_ptr<W_BF16, 4, 1>();
        if (mt == 4 && rw == 2) return kernel_ptr<W_BF16, 4, 2>();
    }
    return nullptr;
}

static int kstep_of(int kind) { return kind == W_BF16 ? 256 : 1024; }

static size_t smem_bytes(int kind, int mt, int S)
{
    const size_t Kpad = (size_t)S * kstep_of(kind);
    const size_t ch = kind == W_INT4 ? 4 : (kind == W_BF16 ? 0 : 1);
    return (size_t)mt * Kpad * 2 + (size_t)mt * (Kpad / 32) * ch * 4;
}

q4_status gemv_plan(const DeviceInfo &dev, int kind, int M, int N, int K, GemvPlan &plan)
{
    plan = GemvPlan{};
    plan.kind = kind;
    plan.S = (K + kstep_of(kind) - 1) / kstep_of(kind);
    int mt = M >= 4 ? 4 : (M >= 2 ? 2 : 1);
    while (mt > 1 && smem_bytes(kind, mt, plan.S) > dev.smem_optin)
        mt /= 2;
    if (smem_bytes(kind, mt, plan.S) > dev.smem_optin)
        return fail(Q4_ERR_SHAPE, "K=%d too large for the streaming kernel's x staging", K);
    plan.mt = mt;
    if (kind == W_BF16) {
        // whole rows per warp (no workspace): the fewest rows per unit that still
        // give every warp of a full grid at least one unit
        const int64_t warps = (int64_t)dev.sms * GEMV_WARPS * 2;
        plan.rw = N >= 8 * warps ? 8 : (N >= 4 * warps ? 4 : (N >= 2 * warps ? 2 : 1));
        plan.gran = plan.S;
    } else {
        // 8 rows per unit when that still gives every SM several units; else 4
        const int64_t units8 = (int64_t)((N + 7) / 8) * plan.S;
        plan.rw = (units8 >= (int64_t)dev.sms * GEMV_WARPS * 2) ? 8 : 4;
        plan.gran = 1;
    }
    plan.G = (N + plan.rw - 1) / plan.rw;
    plan.U = (int64_t)plan.G * plan.S;
    plan.smem = smem_bytes(kind, mt, plan.S);
    const void *k = select_kernel(kind, plan.mt, plan.rw);
    if (!k)
        return fail(Q4_ERR_ARG, "no streaming kernel for kind %d", kind);
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)plan.smem);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaFuncSetAttribute(streaming kernel)");
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, GEMV_THREADS, plan.smem);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
    if (per_sm < 1)
        return fail(Q4_ERR_SHAPE, "streaming kernel does not fit on an SM (smem %zu)", plan.smem);
    const int64_t max_blocks = (int64_t)per_sm * dev.sms;
    const int64_t want = (plan.U / plan.gran + GEMV_WARPS - 1) / GEMV_WARPS;
    plan.grid = (int)(want < max_blocks ? want : max_blocks);
    const bool split = plan.gran == 1 && plan.S > 1;
    plan.ws_floats = split ? (size_t)plan.U * plan.rw * plan.mt : 0;
    plan.tickets = split ? (size_t)plan.G : 0;
    return Q4_OK;
}

q4_status gemv_launch(const GemvPlan &plan, GemvParams p, int M, cudaStream_t stream, bool pdl)
{
    const void *k = select_kernel(plan.kind, plan.mt, plan.rw);
    p.S = plan.S;
    p.G = plan.G;
    p.U = plan.U;
    p.gran = plan.gran;
    p.TW = (int64_t)plan.grid * GEMV_WARPS;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    for (int m0 = 0; m0 < M; m0 += plan.mt) {
        p.m0 = m0;
        p.mcount = (M - m0) < plan.mt ? (M - m0) : plan.mt;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)plan.grid);
        cfg.blockDim = dim3(GEMV_THREADS);
        cfg.dynamicSmemBytes = plan.smem;
        cfg.stream = stream;
        cfg.attrs = pdl ? attr : nullptr;
        cfg.numAttrs = pdl ? 1 : 0;
        void *args[] = {&p};
        cudaError_t e = cudaLaunchKernelExC(&cfg, k, args);
        if (e != cudaSuccess)
            return cuda_fail(e, "launch of the streaming kernel");
    }
    return Q4_OK;
}

}  // namespace q4
