// Bulk-copy (TMA engine) weight-streaming kernel for sm_103a: the decode GEMV of
// both 4-bit layouts for one to four tokens, and the restricted BF16 head.
//
// Same arithmetic as the register-path kernel in gemv.cu (stream_common.cuh:
// prescaled fp16 x, shift-free E2M1 / fp16-magic int4 decode, fp32 accumulation
// by mixed-precision FMAs); what differs is the data movement.
//
//   * Each CTA owns a contiguous range of output rows with their full K, so its
//     share of the packed matrix is one contiguous block.  One producer thread
//     streams it with a few large cp.async.bulk copies per stage (codes, scales,
//     mins: each a contiguous run of rows) into a ring of shared-memory stages.
//     Weights do not depend on the previous kernel, so under programmatic
//     dependent launch the ring (~100 KB, most of a CTA's share) fills while the
//     previous kernel is still running.
//   * x is staged once per CTA in shared memory (stream_common.cuh); consumer warp
//     w owns ONE k-step ks = w % S (1024 4-bit or 256 bf16 columns) and holds its
//     32 (8) x values in registers for the whole kernel; per stage
//     it reads only codes and scales from shared memory for its RPW rows, reduces
//     each row across lanes and parks the per-k-step partial in shared memory.
//     (A warp owning whole rows re-read x for every row: four times the shared
//     memory traffic of the weights themselves, which capped the kernel.)
//   * A final pass sums each row's S partials in k order and stores bf16.  No
//     row is split between CTAs: no workspace, deterministic results.
//
// Synchronisation: per ring slot a "full" mbarrier (producer arrive + bytes of the
// copies) and an "empty" mbarrier (one arrive per consumer warp).  Every wait is
// bounded (mbar_wait) and reports a timeout in the library's device error word.
//
// Eligibility: every copy must start on a 16-byte boundary and be a multiple of
// 16 bytes: int4 K % 1024 == 0, NVFP4 K % 256 == 0, bf16 H % 8 == 0, 16-byte
// aligned scale/min arrays; at most 16 k-steps.  Other shapes use the register
// path.
#include "q4_device.cuh"
#include "q4_internal.h"
#include "stream_common.cuh"

namespace q4 {

__device__ unsigned g_q4_device_error;

// Phase timestamps per CTA (globaltimer ns) for builds with -DQ4_TRACE: kernel
// start, producer done issuing, consumers past griddepcontrol.wait, x staged,
// first stage landed, last stage landed, end.  Not compiled by default.
#ifdef Q4_TRACE
__device__ unsigned long long g_q4_trace[1024 * 40];
__device__ __forceinline__ unsigned long long q4_now()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}
#define Q4_TRACE_AT(slot) g_q4_trace[blockIdx.x * 40 + (slot)] = q4_now()
extern "C" int q4_trace_copy(unsigned long long *host, int n)
{
    return (int)cudaMemcpyFromSymbol(host, g_q4_trace, sizeof(unsigned long long) * n);
}
#else
#define Q4_TRACE_AT(slot) ((void)0)
#endif

// Rows per consumer warp and stage; 0 lets the planner choose (tuning builds).
#ifndef Q4_BULK_RPW
#define Q4_BULK_RPW 0
#endif

constexpr int BK_MAX_C = 16;                        // consumer warps at most
constexpr int BK_MAX_THREADS = (BK_MAX_C + 1) * 32; // + one producer warp
constexpr int BK_BAR_BYTES = 1024;                  // room for 2 x 64 mbarriers
constexpr int BK_MAX_NST = 48;

// Bytes of one row of each array in shared memory (all multiples of 16 for
// eligible shapes): packed codes, then scales, then mins.
struct BulkRow {
    int code, scale, minv;
    __host__ __device__ int total() const { return code + scale + minv; }
};

__host__ __device__ inline BulkRow bulk_row(int kind, int K)
{
    BulkRow r;
    r.code = kind == W_BF16 ? K * 2 : K / 2;
    r.scale = kind == W_INT4 ? (K / 128) * 2 : (kind == W_NVFP4_A16 ? K / 16 : 0);
    r.minv = kind == W_INT4 ? (K / 128) * 2 : 0;
    return r;
}

__device__ __forceinline__ void consumer_barrier(int threads)
{
    asm volatile("bar.sync 1, %0;" ::"r"(threads) : "memory");
}

__device__ __forceinline__ uint32_t lds_u16(const unsigned char *p)
{
    return *reinterpret_cast<const unsigned short *>(p);
}

// Copy logical rows [a, a + cnt) of one array (row stride `stride` bytes, `bytes`
// copied per row) into consecutive rows of shared memory.  Logical rows map to
// physical rows row_begin + n, except the optional extra row after n_rows, so a
// range is at most two contiguous runs.
__device__ __forceinline__ void copy_rows(const GemvParams &p, const uint8_t *base,
                                          int64_t stride, int bytes, int64_t a, int cnt,
                                          uint32_t dst, uint32_t bar)
{
    const int64_t main_end = (int64_t)p.n_rows;
    const int64_t run = (a + cnt <= main_end) ? cnt : (a < main_end ? main_end - a : 0);
    if (run > 0)
        bulk_copy_g2s(dst, base + ((int64_t)p.row_begin + a) * stride,
                      (uint32_t)(run * bytes), bar);
    if (run < cnt)   // the extra row (only the last logical row can be it)
        bulk_copy_g2s(dst + (uint32_t)(run * bytes), base + (int64_t)p.extra_row * stride,
                      (uint32_t)bytes, bar);
}

template <int WK, int MT, int RPW>
__global__ void __launch_bounds__(BK_MAX_THREADS, MT == 1 ? 2 : 1) q4_bulk_kernel(GemvParams p)
{
    extern __shared__ __align__(128) unsigned char smem[];
    constexpr int KSTEP = Kind<WK>::KSTEP;
    constexpr int COLS = Kind<WK>::COLS;
    constexpr int XV = (WK == W_BF16) ? 4 : 16;      // x registers per token
    const int C = p.consumers;                       // consumer warps = S * G
    const int G = C / p.S;                           // warps per k-step
    const int SR = G * RPW;                          // rows per stage
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const BulkRow rb = bulk_row(WK, p.K);
    const int slot_bytes = SR * rb.total();
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);   // full[nst], empty[nst]
    unsigned char *slots = smem + BK_BAR_BYTES;
    constexpr int CH = Kind<WK>::CH;
    const int Kpad = p.S * KSTEP;
    uint16_t *xs = reinterpret_cast<uint16_t *>(slots + (size_t)p.nst * slot_bytes);
    float *cf = reinterpret_cast<float *>(reinterpret_cast<unsigned char *>(xs) +
                                          (size_t)MT * Kpad * 2);
    float *red = cf + (size_t)MT * (Kpad / 32) * CH;        // [row][ks][m] partials
    const int64_t n0 = (int64_t)blockIdx.x * p.N / p.grid;
    const int64_t n1 = ((int64_t)blockIdx.x + 1) * p.N / p.grid;
    const int stages = (int)((n1 - n0 + SR - 1) / SR);

    if (threadIdx.x == 0) {
        for (int i = 0; i < p.nst; ++i) {
            mbar_init(smem_u32(&bars[i]), 1);
            mbar_init(smem_u32(&bars[p.nst + i]), C);
        }
        mbar_init_fence();
        Q4_TRACE_AT(0);
    }
    __syncthreads();

    if (warp == C) {
        // ---------------------------------------------------------- producer
        // Weights and scales do not depend on the previous kernel: they are
        // streamed before (and while) that kernel finishes under PDL.
        pdl_launch_dependents();
        if (lane == 0) {
            for (int i = 0; i < stages; ++i) {
                const int slot = i % p.nst;
                const int use = i / p.nst;
                if (use > 0 && !mbar_wait(smem_u32(&bars[p.nst + slot]), (use - 1) & 1, p.err))
                    break;
                const int64_t a = n0 + (int64_t)i * SR;
                const int cnt = (int)(n1 - a < SR ? n1 - a : SR);
                const uint32_t full = smem_u32(&bars[slot]);
                const uint32_t dst = smem_u32(slots + (size_t)slot * slot_bytes);
                mbar_arrive_expect_tx(full, (uint32_t)cnt * rb.total());
                if (i < 16) Q4_TRACE_AT(24 + i);
                copy_rows(p, p.w, p.w_row_bytes, rb.code, a, cnt, dst, full);
                if (rb.scale)
                    copy_rows(p, static_cast<const uint8_t *>(p.scale), rb.scale, rb.scale, a,
                              cnt, dst + SR * rb.code, full);
                if (rb.minv)
                    copy_rows(p, reinterpret_cast<const uint8_t *>(p.minv), rb.minv, rb.minv, a,
                              cnt, dst + SR * (rb.code + rb.scale), full);
            }
            Q4_TRACE_AT(1);
        }
        return;
    }

    // -------------------------------------------------------------- consumers
    const int ks = warp % p.S;
    const int g = warp / p.S;
    const int col0 = ks * KSTEP + lane * COLS;
    const bool colok = col0 < p.K;
    float gsc = 1.f;
    if constexpr (WK == W_NVFP4_A16)
        gsc = __ldg(p.gscale);                   // a weight-side constant
    pdl_launch_dependents();
    pdl_wait();                                   // x comes from the previous kernel
    if (threadIdx.x == 0) Q4_TRACE_AT(2);
    // x is staged once per CTA (prescaled fp16 + chunk data), then every warp
    // keeps its k-step's slice in registers for the whole kernel
    stage_x<WK, MT>(p, Kpad, xs, cf, (int)threadIdx.x, C * 32);
    consumer_barrier(C * 32);
    if (threadIdx.x == 0) Q4_TRACE_AT(3);
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

    // per-lane partials of NB consecutive stages are reduced across lanes together
    constexpr int PV = RPW * MT;
    constexpr int NB = PV >= 8 ? 1 : 8 / PV;
    float pbuf[NB * PV];
#pragma unroll
    for (int v = 0; v < NB * PV; ++v)
        pbuf[v] = 0.f;
    const int rows_cta = (int)(n1 - n0);

    for (int i = 0; i < stages; ++i) {
        const int slot = i % p.nst;
        const int use = i / p.nst;
        if (!mbar_wait(smem_u32(&bars[slot]), use & 1, p.err))
            break;
        if (threadIdx.x == 0 && i == 0) Q4_TRACE_AT(4);
        if (threadIdx.x == 0 && i == stages - 1) Q4_TRACE_AT(5);
        if (threadIdx.x == 0 && i < 16) Q4_TRACE_AT(8 + i);
        const int64_t a = n0 + (int64_t)i * SR;
        const int cnt = (int)(n1 - a < SR ? n1 - a : SR);
        const unsigned char *sl = slots + (size_t)slot * slot_bytes;
        const unsigned char *scb = sl + SR * rb.code;
        const unsigned char *mnb = scb + SR * rb.scale;
        uint4 q[RPW];
        uint32_t sw[RPW];
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            const int lr = g + G * r;
            q[r] = make_uint4(0u, 0u, 0u, 0u);
            sw[r] = 0u;
            if (lr < cnt && colok) {
                q[r] = *reinterpret_cast<const uint4 *>(sl + (size_t)lr * rb.code +
                                                        (size_t)ks * 512 + lane * 16);
                if constexpr (WK == W_INT4)
                    sw[r] = lds_u16(scb + lr * rb.scale + 2 * (col0 / 128)) |
                            (lds_u16(mnb + lr * rb.minv + 2 * (col0 / 128)) << 16);
                else if constexpr (WK == W_NVFP4_A16)
                    sw[r] = lds_u16(scb + lr * rb.scale + col0 / 16);
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_u32(&bars[p.nst + slot]));

        const int bslot = i % NB;
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            const uint32_t w4[4] = {q[r].x, q[r].y, q[r].z, q[r].w};
            float part[MT];
            if constexpr (WK == W_BF16) {
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    float t = 0.f;
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        t = fma2_bf16(t, w4[j], xr[m][j]);
                    part[m] = t;
                }
            } else if constexpr (WK == W_INT4) {
                float A1[MT], A2[MT];
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    A1[m] = 0.f;
                    A2[m] = 0.f;
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t w8 = w4[j] >> 8;
                    const uint32_t pa = int4_pair_f16_biased<0x000F000Fu>(w4[j]);   // cols 0, 4
                    const uint32_t pb = int4_pair_f16_biased<0x00F000F0u>(w4[j]);   // cols 1, 5
                    const uint32_t pc = int4_pair_f16_biased<0x000F000Fu>(w8);      // cols 2, 6
                    const uint32_t pd = int4_pair_f16_biased<0x00F000F0u>(w8);      // cols 3, 7
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        A1[m] = fma2_f16(A1[m], pa, xr[m][4 * j + 0]);
                        A2[m] = fma2_f16(A2[m], pb, xr[m][4 * j + 1]);
                        A1[m] = fma2_f16(A1[m], pc, xr[m][4 * j + 2]);
                        A2[m] = fma2_f16(A2[m], pd, xr[m][4 * j + 3]);
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
                    part[m] = t * cd[m].x;
                }
            } else {
                float Ta[MT], Tb[MT];
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    Ta[m] = 0.f;
                    Tb[m] = 0.f;
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t h[4];
                    e2m1x8_to_f16x2x4(w4[j], h);
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
                const uint32_t s2 = e4m3x2_to_f16x2(sw[r]);
                const float sa = f16lo_to_f32(s2);
                const float sb = f16hi_to_f32(s2);
#pragma unroll
                for (int m = 0; m < MT; ++m)
                    part[m] = fmaf(Ta[m], sa, Tb[m] * sb) * cd[m].x;
            }
#pragma unroll
            for (int m = 0; m < MT; ++m) {
#pragma unroll
                for (int bb = 0; bb < NB; ++bb)
                    if (bb == bslot)
                        pbuf[(bb * RPW + r) * MT + m] = part[m];
            }
        }
        // every NB stages (and at the end): one transposed lane reduction of the
        // buffered partials, parked per k-step in shared memory
        if (bslot == NB - 1 || i == stages - 1) {
            int idx = 0;
            const float tot = warp_sum_transpose<NB * PV>(pbuf, lane, idx);
            const int bi = idx / PV;
            const int r = (idx / MT) % RPW;
            const int m = idx % MT;
            const int stage = i - bslot + bi;
            const int lr = g + G * r;
            const int row = stage * SR + lr;
            if ((lane & (32 / (NB * PV) - 1)) == 0 && bi <= bslot && row < rows_cta)
                red[((size_t)row * p.S + ks) * MT + m] = tot;
#pragma unroll
            for (int v = 0; v < NB * PV; ++v)
                pbuf[v] = 0.f;
        }
    }

    // ------------------------------------------- sum the k-step partials, store
    consumer_barrier(C * 32);
    const int rows = (int)(n1 - n0);
    for (int e = (int)threadIdx.x; e < rows * MT; e += C * 32) {
        const int row = e / MT, m = e - (e / MT) * MT;
        float s = 0.f;
        for (int k = 0; k < p.S; ++k)
            s += red[((size_t)row * p.S + k) * MT + m];
        if (m < p.mcount)
            p.y[(int64_t)(p.m0 + m) * p.ldy + n0 + row] = f32_to_bf16_bits(s);
    }
    if (threadIdx.x == 0) Q4_TRACE_AT(6);
}

// ------------------------------------------------------------------ host side
template <int WK, int MT, int RPW>
static const void *bulk_ptr()
{
    return reinterpret_cast<const void *>(&q4_bulk_kernel<WK, MT, RPW>);
}

template <int WK>
static const void *bulk_select_kind(int mt, int rpw)
{
#define Q4_B(MT_, R_) if (mt == MT_ && rpw == R_) return bulk_ptr<WK, MT_, R_>();
    Q4_B(1, 1) Q4_B(1, 2) Q4_B(1, 4) Q4_B(2, 1) Q4_B(2, 2) Q4_B(2, 4)
    Q4_B(4, 1) Q4_B(4, 2) Q4_B(4, 4)
#undef Q4_B
    return nullptr;
}

static const void *bulk_select(int kind, int mt, int rpw)
{
    if (kind == W_INT4) return bulk_select_kind<W_INT4>(mt, rpw);
    if (kind == W_NVFP4_A16) return bulk_select_kind<W_NVFP4_A16>(mt, rpw);
    if (kind == W_BF16) return bulk_select_kind<W_BF16>(mt, rpw);
    return nullptr;
}

bool bulk_eligible(int kind, int K)
{
    if (kind == W_INT4) return K % 1024 == 0 && K <= 16384;
    if (kind == W_NVFP4_A16) return K % 256 == 0 && K <= 16384;
    if (kind == W_BF16) return K % 8 == 0 && K <= 4096;
    return false;
}

unsigned *device_error_flags()
{
    static unsigned *addr[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return nullptr;
    if (!addr[dev]) {
        void *a = nullptr;
        if (cudaGetSymbolAddress(&a, g_q4_device_error) != cudaSuccess)
            return nullptr;
        addr[dev] = static_cast<unsigned *>(a);
    }
    return addr[dev];
}

q4_status bulk_plan(const DeviceInfo &dev, int kind, int M, int N, int K, BulkPlan &plan)
{
    plan = BulkPlan{};
    plan.kind = kind;
    const int kstep = kind == W_BF16 ? 256 : 1024;
    const int ch = kind == W_INT4 ? 4 : (kind == W_BF16 ? 0 : 1);
    plan.S = (K + kstep - 1) / kstep;
    if (plan.S > BK_MAX_C)
        return fail(Q4_ERR_SHAPE, "K=%d has more k-steps than the bulk kernel's warps", K);
    const int G = BK_MAX_C / plan.S;
    plan.consumers = G * plan.S;
    const size_t Kpad = (size_t)plan.S * kstep;
    const BulkRow rb = bulk_row(kind, K);
    // Keep one CTA's shared memory near half the SM so that, under programmatic
    // dependent launch, the next kernel's CTA streams its weights beside it; the
    // ring then holds most of a CTA's share of the matrix.
    const size_t budget = dev.smem_optin < 112 * 1024 ? dev.smem_optin : 112 * 1024;
    // rows per warp and stage: stages of at most ~20 KB
    int rpw = 1;
    while (rpw < 4 && (size_t)G * rpw * 2 * rb.total() <= 20 * 1024)
        rpw *= 2;
    if (Q4_BULK_RPW > 0)
        rpw = Q4_BULK_RPW;
    int mt = M >= 4 ? 4 : (M >= 2 ? 2 : 1);
    // one CTA per SM; more (in waves) only when a CTA's per-row partials would
    // not fit in 24 KB of shared memory
    auto grid_for = [&](int m) {
        const int64_t rows_limit = (24 * 1024) / ((int64_t)plan.S * m * 4);
        int64_t grid = N < dev.sms ? N : dev.sms;
        const int64_t need = ((int64_t)N + rows_limit - 1) / rows_limit;
        return need > grid ? need : grid;
    };
    auto fixed_for = [&](int m) {
        const int64_t rows_cap = ((int64_t)N + grid_for(m) - 1) / grid_for(m);
        return (size_t)BK_BAR_BYTES + (size_t)m * Kpad * 2 + (size_t)m * (Kpad / 32) * ch * 4 +
               (size_t)rows_cap * plan.S * m * 4;
    };
    const size_t slot = (size_t)G * rpw * rb.total();
    while (mt > 1 && fixed_for(mt) + 2 * slot > budget)
        mt /= 2;
    if (rpw * mt > 8)
        rpw = 8 / mt;
    const size_t slot2 = (size_t)G * rpw * rb.total();
    const size_t fixed = fixed_for(mt);
    if (fixed + slot2 > dev.smem_optin)
        return fail(Q4_ERR_SHAPE, "K=%d too large for the bulk streaming kernel", K);
    plan.mt = mt;
    plan.rpw = rpw;
    const int64_t grid = grid_for(mt);
    if (grid > 0x7fffffff)
        return fail(Q4_ERR_SHAPE, "N=%d too large", N);
    plan.grid = (int)grid;
    const int64_t rows_per_cta = ((int64_t)N + plan.grid - 1) / plan.grid;
    const int64_t stages = (rows_per_cta + (int64_t)G * rpw - 1) / ((int64_t)G * rpw);
    int64_t nst = budget > fixed + slot2 ? (int64_t)((budget - fixed) / slot2) : 1;
    if (nst < 2 && fixed + 2 * slot2 <= dev.smem_optin)
        nst = 2;     // double buffering beats co-residency under PDL
    if (nst > stages) nst = stages;
    if (nst > BK_MAX_NST) nst = BK_MAX_NST;
    if (nst < 1) nst = 1;
    plan.nst = (int)nst;
    plan.smem = fixed + (size_t)plan.nst * slot2;
    const void *k = bulk_select(kind, plan.mt, plan.rpw);
    if (!k)
        return fail(Q4_ERR_ARG, "no bulk kernel for kind %d (mt %d, rpw %d)", kind, mt, rpw);
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)plan.smem);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaFuncSetAttribute(bulk kernel)");
    plan.ws_floats = 0;
    plan.tickets = 0;
    return Q4_OK;
}

q4_status bulk_launch(const BulkPlan &plan, GemvParams p, int M, cudaStream_t stream, bool pdl)
{
    const void *k = bulk_select(plan.kind, plan.mt, plan.rpw);
    p.S = plan.S;
    p.grid = plan.grid;
    p.nst = plan.nst;
    p.consumers = plan.consumers;
    p.err = device_error_flags();
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    for (int m0 = 0; m0 < M; m0 += plan.mt) {
        p.m0 = m0;
        p.mcount = (M - m0) < plan.mt ? (M - m0) : plan.mt;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)plan.grid);
        cfg.blockDim = dim3((plan.consumers + 1) * 32);
        cfg.dynamicSmemBytes = plan.smem;
        cfg.stream = stream;
        cfg.attrs = pdl ? attr : nullptr;
        cfg.numAttrs = pdl ? 1 : 0;
        void *args[] = {&p};
        cudaError_t e = cudaLaunchKernelExC(&cfg, k, args);
        if (e != cudaSuccess)
            return cuda_fail(e, "launch of the bulk streaming kernel");
    }
    return Q4_OK;
}

}  // namespace q4
