// Bulk-copy (TMA engine) weight-streaming kernel for sm_103a: the decode GEMV of
// both 4-bit layouts for one to four tokens, and the restricted BF16 head.
//
// It computes exactly what the register-path kernel in gemv.cu computes (same
// decode and dot-product code, stream_common.cuh); what changes is how weights
// reach the SM.  Each CTA owns a contiguous range of output rows with their full
// K, so its share of the packed matrix is one contiguous block of memory.  One
// producer thread streams it with a few large cp.async.bulk copies per stage
// (codes, then scales and mins, each a contiguous run of rows) into a ring of
// shared-memory stages; a CTA keeps its whole share (or ~100 KB of it) in flight
// in the memory system at once.  Large copies matter: the TMA engine pays a
// fixed cost per request, so one copy per 512-byte row segment was several
// times slower than one per stage.
//
// Geometry: CTA c owns rows [c*N/grid, (c+1)*N/grid) (+-1 row of balance), in
// stages of SR = 8 * RW rows; consumer warp w decodes rows [w*RW, w*RW + RW) of a
// stage over every k-step (16 bytes of weights per lane and row each), finishes
// them (lane reduction, bf16 store) and releases the stage.  No row is split
// between CTAs, so this path needs no workspace.
//
// Synchronisation: per ring slot a "full" mbarrier (producer arrive + bytes of the
// copies) and an "empty" mbarrier (one arrive per consumer warp).  Every wait is
// bounded (mbar_wait) and reports a timeout in the library's device error word.
//
// Eligibility: every copy must start on a 16-byte boundary and be a multiple of
// 16 bytes: int4 K % 1024 == 0, NVFP4 K % 256 == 0, bf16 H % 8 == 0, 16-byte
// aligned scale/min arrays, and a stage of 8 rows must fit in shared memory.
// Other shapes use the register path.
#include "q4_device.cuh"
#include "q4_internal.h"
#include "stream_common.cuh"

namespace q4 {

__device__ unsigned g_q4_device_error;

constexpr int BK_C = 8;                      // consumer warps per CTA
constexpr int BK_THREADS = (BK_C + 1) * 32;  // + one producer warp
constexpr int BK_BAR_BYTES = 1024;           // room for 2 x 64 mbarriers
constexpr int BK_MAX_NST = 64;

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

__device__ __forceinline__ int64_t bulk_physical_row(const GemvParams &p, int64_t n)
{
    return n < p.n_rows ? (int64_t)p.row_begin + n : (int64_t)p.extra_row;
}

__device__ __forceinline__ void consumer_barrier()
{
    asm volatile("bar.sync 1, %0;" ::"r"(BK_C * 32) : "memory");
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

template <int WK, int MT, int RW>
__global__ void __launch_bounds__(BK_THREADS) q4_bulk_kernel(GemvParams p)
{
    extern __shared__ __align__(128) unsigned char smem[];
    constexpr int SR = BK_C * RW;
    constexpr int KSTEP = Kind<WK>::KSTEP;
    constexpr int COLS = Kind<WK>::COLS;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const BulkRow rb = bulk_row(WK, p.K);
    const int slot_bytes = SR * rb.total();
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);   // full[nst], empty[nst]
    unsigned char *slots = smem + BK_BAR_BYTES;
    const int Kpad = p.S * KSTEP;
    uint16_t *xs = reinterpret_cast<uint16_t *>(slots + (size_t)p.nst * slot_bytes);
    float *cf = reinterpret_cast<float *>(reinterpret_cast<unsigned char *>(xs) +
                                          (size_t)MT * Kpad * 2);
    const int64_t n0 = (int64_t)blockIdx.x * p.N / p.grid;
    const int64_t n1 = ((int64_t)blockIdx.x + 1) * p.N / p.grid;
    const int stages = (int)((n1 - n0 + SR - 1) / SR);

    if (threadIdx.x == 0) {
        for (int i = 0; i < p.nst; ++i) {
            mbar_init(smem_u32(&bars[i]), 1);
            mbar_init(smem_u32(&bars[p.nst + i]), BK_C);
        }
        mbar_init_fence();
    }
    __syncthreads();

    if (warp == BK_C) {
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
                copy_rows(p, p.w, p.w_row_bytes, rb.code, a, cnt, dst, full);
                if (rb.scale)
                    copy_rows(p, static_cast<const uint8_t *>(p.scale), rb.scale, rb.scale, a,
                              cnt, dst + SR * rb.code, full);
                if (rb.minv)
                    copy_rows(p, reinterpret_cast<const uint8_t *>(p.minv), rb.minv, rb.minv, a,
                              cnt, dst + SR * (rb.code + rb.scale), full);
            }
        }
        return;
    }

    // -------------------------------------------------------------- consumers
    pdl_launch_dependents();
    pdl_wait();                                   // x comes from the previous kernel
    stage_x<WK, MT>(p, Kpad, xs, cf, (int)threadIdx.x, BK_C * 32);
    consumer_barrier();
    float gsc = 1.f;
    if constexpr (WK == W_NVFP4_A16)
        gsc = __ldg(p.gscale);

    for (int i = 0; i < stages; ++i) {
        const int slot = i % p.nst;
        const int use = i / p.nst;
        if (!mbar_wait(smem_u32(&bars[slot]), use & 1, p.err))
            break;
        const int64_t a = n0 + (int64_t)i * SR;
        const int cnt = (int)(n1 - a < SR ? n1 - a : SR);
        const unsigned char *sl = slots + (size_t)slot * slot_bytes;
        const unsigned char *sc = sl + SR * rb.code;
        const unsigned char *mn = sc + SR * rb.scale;
        float acc[RW][MT];
#pragma unroll
        for (int r = 0; r < RW; ++r)
#pragma unroll
            for (int m = 0; m < MT; ++m)
                acc[r][m] = 0.f;
        for (int ks = 0; ks < p.S; ++ks) {
            const int col0 = ks * KSTEP + lane * COLS;
            UnitRegs<RW> R;
#pragma unroll
            for (int r = 0; r < RW; ++r) {
                const int srow = warp * RW + r;
                R.q[r] = make_uint4(0u, 0u, 0u, 0u);
                R.s[r] = 0u;
                if (srow < cnt && col0 < p.K) {
                    R.q[r] = *reinterpret_cast<const uint4 *>(
                        sl + (size_t)srow * rb.code + (size_t)ks * 512 + lane * 16);
                    if constexpr (WK == W_INT4)
                        R.s[r] = lds_u16(sc + srow * rb.scale + 2 * (col0 / 128)) |
                                 (lds_u16(mn + srow * rb.minv + 2 * (col0 / 128)) << 16);
                    else if constexpr (WK == W_NVFP4_A16)
                        R.s[r] = lds_u16(sc + srow * rb.scale + col0 / 16);
                }
            }
            compute_unit<WK, MT, RW>(p, R, ks, lane, Kpad, xs, cf, gsc, acc);
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_u32(&bars[p.nst + slot]));
        // lane reduction and bf16 store of this warp's rows of the stage
        if (warp * RW < cnt) {
            constexpr int V = RW * MT;
            float v[V];
#pragma unroll
            for (int r = 0; r < RW; ++r)
#pragma unroll
                for (int m = 0; m < MT; ++m)
                    v[r * MT + m] = acc[r][m];
            int idx = 0;
            const float tot = warp_sum_transpose<V>(v, lane, idx);
            const int r = idx / MT, m = idx - (idx / MT) * MT;
            const int srow = warp * RW + r;
            if ((lane & (32 / V - 1)) == 0 && srow < cnt && m < p.mcount)
                p.y[(int64_t)(p.m0 + m) * p.ldy + a + srow] = f32_to_bf16_bits(tot);
        }
    }
}

// ------------------------------------------------------------------ host side
template <int WK, int MT, int RW>
static const void *bulk_ptr()
{
    return reinterpret_cast<const void *>(&q4_bulk_kernel<WK, MT, RW>);
}

template <int WK>
static const void *bulk_select_kind(int mt, int rw)
{
#define Q4_B(MT_, RW_) if (mt == MT_ && rw == RW_) return bulk_ptr<WK, MT_, RW_>();
    Q4_B(1, 1) Q4_B(1, 2) Q4_B(1, 4)
    Q4_B(2, 1) Q4_B(2, 2) Q4_B(2, 4)
    Q4_B(4, 1) Q4_B(4, 2) Q4_B(4, 4)
#undef Q4_B
    return nullptr;
}

static const void *bulk_select(int kind, int mt, int rw)
{
    if (kind == W_INT4) return bulk_select_kind<W_INT4>(mt, rw);
    if (kind == W_NVFP4_A16) return bulk_select_kind<W_NVFP4_A16>(mt, rw);
    if (kind == W_BF16) return bulk_select_kind<W_BF16>(mt, rw);
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
    const int cols = kind == W_BF16 ? 8 : 32;
    plan.S = (K + kstep - 1) / kstep;
    const size_t Kpad = (size_t)plan.S * kstep;
    const BulkRow rb = bulk_row(kind, K);
    int mt = M >= 4 ? 4 : (M >= 2 ? 2 : 1);
    auto xbytes = [&](int m) { return (size_t)m * Kpad * 2 + (size_t)m * (Kpad / cols) * 4; };
    // keep one CTA's shared memory near half the SM so that, under programmatic
    // dependent launch, the next kernel's CTA can start streaming beside it
    const size_t budget = dev.smem_optin < 112 * 1024 ? dev.smem_optin : 112 * 1024;
    // rows per warp: stages of about 16 KB
    int rw = 1;
    while (rw < 4 && (size_t)BK_C * rw * 2 * rb.total() <= 16 * 1024)
        rw *= 2;
    auto need = [&](int m, int r) {
        return BK_BAR_BYTES + xbytes(m) + 2 * (size_t)BK_C * r * rb.total();
    };
    while (mt > 1 && need(mt, rw) > budget)
        mt /= 2;
    if (need(mt, rw) > dev.smem_optin)
        return fail(Q4_ERR_SHAPE, "K=%d too large for the bulk streaming kernel", K);
    plan.mt = mt;
    plan.rw = rw;
    plan.grid = N < dev.sms ? N : dev.sms;
    const int64_t rows_per_cta = ((int64_t)N + plan.grid - 1) / plan.grid;
    const int64_t stages = (rows_per_cta + BK_C * rw - 1) / (BK_C * rw);
    const size_t slot = (size_t)BK_C * rw * rb.total();
    const size_t fixed = BK_BAR_BYTES + xbytes(mt);
    int64_t nst = budget > fixed ? (int64_t)((budget - fixed) / slot) : 2;
    if (nst > stages) nst = stages;
    if (nst > BK_MAX_NST) nst = BK_MAX_NST;
    if (nst < 1) nst = 1;
    plan.nst = (int)nst;
    plan.smem = fixed + (size_t)plan.nst * slot;
    const void *k = bulk_select(kind, plan.mt, plan.rw);
    if (!k)
        return fail(Q4_ERR_ARG, "no bulk kernel for kind %d", kind);
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
    const void *k = bulk_select(plan.kind, plan.mt, plan.rw);
    p.S = plan.S;
    p.grid = plan.grid;
    p.nst = plan.nst;
    p.err = device_error_flags();
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    for (int m0 = 0; m0 < M; m0 += plan.mt) {
        p.m0 = m0;
        p.mcount = (M - m0) < plan.mt ? (M - m0) : plan.mt;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)plan.grid);
        cfg.blockDim = dim3(BK_THREADS);
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
