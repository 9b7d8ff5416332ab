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
//     dequantise them into the A operand tiles (fp16, K-major, 128-byte
//     swizzle): a thread takes 16 weights of one row per step, and a warp's code
//     reads are 256 contiguous bytes (no bank conflicts).  They also convert the
//     chunk's x tile in place from bf16 to fp16 (for large M a small kernel
//     converts x once per call instead).  int4: w = fp16(c * s + m) (one fused
//     multiply-add, single rounding); NVFP4: w = E2M1 * e4m3 in fp16, exact (the
//     global scale is applied in the epilogue).  An x value outside the fp16
//     range sets Q4_DEVERR_FP16_RANGE.
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
constexpr unsigned kErrFp16Range = 2u;

// Per-CTA timestamps (globaltimer ns) for builds with -DQ4_TRACE.  Ring kernel:
// slots 0..3 start, TMEM ready, final commit seen by the epilogue, end; 8+i
// producer issued stage i, 24+i workers (warp 2) finished stage i, 40+i MMA issued
// stage i; 56..60 warp 2's clock cycles summed over its stages: data waits, x
// conversion, dequant, proxy fence, warp sync + arrive.  Skinny kernel: 0, 1, 2,
// 3 as above, 4 / 6 / 7 / 61 x warps issued their copies / saw step 0 land / had
// step 0 ready / saw the last step land, 5 past the first cluster barrier; 24+s
// and 8+s the MMA thread past the A-full and x-ready waits of step s, 40+s its
// MMAs issued; 56..59 warp 2's cycles in the step's waits and stores.
#ifdef Q4_TRACE
__device__ unsigned long long g_q4_tc_trace[8 * 1024 * 64];   // 8 most recent calls
__device__ __forceinline__ unsigned long long tc_now()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}
#define TC_TRACE(slot) do { if ((slot) < 64 && blockIdx.x < 1024) g_q4_tc_trace[((p.call & 7) * 1024 + blockIdx.x) * 64 + (slot)] = tc_now(); } while (0)
#define TC_CLK(v) long long v = clock64()
#define TC_PHASE(slot, a, b) (tc_ph[(slot) - 56] += (b) - (a))
#define TC_PHASE_DECL long long tc_ph[5] = {0, 0, 0, 0, 0}
#define TC_PHASE_STORE() do { if (warp == 2 && lane == 0 && blockIdx.x < 1024) for (int q_ = 0; q_ < 5; ++q_) g_q4_tc_trace[((p.call & 7) * 1024 + blockIdx.x) * 64 + 56 + q_] = (unsigned long long)tc_ph[q_]; } while (0)
extern "C" int q4_tc_trace_copy(unsigned long long *host, int n)
{
    return (int)cudaMemcpyFromSymbol(host, g_q4_tc_trace, sizeof(unsigned long long) * n);
}
#else
#define TC_TRACE(slot) ((void)0)
#define TC_CLK(v) ((void)0)
#define TC_PHASE(slot, a, b) ((void)0)
#define TC_PHASE_DECL ((void)0)
#define TC_PHASE_STORE() ((void)0)
#endif

struct TcParams {
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
    int x_f16;                 // x already converted to fp16 (large M)
    int call;                  // launch index (phase-trace builds only)
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
__device__ __forceinline__ uint32_t idesc_f16(int n)
{
    return (1u << 4)                    // D format: f32
         | (0u << 7) | (0u << 10)       // A, B format: f16
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

__device__ __forceinline__ uint32_t f16x2_splat(uint32_t h16)
{
    return (h16 & 0xffffu) | (h16 << 16);
}

// Epilogue of both tensor-core kernels, run by the 16 worker warps (w = 0..15)
// once the final MMA commit has been seen (ok): read the accumulator back from
// TMEM (warp w reads lane quadrant (w + 2) % 4, a quarter of its columns),
// release warp 1 to free TMEM after the last read, then store bf16 y -- or, under
// split-K, fp32 partials that the last CTA of the tile to arrive sums in k order.
template <int LAYOUT>
__device__ __forceinline__ void tc_epilogue(const TcParams &p, uint32_t tmem_base, bool ok, int w,
                                            int lane, int n0, int m0, int tile, int ks,
                                            unsigned *last_flag)
{
    const int TN = p.TN;
    const int quad = (w + 2) & 3;            // TMEM lane quadrant of this warp
    const int grp = w >> 2;                  // column share of the quadrant
    const int r = quad * 32 + lane;          // TMEM lane = weight row within the tile
    const int n = n0 + r;
    const bool nok = n < p.N;
    float gsc = 1.f;
    if constexpr (LAYOUT == 1)
        gsc = __ldg(p.gscale);
    const int ncb = (TN + 16 * TC_GROUPS - 1) / (16 * TC_GROUPS);   // same for every worker
    for (int it = 0; it < ncb; ++it) {
        const int cb = grp * 16 + it * 16 * TC_GROUPS;
        uint32_t v[16];
        if (cb < TN)
            tmem_ld16(tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)cb, v);
        if (it == ncb - 1) {
            // last TMEM read done: let warp 1 free the accumulator now
            tc_fence_before();
            asm volatile("bar.arrive 3, %0;" ::"r"((TC_WORKERS + 1) * 32) : "memory");
        }
        if (!ok || cb >= TN)
            continue;
        if (p.KS == 1) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int m = m0 + cb + j;
                if (nok && m < p.M)
                    p.y[(int64_t)m * p.N + n] = f32_to_bf16_bits(__uint_as_float(v[j]) * gsc);
            }
        } else {
            float *dst = p.ws + ((size_t)(tile * p.KS + ks) * TN + cb) * TC_ROWS + r;
#pragma unroll
            for (int j = 0; j < 16; ++j)
                dst[(size_t)j * TC_ROWS] = __uint_as_float(v[j]);
        }
    }
    if (p.KS > 1) {
        // split-K: the last CTA of this tile to arrive sums the partials (every
        // worker reaches both barriers, whatever happened before)
        __threadfence();
        asm volatile("bar.sync 2, %0;" ::"r"(TC_WORKERS * 32) : "memory");
        if (w == 0 && lane == 0)
            *last_flag = (ok && atomicAdd(&p.tickets[tile], 1u) == (unsigned)(p.KS - 1)) ? 1u : 0u;
        asm volatile("bar.sync 2, %0;" ::"r"(TC_WORKERS * 32) : "memory");
        if (*last_flag) {
            __threadfence();
            // Each thread sums groups of four rows of one token column: all KS
            // partials of a group are loaded (16 bytes each) before the adds,
            // which run in k order, so the result does not depend on timing.
            const size_t kstride4 = (size_t)TN * TC_ROWS / 4;
            const float4 *part = reinterpret_cast<const float4 *>(
                p.ws + (size_t)tile * p.KS * TN * TC_ROWS);
            for (int g4 = w * 32 + lane; g4 < TN * (TC_ROWS / 4); g4 += TC_WORKERS * 32) {
                const int c = g4 / (TC_ROWS / 4), q = g4 % (TC_ROWS / 4);
                float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int k0 = 0; k0 < p.KS; k0 += 8) {
                    float4 v[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        if (k0 + j < p.KS)
                            v[j] = __ldcg(part + (k0 + j) * kstride4 + (size_t)c * (TC_ROWS / 4) + q);
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        if (k0 + j < p.KS) {
                            sum.x += v[j].x; sum.y += v[j].y;
                            sum.z += v[j].z; sum.w += v[j].w;
                        }
                }
                const int m = m0 + c;
                const int nb = n0 + 4 * q;
                if (m < p.M) {
                    uint16_t *yr = p.y + (int64_t)m * p.N;
                    const float o[4] = {sum.x, sum.y, sum.z, sum.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if (nb + i < p.N)
                            yr[nb + i] = f32_to_bf16_bits(o[i] * gsc);
                }
            }
            if (w == 0 && lane == 0)
                p.tickets[tile] = 0u;
        }
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

template <int LAYOUT, int SC, int G>   // LAYOUT 0 int4-g128, 1 NVFP4; G worker groups
__global__ void __launch_bounds__(TC_THREADS, 1)
q4_tc_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap,
             TcParams p)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int TN = p.TN;
    const int NS = p.ns;
    const uint32_t x_bytes = (uint32_t)TN * 128;
    const uint32_t x_stride = (x_bytes + 1023) & ~1023u;
    const uint32_t stage_bytes = TcStage<SC>::A + (uint32_t)SC * x_stride + TcStage<SC>::CODE;
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
    const int n0 = tile_n * TC_ROWS;
    const int m0 = tile_m * TN;
    // split-K on super-chunk boundaries
    const int sup_total = (p.chunks + SC - 1) / SC;
    const int u0 = (int)((int64_t)ks * sup_total / p.KS);
    const int u1 = (int)((int64_t)(ks + 1) * sup_total / p.KS);
    const int nsup = u1 - u0;
    const int c0 = u0 * SC;
    const int c1 = (u1 * SC) < p.chunks ? u1 * SC : p.chunks;

    if (threadIdx.x == 0) {
        TC_TRACE(0);
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
    if (threadIdx.x == 0) TC_TRACE(1);

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
                mbar_arrive_expect_tx(full, TcStage<SC>::CODE + (uint32_t)nv * x_bytes);
                // codes of the super-chunk: 128 rows x SC * 32 bytes in one copy
                tma_load_2d(smem_u32(st + TcStage<SC>::A + SC * x_stride), &wmap, kc * (TC_KC / 2),
                            n0, full);
                if (u == 0) {
                    TC_TRACE(61);
                    pdl_wait();                // x comes from the previous kernel
                    TC_TRACE(62);
                }
                for (int c = 0; c < nv; ++c)
                    tma_load_2d(smem_u32(st + TcStage<SC>::A + c * x_stride), &xmap, (kc + c) * TC_KC,
                                m0, full);
                TC_TRACE(8 + u);
                issued = u + 1;
            }
            // drain: every issued copy has landed before the CTA can exit
            for (int u = issued - NS > 0 ? issued - NS : 0; u < issued; ++u)
                mbar_wait(smem_u32(&bars[u % NS]), (u / NS) & 1, p.err);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------- MMA issue
        if (lane == 0) {
            const uint32_t idesc = idesc_f16(TN);
            for (int u = 0; u < nsup; ++u) {
                const int s = u % NS, use = u / NS;
                if (!mbar_wait(smem_u32(&bars[NS + s]), use & 1, p.err))
                    break;
                tc_fence_after();
                const int kc = c0 + u * SC;
                const int nv = (c1 - kc) < SC ? (c1 - kc) : SC;
                const uint32_t st = smem_u32(smem + (size_t)s * stage_bytes);
                const uint64_t ad = smem_desc_sw128(st);
                const uint64_t bd = smem_desc_sw128(st + TcStage<SC>::A);
                const uint32_t alo = (uint32_t)ad, ahi = (uint32_t)(ad >> 32);
                const uint32_t blo = (uint32_t)bd, bhi = (uint32_t)(bd >> 32);
#pragma unroll
                for (int c = 0; c < SC; ++c) {
                    if (c >= nv)
                        break;
#pragma unroll
                    for (int kk = 0; kk < TC_KC / 16; ++kk)
                        mma_f16_2(tmem_base, alo + (uint32_t)c * 1024u + 2u * kk, ahi,
                                  blo + (uint32_t)c * (x_stride >> 4) + 2u * kk, bhi, idesc,
                                  (u > 0 || c > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(smem_u32(&bars[2 * NS + s]));
                TC_TRACE(40 + u);
            }
            mma_commit(smem_u32(&bars[3 * NS]));
        }
        // free the accumulator as soon as every worker has read it back
        __syncwarp();
        asm volatile("bar.sync 3, %0;" ::"r"((TC_WORKERS + 1) * 32) : "memory");
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                     ::"r"(tmem_base), "r"(p.tmem_cols) : "memory");
        if (lane == 0) TC_TRACE(63);
    } else {
        // ------------------------------------------------------------- workers
        // G groups of WG = 16 / G warps take the stages in turn (group gi the
        // stages gi, gi + G, ...), so G stages are dequantised at once.
        // Dequant mapping inside a group: a warp reads 256 contiguous code bytes
        // per step (no bank conflicts): L = 4 SC lanes per code row, 32 / L rows per
        // step, STEPS = SC * G steps.  In step k a lane takes 16 weights: row
        // (128 / WG) wg + (32 / L) k + lane / L, chunk c = (lane % L) / 4, columns
        // 16 (lane % 4) .. + 15 of that chunk.
        constexpr int WG = TC_WORKERS / G;
        constexpr int L = 4 * SC;
        constexpr int RPS = 32 / L;
        constexpr int STEPS = SC * G;
        constexpr int SA = 4;                    // stages of scales loaded ahead
        const int w = warp - 2;                  // 0..15
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
            rowk[k] = (128 / WG) * wg + RPS * k + lane / L;
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
        uint32_t scq[SA][STEPS], mnq[SA][STEPS];
#pragma unroll
        for (int j = 0; j < SA; ++j)
#pragma unroll
            for (int k = 0; k < STEPS; ++k) {
                scq[j][k] = load_scale(gi + j * G, k, p.scale);
                mnq[j][k] = LAYOUT == 0 ? load_scale(gi + j * G, k, p.minv) : 0u;
            }
        bool range_bad = false;
        TC_PHASE_DECL;
        // one stage; false when a wait timed out
        auto stage = [&](int u, const uint32_t (&scs)[STEPS], const uint32_t (&mns)[STEPS]) -> bool {
                const int s = u % NS, use = u / NS;
                const int kc = c0 + u * SC;
                const int nv = (c1 - kc) < SC ? (c1 - kc) : SC;
                unsigned char *st = smem + (size_t)s * stage_bytes;
                TC_CLK(t0);
                if (!mbar_wait_warp(smem_u32(&bars[s]), use & 1, p.err))
                    return false;
                TC_CLK(t1);
                TC_PHASE(56, t0, t1);
                // x sub-tiles: bf16 -> fp16 in place (element-wise, swizzle-agnostic).
                // Only tiles of at most 64 tokens are converted here (larger M arrive
                // in fp16), so a thread has at most SC * G 16-byte vectors: the loop is
                // unrolled and interleaves with the code loads below.
                if (!p.x_f16) {
                    const int per = TN * 8;                  // vectors per sub-tile
    #pragma unroll
                    for (int j = 0; j < SC * G; ++j) {
                        const int v = wt + j * WG * 32;
                        if (v < nv * per) {
                            const int sub = (v >= per) + (v >= 2 * per) + (v >= 3 * per);
                            uint4 *xv = reinterpret_cast<uint4 *>(st + TcStage<SC>::A + sub * x_stride) +
                                        (v - sub * per);
                            const uint4 t = *xv;
                            const uint32_t e[4] = {t.x, t.y, t.z, t.w};
                            uint32_t o[4];
                            float mx = 0.f;
    #pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const float lo = bf16_bits_to_f32(e[q] & 0xffffu);
                                const float hi = bf16_bits_to_f32(e[q] >> 16);
                                mx = fmaxf(mx, fmaxf(fabsf(lo), fabsf(hi)));
                                __half2 h = __floats2half2_rn(lo, hi);
                                o[q] = *reinterpret_cast<uint32_t *>(&h);
                            }
                            if (mx >= 65520.f && mx <= 3.4e38f)
                                range_bad = true;
                            *xv = make_uint4(o[0], o[1], o[2], o[3]);
                        }
                    }
                }
                TC_CLK(t2);
                TC_PHASE(57, t1, t2);
                const unsigned char *codes = st + TcStage<SC>::A + SC * x_stride;
    #pragma unroll
                for (int k = 0; k < STEPS; ++k) {
                    const int rd = rowk[k];
                    const uint2 cw = *reinterpret_cast<const uint2 *>(codes + rd * (SC * 32) + cl * 8);
                    const uint32_t words[2] = {cw.x, cw.y};
                    unsigned char *arow = st + c * 16384 + rd * 128;
                    uint32_t sg = 0u;
                    if constexpr (LAYOUT == 1)
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
                TC_CLK(t3);
                TC_PHASE(58, t2, t3);
                fence_proxy_async();
                TC_CLK(t4);
                TC_PHASE(59, t3, t4);
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(smem_u32(&bars[NS + s]));
                TC_CLK(t5);
                TC_PHASE(60, t4, t5);
                if (warp == 2 && lane == 0) TC_TRACE(24 + u);
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
        TC_PHASE_STORE();
        if (range_bad && p.err)
            atomicOr(p.err, kErrFp16Range);

        // ------------------------------------------------------------ epilogue
        const bool ok = nsup > 0 && mbar_wait_warp(smem_u32(&bars[3 * NS]), 0, p.err);
        tc_fence_after();
        if (warp == 2 && lane == 0) TC_TRACE(2);
        __shared__ unsigned last_flag;
        tc_epilogue<LAYOUT>(p, tmem_base, ok, w, lane, n0, m0, tile_n * p.tiles_m + tile_m, ks,
                            &last_flag);
    }

    __syncthreads();
    if (threadIdx.x == 0) TC_TRACE(3);
}

// ------------------------------------------------------------ skinny kernel
// Batched decode (tiles of at most 64 tokens) reads few bytes of x per weight.
// The ring kernel above stages x, codes and A together through shared memory
// and issues every copy from one thread; for small tiles it is bound by that
// issue rate.  This kernel is built around three measured limits instead:
//   * copies issued by one thread do not overlap much; spread over several
//     warps they reach ~150 GB/s per SM from L2 and the SM's share of HBM.  So
//     the codes of the CTA's whole K range are requested at once (16 KB boxes)
//     before the dependency wait -- weights do not depend on the previous
//     kernel -- and eight x warps each request every eighth step of x after it;
//   * shared-memory bandwidth: the dequantised A tiles never touch shared
//     memory -- each worker writes its row of fp16 weights into tensor memory
//     (tcgen05.st) and the MMA reads A from there, through a ring of six
//     two-chunk slots;
//   * the split-K CTAs of one weight tile form a thread-block cluster: each dumps
//     its fp32 accumulator into its own shared memory, and after a cluster
//     barrier each sums 1/KS of the tile over the KS dumps (read through
//     distributed shared memory) in k order -- deterministic, no workspace.
__device__ __forceinline__ float4 ld_cluster_f4(uint32_t local_addr, uint32_t rank)
{
    uint32_t ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(local_addr), "r"(rank));
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(ra)
                 : "memory");
    return v;
}

__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// 16 codes (one row, 16 consecutive columns) -> 16 fp16 weights: int4
// w = c * s + min (one fused multiply-add, one rounding); NVFP4 w = E2M1 * e4m3,
// exact in fp16 (the global scale is applied in the epilogue).
template <int LAYOUT>
__device__ __forceinline__ void tc_decode16(uint2 cw, uint32_t sc, uint32_t (&o)[8])
{
    const uint32_t words[2] = {cw.x, cw.y};
    if constexpr (LAYOUT == 0) {
        const uint32_t s2 = f16x2_splat(sc & 0xffffu);
        const uint32_t m2 = f16x2_splat(sc >> 16);
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                // byte b -> (1024 + c_lo, 1024 + 16 c_hi) -> (c_lo, c_hi)
                const uint32_t t = prmt(words[j], 0u, (uint32_t)(b | (4 << 4) | (b << 8) | (4 << 12)));
                uint32_t v2;
                asm("lop3.b32 %0, %1, 0x00F0000F, 0x64006400, 0xEA;" : "=r"(v2) : "r"(t));
                v2 = hfma2(v2, 0x2C003C00u, 0xD400E400u);   // * (1, 1/16) + (-1024, -64)
                o[4 * j + b] = hfma2(v2, s2, m2);
            }
    } else {
        const uint32_t sg = f16x2_splat(e4m3x2_to_f16x2(sc & 0xffu) & 0xffffu);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            uint32_t h[4];
            e2m1x8_to_f16x2x4(words[j], h);
#pragma unroll
            for (int b = 0; b < 4; ++b)
                o[4 * j + b] = hmul2(h[b], sg);
        }
    }
}

constexpr int SK_XWARPS = 8;                          // x loading / conversion warps
constexpr int SK_THREADS = TC_THREADS + SK_XWARPS * 32;
constexpr int SK_NA = 6;                              // TMEM A slots of two chunks
constexpr int SK_TMEM_COLS = 512;                     // accumulator (<= 64) + A slots

// tcgen05.mma with the A operand in tensor memory (row i of A in lane i, its K
// values packed two per 32-bit column) and the B descriptor passed as two 32-bit
// halves, so that the issuing loop steps the start-address field (low half) by 2
// per 32 bytes instead of rebuilding a 64-bit descriptor per MMA.
__device__ __forceinline__ void mma_f16_tmem_a2(uint32_t tmem_d, uint32_t tmem_a, uint32_t b_lo,
                                                uint32_t b_hi, uint32_t idesc, uint32_t accumulate)
{
    asm volatile("{\n\t.reg .b64 bd;\n\t.reg .pred p;\n\t"
                 "setp.ne.u32 p, %5, 0;\n\t"
                 "mov.b64 bd, {%2, %3};\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], bd, %4, p;\n\t}"
                 ::"r"(tmem_d), "r"(tmem_a), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate)
                 : "memory");
}

// A warp writes 16 consecutive 32-bit columns of its 32 TMEM lanes (one row each).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
                 "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};"
                 ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]),
                   "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]),
                   "r"(v[13]), "r"(v[14]), "r"(v[15])
                 : "memory");
}

// Shared-memory layout of the skinny kernel (offsets from the 1024-aligned base):
// [x tiles: nch x TN x 128 B][code boxes: ceil(nch / 4) x 128 rows x 128 B][barriers],
// both in the 128-byte swizzle (16-byte unit u of row r stored at u ^ (r % 8)).
// After the final MMA the split-K dump of the accumulator (TN x 128 fp32) reuses
// the start.
struct SkLayout {
    int nch, nstep, nbox;
    uint32_t x_bytes, codes_off, bars_off;
    __host__ __device__ SkLayout(int TN, int nch_)
    {
        nch = nch_;
        nstep = (nch + 1) / 2;                          // steps of two chunks
        nbox = (nch + 3) / 4;                           // code boxes of four chunks
        x_bytes = (uint32_t)TN * 128;
        codes_off = (uint32_t)nch * x_bytes;
        const uint32_t data = codes_off + (uint32_t)nbox * 16384u;
        const uint32_t dump = (uint32_t)TN * TC_ROWS * 4;
        bars_off = ((data > dump ? data : dump) + 7u) & ~7u;
    }
    // barriers: cfull[nbox], xfull[nstep], xready[nstep], afull, aempty, done
    __host__ __device__ uint32_t bytes() const
    {
        return bars_off + (uint32_t)(nbox + 2 * nstep + 2 * SK_NA + 1) * 8 + 16;
    }
};

template <int LAYOUT>
__global__ void __launch_bounds__(SK_THREADS, 1)
q4_tc_skinny_kernel(const __grid_constant__ CUtensorMap xmap,
                    const __grid_constant__ CUtensorMap wmap, TcParams p)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int TN = p.TN;
    const int tile = blockIdx.x / p.KS;
    const int ks = blockIdx.x - tile * p.KS;            // rank within the cluster
    const int n0 = tile * TC_ROWS;
    const int c0 = (int)((int64_t)ks * p.chunks / p.KS);
    const SkLayout L(TN, (int)((int64_t)(ks + 1) * p.chunks / p.KS) - c0);
    const int nch = L.nch, nstep = L.nstep, nbox = L.nbox;
    const uint32_t x_bytes = L.x_bytes;
    unsigned char *xs = smem;
    unsigned char *cs = smem + L.codes_off;
    uint64_t *cfull = reinterpret_cast<uint64_t *>(smem + L.bars_off);   // per code box
    uint64_t *xfull = cfull + nbox;
    uint64_t *xready = xfull + nstep;
    uint64_t *afull = xready + nstep;
    uint64_t *aempty = afull + SK_NA;
    uint64_t *done = aempty + SK_NA;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        TC_TRACE(0);
        for (int i = 0; i < nbox; ++i)
            mbar_init(smem_u32(&cfull[i]), 1);
        for (int st = 0; st < nstep; ++st) {
            mbar_init(smem_u32(&xfull[st]), 1);
            mbar_init(smem_u32(&xready[st]), SK_XWARPS);
        }
        for (int i = 0; i < SK_NA; ++i) {
            mbar_init(smem_u32(&afull[i]), TC_WORKERS);
            mbar_init(smem_u32(&aempty[i]), 1);
        }
        mbar_init(smem_u32(done), 1);
        mbar_init_fence();
        // The codes of the whole K range, requested at once and before the
        // dependency wait (weights do not depend on the previous kernel): boxes
        // of four chunks, 128 rows x 128 bytes, rows beyond N zero-filled.
        for (int b = 0; b < nbox; ++b) {
            mbar_arrive_expect_tx(smem_u32(&cfull[b]), 16384u);
            tma_load_2d(smem_u32(cs + (size_t)b * 16384), &wmap, (c0 + 4 * b) * (TC_KC / 2), n0,
                        smem_u32(&cfull[b]));
        }
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(tmem_slot)), "r"(SK_TMEM_COLS) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    if (threadIdx.x == 0) TC_TRACE(1);
    float gsc = 1.f;                                    // read before the dependency wait:
    if constexpr (LAYOUT == 1)                          // the global scale is a weight
        gsc = __ldg(p.gscale);

    if (warp == 0) {
        // ---------------------------------------------- launch the next kernel early
        pdl_launch_dependents();
    } else if (warp == 1) {
        // ------------------------------------------------------------- MMA issue
        // accumulator in TMEM columns 0 .. TN-1; A slot i in columns 64 + 64 i
        // (chunk h of the step at + 32 h, k-step kk at + 8 kk)
        if (lane == 0) {
            const uint32_t idesc = idesc_f16(TN);
            int sl = 0;
            uint32_t ph = 0;
            for (int s = 0; s < nstep; ++s) {
                if (!mbar_wait(smem_u32(&afull[sl]), ph, p.err))
                    break;
                if (s < 16) TC_TRACE(24 + s);
                if (!mbar_wait(smem_u32(&xready[s]), 0, p.err))
                    break;
                if (s < 16) TC_TRACE(8 + s);
                tc_fence_after();
                const uint32_t a = tmem_base + 64u + 64u * (uint32_t)sl;
                const uint64_t bd = smem_desc_sw128(smem_u32(xs + (size_t)(2 * s) * x_bytes));
                const uint32_t blo = (uint32_t)bd, bhi = (uint32_t)(bd >> 32);
#pragma unroll
                for (int kk = 0; kk < TC_KC / 16; ++kk)        // chunk 2s: +32 bytes per k-step
                    mma_f16_tmem_a2(tmem_base, a + 8u * kk, blo + 2u * kk, bhi, idesc,
                                    (s > 0 || kk > 0) ? 1u : 0u);
                if (nch - 2 * s >= 2)                         // chunk 2s + 1: one x chunk on
#pragma unroll
                    for (int kk = 0; kk < TC_KC / 16; ++kk)
                        mma_f16_tmem_a2(tmem_base, a + 32u + 8u * kk,
                                        blo + (x_bytes >> 4) + 2u * kk, bhi, idesc, 1u);
                mma_commit(smem_u32(&aempty[sl]));
                if (s < 16) TC_TRACE(40 + s);
                if (++sl == SK_NA) {
                    sl = 0;
                    ph ^= 1u;
                }
            }
            mma_commit(smem_u32(done));
        }
        // free the accumulator as soon as every worker has read it back
        __syncwarp();
        asm volatile("bar.sync 3, %0;" ::"r"((TC_WORKERS + 1) * 32) : "memory");
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                     ::"r"(tmem_base), "r"(SK_TMEM_COLS) : "memory");
    } else if (warp >= 2 + TC_WORKERS) {
        // ------------------------------------------------------ x load + convert
        // x comes from the previous kernel, so these warps wait for it.  Lane 0 of
        // x warp i then requests the steps i, i + 8, ...: one tensor copy per x
        // chunk (TN token rows x 128 bytes, 128-byte swizzle, rows beyond M zero)
        // -- spread over eight issuing warps, the copies overlap instead of queuing
        // behind one thread.  All eight warps convert each step bf16 -> fp16 in
        // place once it lands.  A value outside the fp16 range sets
        // Q4_DEVERR_FP16_RANGE.
        const int xw = warp - (2 + TC_WORKERS);
        const int xt = xw * 32 + lane;
        pdl_wait();
        if (lane == 0)
            for (int st = xw; st < nstep; st += SK_XWARPS) {
                const int nv = nch - 2 * st < 2 ? 1 : 2;
                mbar_arrive_expect_tx(smem_u32(&xfull[st]), (uint32_t)nv * x_bytes);
                for (int h = 0; h < nv; ++h)
                    tma_load_2d(smem_u32(xs + (size_t)(2 * st + h) * x_bytes), &xmap,
                                (c0 + 2 * st + h) * TC_KC, 0, smem_u32(&xfull[st]));
            }
        if (xt == 0) TC_TRACE(4);
        bool range_bad = false;
        for (int st = 0; st < nstep; ++st) {
            if (!mbar_wait_warp(smem_u32(&xfull[st]), 0, p.err))
                break;
            if (xt == 0 && st == 0) TC_TRACE(6);
            if (xt == 0 && st == nstep - 1) TC_TRACE(61);
            const int nvec = (nch - 2 * st < 2 ? 1 : 2) * TN * 8;
            uint4 *xv = reinterpret_cast<uint4 *>(xs + (size_t)(2 * st) * x_bytes);
            for (int v = xt; v < nvec; v += SK_XWARPS * 32) {
                const uint4 e4 = xv[v];
                const uint32_t ev[4] = {e4.x, e4.y, e4.z, e4.w};
                uint32_t o[4];
                float mx = 0.f;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float lo = bf16_bits_to_f32(ev[q] & 0xffffu);
                    const float hi = bf16_bits_to_f32(ev[q] >> 16);
                    mx = fmaxf(mx, fmaxf(fabsf(lo), fabsf(hi)));
                    __half2 hh = __floats2half2_rn(lo, hi);
                    o[q] = *reinterpret_cast<uint32_t *>(&hh);
                }
                if (mx >= 65520.f && mx <= 3.4e38f)
                    range_bad = true;
                xv[v] = make_uint4(o[0], o[1], o[2], o[3]);
            }
            fence_proxy_async();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_u32(&xready[st]));
            if (xt == 0 && st == 0) TC_TRACE(7);
        }
        if (range_bad && p.err)
            atomicOr(p.err, kErrFp16Range);
        // every copy this warp requested has landed before the CTA can exit
        if (lane == 0)
            for (int st = xw; st < nstep; st += SK_XWARPS)
                mbar_wait(smem_u32(&xfull[st]), 0, p.err);
    } else {
        // ------------------------------------------------------------- workers
        // A step is two chunks (128 columns).  Warp w may write only TMEM lane
        // quadrant w % 4, so it owns rows 32 (w % 4) + lane; the four warps of a
        // quadrant split the step's columns: g = (w - 2) / 4 takes columns
        // 32 g .. + 31 (chunk g / 2, half g % 2).  A thread reads 16 bytes of its
        // row's codes, dequantises 32 weights and writes them as 16 packed columns
        // of its lane.
        const int w = warp - 2;                  // 0..15
        const int quad = warp & 3;
        const int g = w >> 2;
        const int h = g >> 1;
        const int half = g & 1;
        const int row = quad * 32 + lane;
        const bool rok = n0 + row < p.N;
        const int64_t n = n0 + row;
        const uint32_t t_lane = (uint32_t)(quad * 32) << 16;
        // int4: scale | min << 16 of the thread's group; NVFP4: the e4m3 scales of
        // its two 16-column groups (low byte first)
        auto load_scale = [&](int s) -> uint32_t {
            const int j = 2 * s + h;
            if (!rok || j >= nch)
                return 0u;
            const int kc = c0 + j;
            if constexpr (LAYOUT == 0) {
                const int64_t gi = n * (p.K / 128) + kc / 2;
                return ld_nc_u16(static_cast<const uint16_t *>(p.scale) + gi) |
                       (ld_nc_u16(p.minv + gi) << 16);
            } else {
                return ld_nc_u16(static_cast<const uint8_t *>(p.scale) + n * (p.K / 16) + kc * 4 +
                                     2 * half);
            }
        };
        int sl = 0;                              // A slot of the step
        uint32_t ph = 0;                         // parity of the slot's current use
        TC_PHASE_DECL;
        // one step; false when a wait timed out
        auto step = [&](int s, uint32_t sc) -> bool {
            TC_CLK(t0);
            if (s >= SK_NA && !mbar_wait_warp(smem_u32(&aempty[sl]), ph ^ 1u, p.err))
                return false;
            TC_CLK(t1);
            TC_PHASE(56, t0, t1);
            if ((s & 1) == 0 && !mbar_wait_warp(smem_u32(&cfull[s >> 1]), 0, p.err))
                return false;
            tc_fence_after();
            TC_CLK(t2);
            TC_PHASE(57, t1, t2);
            if (2 * s + h < nch) {
                // unit 4 (s % 2) + g of the row in the box, stored at unit ^ (row % 8)
                const uint4 cw = *reinterpret_cast<const uint4 *>(
                    cs + (size_t)(s >> 1) * 16384 + row * 128 + (((4 * (s & 1) + g) ^ (row & 7)) << 4));
                uint32_t lo[8], hi[8];
                tc_decode16<LAYOUT>(make_uint2(cw.x, cw.y), sc, lo);
                tc_decode16<LAYOUT>(make_uint2(cw.z, cw.w), LAYOUT == 0 ? sc : (sc >> 8), hi);
                const uint32_t v[16] = {lo[0], lo[1], lo[2], lo[3], lo[4], lo[5], lo[6], lo[7],
                                        hi[0], hi[1], hi[2], hi[3], hi[4], hi[5], hi[6], hi[7]};
                tmem_st16(tmem_base + t_lane + 64u + 64u * (uint32_t)sl + 32u * h + 16u * half, v);
            }
            TC_CLK(t3);
            TC_PHASE(58, t2, t3);
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_u32(&afull[sl]));
            if (++sl == SK_NA) {
                sl = 0;
                ph ^= 1u;
            }
            TC_CLK(t4);
            TC_PHASE(59, t3, t4);
            return true;
        };
        // Scales run eight steps ahead in two register sets that take turns, each
        // refilled right after its value is used: no register moves, so no wait on
        // a load that is still in flight.
        uint32_t sa[4], sb[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            sa[i] = load_scale(i);
            sb[i] = load_scale(4 + i);
        }
        bool alive = true;
        for (int g8 = 0; g8 < nstep && alive; g8 += 8) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                if (alive && g8 + i < nstep)
                    alive = step(g8 + i, sa[i]);
                sa[i] = load_scale(g8 + 8 + i);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                if (alive && g8 + 4 + i < nstep)
                    alive = step(g8 + 4 + i, sb[i]);
                sb[i] = load_scale(g8 + 12 + i);
            }
        }
        TC_PHASE_STORE();
        // every code copy has landed before the CTA can exit (the steps wait for
        // them; this covers a step loop that stopped early)
        if (warp == 2 && lane == 0)
            for (int b = 0; b < nbox; ++b)
                mbar_wait(smem_u32(&cfull[b]), 0, p.err);

        // ------------------------------------------------------------ epilogue
        // warp w reads TMEM lane quadrant (w + 2) % 4, columns 16 (w / 4) .. + 15
        const bool ok = mbar_wait_warp(smem_u32(done), 0, p.err);
        tc_fence_after();
        if (warp == 2 && lane == 0) TC_TRACE(2);
        const int cb = g * 16;
        const int r = row;
        uint32_t v[16];
        if (cb < TN)
            tmem_ld16(tmem_base + t_lane + (uint32_t)cb, v);
        tc_fence_before();
        asm volatile("bar.arrive 3, %0;" ::"r"((TC_WORKERS + 1) * 32) : "memory");
        if (ok && cb < TN) {
            if (p.KS == 1) {
                if (n0 + r < p.N)
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (cb + j < p.M)
                            p.y[(int64_t)(cb + j) * p.N + n0 + r] =
                                f32_to_bf16_bits(__uint_as_float(v[j]) * gsc);
            } else {
                // x and codes are idle once the final commit has been seen
                float *dump = reinterpret_cast<float *>(smem);
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    dump[(cb + j) * TC_ROWS + r] = __uint_as_float(v[j]);
            }
        }
    }

    if (p.KS > 1) {
        // Sum this CTA's share of the tile over the KS accumulators of the cluster.
        __syncwarp();
        cluster_sync_all();                      // every dump of the cluster is written
        if (threadIdx.x == 0) TC_TRACE(5);
        const int e4 = TN * (TC_ROWS / 4);       // float4 groups of the tile
        const int g0 = (int)((int64_t)ks * e4 / p.KS);
        const int g1 = (int)((int64_t)(ks + 1) * e4 / p.KS);
        const uint32_t base = smem_u32(smem);
        for (int g = g0 + (int)threadIdx.x; g < g1; g += SK_THREADS) {
            float4 part[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
                if (k < p.KS)
                    part[k] = ld_cluster_f4(base + (uint32_t)g * 16u, (uint32_t)k);
            float4 sum = part[0];
#pragma unroll
            for (int k = 1; k < 8; ++k)
                if (k < p.KS) {
                    sum.x += part[k].x; sum.y += part[k].y;
                    sum.z += part[k].z; sum.w += part[k].w;
                }
            const int m = g / (TC_ROWS / 4);
            const int nb = n0 + 4 * (g % (TC_ROWS / 4));
            if (m < p.M) {
                uint16_t *yr = p.y + (int64_t)m * p.N + nb;
                const uint16_t o[4] = {f32_to_bf16_bits(sum.x * gsc), f32_to_bf16_bits(sum.y * gsc),
                                       f32_to_bf16_bits(sum.z * gsc), f32_to_bf16_bits(sum.w * gsc)};
                if (nb + 3 < p.N && (reinterpret_cast<uintptr_t>(yr) & 7u) == 0) {
                    *reinterpret_cast<uint2 *>(yr) =
                        make_uint2(o[0] | ((uint32_t)o[1] << 16), o[2] | ((uint32_t)o[3] << 16));
                } else {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if (nb + i < p.N)
                            yr[i] = o[i];
                }
            }
        }
        cluster_sync_all();                      // no CTA leaves while its dump is read
    }
    if (threadIdx.x == 0) TC_TRACE(3);
}

// x (bf16) -> fp16 once per call for large M, so that the GEMM's CTAs do not each
// convert the same token tiles.  Out-of-range values set Q4_DEVERR_FP16_RANGE.
__global__ void __launch_bounds__(256) q4_x_to_f16_kernel(const uint4 *__restrict__ x,
                                                          uint4 *__restrict__ out, int64_t n16,
                                                          unsigned *err)
{
    pdl_launch_dependents();
    pdl_wait();
    bool bad = false;
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < n16;
         v += (int64_t)gridDim.x * blockDim.x) {
        const uint4 t = x[v];
        const uint32_t e[4] = {t.x, t.y, t.z, t.w};
        uint32_t o[4];
        float mx = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float lo = bf16_bits_to_f32(e[j] & 0xffffu);
            const float hi = bf16_bits_to_f32(e[j] >> 16);
            mx = fmaxf(mx, fmaxf(fabsf(lo), fabsf(hi)));
            __half2 h = __floats2half2_rn(lo, hi);
            o[j] = *reinterpret_cast<uint32_t *>(&h);
        }
        bad |= (mx >= 65520.f && mx <= 3.4e38f);
        out[v] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (bad && err)
        atomicOr(err, kErrFp16Range);
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

static int tc_tn(int M)
{
    if (M > 256)
        return 256;
    return (M + 15) / 16 * 16 < 16 ? 16 : (M + 15) / 16 * 16;
}

// Split-K factor: as many CTAs as fit in one wave (one CTA per SM) when the tile
// grid is small, keeping at least four K chunks per CTA and at most eight
// partials per tile (the last CTA of a tile sums them; more would lengthen that
// tail more than the extra CTAs shorten the main loop).
static int tc_ks(const DeviceInfo &dev, int M, int N, int K)
{
    const int TN = tc_tn(M);
    const int64_t tiles = (int64_t)((N + TC_ROWS - 1) / TC_ROWS) * ((M + TN - 1) / TN);
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

// x is converted inside the GEMM for tiles of up to 64 tokens (at most SC
// vectors per thread), by a separate pass for more.
static bool tc_preconvert(int M) { return M > 64; }

static size_t tc_xf16_bytes(int M, int K)
{
    return tc_preconvert(M) ? ((size_t)M * K * 2 + 255) / 256 * 256 : 0;
}

static size_t tc_split_bytes(int M, int N, int K, int sms)
{
    DeviceInfo d;
    d.sms = sms;
    const int ks = tc_ks(d, M, N, K);
    if (ks == 1)
        return 0;
    const int TN = tc_tn(M);
    const size_t tiles = (size_t)((N + TC_ROWS - 1) / TC_ROWS) * ((M + TN - 1) / TN);
    return (tiles * 4 + 255) / 256 * 256 + tiles * ks * TN * TC_ROWS * 4;
}

// Workspace layout: [fp16 copy of x (large M)][split-K counters][partials].
size_t tc_workspace_bytes(int M, int N, int K, int sms)
{
    if (K % TC_KC || M < 1 || N < 1)
        return 0;
    return tc_xf16_bytes(M, K) + tc_split_bytes(M, N, K, sms);
}

// Skinny plan: tiles of at most 64 tokens whose K range, split into at most
// eight parts (one cluster of at most eight CTAs per weight tile), keeps all its
// codes and x chunks resident in shared memory (the A tiles live in TMEM).
struct TcSkinnyPlan {
    int ks = 0, ncmax = 0;
    size_t smem = 0;
};

static size_t tc_skinny_smem(int TN, int nch)
{
    return 1024 /* alignment of the base */ + SkLayout(TN, nch).bytes();
}

static bool tc_skinny_plan(const DeviceInfo &dev, int M, int N, int K, TcSkinnyPlan &sp)
{
    const int TN = tc_tn(M);
    if (TN > 64 || K % TC_KC)
        return false;
    const int chunks = K / TC_KC;
    const int64_t tiles = (N + TC_ROWS - 1) / TC_ROWS;
    // the smallest split that fits, then more CTAs -- they pull more bandwidth --
    // while the grid stays one wave and every CTA keeps at least four chunks
    for (int ks = 1; ks <= 8 && ks <= chunks; ++ks) {
        if (tc_skinny_smem(TN, (chunks + ks - 1) / ks) > dev.smem_optin)
            continue;
        while (ks < 8 && tiles * (ks + 1) <= dev.sms && chunks / (ks + 1) >= 4)
            ++ks;
        sp.ks = ks;
        sp.ncmax = (chunks + ks - 1) / ks;
        sp.smem = tc_skinny_smem(TN, sp.ncmax);
        return true;
    }
    return false;
}

// Whether a cluster of ks CTAs of this size can be resident at all (cached).
static bool tc_cluster_fits(const void *k, int device, int ks, size_t smem)
{
    struct Entry {
        const void *k;
        int device, ks;
        size_t smem;
        bool ok;
    };
    static std::mutex mu;
    static Entry cache[64];
    static int used = 0;
    std::lock_guard<std::mutex> g(mu);
    for (int i = 0; i < used; ++i)
        if (cache[i].k == k && cache[i].device == device && cache[i].ks == ks && cache[i].smem == smem)
            return cache[i].ok;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ks);
    cfg.blockDim = dim3(SK_THREADS);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute a[1];
    a[0].id = cudaLaunchAttributeClusterDimension;
    a[0].val.clusterDim.x = (unsigned)ks;
    a[0].val.clusterDim.y = 1;
    a[0].val.clusterDim.z = 1;
    cfg.attrs = a;
    cfg.numAttrs = 1;
    int n = 0;
    const bool ok = cudaOccupancyMaxActiveClusters(&n, k, &cfg) == cudaSuccess && n > 0;
    cudaGetLastError();
    if (used < 64)
        cache[used++] = {k, device, ks, smem, ok};
    return ok;
}

static CUresult tc_encode_maps(EncodeTiledFn enc, CUtensorMap &xmap, CUtensorMap &wmap,
                               const void *xsrc, bool x_f16, const uint8_t *codes, int M, int N,
                               int K, int TN, int code_box_bytes, bool code_swizzle)
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
    cuuint32_t wbox[2] = {(cuuint32_t)code_box_bytes, TC_ROWS};
    return enc(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(codes), wd, wstr, wbox,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               code_swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

template <int LAYOUT>
static const void *tc_select_layout(int sc, int groups)
{
    if (groups == 2)
        return sc == 4 ? reinterpret_cast<const void *>(&q4_tc_kernel<LAYOUT, 4, 2>)
             : sc == 2 ? reinterpret_cast<const void *>(&q4_tc_kernel<LAYOUT, 2, 2>)
                       : reinterpret_cast<const void *>(&q4_tc_kernel<LAYOUT, 1, 2>);
    return sc == 4 ? reinterpret_cast<const void *>(&q4_tc_kernel<LAYOUT, 4, 1>)
         : sc == 2 ? reinterpret_cast<const void *>(&q4_tc_kernel<LAYOUT, 2, 1>)
                   : reinterpret_cast<const void *>(&q4_tc_kernel<LAYOUT, 1, 1>);
}

static const void *tc_select(int kind, int sc, int groups)
{
    return kind == W_INT4 ? tc_select_layout<0>(sc, groups) : tc_select_layout<1>(sc, groups);
}

q4_status tc_launch(int kind, const void *x, const uint8_t *codes, const void *scale,
                    const void *minv, const float *gscale, void *y, int M, int N, int K,
                    void *ws, size_t ws_bytes, cudaStream_t stream, bool pdl,
                    bool skinny)
{
    DeviceInfo dev;
    q4_status s = current_device(dev);
    if (s != Q4_OK)
        return s;
    EncodeTiledFn enc = encode_fn();
    if (!enc)
        return fail(Q4_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    TcParams p = {};
    p.codes = codes;
    p.scale = scale;
    p.minv = static_cast<const uint16_t *>(minv);
    p.gscale = gscale;
    p.y = static_cast<uint16_t *>(y);
    p.err = device_error_flags();
    p.M = M;
    p.N = N;
    p.K = K;
#ifdef Q4_TRACE
    static int trace_calls = 0;
    p.call = trace_calls++;
#endif
    p.TN = tc_tn(M);
    p.tiles_m = (M + p.TN - 1) / p.TN;
    p.KS = tc_ks(dev, M, N, K);
    p.chunks = K / TC_KC;
    int cols = 32;
    while (cols < p.TN)
        cols *= 2;
    p.tmem_cols = cols;
    TcSkinnyPlan sp;
    if (skinny && tc_skinny_plan(dev, M, N, K, sp)) {
        const void *k = kind == W_INT4 ? reinterpret_cast<const void *>(&q4_tc_skinny_kernel<0>)
                                       : reinterpret_cast<const void *>(&q4_tc_skinny_kernel<1>);
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)sp.smem);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaFuncSetAttribute(skinny tensor-core kernel)");
        if (sp.ks == 1 || tc_cluster_fits(k, dev.device, sp.ks, sp.smem)) {
            p.KS = sp.ks;
            p.ns = SK_NA;
            p.tmem_cols = SK_TMEM_COLS;
            p.x_f16 = 0;
            CUtensorMap xmap, wmap;
            const CUresult r = tc_encode_maps(enc, xmap, wmap, x, false, codes, M, N, K, p.TN,
                                              2 * TC_KC, true);
            if (r != CUDA_SUCCESS)
                return fail(Q4_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)(((N + TC_ROWS - 1) / TC_ROWS) * sp.ks));
            cfg.blockDim = dim3(SK_THREADS);
            cfg.dynamicSmemBytes = sp.smem;
            cfg.stream = stream;
            cudaLaunchAttribute a[2];
            unsigned na = 0;
            if (pdl) {
                a[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
                a[na].val.programmaticStreamSerializationAllowed = 1;
                ++na;
            }
            if (sp.ks > 1) {
                a[na].id = cudaLaunchAttributeClusterDimension;
                a[na].val.clusterDim.x = (unsigned)sp.ks;
                a[na].val.clusterDim.y = 1;
                a[na].val.clusterDim.z = 1;
                ++na;
            }
            cfg.attrs = na ? a : nullptr;
            cfg.numAttrs = na;
            void *args[] = {&xmap, &wmap, &p};
            e = cudaLaunchKernelExC(&cfg, k, args);
            if (e != cudaSuccess)
                return cuda_fail(e, "launch of the skinny tensor-core kernel");
            return Q4_OK;
        }
    }
    const size_t need = tc_workspace_bytes(M, N, K, dev.sms);
    if (need > ws_bytes)
        return fail(Q4_ERR_WORKSPACE, "tensor-core path needs %zu bytes of workspace", need);
    const size_t tiles = (size_t)((N + TC_ROWS - 1) / TC_ROWS) * p.tiles_m;
    unsigned char *wsb = static_cast<unsigned char *>(ws);
    const size_t xf16 = tc_xf16_bytes(M, K);
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
        const int64_t n16 = (int64_t)M * K / 8;
        int64_t blocks = (n16 + 255) / 256;
        if (blocks > (int64_t)dev.sms * 8)
            blocks = (int64_t)dev.sms * 8;
        cudaLaunchConfig_t pc = {};
        pc.gridDim = dim3((unsigned)blocks);
        pc.blockDim = dim3(256);
        pc.stream = stream;
        pc.attrs = pdl ? attr : nullptr;
        pc.numAttrs = pdl ? 1 : 0;
        const uint4 *xin = static_cast<const uint4 *>(x);
        uint4 *xo = reinterpret_cast<uint4 *>(wsb);
        void *pargs[] = {&xin, &xo, (void *)&n16, &p.err};
        cudaError_t e0 = cudaLaunchKernelExC(&pc, reinterpret_cast<const void *>(&q4_x_to_f16_kernel),
                                             pargs);
        if (e0 != cudaSuccess)
            return cuda_fail(e0, "launch of the x conversion kernel");
        xsrc = wsb;
        p.x_f16 = 1;
    }
    // Stage = SC chunks (A sub-tiles, x sub-tiles, codes).  The largest SC that
    // still leaves four stages in flight (three, two) amortises each hand-off
    // over more weights without starving the copies.
    const size_t x_stride = ((size_t)p.TN * 128 + 1023) / 1024 * 1024;
    const size_t budget = dev.smem_optin - 1024 /* alignment */ - 1024 /* static */ - 256;
    int sc = 1, ns = 0;
    for (int need = 4; need >= 2 && ns == 0; --need)
        for (int cand = 4; cand >= 1; cand /= 2) {
            const size_t stage = (size_t)cand * (16384 + x_stride + 4096);
            const int fit = (int)(budget / stage);
            if (fit >= need) {
                sc = cand;
                ns = fit > 8 ? 8 : fit;
                break;
            }
        }
#ifdef Q4_TC_SC
    sc = Q4_TC_SC;
    ns = (int)(budget / ((size_t)sc * (16384 + x_stride + 4096)));
    ns = ns > 8 ? 8 : ns;
#endif
    if (ns < 2)
        return fail(Q4_ERR_SHAPE, "tensor-core tile does not fit in shared memory");
    p.ns = ns;
    const size_t stage = (size_t)sc * (16384 + x_stride + 4096);
    const size_t smem = 1024 + (size_t)ns * stage + (3 * ns + 1) * 8 + 16;

    CUtensorMap xmap, wmap;
    {
        const CUresult r = tc_encode_maps(enc, xmap, wmap, xsrc, p.x_f16 != 0, codes, M, N, K, p.TN,
                                          sc * TC_KC / 2, false);
        if (r != CUDA_SUCCESS)
            return fail(Q4_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    }
    // two worker groups, two stages dequantised at once (measured: prefill
    // GEMMs 5-22% faster than one group of 16 warps; batched decode unchanged)
#ifdef Q4_TC_GROUPS
    const int groups = Q4_TC_GROUPS;
#else
    const int groups = 2;
#endif
    const void *k = tc_select(kind, sc, groups);
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaFuncSetAttribute(tensor-core kernel)");
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(tiles * p.KS));
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
