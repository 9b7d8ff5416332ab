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
//   * Eight worker warps dequantise the codes into the A operand tile (fp16,
//     K-major, 128-byte swizzle) and convert the x tile in place from bf16 to
//     fp16.  int4: w = fp16(c * s + m) (one fused multiply-add, single rounding);
//     NVFP4: w = E2M1 * e4m3 in fp16, exact (the global scale is applied in the
//     epilogue).  An x value outside the fp16 range sets Q4_DEVERR_FP16_RANGE.
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
constexpr int TC_WORKERS = 8;          // dequant / epilogue warps
constexpr int TC_THREADS = (2 + TC_WORKERS) * 32;
constexpr unsigned kErrFp16Range = 2u;

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
    int ns;                    // ring stages
    int tmem_cols;             // power of two >= max(32, TN)
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

__device__ __forceinline__ void fence_proxy_async()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
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

__device__ __forceinline__ void mma_f16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "setp.ne.u32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                 ::"r"(tmem_d), "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
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

// ------------------------------------------------------------------ kernel
template <int LAYOUT>   // 0 int4-g128, 1 NVFP4
__global__ void __launch_bounds__(TC_THREADS, 1)
q4_tc_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap,
             TcParams p)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-byte aligned carve-up: [x stages][A stages][code stages][barriers]
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int TN = p.TN;
    const int NS = p.ns;
    const uint32_t x_bytes = (uint32_t)TN * 128;
    const uint32_t x_stride = (x_bytes + 1023) & ~1023u;
    unsigned char *xbuf = smem;
    unsigned char *abuf = xbuf + (size_t)NS * x_stride;                 // 16 KB per stage
    unsigned char *cbuf = abuf + (size_t)NS * 16384;                   // 4 KB per stage
    uint64_t *bars = reinterpret_cast<uint64_t *>(cbuf + (size_t)NS * 4096);
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
    const int c0 = (int)((int64_t)ks * p.chunks / p.KS);
    const int c1 = (int)((int64_t)(ks + 1) * p.chunks / p.KS);
    const int nch = c1 - c0;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(smem_u32(&bars[i]), 1);                  // TMA arrive + bytes
            mbar_init(smem_u32(&bars[NS + i]), TC_WORKERS);    // worker warps
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
            for (int i = 0; i < nch; ++i) {
                const int s = i % NS, use = i / NS;
                if (use > 0 && !mbar_wait(smem_u32(&bars[2 * NS + s]), (use - 1) & 1, p.err))
                    break;
                if (i == 0)
                    pdl_wait();                // x comes from the previous kernel
                const uint32_t full = smem_u32(&bars[s]);
                mbar_arrive_expect_tx(full, x_bytes + 4096);
                const int kc = c0 + i;
                tma_load_2d(smem_u32(xbuf + (size_t)s * x_stride), &xmap, kc * TC_KC, m0, full);
                tma_load_2d(smem_u32(cbuf + (size_t)s * 4096), &wmap, kc * (TC_KC / 2), n0, full);
                issued = i + 1;
            }
            // drain: every issued copy has landed before the CTA can exit
            for (int i = issued - NS > 0 ? issued - NS : 0; i < issued; ++i)
                mbar_wait(smem_u32(&bars[i % NS]), (i / NS) & 1, p.err);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------- MMA issue
        if (lane == 0) {
            const uint32_t idesc = idesc_f16(TN);
            for (int i = 0; i < nch; ++i) {
                const int s = i % NS, use = i / NS;
                if (!mbar_wait(smem_u32(&bars[NS + s]), use & 1, p.err))
                    break;
                tc_fence_after();
                const uint32_t a0 = smem_u32(abuf + (size_t)s * 16384);
                const uint32_t b0 = smem_u32(xbuf + (size_t)s * x_stride);
#pragma unroll
                for (int kk = 0; kk < TC_KC / 16; ++kk)
                    mma_f16(tmem_base, smem_desc_sw128(a0 + kk * 32), smem_desc_sw128(b0 + kk * 32),
                            idesc, (i > 0 || kk > 0) ? 1u : 0u);
                mma_commit(smem_u32(&bars[2 * NS + s]));
            }
            mma_commit(smem_u32(&bars[3 * NS]));
        }
    } else {
        // ------------------------------------------------------------- workers
        const int w = warp - 2;                  // 0..7
        const int quad = warp & 3;               // TMEM lane quadrant of this warp
        const int half = w >> 2;                 // which 32 codes of the row
        const int r = quad * 32 + lane;          // weight row within the tile
        const int n = n0 + r;
        const bool nok = n < p.N;
        const int tid = w * 32 + lane;           // 0..255
        auto load_scale = [&](int kc) -> uint32_t {
            if (!nok)
                return 0u;
            if constexpr (LAYOUT == 0) {
                const int64_t gi = (int64_t)n * (p.K / 128) + (kc * TC_KC) / 128;
                return ld_nc_u16(static_cast<const uint16_t *>(p.scale) + gi) |
                       (ld_nc_u16(p.minv + gi) << 16);
            } else {
                // the two e4m3 scales of this thread's 32 codes
                return ld_nc_u16(static_cast<const uint8_t *>(p.scale) + (int64_t)n * (p.K / 16) +
                                 kc * 4 + half * 2);
            }
        };
        uint32_t sc_next = nch > 0 ? load_scale(c0) : 0u;
        bool range_bad = false;
        for (int i = 0; i < nch; ++i) {
            const int s = i % NS, use = i / NS;
            const uint32_t sc = sc_next;
            if (i + 1 < nch)
                sc_next = load_scale(c0 + i + 1);
            if (!mbar_wait(smem_u32(&bars[s]), use & 1, p.err))
                break;
            // x tile: bf16 -> fp16 in place (element-wise, swizzle-agnostic)
            uint4 *xv = reinterpret_cast<uint4 *>(xbuf + (size_t)s * x_stride);
            for (int v = tid; v < TN * 8; v += TC_WORKERS * 32) {
                const uint4 t = xv[v];
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
                if (mx >= 65520.f && mx <= 3.4e38f)
                    range_bad = true;
                xv[v] = make_uint4(o[0], o[1], o[2], o[3]);
            }
            // A rows: this thread's 32 codes of row r -> four 16-byte fp16 chunks
            const uint4 cw = reinterpret_cast<const uint4 *>(cbuf + (size_t)s * 4096 + r * 32)[half];
            const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
            unsigned char *arow = abuf + (size_t)s * 16384 + (size_t)r * 128;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int chunk = half * 4 + j;          // 8 K columns per chunk
                uint32_t o[4];
                if constexpr (LAYOUT == 0) {
                    const uint32_t s2 = f16x2_splat(sc & 0xffffu);
                    const uint32_t m2 = f16x2_splat(sc >> 16);
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
                    const uint32_t s16 = e4m3x2_to_f16x2(sc);       // two group scales
                    const uint32_t sg = f16x2_splat(j < 2 ? (s16 & 0xffffu) : (s16 >> 16));
#pragma unroll
                    for (int b = 0; b < 4; ++b)
                        o[b] = hmul2(h[b], sg);                     // exact in fp16
                }
                *reinterpret_cast<uint4 *>(arow + ((chunk ^ (r & 7)) << 4)) =
                    make_uint4(o[0], o[1], o[2], o[3]);
            }
            fence_proxy_async();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_u32(&bars[NS + s]));
        }
        if (range_bad && p.err)
            atomicOr(p.err, kErrFp16Range);

        // ------------------------------------------------------------ epilogue
        const bool ok = nch > 0 && mbar_wait(smem_u32(&bars[3 * NS]), 0, p.err);
        tc_fence_after();
        float gsc = 1.f;
        if constexpr (LAYOUT == 1)
            gsc = __ldg(p.gscale);
        const int tile = tile_n * p.tiles_m + tile_m;
        for (int cb = half * 16; cb < TN; cb += 32) {
            uint32_t v[16];
            tmem_ld16(tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)cb, v);
            if (!ok)
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
            __shared__ unsigned last_flag;
            if (tid == 0)
                last_flag = (ok && atomicAdd(&p.tickets[tile], 1u) == (unsigned)(p.KS - 1)) ? 1u : 0u;
            asm volatile("bar.sync 2, %0;" ::"r"(TC_WORKERS * 32) : "memory");
            if (last_flag) {
                __threadfence();
                for (int c = half; c < TN; c += 2) {
                    const int m = m0 + c;
                    float sum = 0.f;
                    for (int k2 = 0; k2 < p.KS; ++k2)
                        sum += __ldcg(p.ws + ((size_t)(tile * p.KS + k2) * TN + c) * TC_ROWS + r);
                    if (nok && m < p.M)
                        p.y[(int64_t)m * p.N + n] = f32_to_bf16_bits(sum * gsc);
                }
                if (tid == 0)
                    p.tickets[tile] = 0u;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                     ::"r"(tmem_base), "r"(p.tmem_cols) : "memory");
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

static int tc_tn(int M)
{
    if (M > 256)
        return 256;
    return (M + 15) / 16 * 16 < 16 ? 16 : (M + 15) / 16 * 16;
}

// Split-K factor: enough CTAs to cover the SMs when the tile grid is small,
// keeping at least four K chunks per CTA.
static int tc_ks(const DeviceInfo &dev, int M, int N, int K)
{
    const int TN = tc_tn(M);
    const int64_t tiles = (int64_t)((N + TC_ROWS - 1) / TC_ROWS) * ((M + TN - 1) / TN);
    const int chunks = K / TC_KC;
    if (tiles * 2 > dev.sms)
        return 1;
    int ks = (int)((dev.sms + tiles - 1) / tiles);
    if (ks > chunks / 4)
        ks = chunks / 4;
    if (ks > 16)
        ks = 16;
    return ks < 1 ? 1 : ks;
}

size_t tc_workspace_bytes(int M, int N, int K, int sms)
{
    if (K % TC_KC || M < 1 || N < 1)
        return 0;
    DeviceInfo d;
    d.sms = sms;
    const int ks = tc_ks(d, M, N, K);
    if (ks == 1)
        return 0;
    const int TN = tc_tn(M);
    const size_t tiles = (size_t)((N + TC_ROWS - 1) / TC_ROWS) * ((M + TN - 1) / TN);
    return (tiles * 4 + 255) / 256 * 256 + tiles * ks * TN * TC_ROWS * 4;
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
    p.codes = codes;
    p.scale = scale;
    p.minv = static_cast<const uint16_t *>(minv);
    p.gscale = gscale;
    p.y = static_cast<uint16_t *>(y);
    p.err = device_error_flags();
    p.M = M;
    p.N = N;
    p.K = K;
    p.TN = tc_tn(M);
    p.tiles_m = (M + p.TN - 1) / p.TN;
    p.KS = tc_ks(dev, M, N, K);
    p.chunks = K / TC_KC;
    int cols = 32;
    while (cols < p.TN)
        cols *= 2;
    p.tmem_cols = cols;
    const size_t need = tc_workspace_bytes(M, N, K, dev.sms);
    if (need > ws_bytes)
        return fail(Q4_ERR_WORKSPACE, "tensor-core path needs %zu bytes of workspace", need);
    const size_t tiles = (size_t)((N + TC_ROWS - 1) / TC_ROWS) * p.tiles_m;
    if (p.KS > 1) {
        unsigned char *b = static_cast<unsigned char *>(ws);
        p.tickets = reinterpret_cast<unsigned *>(b);
        p.ws = reinterpret_cast<float *>(b + (tiles * 4 + 255) / 256 * 256);
    }
    // ring depth: as many stages as fit beside the barriers
    const size_t x_stride = ((size_t)p.TN * 128 + 1023) / 1024 * 1024;
    const size_t stage = x_stride + 16384 + 4096;
    int ns = (int)((dev.smem_optin - 2048) / stage);
    if (ns > 6)
        ns = 6;
    if (ns < 2)
        return fail(Q4_ERR_SHAPE, "tensor-core tile does not fit in shared memory");
    p.ns = ns;
    const size_t smem = 1024 + (size_t)ns * stage + (3 * ns + 1) * 8 + 16;

    CUtensorMap xmap, wmap;
    {
        cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
        cuuint64_t strides[1] = {(cuuint64_t)K * 2};
        cuuint32_t box[2] = {TC_KC, (cuuint32_t)p.TN};
        cuuint32_t estr[2] = {1, 1};
        CUresult r = enc(&xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(x), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS)
            return fail(Q4_ERR_CUDA, "cuTensorMapEncodeTiled(x) failed (%d)", (int)r);
    }
    {
        cuuint64_t dims[2] = {(cuuint64_t)K / 2, (cuuint64_t)N};
        cuuint64_t strides[1] = {(cuuint64_t)K / 2};
        cuuint32_t box[2] = {TC_KC / 2, TC_ROWS};
        cuuint32_t estr[2] = {1, 1};
        CUresult r = enc(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(codes),
                         dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS)
            return fail(Q4_ERR_CUDA, "cuTensorMapEncodeTiled(codes) failed (%d)", (int)r);
    }
    const void *k = kind == W_INT4 ? reinterpret_cast<const void *>(&q4_tc_kernel<0>)
                                   : reinterpret_cast<const void *>(&q4_tc_kernel<1>);
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaFuncSetAttribute(tensor-core kernel)");
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
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
