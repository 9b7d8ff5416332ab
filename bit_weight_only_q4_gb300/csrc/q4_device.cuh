// Device-side helpers shared by the sm_103a kernels of this library: streaming
// loads, in-register decoders of the two 4-bit layouts, mixed-precision FMAs and
// programmatic-dependent-launch controls, mbarriers and bulk async copies.  All
// of it is inline PTX or CUDA intrinsics; nothing here allocates, and the only
// wait (mbar_wait) is bounded.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace q4 {

// ------------------------------------------------------------------ loads
// Weights are read exactly once per call: bypass L1 allocation.
__device__ __forceinline__ uint4 ld_stream_v4(const void *p)
{
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ uint2 ld_stream_v2(const void *p)
{
    uint2 r;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];"
                 : "=r"(r.x), "=r"(r.y)
                 : "l"(p));
    return r;
}

// 16-byte asynchronous global -> shared copy through L2 only (cp.async.cg).
// src_bytes = 0 writes 16 zero bytes and reads nothing.  Completion is tracked
// per thread by commit groups.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;"
                 :: "r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// Wait until at most N of this thread's most recent commit groups are pending.
template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory");
}

// 8- and 16-bit loads straight into 32-bit registers (zero-extended), so no
// widening instruction waits for the load right after it is issued.
__device__ __forceinline__ uint32_t ld_nc_u16(const void *p)
{
    uint32_t r;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=r"(r) : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t ld_nc_u8(const void *p)
{
    uint32_t r;
    asm volatile("ld.global.nc.u8 %0, [%1];" : "=r"(r) : "l"(p));
    return r;
}

// ---------------------------------------------- programmatic dependent launch
// Wait until the grids this one depends on have completed and their writes are
// visible (a no-op when the kernel was not launched with PDL).
__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Allow the next kernel in the stream to be scheduled (its pdl_wait still waits
// for this grid to complete).
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------- int4 code decoding
// Two 4-bit codes at bit positions 0..3 and 16..19 of v become the bf16 pair
// (128 + c_lo, 128 + c_hi): OR the code into the mantissa of 128.0 (0x4300),
// whose last mantissa bit weighs 1.  Exact for c in 0..15.
__device__ __forceinline__ uint32_t int4_pair_bf16_biased(uint32_t v)
{
    uint32_t r;
    asm("lop3.b32 %0, %1, 0x000F000F, 0x43004300, 0xEA;" : "=r"(r) : "r"(v));
    return r;  // (v & 0x000F000F) | 0x43004300
}

// ------------------------------------------------------ mixed-precision FMA
// acc += a.lo * b.lo + a.hi * b.hi with bf16 operands and an fp32 accumulator
// (each product is exact in fp32; two roundings, one per add).
__device__ __forceinline__ float fma2_bf16(float acc, uint32_t a, uint32_t b)
{
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %1;\n\t"
        "mov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.bf16 %0, al, bl, %0;\n\t"
        "fma.rn.f32.bf16 %0, ah, bh, %0;\n\t}"
        : "+f"(acc)
        : "r"(a), "r"(b));
    return acc;
}

// Same with fp16 operands.
__device__ __forceinline__ float fma2_f16(float acc, uint32_t a, uint32_t b)
{
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %1;\n\t"
        "mov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.f16 %0, al, bl, %0;\n\t"
        "fma.rn.f32.f16 %0, ah, bh, %0;\n\t}"
        : "+f"(acc)
        : "r"(a), "r"(b));
    return acc;
}

// Two 16-column groups of fp16 half sums (a: the first group's even and odd
// columns, b: the second's) against their fp16 scales s = (s_a, s_b), in fp32:
// ((a.lo s_a + a.hi s_a) + b.lo s_b) + b.hi s_b, each product exact in fp32 and
// one rounding per add.
__device__ __forceinline__ float f16_group_pair_f32(uint32_t a, uint32_t b, uint32_t s)
{
    float acc;
    asm("{\n\t.reg .b16 al, ah, bl, bh, sl, sh;\n\t"
        "mov.b32 {al, ah}, %1;\n\t"
        "mov.b32 {bl, bh}, %2;\n\t"
        "mov.b32 {sl, sh}, %3;\n\t"
        "fma.rn.f32.f16 %0, al, sl, 0f00000000;\n\t"
        "fma.rn.f32.f16 %0, ah, sl, %0;\n\t"
        "fma.rn.f32.f16 %0, bl, sh, %0;\n\t"
        "fma.rn.f32.f16 %0, bh, sh, %0;\n\t}"
        : "=f"(acc)
        : "r"(a), "r"(b), "r"(s));
    return acc;
}

// Packed fp16 add: a + b per half, one rounding each.
__device__ __forceinline__ uint32_t hadd2_rn(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Packed fp16 fused multiply-add: c + a * b per half, one rounding each.
__device__ __forceinline__ uint32_t hfma2_rn(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t r;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
    return r;
}

// ------------------------------------------------------ NVFP4 decoding
// One byte of two E2M1 codes (low nibble = even column) -> f16x2 (exact).
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte_lo8)
{
    uint32_t r;
    asm("{\n\t.reg .b8 b;\n\t"
        "cvt.u8.u32 b, %1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b;\n\t}"
        : "=r"(r)
        : "r"(byte_lo8));
    return r;
}

// The four bytes of w (eight E2M1 codes, low nibble = even column) -> four f16x2
// pairs: h[b] = (E2M1(code 2b), E2M1(code 2b + 1)).  The byte operands come from a
// vector unpack, which the converter reads in place (no shifts).
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t (&h)[4])
{
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(w));
}

// Two 4-bit codes at bit positions 0..3 and 16..19 (mask 0x000F000F) or 4..7 and
// 20..23 (mask 0x00F000F0) of v become the f16 pair (1024 + c) or (1024 + 16 c):
// OR the masked bits into the mantissa of 1024.0 (0x6400), whose last mantissa
// bit weighs 1.  Exact for c in 0..15.
template <uint32_t MASK>
__device__ __forceinline__ uint32_t int4_pair_f16_biased(uint32_t v)
{
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, 0x64006400, 0xEA;" : "=r"(r) : "r"(v), "n"(MASK));
    return r;  // (v & MASK) | 0x64006400
}

// Integer dot products: c + a.lo16 * b.byte(0|2) + a.hi16 * b.byte(1|3), with a's
// halves signed 16-bit and b's bytes unsigned (.lo takes bytes 0, 1; .hi 2, 3).
__device__ __forceinline__ int dp2a_lo_su(uint32_t a, uint32_t b, int c)
{
    int d;
    asm("dp2a.lo.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ int dp2a_hi_su(uint32_t a, uint32_t b, int c)
{
    int d;
    asm("dp2a.hi.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Two float8_e4m3fn bytes (low 16 bits) -> f16x2 (exact: e4m3 fits in fp16).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes)
{
    uint32_t r;
    unsigned short s = (unsigned short)two_bytes;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(s));
    return r;
}

// The two fp16 halves of h2 as fp32: the pair is unpacked in place (no mask or
// shift) and each half converted once.
__device__ __forceinline__ void f16x2_to_f32x2(uint32_t h2, float &lo, float &hi)
{
    asm("{\n\t.reg .f16 l, h;\n\t"
        "mov.b32 {l, h}, %2;\n\t"
        "cvt.f32.f16 %0, l;\n\t"
        "cvt.f32.f16 %1, h;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(h2));
}

// The low fp16 half of w as fp32 (unpacked in place).
__device__ __forceinline__ float f16lo_unpack_f32(uint32_t w)
{
    float f;
    asm("{\n\t.reg .f16 l, h;\n\t"
        "mov.b32 {l, h}, %1;\n\t"
        "cvt.f32.f16 %0, l;\n\t}"
        : "=f"(f)
        : "r"(w));
    return f;
}

// Two float8_e4m3fn bytes in the low 16 bits of w -> f16x2 (exact), the 16-bit
// operand taken by an in-place unpack.
__device__ __forceinline__ uint32_t e4m3x2lo_to_f16x2(uint32_t w)
{
    uint32_t r;
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "mov.b32 {lo, hi}, %1;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, lo;\n\t}"
        : "=r"(r)
        : "r"(w));
    return r;
}

__device__ __forceinline__ float f16lo_to_f32(uint32_t h2)
{
    return __half2float(__ushort_as_half((unsigned short)(h2 & 0xffffu)));
}

__device__ __forceinline__ float f16hi_to_f32(uint32_t h2)
{
    return __half2float(__ushort_as_half((unsigned short)(h2 >> 16)));
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b16)
{
    return __uint_as_float(b16 << 16);
}

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float v)
{
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}


// ------------------------------------------------ mbarrier + bulk async copy
__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void mbar_init_fence()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// One poll: returns once the phase of the given parity has completed or a short,
// system-dependent time limit has passed.  (A long suspend-time hint made every
// hand-off in the tensor-core pipeline wait far past the phase completion.)
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity)
                 : "memory");
    return ok != 0;
}

// Bounded wait for the phase of the given parity to complete.  Every wait in this
// library ends: after kMbarSpinLimit polls (seconds) the wait sets
// kErrBarrierTimeout in *err and returns false so the kernel can finish instead
// of hanging.
constexpr uint32_t kMbarSpinLimit = 1u << 26;
constexpr unsigned kErrBarrierTimeout = 1u;

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, unsigned *err)
{
    for (uint32_t i = 0; i < kMbarSpinLimit; ++i)
        if (mbar_try_wait(bar, parity))
            return true;
    if (err)
        atomicOr(err, kErrBarrierTimeout);
    return false;
}

// The same wait for a whole (converged) warp: lane 0 polls and the other lanes
// wait at the warp barrier, which orders their later reads after lane 0's
// acquire.  A waiting warp then keeps one poll in the shared-memory pipe instead
// of 32 -- with two dozen warps waiting at once the per-lane polls slowed the
// copies and everything else that shares the pipe.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, unsigned *err)
{
    int ok = 1;
    if ((threadIdx.x & 31) == 0)
        ok = mbar_wait(bar, parity, err) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    return ok != 0;
}

// Order this thread's earlier generic-proxy shared-memory accesses before later
// async-proxy ones (TMA copies, tensor-core operand reads).
__device__ __forceinline__ void fence_proxy_async()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// One contiguous global -> shared copy on the TMA engine; completion is counted
// in bytes on the mbarrier.  dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                              uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes"
                 " [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// ------------------------------------------------------ warp reduction
// Sum V values across the 32 lanes of a warp with a transposing butterfly: at
// each of the first log2(V) steps a lane keeps half of its values and sends the
// other half, so V values cost V-1 + (5 - log2 V) shuffles instead of 5V.
// Returns the total of value index `idx` (written to idx); lanes whose low
// (5 - log2 V) bits are zero hold distinct indices.
template <int V>
__device__ __forceinline__ float warp_sum_transpose(float (&v)[V], int lane, int &idx)
{
    static_assert(V == 1 || V == 2 || V == 4 || V == 8 || V == 16 || V == 32, "V");
    idx = 0;
    int n = V;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        if (n > 1) {
            const bool up = (lane & o) != 0;
#pragma unroll
            for (int i = 0; i < V / 2; ++i) {
                if (i < n / 2) {
                    float send = up ? v[i] : v[i + n / 2];
                    float keep = up ? v[i + n / 2] : v[i];
                    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                }
            }
            if (up)
                idx += n / 2;
            n /= 2;
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
        }
    }
    return v[0];
}

}  // namespace q4
