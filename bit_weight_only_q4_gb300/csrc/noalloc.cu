// q4_linear_int4g128_noalloc: the int4-g128 linear layer for callers that cannot
// allocate device memory, such as code recorded into a CUDA graph after its
// memory pool is frozen, an audio or real-time callback that must never block in
// the allocator, or a plugin whose host application owns every device buffer.
//
// It runs the split-K register-path streaming kernel (gemv.cu) -- the kernel that
// otherwise takes its partial sums and arrival counters from the caller's
// workspace -- with that scratch in the file-scope array below instead.  The
// array is part of the loaded module: every GPU that loads the library holds
// kStaticScratchBytes of it until the process exits.  All calls share it, so
// calls whose kernels overlap on the GPU (different streams, different threads)
// race on it and must be serialised by the caller.
#include <mutex>

#include "q4_internal.h"

namespace q4 {

constexpr size_t kStaticScratchBytes = 4u << 20;   // 4 MiB

static __device__ __align__(256) unsigned char g_q4_static_scratch[kStaticScratchBytes];

// Device address of the scratch array on the current device.  The host-side
// name of a __device__ array is only a host stand-in, so the address is looked up
// with cudaGetSymbolAddress, with the device current, the first time a device is
// used, and cached for that device.  The cache also records the driver context
// the lookup was made in: after a cudaDeviceReset the device gets a new context
// (and the array a new address), so the lookup is made again there.
static q4_status static_scratch_address(void **out)
{
    static std::mutex mu;
    static void *addr[64] = {};
    static void *ctx_of[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64)
        return fail(Q4_ERR_DEVICE, "device ordinal %d out of range", dev);
    void *ctx = current_context();
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev] || !ctx || ctx_of[dev] != ctx) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_q4_static_scratch);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
        addr[dev] = p;
        ctx_of[dev] = ctx;
    }
    *out = addr[dev];
    return Q4_OK;
}

}  // namespace q4

using namespace q4;

extern "C" q4_status q4_linear_int4g128_noalloc(const void *x, const uint8_t *qweight,
                                                const void *scale, const void *minv, void *y,
                                                int M, int N, int K, void *stream)
{
    if (!x || !qweight || !scale || !minv || !y)
        return fail(Q4_ERR_NULL, "x, qweight, scale, min and y must not be NULL");
    if (M < 1 || N < 1)
        return fail(Q4_ERR_SHAPE, "M=%d and N=%d must be >= 1", M, N);
    if (K < 128 || K % 128)
        return fail(Q4_ERR_SHAPE, "int4-g128 needs K >= 128 and K %% 128 == 0 (K=%d)", K);
    auto is_aligned = [](const void *p, size_t a) { return ((uintptr_t)p % a) == 0; };
    if (!is_aligned(x, 16) || !is_aligned(qweight, 16) || !is_aligned(y, 16) ||
        !is_aligned(scale, 2) || !is_aligned(minv, 2))
        return fail(Q4_ERR_ALIGN, "x, qweight, y must be 16-byte and scale/min 2-byte aligned");
    DeviceInfo dev;
    q4_status s = current_device(dev);
    if (s != Q4_OK)
        return s;
    GemvPlan plan;
    if ((s = gemv_plan(dev, W_INT4, M, N, K, plan)) != Q4_OK)
        return s;
    // scratch layout: arrival counters (padded to 256 bytes), then partial sums
    const size_t tickets_bytes = (plan.tickets * 4 + 255) / 256 * 256;
    const size_t need = tickets_bytes + plan.ws_floats * 4;
    if (need > kStaticScratchBytes)
        return fail(Q4_ERR_SHAPE,
                    "M=%d N=%d K=%d needs %zu bytes of split-K scratch; the static scratch "
                    "holds %zu bytes", M, N, K, need, kStaticScratchBytes);
    void *scratch = nullptr;
    if ((s = static_scratch_address(&scratch)) != Q4_OK)
        return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned char *base = static_cast<unsigned char *>(scratch);
    if (plan.tickets > 0) {
        // the counters must start at zero; the array keeps the last call's contents
        cudaError_t e = cudaMemsetAsync(base, 0, plan.tickets * 4, st);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaMemsetAsync(static scratch counters)");
    }
    GemvParams p = {};
    p.x = static_cast<const uint16_t *>(x);
    p.w = qweight;
    p.w_row_bytes = K / 2;
    p.scale = scale;
    p.minv = static_cast<const uint16_t *>(minv);
    p.y = static_cast<uint16_t *>(y);
    p.ldy = N;
    p.N = N;
    p.K = K;
    p.row_begin = 0;
    p.n_rows = N;
    p.extra_row = -1;
    p.tickets = plan.tickets > 0 ? reinterpret_cast<unsigned *>(base) : nullptr;
    p.ws = plan.ws_floats > 0 ? reinterpret_cast<float *>(base + tickets_bytes) : nullptr;
    const bool pdl = (q4_get_launch_flags() & Q4_FLAG_PDL) != 0;
    return gemv_launch(plan, p, M, st, pdl);
}
