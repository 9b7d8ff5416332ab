// The C ABI declared in include/q4.h: host-side validation, kernel selection by
// M, workspace accounting and error reporting.  Nothing here allocates device
// memory or synchronises; every launch goes to the caller's stream.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <cuda.h>
#include <mutex>

#include "q4_internal.h"

namespace q4 {

// The library's device-side error word (Q4_DEVERR_* bits), one per device.
__device__ unsigned g_q4_device_error;

static thread_local char g_last_error[512] = "";
// Smallest M served by the tcgen05 kernel (below it the CUDA-core streaming
// kernels run, one launch per block of up to four tokens).
static constexpr int kTensorCoreMinM = 5;
static std::atomic<unsigned> g_flags{0u};

q4_status fail(q4_status s, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return s;
}

q4_status cuda_fail(cudaError_t e, const char *what)
{
    return fail(Q4_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

q4_status current_device(DeviceInfo &out)
{
    static std::mutex mu;
    static DeviceInfo cache[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64)
        return fail(Q4_ERR_DEVICE, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lock(mu);
    DeviceInfo &c = cache[dev];
    if (c.device != dev) {
        DeviceInfo d;
        d.device = dev;
        int v = 0;
        if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute");
        d.smem_optin = (size_t)v;
        c = d;
    }
    out = c;
    if (out.cc_major != 10 || out.cc_minor != 3)
        return fail(Q4_ERR_DEVICE, "device %d is sm_%d%d; this library is built for sm_103a",
                    dev, out.cc_major, out.cc_minor);
    return Q4_OK;
}

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);

void *current_context()
{
    static CtxGetCurrentFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(p);
    });
    CUcontext c = nullptr;
    if (!fn || fn(&c) != CUDA_SUCCESS)
        return nullptr;
    return c;
}

unsigned *device_error_flags()
{
    static std::mutex mu;
    static void *ctx_of[64] = {};
    static unsigned *addr[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return nullptr;
    void *ctx = current_context();
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev] || !ctx || ctx_of[dev] != ctx) {
        void *a = nullptr;
        if (cudaGetSymbolAddress(&a, g_q4_device_error) != cudaSuccess)
            return nullptr;
        addr[dev] = static_cast<unsigned *>(a);
        ctx_of[dev] = ctx;
    }
    return addr[dev];
}

static bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

// Workspace layout: [tickets: u32, padded to 256 B][partials: fp32].
struct WsLayout {
    size_t tickets_off = 0, partial_off = 0, total = 0;
};

static size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Upper bound over every plan gemv_plan can choose for this shape
// (independent of the device): partial slots for N rows rounded up to a whole
// stage (64 rows) x k-steps x up to 4 tokens, one counter per row group.
static WsLayout stream_ws_layout(int kind, int M, int N, int K)
{
    WsLayout L;
    const int kstep = kind == W_BF16 ? 256 : 1024;
    const size_t S = (size_t)((K + kstep - 1) / kstep);
    const size_t mt = M >= 4 ? 4 : (M >= 2 ? 2 : 1);
    const size_t rows = (size_t)((N + 63) / 64) * 64;
    const size_t tickets = (size_t)N + 64;
    L.tickets_off = 0;
    L.partial_off = round_up(tickets * 4, 256);
    L.total = S > 1 ? L.partial_off + rows * S * mt * 4 : 0;
    return L;
}

static q4_status check_common(int M, int N, int K, void *ws, size_t ws_bytes, size_t need,
                              const void *x, const void *w, const void *y)
{
    if (!x || !w || !y)
        return fail(Q4_ERR_NULL, "x, weights and y must not be NULL");
    if (M < 1 || N < 1)
        return fail(Q4_ERR_SHAPE, "M=%d and N=%d must be >= 1", M, N);
    if (!aligned(x, 16) || !aligned(w, 16) || !aligned(y, 16))
        return fail(Q4_ERR_ALIGN, "x, weights and y must be 16-byte aligned");
    if (need > 0) {
        if (!ws)
            return fail(Q4_ERR_WORKSPACE, "workspace of %zu bytes required, got NULL", need);
        if (ws_bytes < need)
            return fail(Q4_ERR_WORKSPACE, "workspace of %zu bytes required, got %zu", need, ws_bytes);
        if (!aligned(ws, 16))
            return fail(Q4_ERR_ALIGN, "workspace must be 16-byte aligned");
    }
    (void)K;
    return Q4_OK;
}

static q4_status run_stream(int kind, GemvParams p, int M, int N, int K, void *ws,
                            cudaStream_t st)
{
    DeviceInfo dev;
    q4_status s = current_device(dev);
    if (s != Q4_OK)
        return s;
    const WsLayout L = stream_ws_layout(kind, M, N, K);
    const bool pdl = (g_flags.load() & Q4_FLAG_PDL) != 0;
    unsigned char *wsb = static_cast<unsigned char *>(ws);
    p.N = N;
    p.K = K;
    if (rows_eligible(kind, K)) {
        RowsPlan plan;
        if ((s = rows_plan(dev, kind, M, N, K, plan)) == Q4_OK)
            return rows_launch(plan, p, M, st, pdl);
    }
    GemvPlan plan;
    if ((s = gemv_plan(dev, kind, M, N, K, plan)) != Q4_OK)
        return s;
    const bool split = plan.ws_floats > 0;
    if (split && (ws == nullptr || plan.ws_floats * 4 + L.partial_off > L.total ||
                  plan.tickets * 4 > L.partial_off))
        return fail(Q4_ERR_WORKSPACE, "internal: plan exceeds the workspace bound");
    p.tickets = split ? reinterpret_cast<unsigned *>(wsb + L.tickets_off) : nullptr;
    p.ws = split ? reinterpret_cast<float *>(wsb + L.partial_off) : nullptr;
    return gemv_launch(plan, p, M, st, pdl);
}

}  // namespace q4

using namespace q4;

extern "C" {

int q4_abi_version(void) { return Q4_ABI_VERSION; }

const char *q4_status_string(q4_status s)
{
    switch (s) {
    case Q4_OK: return "ok";
    case Q4_ERR_NULL: return "null pointer";
    case Q4_ERR_SHAPE: return "invalid shape";
    case Q4_ERR_ALIGN: return "misaligned pointer";
    case Q4_ERR_WORKSPACE: return "workspace too small";
    case Q4_ERR_ARG: return "invalid argument";
    case Q4_ERR_CUDA: return "CUDA error";
    case Q4_ERR_DEVICE: return "unsupported device";
    }
    return "unknown status";
}

const char *q4_last_error_string(void) { return g_last_error; }

q4_status q4_set_launch_flags(unsigned flags)
{
    const unsigned known =
        Q4_FLAG_PDL | Q4_FLAG_FORCE_CUDA_CORE | Q4_FLAG_FORCE_TENSOR_CORE;
    if (flags & ~known)
        return fail(Q4_ERR_ARG, "unknown launch flags 0x%x", flags & ~known);
    if ((flags & Q4_FLAG_FORCE_CUDA_CORE) && (flags & Q4_FLAG_FORCE_TENSOR_CORE))
        return fail(Q4_ERR_ARG, "cannot force both the CUDA-core and the tensor-core kernel");
    g_flags.store(flags);
    return Q4_OK;
}

unsigned q4_get_launch_flags(void) { return g_flags.load(); }

size_t q4_workspace_bytes(int layout, int M, int N, int K)
{
    if (M < 1 || N < 1 || K < 1)
        return 0;
    int sms = 0, dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        (void)cudaGetLastError();
        sms = 160;   // no device: size for a GB300-class part
    }
    size_t a = 0;
    int kind = 0;
    if (layout == Q4_LAYOUT_INT4G128) {
        if (K % 128)
            return 0;
        kind = W_INT4;
    } else if (layout == Q4_LAYOUT_NVFP4) {
        if (K % 16)
            return 0;
        kind = W_NVFP4_A16;
    } else {
        return 0;
    }
    a = stream_ws_layout(kind, M, N, K).total;
    // the tensor-core path (and its copy of x) only when the call can take it
    const bool tc = M >= kTensorCoreMinM || (g_flags.load() & Q4_FLAG_FORCE_TENSOR_CORE);
    const size_t b = tc ? tc_workspace_bytes(kind, M, N, K, sms) : 0;
    return a > b ? a : b;
}

q4_status q4_linear_int4g128(const void *x, const uint8_t *qweight, const void *scale,
                             const void *minv, void *y, int M, int N, int K, void *workspace,
                             size_t workspace_bytes, void *stream)
{
    if (!scale || !minv)
        return fail(Q4_ERR_NULL, "scale and min must not be NULL");
    if (K < 128 || K % 128)
        return fail(Q4_ERR_SHAPE, "int4-g128 needs K >= 128 and K %% 128 == 0 (K=%d)", K);
    const size_t need = q4_workspace_bytes(Q4_LAYOUT_INT4G128, M, N, K);
    q4_status s = check_common(M, N, K, workspace, workspace_bytes, need, x, qweight, y);
    if (s != Q4_OK)
        return s;
    if (!aligned(scale, 2) || !aligned(minv, 2))
        return fail(Q4_ERR_ALIGN, "scale and min must be 2-byte aligned");
    const unsigned flags = g_flags.load();
    const bool tc_ok = tc_eligible(W_INT4, M, N, K);
    if ((flags & Q4_FLAG_FORCE_TENSOR_CORE) && !tc_ok)
        return fail(Q4_ERR_ARG, "the tensor-core path needs K %% 64 == 0");
    if (tc_ok && !(flags & Q4_FLAG_FORCE_CUDA_CORE) &&
        ((flags & Q4_FLAG_FORCE_TENSOR_CORE) || M >= kTensorCoreMinM))
        return tc_launch(W_INT4, x, qweight, scale, minv, nullptr, y, M, N, K, workspace,
                         workspace_bytes, static_cast<cudaStream_t>(stream),
                         (flags & Q4_FLAG_PDL) != 0);
    GemvParams p = {};
    p.x = static_cast<const uint16_t *>(x);
    p.w = qweight;
    p.w_row_bytes = K / 2;
    p.scale = scale;
    p.minv = static_cast<const uint16_t *>(minv);
    p.y = static_cast<uint16_t *>(y);
    p.ldy = N;
    p.row_begin = 0;
    p.n_rows = N;
    p.extra_row = -1;
    return run_stream(W_INT4, p, M, N, K, workspace, static_cast<cudaStream_t>(stream));
}

q4_status q4_linear_nvfp4(const void *x, const uint8_t *codes, const uint8_t *scale_e4m3,
                          const float *global_scale, void *y, int M, int N, int K,
                          void *workspace, size_t workspace_bytes, void *stream)
{
    if (!scale_e4m3 || !global_scale)
        return fail(Q4_ERR_NULL, "scale_e4m3 and global_scale must not be NULL");
    if (K < 16 || K % 16)
        return fail(Q4_ERR_SHAPE, "NVFP4 needs K >= 16 and K %% 16 == 0 (K=%d)", K);
    const size_t need = q4_workspace_bytes(Q4_LAYOUT_NVFP4, M, N, K);
    q4_status s = check_common(M, N, K, workspace, workspace_bytes, need, x, codes, y);
    if (s != Q4_OK)
        return s;
    if (!aligned(global_scale, 4))
        return fail(Q4_ERR_ALIGN, "global_scale must be 4-byte aligned");
    if (K % 32 == 0 && !aligned(scale_e4m3, 2))
        return fail(Q4_ERR_ALIGN, "scale_e4m3 must be 2-byte aligned");
    const unsigned flags = g_flags.load();
    const bool tc_ok = tc_eligible(W_NVFP4_A16, M, N, K) && aligned(scale_e4m3, 4);
    if ((flags & Q4_FLAG_FORCE_TENSOR_CORE) && !tc_ok)
        return fail(Q4_ERR_ARG, "the tensor-core path needs K %% 64 == 0");
    if (tc_ok && !(flags & Q4_FLAG_FORCE_CUDA_CORE) &&
        ((flags & Q4_FLAG_FORCE_TENSOR_CORE) || M >= kTensorCoreMinM))
        return tc_launch(W_NVFP4_A16, x, codes, scale_e4m3, nullptr, global_scale, y, M, N, K,
                         workspace, workspace_bytes, static_cast<cudaStream_t>(stream),
                         (flags & Q4_FLAG_PDL) != 0);
    GemvParams p = {};
    p.x = static_cast<const uint16_t *>(x);
    p.w = codes;
    p.w_row_bytes = K / 2;
    p.scale = scale_e4m3;
    p.gscale = global_scale;
    p.y = static_cast<uint16_t *>(y);
    p.ldy = N;
    p.row_begin = 0;
    p.n_rows = N;
    p.extra_row = -1;
    const int kind = (K % 32 == 0) ? W_NVFP4_A16 : W_NVFP4_A8;
    return run_stream(kind, p, M, N, K, workspace, static_cast<cudaStream_t>(stream));
}

q4_status audio_head_logits_restricted(const void *h, const void *head, int R_total,
                                       int row_begin, int n_rows, int extra_row, void *logits,
                                       int M, int H, void *stream)
{
    if (!h || !head || !logits)
        return fail(Q4_ERR_NULL, "h, head and logits must not be NULL");
    if (M < 1 || H < 8 || H % 8)
        return fail(Q4_ERR_SHAPE, "head needs M >= 1, H >= 8 and H %% 8 == 0 (M=%d, H=%d)", M, H);
    if (R_total < 1 || row_begin < 0 || n_rows < 0 || (int64_t)row_begin + n_rows > R_total)
        return fail(Q4_ERR_ARG, "rows [%d, %d) outside the head's %d rows", row_begin,
                    row_begin + n_rows, R_total);
    if (extra_row < -1 || extra_row >= R_total)
        return fail(Q4_ERR_ARG, "extra_row %d outside [-1, %d)", extra_row, R_total);
    const int cols = n_rows + (extra_row >= 0 ? 1 : 0);
    if (cols < 1)
        return fail(Q4_ERR_SHAPE, "the restricted head has no output column");
    if (!aligned(h, 16) || !aligned(head, 16) || !aligned(logits, 2))
        return fail(Q4_ERR_ALIGN, "h and head must be 16-byte aligned, logits 2-byte aligned");
    GemvParams p = {};
    p.x = static_cast<const uint16_t *>(h);
    p.w = static_cast<const uint8_t *>(head);
    p.w_row_bytes = (int64_t)H * 2;
    p.y = static_cast<uint16_t *>(logits);
    p.ldy = cols;
    p.row_begin = row_begin;
    p.n_rows = n_rows;
    p.extra_row = extra_row;
    return run_stream(W_BF16, p, M, cols, H, nullptr, static_cast<cudaStream_t>(stream));
}

q4_status q4_device_error_flags(unsigned *flags, int clear)
{
    if (!flags)
        return fail(Q4_ERR_NULL, "flags must not be NULL");
    unsigned *addr = device_error_flags();
    if (!addr)
        return fail(Q4_ERR_CUDA, "cannot locate the device error word");
    cudaError_t e = cudaMemcpy(flags, addr, sizeof(unsigned), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaMemcpy(device error word)");
    if (clear && (e = cudaMemset(addr, 0, sizeof(unsigned))) != cudaSuccess)
        return cuda_fail(e, "cudaMemset(device error word)");
    return Q4_OK;
}

q4_status q4_dequant_int4g128_f32(const uint8_t *qweight, const void *scale, const void *minv,
                                  float *w, int N, int K, void *stream)
{
    if (!qweight || !scale || !minv || !w)
        return fail(Q4_ERR_NULL, "NULL argument");
    if (N < 1 || K < 128 || K % 128)
        return fail(Q4_ERR_SHAPE, "int4-g128 dequant needs N >= 1, K %% 128 == 0");
    if (!aligned(qweight, 4) || !aligned(w, 16) || !aligned(scale, 2) || !aligned(minv, 2))
        return fail(Q4_ERR_ALIGN, "misaligned argument");
    DeviceInfo dev;
    q4_status s = current_device(dev);
    if (s != Q4_OK)
        return s;
    return launch_dequant_int4(qweight, static_cast<const uint16_t *>(scale),
                               static_cast<const uint16_t *>(minv), w, N, K,
                               static_cast<cudaStream_t>(stream));
}

q4_status q4_dequant_nvfp4_f32(const uint8_t *codes, const uint8_t *scale_e4m3,
                               const float *global_scale, float *w, int N, int K, void *stream)
{
    if (!codes || !scale_e4m3 || !global_scale || !w)
        return fail(Q4_ERR_NULL, "NULL argument");
    if (N < 1 || K < 16 || K % 16)
        return fail(Q4_ERR_SHAPE, "NVFP4 dequant needs N >= 1, K %% 16 == 0");
    if (!aligned(codes, 4) || !aligned(w, 16) || !aligned(global_scale, 4))
        return fail(Q4_ERR_ALIGN, "misaligned argument");
    DeviceInfo dev;
    q4_status s = current_device(dev);
    if (s != Q4_OK)
        return s;
    return launch_dequant_nvfp4(codes, scale_e4m3, global_scale, w, N, K,
                                static_cast<cudaStream_t>(stream));
}

q4_status q4_linear_int8(const void *x, const int8_t *qweight, const void *scale, void *y,
                         int M, int N, int K, void *stream)
{
    if (!scale)
        return fail(Q4_ERR_NULL, "scale must not be NULL");
    if (K < 16 || K % 16)
        return fail(Q4_ERR_SHAPE, "INT8 weight-only needs K >= 16 and K %% 16 == 0 (K=%d)", K);
    q4_status s = check_common(M, N, K, nullptr, 0, 0, x, qweight, y);
    if (s != Q4_OK)
        return s;
    if (!aligned(scale, 2))
        return fail(Q4_ERR_ALIGN, "scale must be 2-byte aligned");
    if (!rows_eligible(W_INT8, K))
        return fail(Q4_ERR_SHAPE, "INT8 weight-only supports K up to 8192 (K=%d)", K);
    DeviceInfo dev;
    if ((s = current_device(dev)) != Q4_OK)
        return s;
    GemvParams p = {};
    p.x = static_cast<const uint16_t *>(x);
    p.w = reinterpret_cast<const uint8_t *>(qweight);
    p.w_row_bytes = K;
    p.scale = scale;
    p.y = static_cast<uint16_t *>(y);
    p.ldy = N;
    p.N = N;
    p.K = K;
    p.row_begin = 0;
    p.n_rows = N;
    p.extra_row = -1;
    RowsPlan plan;
    if ((s = rows_plan(dev, W_INT8, M, N, K, plan)) != Q4_OK)
        return s;
    return rows_launch(plan, p, M, static_cast<cudaStream_t>(stream),
                       (g_flags.load() & Q4_FLAG_PDL) != 0);
}

q4_status q4_embedding_int8(const int32_t *ids, const int8_t *qweight, const void *scale,
                            void *out, int M, int V, int H, void *stream)
{
    if (!ids || !qweight || !scale || !out)
        return fail(Q4_ERR_NULL, "NULL argument");
    if (M < 1 || V < 1 || H < 16 || H % 16)
        return fail(Q4_ERR_SHAPE, "embedding gather needs M, V >= 1 and H %% 16 == 0 (H=%d)", H);
    if (!aligned(qweight, 16) || !aligned(out, 16) || !aligned(ids, 4) || !aligned(scale, 2))
        return fail(Q4_ERR_ALIGN, "qweight and out must be 16-byte, ids 4-byte, scale 2-byte aligned");
    DeviceInfo dev;
    q4_status s = current_device(dev);
    if (s != Q4_OK)
        return s;
    const bool pdl = (g_flags.load() & Q4_FLAG_PDL) != 0;
    return launch_embedding_int8(ids, qweight, static_cast<const uint16_t *>(scale),
                                 static_cast<uint16_t *>(out), M, V, H,
                                 static_cast<cudaStream_t>(stream), pdl);
}

q4_status q4_quantize_int4g128(const void *w, uint8_t *qweight, void *scale, void *minv, int N,
                               int K, void *stream)
{
    if (!w || !qweight || !scale || !minv)
        return fail(Q4_ERR_NULL, "NULL argument");
    if (N < 1 || K < 128 || K % 128)
        return fail(Q4_ERR_SHAPE, "int4-g128 quantiser needs N >= 1, K %% 128 == 0");
    if (!aligned(w, 8) || !aligned(qweight, 2) || !aligned(scale, 2) || !aligned(minv, 2))
        return fail(Q4_ERR_ALIGN, "w must be 8-byte, qweight/scale/min 2-byte aligned");
    DeviceInfo dev;
    q4_status s = current_device(dev);
    if (s != Q4_OK)
        return s;
    return launch_quantize_int4(static_cast<const uint16_t *>(w), qweight,
                                static_cast<uint16_t *>(scale), static_cast<uint16_t *>(minv),
                                N, K, static_cast<cudaStream_t>(stream));
}

q4_status q4_quantize_nvfp4(const void *w, uint8_t *codes, uint8_t *scale_e4m3,
                            float *global_scale, int N, int K, void *stream)
{
    if (!w || !codes || !scale_e4m3 || !global_scale)
        return fail(Q4_ERR_NULL, "NULL argument");
    if (N < 1 || K < 16 || K % 16)
        return fail(Q4_ERR_SHAPE, "NVFP4 quantiser needs N >= 1, K %% 16 == 0");
    if (!aligned(w, 16) || !aligned(codes, 8) || !aligned(global_scale, 4))
        return fail(Q4_ERR_ALIGN, "w must be 16-byte, codes 8-byte, global scale 4-byte aligned");
    DeviceInfo dev;
    q4_status s = current_device(dev);
    if (s != Q4_OK)
        return s;
    return launch_quantize_nvfp4(static_cast<const uint16_t *>(w), codes, scale_e4m3,
                                 global_scale, N, K, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
