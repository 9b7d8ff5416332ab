// Host-side internals shared by the translation units of the library: launch
// parameter blocks, per-device properties and the error reporting used by the C
// ABI.  Not part of the public interface (include/q4.h is).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/q4.h"

namespace q4 {

// Per-call parameters of the CUDA-core weight-streaming kernel (GEMV for a few
// tokens, and the restricted head).  The output has N logical rows; logical row
// n reads physical weight row (n < n_rows ? row_begin + n : extra_row).
struct GemvParams {
    const uint16_t *x;        // bf16 [*, K]; this launch reads rows m0 .. m0+mcount-1
    const uint8_t *w;         // weight bytes, row-major
    int64_t w_row_bytes;      // bytes per physical weight row
    const void *scale;        // int4: fp16 [rows, K/128]; nvfp4: e4m3 [rows, K/16]
    const uint16_t *minv;     // int4: fp16 [rows, K/128]
    const float *gscale;      // nvfp4: device fp32 scalar
    uint16_t *y;              // bf16 [*, ldy]
    int64_t ldy;
    float *ws;                // split-K partial sums
    unsigned *tickets;        // one arrival counter per row group (left at zero)
    int mcount, m0;
    int N, K;
    int S;                    // k-steps per row group
    int G;                    // row groups
    int64_t U;                // units = G * S
    int64_t TW;               // warps in the grid
    int64_t gran;             // warp ranges are multiples of gran units (1 or S)
    int row_begin, n_rows, extra_row;
    // whole-row kernels: CTA b owns rows_q (+1 when b < rows_r) rows
    int rows_q, rows_r;
    // whole-row kernels, one token: nanoseconds to hold the prologue's ring
    // requests back (0: issue at once)
    unsigned ring_defer_ns;
    int grid;                 // CTAs
};

enum WeightKind { W_INT4 = 0, W_NVFP4_A16 = 1, W_NVFP4_A8 = 2, W_BF16 = 3, W_INT8 = 4 };

struct DeviceInfo {
    int device = -1;
    int sms = 0;
    int cc_major = 0, cc_minor = 0;
    size_t smem_optin = 0;
};

// Properties of the current device (cached per device).
q4_status current_device(DeviceInfo &out);

// Record an error detail for q4_last_error_string() and return `s`.
q4_status fail(q4_status s, const char *fmt, ...);
q4_status cuda_fail(cudaError_t e, const char *what);

// ---- CUDA-core weight-streaming kernels (gemv.cu)
struct GemvPlan {
    int kind = 0, mt = 1, rw = 4;
    int64_t gran = 1;
    int grid = 0;
    size_t smem = 0;
    int S = 0, G = 0;
    int64_t U = 0;
    size_t ws_floats = 0, tickets = 0;
};
// Choose the launch shape for an [M, N, K] problem of the given weight kind.
q4_status gemv_plan(const DeviceInfo &dev, int kind, int M, int N, int K, GemvPlan &plan);
// Launch ceil(M / plan.mt) kernels on `stream` (parameters filled per launch).
q4_status gemv_launch(const GemvPlan &plan, GemvParams p, int M, cudaStream_t stream,
                      bool pdl);

// ---- register-prefetch weight-streaming kernel (gemv_rows.cu)
struct RowsPlan {
    int kind = 0, mt = 1, w = 1, rb = 4, nb = 2, S = 1, grid = 0;
    bool direct = false;       // one-k-step rows stored from the cross-lane reduction
    size_t smem = 0;
};
bool rows_eligible(int kind, int K);
q4_status rows_plan(const DeviceInfo &dev, int kind, int M, int N, int K, RowsPlan &plan);
q4_status rows_launch(const RowsPlan &plan, GemvParams p, int M, cudaStream_t stream, bool pdl);

// ---- tcgen05 tensor-core GEMM (tc_gemm.cu)
bool tc_eligible(int kind, int M, int N, int K);
size_t tc_workspace_bytes(int kind, int M, int N, int K, int sms);
q4_status tc_launch(int kind, const void *x, const uint8_t *codes, const void *scale,
                    const void *minv, const float *gscale, void *y, int M, int N, int K,
                    void *ws, size_t ws_bytes, cudaStream_t stream, bool pdl);

// Device address of the library's error-flag word in the current context
// (looked up once per device and context; nullptr if the lookup fails).
unsigned *device_error_flags();

// The current CUDA driver context (nullptr when none is current or the driver
// entry point is unavailable); caches of device addresses are keyed on it, so a
// context created after cudaDeviceReset gets fresh lookups.
void *current_context();

// ---- test-only dequantisers (dequant.cu)
q4_status launch_dequant_int4(const uint8_t *q, const uint16_t *s, const uint16_t *m,
                              float *w, int N, int K, cudaStream_t st);
q4_status launch_dequant_nvfp4(const uint8_t *q, const uint8_t *s, const float *g,
                               float *w, int N, int K, cudaStream_t st);

// ---- int8 token-embedding gather (embedding.cu)
q4_status launch_embedding_int8(const int32_t *ids, const int8_t *q, const uint16_t *sc,
                                uint16_t *out, int M, int V, int H, cudaStream_t st, bool pdl);

// ---- round-to-nearest quantisers (quantize.cu)
q4_status launch_quantize_int4(const uint16_t *w, uint8_t *q, uint16_t *s, uint16_t *m, int N,
                               int K, cudaStream_t st);
q4_status launch_quantize_nvfp4(const uint16_t *w, uint8_t *q, uint8_t *s, float *gscale, int N,
                                int K, cudaStream_t st);

}  // namespace q4
