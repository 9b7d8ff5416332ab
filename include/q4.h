/*
 * q4.h -- C ABI of the GB300 (sm_103a) 4-bit weight-only linear library.
 *
 * Every entry point takes plain pointers and sizes.  Unless a comment says
 * otherwise, pointers are DEVICE pointers, tensors are row-major and contiguous,
 * the caller owns (allocates and frees) every buffer, and the library allocates
 * nothing.  Calls are asynchronous on the given stream (`stream` is a
 * cudaStream_t passed as void*; NULL means the legacy default stream) and issue
 * no host synchronisation, so they can be recorded into a CUDA graph.
 *
 * Error behaviour: arguments are validated on the host before anything is
 * launched.  A failed check returns a non-zero q4_status and launches nothing.
 * A failed launch returns Q4_ERR_CUDA.  q4_last_error_string() gives the detail
 * of the last failure on the calling host thread.
 *
 * Weight layouts (the two the source pages fix exactly):
 *   int4-g128-minmax -- "rumik-oss-1-int4", section "Format
 *     (rumik-int4-g128-minmax-v1)": qweight uint8 [N, K/2], two 4-bit codes per
 *     byte, the low nibble holds the even column; scale and min fp16
 *     [N, K/128]; w[n,k] = code[n,k] * scale[n,k/128] + min[n,k/128].
 *     Codes are unsigned 0..15.
 *   NVFP4 weight-only -- "VoxCPM2 NVFP4 (GPTQ)", section "NVFP4 settings":
 *     E2M1 codes uint8 [N, K/2] (same nibble order as int4), float8_e4m3fn group
 *     scales uint8 [N, K/16] (one per 16 columns), one fp32 global scale per
 *     matrix which multiplies: w[n,k] = E2M1(code) * e4m3(scale[n,k/16]) * g.
 *     Activations stay BF16 (there is no activation scale).
 * Activations x and outputs y are bf16; the output is rounded to bf16 (round to
 * nearest even) from an fp32 row sum.  Below five tokens that sum is built from
 * exact int32 dot products (int4, x scaled to int16 per 32 columns) or from fp16
 * partial sums of at most eight products per half group (NVFP4); from five tokens
 * on, the tensor cores multiply 16-bit operands into fp32 accumulators: for
 * int4, fp16 (x scaled per token by a power of two that keeps every bf16 value in
 * the fp16 range, and the weights rounded once to fp16); for NVFP4, bf16 (x as
 * stored, and the weights E2M1 * e4m3, exact in bf16 after a power-of-two share of
 * the global scale, the rest of which is applied to the accumulator).
 */
#ifndef Q4_GB300_H
#define Q4_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define Q4_ABI_VERSION 1

typedef enum {
    Q4_OK = 0,
    Q4_ERR_NULL = 1,       /* a required pointer is NULL                          */
    Q4_ERR_SHAPE = 2,      /* a size is out of range or not a multiple it must be */
    Q4_ERR_ALIGN = 3,      /* a pointer is not 16-byte aligned                    */
    Q4_ERR_WORKSPACE = 4,  /* workspace too small (see q4_workspace_bytes)        */
    Q4_ERR_ARG = 5,        /* any other invalid argument (row index, flag, ...)   */
    Q4_ERR_CUDA = 6,       /* a CUDA runtime call or kernel launch failed         */
    Q4_ERR_DEVICE = 7      /* the current device is not a compute-capability 10.3 GPU */
} q4_status;

/* Layout identifiers for q4_workspace_bytes. */
#define Q4_LAYOUT_INT4G128 0
#define Q4_LAYOUT_NVFP4 1

/* Process-wide launch flags (q4_set_launch_flags).  Default: 0.
 *   Q4_FLAG_PDL: launch with programmatic dependent launch.  A kernel may then
 *     start reading its weights, scales and global scale before the previous
 *     kernel on the stream has finished, so those buffers must not be written
 *     by the immediately preceding kernel.  Activations, outputs and workspace
 *     are touched only after the previous kernel has completed.
 *   Q4_FLAG_FORCE_CUDA_CORE / Q4_FLAG_FORCE_TENSOR_CORE: override the choice of
 *     kernel by M (testing and benchmarking only). */
#define Q4_FLAG_PDL 0x1u
#define Q4_FLAG_FORCE_CUDA_CORE 0x2u
#define Q4_FLAG_FORCE_TENSOR_CORE 0x4u

int q4_abi_version(void);
const char *q4_status_string(q4_status s);
/* Detail of the last non-OK status returned on this host thread ("" if none). */
const char *q4_last_error_string(void);
q4_status q4_set_launch_flags(unsigned flags);
unsigned q4_get_launch_flags(void);

/*
 * Bytes of device workspace that q4_linear_int4g128 (layout 0) or
 * q4_linear_nvfp4 (layout 1) needs for an [M,N,K] call on the current device:
 * split-K partial sums and arrival counters of whichever kernel the call may use
 * under the current launch flags, and for int4 above 64 tokens the per-token
 * prescaled fp16 copy of x and its scales that the tensor-core path reads (the
 * tensor-core part counts from M = 5 on, or for any M while
 * Q4_FLAG_FORCE_TENSOR_CORE is set).
 * The workspace must be zero-filled once after allocation; every call leaves
 * its counters at zero again.  Calls that run concurrently must not share a
 * workspace.  Returns 0 for invalid sizes.
 */
size_t q4_workspace_bytes(int layout, int M, int N, int K);

/*
 * y[M,N] = x[M,K] * W^T for the int4-g128-minmax layout.
 *   x        bf16 [M, K]
 *   qweight  uint8 [N, K/2]     low nibble = even column
 *   scale    fp16 [N, K/128]
 *   minv     fp16 [N, K/128]
 *   y        bf16 [M, N]        written
 * Requirements: M >= 1, N >= 1, K >= 128, K % 128 == 0; x, qweight, y and the
 * workspace 16-byte aligned, scale/minv 2-byte aligned; workspace of at least
 * q4_workspace_bytes(0, M, N, K) bytes (may be NULL when that is 0).
 * M selects the kernel: a CUDA-core GEMV for M <= 4 (one launch per block of up
 * to four tokens), the tcgen05 tensor-core GEMM for M >= 5 when K % 64 == 0.
 */
q4_status q4_linear_int4g128(const void *x, const uint8_t *qweight, const void *scale,
                             const void *minv, void *y, int M, int N, int K,
                             void *workspace, size_t workspace_bytes, void *stream);

/*
 * y[M,N] = x[M,K] * W^T for the NVFP4 weight-only layout.
 *   x             bf16 [M, K]
 *   codes         uint8 [N, K/2]   low nibble = even column, E2M1 (bit 3 = sign)
 *   scale_e4m3    uint8 [N, K/16]  float8_e4m3fn bit patterns
 *   global_scale  fp32 [1]         DEVICE pointer, multiplies every weight
 *   y             bf16 [M, N]      written
 * Requirements: M >= 1, N >= 1, K >= 16, K % 16 == 0; x, codes, y and the
 * workspace 16-byte aligned; workspace as for q4_linear_int4g128 (layout 1).
 */
q4_status q4_linear_nvfp4(const void *x, const uint8_t *codes, const uint8_t *scale_e4m3,
                          const float *global_scale, void *y, int M, int N, int K,
                          void *workspace, size_t workspace_bytes, void *stream);

/*
 * q4_linear_int4g128 for callers that cannot allocate device memory: code that
 * runs where the CUDA allocator must not be called (inside an audio or other
 * real-time callback that may not block, in a plugin whose host application owns
 * every device buffer, after a memory pool has been frozen) and so cannot hand
 * this library a workspace.  The source pages have no counterpart to this entry
 * point; it exists for such deployments.
 *
 * Same arguments, layout and result as q4_linear_int4g128 minus the workspace.
 * It runs the split-K CUDA-core kernel with its scratch (arrival counters and
 * partial sums) in a static device array of 4 MiB that is part of the library:
 * every GPU that loads the library keeps those 4 MiB until the process exits.
 * Shapes whose scratch would exceed 4 MiB are rejected with Q4_ERR_SHAPE (for
 * M <= 4 this covers N * ceil(K / 1024) up to about 250,000 per token block).
 * The call allocates and frees nothing.  The first call on a device looks up the
 * array's device address (with that device current); make that first call
 * before starting any stream capture.  Every call clears the counters it needs
 * with an asynchronous memset on `stream`, then launches the kernel.  All calls
 * share the one array, which keeps the last call's contents: calls whose work
 * overlaps on the GPU (other streams or host threads) race on it and must be
 * serialised by the caller.
 */
q4_status q4_linear_int4g128_noalloc(const void *x, const uint8_t *qweight, const void *scale,
                                     const void *minv, void *y, int M, int N, int K,
                                     void *stream);

/*
 * Restricted output head -- "Rumik TTS Fast Inference", section "What Made It
 * Faster" and Figure 3: project the hidden state only onto the rows of the
 * current codebook (2,048 codes) plus the end token, 2,049 rows instead of the
 * full vocabulary.
 *   h          bf16 [M, H]
 *   head       bf16 [R_total, H]   the (audio) head matrix, row-major
 *   logits     bf16 [M, n_rows + (extra_row >= 0)]   written
 * Column j < n_rows of logits is row (row_begin + j) of head; when
 * extra_row >= 0 the last column is row extra_row (the end token).
 * Requirements: M >= 1, H >= 8, H % 8 == 0, 0 <= row_begin,
 * row_begin + n_rows <= R_total, -1 <= extra_row < R_total, at least one output
 * column; h and head 16-byte aligned.  Uses no workspace.
 */
q4_status audio_head_logits_restricted(const void *h, const void *head, int R_total,
                                       int row_begin, int n_rows, int extra_row,
                                       void *logits, int M, int H, void *stream);

/*
 * Device-side error word of the current device.  Bit 0 (Q4_DEVERR_TIMEOUT) is set
 * when a bounded wait inside a kernel gave up (a copy or a peer warp never
 * arrived); the kernel then returned early and its output is not valid.  This
 * call synchronises with the device (it is a diagnostic, not for the hot path);
 * with clear != 0 the word is reset to zero afterwards.
 */
#define Q4_DEVERR_TIMEOUT 0x1u
/* Bit 2: q4_embedding_int8 met a token id outside 0 .. V-1 and wrote a row of
 * zeros for it. */
#define Q4_DEVERR_INDEX 0x4u
q4_status q4_device_error_flags(unsigned *flags, int clear);

/*
 * Test helpers: decode whole weight matrices to fp32 [N, K] with the same
 * in-register decoders the linear kernels use.  Each weight is the exact value
 * of the layout's formula rounded once to fp32.
 */
q4_status q4_dequant_int4g128_f32(const uint8_t *qweight, const void *scale,
                                  const void *minv, float *w, int N, int K, void *stream);
q4_status q4_dequant_nvfp4_f32(const uint8_t *codes, const uint8_t *scale_e4m3,
                               const float *global_scale, float *w, int N, int K,
                               void *stream);

/*
 * INT8 weight-only linear ("Rumik TTS Fast Inference", "What Made It Faster": INT8
 * weight-only decode projections; the layout is not given there).  Reading, after
 * the int8 scheme "rumik-oss-1-int4" gives for its embedding: qweight int8 [N, K]
 * (signed), scale fp16 [N] (one per output row), w[n, k] = q[n, k] * scale[n].
 * y[M, N] = x[M, K] W^T with x, y bf16, fp32 accumulation, bf16 store.  Runs the
 * whole-row CUDA-core kernel (one launch per 1, 2 or 4 tokens; K > 4096 one token
 * per launch); no workspace.  K % 16 == 0 and K <= 8192; x, qweight, y 16-byte
 * aligned, scale 2-byte.
 */
q4_status q4_linear_int8(const void *x_bf16, const int8_t *qweight, const void *scale_f16,
                         void *y_bf16, int M, int N, int K, void *stream);

/*
 * Token-embedding gather with int8 dequantisation ("rumik-oss-1-int4", "Format":
 * embed_tokens.qweight int8 [V, H], scale fp16 [V]): for each of the M token ids
 * (int32, device memory, typically written by the sampler of the previous step),
 * out[m, k] = bf16(q[ids[m], k] * scale[ids[m]]).  The codes are read as signed
 * two's complement with one symmetric scale per row (the page gives the shapes
 * only); the product is exact in fp32 and rounded once to bf16 (nearest even).
 * An id outside 0 .. V-1 writes a row of zeros and sets Q4_DEVERR_INDEX; nothing
 * outside the table is read.  H % 16 == 0; qweight and out 16-byte aligned, ids
 * 4-byte, scale 2-byte.  With Q4_FLAG_PDL the ids are read after the previous
 * kernel in the stream has finished (griddepcontrol.wait).
 */
q4_status q4_embedding_int8(const int32_t *ids, const int8_t *qweight, const void *scale_f16,
                            void *out_bf16, int M, int V, int H, void *stream);

/*
 * Round-to-nearest quantisers: BF16 weights w [N, K] (row-major, device memory)
 * into the two layouts, for packing a checkpoint (not for the decode path).
 * Every arithmetic step is one IEEE fp32 operation rounded to nearest even.
 *
 * q4_quantize_int4g128 ("rumik-oss-1-int4", "Format (rumik-int4-g128-minmax-v1)";
 * the min/max form the layout's name refers to): per row and group of 128
 * columns, lo = min w, hi = max w; scale = fp16((hi - lo) / 15); min = fp16(lo);
 * code = clamp(rint((w - min) / scale), 0, 15) (0 when the fp16 scale is 0).
 * Outputs qweight [N, K/2] (low nibble = even column), scale and min fp16
 * [N, K/128].  K % 128 == 0; w 8-byte, the outputs 2-byte aligned.  Values whose
 * magnitude exceeds the fp16 range give an infinite scale or min.
 *
 * q4_quantize_nvfp4 ("VoxCPM2 NVFP4 (GPTQ)", "NVFP4 settings": E2M1 codes, group
 * 16, e4m3 group scales, one global scale; the pages' checkpoint used GPTQ, whose
 * error feedback is not reproduced -- this is plain rounding in the same format):
 * G = amax(w) / (6 * 448) (1 for an all-zero matrix); per group of 16 columns
 * s = e4m3((amax_group / 6) / G), nearest even, saturating at 448;
 * code = E2M1(w / (e4m3(s) * G)), nearest even, saturating at 6, magnitude 0
 * stored as +0.  Outputs codes [N, K/2] (low nibble = even column), e4m3 scales
 * [N, K/16] and the fp32 global scale (one float in device memory, overwritten;
 * decoding multiplies by it).  K % 16 == 0; w 16-byte, codes 8-byte, the global
 * scale 4-byte aligned.  Runs three kernels and a 4-byte memset on `stream`.
 *
 * The pages have no counterpart to these entry points' signatures; the layouts
 * they write are the pages'.
 */
q4_status q4_quantize_int4g128(const void *w_bf16, uint8_t *qweight, void *scale_f16,
                               void *min_f16, int N, int K, void *stream);
q4_status q4_quantize_nvfp4(const void *w_bf16, uint8_t *codes, uint8_t *scale_e4m3,
                            float *global_scale, int N, int K, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* Q4_GB300_H */
