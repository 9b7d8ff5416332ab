"""Thin ctypes binding of the C ABI in ``include/q4.h`` (same entry-point names).

Only argument marshalling happens here: tensors are passed as raw device
pointers with their sizes and the current CUDA stream; every step of the
computation runs in the library's sm_103a kernels.  Output and workspace tensors
are allocated with PyTorch when the caller does not pass them (the library
itself never allocates).  If the shared library has not been built, the first
call raises :class:`Q4Error` -- there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

LAYOUT_INT4G128 = 0
LAYOUT_NVFP4 = 1
FLAG_PDL = 0x1
FLAG_FORCE_CUDA_CORE = 0x2
FLAG_FORCE_TENSOR_CORE = 0x4

STATUS = {0: "Q4_OK", 1: "Q4_ERR_NULL", 2: "Q4_ERR_SHAPE", 3: "Q4_ERR_ALIGN",
          4: "Q4_ERR_WORKSPACE", 5: "Q4_ERR_ARG", 6: "Q4_ERR_CUDA", 7: "Q4_ERR_DEVICE"}

_lib = None
_lock = threading.Lock()


class Q4Error(RuntimeError):
    def __init__(self, status: int, detail: str):
        self.status = status
        super().__init__(f"{STATUS.get(status, status)}: {detail}")


def lib_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load the shared library (raises Q4Error if it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = lib_path()
        if not os.path.exists(path):
            raise Q4Error(-1, f"{path} is missing: build it with "
                              f"`python -m bit_weight_only_q4_gb300.build` (no fallback exists)")
        L = ctypes.CDLL(path)
        p, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        st = ctypes.c_int
        sig = {
            "q4_abi_version": ([], ctypes.c_int),
            "q4_status_string": ([st], ctypes.c_char_p),
            "q4_last_error_string": ([], ctypes.c_char_p),
            "q4_set_launch_flags": ([ctypes.c_uint], st),
            "q4_get_launch_flags": ([], ctypes.c_uint),
            "q4_workspace_bytes": ([i, i, i, i], sz),
            "q4_linear_int4g128": ([p, p, p, p, p, i, i, i, p, sz, p], st),
            "q4_linear_nvfp4": ([p, p, p, p, p, i, i, i, p, sz, p], st),
            "q4_linear_int4g128_noalloc": ([p, p, p, p, p, i, i, i, p], st),
            "audio_head_logits_restricted": ([p, p, i, i, i, i, p, i, i, p], st),
            "q4_device_error_flags": ([ctypes.POINTER(ctypes.c_uint), i], st),
            "q4_dequant_int4g128_f32": ([p, p, p, p, i, i, p], st),
            "q4_dequant_nvfp4_f32": ([p, p, p, p, i, i, p], st),
            "q4_quantize_int4g128": ([p, p, p, p, i, i, p], st),
            "q4_embedding_int8": ([p, p, p, p, i, i, i, p], st),
            "q4_linear_int8": ([p, p, p, p, i, i, i, p], st),
            "q4_quantize_nvfp4": ([p, p, p, p, i, i, p], st),
        }
        for name, (args, res) in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
        return L


def symbols() -> list[str]:
    """Entry points the binding expects the library to export."""
    return ["q4_abi_version", "q4_status_string", "q4_last_error_string",
            "q4_set_launch_flags", "q4_get_launch_flags", "q4_workspace_bytes",
            "q4_linear_int4g128", "q4_linear_nvfp4", "audio_head_logits_restricted",
            "q4_linear_int4g128_noalloc", "q4_device_error_flags", "q4_dequant_int4g128_f32",
            "q4_dequant_nvfp4_f32", "q4_quantize_int4g128", "q4_quantize_nvfp4",
            "q4_embedding_int8", "q4_linear_int8"]


def _check(status: int) -> None:
    if status != 0:
        detail = load().q4_last_error_string().decode(errors="replace")
        raise Q4Error(status, detail)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _cuda(t, name, dtype=None):
    if not (isinstance(t, torch.Tensor) and t.is_cuda and t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def set_launch_flags(flags: int) -> None:
    _check(load().q4_set_launch_flags(flags))


def get_launch_flags() -> int:
    return int(load().q4_get_launch_flags())


def device_error_flags(clear: bool = True) -> int:
    """Device error word (bit 0: a bounded in-kernel wait timed out; bit 2: an
    embedding id out of range). Synchronises."""
    v = ctypes.c_uint(0)
    _check(load().q4_device_error_flags(ctypes.byref(v), 1 if clear else 0))
    return int(v.value)


def workspace_bytes(layout: int, M: int, N: int, K: int) -> int:
    return int(load().q4_workspace_bytes(layout, M, N, K))


def alloc_workspace(layout: int, M: int, N: int, K: int, device=None) -> torch.Tensor | None:
    """Zero-filled workspace for the given call shape (None when none is needed)."""
    n = workspace_bytes(layout, M, N, K)
    if n == 0:
        return None
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def _ws_args(ws):
    if ws is None:
        return None, 0
    return ws.data_ptr(), ws.numel() * ws.element_size()


# Workspaces the binding supplies when the caller passes none: one per (device,
# stream, layout and shape), zero-filled once.  Calls of one shape on one stream
# run in order (with programmatic dependent launch a kernel touches the
# workspace only after the previous kernel has finished) and leave its counters
# at zero, so they can share it; a different shape lays counters and partial
# sums out differently and gets its own.  Reuse also keeps allocations, and
# their fill kernels, out of captured CUDA graphs once a stream has made one
# call of each shape.
_ws_cache: dict = {}


def _default_workspace(layout: int, M: int, N: int, K: int, device, stream) -> torch.Tensor | None:
    n = workspace_bytes(layout, M, N, K)
    if n == 0:
        return None
    key = (torch.device(device).index, _stream(stream), layout, M, N, K)
    ws = _ws_cache.get(key)
    if ws is None or ws.numel() < n:     # (a launch flag can change the size)
        if len(_ws_cache) >= 64:        # many distinct shapes: start over (memory is
            _ws_cache.clear()           # returned in stream order by the allocator)
        ws = torch.zeros(n, dtype=torch.uint8, device=device)
        _ws_cache[key] = ws
    return ws


def q4_linear_int4g128(x, qweight, scale, minv, y=None, workspace=None, stream=None):
    """y[M, N] (bf16) = x[M, K] (bf16) W^T, W in the int4-g128-minmax layout."""
    _cuda(x, "x", torch.bfloat16)
    _cuda(qweight, "qweight", torch.uint8)
    _cuda(scale, "scale")
    _cuda(minv, "min")
    M, K = x.shape
    N = qweight.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    if workspace is None:
        workspace = _default_workspace(LAYOUT_INT4G128, M, N, K, x.device, stream)
    wp, wn = _ws_args(workspace)
    _check(load().q4_linear_int4g128(_ptr(x), _ptr(qweight), _ptr(scale), _ptr(minv), _ptr(y),
                                     M, N, K, wp, wn, _stream(stream)))
    return y


def q4_linear_int4g128_noalloc(x, qweight, scale, minv, y, stream=None):
    """As q4_linear_int4g128, for callers that cannot allocate device memory: the
    library's own static scratch replaces the workspace and ``y`` must be given."""
    _cuda(x, "x", torch.bfloat16)
    _cuda(qweight, "qweight", torch.uint8)
    _cuda(scale, "scale")
    _cuda(minv, "min")
    _cuda(y, "y", torch.bfloat16)
    M, K = x.shape
    N = qweight.shape[0]
    _check(load().q4_linear_int4g128_noalloc(_ptr(x), _ptr(qweight), _ptr(scale), _ptr(minv),
                                             _ptr(y), M, N, K, _stream(stream)))
    return y


def q4_linear_nvfp4(x, codes, scale_e4m3, global_scale, y=None, workspace=None, stream=None):
    """y[M, N] (bf16) = x[M, K] (bf16) W^T, W in the NVFP4 weight-only layout;
    ``global_scale`` is a one-element fp32 CUDA tensor."""
    _cuda(x, "x", torch.bfloat16)
    _cuda(codes, "codes", torch.uint8)
    _cuda(scale_e4m3, "scale_e4m3")
    _cuda(global_scale, "global_scale", torch.float32)
    M, K = x.shape
    N = codes.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    if workspace is None:
        workspace = _default_workspace(LAYOUT_NVFP4, M, N, K, x.device, stream)
    wp, wn = _ws_args(workspace)
    _check(load().q4_linear_nvfp4(_ptr(x), _ptr(codes), _ptr(scale_e4m3), _ptr(global_scale),
                                  _ptr(y), M, N, K, wp, wn, _stream(stream)))
    return y


def audio_head_logits_restricted(h, head, row_begin, n_rows, extra_row=-1, logits=None,
                                 stream=None):
    """logits[M, n_rows + (extra_row >= 0)] (bf16) of the restricted head."""
    _cuda(h, "h", torch.bfloat16)
    _cuda(head, "head", torch.bfloat16)
    M, H = h.shape
    cols = n_rows + (1 if extra_row >= 0 else 0)
    if logits is None:
        logits = torch.empty((M, max(cols, 1)), dtype=torch.bfloat16, device=h.device)
    _check(load().audio_head_logits_restricted(_ptr(h), _ptr(head), head.shape[0], row_begin,
                                               n_rows, extra_row, _ptr(logits), M, H,
                                               _stream(stream)))
    return logits


def q4_dequant_int4g128_f32(qweight, scale, minv, stream=None):
    N, K = qweight.shape[0], 2 * qweight.shape[1]
    w = torch.empty((N, K), dtype=torch.float32, device=qweight.device)
    _check(load().q4_dequant_int4g128_f32(_ptr(qweight), _ptr(scale), _ptr(minv), _ptr(w), N, K,
                                          _stream(stream)))
    return w


def q4_dequant_nvfp4_f32(codes, scale_e4m3, global_scale, stream=None):
    N, K = codes.shape[0], 2 * codes.shape[1]
    w = torch.empty((N, K), dtype=torch.float32, device=codes.device)
    _check(load().q4_dequant_nvfp4_f32(_ptr(codes), _ptr(scale_e4m3), _ptr(global_scale),
                                       _ptr(w), N, K, _stream(stream)))
    return w


# Short aliases
linear_int4g128 = q4_linear_int4g128
linear_nvfp4 = q4_linear_nvfp4
dequant_int4g128_f32 = q4_dequant_int4g128_f32
dequant_nvfp4_f32 = q4_dequant_nvfp4_f32


def q4_quantize_int4g128(w, stream=None):
    """(qweight uint8 [N, K/2], scale fp16 [N, K/128], min fp16 [N, K/128]) of the
    round-to-nearest min/max int4-g128 quantisation of bf16 weights w [N, K]."""
    _cuda(w, "w", torch.bfloat16)
    N, K = w.shape
    q = torch.empty((N, K // 2), dtype=torch.uint8, device=w.device)
    s = torch.empty((N, K // 128), dtype=torch.float16, device=w.device)
    m = torch.empty((N, K // 128), dtype=torch.float16, device=w.device)
    _check(load().q4_quantize_int4g128(_ptr(w), _ptr(q), _ptr(s), _ptr(m), N, K,
                                       _stream(stream)))
    return q, s, m


def q4_quantize_nvfp4(w, stream=None):
    """(codes uint8 [N, K/2], e4m3 scales uint8 [N, K/16], global scale fp32 [1]) of
    the round-to-nearest NVFP4 quantisation of bf16 weights w [N, K]."""
    _cuda(w, "w", torch.bfloat16)
    N, K = w.shape
    q = torch.empty((N, K // 2), dtype=torch.uint8, device=w.device)
    s = torch.empty((N, K // 16), dtype=torch.uint8, device=w.device)
    g = torch.empty((1,), dtype=torch.float32, device=w.device)
    _check(load().q4_quantize_nvfp4(_ptr(w), _ptr(q), _ptr(s), _ptr(g), N, K, _stream(stream)))
    return q, s, g


def q4_embedding_int8(ids, qweight, scale, out=None, stream=None):
    """bf16 [M, H] rows of the int8 token embedding for int32 ids [M]."""
    _cuda(ids, "ids", torch.int32)
    _cuda(qweight, "qweight", torch.int8)
    _cuda(scale, "scale", torch.float16)
    V, H = qweight.shape
    M = ids.numel()
    if out is None:
        out = torch.empty((M, H), dtype=torch.bfloat16, device=qweight.device)
    _check(load().q4_embedding_int8(_ptr(ids), _ptr(qweight), _ptr(scale), _ptr(out), M, V, H,
                                    _stream(stream)))
    return out


def q4_linear_int8(x, qweight, scale, y=None, stream=None):
    """y[M, N] (bf16) = x[M, K] (bf16) W^T, W int8 [N, K] with an fp16 scale per row."""
    _cuda(x, "x", torch.bfloat16)
    _cuda(qweight, "qweight", torch.int8)
    _cuda(scale, "scale", torch.float16)
    M, K = x.shape
    N = qweight.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _check(load().q4_linear_int8(_ptr(x), _ptr(qweight), _ptr(scale), _ptr(y), M, N, K,
                                 _stream(stream)))
    return y
