"""CPU oracle for the 4-bit weight-only linear layer -- TEST INFRASTRUCTURE ONLY.

The oracle is the plain definition of what the GPU library computes, written in C
(``oracle.c``) and wrapped here with ctypes and numpy.  It decodes every weight to
fp32 from the format definition and accumulates in fp64.  Only the tests, the
package's ``smoke()`` check and the benchmark's CPU-baseline leg may import it;
the product path never does, and this package never imports the product.

Sources, cited by page title and section:
  * "rumik-oss-1-int4", "Format (rumik-int4-g128-minmax-v1)": the int4 layout and
    ``w = code * scale + min``.
  * "VoxCPM2 NVFP4 (GPTQ)", "NVFP4 settings": E2M1 codes, group 16, e4m3 group
    scales, one global scale per matrix, BF16 activations.
  * "Rumik TTS Fast Inference", "What Made It Faster" / Figure 3: the head
    restricted to the current codebook's 2,049 rows.

The quantisers (round-to-nearest, min/max for int4, amax-based for NVFP4) and the
fp16 / e4m3 / E2M1 encoders they use are written out from the formats'
definitions in ``oracle.c``.

Parity is pinned for every function here by the ``-m "not gpu"`` tests in
``tests/test_oracle_pins.py`` (tables, special cases, brute force, invariants).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle_q4.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` with gcc (OpenMP, no FP contraction) and return the .so path."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    os.makedirs(_OUT_DIR, exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-fopenmp", "-ffp-contract=off", "-fPIC",
           "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    p, i64, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float
    lib.q4o_fp16_value.argtypes = [ctypes.c_uint16]
    lib.q4o_fp16_value.restype = ctypes.c_double
    lib.q4o_bf16_value.argtypes = [ctypes.c_uint16]
    lib.q4o_bf16_value.restype = ctypes.c_double
    lib.q4o_e4m3_value.argtypes = [ctypes.c_uint8]
    lib.q4o_e4m3_value.restype = ctypes.c_double
    lib.q4o_e2m1_value.argtypes = [ctypes.c_uint8]
    lib.q4o_e2m1_value.restype = ctypes.c_double
    lib.q4o_dequant_int4g128.argtypes = [p, p, p, i64, i64, p]
    lib.q4o_dequant_nvfp4.argtypes = [p, p, f32, i64, i64, p]
    lib.q4o_linear_int4g128.argtypes = [p, p, p, p, i64, i64, i64, p, p]
    lib.q4o_linear_nvfp4.argtypes = [p, p, p, f32, i64, i64, i64, p, p]
    lib.q4o_head_restricted.argtypes = [p, p, i64, i64, i64, i64, i64, p, p]
    lib.q4o_num_threads.restype = ctypes.c_int
    for name in ("q4o_f32_to_fp16_array", "q4o_f32_to_e4m3_array", "q4o_f32_to_e2m1_array"):
        getattr(lib, name).argtypes = [p, p, i64]
    lib.q4o_quantize_int4g128.argtypes = [p, i64, i64, p, p, p]
    lib.q4o_quantize_nvfp4.argtypes = [p, i64, i64, p, p, p]
    lib.q4o_embedding_int8.argtypes = [p, p, p, i64, i64, i64, p]
    lib.q4o_dequant_int8.argtypes = [p, p, i64, i64, p]
    lib.q4o_linear_int8.argtypes = [p, p, p, i64, i64, i64, p, p]
    for name in ("q4o_dequant_int4g128", "q4o_dequant_nvfp4", "q4o_linear_int4g128",
                 "q4o_linear_nvfp4", "q4o_head_restricted", "q4o_f32_to_fp16_array",
                 "q4o_f32_to_e4m3_array", "q4o_f32_to_e2m1_array", "q4o_quantize_int4g128",
                 "q4o_quantize_nvfp4", "q4o_embedding_int8", "q4o_dequant_int8",
                 "q4o_linear_int8"):
        getattr(lib, name).restype = None
    _lib = lib
    return lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    return a


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


# ------------------------------------------------------------------ scalars
def fp16_value(bits: int) -> float:
    return _load().q4o_fp16_value(int(bits))


def bf16_value(bits: int) -> float:
    return _load().q4o_bf16_value(int(bits))


def e4m3_value(byte: int) -> float:
    return _load().q4o_e4m3_value(int(byte))


def e2m1_value(nibble: int) -> float:
    return _load().q4o_e2m1_value(int(nibble))


def num_threads() -> int:
    return int(_load().q4o_num_threads())


# ---------------------------------------------------------------- dequantise
def dequant_int4g128(qweight, scale_f16_bits, min_f16_bits) -> np.ndarray:
    """fp32 [N, K] weights of the int4-g128-minmax layout (one rounding each)."""
    q = _c(qweight, np.uint8)
    s = _c(scale_f16_bits, np.uint16)
    m = _c(min_f16_bits, np.uint16)
    N, K = q.shape[0], 2 * q.shape[1]
    if K % 128 or s.shape != (N, K // 128) or m.shape != (N, K // 128):
        raise ValueError("int4g128 shapes: qweight [N,K/2], scale/min [N,K/128]")
    w = np.empty((N, K), np.float32)
    _load().q4o_dequant_int4g128(_ptr(q), _ptr(s), _ptr(m), N, K, _ptr(w))
    return w


def dequant_nvfp4(codes, scale_e4m3, global_scale: float) -> np.ndarray:
    """fp32 [N, K] weights of the NVFP4 weight-only layout (one rounding each)."""
    q = _c(codes, np.uint8)
    s = _c(scale_e4m3, np.uint8)
    N, K = q.shape[0], 2 * q.shape[1]
    if K % 16 or s.shape != (N, K // 16):
        raise ValueError("nvfp4 shapes: codes [N,K/2], scale [N,K/16]")
    w = np.empty((N, K), np.float32)
    _load().q4o_dequant_nvfp4(_ptr(q), _ptr(s), float(np.float32(global_scale)), N, K,
                              _ptr(w))
    return w


# -------------------------------------------------------------------- linear
def linear_int4g128(x_bf16_bits, qweight, scale_f16_bits, min_f16_bits,
                    with_abs: bool = False):
    """fp64 y [M, N] = x [M, K] (bf16 bits) times the decoded weights, transposed.

    With ``with_abs`` also returns sum_k |x[m,k] w[n,k]| per output element.
    """
    x = _c(np.atleast_2d(x_bf16_bits), np.uint16)
    q = _c(qweight, np.uint8)
    s = _c(scale_f16_bits, np.uint16)
    m = _c(min_f16_bits, np.uint16)
    M, K = x.shape
    N = q.shape[0]
    if q.shape[1] * 2 != K or K % 128 or s.shape != (N, K // 128) or m.shape != s.shape:
        raise ValueError("int4g128 linear: shape mismatch")
    y = np.empty((M, N), np.float64)
    a = np.empty((M, N), np.float64) if with_abs else None
    _load().q4o_linear_int4g128(_ptr(x), _ptr(q), _ptr(s), _ptr(m), M, N, K, _ptr(y),
                                _ptr(a) if with_abs else None)
    return (y, a) if with_abs else y


def linear_nvfp4(x_bf16_bits, codes, scale_e4m3, global_scale: float,
                 with_abs: bool = False):
    """fp64 y [M, N] for the NVFP4 weight-only layout (see ``linear_int4g128``)."""
    x = _c(np.atleast_2d(x_bf16_bits), np.uint16)
    q = _c(codes, np.uint8)
    s = _c(scale_e4m3, np.uint8)
    M, K = x.shape
    N = q.shape[0]
    if q.shape[1] * 2 != K or K % 16 or s.shape != (N, K // 16):
        raise ValueError("nvfp4 linear: shape mismatch")
    y = np.empty((M, N), np.float64)
    a = np.empty((M, N), np.float64) if with_abs else None
    _load().q4o_linear_nvfp4(_ptr(x), _ptr(q), _ptr(s), float(np.float32(global_scale)),
                             M, N, K, _ptr(y), _ptr(a) if with_abs else None)
    return (y, a) if with_abs else y


def head_restricted(h_bf16_bits, head_bf16_bits, row_begin: int, n_rows: int,
                    extra_row: int, with_abs: bool = False):
    """fp64 logits [M, n_rows + (extra_row >= 0)] of the restricted output head."""
    h = _c(np.atleast_2d(h_bf16_bits), np.uint16)
    H_ = _c(head_bf16_bits, np.uint16)
    M, Hd = h.shape
    R_total = H_.shape[0]
    if H_.shape[1] != Hd:
        raise ValueError("head: hidden size mismatch")
    if row_begin < 0 or n_rows < 0 or row_begin + n_rows > R_total or extra_row >= R_total:
        raise ValueError("head: row range outside the head")
    cols = n_rows + (1 if extra_row >= 0 else 0)
    out = np.empty((M, cols), np.float64)
    a = np.empty((M, cols), np.float64) if with_abs else None
    _load().q4o_head_restricted(_ptr(h), _ptr(H_), row_begin, n_rows, extra_row, M, Hd,
                                _ptr(out), _ptr(a) if with_abs else None)
    return (out, a) if with_abs else out


# ------------------------------------------------------------------ encoders
def _encode(fn: str, x, out_dtype) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    out = np.empty(a.shape, out_dtype)
    getattr(_load(), fn)(_ptr(a), _ptr(out), a.size)
    return out


def f32_to_fp16_bits(x) -> np.ndarray:
    """IEEE binary16 bits, round to nearest even, overflow to infinity."""
    return _encode("q4o_f32_to_fp16_array", x, np.uint16)


def f32_to_e4m3_bits(x) -> np.ndarray:
    """float8_e4m3fn bits, round to nearest even, saturating at +-448."""
    return _encode("q4o_f32_to_e4m3_array", x, np.uint8)


def f32_to_e2m1_codes(x) -> np.ndarray:
    """E2M1 nibbles (bit 3 sign), nearest with ties to even, saturating at +-6,
    magnitude 0 stored as +0."""
    return _encode("q4o_f32_to_e2m1_array", x, np.uint8)


# ------------------------------------------------------------------ quantise
def quantize_int4g128(w_bf16_bits):
    """(qweight [N,K/2] u8, scale fp16 bits [N,K/128], min fp16 bits [N,K/128])."""
    w = _c(w_bf16_bits, np.uint16)
    N, K = w.shape
    if K % 128:
        raise ValueError("int4g128 quantiser: K % 128 != 0")
    q = np.zeros((N, K // 2), np.uint8)
    s = np.empty((N, K // 128), np.uint16)
    m = np.empty((N, K // 128), np.uint16)
    _load().q4o_quantize_int4g128(_ptr(w), N, K, _ptr(q), _ptr(s), _ptr(m))
    return q, s, m


def quantize_nvfp4(w_bf16_bits):
    """(codes [N,K/2] u8, e4m3 scales [N,K/16] u8, fp32 global scale)."""
    w = _c(w_bf16_bits, np.uint16)
    N, K = w.shape
    if K % 16:
        raise ValueError("nvfp4 quantiser: K % 16 != 0")
    q = np.zeros((N, K // 2), np.uint8)
    s = np.empty((N, K // 16), np.uint8)
    g = np.zeros(1, np.float32)
    _load().q4o_quantize_nvfp4(_ptr(w), N, K, _ptr(q), _ptr(s), _ptr(g))
    return q, s, np.float32(g[0])


# ------------------------------------------------------------------ embedding
def embedding_int8(ids, qweight, scale_f16_bits) -> np.ndarray:
    """fp64 [M, H]: rows ids of the int8 embedding times their fp16 row scale
    (zeros for an id outside 0 .. V-1)."""
    i = _c(np.asarray(ids, dtype=np.int32).reshape(-1), np.int32)
    q = _c(qweight, np.int8)
    s = _c(scale_f16_bits, np.uint16)
    V, H = q.shape
    if s.shape != (V,):
        raise ValueError("embedding: scale must be [V]")
    out = np.empty((i.size, H), np.float64)
    _load().q4o_embedding_int8(_ptr(i), _ptr(q), _ptr(s), i.size, V, H, _ptr(out))
    return out


# ------------------------------------------------------- INT8 weight-only
def dequant_int8(qweight, scale_f16_bits) -> np.ndarray:
    """fp32 [N, K] weights q * scale of the INT8 weight-only layout (exact)."""
    q = _c(qweight, np.int8)
    s = _c(scale_f16_bits, np.uint16)
    N, K = q.shape
    if s.shape != (N,):
        raise ValueError("int8 shapes: qweight [N,K], scale [N]")
    w = np.empty((N, K), np.float32)
    _load().q4o_dequant_int8(_ptr(q), _ptr(s), N, K, _ptr(w))
    return w


def linear_int8(x_bf16_bits, qweight, scale_f16_bits, with_abs: bool = False):
    """fp64 y [M, N] for the INT8 weight-only layout (see ``linear_int4g128``)."""
    x = _c(np.atleast_2d(x_bf16_bits), np.uint16)
    q = _c(qweight, np.int8)
    s = _c(scale_f16_bits, np.uint16)
    M, K = x.shape
    N = q.shape[0]
    if q.shape[1] != K or s.shape != (N,):
        raise ValueError("int8 linear: shape mismatch")
    y = np.empty((M, N), np.float64)
    a = np.empty((M, N), np.float64) if with_abs else None
    _load().q4o_linear_int8(_ptr(x), _ptr(q), _ptr(s), M, N, K, _ptr(y),
                            _ptr(a) if with_abs else None)
    return (y, a) if with_abs else y
