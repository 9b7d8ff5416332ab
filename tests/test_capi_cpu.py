"""Host-side checks of the C ABI that need no GPU: the shared library builds and
loads, exports every entry point include/q4.h declares, and rejects invalid
arguments before launching anything (fake pointers are never dereferenced)."""
import ctypes
import os
import re

import pytest

from bit_weight_only_q4_gb300 import build as q4build
from bit_weight_only_q4_gb300 import layout, q4

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "q4.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", src, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    q4build.build()
    return q4.load()


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for n in ("q4_linear_int4g128", "q4_linear_nvfp4", "audio_head_logits_restricted",
              "q4_workspace_bytes", "q4_dequant_int4g128_f32", "q4_dequant_nvfp4_f32"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(q4.lib_path())
    for name in _declared_functions():
        assert hasattr(raw, name), name
    assert set(q4.symbols()) <= set(_declared_functions())


def test_abi_version_and_status_strings(lib):
    assert lib.q4_abi_version() == 1
    assert lib.q4_status_string(0) == b"ok"
    assert lib.q4_status_string(4) == b"workspace too small"
    assert lib.q4_status_string(99) == b"unknown status"


def test_launch_flags_roundtrip(lib):
    assert q4.get_launch_flags() == 0
    q4.set_launch_flags(q4.FLAG_PDL)
    assert q4.get_launch_flags() == q4.FLAG_PDL
    with pytest.raises(q4.Q4Error):
        q4.set_launch_flags(0x80)
    with pytest.raises(q4.Q4Error):
        q4.set_launch_flags(q4.FLAG_FORCE_CUDA_CORE | q4.FLAG_FORCE_TENSOR_CORE)
    q4.set_launch_flags(0)


def test_workspace_bytes(lib):
    # one 128-column k-range: no CUDA-core kernel splits K, no workspace
    assert q4.workspace_bytes(0, 1, 2048, 128) == 0
    # above 64 tokens the tensor-core path converts x once per call to a
    # prescaled fp16 copy (M x K x 2 bytes) with one scale per token (M x 4),
    # each rounded up to 256 bytes; up to 64 tokens it converts x in the GEMM
    assert q4.workspace_bytes(0, 100, 2048, 128) == 100 * 128 * 2 + 512
    assert q4.workspace_bytes(0, 48, 2048, 128) == 0
    # NVFP4 tensor-core calls take x as stored (bf16 operands): no copy of x
    assert q4.workspace_bytes(1, 100, 2048, 128) == 0
    assert q4.workspace_bytes(1, 2048, 8192, 2048) < 2048 * 2048 * 2 <= \
        q4.workspace_bytes(0, 2048, 8192, 2048)
    # split-K needs counters and partial slots (the bound covers every kernel a
    # call may pick, including the tensor-core path forced by a flag)
    a = q4.workspace_bytes(0, 1, 2048, 2048)
    b = q4.workspace_bytes(0, 1, 2048, 8192)
    assert a > 0 and b > 0
    assert a % 256 == 0 and b % 256 == 0
    assert q4.workspace_bytes(1, 1, 16384, 2048) > 0
    # invalid shapes report 0
    assert q4.workspace_bytes(0, 1, 2048, 100) == 0
    assert q4.workspace_bytes(1, 1, 2048, 24) == 0
    assert q4.workspace_bytes(0, 0, 2048, 2048) == 0
    assert q4.workspace_bytes(7, 1, 2048, 2048) == 0


FAKE = 1 << 20          # a 16-byte aligned address that is never dereferenced


def _int4(lib, x=FAKE, w=FAKE, s=FAKE, m=FAKE, y=FAKE, M=1, N=64, K=128, ws=None, wsb=0):
    return lib.q4_linear_int4g128(x, w, s, m, y, M, N, K, ws, wsb, None)


def _nv(lib, x=FAKE, w=FAKE, s=FAKE, g=FAKE, y=FAKE, M=1, N=64, K=128, ws=None, wsb=0):
    return lib.q4_linear_nvfp4(x, w, s, g, y, M, N, K, ws, wsb, None)


def test_invalid_arguments_are_rejected_before_launch(lib):
    assert _int4(lib, x=None) == 1
    assert _int4(lib, s=None) == 1
    assert _int4(lib, K=1000) == 2
    assert _int4(lib, K=0) == 2
    assert _int4(lib, M=0) == 2
    assert _int4(lib, N=0) == 2
    assert _int4(lib, x=FAKE + 8) == 3
    assert _int4(lib, s=FAKE + 1) == 3
    # K = 2048 needs a workspace
    assert _int4(lib, K=2048) == 4
    need = q4.workspace_bytes(0, 1, 64, 2048)
    assert _int4(lib, K=2048, ws=FAKE, wsb=need - 1) == 4
    assert _int4(lib, K=2048, ws=FAKE + 4, wsb=need) == 3
    assert _nv(lib, K=24) == 2
    assert _nv(lib, g=None) == 1
    assert _nv(lib, g=FAKE + 2) == 3
    assert _nv(lib, y=FAKE + 2) == 3
    assert b"K %" in lib.q4_last_error_string() or lib.q4_last_error_string() != b""


def test_head_arguments_are_rejected_before_launch(lib):
    f = lib.audio_head_logits_restricted
    # (h, head, R_total, row_begin, n_rows, extra_row, logits, M, H, stream)
    assert f(FAKE, FAKE, 100, 0, 101, -1, FAKE, 1, 64, None) == 5
    assert f(FAKE, FAKE, 100, -1, 10, -1, FAKE, 1, 64, None) == 5
    assert f(FAKE, FAKE, 100, 0, 10, 100, FAKE, 1, 64, None) == 5
    assert f(FAKE, FAKE, 100, 0, 10, -2, FAKE, 1, 64, None) == 5
    assert f(FAKE, FAKE, 100, 0, 0, -1, FAKE, 1, 64, None) == 2
    assert f(FAKE, FAKE, 100, 0, 10, -1, FAKE, 1, 60, None) == 2
    assert f(None, FAKE, 100, 0, 10, -1, FAKE, 1, 64, None) == 1
    assert f(FAKE + 8, FAKE, 100, 0, 10, -1, FAKE, 1, 64, None) == 3


def test_dequant_arguments_are_rejected_before_launch(lib):
    assert lib.q4_dequant_int4g128_f32(FAKE, FAKE, FAKE, FAKE, 4, 100, None) == 2
    assert lib.q4_dequant_nvfp4_f32(FAKE, FAKE, None, FAKE, 4, 32, None) == 1
    assert lib.q4_dequant_nvfp4_f32(FAKE, FAKE, FAKE, FAKE + 4, 4, 32, None) == 3



def test_int8_embedding_quantiser_and_noalloc_arguments_are_rejected_before_launch(lib):
    """Every other entry point validates pointers, shapes and alignment on the
    host and launches nothing on failure (status 1 NULL, 2 shape, 3 alignment)."""
    # q4_linear_int8(x, qweight, scale, y, M, N, K, stream): K % 16, K >= 16
    i8 = lambda x=FAKE, w=FAKE, s=FAKE, y=FAKE, M=1, N=64, K=128: \
        lib.q4_linear_int8(x, w, s, y, M, N, K, None)
    assert i8(s=None) == 1 and i8(x=None) == 1 and i8(y=None) == 1
    assert i8(K=24) == 2 and i8(K=8) == 2 and i8(M=0) == 2 and i8(N=0) == 2
    assert i8(x=FAKE + 8) == 3 and i8(w=FAKE + 4) == 3 and i8(s=FAKE + 1) == 3
    assert i8(K=16384) == 2                               # beyond the whole-row kernel
    # q4_embedding_int8(ids, qweight, scale, out, M, V, H, stream): H % 16
    emb = lambda ids=FAKE, w=FAKE, s=FAKE, o=FAKE, M=1, V=100, H=2048: \
        lib.q4_embedding_int8(ids, w, s, o, M, V, H, None)
    assert emb(ids=None) == 1 and emb(o=None) == 1
    assert emb(M=0) == 2 and emb(V=0) == 2 and emb(H=24) == 2
    assert emb(ids=FAKE + 2) == 3 and emb(w=FAKE + 8) == 3 and emb(o=FAKE + 8) == 3
    # quantisers: int4 needs K % 128, NVFP4 K % 16
    qi = lambda w=FAKE, q=FAKE, s=FAKE, m=FAKE, N=4, K=256: \
        lib.q4_quantize_int4g128(w, q, s, m, N, K, None)
    assert qi(m=None) == 1 and qi(K=200) == 2 and qi(N=0) == 2 and qi(w=FAKE + 4) == 3
    qn = lambda w=FAKE, c=FAKE, s=FAKE, g=FAKE, N=4, K=256: \
        lib.q4_quantize_nvfp4(w, c, s, g, N, K, None)
    assert qn(g=None) == 1 and qn(K=24) == 2 and qn(w=FAKE + 8) == 3 and qn(g=FAKE + 2) == 3
    # the allocation-free int4 entry: same checks as the workspace form
    na = lambda x=FAKE, w=FAKE, s=FAKE, m=FAKE, y=FAKE, M=1, N=64, K=2048: \
        lib.q4_linear_int4g128_noalloc(x, w, s, m, y, M, N, K, None)
    assert na(y=None) == 1 and na(K=100) == 2 and na(M=0) == 2 and na(x=FAKE + 8) == 3
    assert lib.q4_last_error_string() != b""

def test_layout_byte_accounting():
    assert layout.int4_bytes_per_weight() == 0.53125
    assert layout.nvfp4_bytes_per_weight() == 0.5625
    assert layout.weight_bytes("int4", 2048, 2048) == 2048 * 1024 + 4 * 2048 * 16
    assert layout.linear_bytes("int4", 1, 2048, 2048) == 2236416
    assert layout.linear_bytes("nvfp4", 1, 16384, 2048) == 18911236

