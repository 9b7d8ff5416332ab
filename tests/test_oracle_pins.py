"""Pins for the CPU oracle: each check ties the oracle to something other than
itself -- a published table, an independent library decode, an exactly
predictable special case, an exact rational result, or brute force on tiny
inputs.  No GPU needed.

A plausible mistake in the oracle (swapped nibble order, k % 128 instead of
k // 128, a dropped min term, a wrong e4m3 bias, the global scale divided instead
of multiplied, a transposed operand in the matmul) fails at least one test here.
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def _pack_codes(C):
    """Pack a [N, K] matrix of 4-bit codes as the pages state it: two codes per
    byte, the low nibble holds the even column."""
    C = np.asarray(C, dtype=np.uint8)
    return (C[:, 0::2] | (C[:, 1::2] << 4)).astype(np.uint8)


def _f16_bits(v):
    return np.asarray(v, dtype=np.float16).view(np.uint16)


def _bf16_bits(v):
    t = torch.as_tensor(np.asarray(v, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


# ------------------------------------------------------------------ scalars
def test_fp16_decode_matches_numpy_all_patterns(oracle_mod):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle_mod.fp16_value(b) for b in bits[::7]])
    r = ref[::7]
    both_nan = np.isnan(got) & np.isnan(r)
    assert np.array_equal(got[~both_nan], r[~both_nan])
    # and every special class explicitly
    for b in (0x0000, 0x8000, 0x0001, 0x03ff, 0x0400, 0x3c00, 0x7bff, 0x7c00, 0xfc00):
        assert oracle_mod.fp16_value(b) == np.uint16(b).view(np.float16).astype(np.float64)
    assert np.isnan(oracle_mod.fp16_value(0x7e00))


def test_bf16_decode_matches_torch(oracle_mod):
    bits = np.arange(0, 65536, 13, dtype=np.int64).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle_mod.bf16_value(b) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_e4m3_decode_matches_torch_all_256(oracle_mod):
    b = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(b).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle_mod.e4m3_value(v) for v in b])
    nan = np.isnan(ref)
    assert nan.sum() == 2                      # 0x7f and 0xff only (no inf in e4m3fn)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_e4m3_published_points(oracle_mod):
    for byte, val in _read_table("e4m3_points.txt"):
        got = oracle_mod.e4m3_value(int(byte, 16))
        if val == "nan":
            assert np.isnan(got)
        else:
            assert got == float(val) and np.signbit(got) == val.startswith("-")


def test_e2m1_published_table(oracle_mod):
    table = _read_table("e2m1_table.txt")
    assert len(table) == 16
    for code, val in table:
        got = oracle_mod.e2m1_value(int(code))
        assert got == float(val) and np.signbit(got) == val.startswith("-")


# ------------------------------------------------------------- int4 dequant
def test_int4_unit_scale_returns_codes(oracle_mod):
    """scale = 1, min = 0: the decoded matrix is the code matrix itself, so the
    nibble order (low nibble = even column) is pinned exactly."""
    rng = np.random.default_rng(11)
    C = rng.integers(0, 16, size=(5, 256))
    q = _pack_codes(C)
    s = _f16_bits(np.ones((5, 2)))
    m = _f16_bits(np.zeros((5, 2)))
    w = oracle_mod.dequant_int4g128(q, s, m)
    assert np.array_equal(w, C.astype(np.float32))


def test_int4_group_index_is_k_div_128(oracle_mod):
    """Distinct power-of-two scales and mins per group make every weight exact; a
    group index of k % 128 or a per-row scale would land on other values."""
    C = np.tile(np.arange(16), (3, 512 // 16))            # [3, 512], 4 groups
    sc = np.array([[2.0 ** g for g in range(4)], [2.0 ** -g for g in range(4)],
                   [1.0, 0.5, 0.25, 4.0]])
    mn = np.array([[-1.0, -2.0, -4.0, -8.0], [0.5, 0.25, 0.125, 1.0], [0, 0, 0, -3.0]])
    w = oracle_mod.dequant_int4g128(_pack_codes(C), _f16_bits(sc), _f16_bits(mn))
    for n in range(3):
        for k in (0, 1, 127, 128, 200, 255, 256, 383, 384, 511):
            g = k // 128
            assert w[n, k] == C[n, k] * sc[n, g] + mn[n, g], (n, k)


def test_int4_symmetric_special_case(oracle_mod):
    """min = -7.5 * scale with codes 7 or 8 gives w = -scale/2 or +scale/2."""
    rng = np.random.default_rng(3)
    s = (2.0 ** rng.integers(-12, -2, size=(4, 2))).astype(np.float64)
    C = rng.choice([7, 8], size=(4, 256))
    w = oracle_mod.dequant_int4g128(_pack_codes(C), _f16_bits(s), _f16_bits(-7.5 * s))
    expect = np.where(C == 8, 0.5, -0.5) * np.repeat(s, 128, axis=1)
    assert np.array_equal(w, expect.astype(np.float32))


def test_int4_zero_codes_give_min(oracle_mod):
    rng = np.random.default_rng(4)
    mn = rng.uniform(-1, 1, size=(3, 2)).astype(np.float16)
    s = rng.uniform(1e-3, 2e-2, size=(3, 2)).astype(np.float16)
    w = oracle_mod.dequant_int4g128(np.zeros((3, 128), np.uint8), s.view(np.uint16),
                                    mn.view(np.uint16))
    assert np.array_equal(w, np.repeat(mn.astype(np.float32), 128, axis=1))


def test_int4_single_rounding_exact_rational(oracle_mod):
    """Each decoded weight equals the exact rational code*scale+min rounded once
    to fp32 (round to nearest even)."""
    rng = np.random.default_rng(5)
    C = rng.integers(0, 16, size=(6, 256))
    s = rng.uniform(1e-3, 2e-2, size=(6, 2)).astype(np.float16)
    mn = (-7.5 * s.astype(np.float64) * rng.uniform(0.8, 1.2, size=s.shape)).astype(np.float16)
    w = oracle_mod.dequant_int4g128(_pack_codes(C), s.view(np.uint16), mn.view(np.uint16))
    for n in range(6):
        for k in range(0, 256, 7):
            g = k // 128
            exact = Fraction(int(C[n, k])) * Fraction(float(s[n, g])) + Fraction(float(mn[n, g]))
            # float(Fraction) is exact here (the value fits in a double); the
            # float32 cast is then the single round-to-nearest-even.
            assert Fraction(float(exact)) == exact
            assert w[n, k] == np.float32(float(exact)), (n, k)


# ------------------------------------------------------------ NVFP4 dequant
def _e2m1_from_table():
    return {int(c): float(v) for c, v in _read_table("e2m1_table.txt")}


def test_nvfp4_unit_scales_give_e2m1_table(oracle_mod):
    rng = np.random.default_rng(6)
    C = rng.integers(0, 16, size=(4, 64))
    one = np.full((4, 4), 0x38, np.uint8)                  # e4m3 1.0
    w = oracle_mod.dequant_nvfp4(_pack_codes(C), one, 1.0)
    tab = _e2m1_from_table()
    assert np.array_equal(w, np.vectorize(tab.get)(C).astype(np.float32))


def test_nvfp4_group_index_and_global_multiplies(oracle_mod):
    """Power-of-two e4m3 scales per group of 16 and a power-of-two global scale
    keep every weight exact: w = e2m1(code) * scale[k // 16] * global."""
    tab = _e2m1_from_table()
    C = np.tile(np.arange(16), (2, 4))                      # [2, 64], 4 groups
    scales = np.array([[0x30, 0x38, 0x40, 0x48], [0x28, 0x20, 0x50, 0x58]], np.uint8)
    sval = {0x20: 0.125, 0x28: 0.25, 0x30: 0.5, 0x38: 1.0, 0x40: 2.0,
            0x48: 4.0, 0x50: 8.0, 0x58: 16.0}
    w = oracle_mod.dequant_nvfp4(_pack_codes(C), scales, 0.125)
    for n in range(2):
        for k in range(64):
            assert w[n, k] == tab[int(C[n, k])] * sval[int(scales[n, k // 16])] * 0.125


def test_nvfp4_single_rounding_exact_rational(oracle_mod):
    """w = E2M1 * e4m3 * global as an exact rational, rounded once to fp32; a
    non-power-of-two global scale makes the rounding matter."""
    rng = np.random.default_rng(7)
    tab = _e2m1_from_table()
    C = rng.integers(0, 16, size=(8, 64))
    sc = torch.from_numpy(rng.uniform(0.25, 4, size=(8, 4)).astype(np.float32)) \
        .to(torch.float8_e4m3fn)
    sbits = sc.view(torch.uint8).numpy()
    sv = sc.to(torch.float64).numpy()
    G = np.float32(1e-2)
    w = oracle_mod.dequant_nvfp4(_pack_codes(C), sbits, G)
    for n in range(8):
        for k in range(64):
            exact = Fraction(tab[int(C[n, k])]) * Fraction(float(sv[n, k // 16])) * Fraction(float(G))
            assert Fraction(float(exact)) == exact
            assert w[n, k] == np.float32(float(exact)), (n, k)


# ---------------------------------------------------------------- linear
def test_linear_int4_integer_case_exact(oracle_mod):
    """Integer codes (scale 1, min 0) and small integer activations: the product
    is an integer matrix product, exact in fp64 and in numpy int64."""
    rng = np.random.default_rng(8)
    M, N, K = 3, 17, 384
    C = rng.integers(0, 16, size=(N, K))
    X = rng.integers(-8, 9, size=(M, K))
    y = oracle_mod.linear_int4g128(_bf16_bits(X), _pack_codes(C),
                                   _f16_bits(np.ones((N, 3))), _f16_bits(np.zeros((N, 3))))
    assert np.array_equal(y, (X.astype(np.int64) @ C.T.astype(np.int64)).astype(np.float64))


def test_linear_one_hot_reads_one_column(oracle_mod):
    rng = np.random.default_rng(9)
    N, K = 9, 256
    C = rng.integers(0, 16, size=(N, K))
    q = _pack_codes(C)
    s = _f16_bits(np.full((N, 2), 0.5))
    m = _f16_bits(np.full((N, 2), -1.0))
    for k in (0, 1, 2, 127, 128, 129, 254, 255):
        x = np.zeros((1, K), np.float32)
        x[0, k] = 1.0
        y = oracle_mod.linear_int4g128(_bf16_bits(x), q, s, m)
        assert np.array_equal(y[0], C[:, k] * 0.5 - 1.0)


def test_linear_matches_numpy_matmul_of_decoded(oracle_mod):
    """Brute force: the oracle's fp64 loops agree with numpy's matmul over the
    (separately pinned) decoded weights, for both layouts, and the returned
    absolute sums agree with |x| @ |w|^T."""
    from bit_weight_only_q4_gb300 import synth
    rng = synth.rng_for(99)
    w4 = synth.int4_matrix(rng, 33, 256)
    wf = synth.nvfp4_matrix(rng, 21, 96)
    x4 = synth.activations(rng, 5, 256)
    xf = synth.activations(rng, 4, 96)
    for x, W, y_a in (
            (x4, oracle_mod.dequant_int4g128(w4.qweight, w4.scale, w4.minv),
             oracle_mod.linear_int4g128(x4, w4.qweight, w4.scale, w4.minv, with_abs=True)),
            (xf, oracle_mod.dequant_nvfp4(wf.codes, wf.scale, wf.global_scale),
             oracle_mod.linear_nvfp4(xf, wf.codes, wf.scale, wf.global_scale, with_abs=True))):
        y, a = y_a
        xd = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).double().numpy()
        ref = xd @ W.astype(np.float64).T
        aref = np.abs(xd) @ np.abs(W.astype(np.float64)).T
        assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)
        assert np.allclose(a, aref, rtol=1e-12, atol=0)


def test_linear_is_affine_in_min(oracle_mod):
    """Invariant of w = c*s + min: raising every min of group g by d raises y by
    d * sum_{k in g} x_k (exact with power-of-two d and small integer x)."""
    rng = np.random.default_rng(10)
    N, K = 4, 256
    C = rng.integers(0, 16, size=(N, K))
    X = rng.integers(-4, 5, size=(1, K)).astype(np.float32)
    s = _f16_bits(np.full((N, 2), 0.25))
    m0 = np.zeros((N, 2))
    m1 = m0.copy()
    m1[:, 1] = 0.5
    y0 = oracle_mod.linear_int4g128(_bf16_bits(X), _pack_codes(C), s, _f16_bits(m0))
    y1 = oracle_mod.linear_int4g128(_bf16_bits(X), _pack_codes(C), s, _f16_bits(m1))
    assert np.array_equal(y1 - y0, np.full((1, N), 0.5 * X[0, 128:].sum()))


# ------------------------------------------------------------------ head
def test_head_selects_rows(oracle_mod):
    """One-hot activations read single head entries; the restricted logits are
    the rows [row_begin, row_begin + n_rows) followed by the extra row."""
    rng = np.random.default_rng(12)
    R, H = 40, 64
    head = rng.integers(-100, 100, size=(R, H)).astype(np.float32)
    hb = _bf16_bits(head)
    for (rb, nr, ex) in ((0, 40, -1), (8, 8, 39), (16, 8, -1), (5, 0, 3)):
        for k in (0, 31, 63):
            x = np.zeros((1, H), np.float32)
            x[0, k] = 1.0
            out = oracle_mod.head_restricted(_bf16_bits(x), hb, rb, nr, ex)
            rows = list(range(rb, rb + nr)) + ([ex] if ex >= 0 else [])
            assert out.shape == (1, len(rows))
            assert np.array_equal(out[0], head[rows, k])


def test_head_matches_numpy(oracle_mod):
    rng = np.random.default_rng(13)
    head = _bf16_bits(rng.standard_normal((50, 48)) * 0.02)
    h = _bf16_bits(rng.standard_normal((3, 48)))
    out, a = oracle_mod.head_restricted(h, head, 10, 32, 49, with_abs=True)
    hd = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).double().numpy()
    Hd = torch.from_numpy(head.view(np.int16)).view(torch.bfloat16).double().numpy()
    rows = list(range(10, 42)) + [49]
    assert np.allclose(out, hd @ Hd[rows].T, rtol=1e-12, atol=1e-14)
    assert np.allclose(a, np.abs(hd) @ np.abs(Hd[rows]).T, rtol=1e-12, atol=0)


# ----------------------------------------------------- page-printed numbers
def test_int4_layout_bytes_reproduce_checkpoint_size():
    """The int4-g128 layout (0.5 B codes + fp16 scale and min per 128 columns)
    applied to the ~3.38B-parameter model, with an int8 embedding of the 277,404
    token vocabulary (+fp16 row scales) and a bf16 [16385, 2048] audio head,
    reproduces the page's 2.13 GB file; a group of 64 or fp32 scales would not."""
    from bit_weight_only_q4_gb300.layout import int4_bytes_per_weight
    nums = {r[0]: float(r[1]) for r in _read_table("pages_numbers.txt")}
    V, H = nums["vocab_rows"], nums["hidden"]
    head_rows = nums["audio_head_rows"]
    emb = V * H
    body = nums["model_params"] - emb
    total = body * int4_bytes_per_weight() + emb * 1 + V * 2 + head_rows * H * 2
    assert abs(total / 1e9 - nums["int4_checkpoint_gb"]) < 0.01
    # fp32 scale and min, groups of 64, or no scale and min at all miss the file size
    for alt in (0.5 + 2 * 4 / 128, 0.5 + 2 * 2 / 64, 0.5):
        alt_total = body * alt + emb * 1 + V * 2 + head_rows * H * 2
        assert abs(alt_total / 1e9 - nums["int4_checkpoint_gb"]) > 0.05, alt
    assert nums["codebook_head_rows"] == 2048 + 1
    assert int4_bytes_per_weight() == 0.5 + 2 * 2 / nums["group_size_int4"]


# ------------------------------------------------------------ int8 embedding
def test_embedding_unit_scale_returns_signed_codes(oracle_mod):
    """Scale 1.0: the gathered rows are the int8 codes themselves, read as
    two's complement (bytes 0x80..0xff are -128..-1)."""
    raw = np.arange(256, dtype=np.uint8).reshape(2, 128)
    q = raw.view(np.int8)
    s = np.full(2, 0x3C00, np.uint16)                  # fp16 1.0
    out = oracle_mod.embedding_int8([1, 0, 1], q, s)
    want = np.where(raw >= 128, raw.astype(np.int64) - 256, raw).astype(np.float64)
    np.testing.assert_array_equal(out, want[[1, 0, 1]])


def test_embedding_row_selection_and_scale(oracle_mod):
    """One-hot rows: id t picks row t and multiplies by scale[t] only."""
    V, H = 5, 16
    q = np.zeros((V, H), np.int8)
    for t in range(V):
        q[t, t] = 1 + t
    s = np.array([0x3800, 0x4000, 0x4400, 0x3400, 0xC000], np.uint16)  # .5 2 4 .25 -2
    sv = np.array([0.5, 2.0, 4.0, 0.25, -2.0])
    out = oracle_mod.embedding_int8([4, 2, 0], q, s)
    for m, t in enumerate([4, 2, 0]):
        want = np.zeros(H)
        want[t] = (1 + t) * sv[t]
        np.testing.assert_array_equal(out[m], want)


def test_embedding_ids_outside_the_table_give_zeros(oracle_mod):
    q = np.ones((3, 8), np.int8)
    s = np.full(3, 0x3C00, np.uint16)
    out = oracle_mod.embedding_int8([-1, 3, 2**31 - 1, 1], q, s)
    assert np.all(out[:3] == 0) and np.all(out[3] == 1)


# --------------------------------------------------- INT8 weight-only linear
def test_int8_linear_integer_case_is_integer_matmul(oracle_mod):
    """Scale 1.0 and small-integer x: the oracle equals numpy's integer matmul of
    the signed codes (two's complement)."""
    rng = np.random.default_rng(21)
    q = rng.integers(-128, 128, (9, 64)).astype(np.int8)
    xi = rng.integers(-3, 4, (2, 64))
    xb = (xi.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)   # exact bf16
    s = np.full(9, 0x3C00, np.uint16)
    y = oracle_mod.linear_int8(xb, q, s)
    np.testing.assert_array_equal(y, xi @ q.astype(np.int64).T)


def test_int8_row_scale_applies_per_output_row(oracle_mod):
    """One-hot x picks column k; row n's output is q[n, k] * scale[n]."""
    q = np.array([[3, -7, 0, 0], [-128, 127, 1, 0]], np.int8)
    s = np.array([0x3800, 0xC200], np.uint16)           # 0.5, -3.0
    for k in range(4):
        x = np.zeros((1, 4), np.float32)
        x[0, k] = 1.0
        xb = (x.view(np.uint32) >> 16).astype(np.uint16)
        y = oracle_mod.linear_int8(xb, q, s)
        np.testing.assert_array_equal(y[0], [q[0, k] * 0.5, q[1, k] * -3.0])
    w = oracle_mod.dequant_int8(q, s)
    np.testing.assert_array_equal(w, q.astype(np.float32) * np.array([[0.5], [-3.0]], np.float32))
