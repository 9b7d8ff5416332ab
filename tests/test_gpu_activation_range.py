"""Activations the staging of x has to survive, on the one-token and few-token
whole-row kernels.

x is staged per 32-column chunk with a power-of-two prescale: int4 as int16 fixed
point (exact for values within 2^7 of the chunk maximum, smaller ones rounded to
the nearest 2^-15 of it), NVFP4 as fp16.  A chunk whose values span many octaves
must stay within the per-element bound of the fp64 oracle; a non-finite value must
make its own token's outputs non-finite and leave the other tokens untouched."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from bit_weight_only_q4_gb300 import synth
from tests import parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q4():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_weight_only_q4_gb300 import build, q4 as lib
    build.build()
    lib.load()
    lib.set_launch_flags(0)
    return lib


def _x_wide(rng: np.random.Generator, M: int, K: int) -> np.ndarray:
    """bf16 bits with random sign, mantissa and an exponent uniform over
    2^-30 .. 2^2, so every chunk spans about 32 octaves."""
    sign = rng.integers(0, 2, (M, K), dtype=np.uint16)
    exp = rng.integers(127 - 30, 127 + 3, (M, K)).astype(np.uint16)
    mant = rng.integers(0, 128, (M, K), dtype=np.uint16)
    return (sign << 15) | (exp << 7) | mant


@pytest.mark.parametrize("M", [1, 3, 4])
def test_int4_wide_range_chunks(q4, oracle_mod, M):
    rng = synth.rng_for(91, M)
    N, K = 640, 2048
    w = synth.int4_matrix(rng, N, K)
    x = _x_wide(rng, M, K)
    y = q4.q4_linear_int4g128(P.bf16_dev(x), *P.int4_dev(w))
    yo, ao = oracle_mod.linear_int4g128(x, w.qweight, w.scale, w.minv, with_abs=True)
    P.check(y, yo, ao, f"int4 wide-range x M={M}")


@pytest.mark.parametrize("M", [1, 3, 4])
def test_nvfp4_wide_range_chunks(q4, oracle_mod, M):
    rng = synth.rng_for(92, M)
    N, K = 640, 2048
    w = synth.nvfp4_matrix(rng, N, K)
    x = _x_wide(rng, M, K)
    y = q4.q4_linear_nvfp4(P.bf16_dev(x), *P.nvfp4_dev(w))
    yo, ao = oracle_mod.linear_nvfp4(x, w.codes, w.scale, w.global_scale, with_abs=True)
    P.check(y, yo, ao, f"nvfp4 wide-range x M={M}")


@pytest.mark.parametrize("layout", ["int4", "nvfp4"])
@pytest.mark.parametrize("bad", [0x7F80, 0xFF80, 0x7FC0])      # +inf, -inf, NaN
@pytest.mark.parametrize("M", [1, 2])
def test_nonfinite_x_poisons_only_its_token(q4, oracle_mod, layout, bad, M):
    rng = synth.rng_for(93, M, bad)
    N, K = 512, 2048
    x = synth.activations(rng, M, K)
    x[0, 777] = bad
    if layout == "int4":
        w = synth.int4_matrix(rng, N, K)
        y = q4.q4_linear_int4g128(P.bf16_dev(x), *P.int4_dev(w))
    else:
        w = synth.nvfp4_matrix(rng, N, K)
        y = q4.q4_linear_nvfp4(P.bf16_dev(x), *P.nvfp4_dev(w))
    yh = y.float().cpu()
    assert not torch.isfinite(yh[0]).any(), "every output of the token holding the value"
    if M > 1:
        if layout == "int4":
            yo, ao = oracle_mod.linear_int4g128(x[1:], w.qweight, w.scale, w.minv, with_abs=True)
        else:
            yo, ao = oracle_mod.linear_nvfp4(x[1:], w.codes, w.scale, w.global_scale, with_abs=True)
        P.check(y[1:], yo, ao, f"{layout} token beside a non-finite one")


def _x_extreme(rng: np.random.Generator, M: int, K: int) -> np.ndarray:
    """N(0,1) bf16 activations with one 32-column chunk of every token moved up by
    2^120 and another moved down by 2^-120 (exact: only the exponent field
    changes), so the prescale of x must reach both ends of the bf16 range."""
    x = synth.activations(rng, M, K)
    e = (x >> 7) & 0xFF
    up = slice(160, 192)
    down = slice(640, 672)
    eu = e[:, up].astype(np.int32)
    x[:, up] = np.where(eu > 0, (x[:, up] & 0x807F) | ((eu + 120).astype(np.uint16) << 7), x[:, up])
    ed = e[:, down].astype(np.int32)
    x[:, down] = np.where(ed > 121, (x[:, down] & 0x807F) | ((ed - 120).astype(np.uint16) << 7),
                          x[:, down])
    return x


@pytest.mark.parametrize("layout", ["int4", "nvfp4"])
@pytest.mark.parametrize("M", [1, 3, 4])
def test_chunks_near_both_ends_of_the_bf16_range(q4, oracle_mod, layout, M):
    """A chunk whose largest |x| is about 2^121 (beyond the reach of a +-100
    prescale) and one about 2^-118: outputs finite and within the oracle's bound."""
    rng = synth.rng_for(94, M)
    N, K = 640, 2048
    x = _x_extreme(rng, M, K)
    assert np.abs(x.view(np.int16).astype(np.int32) & 0x7F80).max() >= (247 << 7)
    if layout == "int4":
        w = synth.int4_matrix(rng, N, K)
        y = q4.q4_linear_int4g128(P.bf16_dev(x), *P.int4_dev(w))
        yo, ao = oracle_mod.linear_int4g128(x, w.qweight, w.scale, w.minv, with_abs=True)
    else:
        w = synth.nvfp4_matrix(rng, N, K)
        y = q4.q4_linear_nvfp4(P.bf16_dev(x), *P.nvfp4_dev(w))
        yo, ao = oracle_mod.linear_nvfp4(x, w.codes, w.scale, w.global_scale, with_abs=True)
    P.check(y, yo, ao, f"{layout} chunks near 2^+-120, M={M}")
