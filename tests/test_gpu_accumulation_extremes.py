"""Worst cases of the partial sums in the whole-row GEMV.

Every x value of a 32-column chunk sits at the top of the prescale range
(|x| = 1.9921875, the largest bf16 below 2) and every code is at the extreme of
one sign.  NVFP4 sums each eight-product half-group in fp16, which then reaches
8 * 6 * 1020 = 48,960, below the fp16 maximum of 65,504; int4 sums c * x' in
int32 with x' in int16, which then reaches 32 * 15 * 32,640 per lane, below 2^24
(exact in fp32).  Outputs must be finite and within the stated tolerance of the
fp64 oracle, for one and four tokens and for K = 2048 and 8192."""
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


def _x_extreme(M: int, K: int) -> np.ndarray:
    """bf16 bits: +-1.9921875 (0x3FFF / 0xBFFF), the sign alternating per 32-column
    chunk and per token."""
    x = np.full((M, K), 0x3FFF, np.uint16)
    chunk = (np.arange(K) // 32)[None, :] + np.arange(M)[:, None]
    x[(chunk % 2) == 1] = 0xBFFF
    return x


@pytest.mark.parametrize("M,K", [(1, 2048), (4, 2048), (1, 8192)])
def test_nvfp4_half_group_sums_at_their_largest(q4, oracle_mod, M, K):
    N = 384
    codes = np.empty((N, K // 2), np.uint8)
    codes[0::3] = 0x77                       # every code +6
    codes[1::3] = 0xFF                       # every code -6
    codes[2::3] = 0x7F                       # -6, +6 alternating
    scale = np.full((N, K // 16), 0x7E, np.uint8)   # e4m3 448, the largest
    scale[1::2] = 0x38                              # e4m3 1.0
    w = synth.Nvfp4Matrix(codes, scale, np.float32(1e-2))
    x = _x_extreme(M, K)
    y = q4.q4_linear_nvfp4(P.bf16_dev(x), *P.nvfp4_dev(w))
    yo, ao = oracle_mod.linear_nvfp4(x, w.codes, w.scale, w.global_scale, with_abs=True)
    P.check(y, yo, ao, f"nvfp4 extremes M={M} K={K}")


@pytest.mark.parametrize("M,K", [(1, 2048), (4, 2048), (1, 8192)])
def test_int4_half_group_sums_at_their_largest(q4, oracle_mod, M, K):
    N = 384
    q = np.empty((N, K // 2), np.uint8)
    q[0::3] = 0xFF                           # every code 15 (c - 8 = 7)
    q[1::3] = 0x00                           # every code 0 (c - 8 = -8)
    q[2::3] = 0x0F                           # 15, 0 alternating
    s = np.full((N, K // 128), 0.02, np.float16)
    mn = np.full((N, K // 128), -0.15, np.float16)
    w = synth.Int4Matrix(q, s.view(np.uint16).copy(), mn.view(np.uint16).copy())
    x = _x_extreme(M, K)
    y = q4.q4_linear_int4g128(P.bf16_dev(x), *P.int4_dev(w))
    yo, ao = oracle_mod.linear_int4g128(x, w.qweight, w.scale, w.minv, with_abs=True)
    P.check(y, yo, ao, f"int4 extremes M={M} K={K}")
