"""INT8 weight-only linear (int8 [N, K] codes, one fp16 scale per row) on the
whole-row CUDA-core kernel, against the fp64 oracle with the usual tolerances."""
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


def _dev(w):
    return (torch.from_numpy(w.qweight).cuda(),
            torch.from_numpy(w.scale.view(np.int16)).view(torch.float16).cuda())


@pytest.mark.parametrize("N,K,M", [(2048, 2048, 1), (16384, 2048, 1), (2048, 8192, 1),
                                   (2048, 8192, 3), (300, 528, 2), (8192, 2048, 4),
                                   (129, 16, 5), (1, 4096, 1)])
def test_int8_linear_matches_oracle(q4, oracle_mod, N, K, M):
    rng = synth.rng_for(60, N, K, M)
    w = synth.int8_matrix(rng, N, K)
    x = synth.activations(rng, M, K)
    y = q4.q4_linear_int8(P.bf16_dev(x), *_dev(w))
    yo, ao = oracle_mod.linear_int8(x, w.qweight, w.scale, with_abs=True)
    P.check(y, yo, ao, f"int8 N={N} K={K} M={M}")


def test_int8_linear_with_pdl_is_identical(q4):
    rng = synth.rng_for(61)
    w = synth.int8_matrix(rng, 4096, 2048)
    xd = P.bf16_dev(synth.activations(rng, 1, 2048))
    wd = _dev(w)
    a = q4.q4_linear_int8(xd, *wd)
    q4.set_launch_flags(q4.FLAG_PDL)
    try:
        b = q4.q4_linear_int8(xd, *wd)
    finally:
        q4.set_launch_flags(0)
    assert torch.equal(a, b)


def test_int8_linear_shape_errors(q4):
    x = torch.zeros((1, 24), dtype=torch.bfloat16, device="cuda")
    q = torch.zeros((4, 24), dtype=torch.int8, device="cuda")
    s = torch.zeros((4,), dtype=torch.float16, device="cuda")
    with pytest.raises(q4.Q4Error):
        q4.q4_linear_int8(x, q, s)                       # K % 16 != 0
    x = torch.zeros((1, 8704), dtype=torch.bfloat16, device="cuda")
    q = torch.zeros((4, 8704), dtype=torch.int8, device="cuda")
    with pytest.raises(q4.Q4Error):
        q4.q4_linear_int8(x, q, s)                       # K > 8192
