"""GPU round-to-nearest quantisers against the oracle: codes, scales, mins and the
global scale are integer / bit-pattern outputs decided in fp32 on both sides, so
they must match bit for bit.  Then the packed result is run through the linear
layer and checked against the oracle's linear on the same packed weights."""
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


def _weights(kind: str, N: int, K: int, seed: int) -> np.ndarray:
    rng = synth.rng_for(40, seed, N, K)
    if kind == "normal":
        w = rng.standard_normal((N, K)) * 0.02
    elif kind == "unit":
        w = rng.standard_normal((N, K))
    elif kind == "outliers":
        w = rng.standard_normal((N, K)) * 0.02
        w[rng.random((N, K)) < 0.002] *= 300.0
    elif kind == "edges":
        w = rng.standard_normal((N, K)) * 0.02
        w[0, :] = 0.0                                   # all-zero row
        w[1 % N, :128] = 0.25                           # constant group
        w[2 % N, :] *= 1e-6                             # tiny values: subnormal fp16 scales
        w[3 % N, 16:32] = -3.0                          # a negative constant group
    else:
        raise ValueError(kind)
    return synth._to_bf16_bits(w.astype(np.float32))


def _dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return P.bf16_dev(bits)


@pytest.mark.parametrize("kind", ["normal", "unit", "outliers", "edges"])
@pytest.mark.parametrize("N,K", [(300, 2048), (7, 128), (129, 384)])
def test_int4_quantiser_bit_exact(q4, oracle_mod, kind, N, K):
    wb = _weights(kind, N, K, 1)
    q, s, m = q4.q4_quantize_int4g128(_dev_bf16(wb))
    qo, so, mo = oracle_mod.quantize_int4g128(wb)
    np.testing.assert_array_equal(q.cpu().numpy(), qo)
    np.testing.assert_array_equal(s.cpu().view(torch.int16).numpy().view(np.uint16), so)
    np.testing.assert_array_equal(m.cpu().view(torch.int16).numpy().view(np.uint16), mo)


@pytest.mark.parametrize("kind", ["normal", "unit", "outliers", "edges"])
@pytest.mark.parametrize("N,K", [(300, 2048), (7, 16), (129, 400)])
def test_nvfp4_quantiser_bit_exact(q4, oracle_mod, kind, N, K):
    wb = _weights(kind, N, K, 2)
    q, s, g = q4.q4_quantize_nvfp4(_dev_bf16(wb))
    qo, so, go = oracle_mod.quantize_nvfp4(wb)
    assert g.cpu().numpy()[0] == go
    np.testing.assert_array_equal(s.cpu().numpy(), so)
    np.testing.assert_array_equal(q.cpu().numpy(), qo)


def test_nvfp4_quantiser_zero_matrix(q4):
    q, s, g = q4.q4_quantize_nvfp4(torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda"))
    assert g.item() == 1.0 and int(q.sum()) == 0 and int(s.sum()) == 0


def test_quantise_then_linear(q4, oracle_mod):
    """Pack a random bf16 matrix on the GPU, then run both linear layers on it."""
    N, K = 1024, 2048
    wb = _weights("normal", N, K, 3)
    x = synth.activations(synth.rng_for(41), 3, K)
    wd = _dev_bf16(wb)
    q, s, m = q4.q4_quantize_int4g128(wd)
    y = q4.q4_linear_int4g128(P.bf16_dev(x), q, s, m)
    yo, ao = oracle_mod.linear_int4g128(x, q.cpu().numpy(),
                                        s.cpu().view(torch.int16).numpy().view(np.uint16),
                                        m.cpu().view(torch.int16).numpy().view(np.uint16),
                                        with_abs=True)
    P.check(y, yo, ao, "int4 quantised then linear")
    c, sc, g = q4.q4_quantize_nvfp4(wd)
    y = q4.q4_linear_nvfp4(P.bf16_dev(x), c, sc, g)
    yo, ao = oracle_mod.linear_nvfp4(x, c.cpu().numpy(), sc.cpu().numpy(), g.cpu().numpy()[0],
                                     with_abs=True)
    P.check(y, yo, ao, "nvfp4 quantised then linear")


def test_quantiser_argument_errors(q4):
    w = torch.zeros((4, 100), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(q4.Q4Error):
        q4.q4_quantize_int4g128(w)                       # K % 128 != 0
    with pytest.raises(q4.Q4Error):
        q4.q4_quantize_nvfp4(torch.zeros((4, 24), dtype=torch.bfloat16, device="cuda"))
