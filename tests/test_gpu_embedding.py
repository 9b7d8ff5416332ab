"""GPU int8 token-embedding gather against the oracle.  The output is the exact
product q * scale rounded once to bf16, so it must match the oracle's exact value
rounded by torch (nearest even) bit for bit."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from bit_weight_only_q4_gb300 import synth

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


def _table(V: int, H: int, seed: int):
    rng = synth.rng_for(50, seed, V, H)
    q = rng.integers(-128, 128, size=(V, H), dtype=np.int8)
    s = rng.uniform(1e-4, 2e-2, size=V).astype(np.float16).view(np.uint16)
    return q, s


def _bf16_bits_of(exact: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(exact.astype(np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("V,H,M", [(16385, 2048, 1), (16385, 2048, 48), (1000, 16, 7),
                                   (277404, 2048, 3)])
def test_embedding_gather_bit_exact(q4, oracle_mod, V, H, M):
    q, s = _table(V, H, 1)
    ids = synth.rng_for(51, V, M).integers(0, V, size=M).astype(np.int32)
    ids[0] = V - 1                                      # last row of the table
    qd = torch.from_numpy(q).cuda()
    sd = torch.from_numpy(s.view(np.int16)).view(torch.float16).cuda()
    out = q4.q4_embedding_int8(torch.from_numpy(ids).cuda(), qd, sd)
    want = _bf16_bits_of(oracle_mod.embedding_int8(ids, q, s))
    got = out.cpu().view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(got, want)


def test_embedding_ids_outside_the_table(q4, oracle_mod):
    V, H = 64, 256
    q, s = _table(V, H, 2)
    ids = np.array([5, -1, 64, 63, 2**31 - 1], np.int32)
    q4.device_error_flags(clear=True)
    out = q4.q4_embedding_int8(torch.from_numpy(ids).cuda(), torch.from_numpy(q).cuda(),
                               torch.from_numpy(s.view(np.int16)).view(torch.float16).cuda())
    flags = q4.device_error_flags(clear=True)
    assert flags & 0x4
    got = out.cpu().view(torch.int16).numpy().view(np.uint16)
    want = _bf16_bits_of(oracle_mod.embedding_int8(ids, q, s))
    np.testing.assert_array_equal(got, want)
    assert np.all(got[[1, 2, 4]] == 0)


def test_embedding_shape_errors(q4):
    q = torch.zeros((8, 24), dtype=torch.int8, device="cuda")
    s = torch.zeros((8,), dtype=torch.float16, device="cuda")
    ids = torch.zeros((2,), dtype=torch.int32, device="cuda")
    with pytest.raises(q4.Q4Error):
        q4.q4_embedding_int8(ids, q, s)                 # H % 16 != 0
