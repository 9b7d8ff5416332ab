"""The allocation-free int4 entry point (q4_linear_int4g128_noalloc), called
through the C ABI: it serves callers that cannot allocate device memory (a
real-time callback, a plugin whose host owns all device buffers), so its split-K
scratch is a static array inside the library.  Its output must match the
workspace entry point within the parity tolerance on two calls in a row (the
second call reuses the scratch the first one left behind), and shapes beyond the
static scratch must be refused.  This file sorts last so that a run stopping at
its first failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

from bit_weight_only_q4_gb300 import synth
from tests import parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_weight_only_q4_gb300 import build, q4
    build.build()
    q4.load()
    q4.set_launch_flags(0)
    return q4


def _noalloc(lib, x, q, s, m, y):
    L = lib.load()
    M, K = x.shape
    N = q.shape[0]
    stream = torch.cuda.current_stream().cuda_stream
    return L.q4_linear_int4g128_noalloc(x.data_ptr(), q.data_ptr(), s.data_ptr(), m.data_ptr(),
                                        y.data_ptr(), M, N, K, ctypes.c_void_p(stream))


@pytest.mark.parametrize("M,N,K", [(1, 2048, 2048), (3, 1000, 3200), (1, 513, 8192)])
def test_noalloc_matches_workspace_entry_point_twice(lib, oracle_mod, M, N, K):
    for call in range(2):
        rng = synth.rng_for(77, M, N, K, call)
        w = synth.int4_matrix(rng, N, K)
        x = synth.activations(rng, M, K)
        q, s, m = P.int4_dev(w)
        xd = P.bf16_dev(x)
        y_ref = lib.q4_linear_int4g128(xd, q, s, m)
        y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert _noalloc(lib, xd, q, s, m, y) == 0, lib.load().q4_last_error_string()
        torch.cuda.synchronize()
        _, ao = oracle_mod.linear_int4g128(x, w.qweight, w.scale, w.minv, with_abs=True)
        ref = y_ref.float().cpu().numpy().astype(np.float64)
        P.check(y, ref, ao, f"noalloc call {call} M={M} N={N} K={K}")


def test_noalloc_rejects_shapes_beyond_the_static_scratch(lib):
    L = lib.load()
    M, N, K = 4, 262144, 16384       # needs far more than 4 MiB of partial sums
    big = 1 << 20                    # aligned fake pointers: rejected before any launch
    st = L.q4_linear_int4g128_noalloc(big, big, big, big, big, M, N, K, None)
    assert st == 2
    assert b"static scratch" in L.q4_last_error_string()
