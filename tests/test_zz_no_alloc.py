"""The allocation-free int4 entry point (q4_linear_int4g128_noalloc), called
through the C ABI.  It serves callers that cannot allocate device memory -- code
in a real-time callback that must not block in the allocator, a plugin whose host
application owns every device buffer, a graph recorded after its memory pool was
frozen -- so its split-K scratch is a static array inside the library instead of
a caller workspace.

Its output must match the fp64 oracle within the parity tolerance, and agree with
the workspace entry point within that same tolerance, on two calls in a row (the
second call reuses the scratch the first one left behind), for one token, for
several launches per call (M >= 5, every launch reusing the counters and partial
sums) and with programmatic dependent launch on; shapes beyond the static scratch
must be refused.  This file sorts last so that a run stopping at its first failure
has already run every other test."""
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


@pytest.mark.parametrize("pdl", [False, True])
@pytest.mark.parametrize("M,N,K", [(1, 2048, 2048), (3, 1000, 3200), (1, 513, 8192),
                                   (7, 700, 4096), (13, 256, 2048)])
def test_noalloc_matches_oracle_twice(lib, oracle_mod, M, N, K, pdl):
    lib.set_launch_flags(lib.FLAG_PDL if pdl else 0)
    try:
        for call in range(2):
            rng = synth.rng_for(77, M, N, K, call)
            w = synth.int4_matrix(rng, N, K)
            x = synth.activations(rng, M, K)
            q, s, m = P.int4_dev(w)
            xd = P.bf16_dev(x)
            y_ws = lib.q4_linear_int4g128(xd, q, s, m)
            y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
            assert _noalloc(lib, xd, q, s, m, y) == 0, lib.load().q4_last_error_string()
            torch.cuda.synchronize()
            yo, ao = oracle_mod.linear_int4g128(x, w.qweight, w.scale, w.minv, with_abs=True)
            P.check(y, yo, ao, f"noalloc call {call} M={M} N={N} K={K} pdl={pdl}")
            # the workspace entry point, within the same tolerance
            ref = y_ws.float().cpu().numpy().astype(np.float64)
            P.check(y, ref, ao, f"noalloc vs workspace call {call} M={M} N={N} K={K}")
    finally:
        lib.set_launch_flags(0)


def test_noalloc_rejects_shapes_beyond_the_static_scratch(lib):
    L = lib.load()
    M, N, K = 4, 262144, 16384       # needs far more than 4 MiB of partial sums
    big = 1 << 20                    # aligned fake pointers: rejected before any launch
    st = L.q4_linear_int4g128_noalloc(big, big, big, big, big, M, N, K, None)
    assert st == 2
    assert b"static scratch" in L.q4_last_error_string()
