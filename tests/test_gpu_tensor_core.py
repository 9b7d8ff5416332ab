"""GPU parity of the tcgen05 tensor-core path (batched decode and prefill) against
the CPU oracle: forced tensor-core launches over ragged shapes, the batched-decode
M sweep, and the prefill GEMM at full size on sampled output rows."""
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


def _run(q4, layout, x, w, flags):
    q4.set_launch_flags(flags)
    try:
        if layout == "int4":
            y = q4.q4_linear_int4g128(P.bf16_dev(x), *P.int4_dev(w))
        else:
            y = q4.q4_linear_nvfp4(P.bf16_dev(x), *P.nvfp4_dev(w))
    finally:
        q4.set_launch_flags(0)
    torch.cuda.synchronize()
    assert q4.device_error_flags() == 0
    return y


def _oracle(oracle_mod, layout, x, w, rows=None):
    if layout == "int4":
        q, s, m = (w.qweight, w.scale, w.minv) if rows is None else \
            (w.qweight[rows], w.scale[rows], w.minv[rows])
        return oracle_mod.linear_int4g128(x, q, s, m, with_abs=True)
    c, s = (w.codes, w.scale) if rows is None else (w.codes[rows], w.scale[rows])
    return oracle_mod.linear_nvfp4(x, c, s, w.global_scale, with_abs=True)


def _mat(layout, rng, N, K):
    return synth.int4_matrix(rng, N, K) if layout == "int4" else synth.nvfp4_matrix(rng, N, K)


@pytest.mark.parametrize("layout", ["int4", "nvfp4"])
@pytest.mark.parametrize("M,N,K", [(16, 128, 128), (1, 128, 128), (5, 200, 256), (48, 1000, 640),
                                   (64, 384, 1024), (200, 130, 2048), (300, 256, 384),
                                   (17, 8192, 128), (48, 96, 8192), (8, 512, 2048),
                                   (33, 2049, 8192), (64, 2048, 8192), (16, 16384, 2048),
                                   (300, 10000, 256), (2048, 2432, 128), (7, 130, 64),
                                   (48, 200, 192)])
def test_forced_tensor_core_shapes(q4, oracle_mod, layout, M, N, K):
    """The tensor-core kernel on every shape (int4: x converted to fp16 in the
    kernel up to 64 tokens, by the pre-pass above; NVFP4: bf16 operands, x as
    stored, and up to 64 tokens A in tensor memory with two chunks per stage,
    here also with a last stage of one chunk (K = 64, 192); A sub-tiles in
    tensor memory from 65 to 255
    tokens; CTAs of two 128-row tiles for 256-token tiles, here with a ragged last
    token tile and a last row pair that ends inside its first tile or at its
    second)."""
    if layout == "int4" and K % 128:
        pytest.skip("int4 needs K % 128")
    rng = synth.rng_for(300, M, N, K)
    w = _mat(layout, rng, N, K)
    x = synth.activations(rng, M, K)
    y = _run(q4, layout, x, w, q4.FLAG_FORCE_TENSOR_CORE)
    yo, ao = _oracle(oracle_mod, layout, x, w)
    P.check(y, yo, ao, f"tc {layout} M={M} N={N} K={K}")


@pytest.mark.parametrize("layout", ["int4", "nvfp4"])
def test_tensor_core_matches_cuda_core(q4, layout):
    """The two kernel families agree with each other as well as with the oracle."""
    rng = synth.rng_for(301)
    w = _mat(layout, rng, 512, 2048)
    x = synth.activations(rng, 8, 2048)
    a = _run(q4, layout, x, w, q4.FLAG_FORCE_TENSOR_CORE).float()
    b = _run(q4, layout, x, w, q4.FLAG_FORCE_CUDA_CORE).float()
    rel = float((a - b).norm() / b.norm())
    assert rel < 3e-3


@pytest.mark.parametrize("layout", ["int4", "nvfp4"])
@pytest.mark.parametrize("shape_index", [0, 1])
def test_prefill_2048_tokens_sampled_rows(q4, oracle_mod, layout, shape_index):
    x, w = synth.prefill(layout, shape_index)
    y = _run(q4, layout, x, w, 0)
    N = w.N
    rows = np.unique(np.concatenate([np.arange(0, 5), np.arange(N - 5, N),
                                     synth.rng_for(302, shape_index).integers(0, N, 22)]))
    yo, ao = _oracle(oracle_mod, layout, x, w, rows)
    P.check(y[:, torch.as_tensor(rows, device=y.device)], yo, ao,
            f"prefill {layout} shape {shape_index}")


def test_tensor_core_is_deterministic(q4):
    """Split-K sums run in k order: repeated calls are bit-identical."""
    rng = synth.rng_for(303)
    w = synth.nvfp4_matrix(rng, 2048, 8192)
    x = synth.activations(rng, 48, 8192)
    y1 = _run(q4, "nvfp4", x, w, 0)
    for _ in range(3):
        y2 = _run(q4, "nvfp4", x, w, 0)
        assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


def _x_tokens_of_many_scales(rng, M, K):
    """bf16 activations whose tokens sit at very different magnitudes: token m is
    N(0,1) times 2^s_m, with s_m cycling over -60, -20, 0, 10, 20 (|x| up to about
    10^6, far beyond the fp16 range), 60 and 120; one column of the first token
    holds 10^6 itself."""
    xf = rng.standard_normal((M, K)).astype(np.float32)
    shifts = np.array([-60, -20, 0, 10, 20, 60, 120], np.float32)
    xf *= np.exp2(shifts[np.arange(M) % shifts.size])[:, None]
    xf[0, 7] = 1.0e6
    return torch.from_numpy(xf).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("layout", ["int4", "nvfp4"])
@pytest.mark.parametrize("M,N,K", [(16, 1024, 2048), (48, 384, 8192), (2048, 256, 2048),
                                   (100, 512, 1024), (300, 10000, 128)])
def test_activations_beyond_the_fp16_range(q4, oracle_mod, layout, M, N, K):
    """Tokens at magnitudes from 2^-60 to 2^120 match the oracle and set no error
    bit.  int4: the MMA operand is fp16 (max 65504), so every token is scaled by
    a power of two before the conversion and its sums scaled back (in-kernel
    conversion up to 64 tokens, the pre-pass above).  NVFP4: bf16 operands take x
    as stored, and the weights carry a power-of-two share of the global scale.
    Both with A in tensor memory at 100 and 2048 tokens and with two-row-tile
    CTAs at 300 tokens x 10000 rows."""
    rng = synth.rng_for(304, M, N, K)
    w = _mat(layout, rng, N, K)
    x = _x_tokens_of_many_scales(rng, M, K)
    q4.device_error_flags()            # clear
    y = _run(q4, layout, x, w, q4.FLAG_FORCE_TENSOR_CORE)
    yo, ao = _oracle(oracle_mod, layout, x, w)
    # the relative Frobenius bound is applied per token (tokens differ by 2^180)
    for m in range(M):
        P.check(y[m:m + 1], yo[m:m + 1], ao[m:m + 1], f"tc {layout} token {m} M={M}")


@pytest.mark.parametrize("M,N,K", [(16, 384, 1024), (48, 2048, 8192), (100, 384, 1024),
                                   (300, 10000, 128)])
def test_nvfp4_global_scale_is_applied_exactly(q4, oracle_mod, M, N, K):
    """NVFP4 on the tensor cores carries a power of two 2^eg of the global scale g
    in its bf16 weights (eg clamped to [-100, 6]) and multiplies the accumulator by
    g * 2^-eg.  Scaling g by a power of two therefore scales every output by the
    same power exactly, wherever eg lands (inside the clamp, at either end of it),
    as long as the outputs stay normal bf16 numbers; g = 0 gives zeros; and a
    non-power-of-two g at either extreme matches the oracle.  Shapes: split-K
    ring kernel, one row tile; A in tensor memory; two-row-tile CTAs."""
    rng = synth.rng_for(305, M, N, K)
    w = synth.nvfp4_matrix(rng, N, K, global_scale=1.0)
    # |x| >= 2^-8, so that no product x * w * 2^eg falls below the fp32 normal range
    xf = rng.standard_normal((M, K)).astype(np.float32)
    xf = np.sign(xf) * np.maximum(np.abs(xf), np.float32(2.0 ** -8))
    x = torch.from_numpy(xf).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    y1 = _run(q4, "nvfp4", x, w, q4.FLAG_FORCE_TENSOR_CORE).float()
    for e in (-120, -100, -40, 6, 7, 40):
        w.global_scale = np.float32(2.0 ** e)
        yg = _run(q4, "nvfp4", x, w, q4.FLAG_FORCE_TENSOR_CORE)
        want = (y1 * (2.0 ** e)).to(torch.bfloat16)
        normal = (want.float().abs() >= 2.0 ** -126) | (y1 == 0)
        assert normal.float().mean().item() > 0.99
        assert torch.equal(yg.view(torch.int16)[normal], want.view(torch.int16)[normal]), e
    w.global_scale = np.float32(0.0)
    assert torch.count_nonzero(_run(q4, "nvfp4", x, w, q4.FLAG_FORCE_TENSOR_CORE)).item() == 0
    for g in (3.1e-33, 1.7e3):
        w.global_scale = np.float32(g)
        y = _run(q4, "nvfp4", x, w, q4.FLAG_FORCE_TENSOR_CORE)
        yo, ao = _oracle(oracle_mod, "nvfp4", x, w)
        P.check(y.float() / g, yo / g, ao / g, f"tc nvfp4 g={g} M={M}")
