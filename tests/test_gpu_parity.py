"""GPU parity: every kernel path through the C ABI against the CPU oracle, on the
seeded synthetic inputs (element-wise tolerance and relative Frobenius error),
plus bit-exact checks of the in-kernel decoders."""
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


def _int4_case(q4, oracle_mod, M, N, K, seed, flags=0, rows=None):
    rng = synth.rng_for(100 + seed, M, N, K)
    w = synth.int4_matrix(rng, N, K)
    x = synth.activations(rng, M, K)
    q, s, m = P.int4_dev(w)
    q4.set_launch_flags(flags)
    try:
        y = q4.q4_linear_int4g128(P.bf16_dev(x), q, s, m)
    finally:
        q4.set_launch_flags(0)
    torch.cuda.synchronize()
    if rows is None:
        yo, ao = oracle_mod.linear_int4g128(x, w.qweight, w.scale, w.minv, with_abs=True)
        return P.check(y, yo, ao, f"int4 M={M} N={N} K={K}")
    yo, ao = oracle_mod.linear_int4g128(x, w.qweight[rows], w.scale[rows], w.minv[rows],
                                        with_abs=True)
    return P.check(y[:, torch.as_tensor(rows, device=y.device)], yo, ao,
                   f"int4 M={M} N={N} K={K} (sampled rows)")


def _nvfp4_case(q4, oracle_mod, M, N, K, seed, flags=0, gscale=1e-2):
    rng = synth.rng_for(200 + seed, M, N, K)
    w = synth.nvfp4_matrix(rng, N, K, gscale)
    x = synth.activations(rng, M, K)
    c, s, g = P.nvfp4_dev(w)
    q4.set_launch_flags(flags)
    try:
        y = q4.q4_linear_nvfp4(P.bf16_dev(x), c, s, g)
    finally:
        q4.set_launch_flags(0)
    torch.cuda.synchronize()
    yo, ao = oracle_mod.linear_nvfp4(x, w.codes, w.scale, w.global_scale, with_abs=True)
    return P.check(y, yo, ao, f"nvfp4 M={M} N={N} K={K}")


# ------------------------------------------------------------ decoders
@pytest.mark.parametrize("N,K", [(2048, 2048), (3, 128), (17, 8192)])
def test_dequant_int4_bit_exact(q4, oracle_mod, N, K):
    w = synth.int4_matrix(synth.rng_for(7, N, K), N, K)
    got = q4.q4_dequant_int4g128_f32(*P.int4_dev(w)).cpu().numpy()
    ref = oracle_mod.dequant_int4g128(w.qweight, w.scale, w.minv)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("N,K,G", [(16384, 2048, 1e-2), (5, 16, 0.37), (9, 48, 3.0)])
def test_dequant_nvfp4_bit_exact(q4, oracle_mod, N, K, G):
    w = synth.nvfp4_matrix(synth.rng_for(8, N, K), N, K, G)
    got = q4.q4_dequant_nvfp4_f32(*P.nvfp4_dev(w)).cpu().numpy()
    ref = oracle_mod.dequant_nvfp4(w.codes, w.scale, w.global_scale)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_dequant_nvfp4_all_code_scale_pairs(q4, oracle_mod):
    """Every E2M1 code against every finite e4m3 scale byte."""
    scales = np.array([b for b in range(256) if (b & 0x7f) != 0x7f], np.uint8)
    N = scales.size
    codes = np.tile(np.array([0x10 * ((2 * j + 1) % 16) + (2 * j) % 16 for j in range(8)],
                             np.uint8), (N, 1))                      # 16 codes per row
    w = synth.Nvfp4Matrix(codes, scales.reshape(N, 1), np.float32(0.7))
    got = q4.q4_dequant_nvfp4_f32(*P.nvfp4_dev(w)).cpu().numpy()
    ref = oracle_mod.dequant_nvfp4(w.codes, w.scale, w.global_scale)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


# ------------------------------------------------- GEMV, batch 1 configs
def test_int4_gemv_2048x2048_seed0(q4, oracle_mod):
    x, w = synth.int4_gemv_2048()
    y = q4.q4_linear_int4g128(P.bf16_dev(x), *P.int4_dev(w))
    yo, ao = oracle_mod.linear_int4g128(x, w.qweight, w.scale, w.minv, with_abs=True)
    P.check(y, yo, ao, "int4 GEMV 2048x2048")


def test_nvfp4_gemv_16384x2048_seed1(q4, oracle_mod):
    x, w = synth.nvfp4_gemv_16384()
    y = q4.q4_linear_nvfp4(P.bf16_dev(x), *P.nvfp4_dev(w))
    yo, ao = oracle_mod.linear_nvfp4(x, w.codes, w.scale, w.global_scale, with_abs=True)
    P.check(y, yo, ao, "nvfp4 GEMV 16384x2048")


# ------------------------------------------------- ragged and edge shapes
@pytest.mark.parametrize("N,K", [(1, 128), (37, 128), (1000, 3200), (3, 8192), (4099, 1152),
                                 (64, 65536)])
def test_int4_ragged_shapes(q4, oracle_mod, N, K):
    _int4_case(q4, oracle_mod, 1, N, K, seed=1)


@pytest.mark.parametrize("N,K", [(1, 16), (5, 16), (77, 48), (300, 2080), (129, 1040),
                                 (2050, 4112), (8, 32)])
def test_nvfp4_ragged_shapes(q4, oracle_mod, N, K):
    _nvfp4_case(q4, oracle_mod, 1, N, K, seed=2)


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8, 16, 33, 48])
def test_m_sweep_small(q4, oracle_mod, M):
    _int4_case(q4, oracle_mod, M, 520, 2048, seed=3)
    _nvfp4_case(q4, oracle_mod, M, 264, 1040, seed=3)


def test_large_n_uses_64bit_offsets(q4, oracle_mod):
    """N*K/2 > 2^31 bytes: sampled rows near the end of the matrix."""
    N, K = 1 << 21, 2048                  # 2 GiB of codes
    rows = np.array([0, 1, N // 2, N - 513, N - 2, N - 1])
    _int4_case(q4, oracle_mod, 1, N, K, seed=4, rows=rows)


# ----------------------------------------------------------------- head
def test_head_2049_rows_config(q4, oracle_mod):
    head = synth.decode_stack_head()
    h = synth.decode_stack_input()
    out = q4.audio_head_logits_restricted(P.bf16_dev(h), P.bf16_dev(head), 0, 2049, -1)
    yo, ao = oracle_mod.head_restricted(h, head, 0, 2049, -1, with_abs=True)
    P.check(out, yo, ao, "head 2049x2048")


@pytest.mark.parametrize("M,codebook", [(1, 0), (3, 5), (2, 7)])
def test_head_16385_row_codebook_slice(q4, oracle_mod, M, codebook):
    rng = synth.rng_for(31, M, codebook)
    head = synth.head_matrix(rng, 16385, 2048)
    h = synth.activations(rng, M, 2048)
    hd = P.bf16_dev(head)
    out = q4.audio_head_logits_restricted(P.bf16_dev(h), hd, 2048 * codebook, 2048, 16384)
    yo, ao = oracle_mod.head_restricted(h, head, 2048 * codebook, 2048, 16384, with_abs=True)
    P.check(out, yo, ao, "head codebook slice")


@pytest.mark.parametrize("rows,H,rb,nr,ex", [(10, 8, 0, 10, -1), (50, 72, 3, 0, 49),
                                              (300, 2056, 7, 291, 0)])
def test_head_edge_shapes(q4, oracle_mod, rows, H, rb, nr, ex):
    rng = synth.rng_for(32, rows, H)
    head = synth.head_matrix(rng, rows, H)
    h = synth.activations(rng, 2, H)
    out = q4.audio_head_logits_restricted(P.bf16_dev(h), P.bf16_dev(head), rb, nr, ex)
    yo, ao = oracle_mod.head_restricted(h, head, rb, nr, ex, with_abs=True)
    P.check(out, yo, ao, "head edge")


# -------------------------------------------------------- determinism / flags
def test_split_k_is_deterministic_and_pdl_is_neutral(q4):
    x, w = synth.nvfp4_gemv_16384()
    xd = P.bf16_dev(x)
    args = P.nvfp4_dev(w)
    y1 = q4.q4_linear_nvfp4(xd, *args)
    y2 = q4.q4_linear_nvfp4(xd, *args)
    q4.set_launch_flags(q4.FLAG_PDL)
    try:
        y3 = q4.q4_linear_nvfp4(xd, *args)
    finally:
        q4.set_launch_flags(0)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    assert torch.equal(y1.view(torch.int16), y3.view(torch.int16))


def test_workspace_too_small_returns_status_and_launches_nothing(q4):
    x, w = synth.int4_gemv_2048()
    q, s, m = P.int4_dev(w)
    y = torch.full((1, 2048), 7.0, dtype=torch.bfloat16, device="cuda")
    need = q4.workspace_bytes(0, 1, 2048, 2048)
    ws = torch.zeros(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(q4.Q4Error) as ei:
        q4.q4_linear_int4g128(P.bf16_dev(x), q, s, m, y=y, workspace=ws)
    assert ei.value.status == 4
    torch.cuda.synchronize()
    assert bool((y.float() == 7.0).all())


# ------------------------------------------------------- decode stack config
def test_decode_stack_layers_per_call_parity(q4, oracle_mod):
    """Config of a 28-layer int4 decode step (projections chained q,k,v <- x;
    o <- v; gate, up <- x; down <- up; next x <- down): first, middle and last
    layer run through the chain, each call checked against the oracle on the
    GPU's own bf16 input."""
    x = synth.decode_stack_input()
    for layer in (0, 13, 27):
        mats = synth.decode_stack_layer(layer)
        dev = {k: P.int4_dev(v) for k, v in mats.items()}
        outs = {}
        src = {"q": "x", "k": "x", "v": "x", "o": "v", "gate": "x", "up": "x", "down": "up"}
        for name, _, _ in synth.DECODE_LAYER_PROJS:
            inp = x if src[name] == "x" else outs[src[name]]
            y = q4.q4_linear_int4g128(P.bf16_dev(inp), *dev[name])
            w = mats[name]
            yo, ao = oracle_mod.linear_int4g128(inp, w.qweight, w.scale, w.minv, with_abs=True)
            P.check(y, yo, ao, f"layer {layer} {name}")
            outs[name] = P.bf16_bits_host(y)
        x = outs["down"]


def test_decode_stack_fused_projections(q4, oracle_mod):
    """Projections sharing an input as one call on concatenated rows (q|k|v,
    gate|up), as the decode-step bench runs them; o and down read their inputs
    as slices of the fused outputs.  Each call is checked against the oracle on
    the concatenated matrix and the GPU's own bf16 input."""
    import numpy as np
    x = synth.decode_stack_input()
    for layer in (0, 27):
        mats = synth.decode_stack_layer(layer)
        cat = lambda names: synth.Int4Matrix(
            np.concatenate([mats[n].qweight for n in names]),
            np.concatenate([mats[n].scale for n in names]),
            np.concatenate([mats[n].minv for n in names]))
        qkv, gu = cat(("q", "k", "v")), cat(("gate", "up"))
        xd = P.bf16_dev(x)
        y_qkv = q4.q4_linear_int4g128(xd, *P.int4_dev(qkv))
        yo, ao = oracle_mod.linear_int4g128(x, qkv.qweight, qkv.scale, qkv.minv, with_abs=True)
        P.check(y_qkv, yo, ao, f"layer {layer} qkv")
        v = y_qkv[:, 4096:]
        y_o = q4.q4_linear_int4g128(v, *P.int4_dev(mats["o"]))
        w = mats["o"]
        yo, ao = oracle_mod.linear_int4g128(P.bf16_bits_host(v), w.qweight, w.scale, w.minv,
                                             with_abs=True)
        P.check(y_o, yo, ao, f"layer {layer} o from the v slice")
        y_gu = q4.q4_linear_int4g128(xd, *P.int4_dev(gu))
        yo, ao = oracle_mod.linear_int4g128(x, gu.qweight, gu.scale, gu.minv, with_abs=True)
        P.check(y_gu, yo, ao, f"layer {layer} gate|up")
        up = y_gu[:, 8192:]
        y_d = q4.q4_linear_int4g128(up, *P.int4_dev(mats["down"]))
        w = mats["down"]
        yo, ao = oracle_mod.linear_int4g128(P.bf16_bits_host(up), w.qweight, w.scale, w.minv,
                                             with_abs=True)
        P.check(y_d, yo, ao, f"layer {layer} down from the up slice")
        x = P.bf16_bits_host(y_d)


# ------------------------------------------------------ batched decode config
@pytest.mark.parametrize("shape_index", [0, 1])
@pytest.mark.parametrize("M", [1, 3, 8, 16, 32, 48])
def test_nvfp4_batched_sweep(q4, oracle_mod, shape_index, M):
    x, w = synth.nvfp4_batched(shape_index, M)
    y = q4.q4_linear_nvfp4(P.bf16_dev(x), *P.nvfp4_dev(w))
    yo, ao = oracle_mod.linear_nvfp4(x, w.codes, w.scale, w.global_scale, with_abs=True)
    P.check(y, yo, ao, f"nvfp4 batched M={M} shape {shape_index}")


# ------------------------------------------- k-step counts that are not powers of two
@pytest.mark.parametrize("K", [3072, 6144, 12288])
@pytest.mark.parametrize("M", [1, 3, 4])
def test_k_not_a_power_of_two_ksteps(q4, oracle_mod, M, K):
    """K = 3072 and 6144 (3 and 6 k-steps of 1024 columns) run the whole-row
    kernel with its k-steps padded to 4 and 8 (the padded ones read nothing);
    K = 12288 (12 k-steps) runs the split-K kernel.  Both layouts, 1-4 tokens."""
    _int4_case(q4, oracle_mod, M, 1000, K, seed=5)
    _nvfp4_case(q4, oracle_mod, M, 1000, K, seed=5)


# ------------------------------------------------------ one-token shapes
@pytest.mark.parametrize("N,K", [(1, 2048), (17, 4096), (151, 2048), (152, 8192), (153, 2048),
                                 (1000, 16384), (4099, 2048), (16384, 4096)])
def test_one_token_shapes_around_the_sm_count(q4, oracle_mod, N, K):
    """One token: rows fewer than, equal to and just above the SM count (one CTA
    per SM), rows per CTA that leave warps without a row, one to sixteen
    1024-column k-steps per row (16384: the split-K kernel)."""
    _int4_case(q4, oracle_mod, 1, N, K, seed=6)
    _nvfp4_case(q4, oracle_mod, 1, N, K, seed=6)
