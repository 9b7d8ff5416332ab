"""The decode step as the bench runs it: dependent calls captured in one CUDA graph
with programmatic dependent launch, replayed, and every call's output compared
with the oracle.

Page "Rumik TTS Fast Inference", section "What Made It Faster": the decode step
runs as a CUDA graph, with projections that share an input packed into one call.
Under programmatic dependent launch call i + 1's CTAs are resident while call i
runs and request their weights before call i has finished, so these tests check
that no call reads its activations, or writes its output, too early.  Each call
writes a buffer of its own, so that every output of the replay can be read back
and fed, as the GPU's own bf16 bits, to the oracle."""
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


def _capture(q4, fn):
    """Capture fn() into a graph on a side stream with PDL launches."""
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    q4.set_launch_flags(q4.FLAG_PDL)
    try:
        with torch.cuda.stream(s):
            fn()                                  # plans and attributes, outside capture
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                fn()
    finally:
        q4.set_launch_flags(0)
    return g, s


def _cat(mats, names):
    return synth.Int4Matrix(np.concatenate([mats[n].qweight for n in names]),
                            np.concatenate([mats[n].scale for n in names]),
                            np.concatenate([mats[n].minv for n in names]))


@pytest.mark.parametrize("fusion", ["all", "pairs"])
def test_decode_step_graph_with_pdl_matches_oracle(q4, oracle_mod, fusion):
    """Four layers of the synthetic 28-layer int4 stack and the 2,049-row
    restricted head in one graph of PDL-chained calls, replayed twice; every
    call checked against the oracle on its own input.  fusion "all": q|k|v|gate|up
    as one call, o and down reading the v and up slices of its output (13
    calls); "pairs": q|k|v and gate|up as two calls (17 calls).  The next layer
    reads down's output."""
    L = 4
    H, F = 2048, 8192
    names = [("q", "k", "v", "gate", "up")] if fusion == "all" else [("q", "k", "v"), ("gate", "up")]
    layers = []
    for layer in range(L):
        mats = synth.decode_stack_layer(layer)
        d = {"o": mats["o"], "down": mats["down"]}
        for nm in names:
            d["|".join(nm)] = _cat(mats, nm)
        layers.append(d)
    dev = [{k: P.int4_dev(v) for k, v in l.items()} for l in layers]
    head = synth.decode_stack_head()
    head_d = P.bf16_dev(head)
    x0 = P.bf16_dev(synth.decode_stack_input())
    width = {"q|k|v|gate|up": 3 * H + 2 * F, "q|k|v": 3 * H, "gate|up": 2 * F, "o": H, "down": H}
    out = [{k: torch.empty((1, width[k]), dtype=torch.bfloat16, device="cuda") for k in l}
           for l in layers]
    # where o and down find their inputs: (output name, first column)
    v_src = ("q|k|v|gate|up", 2 * H) if fusion == "all" else ("q|k|v", 2 * H)
    up_src = ("q|k|v|gate|up", 3 * H + F) if fusion == "all" else ("gate|up", F)
    logits = torch.empty((1, 2049), dtype=torch.bfloat16, device="cuda")

    def step():
        x = x0
        for d, o in zip(dev, out):
            for nm in names:
                key = "|".join(nm)
                q4.q4_linear_int4g128(x, *d[key], y=o[key])
                if key != "gate|up":
                    q4.q4_linear_int4g128(o[v_src[0]][:, v_src[1]:v_src[1] + H], *d["o"], y=o["o"])
            q4.q4_linear_int4g128(o[up_src[0]][:, up_src[1]:up_src[1] + F], *d["down"], y=o["down"])
            x = o["down"]
        q4.audio_head_logits_restricted(x, head_d, 0, 2049, -1, logits=logits)

    q4.device_error_flags()               # clear
    g, s = _capture(q4, step)
    for o in out:
        for t in o.values():
            t.fill_(float("nan"))
    logits.fill_(float("nan"))
    results = []
    for _ in range(2):
        with torch.cuda.stream(s):
            g.replay()
        torch.cuda.synchronize()
        results.append([{k: P.bf16_bits_host(t) for k, t in o.items()} for o in out] +
                       [P.bf16_bits_host(logits)])
    assert q4.device_error_flags() == 0
    # replays are bit-identical (no call depends on timing)
    for a, b in zip(results[0][:L], results[1][:L]):
        for k in a:
            assert np.array_equal(a[k], b[k]), k
    assert np.array_equal(results[0][L], results[1][L])

    host = results[0]
    x = synth.decode_stack_input()
    for li, (lay, o) in enumerate(zip(layers, host)):
        def chk(name, inp, w):
            yo, ao = oracle_mod.linear_int4g128(inp, w.qweight, w.scale, w.minv, with_abs=True)
            y = torch.from_numpy(o[name].view(np.int16)).view(torch.bfloat16)
            P.check(y, yo, ao, f"graph ({fusion}) layer {li} {name}")
        for nm in names:
            chk("|".join(nm), x, lay["|".join(nm)])
        chk("o", np.ascontiguousarray(o[v_src[0]][:, v_src[1]:v_src[1] + H]), lay["o"])
        chk("down", np.ascontiguousarray(o[up_src[0]][:, up_src[1]:up_src[1] + F]), lay["down"])
        x = o["down"]
    yo, ao = oracle_mod.head_restricted(x, head, 0, 2049, -1, with_abs=True)
    P.check(torch.from_numpy(host[L].view(np.int16)).view(torch.bfloat16), yo, ao, "graph head")


def test_nvfp4_16384x2048_chain_with_deferred_ring_requests(q4, oracle_mod):
    """Three dependent one-token NVFP4 16384 x 2048 calls (each reads 2,048 outputs
    of the one before) in a PDL graph: at this shape each warp owns more rows than
    it requests before the dependency wait, so the launch holds the later requests
    back (the deferred-ring case).  Every output checked against the oracle."""
    rng = synth.rng_for(301)
    mats = [synth.nvfp4_matrix(rng, 16384, 2048) for _ in range(3)]
    dev = [P.nvfp4_dev(w) for w in mats]
    x0 = P.bf16_dev(synth.activations(rng, 1, 2048))
    ys = [torch.empty((1, 16384), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    slices = [slice(0, 2048), slice(4096, 6144)]

    def chain():
        x = x0
        for i, (d, y) in enumerate(zip(dev, ys)):
            q4.q4_linear_nvfp4(x, *d, y=y)
            if i < 2:
                x = y[:, slices[i]]

    q4.device_error_flags()               # clear
    g, s = _capture(q4, chain)
    for y in ys:
        y.fill_(float("nan"))
    for _ in range(2):
        with torch.cuda.stream(s):
            g.replay()
    torch.cuda.synchronize()
    assert q4.device_error_flags() == 0
    x = P.bf16_bits_host(x0)
    for i, (w, y) in enumerate(zip(mats, ys)):
        yo, ao = oracle_mod.linear_nvfp4(x, w.codes, w.scale, w.global_scale, with_abs=True)
        P.check(y, yo, ao, f"nvfp4 chain call {i}")
        if i < 2:
            x = np.ascontiguousarray(P.bf16_bits_host(y)[:, slices[i]])
