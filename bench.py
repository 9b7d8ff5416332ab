"""Benchmark of the 4-bit weight-only decode GEMV on one GB300 (or N replicas).

Default workload: NVFP4 weight-only GEMV at batch 1, K=2048 -> N=16384 (seeded
synthetic weights: E2M1 codes uniform over 16 values, e4m3 group-16 scales from
U[0.25, 4], global scale 1e-2; x ~ N(0,1) in bf16).  Each call runs the whole
path (E2M1/e4m3 decode, dot products, bf16 store).

Timing: the calls rotate over enough copies of the weights to cover 4x the L2
cache, so every call streams its weights from HBM.  One step is about 8,192
chained calls: whole passes over that ring of copies, replayed from one CUDA
graph of one pass.  W warm-up steps replay the same graph, then K timed steps
are bracketed by CUDA events on the launching stream with a barrier +
synchronize on both sides; the max over ranks is taken.  `value` is the
effective weight bandwidth (algorithmic bytes / time per call).
The `e2e` key repeats the measurement through the same public call with the
activations copied in from pinned host memory and the result copied back every
step (copies on their own streams, device x and y double-buffered, so one step's
copies overlap the neighbouring steps' kernels; the host results are checked
against the device results).  `--impl reference` times the CPU oracle on the
host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "4-bit decode GEMV µs/call & effective weight GB/s (% of GB300 HBM peak)"
# GB300 HBM3e nominal bandwidth; fractions are reported against it beside the measured peak
HBM_NOMINAL_GBS = 8000.0
# Chained calls per bench step (rounded up to whole passes over the weight ring):
# a step lasts tens of milliseconds, so a 20-step timed region spans several
# clock samples and the per-call time is a steady-state figure.
CALLS_PER_STEP = 8192

# DRAM traffic of one launch of the decode GEMV kernel on a workload, from the ncu
# capture summarised in profiles/ (dram__bytes_read.sum + dram__bytes_write.sum),
# valid only for the kernel sources it was taken on (see _kernel_sha).
TRAFFIC = {
    # workload key: (bytes per launch, _kernel_sha() when captured)
    "nvfp4_gemv": (18919936, "03360da5c802ba8e7bcfcc5c71750e9d1255abd8631d054df1a48f5955185b73"),
}



# ---------------------------------------------------------------- helpers
def _dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, world: int) -> float:
    """Max of a per-rank float over all ranks (identity for one process)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


KERNEL_SOURCES = ("bit_weight_only_q4_gb300/csrc/gemv_rows.cu",
                  "bit_weight_only_q4_gb300/csrc/stream_common.cuh",
                  "bit_weight_only_q4_gb300/csrc/q4_device.cuh")


def _kernel_sha() -> str:
    """Hash of the sources of the decode GEMV kernel (traffic figures are only
    valid for the kernel they were captured on)."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def traffic_for(workload: str):
    """DRAM bytes per launch recorded for `workload` from an ncu capture, or None
    when nothing was recorded or the kernel sources changed since the capture."""
    t = TRAFFIC.get(workload)
    return t[0] if t and t[1] == _kernel_sha() else None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines: list[str] = []
        self.t = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", self.gpu_id],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.t is not None:
                self.t.join(timeout=2)

    def summary(self) -> dict:
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ workloads
class Workload:
    """Seeded inputs on the device, a ring of weight copies and one call per step."""

    def __init__(self, name: str, device):
        import torch
        from bit_weight_only_q4_gb300 import layout, q4, synth
        from bit_weight_only_q4_gb300 import upload as P
        self.name = name
        self.torch = torch
        self.q4 = q4
        self.device = device
        l2 = torch.cuda.get_device_properties(device).L2_cache_size
        self.kernel_launches_per_step = 1
        if name == "nvfp4_gemv":
            c = synth.NVFP4_GEMV_16384
            x, w = synth.nvfp4_gemv_16384()
            self.M, self.N, self.K = c["M"], c["N"], c["K"]
            self.layout = "nvfp4"
            self.desc = c["name"]
            base = P.nvfp4_dev(w)
        elif name == "int8_gemv":
            c = synth.INT8_GEMV_16384
            x, w = synth.int8_gemv_16384()
            self.M, self.N, self.K = c["M"], c["N"], c["K"]
            self.layout = "int8"
            self.desc = c["name"]
            base = P.int8_dev(w)
        elif name == "int4_gemv":
            c = synth.INT4_GEMV_2048
            x, w = synth.int4_gemv_2048()
            self.M, self.N, self.K = c["M"], c["N"], c["K"]
            self.layout = "int4"
            self.desc = c["name"]
            base = P.int4_dev(w)
        else:
            raise ValueError(f"workload {name} has no GEMV bench line")
        self.x_host_bits = x
        self.x = P.bf16_dev(x).to(device)
        self.bytes_per_call = layout.linear_bytes(self.layout, self.M, self.N, self.K)
        wbytes = layout.weight_bytes(self.layout, self.N, self.K)
        self.copies = max(2, math.ceil(4 * l2 / wbytes))
        self.ring = [tuple(t.to(device).clone() for t in base) for _ in range(self.copies)]
        self.y = torch.empty((self.M, self.N), dtype=torch.bfloat16, device=device)
        lay = q4.LAYOUT_NVFP4 if self.layout == "nvfp4" else q4.LAYOUT_INT4G128
        self.ws = None if self.layout == "int8" else \
            q4.alloc_workspace(lay, self.M, self.N, self.K, device)
        self.ring_bytes = self.copies * wbytes
        self.l2 = l2

    def call(self, i: int, x=None, y=None):
        w = self.ring[i % self.copies]
        x = self.x if x is None else x
        y = self.y if y is None else y
        if self.layout == "nvfp4":
            self.q4.q4_linear_nvfp4(x, *w, y=y, workspace=self.ws)
        elif self.layout == "int8":
            self.q4.q4_linear_int8(x, *w, y=y)
        else:
            self.q4.q4_linear_int4g128(x, *w, y=y, workspace=self.ws)


def _capture(torch, fn, n: int, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                fn(i)
    return g


def _time_graphs(torch, stream, graphs, world):
    """Replay graphs [(graph, times)] between two events; returns elapsed ms."""
    barrier(world)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    with torch.cuda.stream(stream):
        for g, times in graphs:
            for _ in range(times):
                g.replay()
    end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    return start.elapsed_time(end)


# ------------------------------------------------------- further workloads
def _graph_time(torch, stream, fn, n_calls, reps, warm=3):
    """Capture fn(0..n_calls-1) once; return ms per replay over `reps` replays."""
    with torch.cuda.stream(stream):
        for i in range(n_calls):
            fn(i)
    torch.cuda.synchronize()
    g = _capture(torch, fn, n_calls, stream)
    _time_graphs(torch, stream, [(g, warm)], 1)
    return _time_graphs(torch, stream, [(g, reps)], 1) / reps


def run_decode_step(args, device):
    """One decode step of the synthetic 28-layer int4 stack (hidden 2048, FFN
    8192): per layer q, k, v, gate, up read x; o reads v; down reads up; the
    next layer's x is down's output; then the restricted head (2049 rows).
    Projections that share an input run as one call on their concatenated rows:
    by default q|k|v|gate|up (N = 22528), then o and down read their inputs as
    slices of that output, 3 calls per layer + the head = 85 per step;
    --fusion pairs runs q|k|v (N = 6144) and gate|up (N = 16384) as two calls
    (113 per step), --fusion none the 7 separate calls per layer (197 per step).
    Replayed from one CUDA graph; 1.007 GB of weights per step."""
    import torch
    from bit_weight_only_q4_gb300 import layout, q4, synth
    from bit_weight_only_q4_gb300 import upload as P
    c = synth.DECODE_STACK_28
    H, F = c["hidden"], c["ffn"]
    fusion = "none" if getattr(args, "no_fuse", False) else getattr(args, "fusion", "all")
    fuse = fusion != "none"
    layers = []
    for layer in range(c["layers"]):
        m = {k: P.int4_dev(v) for k, v in synth.decode_stack_layer(layer).items()}
        cat = lambda names: tuple(torch.cat([m[n][i] for n in names], 0).contiguous()
                                  for i in range(3))
        if fusion == "all":
            layers.append({"f": cat(("q", "k", "v", "gate", "up")), "o": m["o"],
                           "down": m["down"]})
        elif fusion == "pairs":
            layers.append({"qkv": cat(("q", "k", "v")), "o": m["o"],
                           "gu": cat(("gate", "up")), "down": m["down"]})
        else:
            layers.append(m)
    head = P.bf16_dev(synth.decode_stack_head())
    x0 = P.bf16_dev(synth.decode_stack_input())
    logits = torch.empty((1, c["head_rows"]), dtype=torch.bfloat16, device=device)
    shapes = {"all": [(3 * H + 2 * F, H), (H, H), (H, F)],
              "pairs": [(3 * H, H), (H, H), (2 * F, H), (H, F)],
              "none": [(N, K) for _, N, K in synth.DECODE_LAYER_PROJS]}[fusion]
    ws_n = max(q4.workspace_bytes(q4.LAYOUT_INT4G128, 1, N, K) for N, K in shapes)
    ws = torch.zeros(ws_n, dtype=torch.uint8, device=device) if ws_n else None
    wbytes = sum(layout.weight_bytes("int4", N, K) for _, N, K in synth.DECODE_LAYER_PROJS) \
        * c["layers"] + 2 * c["head_rows"] * H
    if fusion == "all":
        y_f = torch.empty((1, 3 * H + 2 * F), dtype=torch.bfloat16, device=device)
        y_o = torch.empty((1, H), dtype=torch.bfloat16, device=device)
        y_down = torch.empty((1, H), dtype=torch.bfloat16, device=device)
        v_view = y_f[:, 2 * H:3 * H]          # v's rows of the fused output
        up_view = y_f[:, 3 * H + F:]          # up's rows

        def step(_):
            x = x0
            for L in layers:
                q4.q4_linear_int4g128(x, *L["f"], y=y_f, workspace=ws)
                q4.q4_linear_int4g128(v_view, *L["o"], y=y_o, workspace=ws)
                q4.q4_linear_int4g128(up_view, *L["down"], y=y_down, workspace=ws)
                x = y_down
            q4.audio_head_logits_restricted(x, head, 0, c["head_rows"], -1, logits=logits)
        launches = 3 * c["layers"] + 1
    elif fusion == "pairs":
        y_qkv = torch.empty((1, 3 * H), dtype=torch.bfloat16, device=device)
        y_o = torch.empty((1, H), dtype=torch.bfloat16, device=device)
        y_gu = torch.empty((1, 2 * F), dtype=torch.bfloat16, device=device)
        y_down = torch.empty((1, H), dtype=torch.bfloat16, device=device)
        v_view = y_qkv[:, 2 * H:]            # v's rows of the fused output
        up_view = y_gu[:, F:]                # up's rows

        def step(_):
            x = x0
            for L in layers:
                q4.q4_linear_int4g128(x, *L["qkv"], y=y_qkv, workspace=ws)
                q4.q4_linear_int4g128(v_view, *L["o"], y=y_o, workspace=ws)
                q4.q4_linear_int4g128(x, *L["gu"], y=y_gu, workspace=ws)
                q4.q4_linear_int4g128(up_view, *L["down"], y=y_down, workspace=ws)
                x = y_down
            q4.audio_head_logits_restricted(x, head, 0, c["head_rows"], -1, logits=logits)
        launches = 4 * c["layers"] + 1
    else:
        buf = {n: torch.empty((1, F if n in ("gate", "up") else H), dtype=torch.bfloat16,
                              device=device) for n in ("q", "k", "v", "o", "gate", "up", "down")}
        src = {"q": "x", "k": "x", "v": "x", "o": "v", "gate": "x", "up": "x", "down": "up"}

        def step(_):
            x = x0
            for L in layers:
                for name, N, K in synth.DECODE_LAYER_PROJS:
                    inp = x if src[name] == "x" else buf[src[name]]
                    q4.q4_linear_int4g128(inp, *L[name], y=buf[name], workspace=ws)
                x = buf["down"]
            q4.audio_head_logits_restricted(x, head, 0, c["head_rows"], -1, logits=logits)
        launches = len(synth.DECODE_LAYER_PROJS) * c["layers"] + 1

    stream = torch.cuda.Stream(device)
    ms = _graph_time(torch, stream, step, 1, max(args.steps, 200))
    peak, _ = _peaks()
    gbs = wbytes / (ms * 1e-3) / 1e9
    return {"workload": c["name"], "ms_per_step": round(ms, 4), "weight_bytes": wbytes,
            "value": round(gbs, 1), "unit": "GB/s", "hbm_frac": round(gbs / peak, 4),
            "hbm_frac_nominal": round(gbs / HBM_NOMINAL_GBS, 4),
            "steps_per_s": round(1e3 / ms, 1), "launches_per_step": launches,
            "fusion": fusion, "fused_projections": fuse, "pdl": not args.no_pdl}


def run_batched(args, device):
    """NVFP4 batched decode at M tokens: K=2048 -> N=8192 then K=8192 -> N=2048
    per step, weights rotating over >= 4x L2; swept over M."""
    import torch
    from bit_weight_only_q4_gb300 import layout, q4, synth
    from bit_weight_only_q4_gb300 import upload as P
    c = synth.NVFP4_BATCHED_48
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    out = {"workload": c["name"], "sweep": []}
    peak, _ = _peaks()
    for M in c["m_sweep"]:
        calls = []
        for si, (N, K) in enumerate(c["shapes"]):
            x, w = synth.nvfp4_batched(si, M)
            base = P.nvfp4_dev(w)
            copies = max(2, math.ceil(2 * l2 / layout.weight_bytes("nvfp4", N, K)))
            ring = [tuple(t.clone() for t in base) for _ in range(copies)]
            xd = P.bf16_dev(x)
            y = torch.empty((M, N), dtype=torch.bfloat16, device=device)
            wsb = q4.alloc_workspace(q4.LAYOUT_NVFP4, M, N, K, device)
            calls.append((ring, xd, y, wsb))
        R = len(calls[0][0])

        def fn(i):
            for ring, xd, y, wsb in calls:
                q4.q4_linear_nvfp4(xd, *ring[i % len(ring)], y=y, workspace=wsb)

        stream = torch.cuda.Stream(device)
        ms = _graph_time(torch, stream, fn, R, max(20, args.steps // R)) / R
        wb = sum(layout.weight_bytes("nvfp4", N, K) for N, K in c["shapes"])
        flops = sum(2 * M * N * K for N, K in c["shapes"])
        gbs = wb / (ms * 1e-3) / 1e9
        out["sweep"].append({"M": M, "us_per_step": round(ms * 1e3, 3), "weight_GBps": round(gbs, 1),
                             "hbm_frac": round(gbs / peak, 4),
                             "hbm_frac_nominal": round(gbs / HBM_NOMINAL_GBS, 4),
                             "tflops": round(flops / (ms * 1e-3) / 1e12, 2)})
    return out


def run_prefill(args, device):
    """Prefill GEMM, M=2048 tokens: int4-g128 and NVFP4, K=2048 -> N=8192 and
    K=8192 -> N=2048 (68.7 GFLOP each), tcgen05 path."""
    import torch
    from bit_weight_only_q4_gb300 import q4, synth
    from bit_weight_only_q4_gb300 import upload as P
    c = synth.PREFILL_2048
    res = {"workload": c["name"], "gemms": []}
    bf16_peak = _bf16_peak()
    for lay in ("int4", "nvfp4"):
        for si, (N, K) in enumerate(c["shapes"]):
            x, w = synth.prefill(lay, si)
            xd = P.bf16_dev(x)
            y = torch.empty((c["M"], N), dtype=torch.bfloat16, device=device)
            if lay == "int4":
                wd = P.int4_dev(w)
                wsb = q4.alloc_workspace(q4.LAYOUT_INT4G128, c["M"], N, K, device)
                fn = lambda i, xd=xd, wd=wd, y=y, wsb=wsb: q4.q4_linear_int4g128(xd, *wd, y=y, workspace=wsb)
            else:
                wd = P.nvfp4_dev(w)
                wsb = q4.alloc_workspace(q4.LAYOUT_NVFP4, c["M"], N, K, device)
                fn = lambda i, xd=xd, wd=wd, y=y, wsb=wsb: q4.q4_linear_nvfp4(xd, *wd, y=y, workspace=wsb)
            stream = torch.cuda.Stream(device)
            ms = _graph_time(torch, stream, fn, 10, max(20, args.steps // 10)) / 10
            tf = 2 * c["M"] * N * K / (ms * 1e-3) / 1e12
            res["gemms"].append({"layout": lay, "N": N, "K": K, "us": round(ms * 1e3, 2),
                                 "tflops": round(tf, 1), "tensor_frac": round(tf / bf16_peak, 4)})
    return res


def run_embedding(args, device):
    """int8 token-embedding gather + dequant ([277404, 2048] table, the full
    vocabulary of the pages' model) for M = 1 and M = 48 tokens per call, chained
    in a CUDA graph with PDL.  Bytes per call: M rows of 2048 int8 codes and one
    fp16 scale read, M x 2048 bf16 written."""
    import torch
    from bit_weight_only_q4_gb300 import q4
    V, H = 277404, 2048
    g = torch.Generator(device="cpu").manual_seed(7)
    q = torch.randint(-128, 128, (V, H), generator=g, dtype=torch.int8).to(device)
    sc = (torch.rand(V, generator=g) * 0.02 + 1e-4).to(torch.float16).to(device)
    peak, _ = _peaks()
    res = {"workload": "int8 embedding gather, V=277404, H=2048", "runs": []}
    for M in (1, 48):
        ids = torch.randint(0, V, (M,), generator=g, dtype=torch.int32).to(device)
        out = torch.empty((M, H), dtype=torch.bfloat16, device=device)
        fn = lambda i, ids=ids, out=out: q4.q4_embedding_int8(ids, q, sc, out=out)
        stream = torch.cuda.Stream(device)
        ms = _graph_time(torch, stream, fn, 50, max(20, args.steps // 50)) / 50
        nbytes = M * (H + 2 + 2 * H + 4)
        res["runs"].append({"M": M, "us_per_call": round(ms * 1e3, 3),
                            "GBps": round(nbytes / (ms * 1e-3) / 1e9, 1)})
    return res


def run_quantize(args, device):
    """Round-to-nearest quantisers from bf16 (packing, not the decode path): a
    16384 x 2048 and an 8192 x 8192 matrix (weights N(0, 0.02)) into both layouts.
    Bytes counted: the bf16 read once plus the packed write (NVFP4 reads the
    matrix a second time for its global amax; that read is not counted)."""
    import torch
    from bit_weight_only_q4_gb300 import layout, q4, synth
    peak, _ = _peaks()
    res = {"workload": "round-to-nearest quantisers, bf16 -> int4-g128 / NVFP4",
           "runs": []}
    for (N, K) in ((16384, 2048), (8192, 8192)):
        g = torch.Generator(device="cpu").manual_seed(N + K)
        w = (torch.randn((N, K), generator=g) * 0.02).to(torch.bfloat16).to(device)
        for lay in ("int4", "nvfp4"):
            if lay == "int4":
                fn = lambda i, w=w: q4.q4_quantize_int4g128(w)
            else:
                fn = lambda i, w=w: q4.q4_quantize_nvfp4(w)
            stream = torch.cuda.Stream(device)
            ms = _graph_time(torch, stream, fn, 5, max(20, args.steps // 5)) / 5
            nbytes = 2 * N * K + layout.weight_bytes(lay, N, K)
            gbs = nbytes / (ms * 1e-3) / 1e9
            res["runs"].append({"layout": lay, "N": N, "K": K, "us": round(ms * 1e3, 2),
                                "GBps": round(gbs, 1), "hbm_frac": round(gbs / peak, 4),
                                "hbm_frac_nominal": round(gbs / HBM_NOMINAL_GBS, 4)})
    return res


def _bf16_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return float(json.load(f)["bf16_tflops"])
    return 1900.0


def run_extra(args, local):
    import torch
    from bit_weight_only_q4_gb300 import build as libbuild
    from bit_weight_only_q4_gb300 import q4
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    libbuild.build()
    q4.load()
    q4.set_launch_flags(q4.FLAG_PDL if not args.no_pdl else 0)
    fn = {"decode_step": run_decode_step, "batched": run_batched, "prefill": run_prefill,
          "quantize": run_quantize, "embedding": run_embedding}
    r = fn[args.workload](args, device)
    r["metric"] = METRIC
    r["data"] = "synthetic (seeded PCG64)"
    print(json.dumps(r), flush=True)


def run_profile(args, local):
    """Plain launches for an ncu capture: W warm-up calls, then K calls, no graphs
    and no timing (a number printed under a profiler is never a bench value).
    GEMV workloads rotate their weight ring; prefill cycles through the int4 and
    the NVFP4 K=2048 -> N=8192 GEMM, then the int4 and the NVFP4 K=8192 -> N=2048
    GEMM, at M=2048 (template argument 0 of the kernel is int4, 1 NVFP4; the int4
    calls also launch the x pre-pass); batched runs the NVFP4 K=8192 ->
    N=2048 GEMM at M=48; decode_step runs the step's distinct calls (fused
    q|k|v|gate|up 22528 x 2048, o 2048 x 2048, down 2048 x 8192, then the
    restricted head) over eight layers' weights (289 MB, beyond L2) in turn."""
    import torch
    from bit_weight_only_q4_gb300 import build as libbuild
    from bit_weight_only_q4_gb300 import q4, synth
    from bit_weight_only_q4_gb300 import upload as P
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    libbuild.build()
    q4.load()
    q4.set_launch_flags(0)
    if args.workload in ("nvfp4_gemv", "int4_gemv", "int8_gemv"):
        wl = Workload(args.workload, device)
        call, desc = wl.call, wl.desc
    elif args.workload == "prefill":
        gemms = []
        for si in (0, 1):
            x, w = synth.prefill("int4", si)
            _, wn = synth.prefill("nvfp4", si)
            xd = P.bf16_dev(x)
            ws = q4.alloc_workspace(q4.LAYOUT_INT4G128, x.shape[0], w.N, w.K, device)
            gemms.append((q4.q4_linear_int4g128, xd, P.int4_dev(w), ws))
            gemms.append((q4.q4_linear_nvfp4, xd, P.nvfp4_dev(wn), ws))

        def call(i):
            f, xd, wd, ws = gemms[i % 4]
            f(xd, *wd, workspace=ws)
        desc = ("prefill M=2048: int4 and nvfp4 K=2048 N=8192, then int4 and nvfp4 "
                "K=8192 N=2048, in turn")
    elif args.workload == "decode_step":
        c = synth.DECODE_STACK_28
        H, F = c["hidden"], c["ffn"]
        nl = 8
        layers = []
        for layer in range(nl):
            m = {k: P.int4_dev(v) for k, v in synth.decode_stack_layer(layer).items()}
            f = tuple(torch.cat([m[n][j] for n in ("q", "k", "v", "gate", "up")], 0).contiguous()
                      for j in range(3))
            layers.append((f, m["o"], m["down"]))
        head = P.bf16_dev(synth.decode_stack_head())
        x0 = P.bf16_dev(synth.decode_stack_input())
        y_f = torch.empty((1, 3 * H + 2 * F), dtype=torch.bfloat16, device=device)
        y_o = torch.empty((1, H), dtype=torch.bfloat16, device=device)
        y_d = torch.empty((1, H), dtype=torch.bfloat16, device=device)
        logits = torch.empty((1, c["head_rows"]), dtype=torch.bfloat16, device=device)
        ws_n = max(q4.workspace_bytes(q4.LAYOUT_INT4G128, 1, N, K)
                   for N, K in ((3 * H + 2 * F, H), (H, H), (H, F)))
        ws = torch.zeros(ws_n, dtype=torch.uint8, device=device) if ws_n else None

        def call(i):
            f, o, d = layers[i % nl]
            q4.q4_linear_int4g128(x0, *f, y=y_f, workspace=ws)
            q4.q4_linear_int4g128(y_f[:, 2 * H:3 * H], *o, y=y_o, workspace=ws)
            q4.q4_linear_int4g128(y_f[:, 3 * H + F:], *d, y=y_d, workspace=ws)
            q4.audio_head_logits_restricted(y_d, head, 0, c["head_rows"], -1, logits=logits)
        desc = "decode-step calls: int4 22528x2048, 2048x2048, 2048x8192, head 2049x2048"
    elif args.workload == "batched":
        x, w = synth.nvfp4_batched(1, 48)
        xd, wd = P.bf16_dev(x), P.nvfp4_dev(w)
        ws = q4.alloc_workspace(q4.LAYOUT_NVFP4, 48, w.N, w.K, device)
        call = lambda i: q4.q4_linear_nvfp4(xd, *wd, workspace=ws)
        desc = "nvfp4 M=48 K=8192 N=2048"
    else:
        raise SystemExit(f"--profile does not cover {args.workload}")
    for i in range(args.warmup + args.steps):
        call(i)
    torch.cuda.synchronize()
    print(json.dumps({"profile_run": desc, "calls": args.warmup + args.steps}))


def run_gpu(args, world, rank, local):
    import torch
    from bit_weight_only_q4_gb300 import build as libbuild
    from bit_weight_only_q4_gb300 import q4

    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if rank == 0:
        libbuild.build()
    barrier(world)
    libbuild.build()
    q4.load()
    q4.set_launch_flags(q4.FLAG_PDL if not args.no_pdl else 0)
    wl = Workload(args.workload, device)
    stream = torch.cuda.Stream(device)
    R = wl.copies
    K, W = args.steps, args.warmup
    # One step = P passes over the R-copy weight ring (R * P chained calls, about
    # CALLS_PER_STEP), replayed from one graph of R calls.  Warm-up replays that
    # same graph, so the timed region never holds a first replay.
    P_ring = max(1, math.ceil(CALLS_PER_STEP / R))
    calls_per_step = R * P_ring

    with torch.cuda.stream(stream):
        for i in range(R):                 # first, uncaptured calls: plans and attributes cached
            wl.call(i)
    torch.cuda.synchronize()
    g_ring = _capture(torch, wl.call, R, stream)
    _time_graphs(torch, stream, [(g_ring, W * P_ring)], world)

    props = torch.cuda.get_device_properties(device)
    gpu_id = str(getattr(props, "uuid", local))
    if gpu_id and not gpu_id.startswith("GPU-") and "-" in gpu_id:
        gpu_id = "GPU-" + gpu_id
    with ClockSampler(gpu_id) as clk:
        ms = _time_graphs(torch, stream, [(g_ring, K * P_ring)], world)
    ms = max_over_ranks(ms, world)
    clocks = clk.summary()

    # End to end through the public call: every step copies its x in from pinned
    # host memory and its y back out to pinned host memory.  The copies run on
    # their own streams with double-buffered device x and y, so that step i + 1's
    # input copy and step i's output copy overlap step i's kernel, as in a
    # serving loop; every copy still happens inside the timed region.
    NBUF = 2
    xh = torch.empty_like(wl.x, device="cpu").pin_memory()
    xh.copy_(wl.x.cpu())
    yh = [torch.empty((wl.M, wl.N), dtype=torch.bfloat16).pin_memory() for _ in range(NBUF)]
    xd = [torch.empty_like(wl.x) for _ in range(NBUF)]
    yd = [torch.empty_like(wl.y) for _ in range(NBUF)]
    s_in = torch.cuda.Stream(device)
    s_out = torch.cuda.Stream(device)
    k_ev = [torch.cuda.Event() for _ in range(NBUF)]     # kernel of the buffer's last step
    x_ev = [torch.cuda.Event() for _ in range(NBUF)]     # input copy landed
    o_ev = [torch.cuda.Event() for _ in range(NBUF)]     # output copy done

    def e2e_steps(n):
        cur = torch.cuda.current_stream()
        s_in.wait_stream(cur)                             # fork (joins a graph capture)
        s_out.wait_stream(cur)
        for i in range(n):
            b = i % NBUF
            if i >= NBUF:
                s_in.wait_event(k_ev[b])                  # step i - 2's kernel read xd[b]
            with torch.cuda.stream(s_in):
                xd[b].copy_(xh, non_blocking=True)
                x_ev[b].record(s_in)
            cur.wait_event(x_ev[b])
            if i >= NBUF:
                cur.wait_event(o_ev[b])                   # step i - 2's output copy read yd[b]
            wl.call(i, x=xd[b], y=yd[b])
            k_ev[b].record(cur)
            s_out.wait_event(k_ev[b])
            with torch.cuda.stream(s_out):
                yh[b].copy_(yd[b], non_blocking=True)
                o_ev[b].record(s_out)
        cur.wait_stream(s_in)                             # join before the graph ends
        cur.wait_stream(s_out)

    def e2e_graph(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                e2e_steps(n)
        return g

    with torch.cuda.stream(stream):
        e2e_steps(3)
    torch.cuda.synchronize()
    ge = e2e_graph(R)
    _time_graphs(torch, stream, [(ge, W * P_ring)], world)
    e2e_ms = _time_graphs(torch, stream, [(ge, K * P_ring)], world)
    e2e_ms = max_over_ranks(e2e_ms, world)
    # each host buffer holds the result of the last step that used it
    torch.cuda.synchronize()
    for b in range(NBUF):
        if not torch.equal(yh[b].view(torch.int16), yd[b].cpu().view(torch.int16)):
            raise SystemExit("end-to-end output copy does not match the device result")

    us_per_call = ms * 1e3 / (K * calls_per_step)
    gbs = wl.bytes_per_call / (us_per_call * 1e-6) / 1e9
    e2e_us = e2e_ms * 1e3 / (K * calls_per_step)
    e2e_gbs = wl.bytes_per_call / (e2e_us * 1e-6) / 1e9
    peak, peak_src = _peaks()
    traffic = traffic_for(args.workload)

    cpu_baseline = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu_baseline = time_oracle(wl.name, budget_s=args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC,
            "value": round(gbs * world, 2),
            "unit": "GB/s",
            "us_per_call": round(us_per_call, 4),
            "hbm_frac": round(gbs / peak, 4),
            "hbm_frac_nominal": round(gbs / HBM_NOMINAL_GBS, 4),
            "n_gpus": world,
            "steps": K,
            "warmup": W,
            "ms_per_step": round(ms / K, 6),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            # NVFP4 whole-row GEMV: fp16 partial sums per 16-column group, fp32 across
            # groups; the other layouts accumulate in fp32
            "dtype": "f16/f32" if wl.layout == "nvfp4" else "f32",
            "data": "synthetic (seeded PCG64; shapes and distributions of the workload)",
            "config": {
                "workload": wl.desc,
                "layout": wl.layout, "M": wl.M, "N": wl.N, "K": wl.K,
                "algorithmic_bytes_per_call": wl.bytes_per_call,
                "l2": f"weights rotate over {wl.copies} copies "
                      f"({wl.ring_bytes / 1e6:.0f} MB, >= 4x the {wl.l2 / 1e6:.0f} MB L2)",
                "calls_per_step": calls_per_step,
                "step": f"{calls_per_step} chained calls: {P_ring} passes over the "
                        f"{R}-copy weight ring, replayed from one CUDA graph of {R} calls "
                        f"(warm-up replays the same graph)",
                "pdl": not args.no_pdl,
                "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
            },
            "roofline": {
                "bound": "hbm",
                "achieved": round(gbs, 2),
                "peak": peak,
                "unit": "GB/s",
                "frac": round(gbs / peak, 4),
                "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
                else "fallback 6.8 TB/s",
                "traffic": traffic,
            },
            "e2e": {
                "value": round(e2e_gbs * world, 2),
                "unit": "GB/s",
                "us_per_call": round(e2e_us, 4),
                "h2d_bytes_per_step": int(wl.x.numel() * 2) * calls_per_step,
                "d2h_bytes_per_step": int(wl.M * wl.N * 2) * calls_per_step,
                "steps": K,
            },
            "gpu_launches": K * calls_per_step * wl.kernel_launches_per_step,
            "clocks": clocks,
            "cpu_baseline": cpu_baseline,
        }
        print(json.dumps(line), flush=True)


# ------------------------------------------------------------- CPU oracle
def time_oracle(workload: str, budget_s: float = 12.0, steps: int | None = None) -> dict:
    """Time the CPU oracle (as it stands) on a bounded sample of the workload."""
    import numpy as np
    import oracle
    from bit_weight_only_q4_gb300 import layout, synth
    if workload == "nvfp4_gemv":
        x, w = synth.nvfp4_gemv_16384()
        N, K, lay = w.N, w.K, "nvfp4"

        def run(rows):
            oracle.linear_nvfp4(x, w.codes[:rows], w.scale[:rows], w.global_scale)
    elif workload == "int8_gemv":
        x, w = synth.int8_gemv_16384()
        N, K, lay = w.N, w.K, "int8"

        def run(rows):
            oracle.linear_int8(x, w.qweight[:rows], w.scale[:rows])
    else:
        x, w = synth.int4_gemv_2048()
        N, K, lay = w.N, w.K, "int4"

        def run(rows):
            oracle.linear_int4g128(x, w.qweight[:rows], w.scale[:rows], w.minv[:rows])
    oracle.build()
    run(min(N, 256))
    t0 = time.perf_counter()
    run(N)
    t_full = time.perf_counter() - t0
    if steps is None:
        calls = max(1, int(budget_s / max(t_full, 1e-6)))
        rows = N
    else:
        # each step a bounded sample of rows: the whole run stays within budget_s
        per_step = budget_s / max(steps, 1)
        rows = int(max(64, min(N, N * per_step / max(t_full, 1e-9))))
        calls = steps
    t0 = time.perf_counter()
    for _ in range(calls):
        run(rows)
    dt = time.perf_counter() - t0
    us_per_call = dt / calls * (N / rows) * 1e6
    gbs = layout.linear_bytes(lay, 1, N, K) / (us_per_call * 1e-6) / 1e9
    return {"value": round(gbs, 4), "unit": "GB/s", "us_per_call": round(us_per_call, 2),
            "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{calls} oracle calls on {rows} of {N} rows (K={K}), "
                      f"time scaled to all rows; {dt:.1f} s"}


def run_reference(args, world, rank):
    if rank != 0:
        return
    wl_desc = {"nvfp4_gemv": "nvfp4 GEMV M=1 N=16384 K=2048",
               "int4_gemv": "int4-g128 GEMV M=1 N=2048 K=2048",
               "int8_gemv": "int8 weight-only GEMV M=1 N=16384 K=2048"}[args.workload]
    budget = min(150.0, max(10.0, 2.0 * (args.steps + args.warmup)))
    cb = time_oracle(args.workload, budget_s=budget, steps=args.steps)
    line = {
        "metric": METRIC, "impl": "reference", "value": cb["value"], "unit": "GB/s",
        "us_per_call": cb["us_per_call"], "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": cb["us_per_call"] * CALLS_PER_STEP / 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded PCG64)",
        "config": {"workload": wl_desc, "calls_per_step": CALLS_PER_STEP,
                   "step": "each timed step runs the oracle once on a sample of rows; "
                           "ms_per_step is the per-call time scaled to a step of "
                           f"{CALLS_PER_STEP} calls"},
        "cpu_baseline": cb,
        "e2e": {"value": cb["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=("nvfp4_gemv", "int4_gemv", "int8_gemv", "decode_step", "batched", "quantize", "embedding",
                                           "prefill"), default="nvfp4_gemv",
                    help="nvfp4_gemv is the bench line; the others print their own "
                         "measurement lines")
    ap.add_argument("--no-pdl", action="store_true")
    ap.add_argument("--no-fuse", action="store_true",
                    help="decode_step: run q, k, v, gate, up as separate calls")
    ap.add_argument("--fusion", choices=("all", "pairs", "none"), default="all",
                    help="decode_step: q|k|v|gate|up as one call (all), q|k|v and "
                         "gate|up (pairs), or separate calls (none)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--profile", action="store_true",
                    help="plain launches for an ncu capture (no timing output)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = _dist_env()
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        if backend == "nccl":
            import torch
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    try:
        if args.impl == "reference":
            run_reference(args, world, rank)
        elif args.profile:
            run_profile(args, local)
        elif args.workload in ("decode_step", "batched", "prefill", "quantize", "embedding"):
            run_extra(args, local)
        else:
            run_gpu(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
