"""Host-side logic of bench.py: max-over-ranks aggregation across 2 gloo ranks
(the multi-GPU replica path, exercised on CPU) and the CPU-oracle timing leg."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_WORKER = r"""
import os, sys
sys.path.insert(0, {root!r})
import torch.distributed as dist
import bench
dist.init_process_group("gloo")
r = dist.get_rank()
v = bench.max_over_ranks(1.5 + 2.0 * r, dist.get_world_size())
bench.barrier(dist.get_world_size())
print("RESULT", r, v, flush=True)
dist.destroy_process_group()
"""


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def test_max_over_ranks_gloo_world2():
    port = _free_port()
    procs = []
    for r in range(2):
        env = dict(os.environ, RANK=str(r), WORLD_SIZE="2", LOCAL_RANK=str(r),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, "-c", _WORKER.format(root=ROOT)],
                                      env=env, stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                                      text=True))
    outs = [p.communicate(timeout=120) for p in procs]
    for p, (o, e) in zip(procs, outs):
        assert p.returncode == 0, e
    vals = sorted(float(o.split()[-1]) for o, _ in outs)
    assert vals == [3.5, 3.5]


def test_reference_arm_prints_one_json_line():
    env = dict(os.environ)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "int4_gemv", "--steps", "3", "--warmup", "3"],
                       capture_output=True, text=True, timeout=300, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_traffic_figure_only_for_the_sources_it_was_captured_on(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    sha = bench._kernel_sha()
    assert len(sha) == 64
    monkeypatch.setattr(bench, "TRAFFIC", {"w": (123, sha), "old": (456, "0" * 64)})
    assert bench.traffic_for("w") == 123
    assert bench.traffic_for("old") is None          # kernel changed since the capture
    assert bench.traffic_for("missing") is None


def test_kernel_hash_covers_the_gemv_sources():
    sys.path.insert(0, ROOT)
    import bench
    for rel in bench.KERNEL_SOURCES:
        assert os.path.exists(os.path.join(ROOT, rel)), rel
    assert any(rel.endswith("gemv_rows.cu") for rel in bench.KERNEL_SOURCES)


def test_recorded_traffic_matches_the_current_gemv_sources():
    """The bench's DRAM-traffic figure for the headline GEMV was captured on the
    kernel sources as they are now: a change to them needs a new ncu capture."""
    sys.path.insert(0, ROOT)
    import bench
    assert bench.traffic_for("nvfp4_gemv") is not None
