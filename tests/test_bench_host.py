"""Host-side logic of bench.py (no GPU): multi-rank timing reduction over gloo, peak/traffic lookup, and
the CPU reference arm's JSON line."""

import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, queue):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    r, local, w = bench.dist_setup()
    bench.barrier(w)
    value = bench.max_over_ranks(1.5 + r, w)
    queue.put((r, w, value))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert out == [(0, 2, 2.5), (1, 2, 2.5)]


def test_single_rank_defaults(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_setup() == (0, 0, 1)
    assert bench.max_over_ranks(3.25, 1) == 3.25


def test_peaks_and_traffic_lookup(monkeypatch, tmp_path):
    sys.path.insert(0, ROOT)
    import bench
    peak, kind = bench.measured_peaks()
    assert peak > 0 and kind in ("measured", "fallback")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_peaks() == (bench.FALLBACK_HBM_GBS, "fallback")
    assert bench.profiled_traffic() is None  # no profile file
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "sgemv_sparse_traffic.txt").write_text(
        "fingerprint: 0000\ndram_bytes_per_step_launch_avg: 123\n")
    monkeypatch.setattr(bench, "lib_fingerprint", lambda: "0000")
    assert bench.profiled_traffic() == 123.0
    monkeypatch.setattr(bench, "lib_fingerprint", lambda: "ffff")
    assert bench.profiled_traffic() is None  # kernel changed since the capture


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                        "--warmup", "3", "--cpu-seconds", "0.5"], capture_output=True, text=True, timeout=600,
                       env={**os.environ, "OMP_NUM_THREADS": "2"})
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
