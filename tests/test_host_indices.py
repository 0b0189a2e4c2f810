"""Index arithmetic of the GEMV kernels, checked on the host (no GPU): tests/host/gemv_indices.cu is
compiled against the library's planner and load cursors and walks every CTA, pass, x tile, warp and lane
of many layer shapes (see its header for the list of checks)."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "int4_weight_only_sgemv_gb300", "csrc")


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    return None


def test_gemv_load_addresses_and_coverage(tmp_path):
    nvcc = _nvcc()
    if nvcc is None:
        pytest.skip("nvcc not found")
    exe = str(tmp_path / "gemv_indices")
    cmd = [nvcc, "-std=c++17", "-O1", "-gencode", "arch=compute_103a,code=sm_103a", "-I", os.path.join(ROOT, "include"),
           "-I", CSRC, os.path.join(ROOT, "tests", "host", "gemv_indices.cu"), os.path.join(CSRC, "abi.cu"),
           os.path.join(ROOT, "tests", "host", "stub_launchers.cu"), "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-4000:]
    assert " 0 failures" in r.stdout, r.stdout[-4000:]


def test_stream_load_addresses_and_coverage(tmp_path):
    """The streaming kernel's planner, unit cursor and addresses (tests/host/stream_indices.cu)."""
    nvcc = _nvcc()
    if nvcc is None:
        pytest.skip("nvcc not found")
    exe = str(tmp_path / "stream_indices")
    cmd = [nvcc, "-std=c++17", "-O1", "-gencode", "arch=compute_103a,code=sm_103a", "-I", os.path.join(ROOT, "include"),
           "-I", CSRC, os.path.join(ROOT, "tests", "host", "stream_indices.cu"), os.path.join(CSRC, "abi.cu"),
           os.path.join(ROOT, "tests", "host", "stub_launchers.cu"), "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-4000:]
    assert " 0 failures" in r.stdout, r.stdout[-4000:]
