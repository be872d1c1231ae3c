"""The optional NVTX ranges: off by default (the macro expands to nothing),
and the sources compile with them switched on (FP8Q_NVTX)."""
import os
import shutil
import subprocess

import pytest

from conftest import ROOT

CSRC = os.path.join(ROOT, "weight_transfer_gb300", "csrc")


def _nvcc():
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        pytest.skip("nvcc not available")
    return path


@pytest.mark.parametrize("define", [None, "-DFP8Q_NVTX=1"])
def test_entry_points_compile_with_and_without_nvtx(tmp_path, define):
    # the AllReduce scheduler: host code only, with two instrumented entry points
    cmd = [_nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-std=c++17", "-Xcompiler", "-fPIC",
           "-I", os.path.join(ROOT, "include"), "-I", CSRC, "-c", os.path.join(CSRC, "ring_allreduce.cu"),
           "-o", str(tmp_path / "ra.o")]
    if define:
        cmd.insert(1, define)
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    nm = subprocess.run(["nm", "-C", str(tmp_path / "ra.o")], capture_output=True, text=True).stdout
    assert ("nvtx" in nm.lower()) == bool(define)


def test_build_script_reads_the_switch(monkeypatch):
    import importlib.util
    spec = importlib.util.spec_from_file_location("_b", os.path.join(ROOT, "weight_transfer_gb300", "build.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    monkeypatch.delenv("FP8Q_NVTX", raising=False)
    assert not b.nvtx_requested()
    monkeypatch.setenv("FP8Q_NVTX", "1")
    assert b.nvtx_requested()
