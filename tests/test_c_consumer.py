"""The C ABI from plain C: a small program (tests/c_abi/consumer.c) that
includes include/fp8q.h, links libfp8q.so and the CUDA runtime, and calls
the library with no Python or torch in between.  Without a GPU it checks the
argument validation; on the GPU it quantizes a file of bf16 values, and the
result is compared with the oracle."""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import gen
from conftest import ROOT, build_lib

CUDA = os.path.dirname(os.path.dirname(shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"))


@pytest.fixture(scope="module")
def consumer(tmp_path_factory):
    lib = build_lib()
    libdir = os.path.dirname(lib)
    exe = str(tmp_path_factory.mktemp("c_abi") / "consumer")
    cmd = ["gcc", "-O2", "-std=c11", os.path.join(ROOT, "tests", "c_abi", "consumer.c"), "-o", exe,
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
           "-L", libdir, "-lfp8q", "-L", os.path.join(CUDA, "lib64"), "-lcudart",
           f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        pytest.skip(f"cannot build the C consumer: {r.stderr[:300]}")
    return exe


def test_c_consumer_argument_checks(consumer):
    r = subprocess.run([consumer, "check"], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "check: ok" in r.stdout


@pytest.mark.gpu
@pytest.mark.parametrize("fmt", [0, 1])
def test_c_consumer_quantize_matches_oracle(consumer, orc, tmp_path, fmt):
    n = 8192 * 5 + 777
    x = gen.normal_bf16(n, 1e-3, seed=900 + fmt, outlier_p=1e-3, outlier_mult=100.0)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    (tmp_path / "in.bin").write_bytes(bits.tobytes())
    r = subprocess.run([consumer, "quantize", str(tmp_path / "in.bin"), str(tmp_path / "out.bin"), str(fmt)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    out = np.frombuffer((tmp_path / "out.bin").read_bytes(), np.uint8)
    ec, es = orc.quantize_blockwise(bits, fmt)
    assert np.array_equal(out[:n], ec)
    assert np.array_equal(out[n:].view(np.uint32), es.view(np.uint32))
