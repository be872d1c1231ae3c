"""The quotient sequence the quantizing kernels use in place of a
per-element IEEE division (per-block correctly rounded reciprocal plus
Markstein corrections; see block_quotients in fp8q_device.cuh) equals
RN(x / s): exhaustively for bf16 dividends, by sampling for binary32
dividends (where Markstein's theorem is the proof), and exhaustively over
whole binades of binary32 dividends for the block scale RN(amax / Fmax),
whose divisor is one of two constants (block_scale in fp8q_device.cuh; the
ring hop passes it the binary32 amax of its fp32 sum)."""
import os
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def checker(tmp_path_factory):
    exe = str(tmp_path_factory.mktemp("fastdiv") / "check")
    subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-pthread", os.path.join(HERE, "fastdiv", "check.c"),
                    "-o", exe, "-lm"], check=True)
    return exe


def test_one_step_exact_for_every_bf16_and_scale_significand(checker):
    r = subprocess.run([checker, "bf16", str(max(1, os.cpu_count() or 1))], capture_output=True, text=True)
    assert "checked 1073741824 pairs, mismatches 0" in r.stdout, r.stdout
    assert r.returncode == 0


def test_two_step_exact_on_sampled_f32_dividends(checker):
    r = subprocess.run([checker, "f32", "30000000", "7"], capture_output=True, text=True)
    assert "mismatches 0" in r.stdout, r.stdout
    assert r.returncode == 0


def test_one_step_block_scale_exact_for_every_f32_amax_in_ten_binades(checker):
    # 2 maxima x 10 binades x 2^23 significands, from 2^-78 to 2^127
    r = subprocess.run([checker, "scale"], capture_output=True, text=True)
    assert "checked 167772160 dividends, mismatches 0" in r.stdout, r.stdout
    assert r.returncode == 0
