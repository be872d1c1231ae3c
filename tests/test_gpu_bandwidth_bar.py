"""The bandwidth bar of the hot path: each of the four kernels moves its
algorithmic bytes at no less than 70% of the GPU's HBM copy peak for
payloads of 64 MiB and more (the measured copy rate of the GB300s
when MEASURED_PEAKS.json is present, else 6.8 TB/s).  Times are CUDA-event
medians of 10 launches, L2 flushed before each; the bench reports the exact
figures, this test only guards the bar."""
import ctypes
import json
import os

import pytest
import torch

from conftest import ROOT

pytestmark = pytest.mark.gpu

BAR = 0.70


def peak_gbs():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"])
    except (OSError, KeyError, ValueError):
        return 6800.0


@pytest.fixture(scope="module")
def w():
    import weight_transfer_gb300 as w
    return w


@pytest.fixture(scope="module")
def flush():
    a = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    b = torch.zeros(64 << 20, dtype=torch.float32, device="cuda")

    def f():
        a.fill_(1)
        b.sum()
    return f


def median_ms(fn, flush, reps=10):
    fn()
    ts = []
    for _ in range(reps):
        flush()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        fn()
        e.record()
        torch.cuda.synchronize()
        ts.append(s.elapsed_time(e))
    return sorted(ts)[len(ts) // 2]


def assert_bar(what, nbytes, ms):
    gbs = nbytes / (ms * 1e-3) / 1e9
    assert gbs >= BAR * peak_gbs(), f"{what}: {gbs:.0f} GB/s is below {BAR:.0%} of {peak_gbs():.0f} GB/s"


N64 = (64 << 20) // 2                       # 64 MiB of bf16


def nsc(n):
    return (n + 127) // 128


def test_quantize_64mib(w, flush):
    x = torch.randn(N64, device="cuda").mul_(1e-4).to(torch.bfloat16)
    c = torch.empty(N64, dtype=torch.uint8, device="cuda")
    s = torch.empty(nsc(N64), dtype=torch.float32, device="cuda")
    ms = median_ms(lambda: w.fp8q_quantize_blockwise(x, "e4m3", codes=c, scales=s), flush)
    assert_bar("quantize", 3 * N64 + 4 * nsc(N64), ms)


def test_fused_reduce_k8_64mib_shards(w, flush):
    k = 8
    cs, ss = [], []
    for r in range(k):
        c, s = w.fp8q_quantize_blockwise(torch.randn(N64, device="cuda").mul_(1e-4).to(torch.bfloat16), "e4m3")
        cs.append(c)
        ss.append(s)
    ob = torch.empty(N64, dtype=torch.bfloat16, device="cuda")
    of = torch.empty(N64, dtype=torch.float32, device="cuda")
    ms = median_ms(lambda: w.fp8q_dequant_reduce(cs, ss, "e4m3", out_bf16=ob, out_fp32=of), flush)
    assert_bar("fused reduce", k * (N64 + 4 * nsc(N64)) + 6 * N64, ms)


def test_ring_hop_64mib(w, flush):
    c, s = w.fp8q_quantize_blockwise(torch.randn(N64, device="cuda").mul_(1e-3).to(torch.bfloat16), "e4m3")
    loc = torch.randn(N64, device="cuda").mul_(1e-3).to(torch.bfloat16)
    oc = torch.empty(N64, dtype=torch.uint8, device="cuda")
    os_ = torch.empty(nsc(N64), dtype=torch.float32, device="cuda")
    ob = torch.empty(N64, dtype=torch.bfloat16, device="cuda")
    ms = median_ms(lambda: w.fp8q_ring_hop(c, s, loc, "e4m3", want_bf16=True, out_codes=oc, out_scales=os_,
                                           out_bf16=ob), flush)
    assert_bar("ring hop", 2 * (N64 + 4 * nsc(N64)) + 2 * N64 + 2 * N64, ms)


def test_mxfp8_expert_batch(w, flush):
    b, m, k = 128, 768, 2048                 # 402 MB of bf16: one expert tensor of the stack
    x = torch.randn((b, m, k), device="cuda").mul_(0.02).to(torch.bfloat16)
    c = torch.empty((b, m, k), dtype=torch.uint8, device="cuda")
    sb = w.mxfp8_swizzled_scale_bytes(b, m, k)
    s = torch.empty(sb, dtype=torch.uint8, device="cuda")
    ms = median_ms(lambda: w.mxfp8_quantize_swizzled(x, codes=c, scales_swizzled=s), flush)
    assert_bar("MXFP8", 3 * b * m * k + sb, ms)
