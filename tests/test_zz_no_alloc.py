"""fp8q_dequant_reduce_unfused_static: the unfused dequantize-then-sum with
the library's own static scratch, for callers that cannot allocate device
memory (an interception layer under a framework whose caching allocator
owns the GPU's memory, or a path where cudaMalloc would synchronize the
device).  Its results must equal those of fp8q_dequant_reduce_unfused,
which takes a caller-owned workspace, bit for bit, call after call, while
the shared scratch still holds the previous call's contents.

This file is collected last on purpose (a run that stops at the first
failure has then already run every other test), and it passes both alone
in a fresh process and after the rest of the suite: the first call on the
device does the one-time lookup of the scratch address.  Each call is
also checked against the oracle directly, one call sits exactly at the
scratch limit, and a call after the first leaves the device's free memory
unchanged."""
import ctypes

import numpy as np
import pytest
import torch

from test_gpu_reduce import random_shards

OK, ERR_SIZE = 0, 2
MAX_FLOATS = 1 << 22


@pytest.fixture(scope="module")
def L():
    import weight_transfer_gb300 as w
    return w.lib()


def _ptrs(ts):
    return (ctypes.c_void_p * len(ts))(*[t.data_ptr() for t in ts])


def _call_both(L, codes, scales, fmt):
    """Through the C ABI: the static-scratch entry point and the existing
    workspace entry point on the same inputs; returns both results."""
    k, n = len(codes), codes[0].size
    dc = [torch.from_numpy(c).cuda() for c in codes]
    ds = [torch.from_numpy(s).cuda() for s in scales]
    cp, sp = _ptrs(dc), _ptrs(ds)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    sb = torch.full((n,), -1, dtype=torch.int16, device="cuda")
    sf = torch.full((n,), float("nan"), dtype=torch.float32, device="cuda")
    st = L.fp8q_dequant_reduce_unfused_static(cp, sp, k, n, fmt, ctypes.c_void_p(sb.data_ptr()),
                                              ctypes.c_void_p(sf.data_ptr()), stream)
    assert st == OK
    ws = torch.empty(k * int(L.fp8q_unfused_stride(n)), dtype=torch.float32, device="cuda")
    wb = torch.full((n,), -1, dtype=torch.int16, device="cuda")
    wf = torch.full((n,), float("nan"), dtype=torch.float32, device="cuda")
    st = L.fp8q_dequant_reduce_unfused(cp, sp, k, n, fmt, ctypes.c_void_p(ws.data_ptr()),
                                       ctypes.c_void_p(wb.data_ptr()), ctypes.c_void_p(wf.data_ptr()), stream)
    assert st == OK
    torch.cuda.synchronize()
    return (sb.cpu().numpy(), sf.cpu().numpy()), (wb.cpu().numpy(), wf.cpu().numpy())


def _check_against_oracle_and_workspace(L, orc, k, n, fmt, seed):
    codes, scales = random_shards(k, n, fmt, seed=seed)
    (sb, sf), (wb, wf) = _call_both(L, codes, scales, fmt)
    assert np.array_equal(sf.view(np.uint32), wf.view(np.uint32)), f"fp32 differs (k={k}, n={n})"
    assert np.array_equal(sb, wb), f"bf16 differs (k={k}, n={n})"
    eb, ef = orc.dequant_reduce(codes, scales, fmt)
    assert np.array_equal(sf.view(np.uint32), ef.view(np.uint32)), f"fp32 differs from the oracle (k={k}, n={n})"
    assert np.array_equal(sb.view(np.uint16), eb), f"bf16 differs from the oracle (k={k}, n={n})"


@pytest.mark.gpu
def test_static_scratch_matches_workspace_entry_point_twice_in_a_row(L, orc):
    # call 1: 8 shards of 50,001 e4m3 values; call 2: 3 shards of 20,007
    # e5m2 values, so the second call finds the first call's data in the
    # scratch beyond and inside the region it uses; both against the
    # workspace entry point and the oracle
    for k, n, fmt, seed in [(8, 50_001, 0, 101), (3, 20_007, 1, 202)]:
        _check_against_oracle_and_workspace(L, orc, k, n, fmt, seed)


@pytest.mark.gpu
def test_static_scratch_call_exactly_at_its_limit(L, orc):
    # k * round_up(n, 4) == FP8Q_STATIC_SCRATCH_FLOATS: the largest call that fits
    k, n = 4, MAX_FLOATS // 4
    assert k * int(L.fp8q_unfused_stride(n)) == MAX_FLOATS
    _check_against_oracle_and_workspace(L, orc, k, n, 0, 303)


@pytest.mark.gpu
def test_static_scratch_call_allocates_no_device_memory(L):
    # after a first call (module load, scratch address lookup), another call
    # leaves the device's free memory exactly where it was
    k, n = 4, 100_000
    codes, scales = random_shards(k, n, 0, seed=404)
    dc = [torch.from_numpy(c).cuda() for c in codes]
    ds = [torch.from_numpy(s).cuda() for s in scales]
    cp, sp = _ptrs(dc), _ptrs(ds)
    ob = torch.empty((n,), dtype=torch.int16, device="cuda")
    of = torch.empty((n,), dtype=torch.float32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    def call():
        st = L.fp8q_dequant_reduce_unfused_static(cp, sp, k, n, 0, ctypes.c_void_p(ob.data_ptr()),
                                                  ctypes.c_void_p(of.data_ptr()), stream)
        torch.cuda.synchronize()
        return st
    assert call() == OK
    free_before, _ = torch.cuda.mem_get_info()
    assert call() == OK
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before


def test_static_scratch_rejects_sizes_beyond_its_limit(L):
    # checked on the host before anything touches the GPU: k * round_up(n, 4)
    # floats must fit in the static array
    c = (ctypes.c_void_p * 2)(0x7F0000000000, 0x7F0001000000)
    s = (ctypes.c_void_p * 2)(0x7F0002000000, 0x7F0003000000)
    n = MAX_FLOATS // 2 + 1
    st = L.fp8q_dequant_reduce_unfused_static(c, s, 2, n, 0, ctypes.c_void_p(0x7F1000000000),
                                              ctypes.c_void_p(0x7F2000000000), None)
    assert st == ERR_SIZE
    # one element past the largest call that fits (k = 4, n = MAX_FLOATS / 4)
    c4 = (ctypes.c_void_p * 4)(0x7F0000000000, 0x7F0001000000, 0x7F0002000000, 0x7F0003000000)
    s4 = (ctypes.c_void_p * 4)(0x7F0004000000, 0x7F0005000000, 0x7F0006000000, 0x7F0007000000)
    st = L.fp8q_dequant_reduce_unfused_static(c4, s4, 4, MAX_FLOATS // 4 + 1, 0, ctypes.c_void_p(0x7F1000000000),
                                              ctypes.c_void_p(0x7F2000000000), None)
    assert st == ERR_SIZE
