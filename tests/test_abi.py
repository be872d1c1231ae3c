"""The C ABI without a GPU: the library loads, exports every function that
include/*.h declares, and rejects bad arguments synchronously with the
documented status before anything is launched.

Every call here fails validation (or is an n == 0 no-op), so no CUDA work is
ever issued; fake device addresses are never dereferenced.
"""
import ctypes
import glob
import os
import re

import pytest

from conftest import ROOT, build_lib

OK, ERR_NULL, ERR_SIZE, ERR_ALIGN, ERR_FORMAT, ERR_K, ERR_CUDA, ERR_ALIAS, ERR_FLAGS = range(9)
A = 0x7F0000000000            # a 16-byte aligned fake device address
MB = 1 << 20


@pytest.fixture(scope="module")
def L():
    build_lib()
    import weight_transfer_gb300 as w
    return w.lib()


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M):
            if not m.group(0).lstrip().startswith(("typedef", "#", "struct")):
                names.add(m.group(1))
    return names


def test_exports_every_declared_function(L):
    names = declared_functions()
    expected = {"fp8q_quantize_blockwise", "fp8q_dequant_reduce", "fp8q_ring_hop", "mxfp8_quantize_swizzled",
                "fp8q_num_scales", "mxfp8_swizzled_scale_bytes", "fp8q_status_string"}
    assert expected <= names, names
    for n in sorted(names):
        assert hasattr(L, n), f"{n} is declared in include/ but not exported"


def test_status_strings(L):
    for s in range(9):
        assert len(L.fp8q_status_string(s)) > 0
    assert L.fp8q_status_string(0) == b"ok"
    assert L.fp8q_status_string(99) == b"unknown status"


def test_launch_overlap_switch(L):
    # host-only state: on by default, each call returns the previous setting
    prev = L.fp8q_set_launch_overlap(0)
    try:
        assert prev == 1
        assert L.fp8q_set_launch_overlap(7) == 0
        assert L.fp8q_set_launch_overlap(1) == 1
    finally:
        L.fp8q_set_launch_overlap(prev)


def test_size_helpers(L, orc):
    for n, nb in [(0, 0), (1, 1), (127, 1), (128, 1), (129, 2), (3_500_000_000, 27_343_750)]:
        assert L.fp8q_num_scales(n) == nb
    for b, m, k in [(1, 256, 256), (2, 129, 32), (128, 768, 2048), (1, 2048, 4096), (3, 1, 96)]:
        assert L.mxfp8_swizzled_scale_bytes(b, m, k) == orc.swizzled_scale_bytes(b, m, k)
    assert L.mxfp8_swizzled_scale_bytes(1, 128, 48) == 0


def test_quantize_validation(L):
    q = L.fp8q_quantize_blockwise
    assert q(A, 1024, 5, A + MB, A + 2 * MB, None) == ERR_FORMAT
    assert q(A, (1 << 42) + 1, 0, A + MB, A + 2 * MB, None) == ERR_SIZE
    assert q(None, 0, 0, None, None, None) == OK                      # empty: no-op
    assert q(None, 1024, 0, A + MB, A + 2 * MB, None) == ERR_NULL
    assert q(A, 1024, 0, None, A + 2 * MB, None) == ERR_NULL
    assert q(A + 2, 1024, 0, A + MB, A + 2 * MB, None) == ERR_ALIGN
    assert q(A, 1024, 0, A + MB + 8, A + 2 * MB, None) == ERR_ALIGN
    assert q(A, 1024, 0, A + 1024, A + 2 * MB, None) == ERR_ALIAS     # codes inside x
    assert q(A, 1024, 1, A + MB, A + MB + 512, None) == ERR_ALIAS     # scales inside codes


def _ptrs(vals):
    return (ctypes.c_void_p * len(vals))(*vals)


def test_dequant_reduce_validation(L):
    r = L.fp8q_dequant_reduce
    c = _ptrs([A + i * MB for i in range(17)])
    s = _ptrs([A + 64 * MB + i * MB for i in range(17)])
    ob, of = A + 200 * MB, A + 300 * MB
    assert r(c, s, 0, 1024, 0, ob, of, None) == ERR_K
    assert r(c, s, 17, 1024, 0, ob, of, None) == ERR_K
    assert r(c, s, 2, 1024, 3, ob, of, None) == ERR_FORMAT
    assert r(c, s, 2, 1024, 0, None, None, None) == ERR_NULL
    assert r(None, s, 2, 1024, 0, ob, of, None) == ERR_NULL
    assert r(_ptrs([A, 0]), s, 2, 1024, 0, ob, of, None) == ERR_NULL
    assert r(c, s, 2, 0, 0, ob, of, None) == OK
    assert r(_ptrs([A, A + MB + 4]), s, 2, 1024, 0, ob, of, None) == ERR_ALIGN
    assert r(c, s, 2, 1024, 0, ob + 2, of, None) == ERR_ALIGN
    assert r(c, s, 2, 1024, 0, c[1], None, None) == ERR_ALIAS         # output over shard 1 codes
    assert r(c, s, 2, 1024, 0, ob, ob + 1024, None) == ERR_ALIAS       # the two outputs overlap
    assert r(c, s, 2, 1 << 43, 0, ob, of, None) == ERR_SIZE


def test_ring_hop_validation(L):
    h = L.fp8q_ring_hop
    ic, isc, loc, oc, osc, ob = (A + i * MB for i in range(6))
    assert h(ic, isc, loc, 1024, 2, oc, osc, ob, None) == ERR_FORMAT
    assert h(ic, isc, None, 1024, 0, oc, osc, ob, None) == ERR_NULL
    assert h(ic, isc, loc, 1024, 0, None, osc, ob, None) == ERR_NULL
    assert h(ic, isc, loc + 4, 1024, 0, oc, osc, ob, None) == ERR_ALIGN
    assert h(ic, isc, loc, 1024, 0, ic, osc, ob, None) == ERR_ALIAS     # out codes over in codes
    assert h(ic, isc, loc, 1024, 0, oc, osc, oc, None) == ERR_ALIAS     # bf16 out over out codes
    assert h(ic, isc, loc, 1024, 0, oc, osc, loc + 16, None) == ERR_ALIAS  # partial overlap with local
    assert h(ic, isc, loc, 0, 0, oc, osc, ob, None) == OK


def test_mxfp8_validation(L):
    f = L.mxfp8_quantize_swizzled
    w, c, s = A, A + 64 * MB, A + 128 * MB
    assert f(w, 1, 128, 48, c, s, None) == ERR_K
    assert f(w, 1, 128, 0, c, s, None) == ERR_K
    assert f(w, 1, 128, -32, c, s, None) == ERR_K
    assert f(w, -1, 128, 64, c, s, None) == ERR_SIZE
    assert f(w, 1, -5, 64, c, s, None) == ERR_SIZE
    assert f(w, 0, 128, 64, c, s, None) == OK
    assert f(w, 1, 0, 64, c, s, None) == OK
    assert f(None, 1, 128, 64, c, s, None) == ERR_NULL
    assert f(w + 8, 1, 128, 64, c, s, None) == ERR_ALIGN
    assert f(w, 1, 128, 64, w + 64, s, None) == ERR_ALIAS
    assert f(w, 1 << 20, 1 << 20, 1 << 20, c, s, None) == ERR_SIZE


def test_other_entry_points_validation(L):
    assert L.fp8q_encode_f32(A, 100, 9, A + MB, None) == ERR_FORMAT
    assert L.fp8q_encode_f32(A, 100, 0, A + 192, None) == ERR_ALIAS
    assert L.fp8q_dequantize(A, A + MB, 100, 0, None, None, None) == ERR_NULL
    c = _ptrs([A, A + MB])
    s = _ptrs([A + 2 * MB, A + 3 * MB])
    assert L.fp8q_dequant_reduce_unfused(c, s, 2, 1024, 0, None, A + 4 * MB, None, None) == ERR_NULL
    assert L.fp8q_dequant_reduce_unfused(c, s, 2, 1024, 0, A + 4 * MB, A + 4 * MB, None, None) == ERR_ALIAS


def test_inputs_ready_flag_validation(L):
    import weight_transfer_gb300 as w
    # unknown flag bits are rejected first; the known flag passes the checks
    assert L.fp8q_quantize_blockwise_ex(A, 1024, 0, A + MB, A + 2 * MB, 2, None) == ERR_FLAGS
    assert L.fp8q_quantize_blockwise_ex(A, 0, 0, A + MB, A + 2 * MB, w.FP8Q_INPUTS_READY, None) == OK
    assert L.fp8q_quantize_blockwise_ex(A, 1024, 9, A + MB, A + 2 * MB, w.FP8Q_INPUTS_READY, None) == ERR_FORMAT
    c = _ptrs([A, A + MB])
    s = _ptrs([A + 2 * MB, A + 3 * MB])
    assert L.fp8q_dequant_reduce_ex(c, s, 2, 1024, 0, A + 4 * MB, None, 4, None) == ERR_FLAGS
    assert L.fp8q_dequant_reduce_ex(c, s, 2, 0, 0, A + 4 * MB, None, w.FP8Q_INPUTS_READY, None) == OK
    T = w.mxfp8_tensor_t
    ok = (T * 1)(T(A, 1, 128, 64, A + MB, A + 2 * MB))
    assert L.mxfp8_quantize_swizzled_group_ex(ok, 1, 8, None) == ERR_FLAGS
    assert L.mxfp8_quantize_swizzled_group_ex(ok, 0, w.FP8Q_INPUTS_READY, None) == ERR_SIZE


def test_quantize_group_validation(L):
    import weight_transfer_gb300 as w
    Q = w.fp8q_quant_t
    g = L.fp8q_quantize_blockwise_group
    ok = Q(A, 1024, A + MB, A + 2 * MB)
    arr = (Q * 17)(*([ok] * 17))
    assert g(arr, 0, 0, 0, None) == ERR_SIZE
    assert g(arr, 17, 0, 0, None) == ERR_SIZE
    assert g(arr, 1, 9, 0, None) == ERR_FORMAT
    assert g(arr, 1, 0, 2, None) == ERR_FLAGS
    assert g(None, 1, 0, 0, None) == ERR_NULL
    # item 1 writes its codes over item 0's input
    alias = (Q * 2)(ok, Q(A + 10 * MB, 1024, A + 512, A + 12 * MB))
    assert g(alias, 2, 0, 0, None) == ERR_ALIAS
    # two items writing the same scales
    same = (Q * 2)(ok, Q(A + 10 * MB, 1024, A + 11 * MB, A + 2 * MB))
    assert g(same, 2, 0, 0, None) == ERR_ALIAS
    bad = (Q * 2)(ok, Q(A + 10 * MB + 8, 1024, A + 11 * MB, A + 12 * MB))
    assert g(bad, 2, 0, 0, None) == ERR_ALIGN
    empty = (Q * 2)(Q(None, 0, None, None), Q(None, 0, None, None))
    assert g(empty, 2, 0, w.FP8Q_INPUTS_READY, None) == OK


def test_mxfp8_dequantize_tile_count_limit(L):
    # 2^32 + 5 one-row matrices of k = 32: n stays below the element limit,
    # but the tile count does not fit the kernel's 32-bit tile index
    G = 1 << 42                   # address spacing: the scale buffer alone is 2 TiB
    batch = (1 << 32) + 5
    assert L.mxfp8_dequantize_swizzled(A, A + G, batch, 1, 32, A + 2 * G, None) == ERR_SIZE
    assert L.mxfp8_dequantize_swizzled(A, A + G, 4, 1, 48, A + 2 * G, None) == ERR_K
    assert L.mxfp8_dequantize_swizzled(A, A + G, 0, 1, 32, A + 2 * G, None) == OK


def test_binding_rejects_cpu_tensors():
    import torch
    import weight_transfer_gb300 as w
    with pytest.raises(ValueError):
        w.fp8q_quantize_blockwise(torch.zeros(256, dtype=torch.bfloat16),
                                  codes=torch.zeros(1), scales=torch.zeros(1))


def test_mxfp8_group_validation(L):
    import weight_transfer_gb300 as w
    T = w.mxfp8_tensor_t
    f = L.mxfp8_quantize_swizzled_group
    ok = T(A, 1, 128, 64, A + 64 * MB, A + 128 * MB)
    arr = (T * 17)(*([ok] * 17))
    assert f(arr, 0, None) == ERR_SIZE
    assert f(arr, 17, None) == ERR_SIZE
    assert f(None, 1, None) == ERR_NULL
    bad_k = (T * 2)(ok, T(A + 200 * MB, 1, 128, 48, A + 264 * MB, A + 328 * MB))
    assert f(bad_k, 2, None) == ERR_K
    # tensor 1 writes its codes over tensor 0's input
    alias = (T * 2)(ok, T(A + 200 * MB, 1, 128, 64, A + 1024, A + 328 * MB))
    assert f(alias, 2, None) == ERR_ALIAS
    empty = (T * 2)(T(None, 0, 128, 64, None, None), T(None, 1, 0, 64, None, None))
    assert f(empty, 2, None) == OK


def test_ring_group_and_allreduce_validation(L):
    import weight_transfer_gb300 as w
    H = w.fp8q_hop_t
    g = L.fp8q_ring_hop_group
    ok = H(A, A + MB, A + 2 * MB, 1024, A + 3 * MB, A + 4 * MB, None)
    arr = (H * 17)(*([ok] * 17))
    assert g(arr, 0, 0, None) == ERR_SIZE
    assert g(arr, 17, 0, None) == ERR_SIZE
    assert g(arr, 1, 9, None) == ERR_FORMAT
    # two hops writing the same output codes
    two = (H * 2)(ok, H(A + 10 * MB, A + 11 * MB, A + 12 * MB, 1024, A + 3 * MB, A + 14 * MB, None))
    assert g(two, 2, 0, None) == ERR_ALIAS
    empty = (H * 1)(H(None, None, None, 0, None, None, None))
    assert g(empty, 1, 0, None) == OK
    gx = L.fp8q_ring_hop_group_ex
    assert gx(arr, 1, 0, 2, None) == ERR_FLAGS                      # unknown flag bit, checked first
    assert gx(arr, 1, 0, 0x80000001, None) == ERR_FLAGS
    assert gx(two, 2, 0, w.FP8Q_HOP_LOCAL_READY, None) == ERR_ALIAS
    assert gx(empty, 1, 0, w.FP8Q_HOP_LOCAL_READY, None) == OK
    assert L.fp8q_ring_allreduce_workspace_bytes(8, 13_107_200) > 0
    assert L.fp8q_ring_allreduce_workspace_bytes(8, 1000) == 0
    assert L.fp8q_ring_allreduce_workspace_bytes(1, 1024) == 0
    pp = (ctypes.c_void_p * 2)(A, A + 10 * MB)
    rp = (ctypes.c_void_p * 2)(A + 20 * MB, A + 30 * MB)
    r = L.fp8q_ring_allreduce_sim
    assert r(pp, rp, 1, 1024, 0, A + 40 * MB, 1 << 20, None, None) == ERR_K
    assert r(pp, rp, 2, 1000, 0, A + 40 * MB, 1 << 20, None, None) == ERR_SIZE
    assert r(pp, rp, 2, 1024, 0, A + 40 * MB, 16, None, None) == ERR_SIZE       # workspace too small
    assert r(pp, rp, 2, 0, 0, None, 0, None, None) == OK
    rx = L.fp8q_ring_allreduce_sim_ex
    assert rx(pp, rp, 2, 1024, 0, A + 40 * MB, 1 << 20, None, 2, None) == ERR_FLAGS      # unknown flag bit
    assert rx(pp, rp, 2, 1024, 9, A + 40 * MB, 1 << 20, None, w.FP8Q_ALLREDUCE_MEAN, None) == ERR_FORMAT
    assert rx(pp, rp, 1, 1024, 0, A + 40 * MB, 1 << 20, None, w.FP8Q_ALLREDUCE_MEAN, None) == ERR_K
    assert rx(pp, rp, 2, 0, 0, None, 0, None, w.FP8Q_ALLREDUCE_MEAN, None) == OK
    # results of two ranks in one place
    same = (ctypes.c_void_p * 2)(A + 20 * MB, A + 20 * MB)
    assert rx(pp, same, 2, 1024, 0, A + 40 * MB, 1 << 20, None, w.FP8Q_ALLREDUCE_MEAN, None) == ERR_ALIAS


def test_selftest_copy_wait_validation(L):
    t = L.fp8q_selftest_copy_wait
    assert t(None, None, 999_999, None) == ERR_SIZE                 # below 1 ms
    assert t(None, None, 2_000_000_001, None) == ERR_SIZE           # above the kernels' own 2 s
    assert t(A, None, 10_000_000, None) == ERR_NULL                  # src without dst
    assert t(None, A, 10_000_000, None) == ERR_NULL
    assert t(A + 8, A + MB, 10_000_000, None) == ERR_ALIGN
    assert t(A, A, 10_000_000, None) == ERR_ALIAS


def test_gather_decode_validation(L):
    gd = L.fp8q_gather_decode
    outs = (ctypes.c_void_p * 2)(A + 8 * MB, A + 16 * MB)
    assert gd(A, A + MB, 4096, 0, outs, 2, 2, None) == ERR_FLAGS
    assert gd(A, A + MB, 4096, 0, outs, 0, 0, None) == ERR_K
    assert gd(A, A + MB, 4096, 0, outs, 17, 0, None) == ERR_K
    assert gd(A, A + MB, 4096, 7, outs, 2, 0, None) == ERR_FORMAT
    assert gd(None, A + MB, 4096, 0, outs, 2, 0, None) == ERR_NULL
    assert gd(A + 4, A + MB, 4096, 0, outs, 2, 0, None) == ERR_ALIGN
    same = (ctypes.c_void_p * 2)(A + 8 * MB, A + 8 * MB + 4096)
    assert gd(A, A + MB, 4096, 0, same, 2, 0, None) == ERR_ALIAS
    over_in = (ctypes.c_void_p * 1)(A)
    assert gd(A, A + MB, 4096, 0, over_in, 1, 0, None) == ERR_ALIAS
    assert gd(None, None, 0, 0, outs, 2, 0, None) == OK                 # empty: no-op
