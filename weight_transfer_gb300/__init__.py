"""weight_transfer_gb300 -- FP8 / MXFP8 transfer codec for GB300 (sm_103a).

Thin Python binding of ``libfp8q.so`` (C ABI declared in ``include/fp8q.h``).
The functions carry the C names; each one only marshals torch CUDA tensors
into device pointers, sizes and the current CUDA stream, calls the library,
and raises ``Fp8qError`` on a non-zero status.  All arithmetic runs in the
library's CUDA kernels; there is no CPU path.  Outputs may be passed in
(reused, caller-owned buffers) or are allocated with torch when omitted.

Importing the package loads the library and fails loudly if it has not been
built (``python weight_transfer_gb300/build.py`` or ``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfp8q.so")

FP8Q_E4M3 = 0
FP8Q_E5M2 = 1
FORMATS = {"e4m3": FP8Q_E4M3, "e5m2": FP8Q_E5M2}
FP8Q_MAX_SHARDS = 16
FP8Q_BLOCK = 128
MXFP8_BLOCK = 32

STATUS = {0: "FP8Q_OK", 1: "FP8Q_ERR_NULL", 2: "FP8Q_ERR_SIZE", 3: "FP8Q_ERR_ALIGN", 4: "FP8Q_ERR_FORMAT",
          5: "FP8Q_ERR_K", 6: "FP8Q_ERR_CUDA", 7: "FP8Q_ERR_ALIAS"}


class Fp8qError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str, cuda_error: int = 0):
        self.status = status
        self.cuda_error = cuda_error
        extra = f" (cudaError {cuda_error})" if status == 6 else ""
        super().__init__(f"{fn}: {STATUS.get(status, status)}: {msg}{extra}")


_vp = ctypes.c_void_p
_sz = ctypes.c_size_t
_i64 = ctypes.c_int64
_int = ctypes.c_int


class fp8q_hop_t(ctypes.Structure):
    """One hop of fp8q_ring_hop_group (same layout as the C struct)."""
    _fields_ = [("in_codes", ctypes.c_void_p), ("in_scales", ctypes.c_void_p), ("local_bf16", ctypes.c_void_p),
                ("n", ctypes.c_size_t), ("out_codes", ctypes.c_void_p), ("out_scales", ctypes.c_void_p),
                ("out_bf16", ctypes.c_void_p)]


FP8Q_MAX_HOP_GROUP = 16


class fp8q_quant_t(ctypes.Structure):
    """One item of fp8q_quantize_blockwise_group (same layout as the C struct)."""
    _fields_ = [("x_bf16", ctypes.c_void_p), ("n", ctypes.c_size_t), ("codes", ctypes.c_void_p),
                ("scales", ctypes.c_void_p)]


FP8Q_MAX_QUANT_GROUP = 16
FP8Q_HOP_LOCAL_READY = 1
FP8Q_INPUTS_READY = 1
FP8Q_ALLREDUCE_MEAN = 1
FP8Q_DEVICE_ERR_COPY_TIMEOUT = 1


class mxfp8_tensor_t(ctypes.Structure):
    """One tensor of mxfp8_quantize_swizzled_group (same layout as the C struct)."""
    _fields_ = [("w_bf16", _vp), ("batch", _i64), ("m", _i64), ("k", _i64), ("codes", _vp),
                ("scales_swizzled", _vp)]


MXFP8_MAX_GROUP = 16


class fp8q_pack_item_t(ctypes.Structure):
    _fields_ = [("codes_bytes", ctypes.c_uint64), ("scales_bytes", ctypes.c_uint64)]


class fp8q_pack_slot_t(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("codes_offset", ctypes.c_uint64), ("scales_offset", ctypes.c_uint64)]


class fp8q_copy_t(ctypes.Structure):
    _fields_ = [("src", ctypes.c_void_p), ("dst", ctypes.c_void_p), ("bytes", ctypes.c_uint64)]


FP8Q_MAX_COPY_SEGMENTS = 96

# name -> (argtypes, restype)
_SIGNATURES = {
    "fp8q_quantize_blockwise": ([_vp, _sz, _int, _vp, _vp, _vp], _int),
    "fp8q_dequant_reduce": ([ctypes.POINTER(_vp), ctypes.POINTER(_vp), _int, _sz, _int, _vp, _vp, _vp], _int),
    "fp8q_ring_hop": ([_vp, _vp, _vp, _sz, _int, _vp, _vp, _vp, _vp], _int),
    "mxfp8_quantize_swizzled": ([_vp, _i64, _i64, _i64, _vp, _vp, _vp], _int),
    "mxfp8_quantize_swizzled_group": ([ctypes.POINTER(mxfp8_tensor_t), _int, _vp], _int),
    "mxfp8_dequantize_swizzled": ([_vp, _vp, _i64, _i64, _i64, _vp, _vp], _int),
    "mxfp8_unswizzle_scales": ([_vp, _i64, _i64, _i64, _vp, _vp], _int),
    "fp8q_count_mismatches": ([_vp, _vp, _sz, _vp, _vp], _int),
    "fp8q_quantize_tensorwise": ([_vp, _sz, _int, _vp, _vp, _vp], _int),
    "fp8q_ring_hop_bf16_requant": ([_vp, _vp, _vp, _sz, _int, _vp, _vp, _vp, _vp], _int),
    "fp8q_pack_plan": ([ctypes.POINTER(fp8q_pack_item_t), _int, ctypes.c_uint64, ctypes.POINTER(fp8q_pack_slot_t),
                        ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(_int)], _int),
    "fp8q_copy_segments": ([ctypes.POINTER(fp8q_copy_t), _int, _vp], _int),
    "fp8q_ring_hop_group": ([ctypes.POINTER(fp8q_hop_t), _int, _int, _vp], _int),
    "fp8q_ring_hop_group_ex": ([ctypes.POINTER(fp8q_hop_t), _int, _int, ctypes.c_uint, _vp], _int),
    "fp8q_quantize_blockwise_ex": ([_vp, _sz, _int, _vp, _vp, ctypes.c_uint, _vp], _int),
    "fp8q_quantize_blockwise_group": ([ctypes.POINTER(fp8q_quant_t), _int, _int, ctypes.c_uint, _vp], _int),
    "fp8q_dequant_reduce_ex": ([ctypes.POINTER(_vp), ctypes.POINTER(_vp), _int, _sz, _int, _vp, _vp, ctypes.c_uint,
                                _vp], _int),
    "mxfp8_quantize_swizzled_group_ex": ([ctypes.POINTER(mxfp8_tensor_t), _int, ctypes.c_uint, _vp], _int),
    "fp8q_ring_allreduce_workspace_bytes": ([_int, _sz], _sz),
    "fp8q_ring_allreduce_sim": ([ctypes.POINTER(_vp), ctypes.POINTER(_vp), _int, _sz, _int, _vp, _sz,
                                 ctypes.POINTER(ctypes.c_uint64), _vp], _int),
    "fp8q_ring_allreduce_sim_ex": ([ctypes.POINTER(_vp), ctypes.POINTER(_vp), _int, _sz, _int, _vp, _sz,
                                    ctypes.POINTER(ctypes.c_uint64), ctypes.c_uint, _vp], _int),
    "fp8q_num_scales": ([_sz], _sz),
    "mxfp8_swizzled_scale_bytes": ([_i64, _i64, _i64], _sz),
    "fp8q_status_string": ([_int], ctypes.c_char_p),
    "fp8q_last_cuda_error": ([], _int),
    "fp8q_set_launch_overlap": ([_int], _int),
    "fp8q_device_errors": ([ctypes.POINTER(ctypes.c_uint), _int], _int),
    "fp8q_selftest_copy_wait": ([_vp, _vp, ctypes.c_uint64, _vp], _int),
    "fp8q_gather_decode": ([_vp, _vp, _sz, _int, ctypes.POINTER(_vp), _int, ctypes.c_uint, _vp], _int),
    "fp8q_encode_f32": ([_vp, _sz, _int, _vp, _vp], _int),
    "fp8q_dequantize": ([_vp, _vp, _sz, _int, _vp, _vp, _vp], _int),
    "fp8q_unfused_stride": ([_sz], _sz),
    "fp8q_dequant_reduce_unfused_static": ([ctypes.POINTER(_vp), ctypes.POINTER(_vp), _int, _sz, _int, _vp, _vp, _vp],
                                           _int),
    "fp8q_dequant_reduce_unfused": ([ctypes.POINTER(_vp), ctypes.POINTER(_vp), _int, _sz, _int, _vp, _vp, _vp, _vp],
                                    _int),
}

_lib: Optional[ctypes.CDLL] = None


def lib() -> ctypes.CDLL:
    """The loaded C library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with `python weight_transfer_gb300/build.py`; "
                              "this package has no CPU fallback")
        L = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


lib()   # fail at import, not at the first call


def _check(fn: str, status: int) -> None:
    if status != 0:
        L = lib()
        raise Fp8qError(fn, status, L.fp8q_status_string(status).decode(), L.fp8q_last_cuda_error())


def _fmt(fmt) -> int:
    if isinstance(fmt, str):
        return FORMATS[fmt]
    return int(fmt)


def _dev(t: Optional[torch.Tensor], what: str, dtype=None, numel: Optional[int] = None) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{what} must be {dtype}, got {t.dtype}")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{what} holds {t.numel()} elements, needs {numel}")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def fp8q_device_errors(clear: bool = True) -> int:
    """Synchronizes the device and returns the kernels' error bits (0 = none)."""
    v = ctypes.c_uint(0)
    _check("fp8q_device_errors", lib().fp8q_device_errors(ctypes.byref(v), int(clear)))
    return int(v.value)


def fp8q_selftest_copy_wait(limit_ns: int, src: Optional[torch.Tensor] = None, dst: Optional[torch.Tensor] = None,
                            stream=None) -> None:
    """Test hook of the kernels' bounded copy wait: with no src/dst the wait
    runs out after limit_ns and raises FP8Q_DEVICE_ERR_COPY_TIMEOUT (read it
    with fp8q_device_errors); with 16-byte src/dst buffers the copy lands and
    src's 16 bytes are written to dst."""
    st = lib().fp8q_selftest_copy_wait(_dev(src, "src", numel=None), _dev(dst, "dst", numel=None), int(limit_ns),
                                       _stream(stream))
    _check("fp8q_selftest_copy_wait", st)


def fp8q_set_launch_overlap(enable: bool) -> bool:
    """Switches programmatic dependent launch for every later launch of the
    library (on by default); returns the previous setting."""
    return bool(lib().fp8q_set_launch_overlap(1 if enable else 0))


def fp8q_num_scales(n: int) -> int:
    return int(lib().fp8q_num_scales(n))


def mxfp8_swizzled_scale_bytes(batch: int, m: int, k: int) -> int:
    return int(lib().mxfp8_swizzled_scale_bytes(batch, m, k))


def fp8q_quantize_blockwise(x: torch.Tensor, fmt="e4m3", codes: Optional[torch.Tensor] = None,
                            scales: Optional[torch.Tensor] = None, stream=None, flags: int = 0):
    """bf16 x -> (codes uint8 [n], scales float32 [ceil(n/128)])."""
    n = x.numel()
    if codes is None:
        codes = torch.empty(n, dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty(max(fp8q_num_scales(n), 1), dtype=torch.float32, device=x.device)
    st = lib().fp8q_quantize_blockwise_ex(_dev(x, "x", torch.bfloat16), n, _fmt(fmt),
                                          _dev(codes, "codes", torch.uint8, n),
                                          _dev(scales, "scales", torch.float32, fp8q_num_scales(n)), flags,
                                          _stream(stream))
    _check("fp8q_quantize_blockwise_ex" if flags else "fp8q_quantize_blockwise", st)
    return codes, scales


def fp8q_quantize_blockwise_ex(x: torch.Tensor, fmt="e4m3", flags: int = 0, codes: Optional[torch.Tensor] = None,
                               scales: Optional[torch.Tensor] = None, stream=None):
    """fp8q_quantize_blockwise with flags (FP8Q_INPUTS_READY)."""
    return fp8q_quantize_blockwise(x, fmt, codes=codes, scales=scales, stream=stream, flags=flags)


def fp8q_quantize_blockwise_group(xs: Sequence[torch.Tensor], fmt="e4m3", flags: int = 0,
                                  codes: Optional[Sequence[torch.Tensor]] = None,
                                  scales: Optional[Sequence[torch.Tensor]] = None, stream=None):
    """Several bf16 arrays quantized blockwise in one launch -> (list of
    codes, list of scales), as one fp8q_quantize_blockwise per array would give."""
    count = len(xs)
    arr = (fp8q_quant_t * max(count, 1))()
    outc, outs = [], []
    for i, x in enumerate(xs):
        n = x.numel()
        c = codes[i] if codes is not None else torch.empty(n, dtype=torch.uint8, device=x.device)
        sc = scales[i] if scales is not None else torch.empty(max(fp8q_num_scales(n), 1), dtype=torch.float32,
                                                              device=x.device)
        arr[i] = fp8q_quant_t(_dev(x, f"xs[{i}]", torch.bfloat16), n, _dev(c, f"codes[{i}]", torch.uint8, n),
                              _dev(sc, f"scales[{i}]", torch.float32, fp8q_num_scales(n)))
        outc.append(c)
        outs.append(sc)
    _check("fp8q_quantize_blockwise_group",
           lib().fp8q_quantize_blockwise_group(arr, count, _fmt(fmt), flags, _stream(stream)))
    return outc, outs


def _ptr_array(ts: Sequence[torch.Tensor], what: str, dtype, numel: int):
    arr = (_vp * len(ts))()
    for i, t in enumerate(ts):
        arr[i] = _dev(t, f"{what}[{i}]", dtype, numel)
    return arr


def fp8q_dequant_reduce(codes: Sequence[torch.Tensor], scales: Sequence[torch.Tensor], fmt="e4m3",
                        out_bf16: Optional[torch.Tensor] = None, out_fp32: Optional[torch.Tensor] = None,
                        want_bf16: bool = True, want_fp32: bool = True, n: Optional[int] = None, stream=None,
                        flags: int = 0):
    """Sum of k FP8 shards in rank order -> (bf16 [n] or None, fp32 [n] or None)."""
    k = len(codes)
    if k != len(scales):
        raise ValueError("codes and scales must have the same length")
    if n is None:
        n = codes[0].numel()
    dev = codes[0].device
    if out_bf16 is None and want_bf16:
        out_bf16 = torch.empty(n, dtype=torch.bfloat16, device=dev)
    if out_fp32 is None and want_fp32:
        out_fp32 = torch.empty(n, dtype=torch.float32, device=dev)
    cp = _ptr_array(codes, "codes", torch.uint8, n)
    sp = _ptr_array(scales, "scales", torch.float32, fp8q_num_scales(n))
    st = lib().fp8q_dequant_reduce_ex(cp, sp, k, n, _fmt(fmt), _dev(out_bf16, "out_bf16", torch.bfloat16, n),
                                      _dev(out_fp32, "out_fp32", torch.float32, n), flags, _stream(stream))
    _check("fp8q_dequant_reduce_ex" if flags else "fp8q_dequant_reduce", st)
    return out_bf16, out_fp32


def fp8q_dequant_reduce_ex(codes: Sequence[torch.Tensor], scales: Sequence[torch.Tensor], fmt="e4m3", flags: int = 0,
                           **kw):
    """fp8q_dequant_reduce with flags (FP8Q_INPUTS_READY); keyword arguments as fp8q_dequant_reduce."""
    return fp8q_dequant_reduce(codes, scales, fmt, flags=flags, **kw)


def fp8q_ring_hop(in_codes: torch.Tensor, in_scales: torch.Tensor, local: torch.Tensor, fmt="e4m3",
                  out_codes: Optional[torch.Tensor] = None, out_scales: Optional[torch.Tensor] = None,
                  out_bf16: Optional[torch.Tensor] = None, want_bf16: bool = False, stream=None):
    """-> (out_codes, out_scales, out_bf16 or None).  out_bf16 may be `local` (in place)."""
    n = local.numel()
    dev = local.device
    if out_codes is None:
        out_codes = torch.empty(n, dtype=torch.uint8, device=dev)
    if out_scales is None:
        out_scales = torch.empty(max(fp8q_num_scales(n), 1), dtype=torch.float32, device=dev)
    if out_bf16 is None and want_bf16:
        out_bf16 = torch.empty(n, dtype=torch.bfloat16, device=dev)
    nb = fp8q_num_scales(n)
    st = lib().fp8q_ring_hop(_dev(in_codes, "in_codes", torch.uint8, n), _dev(in_scales, "in_scales", torch.float32, nb),
                             _dev(local, "local", torch.bfloat16), n, _fmt(fmt),
                             _dev(out_codes, "out_codes", torch.uint8, n),
                             _dev(out_scales, "out_scales", torch.float32, nb),
                             _dev(out_bf16, "out_bf16", torch.bfloat16, n), _stream(stream))
    _check("fp8q_ring_hop", st)
    return out_codes, out_scales, out_bf16


def mxfp8_quantize_swizzled(w: torch.Tensor, codes: Optional[torch.Tensor] = None,
                            scales_swizzled: Optional[torch.Tensor] = None, stream=None):
    """bf16 w [m, k] or [batch, m, k] -> (E4M3 codes uint8 same shape, swizzled E8M0 bytes uint8)."""
    if w.dim() == 2:
        batch, (m, k) = 1, w.shape
    elif w.dim() == 3:
        batch, m, k = w.shape
    else:
        raise ValueError("w must be 2D [m, k] or 3D [batch, m, k]")
    dev = w.device
    sb = mxfp8_swizzled_scale_bytes(batch, m, k)
    if codes is None:
        codes = torch.empty(w.shape, dtype=torch.uint8, device=dev)
    if scales_swizzled is None:
        scales_swizzled = torch.empty(max(sb, 16), dtype=torch.uint8, device=dev)
    st = lib().mxfp8_quantize_swizzled(_dev(w, "w", torch.bfloat16), batch, m, k,
                                       _dev(codes, "codes", torch.uint8, batch * m * k),
                                       _dev(scales_swizzled, "scales_swizzled", torch.uint8, sb), _stream(stream))
    _check("mxfp8_quantize_swizzled", st)
    return codes, scales_swizzled[:sb]


def fp8q_ring_hop_group(hops: Sequence[dict], fmt="e4m3", stream=None):
    """Several independent hops in one launch; each dict has the tensors
    in_codes, in_scales, local and optionally out_codes, out_scales,
    out_bf16 (allocated when missing; out_bf16 only if want_bf16).  Returns
    the list of (out_codes, out_scales, out_bf16 or None)."""
    return fp8q_ring_hop_group_ex(hops, fmt, 0, stream, _name="fp8q_ring_hop_group")


def fp8q_ring_hop_group_ex(hops: Sequence[dict], fmt="e4m3", flags: int = 0, stream=None, _name=None):
    """fp8q_ring_hop_group with flags (FP8Q_HOP_LOCAL_READY: no kernel still
    running when this launch starts writes any hop's local partial)."""
    count = len(hops)
    arr = (fp8q_hop_t * max(count, 1))()
    outs = []
    for i, hp in enumerate(hops):
        loc = hp["local"]
        n = loc.numel()
        nb = fp8q_num_scales(n)
        oc = hp.get("out_codes") if hp.get("out_codes") is not None else torch.empty(n, dtype=torch.uint8,
                                                                                      device=loc.device)
        os_ = hp.get("out_scales") if hp.get("out_scales") is not None else torch.empty(max(nb, 1),
                                                                                        dtype=torch.float32,
                                                                                        device=loc.device)
        ob = hp.get("out_bf16")
        if ob is None and hp.get("want_bf16"):
            ob = torch.empty(n, dtype=torch.bfloat16, device=loc.device)
        arr[i] = fp8q_hop_t(_dev(hp["in_codes"], f"hops[{i}].in_codes", torch.uint8, n),
                            _dev(hp["in_scales"], f"hops[{i}].in_scales", torch.float32, nb),
                            _dev(loc, f"hops[{i}].local", torch.bfloat16), n,
                            _dev(oc, f"hops[{i}].out_codes", torch.uint8, n),
                            _dev(os_, f"hops[{i}].out_scales", torch.float32, nb),
                            _dev(ob, f"hops[{i}].out_bf16", torch.bfloat16, n))
        outs.append((oc, os_, ob))
    if _name == "fp8q_ring_hop_group":
        st = lib().fp8q_ring_hop_group(arr, count, _fmt(fmt), _stream(stream))
    else:
        _name = "fp8q_ring_hop_group_ex"
        st = lib().fp8q_ring_hop_group_ex(arr, count, _fmt(fmt), flags, _stream(stream))
    _check(_name, st)
    return outs


def fp8q_ring_allreduce_sim(partials: Sequence[torch.Tensor], fmt="e4m3", results: Optional[Sequence[torch.Tensor]] = None,
                            workspace: Optional[torch.Tensor] = None, stream=None, mean: bool = False):
    """Ring AllReduce of P ranks' bf16 vectors held on one GPU, over the FP8
    wire format -> (list of P result tensors, wire bytes sent per rank).
    mean=True divides the decoded sum by P (FP8Q_ALLREDUCE_MEAN)."""
    P = len(partials)
    n = partials[0].numel()
    dev = partials[0].device
    if results is None:
        results = [torch.empty(n, dtype=torch.bfloat16, device=dev) for _ in range(P)]
    wb = int(lib().fp8q_ring_allreduce_workspace_bytes(P, n))
    if workspace is None:
        workspace = torch.empty(max(wb, 16), dtype=torch.uint8, device=dev)
    pp = (_vp * P)(*[_dev(t, f"partials[{i}]", torch.bfloat16, n) for i, t in enumerate(partials)])
    rp = (_vp * P)(*[_dev(t, f"results[{i}]", torch.bfloat16, n) for i, t in enumerate(results)])
    wire = ctypes.c_uint64(0)
    flags = FP8Q_ALLREDUCE_MEAN if mean else 0
    st = lib().fp8q_ring_allreduce_sim_ex(pp, rp, P, n, _fmt(fmt), _dev(workspace, "workspace", torch.uint8),
                                          workspace.numel(), ctypes.byref(wire), flags, _stream(stream))
    _check("fp8q_ring_allreduce_sim_ex", st)
    return list(results), int(wire.value)


def fp8q_gather_decode(codes: torch.Tensor, scales: torch.Tensor, count: int, fmt="e4m3",
                       outs: Optional[Sequence[torch.Tensor]] = None, mean: bool = False, stream=None):
    """One FP8 vector decoded once into `count` bf16 outputs (the all-gather
    step of the ring AllReduce); mean=True divides by `count` first."""
    n = codes.numel()
    if outs is None:
        outs = [torch.empty(n, dtype=torch.bfloat16, device=codes.device) for _ in range(count)]
    op = (_vp * count)(*[_dev(t, f"outs[{i}]", torch.bfloat16, n) for i, t in enumerate(outs)])
    st = lib().fp8q_gather_decode(_dev(codes, "codes", torch.uint8), _dev(scales, "scales", torch.float32,
                                                                           fp8q_num_scales(n)),
                                  n, _fmt(fmt), op, count, FP8Q_ALLREDUCE_MEAN if mean else 0, _stream(stream))
    _check("fp8q_gather_decode", st)
    return list(outs)


def mxfp8_quantize_swizzled_group(weights: Sequence[torch.Tensor], codes: Optional[Sequence[torch.Tensor]] = None,
                                  scales: Optional[Sequence[torch.Tensor]] = None, stream=None, flags: int = 0):
    """Several bf16 weights ([m, k] or [batch, m, k]) in one launch ->
    (list of codes, list of swizzled scale buffers), as one
    mxfp8_quantize_swizzled per weight would give."""
    n = len(weights)
    if n > MXFP8_MAX_GROUP:
        raise ValueError(f"at most {MXFP8_MAX_GROUP} tensors per group")
    arr = (mxfp8_tensor_t * max(n, 1))()
    outc, outs = [], []
    for i, w in enumerate(weights):
        if w.dim() == 2:
            b, (m, k) = 1, w.shape
        elif w.dim() == 3:
            b, m, k = w.shape
        else:
            raise ValueError("each weight must be 2D or 3D")
        sb = mxfp8_swizzled_scale_bytes(b, m, k)
        c = codes[i] if codes is not None else torch.empty(w.shape, dtype=torch.uint8, device=w.device)
        sc = scales[i] if scales is not None else torch.empty(max(sb, 16), dtype=torch.uint8, device=w.device)
        arr[i] = mxfp8_tensor_t(_dev(w, f"weights[{i}]", torch.bfloat16), b, m, k,
                                _dev(c, f"codes[{i}]", torch.uint8, b * m * k),
                                _dev(sc, f"scales[{i}]", torch.uint8, sb))
        outc.append(c)
        outs.append(sc[:sb])
    st = lib().mxfp8_quantize_swizzled_group_ex(arr, n, flags, _stream(stream))
    _check("mxfp8_quantize_swizzled_group_ex" if flags else "mxfp8_quantize_swizzled_group", st)
    return outc, outs


def mxfp8_quantize_swizzled_group_ex(weights: Sequence[torch.Tensor], flags: int = 0, **kw):
    """mxfp8_quantize_swizzled_group with flags (FP8Q_INPUTS_READY); keyword
    arguments as mxfp8_quantize_swizzled_group."""
    return mxfp8_quantize_swizzled_group(weights, flags=flags, **kw)


def _mx_shape(codes: torch.Tensor):
    if codes.dim() == 2:
        return 1, codes.shape[0], codes.shape[1]
    if codes.dim() == 3:
        return tuple(codes.shape)
    raise ValueError("codes must be 2D [m, k] or 3D [batch, m, k]")


def mxfp8_dequantize_swizzled(codes: torch.Tensor, scales_swizzled: torch.Tensor,
                              out: Optional[torch.Tensor] = None, stream=None):
    """E4M3 codes [m, k] / [batch, m, k] + swizzled E8M0 bytes -> bf16 weights."""
    b, m, k = _mx_shape(codes)
    if out is None:
        out = torch.empty(codes.shape, dtype=torch.bfloat16, device=codes.device)
    st = lib().mxfp8_dequantize_swizzled(_dev(codes, "codes", torch.uint8),
                                         _dev(scales_swizzled, "scales_swizzled", torch.uint8,
                                              mxfp8_swizzled_scale_bytes(b, m, k)),
                                         b, m, k, _dev(out, "out", torch.bfloat16, b * m * k), _stream(stream))
    _check("mxfp8_dequantize_swizzled", st)
    return out


def mxfp8_unswizzle_scales(scales_swizzled: torch.Tensor, batch: int, m: int, k: int,
                           out: Optional[torch.Tensor] = None, stream=None):
    """Swizzled E8M0 bytes -> row-major uint8 [batch, m, k // 32]."""
    if out is None:
        out = torch.empty((batch, m, k // 32), dtype=torch.uint8, device=scales_swizzled.device)
    st = lib().mxfp8_unswizzle_scales(_dev(scales_swizzled, "scales_swizzled", torch.uint8,
                                           mxfp8_swizzled_scale_bytes(batch, m, k)),
                                      batch, m, k, _dev(out, "out", torch.uint8, batch * m * (k // 32)),
                                      _stream(stream))
    _check("mxfp8_unswizzle_scales", st)
    return out


def fp8q_count_mismatches(a: torch.Tensor, b: torch.Tensor, count: Optional[torch.Tensor] = None, stream=None):
    """Number of differing bytes of two equally sized CUDA tensors (an int64
    device tensor; pass `count` to accumulate into an existing one)."""
    nbytes = a.numel() * a.element_size()
    if b.numel() * b.element_size() != nbytes:
        raise ValueError("a and b must have the same byte size")
    if count is None:
        count = torch.zeros(1, dtype=torch.int64, device=a.device)
    st = lib().fp8q_count_mismatches(_dev(a, "a"), _dev(b, "b"), nbytes, _dev(count, "count", torch.int64, 1),
                                     _stream(stream))
    _check("fp8q_count_mismatches", st)
    return count


def fp8q_quantize_tensorwise(x: torch.Tensor, fmt="e4m3", codes: Optional[torch.Tensor] = None,
                             scale_amax: Optional[torch.Tensor] = None, stream=None):
    """bf16 x -> (codes uint8 [n], float32 [2] device tensor holding (scale, amax))."""
    n = x.numel()
    if codes is None:
        codes = torch.empty(n, dtype=torch.uint8, device=x.device)
    if scale_amax is None:
        scale_amax = torch.empty(4, dtype=torch.float32, device=x.device)
    st = lib().fp8q_quantize_tensorwise(_dev(x, "x", torch.bfloat16), n, _fmt(fmt),
                                        _dev(codes, "codes", torch.uint8, n),
                                        _dev(scale_amax, "scale_amax", torch.float32, 2), _stream(stream))
    _check("fp8q_quantize_tensorwise", st)
    return codes, scale_amax[:2]


def fp8q_ring_hop_bf16_requant(in_codes: torch.Tensor, in_scales: torch.Tensor, local: torch.Tensor, fmt="e4m3",
                               want_bf16: bool = False, stream=None):
    """fp8q_ring_hop that requantizes the bf16-rounded sum -> (codes, scales, bf16 or None)."""
    n = local.numel()
    dev = local.device
    nb = fp8q_num_scales(n)
    oc = torch.empty(n, dtype=torch.uint8, device=dev)
    os_ = torch.empty(max(nb, 1), dtype=torch.float32, device=dev)
    ob = torch.empty(n, dtype=torch.bfloat16, device=dev) if want_bf16 else None
    st = lib().fp8q_ring_hop_bf16_requant(_dev(in_codes, "in_codes", torch.uint8, n),
                                          _dev(in_scales, "in_scales", torch.float32, nb),
                                          _dev(local, "local", torch.bfloat16), n, _fmt(fmt), _dev(oc, "out_codes"),
                                          _dev(os_, "out_scales"), _dev(ob, "out_bf16"), _stream(stream))
    _check("fp8q_ring_hop_bf16_requant", st)
    return oc, os_, ob


def fp8q_pack_plan(pairs: Sequence[tuple], cap_bytes: int):
    """pairs: (codes_bytes, scales_bytes) per weight -> (list of
    (batch, codes_offset, scales_offset), list of batch sizes)."""
    n = len(pairs)
    items = (fp8q_pack_item_t * max(n, 1))(*[fp8q_pack_item_t(int(c), int(s)) for c, s in pairs])
    slots = (fp8q_pack_slot_t * max(n, 1))()
    sizes = (ctypes.c_uint64 * max(n, 1))()
    nb = _int(0)
    _check("fp8q_pack_plan", lib().fp8q_pack_plan(items, n, cap_bytes, slots, sizes, ctypes.byref(nb)))
    return [(slots[i].batch, slots[i].codes_offset, slots[i].scales_offset) for i in range(n)], \
        [int(sizes[b]) for b in range(nb.value)]


def fp8q_copy_segments(segments: Sequence[tuple], stream=None):
    """segments: (src tensor, dst tensor view) pairs of equal byte size; one launch."""
    n = len(segments)
    arr = (fp8q_copy_t * max(n, 1))()
    for i, (src, dst) in enumerate(segments):
        nbytes = src.numel() * src.element_size()
        if dst.numel() * dst.element_size() != nbytes:
            raise ValueError(f"segment {i}: source and destination sizes differ")
        arr[i] = fp8q_copy_t(_dev(src, f"segments[{i}].src"), _dev(dst, f"segments[{i}].dst"), nbytes)
    _check("fp8q_copy_segments", lib().fp8q_copy_segments(arr, n, _stream(stream)))


def fp8q_encode_f32(x: torch.Tensor, fmt="e4m3", codes: Optional[torch.Tensor] = None, stream=None):
    n = x.numel()
    if codes is None:
        codes = torch.empty(n, dtype=torch.uint8, device=x.device)
    st = lib().fp8q_encode_f32(_dev(x, "x", torch.float32), n, _fmt(fmt), _dev(codes, "codes", torch.uint8, n),
                               _stream(stream))
    _check("fp8q_encode_f32", st)
    return codes


def fp8q_dequantize(codes: torch.Tensor, scales: torch.Tensor, fmt="e4m3", out_bf16: Optional[torch.Tensor] = None,
                    out_fp32: Optional[torch.Tensor] = None, want_bf16: bool = False, want_fp32: bool = True,
                    stream=None):
    n = codes.numel()
    dev = codes.device
    if out_bf16 is None and want_bf16:
        out_bf16 = torch.empty(n, dtype=torch.bfloat16, device=dev)
    if out_fp32 is None and want_fp32:
        out_fp32 = torch.empty(n, dtype=torch.float32, device=dev)
    st = lib().fp8q_dequantize(_dev(codes, "codes", torch.uint8, n),
                               _dev(scales, "scales", torch.float32, fp8q_num_scales(n)), n, _fmt(fmt),
                               _dev(out_bf16, "out_bf16", torch.bfloat16, n), _dev(out_fp32, "out_fp32", torch.float32, n),
                               _stream(stream))
    _check("fp8q_dequantize", st)
    return out_bf16, out_fp32


def fp8q_dequant_reduce_unfused(codes: Sequence[torch.Tensor], scales: Sequence[torch.Tensor], fmt="e4m3",
                                workspace: Optional[torch.Tensor] = None, out_bf16: Optional[torch.Tensor] = None,
                                out_fp32: Optional[torch.Tensor] = None, want_bf16: bool = True,
                                want_fp32: bool = True, n: Optional[int] = None, stream=None):
    """The naive dequantize-to-HBM-then-reduce order (comparator); needs a
    k * fp8q_unfused_stride(n) fp32 workspace."""
    k = len(codes)
    if n is None:
        n = codes[0].numel()
    dev = codes[0].device
    stride = int(lib().fp8q_unfused_stride(n))
    if workspace is None:
        workspace = torch.empty(max(k * stride, 1), dtype=torch.float32, device=dev)
    if out_bf16 is None and want_bf16:
        out_bf16 = torch.empty(n, dtype=torch.bfloat16, device=dev)
    if out_fp32 is None and want_fp32:
        out_fp32 = torch.empty(n, dtype=torch.float32, device=dev)
    cp = _ptr_array(codes, "codes", torch.uint8, n)
    sp = _ptr_array(scales, "scales", torch.float32, fp8q_num_scales(n))
    st = lib().fp8q_dequant_reduce_unfused(cp, sp, k, n, _fmt(fmt), _dev(workspace, "workspace", torch.float32, k * stride),
                                           _dev(out_bf16, "out_bf16", torch.bfloat16, n),
                                           _dev(out_fp32, "out_fp32", torch.float32, n), _stream(stream))
    _check("fp8q_dequant_reduce_unfused", st)
    return out_bf16, out_fp32


FP8Q_STATIC_SCRATCH_FLOATS = 1 << 22


def fp8q_dequant_reduce_unfused_static(codes: Sequence[torch.Tensor], scales: Sequence[torch.Tensor], fmt="e4m3",
                                       out_bf16: Optional[torch.Tensor] = None,
                                       out_fp32: Optional[torch.Tensor] = None, want_bf16: bool = True,
                                       want_fp32: bool = True, n: Optional[int] = None, stream=None):
    """The unfused comparator with the library's static scratch instead of a
    workspace, for callers that cannot allocate device memory.  Requires
    k * fp8q_unfused_stride(n) <= FP8Q_STATIC_SCRATCH_FLOATS; calls that
    overlap on the GPU race on the shared scratch."""
    k = len(codes)
    if n is None:
        n = codes[0].numel()
    dev = codes[0].device
    if out_bf16 is None and want_bf16:
        out_bf16 = torch.empty(n, dtype=torch.bfloat16, device=dev)
    if out_fp32 is None and want_fp32:
        out_fp32 = torch.empty(n, dtype=torch.float32, device=dev)
    cp = _ptr_array(codes, "codes", torch.uint8, n)
    sp = _ptr_array(scales, "scales", torch.float32, fp8q_num_scales(n))
    st = lib().fp8q_dequant_reduce_unfused_static(cp, sp, k, n, _fmt(fmt),
                                                  _dev(out_bf16, "out_bf16", torch.bfloat16, n),
                                                  _dev(out_fp32, "out_fp32", torch.float32, n), _stream(stream))
    _check("fp8q_dequant_reduce_unfused_static", st)
    return out_bf16, out_fp32
