"""Oracle for the FP8 transfer codec -- TEST INFRASTRUCTURE ONLY.

A ctypes wrapper around ``liboracle.so``, the plain single-threaded C++
restatement of the codec in ``fp8q_oracle.cpp``.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline / reference leg of
``bench.py`` may import this package.  It shares no code with the CUDA
library and never imports it.

Arrays are numpy arrays on the host: bf16 values travel as ``uint16`` bit
patterns, codes and E8M0 scales as ``uint8``, blockwise scales as ``float32``.

Parity status of each function (what pins it is in ``tests/test_oracle_*``):
  encode / decode, bf16 rounding     pinned (hand table, brute force, torch's
                                     float8 / bfloat16 conversions)
  quantize_blockwise                 pinned (power-of-two worked blocks,
                                     amax invariant, exact error bound)
  dequant_reduce, ring_hop           pinned (exact rational sums within the
                                     fp32 recursive-summation bound)
  mxfp8 block codes and E8M0         pinned (hand examples, invariants)
  quantize_tensorwise                pinned (one block: equals the blockwise
                                     quantizer; power-of-two scales vs torch)
  ring_hop_bf16_requant              pinned (equals quantize of the bf16 sum)
  dequantize_mean                    pinned (the quotient evaluated in float64
                                     and rounded once; divisor 1 is the plain
                                     dequantize)
  mxfp8 dequantize / unswizzle       pinned (torch float8 decode times a power
                                     of two; round trip; the hand swizzle table)
  scale swizzle                      formula pinned by a hand table and a
                                     bijection check; the layout itself is
                                     parity unpinned by the pages.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8q_oracle.cpp")
LIB_PATH = os.path.join(_HERE, "liboracle.so")

E4M3 = 0
E5M2 = 1
FMT_MAX = {E4M3: 448.0, E5M2: 57344.0}
FMT_MAX_CODE = {E4M3: 0x7E, E5M2: 0x7B}


def build(force: bool = False) -> str:
    """Compile liboracle.so in place (g++, -ffp-contract=off, no fast-math)."""
    if not force and os.path.exists(LIB_PATH) and os.path.getmtime(LIB_PATH) >= os.path.getmtime(_SRC):
        return LIB_PATH
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c++17", "-fPIC", "-shared",
           "-o", tmp, _SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


_lib = None

_u8p = ctypes.POINTER(ctypes.c_uint8)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_f32p = ctypes.POINTER(ctypes.c_float)
_sz = ctypes.c_size_t
_i64 = ctypes.c_int64


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(LIB_PATH)
        L.orc_encode.argtypes = [ctypes.c_int, ctypes.c_float]
        L.orc_encode.restype = ctypes.c_uint8
        L.orc_encode_brute.argtypes = [ctypes.c_int, ctypes.c_float]
        L.orc_encode_brute.restype = ctypes.c_uint8
        L.orc_decode.argtypes = [ctypes.c_int, ctypes.c_uint8]
        L.orc_decode.restype = ctypes.c_float
        L.orc_fmt_max.argtypes = [ctypes.c_int]
        L.orc_fmt_max.restype = ctypes.c_float
        L.orc_encode_array.argtypes = [ctypes.c_int, _f32p, _sz, _u8p]
        L.orc_encode_brute_array.argtypes = [ctypes.c_int, _f32p, _sz, _u8p]
        L.orc_encode_pattern_range.argtypes = [ctypes.c_int, ctypes.c_uint64, _sz, _u8p]
        L.orc_decode_array.argtypes = [ctypes.c_int, _u8p, _sz, _f32p]
        L.orc_bf16_to_f32_array.argtypes = [_u16p, _sz, _f32p]
        L.orc_f32_to_bf16_array.argtypes = [_f32p, _sz, _u16p]
        L.orc_num_blocks.argtypes = [_sz]
        L.orc_num_blocks.restype = _sz
        L.orc_quantize_blockwise.argtypes = [_u16p, _sz, ctypes.c_int, _u8p, _f32p]
        L.orc_dequantize.argtypes = [_u8p, _f32p, _sz, ctypes.c_int, _u16p, _f32p]
        L.orc_dequantize_mean.argtypes = [_u8p, _f32p, _sz, ctypes.c_int, ctypes.c_int, _u16p, _f32p]
        L.orc_dequant_reduce.argtypes = [ctypes.POINTER(_u8p), ctypes.POINTER(_f32p), ctypes.c_int, _sz,
                                         ctypes.c_int, _u16p, _f32p]
        L.orc_ring_hop.argtypes = [_u8p, _f32p, _u16p, _sz, ctypes.c_int, _u8p, _f32p, _u16p]
        L.orc_e8m0_of_amax.argtypes = [ctypes.c_float]
        L.orc_e8m0_of_amax.restype = ctypes.c_uint8
        L.orc_mxfp8_block.argtypes = [_u16p, _u8p]
        L.orc_mxfp8_block.restype = ctypes.c_uint8
        L.orc_swizzle_offset.argtypes = [_i64, _i64, _i64, _i64, _i64]
        L.orc_swizzle_offset.restype = ctypes.c_uint64
        L.orc_swizzled_scale_bytes.argtypes = [_i64, _i64, _i64]
        L.orc_swizzled_scale_bytes.restype = ctypes.c_uint64
        L.orc_mxfp8_quantize_swizzled.argtypes = [_u16p, _i64, _i64, _i64, _u8p, _u8p]
        L.orc_mxfp8_quantize_swizzled.restype = ctypes.c_int
        L.orc_mxfp8_unswizzle.argtypes = [_u8p, _i64, _i64, _i64, _u8p]
        L.orc_mxfp8_dequantize.argtypes = [_u8p, _u8p, _i64, _i64, _i64, _u16p]
        L.orc_count_mismatches.argtypes = [_u8p, _u8p, _sz]
        L.orc_count_mismatches.restype = ctypes.c_uint64
        L.orc_quantize_tensorwise.argtypes = [_u16p, _sz, ctypes.c_int, _u8p, _f32p, _f32p]
        L.orc_ring_hop_bf16_requant.argtypes = [_u8p, _f32p, _u16p, _sz, ctypes.c_int, _u8p, _f32p, _u16p]
        _lib = L
    return _lib


def _p(a: np.ndarray, t):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be contiguous"
    return a.ctypes.data_as(t)


def _bf16_bits(x) -> np.ndarray:
    """Accept uint16 bit patterns, or a CPU torch.bfloat16 tensor."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16, "bf16 arrays travel as uint16 bit patterns"
        return np.ascontiguousarray(x)
    import torch  # only for the bit view of a bfloat16 tensor
    assert x.dtype == torch.bfloat16
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


# ------------------------------------------------------------- element level
def encode(fmt: int, v) -> np.ndarray:
    v = np.ascontiguousarray(np.asarray(v, dtype=np.float32).ravel())
    out = np.empty(v.size, np.uint8)
    lib().orc_encode_array(fmt, _p(v, _f32p), v.size, _p(out, _u8p))
    return out


def encode_brute(fmt: int, v) -> np.ndarray:
    v = np.ascontiguousarray(np.asarray(v, dtype=np.float32).ravel())
    out = np.empty(v.size, np.uint8)
    lib().orc_encode_brute_array(fmt, _p(v, _f32p), v.size, _p(out, _u8p))
    return out


def encode_pattern_range(fmt: int, first: int, n: int) -> np.ndarray:
    out = np.empty(n, np.uint8)
    lib().orc_encode_pattern_range(fmt, first, n, _p(out, _u8p))
    return out


def decode(fmt: int, codes) -> np.ndarray:
    c = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8).ravel())
    out = np.empty(c.size, np.float32)
    lib().orc_decode_array(fmt, _p(c, _u8p), c.size, _p(out, _f32p))
    return out


def bf16_to_f32(h) -> np.ndarray:
    h = np.ascontiguousarray(np.asarray(h, dtype=np.uint16).ravel())
    out = np.empty(h.size, np.float32)
    lib().orc_bf16_to_f32_array(_p(h, _u16p), h.size, _p(out, _f32p))
    return out


def f32_to_bf16(f) -> np.ndarray:
    f = np.ascontiguousarray(np.asarray(f, dtype=np.float32).ravel())
    out = np.empty(f.size, np.uint16)
    lib().orc_f32_to_bf16_array(_p(f, _f32p), f.size, _p(out, _u16p))
    return out


def num_blocks(n: int) -> int:
    return (n + 127) // 128


# --------------------------------------------------------------- operations
def quantize_blockwise(x, fmt: int):
    """bf16[n] -> (codes u8[n], scales f32[ceil(n/128)])."""
    x = _bf16_bits(x)
    n = x.size
    codes = np.empty(n, np.uint8)
    scales = np.empty(num_blocks(n), np.float32)
    lib().orc_quantize_blockwise(_p(x, _u16p), n, fmt, _p(codes, _u8p), _p(scales, _f32p))
    return codes, scales


def dequantize(codes, scales, fmt: int):
    """-> (bf16 bits u16[n], f32[n])."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.float32)
    n = codes.size
    ob = np.empty(n, np.uint16)
    of = np.empty(n, np.float32)
    lib().orc_dequantize(_p(codes, _u8p), _p(scales, _f32p), n, fmt, _p(ob, _u16p), _p(of, _f32p))
    return ob, of


def dequantize_mean(codes, scales, fmt: int, ranks: int):
    """dequantize, then the binary32 value divided by ``ranks`` (true
    division) -> (bf16 bits u16[n], f32[n])."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.float32)
    n = codes.size
    ob = np.empty(n, np.uint16)
    of = np.empty(n, np.float32)
    lib().orc_dequantize_mean(_p(codes, _u8p), _p(scales, _f32p), n, fmt, int(ranks), _p(ob, _u16p),
                              _p(of, _f32p))
    return ob, of


def dequant_reduce(codes_list, scales_list, fmt: int):
    """k shards -> (bf16 bits u16[n], f32[n]), summed in list order."""
    k = len(codes_list)
    assert k == len(scales_list) and k >= 1
    cs = [np.ascontiguousarray(c, dtype=np.uint8) for c in codes_list]
    ss = [np.ascontiguousarray(s, dtype=np.float32) for s in scales_list]
    n = cs[0].size
    for c, s in zip(cs, ss):
        assert c.size == n and s.size >= num_blocks(n)
    cp = (_u8p * k)(*[_p(c, _u8p) for c in cs])
    sp = (_f32p * k)(*[_p(s, _f32p) for s in ss])
    ob = np.empty(n, np.uint16)
    of = np.empty(n, np.float32)
    lib().orc_dequant_reduce(cp, sp, k, n, fmt, _p(ob, _u16p), _p(of, _f32p))
    return ob, of


def ring_hop(in_codes, in_scales, local, fmt: int):
    """-> (out codes u8[n], out scales f32[nb], bf16 bits of the fp32 sum u16[n])."""
    in_codes = np.ascontiguousarray(in_codes, dtype=np.uint8)
    in_scales = np.ascontiguousarray(in_scales, dtype=np.float32)
    local = _bf16_bits(local)
    n = in_codes.size
    assert local.size == n
    oc = np.empty(n, np.uint8)
    os_ = np.empty(num_blocks(n), np.float32)
    ob = np.empty(n, np.uint16)
    lib().orc_ring_hop(_p(in_codes, _u8p), _p(in_scales, _f32p), _p(local, _u16p), n, fmt,
                       _p(oc, _u8p), _p(os_, _f32p), _p(ob, _u16p))
    return oc, os_, ob


def e8m0_of_amax(amax: float) -> int:
    return int(lib().orc_e8m0_of_amax(float(amax)))


def mxfp8_block(w32) -> tuple[np.ndarray, int]:
    w32 = _bf16_bits(w32)
    assert w32.size == 32
    codes = np.empty(32, np.uint8)
    e = lib().orc_mxfp8_block(_p(w32, _u16p), _p(codes, _u8p))
    return codes, int(e)


def swizzle_offset(bt: int, r: int, j: int, m: int, kb: int) -> int:
    return int(lib().orc_swizzle_offset(bt, r, j, m, kb))


def swizzled_scale_bytes(batch: int, m: int, k: int) -> int:
    return int(lib().orc_swizzled_scale_bytes(batch, m, k))


def mxfp8_quantize_swizzled(w, batch: int, m: int, k: int):
    """bf16 [batch, m, k] -> (codes u8[batch*m*k], swizzled E8M0 scales u8[...])."""
    w = _bf16_bits(w).ravel()
    assert w.size == batch * m * k
    codes = np.empty(batch * m * k, np.uint8)
    scales = np.empty(max(swizzled_scale_bytes(batch, m, k), 1), np.uint8)
    rc = lib().orc_mxfp8_quantize_swizzled(_p(w, _u16p), batch, m, k, _p(codes, _u8p), _p(scales, _u8p))
    if rc != 0:
        raise ValueError("k must be a positive multiple of 32")
    return codes, scales[: swizzled_scale_bytes(batch, m, k)]


def mxfp8_unswizzle(scales, batch: int, m: int, k: int) -> np.ndarray:
    """Swizzled E8M0 bytes -> plain row-major [batch, m, k/32] uint8."""
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    out = np.empty(batch * m * (k // 32), np.uint8)
    lib().orc_mxfp8_unswizzle(_p(scales, _u8p), batch, m, k, _p(out, _u8p))
    return out


def mxfp8_dequantize(codes, scales, batch: int, m: int, k: int) -> np.ndarray:
    """E4M3 codes + swizzled E8M0 scales -> bf16 bit patterns [batch*m*k]."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8).ravel()
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    out = np.empty(batch * m * k, np.uint16)
    lib().orc_mxfp8_dequantize(_p(codes, _u8p), _p(scales, _u8p), batch, m, k, _p(out, _u16p))
    return out


def count_mismatches(a, b) -> int:
    a = np.ascontiguousarray(a, dtype=np.uint8).ravel()
    b = np.ascontiguousarray(b, dtype=np.uint8).ravel()
    assert a.size == b.size
    return int(lib().orc_count_mismatches(_p(a, _u8p), _p(b, _u8p), a.size))


def quantize_tensorwise(x, fmt: int):
    """bf16[n] -> (codes u8[n], scale, amax) with one scale for the tensor."""
    x = _bf16_bits(x)
    codes = np.empty(x.size, np.uint8)
    sc = np.zeros(1, np.float32)
    am = np.zeros(1, np.float32)
    lib().orc_quantize_tensorwise(_p(x, _u16p), x.size, fmt, _p(codes, _u8p), _p(sc, _f32p), _p(am, _f32p))
    return codes, sc[0], am[0]


def ring_hop_bf16_requant(in_codes, in_scales, local, fmt: int):
    """ring_hop, but requantizing RNE_bf16(y) instead of y."""
    in_codes = np.ascontiguousarray(in_codes, dtype=np.uint8)
    in_scales = np.ascontiguousarray(in_scales, dtype=np.float32)
    local = _bf16_bits(local)
    n = in_codes.size
    oc = np.empty(n, np.uint8)
    os_ = np.empty(num_blocks(n), np.float32)
    ob = np.empty(n, np.uint16)
    lib().orc_ring_hop_bf16_requant(_p(in_codes, _u8p), _p(in_scales, _f32p), _p(local, _u16p), n, fmt,
                                    _p(oc, _u8p), _p(os_, _f32p), _p(ob, _u16p))
    return oc, os_, ob
