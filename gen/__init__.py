"""Seeded synthetic inputs for the FP8 transfer codec (tests, bench, smoke).

The one module both sides of a parity check draw from.  It holds none of the
codec's arithmetic: ``gen.c`` draws binary32 normal samples (SplitMix64
counters + Box-Muller, see its header) and torch casts them to bf16.

Workload recipes (the stand-ins for the pages' real gradients and weights,
which need trained models and datasets that are not available):

* ``pr1``: 1,048,576 gradient values ~ N(0, 1e-3^2), 0.1% outliers x100,
  shard r drawn with seed r (two shards).
* ``ddp``: a 25 MiB DDP bucket, 13,107,200 values ~ N(0, 1e-4^2) per shard,
  shard r with seed r, k = 8 shards.
* ``vec3p5b``: a 3.5e9-element gradient vector ~ N(0, 1e-4^2), 1 in 1e4
  values x1000, 64 zero-filled 128-blocks, shard r with seed 100 + r.
* ``qwen3_layer``: the bf16 weights of one Qwen3-30B-A3B-shaped decoder
  layer, ~ N(0, 0.02^2) with 1% of rows x50 (the row is the outlier unit),
  one seed per (layer, tensor).
* ``ring``: 8 partials per payload size ~ N(0, 1e-3^2), partial r with seed
  200 + r.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
LIB_PATH = os.path.join(_HERE, "libgen.so")

NTHREADS = max(1, min(64, os.cpu_count() or 1))


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB_PATH) and os.path.getmtime(LIB_PATH) >= os.path.getmtime(_SRC):
        return LIB_PATH
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, "-lm"], check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


_lib = None


def _L():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(LIB_PATH)
        u64 = ctypes.c_uint64
        L.gen_normal_f32.argtypes = [u64, u64, u64, u64, ctypes.c_double, ctypes.c_double, ctypes.c_double,
                                     u64, ctypes.POINTER(ctypes.c_float), ctypes.c_int]
        L.gen_distinct_indices.argtypes = [u64, u64, u64, u64, ctypes.POINTER(ctypes.c_uint64)]
        _lib = L
    return _lib


def normal_f32(n: int, sigma: float, seed: int, stream: int = 0, offset: int = 0, outlier_p: float = 0.0,
               outlier_mult: float = 1.0, outlier_group: int = 1, out: np.ndarray | None = None) -> np.ndarray:
    """Samples offset .. offset+n-1 of stream (seed, stream) as float32."""
    if out is None:
        out = np.empty(n, np.float32)
    assert out.dtype == np.float32 and out.size == n and out.flags["C_CONTIGUOUS"]
    _L().gen_normal_f32(seed, stream, offset, n, sigma, outlier_p, outlier_mult, outlier_group,
                        out.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), NTHREADS)
    return out


def to_bf16(f32: np.ndarray) -> torch.Tensor:
    """torch's round-to-nearest-even cast; returns a CPU bfloat16 tensor."""
    return torch.from_numpy(f32).to(torch.bfloat16)


def normal_bf16(n: int, sigma: float, seed: int, **kw) -> torch.Tensor:
    return to_bf16(normal_f32(n, sigma, seed, **kw))


def distinct_indices(count: int, range_: int, seed: int, stream: int = 0) -> np.ndarray:
    out = np.empty(count, np.uint64)
    _L().gen_distinct_indices(seed, stream, count, range_, out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)))
    return out


# ------------------------------------------------------------------ recipes
PR1_N = 1_048_576
DDP_N = 13_107_200
DDP_K = 8
VEC_N = 3_500_000_000
VEC_K = 4
VEC_ZERO_BLOCKS = 64
VEC_CHUNK = 1 << 27              # 256 MiB of bf16 per streamed chunk


def pr1_shard(r: int) -> torch.Tensor:
    return normal_bf16(PR1_N, 1e-3, seed=r, outlier_p=1e-3, outlier_mult=100.0)


def ddp_shard(r: int, n: int = DDP_N) -> torch.Tensor:
    return normal_bf16(n, 1e-4, seed=r)


def vec_zero_blocks(r: int, n: int = VEC_N) -> np.ndarray:
    return np.sort(distinct_indices(VEC_ZERO_BLOCKS, (n + 127) // 128, seed=100 + r, stream=1))


def vec_chunk(r: int, start: int, count: int, n: int = VEC_N) -> torch.Tensor:
    """Elements [start, start+count) of shard r of the 3.5e9 vector."""
    f = normal_f32(count, 1e-4, seed=100 + r, offset=start, outlier_p=1e-4, outlier_mult=1000.0)
    zb = vec_zero_blocks(r, n)
    for b in zb:
        lo, hi = max(int(b) * 128, start), min(int(b) * 128 + 128, start + count)
        if lo < hi:
            f[lo - start:hi - start] = 0.0
    return to_bf16(f)


# Qwen3-30B-A3B-shaped decoder layer, weights stored [out, in] = [M, K]:
# 128 experts x (gate, up: [768, 2048]; down: [2048, 768]),
# q: [4096, 2048], k / v: [512, 2048], o: [2048, 4096].
QWEN3_LAYERS = 48
QWEN3_TENSORS = [
    ("experts.gate", 128, 768, 2048),
    ("experts.up", 128, 768, 2048),
    ("experts.down", 128, 2048, 768),
    ("attn.q", 1, 4096, 2048),
    ("attn.k", 1, 512, 2048),
    ("attn.v", 1, 512, 2048),
    ("attn.o", 1, 2048, 4096),
]


def qwen3_layer_elements() -> int:
    return sum(b * m * k for _, b, m, k in QWEN3_TENSORS)


def qwen3_tensor(layer: int, t: int) -> torch.Tensor:
    """bf16 [batch, M, K] of tensor t of the given layer."""
    _, b, m, k = QWEN3_TENSORS[t]
    f = normal_f32(b * m * k, 0.02, seed=10_000 + 100 * layer + t, outlier_p=0.01, outlier_mult=50.0,
                   outlier_group=k)
    return to_bf16(f).view(b, m, k)


RING_SIZES_BYTES = [1 << p for p in range(10, 29)] + [767 * 1024]
RING_PARTIALS = 8


def ring_partial(r: int, n: int) -> torch.Tensor:
    return normal_bf16(n, 1e-3, seed=200 + r)
