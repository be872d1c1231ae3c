"""The bench's check of its own timed outputs against the oracle (host
logic, on CPU tensors): equal outputs give no mismatch, one changed byte in
any output is counted."""
import types

import numpy as np
import pytest
import torch

import bench
import gen


def _sample(orc):
    n = 4096 + 256
    shards = [gen.normal_bf16(n, 1e-4, seed=r).view(torch.int16).numpy().view(np.uint16) for r in range(8)]
    mats = [(gen.normal_bf16(2 * 128 * 64, 0.02, seed=9).view(torch.int16).numpy().view(np.uint16), 2, 128, 64),
            (gen.normal_bf16(256 * 96, 0.02, seed=10).view(torch.int16).numpy().view(np.uint16), 1, 256, 96)]
    keep = {}
    bench._oracle_step(orc, shards, mats, keep=keep)
    return keep


def _device_set_from(keep):
    """A stand-in for the bench's device set holding the oracle's results,
    laid out as the GPU step lays out its outputs (CPU tensors)."""
    def t(a, dtype=None):
        x = torch.from_numpy(np.ascontiguousarray(a).copy())
        return x.view(dtype) if dtype is not None else x
    q = {f: (torch.stack([t(c) for c, _ in keep["q"][f]]), torch.stack([t(s) for _, s in keep["q"][f]]))
         for f in (0, 1)}
    red = {f: (t(keep["red"][f][0].view(np.int16), torch.bfloat16), t(keep["red"][f][1])) for f in (0, 1)}
    hops = [(t(c), t(s)) for c, s, _ in keep["hops"]]
    ring_bf16 = t(keep["hops"][-1][2].view(np.int16), torch.bfloat16)
    mx = [(t(mc), t(ms), ms.size) for _, _, _, _, mc, ms in keep["mx"]]
    return types.SimpleNamespace(q=q, red=red, hops=hops, ring_bf16=ring_bf16, mx=mx)


def test_equal_outputs_give_no_mismatch(orc):
    keep = _sample(orc)
    r = bench.parity_against_oracle(_device_set_from(keep), keep)
    assert r["mismatches"] == 0
    n = keep["n"]
    assert r["elements"] == 2 * 9 * n + 7 * n + 2 * 128 * 64 + 256 * 96


@pytest.mark.parametrize("where", ["q", "red", "hop", "ring_bf16", "mx_codes", "mx_scales"])
def test_one_changed_byte_is_counted(orc, where):
    keep = _sample(orc)
    ds = _device_set_from(keep)
    if where == "q":
        ds.q[1][0][5, 77] ^= 1
    elif where == "red":
        ds.red[0][1].view(torch.uint8)[13] ^= 1
    elif where == "hop":
        ds.hops[3][1].view(torch.uint8)[2] ^= 1
    elif where == "ring_bf16":
        ds.ring_bf16.view(torch.uint8)[1] ^= 1
    elif where == "mx_codes":
        ds.mx[0][0][300] ^= 1
    else:
        ds.mx[1][1][17] ^= 1
    assert bench.parity_against_oracle(ds, keep)["mismatches"] == 1
