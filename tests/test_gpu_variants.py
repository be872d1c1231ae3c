"""Variants of the codec on the GPU against the oracle: per-tensor scaling
and the ring hop that requantizes the bf16-rounded sum."""
import numpy as np
import pytest
import torch

import gen
from gpu_util import assert_same, assert_same_f32, bf16_from_bits, bits16, u8, varied_bf16
from test_gpu_reduce import random_shards

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w():
    import weight_transfer_gb300 as w
    return w


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("n", [1, 7, 128, 129, 4096 + 17, 1 << 20, 8192 * 3, 8192 * 2 + 9, 8192 * 5 + 8191])
def test_tensorwise_random(w, orc, fmt, n):
    # two 8192-element tiles per CTA: odd tile counts leave the last CTA one
    # tile, staged or ragged
    rng = np.random.default_rng(n + fmt)
    x = (rng.standard_normal(n) * 10.0 ** rng.uniform(-20, 20)).astype(np.float32)
    x[rng.random(n) < 0.001] *= 300.0
    xb = bits16(torch.from_numpy(x).to(torch.bfloat16))
    codes, sa = w.fp8q_quantize_tensorwise(bf16_from_bits(xb), fmt)
    ec, es, ea = orc.quantize_tensorwise(xb, fmt)
    assert_same(u8(codes), ec, "codes")
    assert_same_f32(sa.cpu().numpy(), np.array([es, ea], np.float32), "scale, amax")


def test_tensorwise_varied_and_ddp_shard(w, orc):
    for xb in (varied_bf16(300_001, seed=3), bits16(gen.ddp_shard(0))):
        for fmt in (0, 1):
            codes, sa = w.fp8q_quantize_tensorwise(bf16_from_bits(xb), fmt)
            ec, es, ea = orc.quantize_tensorwise(xb, fmt)
            assert_same(u8(codes), ec, "codes")
            assert_same_f32(sa.cpu().numpy(), np.array([es, ea], np.float32), "scale, amax")


def test_tensorwise_all_zero(w, orc):
    xb = np.zeros(1000, np.uint16)
    xb[5] = 0x8000
    codes, sa = w.fp8q_quantize_tensorwise(bf16_from_bits(xb), 0)
    assert_same(u8(codes), orc.quantize_tensorwise(xb, 0)[0], "codes")
    assert float(sa[0]) == 0.0 and int(u8(codes)[5]) == 0x80


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("n", [1, 129, 4096 * 3 + 5, 200_003])
def test_ring_hop_bf16_requant(w, orc, fmt, n):
    codes, scales = random_shards(1, n, fmt, seed=n + 9 * fmt)
    scales[0] = np.minimum(scales[0], np.float32(1e20))
    loc = varied_bf16(n, seed=n + 1)
    oc, os_, ob = w.fp8q_ring_hop_bf16_requant(torch.from_numpy(codes[0]).cuda(), torch.from_numpy(scales[0]).cuda(),
                                               bf16_from_bits(loc), fmt, want_bf16=True)
    ec, es, eb = orc.ring_hop_bf16_requant(codes[0], scales[0], loc, fmt)
    assert_same(u8(oc), ec, "codes")
    assert_same_f32(os_.cpu().numpy()[:es.size], es, "scales")
    assert_same(bits16(ob), eb, "bf16")
