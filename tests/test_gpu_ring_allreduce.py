"""Grouped ring hops and the simulated FP8 ring AllReduce on the GPU,
against the oracle driven through the same schedule."""
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
def test_hop_group_equals_single_hops(w, orc, fmt):
    # hops of different lengths, including ragged tails between full tiles
    sizes = [4096 * 3 + 77, 128, 1, 4096 * 5, 9000, 0, 4096 + 4095]
    hops, expect = [], []
    for i, n in enumerate(sizes):
        codes, scales = random_shards(1, max(n, 1), fmt, seed=300 + i)
        scales[0] = np.minimum(scales[0], np.float32(1e20))
        loc = varied_bf16(max(n, 1), seed=400 + i)
        if n == 0:
            hops.append({"in_codes": torch.empty(0, dtype=torch.uint8, device="cuda"),
                         "in_scales": torch.empty(1, dtype=torch.float32, device="cuda"),
                         "local": torch.empty(0, dtype=torch.bfloat16, device="cuda")})
            expect.append(None)
            continue
        hops.append({"in_codes": torch.from_numpy(codes[0]).cuda(), "in_scales": torch.from_numpy(scales[0]).cuda(),
                     "local": bf16_from_bits(loc), "want_bf16": i % 2 == 0})
        expect.append(orc.ring_hop(codes[0], scales[0], loc, fmt))
    outs = w.fp8q_ring_hop_group(hops, fmt)
    torch.cuda.synchronize()
    for i, ((oc, os_, ob), e) in enumerate(zip(outs, expect)):
        if e is None:
            continue
        assert_same(u8(oc), e[0], f"hop {i} codes")
        assert_same_f32(os_.cpu().numpy()[:e[1].size], e[1], f"hop {i} scales")
        if ob is not None:
            assert_same(bits16(ob), e[2], f"hop {i} bf16")


def oracle_allreduce(orc, parts, fmt, mean=False):
    """The same ring schedule, step by step, on the oracle."""
    P = len(parts)
    n = parts[0].size
    m = n // P
    msgs = [orc.quantize_blockwise(parts[i][i * m:(i + 1) * m].copy(), fmt) for i in range(P)]
    final = [None] * P
    for s in range(1, P):
        new = [None] * P
        for i in range(P):
            c = (i - s) % P
            oc, os_, _ = orc.ring_hop(msgs[(i - 1) % P][0], msgs[(i - 1) % P][1], parts[i][c * m:(c + 1) * m].copy(),
                                      fmt)
            if s < P - 1:
                new[i] = (oc, os_)
            else:
                final[c] = (oc, os_)
        msgs = new
    codes = np.concatenate([f[0] for f in final])
    scales = np.concatenate([f[1] for f in final])
    ob, _ = orc.dequantize_mean(codes, scales, fmt, P) if mean else orc.dequantize(codes, scales, fmt)
    return ob


@pytest.mark.parametrize("mean", [False, True])
@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("P,n", [(2, 1024), (3, 3 * 512 * 7), (5, 5 * 512 * 11), (8, 8 * 512 * 33),
                                 (16, 16 * 512 * 3)])
def test_ring_allreduce_matches_oracle_schedule(w, orc, fmt, P, n, mean):
    # n = 3 * 512 * 7 and 5 * 512 * 11 end in a ragged 4096-element tile of
    # the all-gather decode; P = 3, 5 make the mean a rounded division
    parts = [bits16(gen.ring_partial(r, n)) for r in range(P)]
    res, wire = w.fp8q_ring_allreduce_sim([bf16_from_bits(p) for p in parts], fmt, mean=mean)
    torch.cuda.synchronize()
    want = oracle_allreduce(orc, parts, fmt, mean)
    for r in range(P):
        assert_same(bits16(res[r]), want, f"rank {r}")
    m = n // P
    assert wire == 2 * (P - 1) * (m + 4 * (m // 128))


@pytest.mark.parametrize("P,n", [(8, 8 * 512 * 33), (3, 3 * 512 * 7)])
def test_ring_allreduce_in_place_mean(w, orc, P, n):
    # results written over the partials (each rank's own), with the mean
    parts = [bits16(gen.ring_partial(r, n)) for r in range(P)]
    dev = [bf16_from_bits(p) for p in parts]
    res, _ = w.fp8q_ring_allreduce_sim(dev, 0, results=dev, mean=True)
    torch.cuda.synchronize()
    want = oracle_allreduce(orc, parts, 0, True)
    for r in range(P):
        assert res[r].data_ptr() == dev[r].data_ptr()
        assert_same(bits16(res[r]), want, f"rank {r}")


def test_ring_allreduce_ddp_bucket_mean(w, orc):
    # the 8-rank bucket at full size, averaged: every rank equals the oracle
    P, n = gen.DDP_K, gen.DDP_N
    parts = [bits16(gen.ddp_shard(r)) for r in range(P)]
    res, _ = w.fp8q_ring_allreduce_sim([bf16_from_bits(p) for p in parts], "e4m3", mean=True)
    torch.cuda.synchronize()
    want = oracle_allreduce(orc, parts, 0, True)
    for r in range(P):
        assert_same(bits16(res[r]), want, f"rank {r}")


def test_ring_allreduce_ddp_bucket_wire_bytes_and_accuracy(w, orc):
    # the 25 MiB bucket of 8 ranks: every rank gets the oracle's result, the
    # wire carries 2 (P-1)/P of the payload at 1.03125 bytes per element,
    # i.e. 48.4% less than the bf16 ring, and the sum is close to the exact one
    P, n = gen.DDP_K, gen.DDP_N
    parts = [bits16(gen.ddp_shard(r)) for r in range(P)]
    res, wire = w.fp8q_ring_allreduce_sim([bf16_from_bits(p) for p in parts], "e4m3")
    torch.cuda.synchronize()
    want = oracle_allreduce(orc, parts, 0)
    for r in range(P):
        assert_same(bits16(res[r]), want, f"rank {r}")
    bf16_ring = 2 * (P - 1) / P * n * 2
    assert wire == 2 * (P - 1) * (n // P) * (1 + 4 / 128)
    assert round(1 - wire / bf16_ring, 4) == 0.4844
    exact = np.sum([(p.astype(np.uint32) << 16).view(np.float32).astype(np.float64) for p in parts], axis=0)
    got = (want.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    # relative to the bucket's scale, the FP8 ring stays within a few e4m3 ulps
    assert np.abs(got - exact).max() < 8 * 2.0 ** -4 * np.abs(exact).max()


def test_ring_allreduce_rejects_bad_sizes(w):
    parts = [torch.zeros(1000, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    with pytest.raises(w.Fp8qError):
        w.fp8q_ring_allreduce_sim(parts)          # 1000 is not a multiple of 512 * 2


@pytest.mark.parametrize("mean", [False, True])
@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("count,n", [(1, 4096), (3, 4096 * 5 + 77), (8, 20_000), (16, 4096 * 2 + 4095)])
def test_gather_decode_matches_oracle(w, orc, fmt, count, n, mean):
    # every output equals the oracle's dequantize (or its mean over `count`),
    # including the ragged last tile
    codes, scales = random_shards(1, n, fmt, seed=500 + count + n)
    sc = np.minimum(scales[0], np.float32(1e30))
    outs = w.fp8q_gather_decode(torch.from_numpy(codes[0]).cuda(), torch.from_numpy(sc).cuda(), count, fmt,
                                mean=mean)
    torch.cuda.synchronize()
    want, _ = orc.dequantize_mean(codes[0], sc, fmt, count) if mean else orc.dequantize(codes[0], sc, fmt)
    for o, t in enumerate(outs):
        assert_same(bits16(t), want, f"output {o}")


@pytest.mark.parametrize("mean", [False, True])
def test_ring_allreduce_256mib_per_rank_sampled(w, orc, mean):
    # the bench's large configuration, 8 ranks x 2^27 elements (256 MiB of
    # bf16 per rank), checked on sampled outputs: the result at a position
    # depends only on that position's 128-block in every rank, through the
    # same ring schedule for its chunk, so the oracle's AllReduce of the
    # sampled pieces (piece c taken from chunk c) gives those outputs exactly
    P, n = 8, 8 * (1 << 24)
    m, L = n // P, 1 << 16
    g = torch.Generator(device="cuda")
    g.manual_seed(1234)
    parts = [torch.randn(n, device="cuda", generator=g).mul_(1e-4).to(torch.bfloat16) for _ in range(P)]
    res, _ = w.fp8q_ring_allreduce_sim(parts, "e4m3", mean=mean)
    torch.cuda.synchronize()
    for off in (0, m // 2 + 128 * 37, m - L):
        idx = torch.cat([torch.arange(c * m + off, c * m + off + L, device="cuda") for c in range(P)])
        sub = [bits16(p[idx]) for p in parts]
        want = oracle_allreduce(orc, sub, 0, mean)
        for r in (0, 3, P - 1):
            assert_same(bits16(res[r][idx]), want, f"rank {r}, offset {off}")
        del idx
    del parts, res
    torch.cuda.empty_cache()
