"""(a) Blockwise quantize and the fp32 -> FP8 conversion on the GPU, against
the oracle, bit for bit.  Calls go through the C ABI via the binding."""
import concurrent.futures as cf

import numpy as np
import pytest
import torch

import gen
from gpu_util import Guarded, assert_same, assert_same_f32, bf16_from_bits, bits16, u8, varied_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w():
    import weight_transfer_gb300 as w
    assert torch.cuda.is_available()
    return w


def run_quant(w, xbits, fmt):
    n = xbits.size
    x = bf16_from_bits(xbits)
    gc = Guarded(n, torch.uint8)
    gs = Guarded(max((n + 127) // 128, 1), torch.float32)
    w.fp8q_quantize_blockwise(x, fmt, codes=gc.t, scales=gs.t)
    torch.cuda.synchronize()
    assert gc.intact() and gs.intact(), "write outside the output buffers"
    return u8(gc.t), gs.t.cpu().numpy()


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("n", [1, 7, 8, 9, 127, 128, 129, 255, 256, 300, 4096 + 17, 128 * 1000 + 77, 1 << 20,
                               8192 * 2 + 5, 8192 * 5, 8192 * 7 + 8191])
def test_quantize_sizes(w, orc, fmt, n):
    # each CTA takes two consecutive 8192-element tiles: an odd tile count
    # leaves the last CTA one tile, staged (8192 * 5) or ragged (8192 * 2 + 5)
    xb = varied_bf16(n, seed=n + 31 * fmt)
    codes, scales = run_quant(w, xb, fmt)
    oc, os_ = orc.quantize_blockwise(xb, fmt)
    assert_same_f32(scales[:os_.size], os_, "scales")
    assert_same(codes, oc, "codes")


@pytest.mark.parametrize("fmt", [0, 1])
def test_quantize_every_bf16_input_for_many_scales(w, orc, fmt):
    # every finite bf16 pattern below each of 64 block amax values
    from test_oracle_ops import _blocks_of_all_bf16_below
    rng = np.random.default_rng(900 + fmt)
    amaxes = list(rng.integers(0x0001, 0x7F7F, size=60)) + [0x0001, 0x0080, 0x3F80, 0x7F7F]
    xb = np.concatenate([_blocks_of_all_bf16_below(np.uint16(a)) for a in amaxes])
    codes, scales = run_quant(w, xb, fmt)
    oc, os_ = orc.quantize_blockwise(xb, fmt)
    assert_same_f32(scales, os_, "scales")
    assert_same(codes, oc, "codes")


def test_quantize_empty(w):
    c, s = w.fp8q_quantize_blockwise(torch.empty(0, dtype=torch.bfloat16, device="cuda"))
    assert c.numel() == 0


@pytest.mark.parametrize("fmt", [0, 1])
def test_quantize_pr1_config(w, orc, fmt):
    for r in range(2):
        x = gen.pr1_shard(r)
        xb = bits16(x)
        codes, scales = run_quant(w, xb, fmt)
        oc, os_ = orc.quantize_blockwise(xb, fmt)
        assert_same_f32(scales, os_, f"scales shard {r}")
        assert_same(codes, oc, f"codes shard {r}")


@pytest.mark.parametrize("fmt", [0, 1])
def test_quantize_ddp_bucket_config(w, orc, fmt):
    # 25 MiB bucket, 8 shards, at full size and with the bench's launch shape
    def oracle(r):
        return orc.quantize_blockwise(bits16(gen.ddp_shard(r)), fmt)
    with cf.ThreadPoolExecutor(8) as ex:
        expected = list(ex.map(oracle, range(gen.DDP_K)))
    # one launch over the [8, n] bucket, as the bench quantizes it (n is a
    # multiple of 128, so no block straddles two shards)
    n, k = gen.DDP_N, gen.DDP_K
    bucket = torch.empty((k, n), dtype=torch.bfloat16, device="cuda")
    for r in range(k):
        bucket[r].copy_(gen.ddp_shard(r))
    c, s = w.fp8q_quantize_blockwise(bucket.view(-1), fmt)
    c, s = u8(c).reshape(k, n), s.cpu().numpy().reshape(k, n // 128)
    for r in range(k):
        assert_same_f32(s[r], expected[r][1], f"scales shard {r}")
        assert_same(c[r], expected[r][0], f"codes shard {r}")


@pytest.mark.parametrize("fmt", [0, 1])
def test_encode_f32_all_2_32_patterns(w, orc, fmt):
    # the native satfinite RNE conversion against the oracle's encoder for
    # every binary32 bit pattern (NaN inputs only need a NaN code back)
    chunk = 1 << 28
    pool = cf.ThreadPoolExecutor(16)
    for c0 in range(0, 1 << 32, chunk):
        idx = torch.arange(c0, c0 + chunk, dtype=torch.int64, device="cuda")
        # the int32 whose two's-complement bits are the pattern
        x = (idx - (1 << 32) if c0 >= (1 << 31) else idx).to(torch.int32).view(torch.float32)
        got = u8(w.fp8q_encode_f32(x, fmt))
        del idx, x
        parts = list(pool.map(lambda s: orc.encode_pattern_range(fmt, c0 + s, chunk // 16),
                              range(0, chunk, chunk // 16)))
        want = np.concatenate(parts)
        pat = np.arange(c0, c0 + chunk, dtype=np.uint64).astype(np.uint32)
        nan = (pat & 0x7FFFFFFF) > 0x7F800000
        assert_same(got[~nan], want[~nan], f"chunk {c0:#x}")
        g = got[nan]
        if fmt == 0:
            assert ((g & 0x7F) == 0x7F).all()
        else:
            assert (((g & 0x7C) == 0x7C) & ((g & 3) != 0)).all()
    pool.shutdown()


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("flags", [0, 1])
def test_quantize_group_mixed_sizes(w, orc, fmt, flags):
    # items of every shape: a single element, one partial block, whole tiles,
    # a ragged tile in the middle of the group's tile sequence, an empty item
    # and large varied inputs; each equals one fp8q_quantize_blockwise
    sizes = [1, 129, 8192, 8192 * 3 + 77, 0, 100_003, 8192 * 2, 300]
    xs = [varied_bf16(n, seed=700 + i) if n else np.zeros(0, np.uint16) for i, n in enumerate(sizes)]
    dx = [bf16_from_bits(x) if x.size else torch.empty(0, dtype=torch.bfloat16, device="cuda") for x in xs]
    gc = [Guarded(n, torch.uint8) if n else None for n in sizes]
    gs = [Guarded((n + 127) // 128, torch.float32) if n else None for n in sizes]
    codes = [g.t if g else torch.empty(0, dtype=torch.uint8, device="cuda") for g in gc]
    scales = [g.t if g else torch.empty(1, dtype=torch.float32, device="cuda") for g in gs]
    w.fp8q_quantize_blockwise_group(dx, fmt, flags, codes=codes, scales=scales)
    torch.cuda.synchronize()
    for i, n in enumerate(sizes):
        if n == 0:
            continue
        assert gc[i].intact() and gs[i].intact(), f"item {i} wrote outside its buffers"
        ec, es = orc.quantize_blockwise(xs[i], fmt)
        assert_same_f32(gs[i].t.cpu().numpy(), es, f"item {i} scales")
        assert_same(u8(gc[i].t), ec, f"item {i} codes")
