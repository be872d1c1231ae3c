"""(d) BF16 -> MXFP8 prequantization with the swizzled E8M0 scales on the
GPU, against the oracle: codes and the whole scale buffer (padding
included) bit for bit."""
import concurrent.futures as cf

import numpy as np
import pytest
import torch

import gen
from gpu_util import Guarded, assert_same, bf16_from_bits, bits16, u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w():
    import weight_transfer_gb300 as w
    return w


def weight_bits(b, m, k, seed):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((b, m, k)) * 0.02).astype(np.float32)
    rows = rng.random((b, m)) < 0.05
    x[rows] *= 50.0
    blk = x.reshape(b, m, k // 32, 32)
    z = rng.random((b, m, k // 32)) < 0.03
    blk[z] = 0.0                                           # zero-scale clamp
    t = rng.random((b, m, k // 32)) < 0.02
    blk[t] *= 1e-36                                        # tiny / subnormal blocks
    h = rng.random((b, m, k // 32)) < 0.01
    blk[h] *= 1e30                                         # huge blocks
    bits = torch.from_numpy(x.ravel()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()
    if bits.size > 64:
        bits[7] = 0x7F7F                                   # largest bf16
        bits[40] = 0x8000                                  # negative zero
    bits[(bits & 0x7F80) == 0x7F80] = 0x3C00
    return bits


def run(w, bits, b, m, k):
    x = bf16_from_bits(bits).view(b, m, k)
    gc = Guarded(b * m * k, torch.uint8)
    sb = w.mxfp8_swizzled_scale_bytes(b, m, k)
    gs = Guarded(sb, torch.uint8)
    w.mxfp8_quantize_swizzled(x, codes=gc.t.view(b, m, k), scales_swizzled=gs.t)
    torch.cuda.synchronize()
    assert gc.intact() and gs.intact(), "write outside the output buffers"
    return u8(gc.t), u8(gs.t)


@pytest.mark.parametrize("b,m,k", [(1, 1, 32), (1, 1, 64), (1, 127, 64), (1, 128, 128), (1, 129, 96), (3, 129, 32),
                                   (2, 256, 768), (1, 300, 2048), (5, 64, 160), (1, 4096, 2048), (2, 768, 2048)])
def test_mxfp8_shapes(w, orc, b, m, k):
    bits = weight_bits(b, m, k, seed=b * 7 + m + k)
    gc, gs = run(w, bits, b, m, k)
    ec, es = orc.mxfp8_quantize_swizzled(bits, b, m, k)
    assert_same(gs, es, "swizzled scales")
    assert_same(gc, ec, "codes")


def test_mxfp8_k32_scale_column_survives(w, orc):
    # K == 32: one real scale column per row, padded to a 4-wide tile
    bits = weight_bits(1, 200, 32, seed=5)
    gc, gs = run(w, bits, 1, 200, 32)
    ec, es = orc.mxfp8_quantize_swizzled(bits, 1, 200, 32)
    assert gs.size == 2 * 512
    assert_same(gs, es, "scales")
    assert_same(gc, ec, "codes")


def test_mxfp8_2d_call(w, orc):
    bits = weight_bits(1, 256, 512, seed=11)
    c, s = w.mxfp8_quantize_swizzled(bf16_from_bits(bits).view(256, 512))
    ec, es = orc.mxfp8_quantize_swizzled(bits, 1, 256, 512)
    assert c.shape == (256, 512)
    assert_same(u8(c).ravel(), ec, "codes")
    assert_same(u8(s), es, "scales")


def test_mxfp8_qwen3_layer_full_size(w, orc):
    # every tensor of one Qwen3-30B-A3B-shaped layer (all 48 layers have the
    # same shapes), checked in full; the oracle runs on expert slices in
    # parallel (the swizzled buffer is a concatenation over the batch)
    pool = cf.ThreadPoolExecutor(16)
    for t, (name, b, m, k) in enumerate(gen.QWEN3_TENSORS):
        x = gen.qwen3_tensor(0, t)
        c, s = w.mxfp8_quantize_swizzled(x.cuda())
        hb = bits16(x).reshape(b, m * k)
        per = w.mxfp8_swizzled_scale_bytes(1, m, k)
        step = max(1, b // 16)
        jobs = [(i, min(b, i + step)) for i in range(0, b, step)]
        res = list(pool.map(lambda ij: orc.mxfp8_quantize_swizzled(hb[ij[0]:ij[1]].copy(), ij[1] - ij[0], m, k), jobs))
        ec = np.concatenate([r[0] for r in res])
        es = np.concatenate([r[1] for r in res])
        assert es.size == b * per
        assert_same(u8(s), es, f"{name} scales")
        assert_same(u8(c).ravel(), ec, f"{name} codes")
        del c, s, x
    pool.shutdown()


def test_mxfp8_group_mixed_shapes_equals_per_tensor_oracle(w, orc):
    shapes = [(1, 1, 32), (3, 129, 96), (1, 0, 64), (2, 256, 768), (1, 300, 2048), (5, 64, 160), (1, 127, 64)]
    bits = [weight_bits(b, m, k, seed=70 + i) if b * m * k else np.zeros(0, np.uint16)
            for i, (b, m, k) in enumerate(shapes)]
    xs = [bf16_from_bits(x).view(b, m, k) for x, (b, m, k) in zip(bits, shapes)]
    codes, scales = w.mxfp8_quantize_swizzled_group(xs)
    torch.cuda.synchronize()
    for x, c, s, (b, m, k) in zip(bits, codes, scales, shapes):
        ec, es = orc.mxfp8_quantize_swizzled(x, b, m, k)
        assert_same(u8(s), es, f"scales {b}x{m}x{k}")
        assert_same(u8(c).ravel(), ec, f"codes {b}x{m}x{k}")


def test_mxfp8_group_whole_qwen3_layer(w, orc):
    # all 7 tensors of a Qwen3-30B-A3B-shaped layer (layer 1) in one launch,
    # checked in full against the oracle run per tensor on expert slices
    pool = cf.ThreadPoolExecutor(16)
    xs = [gen.qwen3_tensor(1, t) for t in range(len(gen.QWEN3_TENSORS))]
    codes, scales = w.mxfp8_quantize_swizzled_group([x.cuda() for x in xs])
    torch.cuda.synchronize()
    for t, (name, b, m, k) in enumerate(gen.QWEN3_TENSORS):
        hb = bits16(xs[t]).reshape(b, m * k)
        step = max(1, b // 16)
        jobs = [(i, min(b, i + step)) for i in range(0, b, step)]
        res = list(pool.map(lambda ij: orc.mxfp8_quantize_swizzled(hb[ij[0]:ij[1]].copy(), ij[1] - ij[0], m, k), jobs))
        assert_same(u8(scales[t]), np.concatenate([r[1] for r in res]), f"{name} scales")
        assert_same(u8(codes[t]).ravel(), np.concatenate([r[0] for r in res]), f"{name} codes")
    pool.shutdown()


@pytest.mark.parametrize("layer", [0, 23, 47])
def test_mxfp8_stack_layers_sampled(w, orc, layer):
    # the first, a middle and the last layer of the 48-layer stack, each in
    # the bench's one grouped launch; the oracle checks every attention
    # matrix in full and experts 0, 64 and 127 of each expert tensor
    xs = [gen.qwen3_tensor(layer, t) for t in range(len(gen.QWEN3_TENSORS))]
    codes, scales = w.mxfp8_quantize_swizzled_group([x.cuda() for x in xs])
    torch.cuda.synchronize()
    for t, (name, b, m, k) in enumerate(gen.QWEN3_TENSORS):
        hb = bits16(xs[t]).reshape(b, m * k)
        per = w.mxfp8_swizzled_scale_bytes(1, m, k)
        gc = u8(codes[t]).reshape(b, m * k)
        gs = u8(scales[t]).reshape(b, per)
        for e in ([0] if b == 1 else [0, 64, 127]):
            ec, es = orc.mxfp8_quantize_swizzled(hb[e].copy(), 1, m, k)
            assert_same(gs[e], es, f"layer {layer} {name}[{e}] scales")
            assert_same(gc[e], ec, f"layer {layer} {name}[{e}] codes")


# ----------------------------------------------------------- receiver side
@pytest.mark.parametrize("b,m,k", [(1, 1, 32), (3, 129, 96), (2, 256, 768), (1, 300, 2048)])
def test_mxfp8_dequantize_and_unswizzle(w, orc, b, m, k):
    # inputs from the oracle's quantizer, plus random codes with random scale
    # bytes (every e8m0 value, subnormal results included)
    bits = weight_bits(b, m, k, seed=b + m + k)
    codes, sc = orc.mxfp8_quantize_swizzled(bits, b, m, k)
    rng = np.random.default_rng(b * m + k)
    rcodes = rng.integers(0, 256, codes.size, dtype=np.uint8)
    rcodes[(rcodes & 0x7F) == 0x7F] = 0x41
    rsc = rng.integers(0, 255, sc.size, dtype=np.uint8)
    for cc, ss in ((codes, sc), (rcodes, rsc)):
        dc = torch.from_numpy(cc.reshape(b, m, k).copy()).cuda()
        ds = torch.from_numpy(ss.copy()).cuda()
        out = w.mxfp8_dequantize_swizzled(dc, ds)
        plain = w.mxfp8_unswizzle_scales(ds, b, m, k)
        torch.cuda.synchronize()
        assert_same(bits16(out).ravel(), orc.mxfp8_dequantize(cc, ss, b, m, k), "dequantized weights")
        assert_same(u8(plain).ravel(), orc.mxfp8_unswizzle(ss, b, m, k), "row-major scales")


@pytest.mark.parametrize("b,m,k", [(30, 200, 4000), (40, 768, 2048)])
def test_mxfp8_dequantize_many_tiles_per_cta(w, orc, b, m, k):
    # more tiles than three per CTA, so every shared-memory stage is refilled;
    # (30, 200, 4000): rows past each matrix's end and a partial column tile
    rng = np.random.default_rng(m + k)
    codes = rng.integers(0, 256, b * m * k, dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3A
    sb = w.mxfp8_swizzled_scale_bytes(b, m, k)
    sc = rng.integers(100, 140, sb, dtype=np.uint8)
    out = w.mxfp8_dequantize_swizzled(torch.from_numpy(codes.reshape(b, m, k)).cuda(), torch.from_numpy(sc).cuda())
    torch.cuda.synchronize()
    assert_same(bits16(out).ravel(), orc.mxfp8_dequantize(codes, sc, b, m, k), "dequantized weights")


def test_count_mismatches(w, orc):
    rng = np.random.default_rng(5)
    for n in (1, 15, 16, 17, 4096 + 7, 3_000_001):
        a = rng.integers(0, 256, n, dtype=np.uint8)
        b = a.copy()
        flip = rng.choice(n, size=min(n, 1 + n // 1000), replace=False)
        b[flip] ^= rng.integers(1, 256, flip.size, dtype=np.uint8)
        got = w.fp8q_count_mismatches(torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda())
        same = w.fp8q_count_mismatches(torch.from_numpy(a).cuda(), torch.from_numpy(a).cuda())
        assert int(got.item()) == orc.count_mismatches(a, b) == flip.size
        assert int(same.item()) == 0
