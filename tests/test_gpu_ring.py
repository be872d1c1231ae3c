"""(c) The ring hop on the GPU against the oracle: single hops on adversarial
inputs, and the 7-hop chain of a ring of 8 over the payload sweep."""
import numpy as np
import pytest
import torch

import gen
from gpu_util import Guarded, assert_same, assert_same_f32, bf16_from_bits, bits16, u8, varied_bf16
from test_gpu_reduce import random_shards

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w():
    import weight_transfer_gb300 as w
    return w


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("n", [1, 15, 16, 17, 127, 128, 129, 4096 + 17, 200_003])
@pytest.mark.parametrize("with_bf16", [True, False])
def test_single_hop(w, orc, fmt, n, with_bf16):
    codes, scales = random_shards(1, n, fmt, seed=n + 17 * fmt)
    # keep the incoming values in a range where adding the local partial
    # stays finite
    scales[0] = np.minimum(scales[0], np.float32(1e20))
    loc = varied_bf16(n, seed=n + 5)
    gc = Guarded(n, torch.uint8)
    gs = Guarded((n + 127) // 128, torch.float32)
    gb = Guarded(n, torch.bfloat16) if with_bf16 else None
    w.fp8q_ring_hop(torch.from_numpy(codes[0]).cuda(), torch.from_numpy(scales[0]).cuda(), bf16_from_bits(loc), fmt,
                    out_codes=gc.t, out_scales=gs.t, out_bf16=gb.t if gb else None)
    torch.cuda.synchronize()
    assert gc.intact() and gs.intact() and (gb is None or gb.intact())
    oc, os_, ob = orc.ring_hop(codes[0], scales[0], loc, fmt)
    assert_same_f32(gs.t.cpu().numpy(), os_, "scales")
    assert_same(u8(gc.t), oc, "codes")
    if gb:
        assert_same(bits16(gb.t), ob, "bf16")


def test_hop_in_place_local_update(w, orc):
    n = 100_000
    codes, scales = random_shards(1, n, 0, seed=4)
    scales[0] = np.minimum(scales[0], np.float32(1e20))
    loc = varied_bf16(n, seed=9)
    dloc = bf16_from_bits(loc)
    oc, os_, ob = w.fp8q_ring_hop(torch.from_numpy(codes[0]).cuda(), torch.from_numpy(scales[0]).cuda(), dloc, 0,
                                  out_bf16=dloc)
    ec, es, eb = orc.ring_hop(codes[0], scales[0], loc, 0)
    assert_same(bits16(dloc), eb, "in-place bf16")
    assert_same(u8(oc), ec, "codes")


def run_chain_gpu(w, parts, fmt):
    """hop 0 = quantize of partial 0; hops 1..7 add partials 1..7; the last
    hop also writes bf16.  Returns per-hop (codes, scales) and the final bf16."""
    hops = [w.fp8q_quantize_blockwise(parts[0], fmt)]
    last = None
    for h in range(1, len(parts)):
        c, s, b = w.fp8q_ring_hop(hops[-1][0], hops[-1][1], parts[h], fmt, want_bf16=h == len(parts) - 1)
        hops.append((c, s))
        last = b
    return hops, last


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("payload", [1 << p for p in range(10, 25)] + [767 * 1024])
def test_ring_chain_full_check(w, orc, fmt, payload):
    # per-hop payloads 1 KiB .. 16 MiB and 767 KiB, every element checked
    n = payload // 2
    host = [gen.ring_partial(r, n) for r in range(gen.RING_PARTIALS)]
    hops, last = run_chain_gpu(w, [p.cuda() for p in host], fmt)
    c, s = orc.quantize_blockwise(bits16(host[0]), fmt)
    for h in range(1, gen.RING_PARTIALS):
        assert_same(u8(hops[h - 1][0]), c, f"codes after hop {h - 1}")
        assert_same_f32(hops[h - 1][1].cpu().numpy(), s, f"scales after hop {h - 1}")
        c, s, b = orc.ring_hop(c, s, bits16(host[h]), fmt)
    assert_same(u8(hops[-1][0]), c, "final codes")
    assert_same(bits16(last), b, "final bf16")


@pytest.mark.parametrize("fmt,payload", [(0, 1 << 25), (0, 1 << 26), (0, 1 << 27), (0, 1 << 28), (1, 1 << 26),
                                         (1, 1 << 28)])
def test_ring_chain_large_sampled(w, orc, fmt, payload):
    # 32 MiB .. 256 MiB per-hop payloads, checked on sampled 128-blocks:
    # every hop is block-local, so the oracle replays the chain of a block
    # from that block's slice of the 8 partials
    n = payload // 2
    host = [gen.ring_partial(r, n) for r in range(gen.RING_PARTIALS)]
    hops, last = run_chain_gpu(w, [p.cuda() for p in host], fmt)
    nb = n // 128
    rng = np.random.default_rng(payload >> 20)
    blocks = np.unique(np.concatenate([rng.integers(0, nb, 400), [0, nb - 1]]))
    hb = [bits16(p) for p in host]
    gpu_codes = [u8(c) for c, _ in hops]
    gpu_scales = [s.cpu().numpy() for _, s in hops]
    gpu_last = bits16(last)
    for b in blocks:
        sl = slice(128 * b, 128 * b + 128)
        c, s = orc.quantize_blockwise(hb[0][sl].copy(), fmt)
        for h in range(1, gen.RING_PARTIALS):
            assert_same(gpu_codes[h - 1][sl], c, f"block {b} hop {h - 1}")
            assert gpu_scales[h - 1][b] == s[0]
            c, s, bf = orc.ring_hop(c, s, hb[h][sl].copy(), fmt)
        assert_same(gpu_codes[-1][sl], c, f"block {b} final")
        assert_same(gpu_last[sl], bf, f"block {b} bf16")


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("want_bf16", [True, False])
def test_hop_signed_zeros_and_cancellation(w, orc, fmt, want_bf16):
    # power-of-two block scales make every dequantized value exact in bf16,
    # so the local partial can cancel it exactly: sums of +0 from opposite
    # signs, -0 + -0, all-zero blocks after cancellation, zero scales,
    # subnormal sums and near-cancellation, over a ragged tail
    rng = np.random.default_rng(321 + fmt)
    nb = 96
    n = nb * 128 - 45
    codes = rng.integers(0, 256, n, dtype=np.uint8)
    nan_bits = 0x7F if fmt == 0 else 0x7C
    codes[(codes & nan_bits) == nan_bits] = 0x23
    kind = np.arange(nb) % 6
    scales = np.ldexp(np.float32(1.0), rng.integers(-60, 60, nb)).astype(np.float32)
    scales[kind == 3] = 0.0
    scales[kind == 4] = np.float32(2.0 ** -140)
    ek = np.repeat(kind, 128)[:n]
    zc = ek == 1
    codes[zc] = np.where(rng.random(zc.sum()) < 0.5, 0x00, 0x80).astype(np.uint8)
    a = orc.dequantize(codes, scales, fmt)[1]
    sz = np.where(rng.random(n) < 0.5, np.float32(0.0), np.float32(-0.0)).astype(np.float32)
    loc = np.where(ek == 0, -a, sz)
    half = (ek == 2) & (rng.random(n) < 0.5)
    loc = np.where(half, -a, np.where(ek == 2, rng.standard_normal(n).astype(np.float32) * np.abs(a), loc))
    loc = np.where(ek == 5, -a * np.float32(1.0078125), loc)
    lb = orc.f32_to_bf16(loc.astype(np.float32))
    assert np.array_equal(orc.bf16_to_f32(lb)[ek == 0], -a[ek == 0])      # the cancellation is exact
    dc, ds = torch.from_numpy(codes).cuda(), torch.from_numpy(scales).cuda()
    oc, os_, ob = w.fp8q_ring_hop(dc, ds, bf16_from_bits(lb), fmt, want_bf16=want_bf16)
    ec, es, eb = orc.ring_hop(codes, scales, lb, fmt)
    assert np.signbit(orc.bf16_to_f32(eb)).any() and (eb == 0).any()      # both zero signs occur
    assert_same_f32(os_.cpu().numpy(), es, "scales")
    assert_same(u8(oc), ec, "codes")
    if want_bf16:
        assert_same(bits16(ob), eb, "bf16")


def _near_boundary_blocks(orc, fmt, nblocks, seed):
    """Incoming codes, scales and local partials for `nblocks` blocks in which
    the quotients y / s (y the fp32 sums, s the block's new scale) lie within
    a few binary32 ulps of FP8 rounding boundaries, where a quotient one ulp
    off changes the code.  Element 0 of a block is a zero code with a bf16
    local A, which fixes the amax, so s = RN(A / Fmax).  The incoming scale is
    then s_in = RN(m * s / d) for a random code value d and a random midpoint
    m between two adjacent FP8 values: every code d * 2^j (either sign) of a
    lane decodes to a product within an ulp or two of m * 2^j * s, and the
    lane's local adds k ulps of that product (|k| <= 3, exact in bf16)."""
    rng = np.random.default_rng(seed)
    F = 448.0 if fmt == 0 else 57344.0
    min_normal = 2.0 ** (-6 if fmt == 0 else -14)
    vals = orc.decode(fmt, np.arange(0x80, dtype=np.uint8)).astype(np.float64)   # the positive codes, ascending
    fin = np.isfinite(vals)
    codes, scales, local = [], [], []
    for _ in range(nblocks):
        A = float(orc.bf16_to_f32(orc.f32_to_bf16(np.float32(rng.uniform(1, 2) * 2.0 ** int(rng.integers(-8, 8)))))[0])
        s = np.float32(np.float32(A) / np.float32(F))
        # a midpoint m between adjacent normal values below F / 4, a normal code value d
        lo_i = int(rng.choice(np.nonzero(fin & (vals >= min_normal) & (vals < F / 4))[0]))
        m = (vals[lo_i] + vals[lo_i + 1]) / 2
        d_i = int(rng.choice(np.nonzero(fin & (vals >= min_normal) & (vals <= F / 2))[0]))
        d = vals[d_i]
        s_in = np.float32(m * float(s) / d)
        # the lanes' codes: d * 2^j with m * 2^j in [min_normal, F / 2] and d * 2^j a normal code
        cand = [c for c in range(1, 0x7F) if fin[c] and vals[c] >= min_normal and
                (vals[c] / d) == 2.0 ** np.round(np.log2(vals[c] / d)) and
                min_normal <= m * vals[c] / d <= F / 2]
        assert cand
        lanes = rng.choice(cand, 127) | (rng.integers(0, 2, 127) << 7)
        p = (orc.decode(fmt, lanes.astype(np.uint8)) * s_in).astype(np.float32)
        ulp = np.spacing(np.abs(p)).astype(np.float32)
        k = rng.integers(-3, 4, 127).astype(np.float32)
        lb = orc.f32_to_bf16((k * ulp).astype(np.float32))
        assert np.array_equal(orc.bf16_to_f32(lb), (k * ulp).astype(np.float32))     # exact in bf16
        codes.append(np.concatenate([[0], lanes]).astype(np.uint8))
        local.append(np.concatenate([orc.f32_to_bf16(np.float32(A)), lb]).astype(np.uint16))
        scales.append(s_in)
    return np.concatenate(codes), np.array(scales, np.float32), np.concatenate(local)


@pytest.mark.parametrize("fmt", [0, 1])
def test_hop_quotients_near_fp8_boundaries(w, orc, fmt):
    # the hop's quotient y / s in the two-step reciprocal form must equal the
    # IEEE quotient wherever it decides a code: 48 staged blocks and a ragged
    # partial block, through the single-hop kernel and a group of two hops
    codes, scales, lb = _near_boundary_blocks(orc, fmt, 49, seed=77 + fmt)
    n = 48 * 128 + 77
    codes, lb = codes[:n], lb[:n]
    ec, es, eb = orc.ring_hop(codes, scales, lb, fmt)
    dc, ds, dl = torch.from_numpy(codes).cuda(), torch.from_numpy(scales).cuda(), bf16_from_bits(lb)
    oc, os_, ob = w.fp8q_ring_hop(dc, ds, dl, fmt, want_bf16=True)
    assert_same_f32(os_.cpu().numpy(), es, "scales")
    assert_same(u8(oc), ec, "codes")
    assert_same(bits16(ob), eb, "bf16")
    outs = w.fp8q_ring_hop_group([{"in_codes": dc, "in_scales": ds, "local": dl},
                                  {"in_codes": dc, "in_scales": ds, "local": dl, "want_bf16": True}], fmt)
    for gc, gs, gb in outs:
        assert_same_f32(gs.cpu().numpy(), es, "group scales")
        assert_same(u8(gc), ec, "group codes")
    assert_same(bits16(outs[1][2]), eb, "group bf16")
