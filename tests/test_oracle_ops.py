"""Pins for the oracle's four operations: blockwise quantize, fused
dequant-reduce, ring hop and MXFP8 prequantization with the scale swizzle.

Nothing here re-types the oracle's formulas.  Expected values come from
hand-worked fixtures (tests/golden/), exact rational arithmetic
(fractions.Fraction) with the fp32 rounding-error bounds, torch's float8
conversion on power-of-two scalings (which are exact), and invariants that
follow from the definitions.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

from conftest import read_golden

U = Fraction(1, 2 ** 24)          # unit roundoff of binary32
FMAX = {0: 448.0, 1: 57344.0}
MAXC = {0: 0x7E, 1: 0x7B}
TD = {0: torch.float8_e4m3fn, 1: torch.float8_e5m2}


def bf16_bits(f32):
    return torch.from_numpy(np.asarray(f32, np.float32).copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_val(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def torch_fp8(fmt, v):
    """torch's RNE conversion (values must be within the format's range)."""
    return torch.from_numpy(np.asarray(v, np.float32).copy()).to(TD[fmt]).view(torch.uint8).numpy()


def torch_fp8_decode(fmt, c):
    return torch.from_numpy(np.asarray(c, np.uint8).copy()).view(TD[fmt]).float().numpy()


def fp8_half_ulp(fmt, q):
    """Half an ulp of the FP8 grid at |q| (exact Fraction)."""
    m = 3 if fmt == 0 else 2
    emin = -6 if fmt == 0 else -14
    q = abs(Fraction(q))
    if q == 0:
        e = emin
    else:
        e = q.numerator.bit_length() - q.denominator.bit_length()
        if Fraction(2) ** e > q:
            e -= 1
        e = max(e, emin)
    return Fraction(2) ** (e - m) / 2


# ------------------------------------------------------------ quantize ----
@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("j", [-30, -12, 0, 5])
def test_quantize_power_of_two_scale_block(orc, fmt, j):
    # amax = Fmax * 2^j gives s = 2^j exactly, so the codes are the plain
    # conversion of x * 2^-j, which torch computes independently.
    rng = np.random.default_rng(100 + j + 7 * fmt)
    x = (rng.standard_normal(128) * FMAX[fmt] * 2.0 ** j / 4).astype(np.float32)
    x = np.clip(x, -FMAX[fmt] * 2.0 ** j, FMAX[fmt] * 2.0 ** j)
    x[17] = -FMAX[fmt] * 2.0 ** j
    xb = bf16_bits(x)
    xv = bf16_val(xb)
    codes, scales = orc.quantize_blockwise(xb, fmt)
    assert scales[0] == np.float32(2.0 ** j)
    assert np.array_equal(codes, torch_fp8(fmt, xv * np.float32(2.0 ** -j)))


@pytest.mark.parametrize("fmt", [0, 1])
def test_quantize_amax_invariant_and_error_bound(orc, fmt):
    rng = np.random.default_rng(11 + fmt)
    n = 128 * 40 + 37                 # ragged tail
    mags = 10.0 ** rng.uniform(-30, 30, size=(n + 127) // 128)
    x = rng.standard_normal(n) * np.repeat(mags, 128)[:n]
    xb = bf16_bits(x.astype(np.float32))
    xv = bf16_val(xb)
    codes, scales = orc.quantize_blockwise(xb, fmt)
    assert scales.size == (n + 127) // 128
    dec = torch_fp8_decode(fmt, codes)
    for b in range(scales.size):
        blk = slice(128 * b, min(n, 128 * b + 128))
        amax = np.abs(xv[blk]).max()
        s = Fraction(float(scales[b]))
        # s is amax/Fmax rounded once to binary32
        assert abs(s - Fraction(float(amax)) / Fraction(FMAX[fmt])) <= U * Fraction(float(amax)) / Fraction(FMAX[fmt])
        if s >= Fraction(2) ** -126:
            # the block's largest element lands on the largest code
            assert (codes[blk] & 0x7F).max() == MAXC[fmt]
        for i in range(blk.start, blk.stop, 7):
            q = Fraction(float(xv[i])) / s
            if abs(q) >= FMAX[fmt]:
                assert codes[i] & 0x7F == MAXC[fmt]
                continue
            err = abs(Fraction(float(dec[i])) - q)
            assert err <= fp8_half_ulp(fmt, q) + U * abs(q), (b, i)
            assert np.signbit(dec[i]) == np.signbit(xv[i]) or dec[i] == 0


def _blocks_of_all_bf16_below(amax_bits):
    """Blocks of 128 bf16 values: every bf16 pattern with |x| <= amax, each
    block led by amax itself so that every block has the same scale."""
    h = np.arange(65536, dtype=np.uint16)
    v = bf16_val(h)
    amax = bf16_val(np.array([amax_bits], np.uint16))[0]
    keep = np.isfinite(v) & (np.abs(v) <= amax)
    xs = h[keep]
    nblk = (xs.size + 126) // 127
    xs = np.concatenate([xs, np.zeros(nblk * 127 - xs.size, np.uint16)]).reshape(nblk, 127)
    return np.concatenate([np.full((nblk, 1), amax_bits, np.uint16), xs], axis=1).ravel()


@pytest.mark.parametrize("fmt", [0, 1])
def test_quantize_is_true_division_over_all_bf16_inputs(orc, fmt):
    # For a set of block amax values, every bf16 x in the block's range.  The
    # expected quotient is x / s rounded once to binary32, obtained here from
    # a float64 division (correctly rounded) then a cast to float32: double
    # rounding 53 -> 24 bits is innocuous for a quotient of 24-bit operands
    # (Figueroa, "When is double rounding innocuous?", 1995).  A multiply by
    # the reciprocal of s differs from it near FP8 rounding boundaries.
    rng = np.random.default_rng(500 + fmt)
    amaxes = list(rng.integers(0x0080, 0x7F7F, size=24)) + [0x3F80, 0x0001, 0x0003, 0x7F7F, 0x3A83]
    for ab in amaxes:
        x = _blocks_of_all_bf16_below(np.uint16(ab))
        codes, scales = orc.quantize_blockwise(x, fmt)
        assert (scales == scales[0]).all()
        s = np.float64(scales[0])
        q = (bf16_val(x).astype(np.float64) / s).astype(np.float32)
        q = np.clip(q, -FMAX[fmt], FMAX[fmt])
        assert np.array_equal(codes, torch_fp8(fmt, q)), hex(ab)


@pytest.mark.parametrize("fmt", [0, 1])
def test_quantize_zero_blocks_and_signed_zeros(orc, fmt):
    x = np.zeros(300, np.float32)
    x[128:256] = np.linspace(-1, 1, 128)
    x[5] = -0.0
    xb = bf16_bits(x)
    codes, scales = orc.quantize_blockwise(xb, fmt)
    assert scales[0] == 0.0 and scales[2] == 0.0 and scales[1] > 0
    assert codes[5] == 0x80 and codes[4] == 0x00
    assert (codes[256:] == 0).all()


def test_quantize_tail_block_is_independent(orc):
    rng = np.random.default_rng(3)
    x = bf16_bits(rng.standard_normal(128 * 3 + 5).astype(np.float32))
    c_all, s_all = orc.quantize_blockwise(x, 0)
    for b in range(4):
        c, s = orc.quantize_blockwise(x[128 * b:128 * b + 128].copy(), 0)
        assert s[0] == s_all[b]
        assert np.array_equal(c, c_all[128 * b:128 * b + 128])


def test_quantize_n1(orc):
    c, s = orc.quantize_blockwise(bf16_bits([-3.0]), 0)
    assert s[0] == np.float32(3.0) / np.float32(448.0) and c[0] == 0xFE


def test_wire_bytes_closed_form():
    d = {r[0]: float(r[1]) for r in read_golden("wire_bytes.txt")}
    per_elem = 1 + 4 / 128                         # one fp32 scale per 128 codes
    assert per_elem == d["blockwise_bytes_per_element"]
    saving = 1 - per_elem / d["bf16_bytes_per_element"]
    assert saving == d["saving_fraction"]
    assert round(100 * saving, 1) == d["saving_percent_printed"]
    p = d["ring_allreduce_ranks"]
    assert 2 * (p - 1) / p * d["ring_allreduce_gb_payload"] == d["ring_allreduce_gb_moved"]


# ------------------------------------------------------ dequant-reduce ----
def test_reduce_hand_example(orc):
    # shard 0: code 0x38 (1.0) scale 1; shard 1: code 0x40 (2.0) scale 0.5 -> 2.0
    c0 = np.full(128, 0x38, np.uint8)
    c1 = np.full(128, 0x40, np.uint8)
    ob, of = orc.dequant_reduce([c0, c1], [np.array([1.0], np.float32), np.array([0.5], np.float32)], 0)
    assert (of == 2.0).all() and (ob == 0x4000).all()


def test_reduce_is_rank_ordered(orc):
    # d0 = 2^24, d1 = 1, d2 = -2^24: (2^24 + 1) ties back to 2^24 (even), so the
    # rank-order sum is 0; any other order that adds d1 last gives 1.
    c = np.full(128, 0x38, np.uint8)
    cn = np.full(128, 0xB8, np.uint8)
    s_big = np.array([2.0 ** 24], np.float32)
    s_one = np.array([1.0], np.float32)
    _, of = orc.dequant_reduce([c, c, cn], [s_big, s_one, s_big], 0)
    assert (of == 0.0).all()
    _, of2 = orc.dequant_reduce([c, cn, c], [s_big, s_big, s_one], 0)
    assert (of2 == 1.0).all()


def test_reduce_starts_from_positive_zero(orc):
    c = np.full(128, 0x80, np.uint8)        # -0.0 in e4m3
    ob, of = orc.dequant_reduce([c, c], [np.ones(1, np.float32)] * 2, 0)
    assert (of.view(np.uint32) == 0).all() and (ob == 0).all()


@pytest.mark.parametrize("k", [1, 2, 4, 8, 16])
def test_reduce_identical_power_of_two_shards_exact(orc, k):
    rng = np.random.default_rng(k)
    c = rng.integers(0, 256, 1000, dtype=np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x10                       # no NaN codes
    s = (2.0 ** rng.integers(-20, 20, 8)).astype(np.float32)
    ob, of = orc.dequant_reduce([c] * k, [s] * k, 0)
    expect = torch_fp8_decode(0, c) * np.repeat(s, 128)[:1000] * k
    assert np.array_equal(of, expect.astype(np.float32))
    assert np.array_equal(ob, bf16_bits(of))


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("k", [2, 3, 8])
def test_reduce_within_recursive_summation_bound(orc, fmt, k):
    rng = np.random.default_rng(40 + k + fmt)
    n = 128 * 6 + 9
    nb = (n + 127) // 128
    codes, scales = [], []
    for r in range(k):
        c = rng.integers(0, 256, n, dtype=np.uint8)
        dec = torch_fp8_decode(fmt, c)
        c[~np.isfinite(dec)] = 0x21
        codes.append(c)
        # scales spread over many binades so a wrong block or shard index shows
        scales.append((10.0 ** rng.uniform(-8, 8, nb)).astype(np.float32))
    ob, of = orc.dequant_reduce(codes, scales, fmt)
    g = (k - 1) * U / (1 - (k - 1) * U)
    for i in range(0, n, 5):
        terms = [Fraction(float(torch_fp8_decode(fmt, codes[r][i:i + 1])[0])) * Fraction(float(scales[r][i // 128]))
                 for r in range(k)]
        exact = sum(terms, Fraction(0))
        bound = (g + U * (1 + g)) * sum(abs(t) for t in terms)
        assert abs(Fraction(float(of[i])) - exact) <= bound, i
    assert np.array_equal(ob, bf16_bits(of))


def test_dequantize_power_of_two(orc):
    rng = np.random.default_rng(9)
    c = rng.integers(0, 256, 384, dtype=np.uint8)
    c[(c & 0x7F) == 0x7F] = 0
    s = np.array([0.25, 2.0 ** 40, 2.0 ** -60], np.float32)
    _, of = orc.dequantize(c, s, 0)
    assert np.array_equal(of, (torch_fp8_decode(0, c) * np.repeat(s, 128)).astype(np.float32))


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("ranks", [2, 3, 5, 7, 8, 16])
def test_dequantize_mean_is_one_true_division(orc, fmt, ranks):
    # The product decode(c) * s is exact in float64 and the quotient of two
    # binary32 values rounded to float64 and then to binary32 equals the
    # single binary32 rounding (53 >= 2*24 + 2; Figueroa 1995).  The scales
    # span normal and subnormal binary32 quotients; a multiply by RN(1/P)
    # instead of the division, a division of the bf16 value, or a dropped
    # divisor each fail here.
    rng = np.random.default_rng(70 + 10 * fmt + ranks)
    n = 128 * 48
    c = rng.integers(0, 256, n, dtype=np.uint8)
    dec = torch_fp8_decode(fmt, c)
    c[~np.isfinite(dec)] = 0x21
    dec = torch_fp8_decode(fmt, c)
    s = (2.0 ** rng.uniform(-140, 40, n // 128)).astype(np.float32)
    s[:4] = [0.0, 1.0, 2.0 ** -126, 2.0 ** -149]
    ob, of = orc.dequantize_mean(c, s, fmt, ranks)
    d = (dec.astype(np.float64) * np.repeat(s, 128).astype(np.float64)).astype(np.float32)
    q = (d.astype(np.float64) / ranks).astype(np.float32)
    assert np.array_equal(of.view(np.uint32), q.view(np.uint32))
    assert np.array_equal(ob, bf16_bits(q))
    if ranks == 3:
        # a hand case: 0x38 (1.0) at s = 1.5 is 1.5, and 1.5 / 3 = 0.5 exactly
        ob1, of1 = orc.dequantize_mean(np.array([0x38 if fmt == 0 else 0x3C], np.uint8),
                                       np.array([1.5], np.float32), fmt, 3)
        assert of1[0] == 0.5 and ob1[0] == 0x3F00


@pytest.mark.parametrize("fmt", [0, 1])
def test_dequantize_mean_by_one_is_dequantize(orc, fmt):
    rng = np.random.default_rng(80 + fmt)
    c = rng.integers(0, 256, 128 * 9 + 5, dtype=np.uint8)
    s = (2.0 ** rng.uniform(-100, 30, 10)).astype(np.float32)
    ob, of = orc.dequantize(c, s, fmt)
    mb, mf = orc.dequantize_mean(c, s, fmt, 1)
    assert np.array_equal(ob, mb) and np.array_equal(of.view(np.uint32), mf.view(np.uint32))


# ------------------------------------------------------------ ring hop ----
@pytest.mark.parametrize("fmt", [0, 1])
def test_ring_hop_zero_local_is_requant_identity(orc, fmt):
    # power-of-two scales: dequant is exact and requant reproduces the input
    rng = np.random.default_rng(21 + fmt)
    n = 128 * 8 + 30
    x = rng.standard_normal(n).astype(np.float32) * np.float32(FMAX[fmt] / 3)
    x = np.clip(x, -FMAX[fmt], FMAX[fmt])
    x[::128] = FMAX[fmt]                                   # amax = Fmax -> s = 1
    xb = bf16_bits(x * np.float32(2.0 ** -7))              # s = 2^-7 in every block
    c, s = orc.quantize_blockwise(xb, fmt)
    assert (s == np.float32(2.0 ** -7)).all()
    oc, os_, ob = orc.ring_hop(c, s, np.zeros(n, np.uint16), fmt)
    assert np.array_equal(os_, s) and np.array_equal(oc, c)


@pytest.mark.parametrize("fmt", [0, 1])
def test_ring_hop_matches_quantize_of_exact_sum(orc, fmt):
    # inputs on coarse grids so that d + local is exact and bf16-representable;
    # then the hop must equal blockwise quantize of that sum (pinned above).
    rng = np.random.default_rng(31 + fmt)
    n = 128 * 5 + 77
    nb = (n + 127) // 128
    in_codes = rng.choice(np.array([0x30, 0x38, 0x40, 0x44, 0xB8, 0xC0, 0x00], np.uint8), n)
    in_scales = (2.0 ** rng.integers(-10, 3, nb)).astype(np.float32)
    loc = rng.integers(-8, 9, n).astype(np.float32) * np.repeat(in_scales, 128)[:n]
    locb = bf16_bits(loc)
    d = torch_fp8_decode(fmt, in_codes) * np.repeat(in_scales, 128)[:n]
    y = (d + bf16_val(locb)).astype(np.float32)
    yb = bf16_bits(y)
    assert np.array_equal(bf16_val(yb), y)                # exact by construction
    oc, os_, ob = orc.ring_hop(in_codes, in_scales, locb, fmt)
    qc, qs = orc.quantize_blockwise(yb, fmt)
    assert np.array_equal(ob, yb)
    assert np.array_equal(os_, qs) and np.array_equal(oc, qc)


@pytest.mark.parametrize("fmt", [0, 1])
def test_ring_hop_requantizes_the_fp32_sum_by_true_division(orc, fmt):
    # Every rounding of the hop evaluated in float64 and cast once to float32:
    # a product of a 4-bit and a 24-bit significand is exact in float64, and a
    # sum or quotient of two binary32 values rounded to float64 first and then
    # to binary32 equals the single binary32 rounding (53 >= 2*24 + 2;
    # Figueroa 1995).  This catches requantizing RNE_bf16(y) instead of y, and
    # a multiply by the reciprocal of the scale instead of the division.
    rng = np.random.default_rng(61 + fmt)
    n = 128 * 64
    nb = n // 128
    in_codes = rng.integers(0, 256, n, dtype=np.uint8)
    dec = torch_fp8_decode(fmt, in_codes)
    in_codes[~np.isfinite(dec)] = 0x11
    dec = torch_fp8_decode(fmt, in_codes)
    in_scales = (10.0 ** rng.uniform(-6, -2, nb)).astype(np.float32)
    locb = bf16_bits((rng.standard_normal(n) * 1e-3).astype(np.float32))
    oc, os_, ob = orc.ring_hop(in_codes, in_scales, locb, fmt)
    d = (dec.astype(np.float64) * np.repeat(in_scales, 128).astype(np.float64)).astype(np.float32)
    y = (d.astype(np.float64) + bf16_val(locb).astype(np.float64)).astype(np.float32)
    assert np.array_equal(ob, bf16_bits(y))
    amax = np.abs(y.reshape(nb, 128)).max(axis=1)
    sc = (amax.astype(np.float64) / FMAX[fmt]).astype(np.float32)
    assert np.array_equal(os_, sc)
    q = (y.astype(np.float64) / np.repeat(sc, 128).astype(np.float64)).astype(np.float32)
    q = np.clip(q, -FMAX[fmt], FMAX[fmt])
    assert np.array_equal(oc, torch_fp8(fmt, q))


def test_ring_hop_division_on_fp8_rounding_boundaries(orc):
    # Blocks searched so that RN(y / s) and RN(y * RN(1/s)) fall on different
    # sides of an e4m3 rounding boundary for some element; the hop must give
    # the true-division code there (expected values as in the test above).
    # Element 0 carries code 0x7E (the block amax, 448 * s_in); the others
    # carry 1.0 * s_in plus a bf16 local near 0.0625 * s_in, which puts y / s
    # next to the e4m3 midpoint 1.0625.
    rng = np.random.default_rng(71)
    rows = 800_000
    s_in = (10.0 ** rng.uniform(-6, 0, rows)).astype(np.float32)
    base = bf16_bits(np.float32(0.0625) * s_in).astype(np.int32)
    offs = np.arange(-8, 9, dtype=np.int32)
    loc = (base[:, None] + offs[None, :]).astype(np.uint16)            # 17 bf16 neighbours
    y = np.empty((rows, 18), np.float32)
    y[:, 0] = (448.0 * s_in.astype(np.float64)).astype(np.float32)
    y[:, 1:] = (s_in[:, None].astype(np.float64) + bf16_val(loc).astype(np.float64)).astype(np.float32)
    sc = (y[:, 0].astype(np.float64) / 448.0).astype(np.float32)
    q_true = (y.astype(np.float64) / sc[:, None].astype(np.float64)).astype(np.float32)
    q_recip = (y * (np.float32(1.0) / sc)[:, None]).astype(np.float32)
    c_true = torch_fp8(0, np.clip(q_true, 0, 448).ravel()).reshape(y.shape)
    c_recip = torch_fp8(0, np.clip(q_recip, 0, 448).ravel()).reshape(y.shape)
    hit = np.unique(np.nonzero(c_true != c_recip)[0])[:64]
    assert hit.size >= 12, f"search found {hit.size} boundary cases"
    in_codes = np.zeros((hit.size, 128), np.uint8)
    in_codes[:, 0] = 0x7E
    in_codes[:, 1:18] = 0x38
    local = np.zeros((hit.size, 128), np.uint16)
    local[:, 1:18] = loc[hit]
    oc, os_, _ = orc.ring_hop(in_codes.ravel(), s_in[hit], local.ravel(), 0)
    assert np.array_equal(os_, sc[hit])
    assert np.array_equal(oc.reshape(hit.size, 128)[:, :18], c_true[hit])


def test_ring_chain_tracks_exact_sum(orc):
    # 8 partials, hop 0 = quantize, hops 1..7 add one partial each; the final
    # bf16 stays within the accumulated e4m3 quantization error of the sum.
    rng = np.random.default_rng(8)
    n = 128 * 4 + 11
    parts = [bf16_bits((rng.standard_normal(n) * 1e-3).astype(np.float32)) for _ in range(8)]
    c, s = orc.quantize_blockwise(parts[0], 0)
    bound = np.repeat(s, 128)[:n].astype(np.float64) * 16     # half an e4m3 ulp at the top is 16 * s
    for h in range(1, 8):
        c, s, ob = orc.ring_hop(c, s, parts[h], 0)
        bound += np.repeat(s, 128)[:n] * 16
    exact = np.sum([bf16_val(p).astype(np.float64) for p in parts], axis=0)
    final = bf16_val(ob).astype(np.float64)
    assert (np.abs(final - exact) <= bound + np.abs(exact) * 2.0 ** -8).all()


# ----------------------------------------------------------- MXFP8 --------
def test_mxfp8_golden_blocks(orc):
    rows = read_golden("mxfp8_worked.txt")
    assert len(rows) >= 8
    for amax_tok, e_hex, code_hex, *_ in rows:
        amax = float.fromhex(amax_tok) if "0x" in amax_tok else float(amax_tok)
        w = np.zeros(32, np.float32)
        w[9] = amax
        w[3] = -amax / 4
        w[20] = amax / 3
        wb = bf16_bits(w)
        assert bf16_val(wb)[9] == np.float32(amax), amax_tok
        codes, e = orc.mxfp8_block(wb)
        assert e == int(e_hex, 16), amax_tok
        assert codes[9] == int(code_hex, 16), amax_tok
        assert orc.e8m0_of_amax(amax) == int(e_hex, 16)


def test_mxfp8_exponent_brackets_amax(orc):
    # for every positive finite bf16 amax whose e is not clamped, the scaled
    # amax lands in [256, 512): e is floor(log2 amax) - 8 + 127.
    h = np.arange(1, 0x7F80, dtype=np.uint16)
    a = bf16_val(h)
    for i in range(0, h.size, 3):
        e = orc.e8m0_of_amax(float(a[i]))
        t = Fraction(float(a[i])) * Fraction(2) ** (127 - e)
        if e > 0:
            assert Fraction(256) <= t < Fraction(512), float(a[i])
        else:
            assert t < Fraction(512)


def test_mxfp8_codes_match_torch_after_power_of_two_scaling(orc):
    rng = np.random.default_rng(12)
    m, k = 64, 256
    w = (rng.standard_normal((m, k)) * 0.02).astype(np.float32)
    w[rng.random(m) < 0.1] *= 50
    w[3, 32:64] = 0.0
    wb = bf16_bits(w.ravel())
    codes, sc = orc.mxfp8_quantize_swizzled(wb, 1, m, k)
    wv = bf16_val(wb).reshape(m, k)
    cv = codes.reshape(m, k)
    for r in range(m):
        for j in range(k // 32):
            e = sc[orc.swizzle_offset(0, r, j, m, k // 32)]
            blk = wv[r, 32 * j:32 * j + 32]
            t = (blk.astype(np.float64) * 2.0 ** (127 - int(e))).astype(np.float32)
            t = np.clip(t, -448, 448)                       # satfinite
            assert np.array_equal(cv[r, 32 * j:32 * j + 32], torch_fp8(0, t)), (r, j)
            if np.abs(blk).max() == 0:
                assert e == 0
            elif e > 0:
                assert 0x78 <= (cv[r, 32 * j:32 * j + 32] & 0x7F).max() <= 0x7E


def test_swizzle_hand_table(orc):
    rows = read_golden("swizzle_m256_kb8.txt")
    for bt, r, j, off in rows:
        assert orc.swizzle_offset(int(bt), int(r), int(j), 256, 8) == int(off)
    assert orc.swizzled_scale_bytes(2, 256, 256) == 4096


@pytest.mark.parametrize("m,kb", [(256, 8), (129, 3), (1, 1), (384, 24), (128, 64)])
def test_swizzle_is_a_bijection_onto_the_unpadded_cells(orc, m, kb):
    total = orc.swizzled_scale_bytes(2, m, kb * 32)
    seen = set()
    for bt in range(2):
        for r in range(m):
            for j in range(kb):
                off = orc.swizzle_offset(bt, r, j, m, kb)
                assert 0 <= off < total
                seen.add(off)
    assert len(seen) == 2 * m * kb
    if m % 128 == 0 and kb % 4 == 0:
        assert len(seen) == total                     # no padding: onto


def tiled_128x4(nat, m, kb):
    """The block-scaled GEMM scale layout written as array reshapes (NVIDIA
    cuBLAS documentation, "1D Block Scaling Factors Layout"): a [rows, K/32]
    scale matrix is zero-padded to whole 128 x 4 tiles; tile (row tile a,
    column tile b) holds 32 lines of 16 bytes, line i carrying, for rows
    i, i + 32, i + 64 and i + 96 of the row tile, their 4 scales; tiles are
    stored row tile by row tile.  nat: [batch, m, kb] -> flat [batch, ...]."""
    bt = nat.shape[0]
    mp, kp = -(-m // 128) * 128, -(-kb // 4) * 4
    pad = np.zeros((bt, mp, kp), nat.dtype)
    pad[:, :m, :kb] = nat
    # row = a*128 + g*32 + i, column = b*4 + c  ->  order (a, b, i, g, c)
    t = pad.reshape(bt, mp // 128, 4, 32, kp // 4, 4).transpose(0, 1, 4, 3, 2, 5)
    return t.reshape(-1)


@pytest.mark.parametrize("bt,m,kb", [(1, 1, 1), (2, 129, 3), (1, 256, 8), (2, 384, 24), (1, 200, 64)])
def test_swizzle_equals_the_reshape_form_of_128x4_tiles(orc, bt, m, kb):
    ids = np.arange(1, bt * m * kb + 1, dtype=np.int64).reshape(bt, m, kb)
    want = tiled_128x4(ids, m, kb)
    got = np.zeros(orc.swizzled_scale_bytes(bt, m, kb * 32), np.int64)
    for b in range(bt):
        for r in range(m):
            for j in range(kb):
                got[orc.swizzle_offset(b, r, j, m, kb)] = ids[b, r, j]
    assert np.array_equal(got, want)


def test_swizzled_scales_are_the_reshape_form_of_the_row_major_exponents(orc):
    # the whole scale buffer of a ragged batch: the E8M0 byte of each
    # 32-block, from the block amax alone, laid out by the reshape form
    rng = np.random.default_rng(11)
    bt, m, k = 2, 200, 96
    x = (rng.standard_normal((bt, m, k)) * np.exp2(rng.integers(-20, 20, (bt, m, 1)))).astype(np.float32)
    x[0, 3, 32:64] = 0.0                                      # a zero block
    w = bf16_bits(x.ravel())
    amax = np.abs(bf16_val(w).reshape(bt, m, k // 32, 32)).max(axis=3)
    nat = np.vectorize(orc.e8m0_of_amax)(amax).astype(np.int64)
    assert nat[0, 3, 1] == 0
    _, sc = orc.mxfp8_quantize_swizzled(w, bt, m, k)
    assert np.array_equal(sc.astype(np.int64), tiled_128x4(nat, m, k // 32))


def test_mxfp8_k32_keeps_its_scale_column_and_zero_padding(orc):
    # K == 32: one real scale column, padded to a 4-wide tile with zeros
    rng = np.random.default_rng(4)
    m = 130
    w = bf16_bits((rng.standard_normal(m * 32) + 3).astype(np.float32))
    codes, sc = orc.mxfp8_quantize_swizzled(w, 1, m, 32)
    assert sc.size == 2 * 512
    real = {orc.swizzle_offset(0, r, 0, m, 1) for r in range(m)}
    for off in range(sc.size):
        if off not in real:
            assert sc[off] == 0
        else:
            assert sc[off] != 0


def test_mxfp8_batch_equals_flattened_rows_when_m_is_tile_aligned(orc):
    rng = np.random.default_rng(6)
    b, m, k = 3, 128, 96
    w = bf16_bits((rng.standard_normal(b * m * k) * 0.02).astype(np.float32))
    c3, s3 = orc.mxfp8_quantize_swizzled(w, b, m, k)
    c2, s2 = orc.mxfp8_quantize_swizzled(w, 1, b * m, k)
    assert np.array_equal(c3, c2) and np.array_equal(s3, s2)


def test_mxfp8_codes_to_scales_ratio(orc):
    # "a prequantized weight is ~32x its scale": 1 byte per element, 1 per block
    m, k = 768, 2048
    assert (m * k) / orc.swizzled_scale_bytes(1, m, k) == 32


def test_mxfp8_rejects_k_not_multiple_of_32(orc):
    with pytest.raises(ValueError):
        orc.mxfp8_quantize_swizzled(np.zeros(48, np.uint16), 1, 1, 48)


# ----------------------------------------------------- MXFP8 receiver -----
def test_mxfp8_dequantize_is_exact_power_of_two_scaling(orc):
    # every code times 2^(e-127), computed in float64 from torch's e4m3
    # decode and cast to bf16 by torch, for many scale bytes
    rng = np.random.default_rng(81)
    b, m, k = 2, 130, 96
    codes = rng.integers(0, 256, b * m * k, dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3C
    kb = k // 32
    plain = rng.integers(0, 255, b * m * kb, dtype=np.uint8)
    sc = np.zeros(orc.swizzled_scale_bytes(b, m, k), np.uint8)
    for bt in range(b):
        for r in range(m):
            for j in range(kb):
                sc[orc.swizzle_offset(bt, r, j, m, kb)] = plain[(bt * m + r) * kb + j]
    got = orc.mxfp8_dequantize(codes, sc, b, m, k)
    e = np.repeat(plain.astype(np.int64), 32)
    val = torch_fp8_decode(0, codes).astype(np.float64) * np.exp2(e - 127.0)
    want = torch.from_numpy(val.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)
    assert np.array_equal(orc.mxfp8_unswizzle(sc, b, m, k), plain)


def test_mxfp8_round_trip_within_half_ulp(orc):
    rng = np.random.default_rng(82)
    m, k = 64, 256
    w = (rng.standard_normal(m * k) * 0.02).astype(np.float32)
    wb = bf16_bits(w)
    codes, sc = orc.mxfp8_quantize_swizzled(wb, 1, m, k)
    back = bf16_val(orc.mxfp8_dequantize(codes, sc, 1, m, k)).astype(np.float64)
    wv = bf16_val(wb).astype(np.float64)
    e = orc.mxfp8_unswizzle(sc, 1, m, k).astype(np.int64)
    unit = np.exp2(np.repeat(e, 32) - 127.0)            # the block's 2^(e-127)
    scaled = np.abs(wv) / unit                           # in [0, 512)
    # |error| <= half an e4m3 ulp of the scaled value (<= 16 below 512), or
    # the saturation above 448, times the scale
    bound = np.maximum(16.0, scaled - 448.0) * unit
    assert (np.abs(back - wv) <= bound + 2.0 ** -133).all()
    assert (scaled < 512).all()


def test_count_mismatches(orc):
    a = np.arange(1000, dtype=np.uint32).astype(np.uint8)
    b = a.copy()
    b[[3, 500, 999]] ^= 1
    assert orc.count_mismatches(a, a) == 0 and orc.count_mismatches(a, b) == 3


# --------------------------------------------------------- NEXT variants --
@pytest.mark.parametrize("fmt", [0, 1])
def test_tensorwise_equals_blockwise_on_one_block(orc, fmt):
    # with n <= 128 the tensor is one block: both recipes must agree
    for n in (1, 77, 128):
        xb = bf16_bits((np.random.default_rng(n).standard_normal(n) * 3e-3).astype(np.float32))
        c1, s1 = orc.quantize_blockwise(xb, fmt)
        c2, s2, a2 = orc.quantize_tensorwise(xb, fmt)
        assert np.array_equal(c1, c2) and s1[0] == s2
        assert a2 == np.abs(bf16_val(xb)).max()


@pytest.mark.parametrize("fmt", [0, 1])
def test_tensorwise_power_of_two_scale(orc, fmt):
    # amax = Fmax * 2^-9 over many blocks -> s = 2^-9, codes are torch's
    # conversion of x * 2^9
    rng = np.random.default_rng(90 + fmt)
    x = np.clip(rng.standard_normal(5000) * FMAX[fmt] * 2.0 ** -11, -FMAX[fmt] * 2.0 ** -9, FMAX[fmt] * 2.0 ** -9)
    x[1234] = FMAX[fmt] * 2.0 ** -9
    xb = bf16_bits(x.astype(np.float32))
    codes, s, amax = orc.quantize_tensorwise(xb, fmt)
    assert s == np.float32(2.0 ** -9) and amax == np.float32(FMAX[fmt] * 2.0 ** -9)
    assert np.array_equal(codes, torch_fp8(fmt, bf16_val(xb) * np.float32(2.0 ** 9)))


def test_ring_hop_bf16_requant_equals_quantize_of_bf16_sum(orc):
    rng = np.random.default_rng(91)
    n = 128 * 9 + 5
    codes, scales = orc.quantize_blockwise(bf16_bits((rng.standard_normal(n) * 1e-3).astype(np.float32)), 0)
    loc = bf16_bits((rng.standard_normal(n) * 1e-3).astype(np.float32))
    oc, os_, ob = orc.ring_hop_bf16_requant(codes, scales, loc, 0)
    _, _, ob32 = orc.ring_hop(codes, scales, loc, 0)
    assert np.array_equal(ob, ob32)                      # same bf16 partial
    qc, qs = orc.quantize_blockwise(ob, 0)               # requantized from it
    assert np.array_equal(oc, qc) and np.array_equal(os_, qs)
