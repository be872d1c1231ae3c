"""Pins for the oracle's element codecs (FP8 encode/decode, bf16 rounding).

Each test checks the oracle against something other than itself: the
hand-worked table in tests/golden/fp8_encodings.txt (OFP8 bit layouts),
a brute-force nearest-code search, and torch's own float8 / bfloat16
conversions (library routines that share nothing with the oracle).
"""
import math

import numpy as np
import pytest
import torch

from conftest import read_golden

FMT = {"e4m3": 0, "e5m2": 1}


def _val(tok):
    if tok in ("inf", "-inf"):
        return float(tok)
    return float.fromhex(tok) if "0x" in tok else float(tok)


def test_golden_encodings(orc):
    rows = read_golden("fp8_encodings.txt")
    assert len(rows) >= 40
    for fmt, val, code, *_ in rows:
        got = orc.encode(FMT[fmt], [_val(val)])[0]
        assert got == int(code, 16), f"{fmt} {val}: got {got:#04x}, want {code}"
        # the brute-force search must agree on every hand-worked case too
        assert orc.encode_brute(FMT[fmt], [_val(val)])[0] == int(code, 16)


@pytest.mark.parametrize("fmt,tdtype", [(0, torch.float8_e4m3fn), (1, torch.float8_e5m2)])
def test_decode_table_matches_torch(orc, fmt, tdtype):
    codes = np.arange(256, dtype=np.uint8)
    mine = orc.decode(fmt, codes)
    ref = torch.from_numpy(codes.copy()).view(tdtype).float().numpy()
    both_nan = np.isnan(mine) & np.isnan(ref)
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    assert np.array_equal(mine[~both_nan], ref[~both_nan])
    assert np.array_equal(np.signbit(mine[~both_nan]), np.signbit(ref[~both_nan]))


@pytest.mark.parametrize("fmt", [0, 1])
def test_decode_special_values(orc, fmt):
    d = orc.decode(fmt, np.arange(256, dtype=np.uint8))
    if fmt == 0:
        assert np.isnan(d[0x7F]) and np.isnan(d[0xFF]) and np.isnan(d).sum() == 2
        assert not np.isinf(d).any()
        assert d[0x7E] == 448.0 and d[0x01] == 2.0 ** -9 and d[0x08] == 2.0 ** -6
    else:
        assert np.isinf(d[0x7C]) and np.isinf(d[0xFC]) and np.isinf(d).sum() == 2
        assert np.isnan(d).sum() == 6
        assert d[0x7B] == 57344.0 and d[0x01] == 2.0 ** -16 and d[0x04] == 2.0 ** -14


@pytest.mark.parametrize("fmt", [0, 1])
def test_encode_decode_roundtrip(orc, fmt):
    codes = np.arange(256, dtype=np.uint8)
    vals = orc.decode(fmt, codes)
    finite = np.isfinite(vals)
    back = orc.encode(fmt, vals[finite])
    assert np.array_equal(back, codes[finite])


@pytest.mark.parametrize("fmt", [0, 1])
def test_encoder_vs_bruteforce_all_bf16_patterns(orc, fmt):
    # every bf16 bit pattern (as binary32) and the same patterns divided by a
    # few scales (the quotients the quantizer feeds the encoder)
    h = np.arange(65536, dtype=np.uint32)
    v = (h << 16).view(np.float32)
    v = v[~np.isnan(v)]
    for s in (1.0, 3.0, 448.0 / 1e-3, 1.0 / 7.0, 2.0 ** -20):
        with np.errstate(over="ignore"):
            q = (v / np.float32(s)).astype(np.float32)
        assert np.array_equal(orc.encode(fmt, q), orc.encode_brute(fmt, q)), f"scale {s}"


@pytest.mark.parametrize("fmt", [0, 1])
def test_encoder_vs_bruteforce_random_f32(orc, fmt):
    rng = np.random.default_rng(1234 + fmt)
    bits = rng.integers(0, 2 ** 32, size=400_000, dtype=np.uint64).astype(np.uint32)
    v = bits.view(np.float32)
    v = v[~np.isnan(v)]
    # also values concentrated in the format's range, where the rounding work happens
    lim = 448.0 if fmt == 0 else 57344.0
    w = (rng.standard_normal(400_000) * lim / 4).astype(np.float32)
    t = (rng.random(400_000) * 2.0 ** -8).astype(np.float32)   # subnormal region of both formats
    for arr in (v, w, t):
        assert np.array_equal(orc.encode(fmt, arr), orc.encode_brute(fmt, arr))


@pytest.mark.parametrize("fmt,tdtype", [(0, torch.float8_e4m3fn), (1, torch.float8_e5m2)])
def test_encoder_matches_torch_in_range(orc, fmt, tdtype):
    # torch's float32 -> float8 conversion rounds to nearest even; it does not
    # saturate, so compare where |v| <= max finite and check saturation apart.
    rng = np.random.default_rng(77 + fmt)
    lim = 448.0 if fmt == 0 else 57344.0
    parts = [
        (rng.standard_normal(300_000) * lim / 3).astype(np.float32),
        (rng.random(300_000) * 2.0 ** -6).astype(np.float32),
        rng.integers(0, 2 ** 32, 300_000, dtype=np.uint64).astype(np.uint32).view(np.float32),
    ]
    v = np.concatenate(parts)
    v = v[np.isfinite(v) & (np.abs(v) <= lim)]
    ref = torch.from_numpy(v.copy()).to(tdtype).view(torch.uint8).numpy()
    assert np.array_equal(orc.encode(fmt, v), ref)
    big = np.array([lim * 1.01, lim * 1000, -lim * 3, np.inf, -np.inf], np.float32)
    sat = orc.encode(fmt, big)
    maxc = 0x7E if fmt == 0 else 0x7B
    assert list(sat) == [maxc, maxc, 0x80 | maxc, maxc, 0x80 | maxc]


def test_nan_input_gives_nan_code(orc):
    for fmt in (0, 1):
        c = orc.encode(fmt, [float("nan")])[0]
        assert math.isnan(orc.decode(fmt, [c])[0])


def test_bf16_rounding_matches_torch(orc):
    rng = np.random.default_rng(5)
    bits = rng.integers(0, 2 ** 32, size=1_000_000, dtype=np.uint64).astype(np.uint32)
    # add exact ties and near-ties around the bf16 grid
    base = rng.integers(0, 2 ** 16, size=50_000, dtype=np.uint64).astype(np.uint32) << 16
    bits = np.concatenate([bits, base | 0x8000, base | 0x7FFF, base | 0x8001, base])
    f = bits.view(np.float32)
    f = f[~np.isnan(f)]
    mine = orc.f32_to_bf16(f)
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(mine, ref)


def test_bf16_to_f32_is_exact_widening(orc):
    h = np.arange(65536, dtype=np.uint16)
    f = orc.bf16_to_f32(h)
    ref = torch.from_numpy(h.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(f), nan)
    assert np.array_equal(f[~nan].view(np.uint32), ref[~nan].view(np.uint32))
