"""Pins for the oracle's number formats (CPU only).

Each check compares the oracle against something that does not reuse its code:
the format definitions enumerated by brute force with exact rational arithmetic,
torch's own float8_e4m3fn / bfloat16 casts (an independent library routine), and
tie cases worked out by hand.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

# --- format definitions, enumerated independently of the oracle -------------

def _e4m3_table():
    """All finite E4M3 ("fn") values by code, from the format: bias 7, 3 mantissa bits."""
    vals = {}
    for c in range(256):
        s, e, m = c >> 7, (c >> 3) & 15, c & 7
        if e == 15 and m == 7:
            continue  # NaN
        mag = Fraction(m, 8) * Fraction(1, 64) if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
        vals[c] = -mag if s else mag
    return vals


def _e2m1_table():
    vals = {}
    for c in range(16):
        s, e, m = c >> 3, (c >> 1) & 3, c & 1
        mag = Fraction(m, 2) if e == 0 else (1 + Fraction(m, 2)) * Fraction(2) ** (e - 1)
        vals[c] = -mag if s else mag
    return vals


E4M3 = _e4m3_table()
E2M1 = _e2m1_table()


def _nearest(table, x: Fraction, sign_bit: int, maxcode: int) -> int:
    """Brute-force round-to-nearest, ties to the even code, saturating, sign kept."""
    neg = x < 0
    a = abs(x)
    cands = [(abs(v - a), c & 1, c) for c, v in table.items() if v >= 0 and c <= maxcode]
    best = min(cands)
    c = best[2]
    return (c | sign_bit) if neg else c


# --- E4M3 --------------------------------------------------------------------

def test_e4m3_decode_all_codes_matches_format_and_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    tv = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        o = oracle.e4m3_to_float(c)
        if c in (0x7F, 0xFF):
            assert np.isnan(o) and np.isnan(tv[c])
            continue
        assert o == float(E4M3[c]) == tv[c], hex(c)


def test_e4m3_encode_roundtrips_every_code():
    for c, v in E4M3.items():
        if v == 0:
            # a Fraction has no signed zero: feed +0.0 / -0.0 explicitly
            assert oracle.e4m3_from_float(-0.0 if c & 0x80 else 0.0) == c
        else:
            got = oracle.e4m3_from_float(float(v))
            assert got == c, (hex(c), float(v), hex(got))


def test_e4m3_ties_and_saturation_by_hand():
    # midpoint of 0 and the smallest subnormal 2^-9 -> even (0)
    assert oracle.e4m3_from_float(2.0 ** -10) == 0x00
    # midpoint of 2^-9 (code 1) and 2^-8 (code 2) -> even code 2
    assert oracle.e4m3_from_float(1.5 * 2.0 ** -9) == 0x02
    # 1.0 = 0x38; 1.0625 halfway to 1.125 (0x39) -> even 0x38; 1.1875 -> 0x3A
    assert oracle.e4m3_from_float(1.0625) == 0x38
    assert oracle.e4m3_from_float(1.1875) == 0x3A
    # largest finite and beyond
    assert oracle.e4m3_from_float(448.0) == 0x7E
    assert oracle.e4m3_from_float(464.0) == 0x7E      # tie 448/480 -> 448
    assert oracle.e4m3_from_float(1e6) == 0x7E
    assert oracle.e4m3_from_float(-1e30) == 0xFE
    assert oracle.e4m3_from_float(float("inf")) == 0x7E
    # a negative value that rounds to zero keeps its sign
    assert oracle.e4m3_from_float(-1e-5) == 0x80


def test_e4m3_encode_matches_torch_cast_on_dense_sample():
    rng = np.random.default_rng(1)
    # log-uniform magnitudes over the whole E4M3 range and below, both signs
    mags = np.exp2(rng.uniform(-14, np.log2(464.0), 60000)).astype(np.float32)
    signs = np.where(rng.random(mags.size) < 0.5, -1, 1).astype(np.float32)
    sample = mags * signs
    # every midpoint between adjacent positive codes, and one float32 ulp either side
    pos = sorted(float(v) for c, v in E4M3.items() if v >= 0 and c < 0x80)
    mids = np.array([(a + b) / 2 for a, b in zip(pos, pos[1:])], dtype=np.float64)
    mids32 = mids.astype(np.float32)
    around = np.concatenate([mids32, np.nextafter(mids32, np.float32(np.inf)),
                             np.nextafter(mids32, np.float32(0))])
    vals = np.concatenate([sample, around, -around]).astype(np.float32)
    vals = vals[np.abs(vals) <= 464.0]
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_from_float(v) for v in vals], dtype=np.uint8)
    bad = np.nonzero(ref != got)[0]
    assert bad.size == 0, [(float(vals[i]), hex(ref[i]), hex(got[i])) for i in bad[:5]]


def test_e4m3_encode_matches_bruteforce_nearest():
    rng = np.random.default_rng(2)
    vals = np.concatenate([
        rng.uniform(-500, 500, 300), rng.uniform(-0.05, 0.05, 300),
        np.array([0.0, 2.0 ** -10, 3 * 2.0 ** -10, 240.0, 248.0, 464.0, 472.0]),
    ]).astype(np.float32)
    for v in vals:
        x = Fraction(float(v))
        want = _nearest(E4M3, x, 0x80, 0x7E)
        assert oracle.e4m3_from_float(float(v)) == want, float(v)


# --- E2M1 --------------------------------------------------------------------

def test_e2m1_decode_table():
    assert [oracle.e2m1_to_float(c) for c in range(8)] == [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    assert [oracle.e2m1_to_float(c) for c in range(8, 16)] == [-0.0, -0.5, -1, -1.5, -2, -3, -4, -6]
    for c in range(16):
        assert oracle.e2m1_to_float(c) == float(E2M1[c])


def test_e2m1_tie_cases_by_hand():
    cases = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6, 7.0: 7, 100.0: 7,
             0.24: 0, 0.26: 1, 5.01: 7, 4.99: 6}
    for v, c in cases.items():
        assert oracle.e2m1_from_float(v) == c, v
        assert oracle.e2m1_from_float(-v) == c | 8, -v
    assert oracle.e2m1_from_float(-0.1) == 0x8


def test_e2m1_encode_matches_bruteforce_nearest():
    grid = np.arange(-8.0, 8.0, 1.0 / 64, dtype=np.float32)
    rng = np.random.default_rng(3)
    vals = np.concatenate([grid, rng.uniform(-7, 7, 500).astype(np.float32)])
    for v in vals:
        want = _nearest(E2M1, Fraction(float(v)), 0x8, 0x7)
        assert oracle.e2m1_from_float(float(v)) == want, float(v)


# --- bf16 rounding of the binary64 combine sum ---------------------------------

def _bf16_value(bits: int) -> Fraction:
    f = np.array([bits << 16], dtype=np.uint32).view(np.float32)[0]
    return Fraction(float(f))


def test_bf16_from_double_matches_bruteforce_nearest():
    rng = np.random.default_rng(4)
    vals = np.concatenate([rng.standard_normal(400) * 10.0 ** rng.integers(-30, 30, 400),
                           rng.standard_normal(100) * 1e-39,     # bf16 subnormal range
                           np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 3.3895313892515355e38])])
    for v in vals:
        got = oracle.bf16_from_double(float(v))
        x = Fraction(float(v))
        # candidates: the truncation of the float32 nearest and its neighbours
        f32bits = int(np.array([v], dtype=np.float32).view(np.uint32)[0])
        base = f32bits >> 16
        cands = [b for b in (base - 1, base, base + 1) if 0 <= (b & 0x7FFF) < 0x7F80]
        best = min(cands, key=lambda b: (abs(_bf16_value(b) - x), b & 1))
        assert got == best, (float(v), hex(got), hex(best))


def test_bf16_from_double_matches_torch_on_float32_inputs():
    rng = np.random.default_rng(5)
    f = (rng.standard_normal(20000) * np.exp2(rng.integers(-60, 60, 20000))).astype(np.float32)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_from_double(float(v)) for v in f], dtype=np.uint16)
    assert np.array_equal(ref, got)
