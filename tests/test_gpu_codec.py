"""GPU codec check: the e4m3 / e2m1 conversions the quantising kernels use, run through
moe_convert_probe, against the oracle's format definitions on every decision point --
each representable value, every midpoint between neighbours and the float32 values up
to 3 ulps either side of it, saturation, signed zeros, float32 subnormals -- plus a
million log-uniform random values; and exhaustively over every float32 whose conversion is
not a trivial saturation or flush to zero. Also fixes the packing order: the even element
goes to the low byte (e4m3 pair) / low nibble (e2m1 pair)."""
import numpy as np
import pytest
import torch

import oracle

from _harness import moe

pytestmark = pytest.mark.gpu


def _around(points: np.ndarray, ulps: int = 3) -> np.ndarray:
    p = points.astype(np.float32)
    out = [p]
    up, dn = p.copy(), p.copy()
    for _ in range(ulps):
        up = np.nextafter(up, np.float32(np.inf))
        dn = np.nextafter(dn, np.float32(-np.inf))
        out += [up, dn]
    return np.concatenate(out)


def _decision_points():
    e4 = np.array([oracle.e4m3_to_float(c) for c in range(0x7F)], np.float64)       # 0 .. 448
    e2 = np.array([oracle.e2m1_to_float(c) for c in range(8)], np.float64)          # 0 .. 6
    mids = np.concatenate([(e4[1:] + e4[:-1]) / 2, (e2[1:] + e2[:-1]) / 2])
    special = np.array([448.0, 464.0, 480.0, 500.0, 1e6, 3.0e38, 6.0, 7.0, 8.0, 1e-30, 1e-40, 2.0 ** -10,
                        2.0 ** -126, 2.0 ** -149], np.float64)
    pos = np.concatenate([_around(e4), _around(e2), _around(mids), _around(special)])
    pos = pos[np.isfinite(pos) & (pos >= 0)]
    rng = np.random.default_rng(0)
    rand = np.exp2(rng.uniform(-20, 10, 1 << 20)).astype(np.float32)
    vals = np.concatenate([pos, rand, [0.0]]).astype(np.float32)
    vals = np.concatenate([vals, -vals])
    if vals.size % 2:
        vals = np.append(vals, np.float32(1.0))
    return vals


def test_convert_probe_matches_oracle_formats():
    m = moe()
    v = _decision_points()
    x = torch.from_numpy(v).cuda()
    e4 = torch.empty(v.size, dtype=torch.uint8, device="cuda")
    e2 = torch.empty(v.size // 2, dtype=torch.uint8, device="cuda")
    dv = torch.empty(v.size, dtype=torch.float32, device="cuda")
    m.moe_convert_probe(x, e4, e2, dv)
    torch.cuda.synchronize()
    g4, g2, gd = e4.cpu().numpy(), e2.cpu().numpy(), dv.cpu().numpy()

    o4 = oracle.e4m3_from_float_array(v)
    bad = np.nonzero(g4 != o4)[0]
    assert bad.size == 0, [(float(v[i]), hex(g4[i]), hex(o4[i])) for i in bad[:8]]

    o2 = oracle.e2m1_from_float_array(v)
    packed = (o2[0::2] | (o2[1::2] << 4)).astype(np.uint8)
    bad = np.nonzero(g2 != packed)[0]
    assert bad.size == 0, [(float(v[2 * i]), float(v[2 * i + 1]), hex(g2[i]), hex(packed[i])) for i in bad[:8]]

    od = np.array([oracle.e4m3_to_float(c) for c in range(256)], np.float64)[o4].astype(np.float32)
    ok = ~np.isnan(od)
    assert np.array_equal(gd[ok].view(np.uint32), od[ok].view(np.uint32))


def test_convert_probe_exhaustive_over_the_rounding_range():
    """Every float32 of both signs with magnitude in [2^-11, 2^11) -- the range in which an
    e4m3 or e2m1 conversion neither saturates trivially nor flushes to zero (e4m3: smallest
    subnormal 2^-9, largest finite 448; e2m1: 0.5 .. 6) -- in chunks of 2^25 values:
    369 million conversions of each kind compared with the oracle's definitions."""
    m = moe()
    lo, hi = (127 - 11) << 23, (127 + 11) << 23
    chunk = 1 << 25
    table = np.array([oracle.e4m3_to_float(c) for c in range(256)], np.float64).astype(np.float32)
    x = torch.empty(chunk, dtype=torch.float32, device="cuda")
    e4 = torch.empty(chunk, dtype=torch.uint8, device="cuda")
    e2 = torch.empty(chunk // 2, dtype=torch.uint8, device="cuda")
    dv = torch.empty(chunk, dtype=torch.float32, device="cuda")
    checked = 0
    for sign in (0, 1 << 31):
        for start in range(lo, hi, chunk):
            n = min(chunk, hi - start)
            bits = np.arange(start, start + n, dtype=np.uint64).astype(np.uint32) | np.uint32(sign)
            v = bits.view(np.float32)
            x[:n].copy_(torch.from_numpy(v))
            m.moe_convert_probe(x[:n], e4[:n], e2[: n // 2], dv[:n])
            g4, g2, gd = e4[:n].cpu().numpy(), e2[: n // 2].cpu().numpy(), dv[:n].cpu().numpy()
            o4 = oracle.e4m3_from_float_array(v)
            bad = np.nonzero(g4 != o4)[0]
            assert bad.size == 0, [(float(v[i]), hex(g4[i]), hex(o4[i])) for i in bad[:8]]
            o2 = oracle.e2m1_from_float_array(v)
            packed = (o2[0::2] | (o2[1::2] << 4)).astype(np.uint8)
            bad = np.nonzero(g2 != packed)[0]
            assert bad.size == 0, [(float(v[2 * i]), hex(g2[i]), hex(packed[i])) for i in bad[:8]]
            od = table[o4]
            ok = ~np.isnan(od)
            assert np.array_equal(gd[ok].view(np.uint32), od[ok].view(np.uint32))
            checked += n
    assert checked == 2 * (hi - lo)


def test_fp8_division_matches_ieee_over_the_quantiser_domain():
    """The FP8 quantiser's x / s (reciprocal + one correction step) gives the same e4m3 code
    as the IEEE binary32 division for every bf16 group maximum and every bf16 x it can divide
    (about 10^9 pairs, checked exhaustively on the GPU), and the same quotient wherever
    |x / s| >= 2^-12."""
    m = moe()
    res = torch.full((4,), -1, dtype=torch.int64, device="cuda")
    m.moe_fp8_division_check(res)
    code_mism, first, big_mism, all_mism = (int(v) for v in res.cpu().tolist())
    x_bits, s_bits = (first >> 32) & 0xFFFFFFFF, first & 0xFFFFFFFF
    assert code_mism == 0, (code_mism, hex(x_bits), hex(s_bits))
    assert big_mism == 0, big_mism
    assert all_mism >= 0
