"""Pins for the oracle's metadata, quantisation, gather and combine (CPU only).

Nothing here re-types the oracle's own loops: the metadata is checked against a
brute-force pair count and numpy's stable argsort, the quantisers against the
hand-worked examples in tests/golden and against bounds the formats fix, the
gather against its inverse, and the combine against exact rational arithmetic
and closed forms (identity experts).
"""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from workloads import bf16_bits_to_f32, f32_to_bf16_bits, make_case, make_workload

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    rows = {}
    multi = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            if key in rows:
                multi.setdefault(key, [rows[key]]).append(vals)
            rows[key] = vals
    return rows, multi


def _ints(vals):
    return [int(v, 0) for v in vals]


# --- metadata ------------------------------------------------------------------

def _bruteforce_meta(ids, E):
    """src2dst[i] = #valid pairs with a smaller id + #earlier pairs with the same id."""
    flat = ids.reshape(-1)
    valid = (flat >= 0) & (flat < E)
    s2d = np.full(flat.size, -1, np.int64)
    for i in range(flat.size):
        if not valid[i]:
            continue
        below = sum(1 for j in range(flat.size) if valid[j] and flat[j] < flat[i])
        before = sum(1 for j in range(i) if valid[j] and flat[j] == flat[i])
        s2d[i] = below + before
    return s2d


def test_route_meta_golden_worked_example():
    g, _ = _read_golden("route_meta_worked.txt")
    T, K, E, P = (int(g[k][0]) for k in ("T", "K", "E", "P"))
    ids = np.array(_ints(g["topk_ids"]), np.int32).reshape(T, K)
    m2 = oracle.route_meta(ids, E, P=P, M=2)
    assert m2.seg_indptr.tolist() == _ints(g["seg_indptr"])
    assert m2.src2dst.tolist() == _ints(g["src2dst"])
    assert m2.reorder_topk_ids.tolist() == _ints(g["reorder_topk_ids"])
    assert m2.masked_m.tolist() == _ints(g["masked_m_M2"])
    assert m2.partition_counts.tolist() == _ints(g["partition_counts_P2"])
    assert m2.expected_m == int(g["expected_m"][0])
    assert m2.status == 0
    m1 = oracle.route_meta(ids, E, P=P, M=1)
    assert m1.masked_m.tolist() == _ints(g["masked_m_M1"])
    assert m1.status == oracle.CAPACITY
    # masked rows e*M + rank from the oracle's own masked dispatch
    x = np.arange(T * 8, dtype=np.uint16).reshape(T, 8) + 1
    q, _ = oracle.dispatch("masked", "none", x, ids, m2, E, M=2)
    rows = q.reshape(E * 2, 8)
    for i, r in enumerate(_ints(g["masked_rows_M2"])):
        if r >= 0:
            assert rows[r].tolist() == x[i // K].tolist()


@pytest.mark.parametrize("seed", range(40))
def test_route_meta_bruteforce_tiny(seed):
    rng = np.random.default_rng(seed)
    T, K, E = int(rng.integers(0, 7)), int(rng.integers(1, 4)), int(rng.integers(1, 6))
    ids = rng.integers(-1, E, size=(T, K)).astype(np.int32)
    m = oracle.route_meta(ids, E)
    assert m.src2dst.tolist() == _bruteforce_meta(ids, E).tolist()
    assert m.status == 0


@pytest.mark.parametrize("seed", range(5))
def test_route_meta_matches_stable_argsort(seed):
    w = make_case(300, 8, 37, 5, seed=seed, routing="replace", invalid_rate=0.1)
    flat = w.topk_ids.reshape(-1)
    key = np.where(flat >= 0, flat, 37)                  # invalid pairs sort last
    order = np.argsort(key, kind="stable")
    n = int((flat >= 0).sum())
    want = np.full(flat.size, -1, np.int64)
    want[order[:n]] = np.arange(n)
    m = oracle.route_meta(w.topk_ids, 37)
    assert np.array_equal(m.src2dst, want)
    assert np.array_equal(m.seg_indptr, np.concatenate([[0], np.cumsum(np.bincount(flat[flat >= 0], minlength=37))]))
    assert np.array_equal(m.reorder_topk_ids, flat[order[:n]])


@pytest.mark.parametrize("name", ["tiny", "decode", "prefill"])
def test_route_meta_invariants_on_workloads(name):
    w = make_workload(name)
    m = oracle.route_meta(w.topk_ids, w.E, P=w.P, M=w.M)
    flat = w.topk_ids.reshape(-1)
    valid = (flat >= 0) & (flat < w.E)
    n = int(valid.sum())
    assert m.seg_indptr[-1] == n                                  # seg_indptr[E] = #valid pairs
    assert sorted(m.src2dst[valid].tolist()) == list(range(n))    # bijection onto [0, N)
    assert (m.src2dst[~valid] == -1).all()
    assert (np.diff(m.reorder_topk_ids) >= 0).all()               # non-decreasing
    assert np.array_equal(m.reorder_topk_ids[m.src2dst[valid]], flat[valid])
    assert m.partition_counts.sum() == n
    assert m.expected_m == (w.T * w.K + w.E) // w.E


def test_route_meta_empty_batch_and_all_invalid():
    m = oracle.route_meta(np.zeros((0, 8), np.int32), 16)
    assert m.seg_indptr.tolist() == [0] * 17 and m.src2dst.size == 0 and m.num_valid == 0
    m = oracle.route_meta(np.full((5, 3), -1, np.int32), 4, M=2)
    assert m.seg_indptr.tolist() == [0] * 5 and (m.src2dst == -1).all() and m.status == 0


def test_route_meta_flags_out_of_range_ids():
    ids = np.array([[0, 4], [-3, 1]], np.int32)
    m = oracle.route_meta(ids, 4)
    assert m.status == oracle.BAD_ID
    assert m.src2dst.tolist() == [0, -1, -1, 1]


def test_closed_forms_from_the_pages():
    g, multi = _read_golden("closed_forms.txt")
    assert oracle.dispatch_payload_bytes(7168, 8, True) == int(g["payload_nvfp4_H7168_K8"][0])
    assert oracle.dispatch_payload_bytes(7168, 8, False) == int(g["payload_bf16_H7168_K8"][0])
    for T, K, E, em in (map(int, r) for r in multi["expected_m"]):
        assert oracle.expected_m(T, K, E) == em


# --- FP8 group-128 ----------------------------------------------------------------

def _bits(vals):
    return f32_to_bf16_bits(np.array(vals, np.float32))


def test_fp8_golden_group():
    g, _ = _read_golden("quant_worked.txt")
    x = np.zeros(128, np.float32)
    xv = [float(v) for v in g["fp8_group_x"]]
    x[: len(xv)] = xv
    q, s = oracle.quant_fp8_row(_bits(x))
    codes = _ints(g["fp8_group_codes"])
    assert q[: len(codes)].tolist() == codes and (q[len(codes):] == 0).all()
    num, den = map(int, g["fp8_group_scale_rational"][0].split("/"))
    exact = Fraction(num, den)
    ulp = Fraction(2) ** (int(np.floor(np.log2(float(exact)))) - 23)
    assert abs(Fraction(float(s[0])) - exact) <= ulp / 2


def test_fp8_constant_and_zero_groups():
    row = np.concatenate([np.full(128, 0.3, np.float32), np.zeros(128, np.float32),
                          np.full(128, -5.0, np.float32)])
    q, s = oracle.quant_fp8_row(_bits(row))
    assert (q[:128] == 0x7E).all() and (q[128:256] == 0).all() and (q[256:] == 0xFE).all()
    assert s[1] == np.float32(np.float32(1e-10) / np.float32(448.0))
    c = float(bf16_bits_to_f32(_bits([0.3]))[0])
    assert abs(Fraction(float(s[0])) - Fraction(c) / 448) <= Fraction(float(s[0])) * Fraction(1, 2 ** 24)


def test_fp8_dequant_error_within_half_ulp():
    w = make_case(4, 7168, 8, 1, seed=11)
    for t in range(4):
        q, s = oracle.quant_fp8_row(w.x[t])
        x = bf16_bits_to_f32(w.x[t]).astype(np.float64).reshape(-1, 128)
        dq = np.array([oracle.e4m3_to_float(c) for c in q], np.float64).reshape(-1, 128)
        y = x / s[:, None].astype(np.float64)          # exact quotient the codes approximate
        # e4m3 spacing at |y| (3 mantissa bits, subnormal quantum 2^-9), half of it
        e = np.floor(np.log2(np.maximum(np.abs(y), 2.0 ** -6)))
        half = np.exp2(e - 3) / 2
        assert (np.abs(dq - y) <= half * (1 + 1e-6) + 1e-30).all()
        # the largest element of every group maps to +-448
        amax_pos = np.abs(x).argmax(axis=1)
        assert (np.abs(dq[np.arange(dq.shape[0]), amax_pos]) == 448).all()


# --- NVFP4 block-16 -------------------------------------------------------------------

@pytest.mark.parametrize("case", ["A", "B"])
def test_nvfp4_golden_blocks(case):
    g, _ = _read_golden("quant_worked.txt")
    x = np.zeros(16, np.float32)
    xv = [float(v) for v in g[f"nvfp4_{case}_x"]]
    x[: len(xv)] = xv
    q, sf = oracle.quant_nvfp4_row(_bits(x), float(g[f"nvfp4_{case}_g"][0]))
    want = _ints(g[f"nvfp4_{case}_bytes"])
    assert sf.tolist() == _ints(g[f"nvfp4_{case}_sf"])
    assert q[: len(want)].tolist() == want and (q[len(want):] == 0).all()


def test_nvfp4_zero_block_and_max_element():
    w = make_case(3, 7168, 8, 1, seed=12, quant="nvfp4b16", std=1.4142135)
    g = w.global_scale
    x = w.x.copy()
    x[0, :16] = 0
    for t in range(3):
        q, sf = oracle.quant_nvfp4_row(x[t], g)
        codes = np.stack([q & 15, q >> 4], axis=1).reshape(-1, 16)
        xb = bf16_bits_to_f32(x[t]).reshape(-1, 16)
        sff = np.array([oracle.e4m3_to_float(c) for c in sf])
        for b in range(codes.shape[0]):
            if sff[b] == 0:
                assert (codes[b] == 0).all()
                continue
            # sf is within half an e4m3 step of amax*g/6, so the largest element maps to 6
            j = int(np.abs(xb[b]).argmax())
            assert codes[b, j] & 7 == 7
            # every element within half an e2m1 step (after scaling) of its code
            y = xb[b].astype(np.float64) * (g / sff[b])
            dq = np.array([oracle.e2m1_to_float(c) for c in codes[b]])
            step = np.where(np.abs(y) < 2, 0.5, np.where(np.abs(y) < 4, 1.0, 2.0))
            assert (np.abs(dq - np.clip(y, -6, 6)) <= step / 2 + 1e-6).all()
        if t == 0:
            assert sf[0] == 0 and (q[:8] == 0).all()


# --- gather ----------------------------------------------------------------------------

@pytest.mark.parametrize("mode", ["normal", "masked"])
def test_dispatch_unpermute_returns_input(mode):
    w = make_case(50, 64, 12, 4, seed=13, invalid_rate=0.1)
    M = 60 if mode == "masked" else 0
    m = oracle.route_meta(w.topk_ids, w.E, M=M)
    q, _ = oracle.dispatch(mode, "none", w.x, w.topk_ids, m, w.E, M=M, fill=0xAB)
    rows = q.reshape(-1, 64)
    flat = w.topk_ids.reshape(-1)
    touched = np.zeros(rows.shape[0], bool)
    for i, d in enumerate(m.src2dst):
        if d < 0:
            continue
        r = d if mode == "normal" else flat[i] * M + (d - m.seg_indptr[flat[i]])
        assert np.array_equal(rows[r], w.x[i // 4])
        touched[r] = True
    assert (rows[~touched] == 0xABAB).all()


def test_dispatch_masked_capacity_drops_late_pairs():
    w = make_case(20, 32, 2, 1, seed=14, routing="hot")     # every token -> expert 0
    m = oracle.route_meta(w.topk_ids, 2, M=5)
    assert m.status == oracle.CAPACITY and m.masked_m.tolist() == [5, 0]
    q, _ = oracle.dispatch("masked", "none", w.x, w.topk_ids, m, 2, M=5)
    assert np.array_equal(q[0, :5], w.x[:5])               # the first five tokens in order


# --- combine ---------------------------------------------------------------------------

def test_combine_identity_experts_return_input():
    w = make_case(64, 256, 8, 4, seed=15)
    m = oracle.route_meta(w.topk_ids, w.E)
    q, _ = oracle.dispatch("normal", "none", w.x, w.topk_ids, m, w.E)
    y = oracle.combine("normal", q[: m.num_valid], w.topk_ids, w.topk_weights, m, w.E)
    assert np.array_equal(y, w.x)


def test_combine_single_slot_unit_weight_is_exact():
    w = make_case(33, 96, 5, 1, seed=16)
    m = oracle.route_meta(w.topk_ids, w.E, M=40)
    q, _ = oracle.dispatch("masked", "none", w.x, w.topk_ids, m, w.E, M=40)
    y = oracle.combine("masked", q, w.topk_ids, np.ones((33, 1), np.float32), m, w.E, M=40)
    assert np.array_equal(y, w.x)


def test_combine_two_rows_matches_exact_rational_rounding():
    rng = np.random.default_rng(17)
    a = f32_to_bf16_bits(rng.standard_normal(512).astype(np.float32))
    b = f32_to_bf16_bits(rng.standard_normal(512).astype(np.float32))
    eo = np.stack([a, b])
    ids = np.array([[0, 1]], np.int32)
    wts = np.array([[0.5, 0.5]], np.float32)
    m = oracle.route_meta(ids, 2)
    y = oracle.combine("normal", eo, ids, wts, m, 2)[0]
    fa, fb = bf16_bits_to_f32(a), bf16_bits_to_f32(b)
    for h in range(512):
        exact = (Fraction(float(fa[h])) + Fraction(float(fb[h]))) / 2
        f32 = np.float32(float(exact))
        base = int(np.array([f32]).view(np.uint32)[0]) >> 16
        cands = [c for c in (base - 1, base, base + 1) if (c & 0x7FFF) < 0x7F80]
        val = lambda c: Fraction(float(np.array([c << 16], np.uint32).view(np.float32)[0]))
        best = min(cands, key=lambda c: (abs(val(c) - exact), c & 1))
        assert int(y[h]) == best


def test_combine_token_without_valid_slot_is_zero():
    ids = np.array([[-1, -1], [0, 1]], np.int32)
    m = oracle.route_meta(ids, 2)
    eo = f32_to_bf16_bits(np.ones((2, 16), np.float32))
    y = oracle.combine("normal", eo, ids, np.full((2, 2), 0.5, np.float32), m, 2)
    assert (y[0] == 0).all() and (bf16_bits_to_f32(y[1]) == 1.0).all()


def test_tiny_workload_scaled_experts_roundtrip():
    """Expert e returns x*(e+1)/8 (exact in bf16 for e+1 a power of two); combine of the
    scaled rows with weights w equals sum_k w_k*(e_k+1)/8 * x in exact arithmetic."""
    w = make_workload("tiny")
    m = oracle.route_meta(w.topk_ids, w.E)
    q, _ = oracle.dispatch("normal", "none", w.x, w.topk_ids, m, w.E)
    rows = bf16_bits_to_f32(q[: m.num_valid]).astype(np.float64)
    scale = (m.reorder_topk_ids.astype(np.float64) + 1) / 8
    eo = f32_to_bf16_bits((rows * scale[:, None]).astype(np.float32))
    y = bf16_bits_to_f32(oracle.combine("normal", eo, w.topk_ids, w.topk_weights, m, w.E))
    pow2 = [0, 1, 3, 7]                                     # (e+1)/8 in {1/8, 1/4, 1/2, 1}
    x = bf16_bits_to_f32(w.x).astype(np.float64)
    for t in range(w.T):
        e0, e1 = w.topk_ids[t]
        if e0 in pow2 and e1 in pow2:
            want = (float(w.topk_weights[t, 0]) * (e0 + 1) / 8 + float(w.topk_weights[t, 1]) * (e1 + 1) / 8) * x[t]
            assert np.allclose(y[t], want, rtol=2 ** -8, atol=0)
