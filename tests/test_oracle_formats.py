"""Pins for the oracle's DeepGEMM consumer formats (CPU only): expert-aligned metadata and
FP8 group-128 quantisation with power-of-two UE8M0 scales.

Aligned metadata is checked against the unaligned metadata (pinned separately) through
the closed-form shift of every segment, against bincount, and by brute force; UE8M0 scales
against exact rational bounds (2^(b-128) < amax/448 <= 2^(b-127), amax/448 taken in binary32
as the definition states) and the codes against torch's float8_e4m3fn cast of the exactly
scaled values.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from workloads import bf16_bits_to_f32, f32_to_bf16_bits, make_case


@pytest.mark.parametrize("A", [1, 2, 8, 128])
@pytest.mark.parametrize("seed", range(4))
def test_aligned_metadata_is_the_unaligned_one_shifted(A, seed):
    w = make_case(200, 16, 24, 6, seed=seed, routing="replace", invalid_rate=0.1)
    u = oracle.route_meta(w.topk_ids, w.E, P=4)
    a = oracle.route_meta_aligned(w.topk_ids, w.E, A, P=4)
    flat = w.topk_ids.reshape(-1)
    cnt = np.bincount(flat[flat >= 0], minlength=w.E)
    assert a.seg_indptr.tolist() == [0] + np.cumsum((cnt + A - 1) // A * A).tolist()
    assert (a.seg_indptr % A == 0).all()
    v = flat >= 0
    shift = a.seg_indptr[flat[v]] - u.seg_indptr[flat[v]]
    assert np.array_equal(a.src2dst[v], u.src2dst[v] + shift)
    assert (a.src2dst[~v] == -1).all()
    assert np.array_equal(a.masked_m, u.masked_m) and np.array_equal(a.partition_counts, u.partition_counts)
    # reorder: the expert of every real row, -1 on every padding row
    want = np.full(int(a.seg_indptr[-1]), -1)
    want[a.src2dst[v]] = flat[v]
    assert np.array_equal(a.reorder_topk_ids, want)
    if A == 1:
        assert np.array_equal(a.seg_indptr, u.seg_indptr) and np.array_equal(a.src2dst, u.src2dst)


def test_ue8m0_scales_and_codes():
    w = make_case(6, 1024, 4, 1, seed=41, std=3.0, zero_tokens=1)
    for t in range(w.T):
        q, b = oracle.quant_fp8_ue8m0_row(w.x[t])
        x = bf16_bits_to_f32(w.x[t]).reshape(-1, 128)
        for g in range(x.shape[0]):
            amax = float(np.abs(x[g]).max())
            s = Fraction(float(np.float32(max(amax, np.float32(1e-10))) / np.float32(448.0)))
            k = int(b[g]) - 127
            assert Fraction(2) ** (k - 1) < s <= Fraction(2) ** k          # the power of two just above
            scaled = (x[g].astype(np.float64) * 2.0 ** (-k)).astype(np.float32)  # exact: power-of-two scaling
            assert np.all(np.abs(scaled) <= 448)
            ref = torch.from_numpy(scaled).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            assert np.array_equal(q[g * 128:(g + 1) * 128], ref)


def test_ue8m0_constant_group_uses_powers_of_two():
    row = f32_to_bf16_bits(np.concatenate([np.full(128, 448.0), np.full(128, 1.0)]).astype(np.float32))
    q, b = oracle.quant_fp8_ue8m0_row(row)
    assert b.tolist() == [127, 127 - 8]                 # 448/448 = 2^0; 1/448 -> 2^-8
    assert (q[:128] == 0x7E).all()                       # 448 / 1 = 448
    assert (q[128:] == 0x78).all()                       # 1 / 2^-8 = 256 = 2^8 -> e4m3 0x78


@pytest.mark.parametrize("mode", ["normal", "masked"])
def test_fp8_passthrough_rows_are_byte_copies(mode):
    """Per-tensor FP8 rows (already one-byte codes) are copied unchanged to their destinations."""
    w = make_case(30, 96, 6, 3, seed=61, invalid_rate=0.1)
    codes = np.random.default_rng(62).integers(0, 256, size=(w.T, w.H), dtype=np.uint8)
    M = 40 if mode == "masked" else 0
    m = oracle.route_meta(w.topk_ids, w.E, M=M)
    q, s = oracle.dispatch(mode, "fp8_passthrough", codes, w.topk_ids, m, w.E, M=M, fill=0xC3)
    assert s is None
    rows = q.reshape(-1, w.H)
    flat = w.topk_ids.reshape(-1)
    hit = np.zeros(rows.shape[0], bool)
    for i, d in enumerate(m.src2dst):
        if d < 0:
            continue
        r = d if mode == "normal" else flat[i] * M + d - m.seg_indptr[flat[i]]
        assert np.array_equal(rows[r], codes[i // w.K])
        hit[r] = True
    assert (rows[~hit] == 0xC3).all()


# --- interleaved NVFP4 block scales (nvfp4_block_scale_interleave) ---------------------------

def _interleave_by_reshape(sf: np.ndarray) -> np.ndarray:
    """The same layout stated as array reshapes: rows r = 128*rt + 32*i + j, columns
    c = 4*ct + cc; the tile (rt, ct) is stored as [j][i][cc]."""
    rows, cols = sf.shape
    Rp, Cp = (rows + 127) // 128 * 128, (cols + 3) // 4 * 4
    pad = np.zeros((Rp, Cp), np.uint8)
    pad[:rows, :cols] = sf
    t = pad.reshape(Rp // 128, 4, 32, Cp // 4, 4)       # rt, i, j, ct, cc
    return t.transpose(0, 3, 2, 1, 4).reshape(-1)        # rt, ct, j, i, cc


@pytest.mark.parametrize("rows,cols", [(128, 4), (256, 448), (77, 448), (300, 6), (1, 1), (1024, 256)])
def test_sf_interleave_matches_reshape_definition(rows, cols):
    sf = np.random.default_rng(rows * 7 + cols).integers(0, 256, (rows, cols), dtype=np.uint8)
    got = oracle.nvfp4_sf_interleave(sf)
    assert got.shape == ((rows + 127) // 128 * 128 * ((cols + 3) // 4 * 4),)
    assert np.array_equal(got, _interleave_by_reshape(sf))


def test_sf_interleave_first_lines_and_padding():
    """Each 16-byte line holds rows j, j+32, j+64, j+96 of the tile's 4 columns; the next
    4 columns start a new 512-byte tile; padded rows and columns are zero."""
    rows, cols = 100, 6
    sf = (np.arange(rows * cols) % 251 + 1).astype(np.uint8).reshape(rows, cols)  # no zeros
    got = oracle.nvfp4_sf_interleave(sf)
    assert list(got[0:4]) == list(sf[0, 0:4])
    assert list(got[4:8]) == list(sf[32, 0:4])
    assert list(got[8:12]) == list(sf[64, 0:4])
    assert list(got[12:16]) == list(sf[96, 0:4])
    assert list(got[16:20]) == list(sf[1, 0:4])
    assert list(got[512:514]) == list(sf[0, 4:6]) and list(got[514:516]) == [0, 0]   # cols 6, 7 pad
    assert list(got[12 + 16 * 4: 16 + 16 * 4]) == [0, 0, 0, 0]                         # row 100 pad
    assert int(np.count_nonzero(got)) == rows * cols


def test_sf_interleave_is_a_permutation_of_full_tiles():
    """On whole tiles every source byte lands in exactly one place: tracking a 16-bit index
    through the interleave as two byte planes recovers a permutation."""
    rows, cols = 256, 8
    idx = np.arange(rows * cols, dtype=np.uint16).reshape(rows, cols)
    lo = oracle.nvfp4_sf_interleave((idx & 0xFF).astype(np.uint8))
    hi = oracle.nvfp4_sf_interleave((idx >> 8).astype(np.uint8))
    where = lo.astype(np.int64) | (hi.astype(np.int64) << 8)
    assert np.array_equal(np.sort(where), np.arange(rows * cols))


def test_swizzled_expectation_helper_matches_a_direct_construction():
    """The test-side expectation of the swizzled scale buffer (tests/_harness.py) equals a direct,
    element-by-element construction from the layout's definition: scale (r, c) at byte
    ((r/128)*(C/4) + c/4)*512 + (r%32)*16 + ((r%128)/32)*4 + c%4; the rows of a touched 128-row
    block that no pair maps to, and the padding rows, are zero; other blocks keep the fill."""
    from _harness import swizzled_scales_expected
    rng = np.random.default_rng(3)
    for R, C in ((300, 8), (128, 4), (513, 12)):
        fill = 0xA5
        osf = np.full((R, C), fill, np.uint8)
        written = rng.random(R) < 0.6
        osf[written] = rng.integers(0, 0x7F, size=(int(written.sum()), C), dtype=np.uint8)
        touched = np.zeros(R, bool)
        touched[rng.integers(0, R, size=3)] = True
        got = swizzled_scales_expected(osf, written, touched)
        Rp = (R + 127) // 128 * 128
        want = np.full(Rp * C, fill, np.uint8)
        blk_touched = np.zeros(Rp // 128, bool)
        blk_touched[np.nonzero(touched)[0] // 128] = True
        if R % 128:
            blk_touched[-1] = True
        for r in range(Rp):
            for c in range(C):
                off = ((r // 128) * (C // 4) + c // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + c % 4
                if r >= R:
                    v = 0
                elif blk_touched[r // 128] and not written[r]:
                    v = 0
                else:
                    v = osf[r, c]
                want[off] = v
        assert np.array_equal(got, want)
