"""GPU parity of the DeepGEMM consumer formats against the oracle: expert-aligned metadata
(moe_route_meta_ex), FP8 group-128 with power-of-two UE8M0 scales, and the column-major
(MN-major, TMA-aligned) scale layouts of moe_dispatch_ex; combine over aligned segments
(moe_combine_ex). All integer and quantised outputs bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from workloads import make_case, make_workload, random_bf16

from _harness import (_all_bytes_are, _sentinel_buffer, SENTINEL, bytes_of, check_combine, filled, masked_rows, masked_touched_rows, moe, to_dev,
                      swizzled_scales_expected)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T,E,K,A", [(100, 16, 4, 128), (3000, 37, 8, 8), (64, 8, 2, 1), (20000, 256, 8, 128)])
def test_aligned_route_meta_matches_oracle(T, E, K, A):
    m = moe()
    w = make_case(T, 16, E, K, seed=T + A, routing="zipf" if E >= K else "replace", invalid_rate=0.05)
    _, ids, _ = to_dev(w)
    cap = T * K + E * (A - 1)
    seg = torch.empty(E + 1, dtype=torch.int64, device="cuda")
    s2d = torch.empty(T * K, dtype=torch.int32, device="cuda")
    reo = torch.full((cap,), -7, dtype=torch.int32, device="cuda")
    mm = torch.empty(E, dtype=torch.int32, device="cuda")
    pc = torch.empty(1, dtype=torch.int32, device="cuda")
    st = m.new_status()
    m.moe_route_meta_ex(ids, E, seg, s2d, reo, mm, st, m.new_workspace(T, K, E), 1, 0, A, pc)
    om = oracle.route_meta_aligned(w.topk_ids, E, A)
    torch.cuda.synchronize()
    n = int(om.seg_indptr[-1])
    assert np.array_equal(seg.cpu().numpy(), om.seg_indptr)
    assert np.array_equal(s2d.cpu().numpy(), om.src2dst)
    assert np.array_equal(reo[:n].cpu().numpy(), om.reorder_topk_ids)
    assert (reo[n:].cpu().numpy() == -7).all()
    assert np.array_equal(mm.cpu().numpy(), om.masked_m) and int(pc.item()) == int(om.partition_counts[0])
    assert int(st.item()) == 0


def _colmajor_fp32(rowmajor, R4):
    rows, G = rowmajor.shape
    out = np.full((G, R4), SENTINEL * 0x01010101, np.uint32)
    out[:, :rows] = rowmajor.view(np.uint32).T
    return out


def _colmajor_ue8m0(rowmajor, R4):
    rows, G = rowmajor.shape
    G4 = (G + 3) // 4
    out = np.full((G4, R4, 4), SENTINEL, np.uint8)
    for g in range(G):
        out[g // 4, :rows, g % 4] = rowmajor[:, g]
    return out


@pytest.mark.parametrize("T", [300, 1100])   # register path; bulk kernel with thread-stored scales
@pytest.mark.parametrize("quant", ["fp8g128", "fp8g128_ue8m0"])
@pytest.mark.parametrize("layout", ["row", "col"])
def test_aligned_dispatch_and_combine(quant, layout, T):
    """Normal layout over 128-aligned segments, both scale layouts (H = 640: 5 groups, so
    neither scale row is a 16-byte multiple)."""
    m = moe()
    H, E, K, A = 640, 24, 6, 128
    w = make_case(T, H, E, K, seed=51, routing="zipf", invalid_rate=0.05)
    x, ids, wt = to_dev(w)
    cap = T * K + E * (A - 1)
    om = oracle.route_meta_aligned(w.topk_ids, E, A)
    seg = torch.from_numpy(om.seg_indptr).cuda()
    s2d = torch.from_numpy(om.src2dst).cuda()
    G = H // 128
    q = filled((cap, H), torch.uint8)
    R4 = (cap + 3) // 4 * 4
    if quant == "fp8g128":
        scales = filled((cap, G) if layout == "row" else (G, R4), torch.float32)
    else:
        scales = filled((cap, G) if layout == "row" else ((G + 3) // 4, R4, 4), torch.uint8)
    st = m.new_status()
    m.moe_dispatch_ex("normal", quant, layout, x, ids, E, s2d, seg, q, scales, st, out_rows=cap)
    torch.cuda.synchronize()
    gq = q.cpu().numpy()
    rows_written = np.zeros(cap, bool)
    ref_scale = np.zeros((cap, G), np.float32 if quant == "fp8g128" else np.uint8)
    for i, d in enumerate(om.src2dst):
        if d < 0:
            continue
        t = i // K
        if quant == "fp8g128":
            oq, os_ = oracle.quant_fp8_row(w.x[t])
        else:
            oq, os_ = oracle.quant_fp8_ue8m0_row(w.x[t])
        assert np.array_equal(gq[d], oq)
        ref_scale[d] = os_
        rows_written[d] = True
    assert (gq[~rows_written] == SENTINEL).all()          # padding rows and unused capacity untouched
    gs = scales.cpu().numpy()
    if layout == "row":
        got = gs[rows_written]
        want = ref_scale[rows_written]
        assert np.array_equal(got.view(np.uint8), want.view(np.uint8))
    else:
        if quant == "fp8g128":
            full = _colmajor_fp32(np.where(rows_written[:, None], ref_scale, np.float32(0)).astype(np.float32), R4)
            mask = np.zeros((G, R4), bool)
            mask[:, :cap] = rows_written[None, :]
            assert np.array_equal(gs.view(np.uint32)[mask], full[mask])
            assert (gs.view(np.uint32)[~mask] == SENTINEL * 0x01010101).all()
        else:
            full = _colmajor_ue8m0(ref_scale, R4)
            mask = np.zeros(((G + 3) // 4, R4, 4), bool)
            for g in range(G):
                mask[g // 4, :cap, g % 4] = rows_written
            assert np.array_equal(gs[mask], full[mask])
            assert (gs[~mask] == SENTINEL).all()
    # combine over the aligned rows
    eo_h = random_bf16(np.random.default_rng(52), (cap, H))
    eo = torch.from_numpy(eo_h.view(np.int16)).cuda().view(torch.bfloat16)
    out = filled((T, H), torch.bfloat16)
    m.moe_combine_ex("normal", eo, ids, wt, E, s2d, seg, out, st, expert_out_rows=cap)
    meta = oracle.Meta(om.seg_indptr, om.src2dst, om.reorder_topk_ids, om.masked_m, om.partition_counts, 0, 0)
    want = oracle.combine("normal", eo_h, w.topk_ids, w.topk_weights, meta, E)
    torch.cuda.synchronize()
    check_combine(bytes_of(out).view(np.uint16).reshape(T, H), want)
    assert int(st.item()) == 0


@pytest.mark.parametrize("T,M", [(96, 30), (1100, 300)])   # register path; bulk kernel
@pytest.mark.parametrize("quant", ["fp8g128", "fp8g128_ue8m0"])
def test_masked_colmajor_scales(quant, T, M):
    """Masked layout [E, M, .] with per-expert column-major scales [E, G, roundup(M, 4)]."""
    m = moe()
    H, E, K = 1024, 16, 4
    w = make_case(T, H, E, K, seed=53, invalid_rate=0.05)
    x, ids, _ = to_dev(w)
    om = oracle.route_meta(w.topk_ids, E, M=M)
    seg = torch.from_numpy(om.seg_indptr).cuda()
    s2d = torch.from_numpy(om.src2dst).cuda()
    G, M4 = H // 128, (M + 3) // 4 * 4
    q = filled((E, M, H), torch.uint8)
    if quant == "fp8g128":
        scales = filled((E, G, M4), torch.float32)
    else:
        scales = filled((E, (G + 3) // 4, M4, 4), torch.uint8)
    st = m.new_status()
    m.moe_dispatch_ex("masked", quant, "col", x, ids, E, s2d, seg, q, scales, st, max_tokens_per_expert=M)
    torch.cuda.synchronize()
    gq, gs = q.cpu().numpy(), scales.cpu().numpy()
    flat = w.topk_ids.reshape(-1)
    for i, d in enumerate(om.src2dst):
        if d < 0:
            continue
        e, r = int(flat[i]), int(d - om.seg_indptr[flat[i]])
        if r >= M:
            continue
        if quant == "fp8g128":
            oq, os_ = oracle.quant_fp8_row(w.x[i // K])
            assert np.array_equal(gs[e, :, r].view(np.uint32), os_.view(np.uint32))
        else:
            oq, os_ = oracle.quant_fp8_ue8m0_row(w.x[i // K])
            assert np.array_equal(np.array([gs[e, g // 4, r, g % 4] for g in range(G)], np.uint8), os_)
        assert np.array_equal(gq[e, r], oq)


def test_ue8m0_through_fused_route_dispatch():
    """moe_route_dispatch with UE8M0 scales (the fused small-batch kernel), masked layout."""
    m = moe()
    w = make_case(128, 7168, 256, 8, seed=54, mode="masked", M=128, routing="softmax")
    x, ids, _ = to_dev(w)
    d = m.MoEDispatcher(128, 7168, 8, 256, mode="masked", quant="fp8g128_ue8m0", max_tokens_per_expert=128)
    d.route_dispatch(x, ids)
    om = oracle.route_meta(w.topk_ids, 256, M=128)
    torch.cuda.synchronize()
    gq, gs = d.out_q.cpu().numpy(), d.out_scales.cpu().numpy()
    flat = w.topk_ids.reshape(-1)
    for i, dd in enumerate(om.src2dst):
        e, r = int(flat[i]), int(dd - om.seg_indptr[flat[i]])
        oq, os_ = oracle.quant_fp8_ue8m0_row(w.x[i // 8])
        assert np.array_equal(gq[e, r], oq) and np.array_equal(gs[e, r], os_)
    d.check()


# --- f4: int64 topk_ids and per-tensor FP8 pass-through rows ---------------------------------

@pytest.mark.parametrize("T,K,E", [(128, 8, 256), (5000, 8, 64)])
def test_int64_ids_match_int32_metadata(T, K, E):
    m = moe()
    w = make_case(T, 16, E, K, seed=T + 71, invalid_rate=0.05, bad_rate=0.01)
    ids64 = w.topk_ids.astype(np.int64)
    # a few ids whose low 32 bits alias valid experts: they must count as bad, not as experts
    ids64.reshape(-1)[::97] = (np.int64(1) << 40) + 3
    want_ids = np.where((ids64 >= -(1 << 31)) & (ids64 < (1 << 31)), ids64, np.int64(1 << 31) - 1).astype(np.int32)
    om = oracle.route_meta(want_ids, E)
    d64 = torch.from_numpy(ids64).cuda()
    seg = torch.empty(E + 1, dtype=torch.int64, device="cuda")
    s2d = torch.empty(T * K, dtype=torch.int32, device="cuda")
    reo = torch.empty(T * K, dtype=torch.int32, device="cuda")
    mm = torch.empty(E, dtype=torch.int32, device="cuda")
    i32 = torch.empty((T, K), dtype=torch.int32, device="cuda")
    st = m.new_status()
    m.moe_route_meta_ex(d64, E, seg, s2d, reo, mm, st, m.new_workspace(T, K, E), topk_ids_i32_out=i32)
    torch.cuda.synchronize()
    n = om.num_valid
    assert np.array_equal(seg.cpu().numpy(), om.seg_indptr)
    assert np.array_equal(s2d.cpu().numpy(), om.src2dst)
    assert np.array_equal(reo[:n].cpu().numpy(), om.reorder_topk_ids)
    assert np.array_equal(i32.cpu().numpy(), want_ids)
    assert int(st.item()) == m.MOE_ERR_BAD_EXPERT_ID


@pytest.mark.parametrize("mode,M", [("normal", 0), ("masked", 64)])
def test_fp8_passthrough_dispatch(mode, M):
    m = moe()
    T, H, E, K = 200, 2048, 32, 4
    w = make_case(T, H, E, K, seed=72, invalid_rate=0.05)
    codes = np.random.default_rng(73).integers(0, 256, size=(T, H), dtype=np.uint8)
    xc = torch.from_numpy(codes).cuda()
    _, ids, _ = to_dev(w)
    om = oracle.route_meta(w.topk_ids, E, M=M)
    seg = torch.from_numpy(om.seg_indptr).cuda()
    s2d = torch.from_numpy(om.src2dst).cuda()
    q = filled((T * K, H) if mode == "normal" else (E, M, H), torch.uint8)
    st = m.new_status()
    m.moe_dispatch(mode, "fp8_passthrough", xc, ids, E, s2d, seg, q, None, st, M)
    want, _ = oracle.dispatch(mode, "fp8_passthrough", codes, w.topk_ids, om, E, M=M, fill=SENTINEL)
    torch.cuda.synchronize()
    assert np.array_equal(q.cpu().numpy(), want)
    # the same through the fused small-batch call
    d = m.MoEDispatcher(T, H, K, E, mode=mode, quant="fp8_passthrough", max_tokens_per_expert=M)
    d.out_q = filled(tuple(q.shape), torch.uint8)
    d.route_dispatch(xc, ids)
    torch.cuda.synchronize()
    assert np.array_equal(d.out_q.cpu().numpy(), want)
    d.check()


def test_ue8m0_bulk_path_normal_layout():
    """>= 1024 tokens with 16-byte UE8M0 scale rows (H = 2048): the bulk dispatch path."""
    m = moe()
    T, H, E, K = 1200, 2048, 64, 8
    w = make_case(T, H, E, K, seed=81, routing="zipf", invalid_rate=0.05)
    x, ids, _ = to_dev(w)
    om = oracle.route_meta(w.topk_ids, E)
    seg = torch.from_numpy(om.seg_indptr).cuda()
    s2d = torch.from_numpy(om.src2dst).cuda()
    q = filled((T * K, H), torch.uint8)
    sc = filled((T * K, H // 128), torch.uint8)
    st = m.new_status()
    m.moe_dispatch("normal", "fp8g128_ue8m0", x, ids, E, s2d, seg, q, sc, st)
    torch.cuda.synchronize()
    gq, gs = q.cpu().numpy(), sc.cpu().numpy()
    for i, d in enumerate(om.src2dst):
        if d < 0:
            continue
        oq, oe = oracle.quant_fp8_ue8m0_row(w.x[i // K])
        assert np.array_equal(gq[d], oq) and np.array_equal(gs[d], oe)
    n = om.num_valid
    assert (gq[n:] == SENTINEL).all() and (gs[n:] == SENTINEL).all()
    assert int(st.item()) == 0


# --- NVFP4 block scales in the 128 x 4 swizzled layout (nvfp4_block_scale_interleave) --------

@pytest.mark.parametrize("mode,T,H,E,K,M,offset", [
    ("normal", 300, 1024, 24, 6, 0, 4),      # scale buffer 4-byte aligned only: words stored in place
    ("masked", 1100, 7168, 64, 8, 200, 4),
    ("masked", 96, 1024, 16, 4, 30, 12),
])
def test_nvfp4_swizzled_scales_unaligned_buffer(mode, T, H, E, K, M, offset):
    """A swizzled scale buffer that is 4- but not 16-byte aligned gets the same bytes (its tiles
    cleared, then every scale word stored at its tile position) as an aligned one."""
    _swizzled_case(mode, T, H, E, K, M, offset)


@pytest.mark.parametrize("mode,T,H,E,K,M", [
    ("normal", 300, 1024, 24, 6, 0),     # 1800 rows -> padded to 1920
    ("normal", 1500, 2048, 64, 8, 0),    # >= 1024 tokens: the bulk kernel, its threads storing the scales
    ("normal", 1030, 256, 16, 3, 0),     # bulk kernel, 3090 rows -> padded to 3200
    ("masked", 96, 1024, 16, 4, 30),     # E*M = 480 rows -> padded to 512
    ("masked", 128, 7168, 256, 8, 128),  # the decode shape: 32768 rows, no padding
    ("masked", 1100, 7168, 64, 8, 200),  # bulk kernel, masked rows
    ("masked", 1100, 1088, 64, 8, 200),  # H % 256 != 0: the bulk kernel still stores the swizzled words
])
def test_nvfp4_swizzled_scales_match_oracle_interleave(mode, T, H, E, K, M):
    """The whole scale buffer equals the oracle's row-major scales passed through the interleave,
    where every 128-row block the call touches is written in full (rows no pair maps to are zero,
    and so are the padding rows) and every other block keeps its fill; codes unchanged."""
    _swizzled_case(mode, T, H, E, K, M, 0)


def _swizzled_case(mode, T, H, E, K, M, offset):
    m = moe()
    w = make_case(T, H, E, K, seed=T + H, mode=mode, quant="nvfp4b16", M=M, invalid_rate=0.05)
    x, ids, _ = to_dev(w)
    om = oracle.route_meta(w.topk_ids, E, M=M)
    seg = torch.from_numpy(om.seg_indptr).cuda()
    s2d = torch.from_numpy(om.src2dst).cuda()
    R = T * K if mode == "normal" else E * M
    q = filled((R, H // 2), torch.uint8)
    nsf = m.swizzled_scale_bytes(R, H)
    sf = filled((nsf + 16,), torch.uint8)[offset:offset + nsf]
    st = m.new_status()
    m.moe_dispatch_ex(mode, "nvfp4b16", "swizzled", x, ids, E, s2d, seg, q, sf, st, max_tokens_per_expert=M,
                      input_global_scale=w.global_scale)
    oq, osf = oracle.dispatch(mode, "nvfp4b16", w.x, w.topk_ids, om, E, M=M, global_scale=w.global_scale,
                              rows=R if mode == "normal" else None, fill=SENTINEL)
    written = np.zeros(R, bool)
    rows = om.src2dst[om.src2dst >= 0] if mode == "normal" else masked_rows(w, om)
    written[rows[rows >= 0]] = True
    touched = np.ones(R, bool) if mode == "normal" else masked_touched_rows(om.seg_indptr, E, M)
    want_sf = swizzled_scales_expected(osf.reshape(R, H // 16), written, touched)
    torch.cuda.synchronize()
    assert np.array_equal(bytes_of(q).reshape(-1), oq.reshape(-1))
    assert np.array_equal(sf.cpu().numpy(), want_sf)
    assert int(st.item()) == 0    # the dispatch drops pairs past capacity silently (route_meta reports them)


def test_nvfp4_masked_swizzled_workload_in_full():
    """The nvfp4 workload (T=8192, H=7168, E=256, K=8, M=8192) with swizzled scales, in the
    benchmark's launch configuration: every written code row against the oracle; every touched
    128-row block of the [E*M, H/16] scale matrix equal to the oracle's interleave of its
    expected rows (the expert's scale rows, zeros below the block's end); every other byte of
    both buffers still the fill. The host builds the touched blocks only (the buffers are
    7.5 GB and 0.9 GB)."""
    m = moe()
    w = make_workload("nvfp4")
    x, ids, _ = to_dev(w)
    E, M, H, K = w.E, w.M, w.H, w.K
    C = H // 16
    om = oracle.route_meta(w.topk_ids, E, M=M)
    seg = torch.from_numpy(om.seg_indptr).cuda()
    s2d = torch.from_numpy(om.src2dst).cuda()
    R = E * M
    q = _sentinel_buffer((R, H // 2), torch.uint8)
    nsf = m.swizzled_scale_bytes(R, H)
    assert nsf == R * C
    sf = _sentinel_buffer((nsf,), torch.uint8)
    st = m.new_status()
    m.moe_dispatch_ex("masked", "nvfp4b16", "swizzled", x, ids, E, s2d, seg, q, sf, st, max_tokens_per_expert=M,
                      input_global_scale=w.global_scale)
    n = om.num_valid
    valid = om.src2dst >= 0
    pair_of_slot = np.empty(n, np.int64)
    pair_of_slot[om.src2dst[valid]] = np.nonzero(valid)[0]
    dst = masked_rows(w, om)[pair_of_slot]        # masked row of contiguous slot j
    assert (dst >= 0).all()
    oq, osc = oracle.dispatch("normal", "nvfp4b16", w.x, w.topk_ids, om, E, global_scale=w.global_scale, rows=n)
    osc = np.ascontiguousarray(osc[:n]).view(np.uint8).reshape(n, C)
    dst_d = torch.from_numpy(dst).cuda()
    got = q.index_select(0, dst_d)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert np.array_equal(got.cpu().numpy(), np.ascontiguousarray(oq[:n]).view(np.uint8).reshape(n, -1)), "codes"
    q.index_fill_(0, dst_d, SENTINEL)
    assert _all_bytes_are(q, SENTINEL), "rows no pair maps to were written"
    del q, got

    blk = np.unique(np.nonzero(masked_touched_rows(om.seg_indptr, E, M))[0] // 128)
    slot_of_row = np.full(R, -1, np.int64)
    slot_of_row[dst] = np.arange(n)
    sl = slot_of_row[(blk[:, None] * 128 + np.arange(128)).reshape(-1)]
    rows = np.zeros((blk.size * 128, C), np.uint8)
    rows[sl >= 0] = osc[sl[sl >= 0]]
    want = oracle.nvfp4_sf_interleave(rows).reshape(blk.size, 128 * C)
    sf2 = sf.view(R // 128, 128 * C)
    blk_d = torch.from_numpy(blk).cuda()
    assert np.array_equal(sf2.index_select(0, blk_d).cpu().numpy(), want), "touched scale blocks"
    sf2.index_fill_(0, blk_d, SENTINEL)
    assert _all_bytes_are(sf2, SENTINEL), "untouched scale blocks were written"
