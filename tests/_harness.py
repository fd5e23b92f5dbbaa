"""Test harness: runs one seeded workload through the CUDA library (via the C ABI
binding) and through the CPU oracle, and compares them.

Bars (the method's own): bit-exact for the metadata, the gathered bf16 rows and the
quantised bytes/scales; the combine within 1e-2 relative / 1e-3 absolute of the
oracle's binary64 sum rounded to bf16 (elementwise |gpu - oracle| <= 1e-3 + 1e-2*|oracle|).
"""
from __future__ import annotations

from typing import Optional

import numpy as np
import torch

import oracle
from workloads import Workload, bf16_bits_to_f32, random_bf16

RTOL = 1e-2
ATOL = 1e-3
SENTINEL = 0xA5

STATUS_OF_ORACLE = {0: {0}, oracle.BAD_ID: {4}, oracle.CAPACITY: {3}, oracle.BAD_ID | oracle.CAPACITY: {3, 4}}


def moe():
    import combine_moe_route_meta_gb300 as m
    return m


def to_dev(w: Workload):
    x = torch.from_numpy(np.ascontiguousarray(w.x).view(np.int16)).cuda().view(torch.bfloat16)
    ids = torch.from_numpy(np.ascontiguousarray(w.topk_ids)).cuda()
    wt = torch.from_numpy(np.ascontiguousarray(w.topk_weights)).cuda()
    return x, ids, wt


def bytes_of(t: torch.Tensor) -> np.ndarray:
    """Host copy of a device tensor's raw bytes, shaped [rows, row_bytes]."""
    rows = t.shape[0] if t.dim() > 1 else 1
    a = t.contiguous().view(torch.uint8).cpu().numpy()
    width = a.size // rows if rows else 0
    return a.reshape(rows, width)


GUARD_BYTES = 4096
_GUARDED = []  # (whole allocation, inner bytes, fill) of every buffer made by filled()


def filled(shape, dtype, fill=SENTINEL) -> torch.Tensor:
    """A device buffer of `shape` filled with the byte `fill`, placed between two guard
    margins of GUARD_BYTES holding the same byte; check_guards() verifies that no kernel
    wrote outside the buffer (the canary check used instead of a memory checker)."""
    n = int(np.prod(shape)) * torch.empty(0, dtype=dtype).element_size()
    whole = torch.full((n + 2 * GUARD_BYTES,), fill, dtype=torch.uint8, device="cuda")
    _GUARDED.append((whole, n, fill))
    return whole[GUARD_BYTES:GUARD_BYTES + n].view(dtype).view(shape)


def check_guards():
    """Every guard margin of the buffers made by filled() since the last check still holds
    its fill byte."""
    torch.cuda.synchronize()
    try:
        for whole, n, fill in _GUARDED:
            margins = torch.cat([whole[:GUARD_BYTES], whole[GUARD_BYTES + n:]])
            bad = int((margins != fill).sum().item())
            assert bad == 0, f"{bad} guard bytes around a {n}-byte output buffer were overwritten"
    finally:
        _GUARDED.clear()


def check_meta(w: Workload, om: oracle.Meta, gm, status: torch.Tensor):
    n = om.num_valid
    assert np.array_equal(gm.seg_indptr.cpu().numpy(), om.seg_indptr), "seg_indptr"
    assert np.array_equal(gm.src2dst.cpu().numpy(), om.src2dst), "src2dst"
    assert np.array_equal(gm.reorder_topk_ids[:n].cpu().numpy(), om.reorder_topk_ids), "reorder_topk_ids"
    assert np.array_equal(gm.masked_m.cpu().numpy(), om.masked_m), "masked_m"
    assert np.array_equal(gm.partition_counts.cpu().numpy(), om.partition_counts), "partition_counts"
    assert gm.expected_m == om.expected_m
    assert int(status.item()) in STATUS_OF_ORACLE[om.status], (int(status.item()), om.status)


def gpu_meta(w: Workload, ids: torch.Tensor):
    m = moe()
    status = m.new_status()
    gm = m.route_meta(ids, w.E, num_partitions=w.P, max_tokens_per_expert=w.M, dev_status=status)
    return gm, status


def check_combine(got_bits: np.ndarray, want_bits: np.ndarray, what="combine"):
    g = bf16_bits_to_f32(got_bits).astype(np.float64)
    o = bf16_bits_to_f32(want_bits).astype(np.float64)
    err = np.abs(g - o)
    bad = err > ATOL + RTOL * np.abs(o)
    assert not bad.any(), f"{what}: {int(bad.sum())} elements out of tolerance, max err {err.max()}"


def masked_rows(w: Workload, om: oracle.Meta):
    """Masked-layout row of every valid pair (flattened pair order), -1 where dropped/invalid."""
    flat = w.topk_ids.reshape(-1)
    rows = np.full(flat.size, -1, np.int64)
    v = om.src2dst >= 0
    e = flat[v].astype(np.int64)
    rank = om.src2dst[v].astype(np.int64) - om.seg_indptr[e]
    r = np.where(rank < w.M, e * w.M + rank, -1)
    rows[np.nonzero(v)[0]] = r
    return rows


def run_full(w: Workload, *, expert_seed: int = 1234, check_untouched: bool = True):
    """Meta + dispatch + combine on the GPU, each compared in full with the oracle."""
    m = moe()
    x, ids, wt = to_dev(w)
    om = oracle.route_meta(w.topk_ids, w.E, P=w.P, M=w.M)
    gm, status = gpu_meta(w, ids)
    torch.cuda.synchronize()
    check_meta(w, om, gm, status)

    # ---- dispatch ----
    qs, qd, ss, sd = m.dispatch_out_shapes(w.mode, w.quant, w.T, w.H, w.K, w.E, w.M)
    q = filled(qs, qd)
    s = filled(ss, sd) if ss is not None else None
    st2 = m.new_status()
    if w.T:
        m.moe_dispatch(w.mode, w.quant, x, ids, w.E, gm.src2dst, gm.seg_indptr, q, s, st2, w.M,
                       w.global_scale or 0.0)
    oq, osc = oracle.dispatch(w.mode, w.quant, w.x, w.topk_ids, om, w.E, M=w.M,
                              global_scale=w.global_scale or 0.0, fill=SENTINEL)
    torch.cuda.synchronize()
    gq = bytes_of(q)
    oqb = np.ascontiguousarray(oq).view(np.uint8).reshape(gq.shape)
    if check_untouched:
        assert np.array_equal(gq, oqb), "dispatch rows (incl. untouched sentinel rows)"
    else:
        n = om.num_valid
        assert np.array_equal(gq[:n], oqb[:n])
    if s is not None:
        gs = bytes_of(s)
        osb = np.ascontiguousarray(osc).view(np.uint8).reshape(gs.shape)
        assert np.array_equal(gs, osb), "dispatch scales"
    assert int(st2.item()) == 0

    # ---- combine ----
    rng = np.random.default_rng(expert_seed)
    if w.mode == "normal":
        eo_host = random_bf16(rng, (max(w.T * w.K, 1), w.H))
    else:
        eo_host = random_bf16(rng, (w.E * w.M, w.H))
    eo = torch.from_numpy(eo_host.view(np.int16)).cuda().view(torch.bfloat16)
    out = filled((w.T, w.H), torch.bfloat16)
    st3 = m.new_status()
    if w.T:
        m.moe_combine(w.mode, eo, ids, wt, w.E, gm.src2dst, gm.seg_indptr, out, st3, w.M)
    want = oracle.combine(w.mode, eo_host, w.topk_ids, w.topk_weights, om, w.E, M=w.M)
    torch.cuda.synchronize()
    check_combine(bytes_of(out).view(np.uint16).reshape(w.T, w.H), want)
    assert int(st3.item()) == 0
    return om


def swizzled_scales_expected(osf: np.ndarray, written: np.ndarray, touched_rows: np.ndarray) -> np.ndarray:
    """The expected swizzled NVFP4 scale buffer: the oracle's row-major scales osf [R, C] (rows no
    pair maps to hold the fill) with every unwritten row of a touched 128-row block set to zero,
    through the oracle's interleave (which zero-pads to a multiple of 128 rows).

    written:      bool [R], the rows a pair maps to.
    touched_rows: bool [R], the rows that decide which blocks the call touches (the block holding
                  the padding rows, if any, is touched as well)."""
    R = osf.shape[0]
    nb = (R + 127) // 128
    blk = np.zeros(nb, bool)
    idx = np.nonzero(touched_rows)[0]
    blk[idx // 128] = True
    if R % 128:
        blk[-1] = True
    in_touched = np.repeat(blk, 128)[:R]
    out = osf.copy()
    out[in_touched & ~written] = 0
    return oracle.nvfp4_sf_interleave(out)


def masked_touched_rows(seg: np.ndarray, E: int, M: int) -> np.ndarray:
    """Rows e*M + [0, min(M, seg[e+1] - seg[e])) of the masked layout [E*M]."""
    rows = np.zeros(E * M, bool)
    for e in range(E):
        n = min(M, int(seg[e + 1] - seg[e]))
        rows[e * M:e * M + n] = True
    return rows


def partitioned_routed(topk_ids: np.ndarray, E: int, P: int, S: int) -> np.ndarray:
    """bool [P*S]: slot t of partition p receives token t (some valid id of t lies in p)."""
    T, K = topk_ids.shape
    ep = E // P
    routed = np.zeros((P, S), bool)
    for k in range(K):
        e = topk_ids[:, k]
        ok = (e >= 0) & (e < E)
        routed[e[ok] // ep, np.nonzero(ok)[0]] = True
    return routed.reshape(-1)


def partitioned_touched_rows(P: int, S: int, T: int) -> np.ndarray:
    """Slots [0, T) of every partition's S receive slots."""
    rows = np.zeros((P, S), bool)
    rows[:, :T] = True
    return rows.reshape(-1)


def _sentinel_buffer(shape, dtype) -> torch.Tensor:
    """A device buffer of `shape` whose every byte is SENTINEL."""
    n = int(np.prod(shape)) * torch.empty(0, dtype=dtype).element_size()
    return torch.full((n,), SENTINEL, dtype=torch.uint8, device="cuda").view(dtype).view(shape)


def _all_bytes_are(t2d: torch.Tensor, value: int, chunk_bytes: int = 1 << 30) -> bool:
    """Every byte of a [rows, bytes] uint8 device tensor equals `value` (checked in row chunks,
    so no temporary the size of a multi-GB buffer is made)."""
    rows = max(1, chunk_bytes // max(1, t2d.shape[1]))
    for r0 in range(0, t2d.shape[0], rows):
        if bool((t2d[r0:r0 + rows] != value).any()):
            return False
    return True


def run_full_large(w: Workload, *, expert_seed: int = 4321):
    """A full-size workload in the benchmark's launch configuration, compared in full.

    Metadata: every entry. Dispatch: every written row and scale row, bit for bit, against
    the oracle's rows in src2dst order (the contiguous layout: out[src2dst[i]] = Q(x[t]));
    in the masked layout each row e*M + rank is the contiguous row seg_indptr[e] + rank by
    definition, so the GPU's masked rows are gathered into that order on the device first.
    Every other row of the output (beyond N, or at slots >= masked_m[e]) must still hold the
    sentinel fill. Combine: every element of every token, against the oracle's binary64 sum
    over the compact expert rows (the masked buffer holds the same rows at e*M + rank).
    The host never materialises the [E, M, .] buffers, which run to tens of GB."""
    m = moe()
    x, ids, wt = to_dev(w)
    om = oracle.route_meta(w.topk_ids, w.E, P=w.P, M=w.M)
    gm, status = gpu_meta(w, ids)
    torch.cuda.synchronize()
    check_meta(w, om, gm, status)
    assert om.status == 0

    qs, qd, ss, sd = m.dispatch_out_shapes(w.mode, w.quant, w.T, w.H, w.K, w.E, w.M)
    q = _sentinel_buffer(qs, qd)
    s = _sentinel_buffer(ss, sd) if ss is not None else None
    st2 = m.new_status()
    m.moe_dispatch(w.mode, w.quant, x, ids, w.E, gm.src2dst, gm.seg_indptr, q, s, st2, w.M,
                   w.global_scale or 0.0)

    n = om.num_valid
    valid = om.src2dst >= 0
    pair_of_slot = np.empty(n, np.int64)
    pair_of_slot[om.src2dst[valid]] = np.nonzero(valid)[0]
    rows = om.src2dst.astype(np.int64) if w.mode == "normal" else masked_rows(w, om)
    dst = rows[pair_of_slot]                      # output row of contiguous slot j
    assert (dst >= 0).all()                       # no capacity drops in these workloads

    # oracle: the contiguous layout of all N rows
    oq, osc = oracle.dispatch("normal", w.quant, w.x, w.topk_ids, om, w.E, global_scale=w.global_scale or 0.0,
                              rows=max(n, 1))
    q2 = q.view(torch.uint8).view(int(np.prod(qs[:-1])), -1)
    dst_d = torch.from_numpy(dst).cuda()
    got_rows = q2.index_select(0, dst_d)
    torch.cuda.synchronize()
    assert int(st2.item()) == 0
    assert np.array_equal(got_rows.cpu().numpy(), np.ascontiguousarray(oq[:n]).view(np.uint8).reshape(n, -1)), \
        "dispatch rows"
    # the written rows are checked: overwrite them with the fill, then every byte must be the fill
    q2.index_fill_(0, dst_d, SENTINEL)
    assert _all_bytes_are(q2, SENTINEL), "rows no pair maps to were written"
    if s is not None:
        s2 = s.view(torch.uint8).view(q2.shape[0], -1)
        got_sc = s2.index_select(0, dst_d)
        assert np.array_equal(got_sc.cpu().numpy(), np.ascontiguousarray(osc[:n]).view(np.uint8).reshape(n, -1)), \
            "dispatch scales"
        s2.index_fill_(0, dst_d, SENTINEL)
        assert _all_bytes_are(s2, SENTINEL), "scale rows no pair maps to were written"
    del q, s, q2, got_rows

    # combine over compact expert rows (row j of eo_compact is the expert output of slot j)
    rng = np.random.default_rng(expert_seed)
    eo_compact = random_bf16(rng, (max(n, 1), w.H))
    eo_c = torch.from_numpy(eo_compact.view(np.int16)).cuda().view(torch.bfloat16)
    if w.mode == "normal":
        eo = eo_c
    else:
        eo = torch.zeros((w.E * w.M, w.H), dtype=torch.bfloat16, device="cuda")
        eo.index_copy_(0, dst_d, eo_c[:n])
    out = filled((w.T, w.H), torch.bfloat16)
    st3 = m.new_status()
    m.moe_combine(w.mode, eo, ids, wt, w.E, gm.src2dst, gm.seg_indptr, out, st3, w.M)
    want = oracle.combine("normal", eo_compact, w.topk_ids, w.topk_weights, om, w.E)
    torch.cuda.synchronize()
    assert int(st3.item()) == 0
    check_combine(bytes_of(out).view(np.uint16).reshape(w.T, w.H), want)
    return om


def run_partitioned_dispatch(w: Workload, P: int, S: int, layout: str, invalid_id: int = -1):
    """moe_dispatch_partitioned_ex of an NVFP4 workload against oracle.dispatch_partitioned, in
    full: every receive code row (untouched rows keep the fill), the scales (row-major, or the
    swizzled layout's expected bytes), ids and weights, and the status word."""
    m = moe()
    x, ids, wt = to_dev(w)
    H, E, K = w.H, w.E, w.K
    g = w.global_scale if w.global_scale is not None else 0.0
    rx = filled((P, S, H // 2), torch.uint8)
    rsf = filled((m.swizzled_scale_bytes(P * S, H),) if layout == "swizzled" else (P, S, H // 16), torch.uint8)
    rids = filled((P, S, K), torch.int32)
    rw = filled((P, S, K), torch.float32)
    st = m.new_status()
    m.moe_dispatch_partitioned_ex("nvfp4b16", layout, x, ids, wt, E, P, rx, rsf, rids, rw, st,
                                  invalid_expert_id=invalid_id, input_global_scale=g)
    ox, osf, oids, ow = oracle.dispatch_partitioned("nvfp4b16", w.x, w.topk_ids, w.topk_weights, E, P,
                                                    invalid_id=invalid_id, global_scale=g, num_slots=S, fill=SENTINEL)
    torch.cuda.synchronize()
    assert np.array_equal(bytes_of(rx).reshape(-1), np.ascontiguousarray(ox).view(np.uint8).reshape(-1)), "codes"
    if layout == "swizzled":
        want = swizzled_scales_expected(osf.reshape(P * S, H // 16), partitioned_routed(w.topk_ids, E, P, S),
                                        partitioned_touched_rows(P, S, w.T))
    else:
        want = osf
    assert np.array_equal(rsf.cpu().numpy().reshape(-1), np.asarray(want).reshape(-1)), "scales"
    assert np.array_equal(rids.cpu().numpy(), oids), "ids"
    assert np.array_equal(rw.cpu().numpy().view(np.uint32), ow.view(np.uint32)), "weights"
    assert int(st.item()) == 0
    check_guards()
