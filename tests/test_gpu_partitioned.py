"""GPU parity of the per-partition layout (moe_dispatch_layout) and the FlashInfer
all-to-all layout (moe_dispatch_partitioned / moe_combine_partitioned) against the oracle.

Layout, receive rows, sanitised ids, weights and NVFP4 codes/scales are compared bit for
bit, including the payload the kernels must leave untouched; the combine within
1e-2 relative / 1e-3 absolute.
"""
import numpy as np
import pytest
import torch

import oracle
from workloads import make_case, make_workload, random_bf16

from _harness import (SENTINEL, bytes_of, check_combine, filled, moe, partitioned_routed, partitioned_touched_rows,
                      run_partitioned_dispatch,
                      swizzled_scales_expected, to_dev)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T,E,K,P,bad", [
    (0, 16, 4, 4, 0.0), (1, 8, 2, 1, 0.0), (300, 64, 6, 8, 0.0), (5000, 256, 8, 32, 0.02), (16384, 128, 8, 8, 0.0),
    (500, 256, 8, 8, 0.02),        # one block, bad ids reported
    (512, 1024, 8, 1024, 0.0),     # the largest one-block case: 4096 ids and 2 x 1024 counters in shared memory
    (513, 1024, 8, 1024, 0.0),     # one token more: the multi-block kernel
])
def test_dispatch_layout_matches_oracle(T, E, K, P, bad):
    m = moe()
    w = make_case(T, 16, E, K, seed=T + P, invalid_rate=0.05, bad_rate=bad,
                  routing="replace" if T == 5000 else "uniform")
    _, ids, _ = to_dev(w)
    ntr = torch.full((P,), -1, dtype=torch.int32, device="cuda")
    itr = torch.full((max(T, 1), P), 7, dtype=torch.uint8, device="cuda")[:T]
    nte = torch.full((E,), -1, dtype=torch.int32, device="cuda")
    st = m.new_status()
    m.moe_dispatch_layout(ids, E, P, ntr, itr, st, nte)
    o_ntr, o_itr, o_nte = oracle.dispatch_layout(w.topk_ids, E, P)
    torch.cuda.synchronize()
    assert np.array_equal(ntr.cpu().numpy(), o_ntr)
    assert np.array_equal(itr.cpu().numpy().astype(bool), o_itr)
    assert np.array_equal(nte.cpu().numpy(), o_nte)
    assert int(st.item()) == (m.MOE_ERR_BAD_EXPERT_ID if bad else 0)


@pytest.mark.parametrize("T,S,H,E,K,P,quant,inv", [
    (64, 64, 256, 16, 4, 4, "none", -1),
    (50, 61, 1040, 32, 6, 8, "nvfp4b16", 32),       # padding slots, ragged 512-slice, invalid id = E
    (128, 128, 7168, 256, 8, 8, "nvfp4b16", -1),    # the FlashInfer NVFP4 payload shape (decode-sized)
    (512, 600, 4096, 128, 8, 8, "none", 128),
    (37, 37, 128, 64, 16, 32, "none", -1),          # P = 32 (one lane per partition), K = 16
    (20, 20, 64, 4, 2, 1, "nvfp4b16", -1),          # a single partition
    # >= 1024 tokens with 16-byte row geometry: the bulk (TMA) kernels
    (1100, 1200, 2048, 64, 8, 8, "nvfp4b16", -1),   # padding slots
    (1030, 1030, 512, 32, 4, 4, "none", 32),        # invalid id = E
    (2000, 2050, 256, 64, 16, 32, "nvfp4b16", -1),  # K = 16, P = 32
    (1024, 1024, 1088, 16, 2, 2, "nvfp4b16", -1),   # H % 256 != 0: bulk kernel, scale bytes stored by its threads
])
def test_partitioned_dispatch_and_combine_match_oracle(T, S, H, E, K, P, quant, inv):
    m = moe()
    w = make_case(T, H, E, K, seed=T * 3 + P, quant=quant, invalid_rate=0.05)
    x, ids, wt = to_dev(w)
    g = w.global_scale or 0.0
    if quant == "nvfp4b16":
        rx = filled((P, S, H // 2), torch.uint8)
        rsf = filled((P, S, H // 16), torch.uint8)
    else:
        rx = filled((P, S, H), torch.bfloat16)
        rsf = None
    rids = filled((P, S, K), torch.int32)
    rw = filled((P, S, K), torch.float32)
    st = m.new_status()
    m.moe_dispatch_partitioned(quant, x, ids, wt, E, P, rx, rsf, rids, rw, st, invalid_expert_id=inv,
                               input_global_scale=g)
    ox, osf, oids, ow = oracle.dispatch_partitioned(quant, w.x, w.topk_ids, w.topk_weights, E, P, invalid_id=inv,
                                                    global_scale=g, num_slots=S, fill=SENTINEL)
    torch.cuda.synchronize()
    assert np.array_equal(bytes_of(rx), np.ascontiguousarray(ox).view(np.uint8).reshape(P, -1))
    if rsf is not None:
        assert np.array_equal(bytes_of(rsf), osf.reshape(P, -1))
    assert np.array_equal(rids.cpu().numpy(), oids)
    assert np.array_equal(rw.cpu().numpy().view(np.uint32), ow.view(np.uint32))
    assert int(st.item()) == 0

    partial_h = random_bf16(np.random.default_rng(T + S), (P, S, H))
    partial = torch.from_numpy(partial_h.view(np.int16)).cuda().view(torch.bfloat16)
    out = filled((T, H), torch.bfloat16)
    m.moe_combine_partitioned(partial, ids, E, P, out, st)
    want = oracle.combine_partitioned(partial_h, w.topk_ids, E, P)
    torch.cuda.synchronize()
    check_combine(bytes_of(out).view(np.uint16).reshape(T, H), want)


@pytest.mark.parametrize("layout", ["row", "swizzled", "swizzled_pad"])
def test_partitioned_nvfp4_workload_in_full(layout):
    """The nvfp4 workload (T=8192, H=7168, E=256, K=8, P=8, one receive slot per token) through
    the FlashInfer layout, in the benchmark's launch configuration: every receive row, scale,
    sanitised id and weight (row-major or swizzled scales), the untouched payload of slots a
    partition does not receive, and every element of the partitioned combine. swizzled_pad: 64
    padding slots per partition, so that tiles straddle partitions (the interleave pass)."""
    m = moe()
    w = make_workload("nvfp4")
    x, ids, wt = to_dev(w)
    P, S, K, H, E = w.P, w.T + (64 if layout == "swizzled_pad" else 0), w.K, w.H, w.E
    layout = "swizzled" if layout.startswith("swizzled") else layout
    rx = filled((P, S, H // 2), torch.uint8)
    rsf = filled((m.swizzled_scale_bytes(P * S, H),) if layout == "swizzled" else (P, S, H // 16), torch.uint8)
    rids = filled((P, S, K), torch.int32)
    rw = filled((P, S, K), torch.float32)
    st = m.new_status()
    m.moe_dispatch_partitioned_ex("nvfp4b16", layout, x, ids, wt, E, P, rx, rsf, rids, rw, st,
                                  input_global_scale=w.global_scale)
    ox, osf, oids, ow = oracle.dispatch_partitioned("nvfp4b16", w.x, w.topk_ids, w.topk_weights, E, P,
                                                    global_scale=w.global_scale, num_slots=S, fill=SENTINEL)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert np.array_equal(bytes_of(rx), np.ascontiguousarray(ox).view(np.uint8).reshape(P, -1))
    if layout == "swizzled":
        want = swizzled_scales_expected(osf.reshape(P * S, H // 16), partitioned_routed(w.topk_ids, E, P, S),
                                        partitioned_touched_rows(P, S, w.T))
        assert np.array_equal(rsf.cpu().numpy(), want)
    else:
        assert np.array_equal(bytes_of(rsf), osf.reshape(P, -1))
    assert np.array_equal(rids.cpu().numpy(), oids)
    assert np.array_equal(rw.cpu().numpy().view(np.uint32), ow.view(np.uint32))
    del rx, rsf, rids, rw, ox, osf

    partial_h = random_bf16(np.random.default_rng(77), (P, S, H))
    partial = torch.from_numpy(partial_h.view(np.int16)).cuda().view(torch.bfloat16)
    out = filled((w.T, H), torch.bfloat16)
    m.moe_combine_partitioned(partial, ids, E, P, out, st)
    want = oracle.combine_partitioned(partial_h, w.topk_ids, E, P)
    torch.cuda.synchronize()
    check_combine(bytes_of(out).view(np.uint16).reshape(w.T, H), want)
    assert int(st.item()) == 0


@pytest.mark.parametrize("T,S,H,E,K,P", [
    (20, 20, 64, 4, 2, 1),            # 20 rows -> padded to 128
    (50, 61, 1024, 32, 6, 8),         # 488 rows -> padded to 512, padding slots
    (128, 128, 7168, 256, 8, 8),      # the FlashInfer NVFP4 payload shape, 1024 rows
    (1100, 1130, 2048, 64, 8, 8),     # >= 1024 tokens: the bulk kernel, padding slots
    (1030, 1030, 256, 96, 6, 32),     # bulk kernel, 32 partitions, 32960 rows -> padded to 33024
    # num_slots % 128 == 0: every tile lies in one partition and is built whole in shared memory
    (1000, 1024, 1088, 64, 8, 8),     # ragged last token group (104 slots) and last column slice (1 tile)
    (300, 512, 256, 96, 6, 32),       # 32 partitions; the last slot group of each partition untouched
    (0, 128, 64, 4, 2, 1),            # no tokens: padding ids only, no tile touched
    (4096, 4096, 4096, 128, 8, 4),    # many units per CTA
    (700, 768, 512, 64, 16, 16),      # top-16, 16 partitions
])
def test_partitioned_swizzled_scales_match_oracle_interleave(T, S, H, E, K, P):
    """moe_dispatch_partitioned_ex with swizzled scales equals the row-major receive scales
    [P*S, H/16] passed through nvfp4_block_scale_interleave, where every 128-row block holding a
    slot t < T (or a padding row) is written in full: slots a partition does not receive are
    zero there, padding rows zero, other blocks keep their fill; codes, ids and weights as in
    the row-major layout."""
    m = moe()
    w = make_case(T, H, E, K, seed=T * 5 + P, quant="nvfp4b16", invalid_rate=0.05)
    x, ids, wt = to_dev(w)
    rx = filled((P, S, H // 2), torch.uint8)
    rsf = filled((m.swizzled_scale_bytes(P * S, H),), torch.uint8)
    rids = filled((P, S, K), torch.int32)
    rw = filled((P, S, K), torch.float32)
    st = m.new_status()
    m.moe_dispatch_partitioned_ex("nvfp4b16", "swizzled", x, ids, wt, E, P, rx, rsf, rids, rw, st,
                                  input_global_scale=w.global_scale or 0.0)
    ox, osf, oids, ow = oracle.dispatch_partitioned("nvfp4b16", w.x, w.topk_ids, w.topk_weights, E, P,
                                                    global_scale=w.global_scale or 0.0, num_slots=S, fill=SENTINEL)
    torch.cuda.synchronize()
    assert np.array_equal(bytes_of(rx), np.ascontiguousarray(ox).view(np.uint8).reshape(P, -1))
    want = swizzled_scales_expected(osf.reshape(P * S, H // 16), partitioned_routed(w.topk_ids, E, P, S),
                                    partitioned_touched_rows(P, S, T))
    assert np.array_equal(rsf.cpu().numpy(), want)
    assert np.array_equal(rids.cpu().numpy(), oids)
    assert np.array_equal(rw.cpu().numpy().view(np.uint32), ow.view(np.uint32))
    assert int(st.item()) == 0


@pytest.mark.parametrize("T,S,offset", [(200, 256, 4), (1100, 1152, 12)])
def test_partitioned_swizzled_scales_unaligned_buffer(T, S, offset):
    """A swizzled receive-scale buffer that is 4- but not 16-byte aligned (num_slots a multiple
    of 128): the tiles are cleared and the scale words stored one by one, with the same bytes as
    nvfp4_block_scale_interleave of the row-major receive scales."""
    m = moe()
    H, E, K, P = 1024, 64, 8, 8
    w = make_case(T, H, E, K, seed=T + offset, quant="nvfp4b16", invalid_rate=0.05)
    x, ids, wt = to_dev(w)
    rx = filled((P, S, H // 2), torch.uint8)
    nsf = m.swizzled_scale_bytes(P * S, H)
    base = filled((nsf + 16,), torch.uint8)
    rsf = base[offset:offset + nsf]
    rids = filled((P, S, K), torch.int32)
    rw = filled((P, S, K), torch.float32)
    st = m.new_status()
    m.moe_dispatch_partitioned_ex("nvfp4b16", "swizzled", x, ids, wt, E, P, rx, rsf, rids, rw, st,
                                  input_global_scale=w.global_scale)
    ox, osf, oids, ow = oracle.dispatch_partitioned("nvfp4b16", w.x, w.topk_ids, w.topk_weights, E, P,
                                                    global_scale=w.global_scale, num_slots=S, fill=SENTINEL)
    torch.cuda.synchronize()
    assert np.array_equal(bytes_of(rx), np.ascontiguousarray(ox).view(np.uint8).reshape(P, -1))
    want = swizzled_scales_expected(osf.reshape(P * S, H // 16), partitioned_routed(w.topk_ids, E, P, S),
                                    partitioned_touched_rows(P, S, T))
    got = base.cpu().numpy()
    assert np.array_equal(got[offset:offset + nsf], want)
    assert np.all(got[:offset] == SENTINEL) and np.all(got[offset + nsf:] == SENTINEL)
    assert np.array_equal(rids.cpu().numpy(), oids)
    assert np.array_equal(rw.cpu().numpy().view(np.uint32), ow.view(np.uint32))
    assert int(st.item()) == 0


@pytest.mark.parametrize("P,K,layout", [(1, 8, "row"), (4, 8, "row"), (16, 8, "row"), (32, 16, "row"),
                                        (4, 8, "swizzled"), (32, 16, "swizzled")])
def test_partitioned_nvfp4_ring_and_tiles_across_partition_counts(P, K, layout):
    """2048 tokens of the nvfp4 shape (H = 7168, E = 256) through the ring dispatch (row-major
    scales) and the whole-tile dispatch (swizzled, num_slots = T), from one partition to 32 and
    up to top-16: every receive row, scale, id and weight against the oracle."""
    w = make_case(2048, 7168, 256, K, seed=P * 31 + K, quant="nvfp4b16", invalid_rate=0.03)
    run_partitioned_dispatch(w, P, w.T, layout)


@pytest.mark.parametrize("T", [200, 1100])
def test_partitioned_nvfp4_row_scales_at_an_odd_address(T):
    """Row-major receive scales may start at any byte: a buffer at an odd address (no 16-byte
    bulk stores possible) gets the same bytes, stored by the threads."""
    m = moe()
    H, E, K, P, S = 1024, 64, 8, 8, T + 8
    w = make_case(T, H, E, K, seed=T + 7, quant="nvfp4b16", invalid_rate=0.05)
    x, ids, wt = to_dev(w)
    rx = filled((P, S, H // 2), torch.uint8)
    n = P * S * (H // 16)
    base = filled((n + 16,), torch.uint8)
    rsf = base[1:1 + n]
    rids = filled((P, S, K), torch.int32)
    rw = filled((P, S, K), torch.float32)
    st = m.new_status()
    m.moe_dispatch_partitioned_ex("nvfp4b16", "row", x, ids, wt, E, P, rx, rsf, rids, rw, st,
                                  input_global_scale=w.global_scale)
    ox, osf, oids, ow = oracle.dispatch_partitioned("nvfp4b16", w.x, w.topk_ids, w.topk_weights, E, P,
                                                    global_scale=w.global_scale, num_slots=S, fill=SENTINEL)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert np.array_equal(bytes_of(rx), np.ascontiguousarray(ox).view(np.uint8).reshape(P, -1))
    got = base.cpu().numpy()
    assert np.array_equal(got[1:1 + n], np.asarray(osf).reshape(-1))
    assert got[0] == SENTINEL and np.all(got[1 + n:] == SENTINEL)
    assert np.array_equal(rids.cpu().numpy(), oids)
    assert np.array_equal(rw.cpu().numpy().view(np.uint32), ow.view(np.uint32))


def test_partition_kernels_on_concurrent_streams():
    """The ring dispatch (row-major scales), the whole-tile dispatch (swizzled scales) and the
    ring combine of three different batches on three streams, their launches interleaved: none
    of them keeps state outside its caller's buffers, so each stream's results match the oracle."""
    m = moe()
    H, E, P = 1024, 64, 8
    specs = [(1500, 8, "row"), (1280, 6, "swizzled"), (2000, 8, "row")]
    runs = []
    for n, (T, K, layout) in enumerate(specs):
        w = make_case(T, H, E, K, seed=300 + n, quant="nvfp4b16", invalid_rate=0.03)
        x, ids, wt = to_dev(w)
        S = T
        rx = filled((P, S, H // 2), torch.uint8)
        rsf = filled((m.swizzled_scale_bytes(P * S, H),) if layout == "swizzled" else (P, S, H // 16), torch.uint8)
        rids = filled((P, S, K), torch.int32)
        rw = filled((P, S, K), torch.float32)
        partial_h = random_bf16(np.random.default_rng(400 + n), (P, S, H))
        partial = torch.from_numpy(partial_h.view(np.int16)).cuda().view(torch.bfloat16)
        out = filled((T, H), torch.bfloat16)
        runs.append((w, layout, torch.cuda.Stream(), x, ids, wt, rx, rsf, rids, rw, partial, partial_h, out,
                     m.new_status()))
    torch.cuda.synchronize()
    for step in range(2):
        for w, layout, s, x, ids, wt, rx, rsf, rids, rw, partial, _, out, st in runs:
            with torch.cuda.stream(s):
                if step == 0:
                    m.moe_dispatch_partitioned_ex("nvfp4b16", layout, x, ids, wt, E, P, rx, rsf, rids, rw, st,
                                                  input_global_scale=w.global_scale)
                else:
                    m.moe_combine_partitioned(partial, ids, E, P, out, st)
    torch.cuda.synchronize()
    for w, layout, s, x, ids, wt, rx, rsf, rids, rw, partial, partial_h, out, st in runs:
        assert int(st.item()) == 0
        S = w.T
        ox, osf, oids, ow = oracle.dispatch_partitioned("nvfp4b16", w.x, w.topk_ids, w.topk_weights, E, P,
                                                        global_scale=w.global_scale, num_slots=S, fill=SENTINEL)
        assert np.array_equal(bytes_of(rx), np.ascontiguousarray(ox).view(np.uint8).reshape(P, -1))
        if layout == "swizzled":
            want = swizzled_scales_expected(osf.reshape(P * S, H // 16), partitioned_routed(w.topk_ids, E, P, S),
                                            partitioned_touched_rows(P, S, w.T))
            assert np.array_equal(rsf.cpu().numpy(), want)
        else:
            assert np.array_equal(bytes_of(rsf), osf.reshape(P, -1))
        assert np.array_equal(rids.cpu().numpy(), oids)
        assert np.array_equal(rw.cpu().numpy().view(np.uint32), ow.view(np.uint32))
        want = oracle.combine_partitioned(partial_h, w.topk_ids, E, P)
        check_combine(bytes_of(out).view(np.uint16).reshape(w.T, H), want)
