"""Randomised GPU parity: seeded random shapes, modes, quantisations, routing skew,
invalid/out-of-range slots and duplicate experts, each run through route_meta, dispatch
and combine (and the fused route_dispatch) and compared with the oracle in full; the
one-row-per-partition layout; expert-aligned metadata from int32 or int64 ids.

MOE_RANDOM_SEEDS (default 40) sets the number of full-path seeds; the partitioned and the
aligned-metadata tests run a quarter and three quarters as many (at least 10 and 30)."""
import os

import numpy as np
import pytest
import torch

import oracle
from workloads import make_case

from _harness import (SENTINEL, bytes_of, check_meta, filled, moe, partitioned_routed, partitioned_touched_rows,
                      run_full, swizzled_scales_expected, to_dev)

pytestmark = pytest.mark.gpu

QUANTS = ["none", "fp8g128", "nvfp4b16", "fp8g128_ue8m0"]
N_SEEDS = max(1, int(os.environ.get("MOE_RANDOM_SEEDS", "40")))


def _random_case(seed):
    rng = np.random.default_rng(1000 + seed)
    quant = QUANTS[seed % 4]
    mode = "masked" if rng.random() < 0.5 else "normal"
    unit = 128 if quant.startswith("fp8") else 16
    H = int(rng.integers(1, 24)) * unit
    P = int(rng.choice([1, 2, 4, 8]))
    E = P * int(rng.integers(1, 33))
    K = int(rng.integers(1, min(16, E) + 1)) if seed % 3 else int(rng.integers(1, 17))
    T = int(rng.integers(0, 3000)) if seed % 5 else int(rng.integers(0, 40))
    routing = "replace" if K > E or seed % 7 == 0 else ("zipf" if seed % 2 else "uniform")
    M = int(rng.integers(1, max(2, 2 * T * K // max(E, 1) + 2))) if mode == "masked" else 0
    return make_case(T, H, E, K, seed=seed, mode=mode, quant=quant if quant != "fp8g128_ue8m0" else "fp8g128",
                     M=M, P=P, invalid_rate=float(rng.choice([0.0, 0.05, 0.3])),
                     bad_rate=float(rng.choice([0.0, 0.0, 0.01])), routing=routing), quant


@pytest.mark.parametrize("seed", range(N_SEEDS))
def test_random_configurations(seed):
    w, quant = _random_case(seed)
    if quant != "fp8g128_ue8m0":
        run_full(w)
        return
    # UE8M0 through the fused / unfused route_dispatch call, compared row by row
    m = moe()
    x, ids, _ = to_dev(w)
    d = m.MoEDispatcher(w.T, w.H, w.K, w.E, mode=w.mode, quant=quant, num_partitions=w.P,
                        max_tokens_per_expert=w.M)
    qs, qd, ss, sd = m.dispatch_out_shapes(w.mode, quant, w.T, w.H, w.K, w.E, w.M)
    d.out_q = filled(qs, qd)
    d.out_scales = filled(ss, sd)
    if w.T:
        d.route_dispatch(x, ids)
    om = oracle.route_meta(w.topk_ids, w.E, P=w.P, M=w.M)
    torch.cuda.synchronize()
    if w.T == 0:
        return
    meta = m.RouteMeta(d.seg_indptr, d.src2dst, d.reorder_topk_ids, d.masked_m, d.partition_counts, d.expected_m)
    check_meta(w, om, meta, d.status)
    gq = bytes_of(d.out_q).reshape(-1, w.H)
    gs = bytes_of(d.out_scales).reshape(-1, w.H // 128)
    flat = w.topk_ids.reshape(-1)
    written = np.zeros(gq.shape[0], bool)
    for i, dd in enumerate(om.src2dst):
        if dd < 0:
            continue
        r = dd if w.mode == "normal" else flat[i] * w.M + dd - om.seg_indptr[flat[i]]
        if w.mode == "masked" and dd - om.seg_indptr[flat[i]] >= w.M:
            continue
        q, e = oracle.quant_fp8_ue8m0_row(w.x[i // w.K])
        assert np.array_equal(gq[r], q) and np.array_equal(gs[r], e)
        written[r] = True
    assert (gq[~written] == SENTINEL).all()


@pytest.mark.parametrize("seed", range(max(10, N_SEEDS // 4)))
def test_random_partitioned_layouts(seed):
    """The FlashInfer one-row-per-partition layout and its combine on seeded random shapes,
    against the oracle in full (bf16 or NVFP4 payload, row-major or swizzled scales)."""
    rng = np.random.default_rng(5000 + seed)
    quant = "nvfp4b16" if seed % 2 else "none"
    layout = "swizzled" if seed % 4 == 1 else "row"
    P = int(rng.choice([1, 2, 4, 8, 16, 32]))
    E = P * int(rng.integers(1, 9))
    K = int(rng.integers(1, min(16, E) + 1))
    H = int(rng.integers(1, 20)) * 64
    T = int(rng.integers(0, 1500))
    S = T + int(rng.integers(0, 40))
    if seed % 8 == 1:  # swizzled scales with num_slots a multiple of 128 (whole tiles per partition)
        S = (S + 127) // 128 * 128
    w = make_case(T, H, E, K, seed=seed, quant=quant, invalid_rate=float(rng.choice([0.0, 0.1])),
                  routing="uniform" if K <= E else "replace")
    m = moe()
    x, ids, wt = to_dev(w)
    g = w.global_scale or 0.0
    inv = int(rng.choice([-1, E]))
    if quant == "nvfp4b16":
        rx = filled((P, S, H // 2), torch.uint8)
        rsf = filled((m.swizzled_scale_bytes(P * S, H),) if layout == "swizzled" else (P, S, H // 16), torch.uint8)
    else:
        rx = filled((P, S, H), torch.bfloat16)
        rsf = None
    rids = filled((P, S, K), torch.int32)
    rw = filled((P, S, K), torch.float32)
    st = m.new_status()
    if S:
        m.moe_dispatch_partitioned_ex(quant, layout, x, ids, wt, E, P, rx, rsf, rids, rw, st, invalid_expert_id=inv,
                                      input_global_scale=g)
    ox, osf, oids, ow = oracle.dispatch_partitioned(quant, w.x, w.topk_ids, w.topk_weights, E, P, invalid_id=inv,
                                                    global_scale=g, num_slots=S, fill=SENTINEL)
    torch.cuda.synchronize()
    assert np.array_equal(bytes_of(rx).reshape(-1), np.ascontiguousarray(ox).view(np.uint8).reshape(-1))
    if rsf is not None:
        want = (swizzled_scales_expected(osf.reshape(P * S, H // 16), partitioned_routed(w.topk_ids, E, P, S),
                                         partitioned_touched_rows(P, S, T))
                if layout == "swizzled" else osf.reshape(-1))
        assert np.array_equal(rsf.cpu().numpy().reshape(-1), want.reshape(-1))
    assert np.array_equal(rids.cpu().numpy(), oids)
    assert np.array_equal(rw.cpu().numpy().view(np.uint32), ow.view(np.uint32))
    assert int(st.item()) == 0
    if T == 0:
        return
    from workloads import random_bf16
    from _harness import check_combine
    partial_h = random_bf16(np.random.default_rng(seed + 77), (P, S, H))
    partial = torch.from_numpy(partial_h.view(np.int16)).cuda().view(torch.bfloat16)
    out = filled((T, H), torch.bfloat16)
    m.moe_combine_partitioned(partial, ids, E, P, out, st)
    want = oracle.combine_partitioned(partial_h, w.topk_ids, E, P)
    torch.cuda.synchronize()
    check_combine(bytes_of(out).view(np.uint16).reshape(T, H), want)


@pytest.mark.parametrize("seed", range(max(30, 3 * N_SEEDS // 4)))
def test_random_aligned_route_meta(seed):
    """moe_route_meta_ex on seeded random shapes: expert alignment A in {1, 2, 8, 128, 1024},
    int32 or int64 ids (with the int32 copy), partitions, capacity checks, invalid and
    out-of-range ids; every output against the oracle, the padding tail of
    reorder_topk_ids untouched."""
    rng = np.random.default_rng(9000 + seed)
    m = moe()
    P = int(rng.choice([1, 2, 4, 8]))
    E = min(P * int(rng.integers(1, 129)), 1024)
    K = int(rng.integers(1, min(16, E) + 1))
    T = int(rng.integers(0, 6000)) if seed % 3 else int(rng.integers(0, 300))
    A = int(rng.choice([1, 2, 8, 128, 1024]))
    M = int(rng.integers(0, max(2, 2 * T * K // E + 2)))
    w = make_case(T, 16, E, K, seed=seed, routing="zipf" if seed % 2 else "uniform",
                  invalid_rate=float(rng.choice([0.0, 0.05])), bad_rate=float(rng.choice([0.0, 0.01])))
    use64 = seed % 2 == 0
    ids = torch.from_numpy(np.ascontiguousarray(w.topk_ids.astype(np.int64) if use64 else w.topk_ids)).cuda()
    cap = T * K + E * (A - 1)
    seg = filled((E + 1,), torch.int64)
    s2d = filled((T * K,), torch.int32)
    reo = filled((cap,), torch.int32)
    mm = filled((E,), torch.int32)
    pc = filled((P,), torch.int32)
    i32 = filled((T, K), torch.int32) if use64 else None
    st = m.new_status()
    em = m.moe_route_meta_ex(ids, E, seg, s2d, reo, mm, st, m.new_workspace(T, K, E), P, M, A, pc,
                             topk_ids_i32_out=i32)
    om = oracle.route_meta_aligned(w.topk_ids, E, A, P=P, M=M)
    torch.cuda.synchronize()
    n = int(om.seg_indptr[-1])
    assert np.array_equal(seg.cpu().numpy(), om.seg_indptr)
    assert np.array_equal(s2d.cpu().numpy(), om.src2dst)
    assert np.array_equal(reo[:n].cpu().numpy(), om.reorder_topk_ids)
    assert (bytes_of(reo[n:]) == SENTINEL).all()
    assert np.array_equal(mm.cpu().numpy(), om.masked_m)
    assert np.array_equal(pc.cpu().numpy(), om.partition_counts)
    assert em == om.expected_m
    if use64:
        assert np.array_equal(i32.cpu().numpy(), w.topk_ids)
    # first error wins on the GPU: with both a bad id and an overflow either code may land
    assert (int(st.item()) == 0) == (om.status == 0)
