"""Randomised GPU parity: seeded random shapes, modes, quantisations, routing skew,
invalid/out-of-range slots and duplicate experts, each run through route_meta, dispatch
and combine (and the fused route_dispatch) and compared with the oracle in full."""
import numpy as np
import pytest
import torch

import oracle
from workloads import make_case

from _harness import SENTINEL, bytes_of, check_meta, filled, moe, run_full, to_dev

pytestmark = pytest.mark.gpu

QUANTS = ["none", "fp8g128", "nvfp4b16", "fp8g128_ue8m0"]


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


@pytest.mark.parametrize("seed", range(24))
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
