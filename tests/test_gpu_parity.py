"""GPU parity: the CUDA library (through the C ABI) against the CPU oracle.

Small and medium cases are compared in full (every metadata entry, every output byte
including the rows the kernels must leave untouched, every combined element); the
full-size workloads run in the benchmark's launch configuration and are compared in full
too: every metadata entry, every written row and scale row, the sentinel left in every row
no pair maps to, and every combined element.
"""
import numpy as np
import pytest
import torch

import oracle
from workloads import bf16_bits_to_f32, f32_to_bf16_bits, make_case, make_workload, random_bf16

from _harness import (bytes_of, check_combine, gpu_meta, moe, run_full, run_full_large, to_dev)

pytestmark = pytest.mark.gpu


# --- the named workloads ---------------------------------------------------------

def test_tiny_workload_with_scaled_experts():
    """tiny: normal / none; expert e returns x * (e+1)/8 (computed on the host, shared)."""
    m = moe()
    w = make_workload("tiny")
    x, ids, wt = to_dev(w)
    om = oracle.route_meta(w.topk_ids, w.E)
    gm, st = gpu_meta(w, ids)
    d = m.dispatch(x, ids, wt, gm, w.E, mode="normal", quant="none", dev_status=st)
    oq, _ = oracle.dispatch("normal", "none", w.x, w.topk_ids, om, w.E)
    torch.cuda.synchronize()
    n = om.num_valid
    assert np.array_equal(bytes_of(d.hidden_states)[:n], oq[:n].view(np.uint8))
    rows = bf16_bits_to_f32(oq[:n]).astype(np.float32)
    scale = ((om.reorder_topk_ids + 1) / 8).astype(np.float32)
    eo_host = f32_to_bf16_bits(rows * scale[:, None])
    eo = torch.from_numpy(eo_host.view(np.int16)).cuda().view(torch.bfloat16)
    y = m.combine(eo, ids, wt, gm, w.E, dev_status=st)
    want = oracle.combine("normal", eo_host, w.topk_ids, w.topk_weights, om, w.E)
    torch.cuda.synchronize()
    check_combine(bytes_of(y).view(np.uint16).reshape(w.T, w.H), want)
    assert int(st.item()) == 0


def test_decode_workload_full():
    """decode (T=128, H=7168, E=256, top-8, masked M=128, FP8 g128): full comparison."""
    run_full(make_workload("decode"))


@pytest.mark.parametrize("name", ["prefill", "qwen3", "nvfp4"])
def test_full_size_workloads_in_full(name):
    """prefill (normal FP8, Zipf routing, H=7168), qwen3 (normal bf16, 5 % empty slots) and nvfp4
    (masked NVFP4, M=8192): every byte and every combined element against the oracle."""
    run_full_large(make_workload(name))


def test_qwen3_masked_secondary():
    """qwen3 routing in the masked layout with M = T (no capacity drops), compared in full."""
    w = make_workload("qwen3")
    w.mode, w.M = "masked", w.T
    run_full_large(w)


# --- shapes: ragged slices, several blocks, limits ------------------------------

@pytest.mark.parametrize("T,H,E,K,mode,quant,M", [
    (1, 16, 1, 1, "normal", "none", 0),
    (3, 48, 3, 2, "masked", "none", 4),
    (37, 272, 5, 3, "normal", "none", 0),          # ragged 512-slice (17 active lanes)
    (50, 640, 12, 4, "normal", "fp8g128", 0),      # one full + one ragged slice
    (50, 384, 12, 4, "masked", "fp8g128", 40),
    (61, 1040, 16, 6, "normal", "nvfp4b16", 0),    # 1040 = 2*512 + 16
    (61, 208, 16, 6, "masked", "nvfp4b16", 61),
    (300, 4096, 128, 8, "normal", "none", 0),
    (200, 7168, 256, 8, "normal", "fp8g128", 0),
    (200, 7168, 256, 8, "masked", "nvfp4b16", 64),
    (2500, 256, 37, 8, "normal", "fp8g128", 0),    # 20000 pairs: several route blocks, E not 2^k
    (3000, 128, 8, 8, "masked", "none", 3000),     # several route blocks with E < 32
    (1200, 128, 1024, 16, "normal", "none", 0),    # E and K at their limits, several blocks
    (40, 128, 1024, 16, "masked", "fp8g128", 8),   # E = 1024 in one block
    # >= 1024 tokens with 16-byte row geometry: the bulk (TMA) dispatch path
    (1500, 1024, 64, 8, "normal", "fp8g128", 0),
    (1100, 2048, 32, 6, "masked", "nvfp4b16", 400),
    (1030, 512, 16, 4, "masked", "none", 500),
    (2048, 4096, 128, 8, "normal", "none", 0),
    # other models' hidden sizes: 16384 (32 slices, so warps loop), 5120, 2880 (ragged slice)
    (96, 16384, 64, 4, "normal", "fp8g128", 0),
    (1100, 16384, 64, 4, "masked", "nvfp4b16", 200),
    (300, 5120, 160, 6, "normal", "fp8g128", 0),
    (1024, 5120, 160, 6, "masked", "fp8g128", 64),
    (200, 2880, 32, 4, "normal", "none", 0),
    (1100, 2880, 32, 4, "masked", "nvfp4b16", 300),
    # >= 1024 tokens whose rows do not fit the bulk ring's shared memory: the register path
    (1030, 32768, 16, 2, "normal", "none", 0),
    (1030, 32768, 16, 2, "masked", "fp8g128", 200),
    # many short rows: each bulk CTA cycles its ring (and its mbarrier phases) 100+ times
    (200000, 128, 16, 2, "normal", "none", 0),
    (100000, 512, 16, 2, "masked", "fp8g128", 15000),
    (100000, 256, 16, 2, "normal", "nvfp4b16", 0),
])
def test_shapes_full(T, H, E, K, mode, quant, M):
    w = make_case(T, H, E, K, seed=T + H + E + K, mode=mode, quant=quant, M=M, invalid_rate=0.05)
    run_full(w)


def test_large_route_meta_many_rounds():
    """2^21 pairs: 16 rounds per warp and 128 blocks; metadata compared in full."""
    w = make_case(262144, 16, 256, 8, seed=5, routing="zipf")
    _, ids, _ = to_dev(w)
    om = oracle.route_meta(w.topk_ids, w.E)
    gm, st = gpu_meta(w, ids)
    torch.cuda.synchronize()
    assert np.array_equal(gm.src2dst.cpu().numpy(), om.src2dst)
    assert np.array_equal(gm.seg_indptr.cpu().numpy(), om.seg_indptr)
    assert np.array_equal(gm.reorder_topk_ids[: om.num_valid].cpu().numpy(), om.reorder_topk_ids)


@pytest.mark.parametrize("T,K,E,routing", [
    (400000, 8, 256, "uniform"),  # 196 blocks of 16 rounds (more than one wave)
    (20000, 8, 1024, "zipf"),     # 79 blocks of 2 rounds, E = 1024: the largest shared-memory footprint
    (9000, 1, 7, "uniform"),      # 9 blocks, odd E smaller than a warp
    (256, 8, 256, "zipf"),        # 2048 pairs: the largest one-block case, 2 rounds per warp
    (257, 8, 256, "zipf"),        # one token more: count + place over 3 blocks
    (250, 8, 1024, "uniform"),    # 2000 pairs with E = 1024 in one block
    (1024, 8, 256, "zipf"),       # 8192 pairs: count + place over 8 blocks
])
def test_multi_block_route_meta_paths(T, K, E, routing):
    """Metadata in full across the size classes: one block up to 2048 pairs, then the count
    and place kernels (up to more blocks than fit on the GPU at once); the workspace is
    reused across calls."""
    w = make_case(T, 16, E, K, seed=T + E, routing=routing, invalid_rate=0.03)
    _, ids, _ = to_dev(w)
    om = oracle.route_meta(w.topk_ids, w.E)
    m = moe()
    d = m.MoEDispatcher(w.T, w.H, w.K, w.E)
    for _ in range(2):
        d.route(ids)
        torch.cuda.synchronize()
        assert np.array_equal(d.src2dst.cpu().numpy(), om.src2dst)
        assert np.array_equal(d.seg_indptr.cpu().numpy(), om.seg_indptr)
        assert np.array_equal(d.reorder_topk_ids[: om.num_valid].cpu().numpy(), om.reorder_topk_ids)
        assert np.array_equal(d.masked_m.cpu().numpy(), om.masked_m)
    d.check()


# --- degenerate inputs ---------------------------------------------------------------

def test_empty_batch():
    for mode, quant, M in (("normal", "none", 0), ("masked", "fp8g128", 8), ("masked", "nvfp4b16", 8)):
        w = make_case(0, 256, 16, 4, mode=mode, quant=quant, M=M)
        run_full(w)


def test_all_slots_invalid():
    w = make_case(100, 256, 16, 4, seed=3, invalid_rate=1.0)
    om = run_full(w)
    assert om.num_valid == 0


def test_every_pair_to_one_expert():
    """All pairs hit expert 0: the warp-match groups are the whole warp."""
    w = make_case(20000, 128, 4, 1, seed=4, routing="hot", quant="fp8g128")
    run_full(w)


def test_duplicate_experts_in_a_token():
    w = make_case(500, 256, 6, 8, seed=6, routing="replace", quant="fp8g128")
    run_full(w)


def test_zero_rows_quantise_to_zero_codes():
    for quant in ("fp8g128", "nvfp4b16"):
        w = make_case(64, 512, 8, 2, seed=8, quant=quant, zero_tokens=10)
        run_full(w)


@pytest.mark.parametrize("T,M", [(400, 100), (1600, 300)])  # register / ring (>= 1024 tokens) combine
def test_capacity_overflow_drops_late_pairs_and_reports(T, M):
    w = make_case(T, 256, 4, 2, seed=9, mode="masked", quant="fp8g128", M=M)
    om = run_full(w)
    assert om.status == oracle.CAPACITY
    assert (om.masked_m == M).any()


@pytest.mark.parametrize("T,mode,M", [(300, "normal", 0), (1500, "normal", 0), (1500, "masked", 1500)])
def test_out_of_range_ids_are_skipped_and_reported(T, mode, M):
    w = make_case(T, 256, 16, 4, seed=10, mode=mode, M=M, bad_rate=0.02, invalid_rate=0.02)
    om = run_full(w)
    assert om.status == oracle.BAD_ID


def test_status_word_is_sticky_first_error_wins():
    m = moe()
    w = make_case(64, 256, 8, 2, seed=11, bad_rate=0.1)
    _, ids, _ = to_dev(w)
    st = m.new_status()
    m.route_meta(ids, w.E, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == m.MOE_ERR_BAD_EXPERT_ID
    w2 = make_case(64, 256, 8, 2, seed=12, mode="masked", M=1)
    _, ids2, _ = to_dev(w2)
    m.route_meta(ids2, w2.E, max_tokens_per_expert=1, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == m.MOE_ERR_BAD_EXPERT_ID
    with pytest.raises(m.MoEError):
        m.check_status(st)


def test_host_errors_raise_before_launch():
    m = moe()
    w = make_case(8, 100, 8, 2)
    x = torch.zeros((8, 100), dtype=torch.bfloat16, device="cuda")
    _, ids, _ = to_dev(w)
    gm, st = gpu_meta(w, ids)
    with pytest.raises(m.MoEError) as e:
        m.dispatch(x, ids, None, gm, w.E, quant="fp8g128", dev_status=st)
    assert e.value.status == m.MOE_ERR_INVALID_ARG


def test_repeated_calls_reuse_workspace():
    """The multi-block route workspace is left ready for the next call."""
    m = moe()
    w = make_case(5000, 64, 64, 8, seed=13, routing="zipf")
    _, ids, _ = to_dev(w)
    om = oracle.route_meta(w.topk_ids, w.E)
    d = m.MoEDispatcher(w.T, w.H, w.K, w.E)
    for _ in range(4):
        d.route(ids)
        torch.cuda.synchronize()
        assert np.array_equal(d.src2dst.cpu().numpy(), om.src2dst)
        assert np.array_equal(d.seg_indptr.cpu().numpy(), om.seg_indptr)
    d.check()


@pytest.mark.parametrize("case", ["decode", "normal_4096"])
def test_dispatcher_graph_capture_replays_correctly(case):
    """route + dispatch + combine captured in one CUDA graph and replayed (decode: one-block
    metadata; normal_4096: the count and place metadata kernels and the bulk dispatch)."""
    m = moe()
    if case == "decode":
        w = make_workload("decode")
    else:
        w = make_case(4096, 1024, 256, 8, seed=21, quant="fp8g128", routing="zipf", invalid_rate=0.02)
    x, ids, wt = to_dev(w)
    d = m.MoEDispatcher(w.T, w.H, w.K, w.E, mode=w.mode, quant=w.quant, num_partitions=w.P,
                        max_tokens_per_expert=w.M)
    eo_rows = w.E * w.M if w.mode == "masked" else w.T * w.K
    eo = torch.randn((eo_rows, w.H), dtype=torch.bfloat16, device="cuda")
    d.out_q.zero_()            # slots past masked_m are never written: start both runs from zeros
    d.out.zero_()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        d.route(ids)
        d.dispatch(x, ids)
        d.combine(eo, ids, wt)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    ref_q = d.out_q.clone()
    ref_out = d.out.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        d.route(ids)
        d.dispatch(x, ids)
        d.combine(eo, ids, wt)
    d.out_q.zero_()
    d.out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(d.out_q, ref_q)
    assert torch.equal(d.out, ref_out)
    d.check()


def test_concurrent_streams_keep_their_own_results():
    """Four dispatchers on four streams, their launches interleaved with no ordering between
    the streams (fused small batch, count + place metadata with the bulk FP8 dispatch,
    NVFP4 masked, bf16 register path): every call works only on its caller's buffers, so
    each stream's results match the oracle."""
    import oracle as orc
    m = moe()
    cases = [make_case(96, 1024, 32, 4, seed=61, mode="masked", quant="fp8g128", M=48, invalid_rate=0.05),
             make_case(3000, 1024, 64, 8, seed=62, quant="fp8g128", routing="zipf"),
             make_case(1500, 512, 16, 4, seed=63, mode="masked", quant="nvfp4b16", M=600),
             make_case(700, 768, 24, 3, seed=64)]
    streams = [torch.cuda.Stream() for _ in cases]
    runs = []
    for w, s in zip(cases, streams):
        x, ids, wt = to_dev(w)
        d = m.MoEDispatcher(w.T, w.H, w.K, w.E, mode=w.mode, quant=w.quant, num_partitions=w.P,
                            max_tokens_per_expert=w.M)
        eo_rows = w.E * w.M if w.mode == "masked" else w.T * w.K
        eo_h = random_bf16(np.random.default_rng(w.seed), (eo_rows, w.H))
        eo = torch.from_numpy(eo_h.view(np.int16)).cuda().view(torch.bfloat16)
        runs.append((w, s, d, x, ids, wt, eo, eo_h))
    torch.cuda.synchronize()
    for step in range(3):  # interleave the streams' launches call by call
        for w, s, d, x, ids, wt, eo, _ in runs:
            with torch.cuda.stream(s):
                if step == 0:
                    d.route(ids)
                elif step == 1:
                    d.dispatch(x, ids, w.global_scale or 0.0)
                else:
                    d.combine(eo, ids, wt)
    torch.cuda.synchronize()
    for w, s, d, x, ids, wt, eo, eo_h in runs:
        d.check()
        om = orc.route_meta(w.topk_ids, w.E, P=w.P, M=w.M)
        assert np.array_equal(d.src2dst.cpu().numpy(), om.src2dst)
        oq, osc = orc.dispatch(w.mode, w.quant, w.x, w.topk_ids, om, w.E, M=w.M,
                               global_scale=w.global_scale or 0.0)
        pairs = [(bytes_of(d.out_q), np.ascontiguousarray(oq).view(np.uint8))]
        if osc is not None:
            pairs.append((bytes_of(d.out_scales), np.ascontiguousarray(osc).view(np.uint8)))
        for got, ref in pairs:
            if w.mode == "masked":
                got, ref = got.reshape(w.E, w.M, -1), ref.reshape(w.E, w.M, -1)
                for e in range(w.E):
                    n = int(om.masked_m[e])
                    assert np.array_equal(got[e, :n], ref[e, :n])
            else:
                n = om.num_valid
                got, ref = got.reshape(w.T * w.K, -1), ref.reshape(w.T * w.K, -1)
                assert np.array_equal(got[:n], ref[:n])
        want = orc.combine(w.mode, eo_h, w.topk_ids, w.topk_weights, om, w.E, M=w.M)
        check_combine(d.out.view(torch.int16).cpu().numpy().view(np.uint16), want)


# --- moe_route_dispatch: route + dispatch in one call -------------------------------------

@pytest.mark.parametrize("T,H,E,K,mode,quant,M,P", [
    (64, 16384, 64, 4, "masked", "fp8g128", 64, 4),     # 32 slices per token: warps loop
    (100, 2880, 32, 4, "normal", "nvfp4b16", 0, 2),     # ragged last slice
    (128, 7168, 256, 8, "masked", "fp8g128", 128, 8),   # the decode shape: one fused kernel
    (1, 16, 1, 1, "normal", "none", 0, 1),
    (33, 272, 5, 3, "masked", "none", 9, 5),             # capacity drops inside the fused kernel
    (100, 1040, 64, 6, "normal", "nvfp4b16", 0, 4),
    (256, 4096, 128, 16, "masked", "nvfp4b16", 64, 8),   # 4096 pairs: the largest fused batch
    (512, 256, 64, 2, "normal", "fp8g128", 0, 2),        # 512 tokens: the largest fused batch by tokens
    (1024, 128, 1024, 4, "normal", "fp8g128", 0, 2),     # 1024 tokens (past the fused limit), E at its limit
    (4096, 512, 256, 8, "normal", "fp8g128", 0, 8),      # beyond the fused limits: route kernels + dispatch
    (513, 256, 16, 8, "masked", "none", 600, 4),         # 4104 pairs: just past the fused limit
])
def test_route_dispatch_matches_oracle(T, H, E, K, mode, quant, M, P):
    import oracle as orc
    from _harness import SENTINEL, check_meta, filled
    m = moe()
    w = make_case(T, H, E, K, seed=T * 7 + H, mode=mode, quant=quant, M=M, P=P, invalid_rate=0.05,
                  routing="zipf" if E >= K else "replace")
    x, ids, _ = to_dev(w)
    d = m.MoEDispatcher(T, H, K, E, mode=mode, quant=quant, num_partitions=P, max_tokens_per_expert=M)
    qs, qd, ss, sd = m.dispatch_out_shapes(mode, quant, T, H, K, E, M)
    d.out_q = filled(qs, qd)
    d.out_scales = filled(ss, sd) if ss is not None else None
    d.route_dispatch(x, ids, w.global_scale or 0.0)
    om = orc.route_meta(w.topk_ids, E, P=P, M=M)
    oq, osc = orc.dispatch(mode, quant, w.x, w.topk_ids, om, E, M=M, global_scale=w.global_scale or 0.0,
                           fill=SENTINEL)
    torch.cuda.synchronize()
    meta = m.RouteMeta(d.seg_indptr, d.src2dst, d.reorder_topk_ids, d.masked_m, d.partition_counts, d.expected_m)
    check_meta(w, om, meta, d.status)
    gq = bytes_of(d.out_q)
    assert np.array_equal(gq, np.ascontiguousarray(oq).view(np.uint8).reshape(gq.shape))
    if d.out_scales is not None:
        gs = bytes_of(d.out_scales)
        assert np.array_equal(gs, np.ascontiguousarray(osc).view(np.uint8).reshape(gs.shape))


def test_route_dispatch_bad_ids_reported_once():
    m = moe()
    w = make_case(64, 256, 16, 4, seed=21, bad_rate=0.05)
    x, ids, _ = to_dev(w)
    d = m.MoEDispatcher(64, 256, 4, 16)
    d.route_dispatch(x, ids)
    torch.cuda.synchronize()
    assert int(d.status.item()) == m.MOE_ERR_BAD_EXPERT_ID
    om = oracle.route_meta(w.topk_ids, 16)
    assert np.array_equal(d.src2dst.cpu().numpy(), om.src2dst)
