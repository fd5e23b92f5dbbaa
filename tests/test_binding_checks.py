"""The Python binding rejects, before any launch, buffers that the kernels would access past
their end or with the wrong element type (the C ABI only sees raw pointers). CPU only: the
checks run before the binding asks for device tensors."""
import pytest
import torch

import combine_moe_route_meta_gb300 as moe

T, H, K, E, M = 16, 256, 2, 8, 8


def _meta():
    return dict(seg_indptr=torch.zeros(E + 1, dtype=torch.int64), src2dst=torch.zeros(T * K, dtype=torch.int32),
                reorder_topk_ids=torch.zeros(T * K, dtype=torch.int32), masked_m=torch.zeros(E, dtype=torch.int32),
                dev_status=torch.zeros(1, dtype=torch.int32))


def test_route_meta_checks_sizes_and_dtypes():
    ids = torch.zeros((T, K), dtype=torch.int32)
    b = _meta()
    b["seg_indptr"] = torch.zeros(E + 1, dtype=torch.int32)
    with pytest.raises(ValueError, match="seg_indptr"):
        moe.moe_route_meta(ids, E, **b)
    b = _meta()
    b["src2dst"] = torch.zeros(T * K - 1, dtype=torch.int32)
    with pytest.raises(ValueError, match="src2dst"):
        moe.moe_route_meta(ids, E, **b)
    with pytest.raises(ValueError, match="topk_ids"):
        moe.moe_route_meta(ids.to(torch.int64), E, **_meta())
    b = _meta()
    with pytest.raises(ValueError, match="partition_counts"):
        moe.moe_route_meta(ids, E, num_partitions=4, partition_counts=torch.zeros(3, dtype=torch.int32), **b)


def test_dispatch_checks_output_sizes():
    x = torch.zeros((T, H), dtype=torch.bfloat16)
    ids = torch.zeros((T, K), dtype=torch.int32)
    s2d = torch.zeros(T * K, dtype=torch.int32)
    seg = torch.zeros(E + 1, dtype=torch.int64)
    st = torch.zeros(1, dtype=torch.int32)
    q = torch.zeros((E, M, H), dtype=torch.uint8)
    sc = torch.zeros((E, M, H // 128), dtype=torch.float32)
    with pytest.raises(ValueError, match="out_q"):
        moe.moe_dispatch("masked", "fp8g128", x, ids, E, s2d, seg, q[:-1], sc, st, M)
    with pytest.raises(ValueError, match="out_scales"):
        moe.moe_dispatch("masked", "fp8g128", x, ids, E, s2d, seg, q, None, st, M)
    with pytest.raises(ValueError, match="out_scales"):
        moe.moe_dispatch("masked", "fp8g128", x, ids, E, s2d, seg, q, sc[:, :-1], st, M)
    with pytest.raises(ValueError, match="seg_indptr"):
        moe.moe_dispatch("masked", "fp8g128", x, ids, E, s2d, seg[:-1], q, sc, st, M)
    with pytest.raises(ValueError, match="device tensor"):     # right sizes: only the device check is left
        moe.moe_dispatch("masked", "fp8g128", x, ids, E, s2d, seg, q, sc, st, M)


def test_combine_checks_input_and_output_sizes():
    ids = torch.zeros((T, K), dtype=torch.int32)
    w = torch.zeros((T, K), dtype=torch.float32)
    s2d = torch.zeros(T * K, dtype=torch.int32)
    seg = torch.zeros(E + 1, dtype=torch.int64)
    st = torch.zeros(1, dtype=torch.int32)
    out = torch.zeros((T, H), dtype=torch.bfloat16)
    eo_masked = torch.zeros((E * M, H), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="expert_out"):
        moe.moe_combine("masked", eo_masked[:-1], ids, w, E, s2d, seg, out, st, M)
    with pytest.raises(ValueError, match="topk_weights"):
        moe.moe_combine("masked", eo_masked, ids, w.to(torch.float16), E, s2d, seg, out, st, M)
    with pytest.raises(ValueError, match="device tensor"):
        moe.moe_combine("masked", eo_masked, ids, w, E, s2d, seg, out, st, M)
    # the contiguous layout reads N = seg_indptr[E] rows, which only the device knows: a
    # compact buffer of fewer than T*K rows is legal and passes to the device check
    with pytest.raises(ValueError, match="device tensor"):
        moe.moe_combine("normal", torch.zeros((T * K - 3, H), dtype=torch.bfloat16), ids, w, E, s2d, seg, out, st)
    with pytest.raises(ValueError, match="expert_out"):
        moe.moe_combine_ex("normal", torch.zeros((T * K - 3, H), dtype=torch.bfloat16), ids, w, E, s2d, seg, out,
                           st, expert_out_rows=T * K)


def test_ex_and_partitioned_wrappers_check_sizes():
    x = torch.zeros((T, H), dtype=torch.bfloat16)
    ids = torch.zeros((T, K), dtype=torch.int32)
    w = torch.zeros((T, K), dtype=torch.float32)
    s2d = torch.zeros(T * K, dtype=torch.int32)
    seg = torch.zeros(E + 1, dtype=torch.int64)
    st = torch.zeros(1, dtype=torch.int32)
    cap = T * K + 5
    q = torch.zeros((cap, H), dtype=torch.uint8)
    G, R4 = H // 128, (cap + 3) // 4 * 4
    col = torch.zeros((G, R4), dtype=torch.float32)
    with pytest.raises(ValueError, match="out_scales"):        # column-major needs R4 = roundup(out_rows, 4)
        moe.moe_dispatch_ex("normal", "fp8g128", "col", x, ids, E, s2d, seg, q, col[:, :-4], st, out_rows=cap)
    with pytest.raises(ValueError, match="out_q"):
        moe.moe_dispatch_ex("normal", "fp8g128", "col", x, ids, E, s2d, seg, q[:-1], col, st, out_rows=cap)
    sw = torch.zeros(moe.swizzled_scale_bytes(T * K, H) - 1, dtype=torch.uint8)
    with pytest.raises(ValueError, match="out_scales"):
        moe.moe_dispatch_ex("normal", "nvfp4b16", "swizzled", x, ids, E, s2d, seg,
                            torch.zeros((T * K, H // 2), dtype=torch.uint8), sw, st)
    with pytest.raises(ValueError, match="reorder_topk_ids"):  # alignment padding rows need room
        moe.moe_route_meta_ex(ids, E, seg, s2d, torch.zeros(T * K, dtype=torch.int32),
                              torch.zeros(E, dtype=torch.int32), st, expert_alignment=4)
    P, S = 2, T
    rx = torch.zeros((P, S, H // 2), dtype=torch.uint8)
    rsf = torch.zeros((P, S, H // 16), dtype=torch.uint8)
    rids = torch.zeros((P, S, K), dtype=torch.int32)
    rw = torch.zeros((P, S, K), dtype=torch.float32)
    with pytest.raises(ValueError, match="recv_scales"):       # swizzled: rows padded to 128
        moe.moe_dispatch_partitioned_ex("nvfp4b16", "swizzled", x, ids, w, E, P, rx, rsf, rids, rw, st)
    with pytest.raises(ValueError, match="recv_x"):
        moe.moe_dispatch_partitioned("nvfp4b16", x, ids, w, E, P, rx[:1], rsf, rids, rw, st)
    with pytest.raises(ValueError, match="partial"):
        moe.moe_combine_partitioned(torch.zeros((1, S, H), dtype=torch.bfloat16), ids, E, P,
                                    torch.zeros((T, H), dtype=torch.bfloat16), st)
