"""moe_route_meta_noalloc: the metadata entry point for callers that cannot allocate.

Some callers cannot hand the library a workspace -- an engine whose memory pool already
owns the GPU's memory, or a plugin interface that passes only inputs and outputs -- so
moe_route_meta_noalloc takes its scratch from a fixed array inside the library. These
tests call it through the C ABI and require outputs identical to moe_route_meta and to
the CPU oracle (the metadata is integer work, compared bit for bit): on two calls in a
row, on calls that alternate between routings of different block counts (so each call
starts from the table another call left behind), and at the largest size the array
holds. This file is collected last and also passes when run alone in a fresh process.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 1 << 20


def _outputs(T, K, E, P):
    dev = "cuda"
    return dict(seg_indptr=torch.full((E + 1,), -7, dtype=torch.int64, device=dev),
                src2dst=torch.full((T * K,), -7, dtype=torch.int32, device=dev),
                reorder_topk_ids=torch.full((max(T * K, 1),), -7, dtype=torch.int32, device=dev),
                masked_m=torch.full((E,), -7, dtype=torch.int32, device=dev),
                partition_counts=torch.full((P,), -7, dtype=torch.int32, device=dev))


def _host(o, n_valid):
    return (o["seg_indptr"].cpu().numpy(), o["src2dst"].cpu().numpy(),
            o["reorder_topk_ids"][:n_valid].cpu().numpy(), o["masked_m"].cpu().numpy(),
            o["partition_counts"].cpu().numpy())


def _oracle(ids_host, E, P, M):
    om = oracle.route_meta(ids_host, E, P=P, M=M)
    return om, (om.seg_indptr, om.src2dst, om.reorder_topk_ids, om.masked_m, om.partition_counts)


def _noalloc(moe, ids, E, P, M):
    T, K = ids.shape
    got = _outputs(T, K, E, P)
    st = moe.new_status()
    em = moe.moe_route_meta_noalloc(ids, E, got["seg_indptr"], got["src2dst"], got["reorder_topk_ids"],
                                    got["masked_m"], st, P, M, got["partition_counts"])
    return got, st, em


def _assert_same(got, want, n_valid):
    names = ("seg_indptr", "src2dst", "reorder_topk_ids", "masked_m", "partition_counts")
    for name, a, b in zip(names, _host(got, n_valid), want):
        assert np.array_equal(a, b), name


@pytest.mark.parametrize("T,K,E,P,M,routing", [
    (128, 8, 256, 8, 128, "softmax"),     # one block: no scratch needed
    (4096, 8, 256, 8, 0, "zipf"),         # 32 blocks
    (16384, 8, 128, 8, 16384, "uniform"), # 128 blocks
    (3000, 8, 8, 2, 0, "uniform"),        # several blocks, fewer experts than a warp
])
def test_noalloc_matches_route_meta_and_oracle_twice(T, K, E, P, M, routing):
    import combine_moe_route_meta_gb300 as moe
    from workloads import make_case

    w = make_case(T, 16, E, K, seed=T + E, routing=routing, invalid_rate=0.05)
    ids = torch.from_numpy(w.topk_ids).cuda()

    ref = _outputs(T, K, E, P)
    st_ref = moe.new_status()
    em_ref = moe.moe_route_meta(ids, E, ref["seg_indptr"], ref["src2dst"], ref["reorder_topk_ids"],
                                ref["masked_m"], st_ref, moe.new_workspace(T, K, E), P, M,
                                ref["partition_counts"])
    torch.cuda.synchronize()
    om, want = _oracle(w.topk_ids, E, P, M)
    _assert_same(ref, want, om.num_valid)
    assert em_ref == om.expected_m

    for _ in range(2):
        got, st, em = _noalloc(moe, ids, E, P, M)
        torch.cuda.synchronize()
        assert em == em_ref
        _assert_same(got, want, om.num_valid)
        assert int(st.item()) == int(st_ref.item())


def test_noalloc_alternating_routings_each_match_the_oracle():
    """Two routings with different block counts and expert counts, called A, B, A, B: the
    table each call reads was last written by the other routing."""
    import combine_moe_route_meta_gb300 as moe
    from workloads import make_case

    cases = []
    for T, K, E, P, routing in ((4096, 8, 256, 8, "zipf"), (9000, 3, 64, 4, "replace")):
        w = make_case(T, 16, E, K, seed=31 + T, routing=routing, invalid_rate=0.03)
        om, want = _oracle(w.topk_ids, E, P, 0)
        cases.append((torch.from_numpy(w.topk_ids).cuda(), E, P, om, want))
    blocks = [moe.moe_route_meta_workspace_size(c[0].shape[0], c[0].shape[1], c[1]) // (4 * c[1]) for c in cases]
    assert blocks[0] != blocks[1] and min(blocks) > 1
    for rep in range(4):
        ids, E, P, om, want = cases[rep % 2]
        got, st, em = _noalloc(moe, ids, E, P, 0)
        torch.cuda.synchronize()
        _assert_same(got, want, om.num_valid)
        assert em == om.expected_m
        assert int(st.item()) == 0


def test_noalloc_at_its_capacity_and_one_pair_beyond():
    """E = 1024, K = 1: 4,194,304 pairs fill the 1 MiB table exactly (256 blocks x 1024
    experts x 4 bytes) and match the oracle; one pair more is rejected before any launch."""
    import combine_moe_route_meta_gb300 as moe

    E, K, P = 1024, 1, 8
    T = 4194304
    assert moe.moe_route_meta_workspace_size(T, K, E) == SCRATCH_BYTES
    assert moe.moe_route_meta_workspace_size(T + 1, K, E) > SCRATCH_BYTES
    rng = np.random.default_rng(2024)
    ids_host = rng.integers(-1, E, size=(T, K), dtype=np.int32)
    ids = torch.from_numpy(ids_host).cuda()
    got, st, em = _noalloc(moe, ids, E, P, 0)
    om, want = _oracle(ids_host, E, P, 0)
    torch.cuda.synchronize()
    _assert_same(got, want, om.num_valid)
    assert em == om.expected_m and int(st.item()) == 0

    ids1 = torch.zeros((T + 1, K), dtype=torch.int32, device="cuda")
    o = _outputs(T + 1, K, E, P)
    st = moe.new_status()
    with pytest.raises(moe.MoEError) as e:
        moe.moe_route_meta_noalloc(ids1, E, o["seg_indptr"], o["src2dst"], o["reorder_topk_ids"],
                                   o["masked_m"], st, P, 0, o["partition_counts"])
    assert e.value.status == moe.MOE_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert int(o["seg_indptr"][0].item()) == -7     # nothing was launched


def test_noalloc_rejects_bad_arguments_before_any_launch():
    """A call with E % P != 0 returns MOE_ERR_INVALID_ARG and leaves every output as it was."""
    import combine_moe_route_meta_gb300 as moe

    T, K, E = 4096, 8, 256
    ids = torch.zeros((T, K), dtype=torch.int32, device="cuda")
    o = _outputs(T, K, E, 3)
    st = moe.new_status()
    with pytest.raises(moe.MoEError) as e:
        moe.moe_route_meta_noalloc(ids, E, o["seg_indptr"], o["src2dst"], o["reorder_topk_ids"],
                                   o["masked_m"], st, 3, 0, o["partition_counts"])
    assert e.value.status == moe.MOE_ERR_INVALID_ARG
    torch.cuda.synchronize()
    for name, t in o.items():
        assert bool((t == -7).all()), name
    assert int(st.item()) == 0
