"""moe_route_meta_noalloc: the metadata entry point for callers that cannot allocate.

Some callers cannot hand the library a workspace -- an engine whose memory pool already
owns the GPU's memory, or a plugin interface that passes only inputs and outputs -- so
moe_route_meta_noalloc takes its scratch from a fixed array inside the library. These
tests call it through the C ABI and require outputs identical to moe_route_meta (the
metadata is integer work, compared bit for bit) on two calls in a row, the second of
which starts from the scratch the first one left behind. This file is collected last
and also passes when run alone in a fresh process.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


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


@pytest.mark.parametrize("T,K,E,P,M,routing", [
    (128, 8, 256, 8, 128, "softmax"),     # one block: no scratch needed
    (4096, 8, 256, 8, 0, "zipf"),         # 32 blocks
    (16384, 8, 128, 8, 16384, "uniform"), # 128 blocks
    (3000, 8, 8, 2, 0, "uniform"),        # several blocks, fewer experts than a warp
])
def test_noalloc_matches_route_meta_twice(T, K, E, P, M, routing):
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
    n_valid = int(ref["seg_indptr"][-1].item())
    want = _host(ref, n_valid)

    for _ in range(2):
        got = _outputs(T, K, E, P)
        st = moe.new_status()
        em = moe.moe_route_meta_noalloc(ids, E, got["seg_indptr"], got["src2dst"], got["reorder_topk_ids"],
                                        got["masked_m"], st, P, M, got["partition_counts"])
        torch.cuda.synchronize()
        assert em == em_ref
        for a, b in zip(_host(got, n_valid), want):
            assert np.array_equal(a, b)
        assert int(st.item()) == int(st_ref.item())


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import combine_moe_route_meta_gb300 as moe

    T, K, E = 600000, 8, 1024          # needs a 1.2 MB table: over the 1 MiB scratch
    assert moe.moe_route_meta_workspace_size(T, K, E) > (1 << 20)
    ids = torch.zeros((T, K), dtype=torch.int32, device="cuda")
    o = _outputs(T, K, E, 1)
    st = moe.new_status()
    with pytest.raises(moe.MoEError) as e:
        moe.moe_route_meta_noalloc(ids, E, o["seg_indptr"], o["src2dst"], o["reorder_topk_ids"],
                                   o["masked_m"], st)
    assert e.value.status == moe.MOE_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert int(o["seg_indptr"][0].item()) == -7     # nothing was launched
