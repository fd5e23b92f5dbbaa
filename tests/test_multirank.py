"""World-size-2 checks of the benchmark's multi-rank host logic on CPU (gloo).

The N>1 path runs one process per GPU, each on its own seeded batch, with no data-path
collective; only the per-rank step time is max-reduced. These tests run that logic with
two gloo ranks on the host: per-rank seeds give distinct batches, every rank sees the
same max, the whole-job throughput counts all ranks' tokens over the slowest rank, and
the reference arm runs on rank 0 only.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import oracle
    from workloads import make_workload

    w = make_workload("tiny", seed=bench.rank_seed(rank))
    meta = oracle.route_meta(w.topk_ids, w.E)              # a host stand-in for one step
    fake_ms = 1.0 + rank                                    # rank 1 is the slow one
    ms = bench.max_over_ranks(fake_ms, dist)
    value = bench.job_throughput(w.T, world, ms)

    class A:
        steps, warmup = 1, 3
    ref = bench.run_reference(A, w, rank, world)
    np.savez(os.path.join(out_dir, f"r{rank}.npz"), ids=w.topk_ids, ms=ms, value=value,
             n_valid=meta.num_valid, ref_is_none=ref is None,
             ref_value=(ref or {}).get("value", -1.0))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    r0 = np.load(tmp_path / "r0.npz")
    r1 = np.load(tmp_path / "r1.npz")
    assert not np.array_equal(r0["ids"], r1["ids"])          # distinct per-rank batches
    assert float(r0["ms"]) == float(r1["ms"]) == 2.0          # max over ranks
    assert float(r0["value"]) == pytest.approx(64 * 2 / 2e-3)
    assert not bool(r0["ref_is_none"]) and float(r0["ref_value"]) > 0
    assert bool(r1["ref_is_none"])                            # reference arm: rank 0 only
