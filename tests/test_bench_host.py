"""CPU checks of the benchmark's host logic and of the seeded workloads."""
import os

import numpy as np
import pytest

import bench
from workloads import bf16_bits_to_f32, make_workload


def test_row_bytes():
    assert bench.row_bytes("none", 7168) == 14336
    assert bench.row_bytes("fp8g128", 7168) == 7168 + 224
    assert bench.row_bytes("nvfp4b16", 7168) == 3584 + 448


def test_decode_byte_model_totals():
    """decode: every pair valid and inside capacity -> N = T*K rows of H + 4H/128 bytes."""
    w = make_workload("decode")
    algo = bench.algorithmic_bytes(w, n_valid=1024, n_rows=1024)
    assert algo["dispatch"] == 2 * 128 * 7168 + 8 * 1024 + 8 * 256 + 1024 * 7392
    assert algo["combine"] == 1024 * 14336 + 12 * 1024 + 8 * 256 + 2 * 128 * 7168
    assert sum(algo.values()) == 25959464


def test_profiled_traffic_requires_matching_source(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    os.makedirs(tmp_path / "profiles")
    os.makedirs(tmp_path / "combine_moe_route_meta_gb300" / "csrc")
    src = tmp_path / "combine_moe_route_meta_gb300" / "csrc" / "combine.cu"
    src.write_text("kernel v1")
    digest = bench.source_digest("combine")
    (tmp_path / "profiles" / "combine_decode.md").write_text(
        f"# x\n- source_sha256: {digest}\n- dram_bytes_per_launch: 1234\n")
    assert bench.profiled_traffic("combine", "decode") == 1234
    src.write_text("kernel v2")                       # the kernel changed since the capture
    assert bench.profiled_traffic("combine", "decode") is None
    assert bench.profiled_traffic("combine", "prefill") is None


def test_job_throughput_and_single_rank_max():
    assert bench.max_over_ranks(3.5, None) == 3.5
    assert bench.job_throughput(128, 1, 0.02) == pytest.approx(128 / 20e-6)


@pytest.mark.parametrize("name,T,H,E,K", [("tiny", 64, 256, 8, 2), ("decode", 128, 7168, 256, 8)])
def test_workloads_are_deterministic_and_shaped(name, T, H, E, K):
    a, b = make_workload(name), make_workload(name)
    assert a.x.shape == (T, H) and a.topk_ids.shape == (T, K) and a.topk_weights.shape == (T, K)
    assert np.array_equal(a.x, b.x) and np.array_equal(a.topk_ids, b.topk_ids)
    assert np.allclose(a.topk_weights.sum(axis=1), 1.0, atol=1e-6)
    assert ((a.topk_ids >= 0) & (a.topk_ids < E)).all()
    assert all(len(set(r)) == K for r in a.topk_ids.tolist())            # distinct experts per token
    assert not np.array_equal(make_workload(name, seed=1).x, a.x)


def test_nvfp4_global_scale_is_448x6_over_amax():
    w = make_workload("nvfp4")
    amax = float(np.abs(bf16_bits_to_f32(w.x)).max())
    assert w.global_scale == float(np.float32(2688.0) / np.float32(amax))
    assert w.M == 8192 and w.mode == "masked" and w.quant == "nvfp4b16"
