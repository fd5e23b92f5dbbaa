"""bench.py end to end on the tiny workload: one JSON line with the keys and value types the
benchmark contract asks for (run as a subprocess, as the driver runs it)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                         cwd=ROOT, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]
    return json.loads(lines[0])


def test_bench_line_has_the_contract_keys():
    d = _run("--workload", "tiny", "--per-config", "none", "--steps", "4", "--warmup", "3", "--no-cpu-baseline")
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 4 and d["warmup"] == 3 and d["higher_is_better"] is True
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["unit"] == "tokens/s"
    assert d["config"]["workload"] == "tiny"
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and 0 < r["frac"] and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] == 64 * 256 * 2
    assert d["gpu_launches"] == 4 * 2                 # fused route+dispatch, then combine
    assert set(d["graph_replay"]) >= {"cold_l2", "warm_l2"}


def test_graph_mode_line():
    """--graph: the timed steps are replays of one captured step; the line says so and keeps the
    contract keys."""
    d = _run("--workload", "tiny", "--per-config", "none", "--steps", "4", "--warmup", "3", "--no-cpu-baseline",
             "--no-e2e", "--graph")
    assert d["timing"].startswith("CUDA graph of one step")
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["roofline"]["frac"] > 0


def test_per_config_entries():
    """--per-config: each listed workload gets an entry measured in the same run, with its own
    config (the one the reference arm prints for it), step time, roofline and e2e."""
    import bench
    from workloads import make_workload
    d = _run("--workload", "tiny", "--per-config", "decode", "--steps", "3", "--warmup", "3", "--no-cpu-baseline")
    assert set(d["per_config"]) == {"decode"}
    p = d["per_config"]["decode"]
    assert p["config"] == bench.config_of(make_workload("decode"))
    assert p["value"] > 0 and p["ms_per_step"] > 0 and p["unit"] == "tokens/s"
    r = p["roofline"]
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    assert abs(r["frac_vs_8tbs"] - r["achieved"] / 8000.0) < 1e-9
    assert abs(p["frac_step"] - p["achieved_gbs_step"] / r["peak"]) < 1e-9
    assert p["e2e"]["value"] > 0 and p["e2e"]["h2d_bytes_per_step"] > 0
    assert d["config"] == bench.config_of(make_workload("tiny"))
    assert d["clocks"]["samples"] >= 1


def test_next_rows_lines():
    """bench.py --next-rows: one well-formed line per NEXT-row call (f1-f4), each a positive time
    and a fraction equal to GB/s over the peak."""
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--next-rows", "--steps", "3",
                          "--warmup", "3"], capture_output=True, text=True, cwd=ROOT, timeout=900)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [json.loads(l) for l in out.stdout.splitlines() if l.strip().startswith("{")]
    assert {d["row"] for d in lines} == {"f1", "f2", "f3", "f4", "f3+f4"}
    for d in lines:
        assert d["us"] > 0 and d["algorithmic_bytes"] > 0 and d["peak"] > 0
        assert abs(d["gbs"] - d["algorithmic_bytes"] / d["us"] / 1e3) < 1e-6 * d["gbs"]
        assert abs(d["frac"] - d["gbs"] / d["peak"]) < 1e-9
        assert d["kernels"] and d["launches_per_call"] >= 1
