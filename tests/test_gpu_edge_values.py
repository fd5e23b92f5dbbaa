"""Degenerate values through the quantising dispatch, bit for bit against the oracle: rows
of zeros and negative zeros, magnitudes near the top and the bottom of the bf16 range,
groups where one huge element sends the rest to code zero, constant rows (the maximum
code), and NVFP4 global scales of 0, 1e-30 and 1e30 (every block scale zero, or every
block scale and code saturated). All intermediate values stay finite: the pages do not
say what infinities or NaNs in hidden_states should produce."""
import dataclasses

import numpy as np
import pytest

from workloads import make_case

from _harness import run_full, run_partitioned_dispatch

pytestmark = pytest.mark.gpu


def _bf16(a) -> np.ndarray:
    """float -> bf16 bits by truncation (any bit pattern is a valid input)."""
    return (np.asarray(a, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _with_rows(w, rows):
    x = w.x.copy()
    for i, r in enumerate(rows):
        x[i] = r
    return dataclasses.replace(w, x=x)


def _extreme_rows(H, rng, huge: bool):
    z = np.clip(rng.standard_normal(H), -3.0, 3.0).astype(np.float32)
    rows = [np.zeros(H, np.uint16),                 # +0 everywhere
            np.full(H, 0x8000, np.uint16),          # -0 everywhere
            _bf16(z * np.float32(1e-38)),           # normal and subnormal bf16 near the bottom
            _bf16(np.full(H, 1.0, np.float32)),     # constant: every element the group maximum
            _bf16(np.full(H, -1344.0, np.float32))]
    mixed = _bf16(z * np.float32(1e-30))
    mixed[::16] = _bf16(np.float32(3e3))            # one large element per 16-block
    rows.append(mixed)
    if huge:
        rows.append(_bf16(z * np.float32(1e38)))    # near the top of the range (|x| <= 3e38)
        m2 = _bf16(z * np.float32(1e-20))
        m2[5::128] = _bf16(np.float32(-2e38))       # one huge element per 128-group
        rows.append(m2)
    return rows


@pytest.mark.parametrize("mode,M", [("normal", 0), ("masked", 24)])
@pytest.mark.parametrize("quant", ["fp8g128", "nvfp4b16"])
def test_extreme_magnitudes(quant, mode, M):
    w = make_case(24, 512, 8, 2, seed=91, mode=mode, quant=quant, M=M)
    w = _with_rows(w, _extreme_rows(w.H, np.random.default_rng(92), huge=True))
    if quant == "nvfp4b16":
        w = dataclasses.replace(w, global_scale=1.0)
    run_full(w)


@pytest.mark.parametrize("g", [0.0, 1e-30, 1e30])
@pytest.mark.parametrize("mode,M", [("normal", 0), ("masked", 24)])
def test_nvfp4_degenerate_global_scales(g, mode, M):
    w = make_case(24, 512, 8, 2, seed=93, mode=mode, quant="nvfp4b16", M=M)
    w = _with_rows(w, _extreme_rows(w.H, np.random.default_rng(94), huge=False))
    run_full(dataclasses.replace(w, global_scale=g))


@pytest.mark.parametrize("g", [1.0, 0.0, 1e-30, 1e30])
@pytest.mark.parametrize("layout,T,S", [("swizzled", 24, 128), ("row", 24, 24), ("swizzled", 1100, 1152),
                                        ("row", 1100, 1100)])
def test_partitioned_nvfp4_extreme_values(g, layout, T, S):
    """The same degenerate rows and global scales through the FlashInfer partition layout: the
    kernel that builds whole swizzled tiles (num_slots % 128 == 0) has a quantiser of its own."""
    w = make_case(T, 512, 16, 4, seed=93, quant="nvfp4b16")
    rows = _extreme_rows(w.H, np.random.default_rng(94), huge=True)
    x = w.x.copy()
    for i, r in enumerate(rows):
        x[(i * 137) % T] = r
    w = dataclasses.replace(w, x=x, global_scale=g)
    run_partitioned_dispatch(w, 4, S, layout)
