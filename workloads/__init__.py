"""Seeded synthetic inputs for the MoE dispatch/combine hot path.

This module is the one piece of code that both the CUDA path's tests/benchmark
and the CPU oracle consume. It draws random numbers and shapes them into the
tensors the dispatcher pages pass around (``hidden_states``, ``topk_ids``,
``topk_weights``, ``input_global_scale``); it performs none of the method's own
arithmetic (no histogram, scan, rank, gather, quantisation or combine).

Every array is produced on the host with numpy's PCG64 (``default_rng(seed)``)
and returned as plain numpy arrays:

* ``x``            uint16 [T, H]  -- bf16 bit patterns of ``hidden_states``
* ``topk_ids``     int32  [T, K]  -- expert id per (token, slot), -1 = invalid slot
* ``topk_weights`` float32 [T, K] -- router weights, renormalised over the K slots

The five named workloads follow the shapes, distributions and routing skew of the
dispatcher pages' deployments (DeepSeek-V3-shaped decode and prefill, a
Qwen3-MoE-shaped layer with dropped slots, and the FlashInfer NVFP4 payload).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

__all__ = [
    "Workload",
    "WORKLOADS",
    "make_workload",
    "make_case",
    "random_bf16",
    "f32_to_bf16_bits",
    "bf16_bits_to_f32",
]


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 samples to bf16 (round-to-nearest-even) and return bit patterns.

    Used only to turn freshly drawn float32 random numbers into bf16 inputs; the
    conversion is delegated to torch's CPU cast so that this module carries no
    rounding code of its own.
    """
    import torch

    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (b.astype(np.uint32) << 16).view(np.float32)


def random_bf16(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    """bf16 bit patterns of N(0, std^2) samples."""
    return f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32) * np.float32(std))


def _softmax_rows(z: np.ndarray) -> np.ndarray:
    z = z.astype(np.float64)
    z = z - z.max(axis=1, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=1, keepdims=True)


def _renormalised_weights(logits_at_ids: np.ndarray) -> np.ndarray:
    """softmax over the K chosen logits == softmax over all, restricted and renormalised."""
    return _softmax_rows(logits_at_ids).astype(np.float32)


@dataclass
class Workload:
    name: str
    T: int
    H: int
    E: int
    K: int
    P: int                      # logical expert-parallel partitions (E % P == 0)
    M: int                      # masked capacity per expert (0 = not masked)
    mode: str                   # "normal" | "masked"
    quant: str                  # "none" | "fp8g128" | "nvfp4b16"
    seed: int
    x: np.ndarray               # uint16 [T, H] bf16 bits
    topk_ids: np.ndarray        # int32  [T, K]
    topk_weights: np.ndarray    # float32 [T, K]
    global_scale: Optional[float] = None   # NVFP4 input_global_scale
    recipe: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def pairs(self) -> int:
        return self.T * self.K


# ---------------------------------------------------------------------------
# routing generators
# ---------------------------------------------------------------------------

def _route_topk_softmax(rng, T, E, K):
    """top-K experts by N(0,1) router logit (ties -> lower id), renormalised softmax."""
    logits = rng.standard_normal((T, E), dtype=np.float32)
    order = np.argsort(-logits, axis=1, kind="stable")[:, :K]
    ids = order.astype(np.int32)
    w = _renormalised_weights(np.take_along_axis(logits, order, axis=1))
    return ids, w


def _route_uniform(rng, T, E, K):
    """K distinct experts per token, uniformly at random, in random slot order."""
    keys = rng.random((T, E))
    ids = np.argsort(keys, axis=1, kind="stable")[:, :K].astype(np.int32)
    w = _renormalised_weights(rng.standard_normal((T, K), dtype=np.float32))
    return ids, w


def _route_zipf(rng, T, E, K, s):
    """Expert popularity p_e ~ rank_e^-s (rank = seeded permutation of 1..E);
    K experts per token drawn without replacement from p."""
    rank = rng.permutation(E) + 1
    p = rank.astype(np.float64) ** (-s)
    p /= p.sum()
    ids = np.empty((T, K), dtype=np.int32)
    for t in range(T):
        ids[t] = rng.choice(E, size=K, replace=False, p=p)
    w = _renormalised_weights(rng.standard_normal((T, K), dtype=np.float32))
    return ids, w


def _drop_slots(rng, ids, rate):
    """Set a Bernoulli(rate) subset of (token, slot) entries to the invalid id -1."""
    if rate <= 0:
        return ids
    mask = rng.random(ids.shape) < rate
    out = ids.copy()
    out[mask] = -1
    return out


# ---------------------------------------------------------------------------
# the five named workloads
# ---------------------------------------------------------------------------

def _tiny(seed):
    rng = np.random.default_rng(seed)
    T, H, E, K = 64, 256, 8, 2
    x = random_bf16(rng, (T, H))
    ids, w = _route_topk_softmax(rng, T, E, K)
    return Workload("tiny", T, H, E, K, 1, 0, "normal", "none", seed, x, ids, w,
                    recipe="T=64 H=256 bf16 N(0,1); E=8 top-2 by N(0,1) logit, renormalised "
                           "softmax weights; expert output = input*(e+1)/8")


def _decode(seed):
    rng = np.random.default_rng(seed)
    T, H, E, K = 128, 7168, 256, 8
    x = random_bf16(rng, (T, H))
    ids, w = _route_topk_softmax(rng, T, E, K)
    return Workload("decode", T, H, E, K, 8, 128, "masked", "fp8g128", seed, x, ids, w,
                    recipe="T=128 H=7168 bf16 N(0,1); E=256 top-8 by N(0,1) logit, "
                           "renormalised softmax; 8 partitions x 32 experts; M=128")


def _prefill(seed):
    rng = np.random.default_rng(seed)
    T, H, E, K = 4096, 7168, 256, 8
    x = random_bf16(rng, (T, H))
    ids, w = _route_zipf(rng, T, E, K, 1.2)
    return Workload("prefill", T, H, E, K, 8, 0, "normal", "fp8g128", seed, x, ids, w,
                    recipe="T=4096 H=7168 bf16 N(0,1); E=256, Zipf(s=1.2) expert popularity "
                           "over a seeded rank permutation, 8 per token without replacement")


def _qwen3(seed):
    rng = np.random.default_rng(seed)
    T, H, E, K = 16384, 4096, 128, 8
    x = random_bf16(rng, (T, H))
    ids, w = _route_uniform(rng, T, E, K)
    ids = _drop_slots(rng, ids, 0.05)
    return Workload("qwen3", T, H, E, K, 8, 0, "normal", "none", seed, x, ids, w,
                    recipe="T=16384 H=4096 bf16 N(0,1); E=128, 8 uniform without replacement; "
                           "5% of slots set to -1 (Bernoulli per slot); 8 partitions x 16")


def _nvfp4(seed):
    rng = np.random.default_rng(seed)
    T, H, E, K = 8192, 7168, 256, 8
    # N(0, 2): mean 0, variance 2
    x = random_bf16(rng, (T, H), std=float(np.sqrt(2.0)))
    ids, w = _route_uniform(rng, T, E, K)
    amax = float(np.abs(bf16_bits_to_f32(x)).max())
    g = float(np.float32(2688.0) / np.float32(amax))
    return Workload("nvfp4", T, H, E, K, 8, 8192, "masked", "nvfp4b16", seed, x, ids, w,
                    global_scale=g,
                    recipe="T=8192 H=7168 bf16 N(0,2) (variance 2); E=256, 8 uniform without "
                           "replacement; input_global_scale = 448*6/amax(x); M=8192, 8 partitions")


WORKLOADS = {
    "tiny": _tiny,
    "decode": _decode,
    "prefill": _prefill,
    "qwen3": _qwen3,
    "nvfp4": _nvfp4,
}


def make_workload(name: str, seed: int = 0) -> Workload:
    return WORKLOADS[name](seed)


def make_case(T: int, H: int, E: int, K: int, *, seed: int = 0, mode: str = "normal",
              quant: str = "none", M: int = 0, P: int = 1, invalid_rate: float = 0.0,
              bad_rate: float = 0.0, routing: str = "uniform", zipf_s: float = 1.2,
              std: float = 1.0, global_scale: Optional[float] = None,
              zero_tokens: int = 0) -> Workload:
    """A seeded case of arbitrary shape for parity and property tests.

    routing: "uniform" (distinct experts), "zipf" (skewed, distinct), "softmax"
    (top-K by logit), "hot" (every slot of every token -> expert 0 when K == 1,
    otherwise K distinct lowest ids), or "replace" (independent draws, duplicates allowed).
    bad_rate sets that fraction of slots to out-of-range ids (E, E+7 or -3).
    zero_tokens: the first `zero_tokens` rows of x are all zero.
    """
    rng = np.random.default_rng(seed)
    x = random_bf16(rng, (T, H), std=std) if T * H else np.zeros((T, H), np.uint16)
    if zero_tokens:
        x[:zero_tokens] = 0
    if T == 0:
        ids = np.zeros((0, K), np.int32)
        w = np.zeros((0, K), np.float32)
    elif routing == "uniform":
        ids, w = _route_uniform(rng, T, E, K)
    elif routing == "zipf":
        ids, w = _route_zipf(rng, T, E, K, zipf_s)
    elif routing == "softmax":
        ids, w = _route_topk_softmax(rng, T, E, K)
    elif routing == "hot":
        ids = np.tile(np.arange(K, dtype=np.int32), (T, 1))
        w = _renormalised_weights(rng.standard_normal((T, K), dtype=np.float32))
    elif routing == "replace":
        ids = rng.integers(0, E, size=(T, K), dtype=np.int32)
        w = _renormalised_weights(rng.standard_normal((T, K), dtype=np.float32))
    else:
        raise ValueError(routing)
    if T:
        ids = _drop_slots(rng, ids, invalid_rate)
        if bad_rate > 0:
            bad = rng.random(ids.shape) < bad_rate
            choices = np.array([E, E + 7, -3], dtype=np.int32)
            ids = np.where(bad, choices[rng.integers(0, 3, size=ids.shape)], ids).astype(np.int32)
    if quant == "nvfp4b16" and global_scale is None and T * H:
        amax = float(np.abs(bf16_bits_to_f32(x)).max())
        global_scale = float(np.float32(2688.0) / np.float32(amax)) if amax > 0 else 1.0
    return Workload("case", T, H, E, K, P, M, mode, quant, seed, x,
                    np.ascontiguousarray(ids, dtype=np.int32),
                    np.ascontiguousarray(w, dtype=np.float32),
                    global_scale=global_scale)
