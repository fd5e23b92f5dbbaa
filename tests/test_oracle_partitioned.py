"""Pins for the oracle's per-partition layout (get_dispatch_layout) and its FlashInfer
all-to-all layout (one source rank, P partitions), CPU only.

Checked against brute force over Python sets, numpy's bincount, and closed forms of the
combine (one partition per token gives the partial back exactly; a token routed nowhere
gives zeros; two partials round like the exact rational sum).
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from workloads import bf16_bits_to_f32, f32_to_bf16_bits, make_case


def _partitions_of(ids_row, E, P):
    ep = E // P
    return {int(e) // ep for e in ids_row if 0 <= e < E}


@pytest.mark.parametrize("seed", range(12))
def test_dispatch_layout_bruteforce(seed):
    rng = np.random.default_rng(seed)
    P = int(rng.choice([1, 2, 4, 8]))
    E = P * int(rng.integers(1, 6))
    T, K = int(rng.integers(0, 30)), int(rng.integers(1, 5))
    ids = rng.integers(-2, E + 2, size=(T, K)).astype(np.int32)
    ntr, itr, nte = oracle.dispatch_layout(ids, E, P)
    for t in range(T):
        parts = _partitions_of(ids[t], E, P)
        assert {p for p in range(P) if itr[t, p]} == parts
    assert ntr.tolist() == [sum(1 for t in range(T) if p in _partitions_of(ids[t], E, P)) for p in range(P)]
    flat = ids.reshape(-1)
    assert nte.tolist() == np.bincount(flat[(flat >= 0) & (flat < E)], minlength=E).tolist()


@pytest.mark.parametrize("quant", ["none", "nvfp4b16"])
def test_partitioned_dispatch_rows_ids_and_padding(quant):
    w = make_case(40, 64, 16, 4, seed=31, quant=quant, invalid_rate=0.1)
    P, S, INV = 4, 44, 16
    rx, rsf, rids, rw = oracle.dispatch_partitioned(quant, w.x, w.topk_ids, w.topk_weights, w.E, P,
                                                    invalid_id=INV, global_scale=w.global_scale or 0.0,
                                                    num_slots=S, fill=0x5A)
    ep = w.E // P
    sent = 0
    for p in range(P):
        for t in range(S):
            routed = t < w.T and p in _partitions_of(w.topk_ids[t], w.E, P)
            if not routed:
                assert (rids[p, t] == INV).all()
                assert (rx[p, t].view(np.uint8) == 0x5A).all()      # payload left untouched
                continue
            sent += 1
            for k in range(w.K):
                e = int(w.topk_ids[t, k])
                assert rids[p, t, k] == (e if 0 <= e < w.E and e // ep == p else INV)
                assert rw[p, t, k] == w.topk_weights[t, k]
            if quant == "none":
                assert np.array_equal(rx[p, t], w.x[t])
            else:
                q, sf = oracle.quant_nvfp4_row(w.x[t], w.global_scale)
                assert np.array_equal(rx[p, t], q) and np.array_equal(rsf[p, t], sf)
    ntr, _, _ = oracle.dispatch_layout(w.topk_ids, w.E, P)
    assert sent == int(ntr.sum())
    # every valid pair survives sanitising in exactly one partition
    valid = (w.topk_ids >= 0) & (w.topk_ids < w.E)
    kept = (rids[:, : w.T, :] != INV).sum(axis=0)
    assert np.array_equal(kept, valid.astype(kept.dtype))


def test_partitioned_combine_single_partition_is_exact():
    w = make_case(30, 48, 8, 1, seed=32)          # K = 1: each token lives in one partition
    P = 4
    rng = np.random.default_rng(3)
    partial = f32_to_bf16_bits(rng.standard_normal((P, w.T, w.H)).astype(np.float32))
    y = oracle.combine_partitioned(partial, w.topk_ids, w.E, P)
    for t in range(w.T):
        p = int(w.topk_ids[t, 0]) // (w.E // P)
        assert np.array_equal(y[t], partial[p, t])


def test_partitioned_combine_two_partials_round_once():
    ids = np.array([[0, 3]], np.int32)            # E = 4, P = 2: experts 0 and 3 -> partitions 0, 1
    rng = np.random.default_rng(4)
    partial = f32_to_bf16_bits(rng.standard_normal((2, 1, 256)).astype(np.float32))
    y = oracle.combine_partitioned(partial, ids, 4, 2)[0]
    a, b = bf16_bits_to_f32(partial[0, 0]), bf16_bits_to_f32(partial[1, 0])
    for h in range(256):
        exact = Fraction(float(a[h])) + Fraction(float(b[h]))
        assert Fraction(float(exact)) == exact                    # the sum is exact in binary64
        assert int(y[h]) == oracle.bf16_from_double(float(exact))  # one rounding (pinned separately)


def test_partitioned_combine_unrouted_token_is_zero():
    ids = np.array([[-1, -1], [1, 2]], np.int32)
    partial = np.full((2, 2, 16), 0x3F80, np.uint16)   # 1.0 everywhere
    y = oracle.combine_partitioned(partial, ids, 4, 2)
    assert (y[0] == 0).all()
    assert (bf16_bits_to_f32(y[1]) == 2.0).all()       # experts 1 and 2 live in partitions 0 and 1
