"""CPU oracle for the MoE dispatch/combine hot path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's ``cpu_baseline``
and ``--impl reference`` legs may import this package. The product path (the CUDA
library and its binding in ``combine_moe_route_meta_gb300``) never imports, links
or executes anything here, and this package imports nothing from it.

The arithmetic lives in plain C (``moe_oracle.c``: single-threaded, binary32
quantisation in the kernel's precision, binary64 combine). This module compiles
it with gcc (``-O2 -ffp-contract=off``, no fast-math) and wraps it for numpy.
Status bits returned by the metadata and dispatch routines:
``BAD_ID`` (an id outside [-1, E) was skipped) and ``CAPACITY`` (an expert got
more than M pairs in masked mode).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "libmoe_oracle.so")

BAD_ID = 1
CAPACITY = 2

MODES = {"normal": 0, "masked": 1}
QUANTS = {"none": 0, "fp8g128": 1, "nvfp4b16": 2, "fp8_passthrough": 4}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/libmoe_oracle.so`` (gcc, a second or two)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i64, f32 = ctypes.c_int64, ctypes.c_float
        sig = {
            "oracle_bf16_to_float": (f32, [ctypes.c_uint16]),
            "oracle_bf16_from_double": (ctypes.c_uint16, [ctypes.c_double]),
            "oracle_e4m3_to_double": (ctypes.c_double, [ctypes.c_uint8]),
            "oracle_e4m3_from_float": (ctypes.c_uint8, [f32]),
            "oracle_e2m1_to_double": (ctypes.c_double, [ctypes.c_uint8]),
            "oracle_e2m1_from_float": (ctypes.c_uint8, [f32]),
            "oracle_e4m3_from_float_array": (None, [P, i64, P]),
            "oracle_e2m1_from_float_array": (None, [P, i64, P]),
            "oracle_route_meta": (ctypes.c_int, [P, i64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                 ctypes.c_int, P, P, P, P, P]),
            "oracle_expected_m": (i64, [i64, ctypes.c_int, ctypes.c_int]),
            "oracle_dispatch_payload_bytes": (i64, [ctypes.c_int, ctypes.c_int, ctypes.c_int]),
            "oracle_quant_fp8_g128_row": (None, [P, ctypes.c_int, P, P]),
            "oracle_quant_nvfp4_b16_row": (None, [P, ctypes.c_int, f32, P, P]),
            "oracle_dispatch": (None, [ctypes.c_int, ctypes.c_int, P, i64, ctypes.c_int, P,
                                       ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, f32, P, P]),
            "oracle_combine": (None, [ctypes.c_int, P, i64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_int, P, P, P, P, P]),
            "oracle_dispatch_layout": (None, [P, i64, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, P]),
            "oracle_route_meta_aligned": (ctypes.c_int, [P, i64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                         ctypes.c_int, ctypes.c_int, P, P, P, P, P]),
            "oracle_quant_fp8_g128_ue8m0_row": (None, [P, ctypes.c_int, P, P]),
            "oracle_dispatch_partitioned": (None, [ctypes.c_int, P, i64, i64, ctypes.c_int, P, P, ctypes.c_int,
                                                   ctypes.c_int, ctypes.c_int, ctypes.c_int32, f32, P, P, P, P]),
            "oracle_combine_partitioned": (None, [P, i64, i64, ctypes.c_int, P, ctypes.c_int, ctypes.c_int,
                                                  ctypes.c_int, P]),
            "oracle_nvfp4_sf_interleave": (None, [P, i64, ctypes.c_int, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _ptr(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


# ---------------------------------------------------------------------------
# scalar codecs (exposed for the pins)
# ---------------------------------------------------------------------------

def e4m3_from_float(v: float) -> int:
    return int(_load().oracle_e4m3_from_float(float(v)))


def e4m3_to_float(c: int) -> float:
    return float(_load().oracle_e4m3_to_double(int(c)))


def e2m1_from_float(v: float) -> int:
    return int(_load().oracle_e2m1_from_float(float(v)))


def e2m1_to_float(c: int) -> float:
    return float(_load().oracle_e2m1_to_double(int(c)))


def e4m3_from_float_array(v: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.size, np.uint8)
    _load().oracle_e4m3_from_float_array(_ptr(v), v.size, _ptr(out))
    return out


def e2m1_from_float_array(v: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.size, np.uint8)
    _load().oracle_e2m1_from_float_array(_ptr(v), v.size, _ptr(out))
    return out


def bf16_from_double(v: float) -> int:
    return int(_load().oracle_bf16_from_double(float(v)))


def expected_m(T: int, K: int, E: int) -> int:
    return int(_load().oracle_expected_m(T, K, E))


def dispatch_payload_bytes(H: int, K: int, nvfp4: bool) -> int:
    return int(_load().oracle_dispatch_payload_bytes(H, K, int(bool(nvfp4))))


# ---------------------------------------------------------------------------
# the path
# ---------------------------------------------------------------------------

@dataclass
class Meta:
    seg_indptr: np.ndarray        # int64 [E+1]
    src2dst: np.ndarray           # int32 [T*K]
    reorder_topk_ids: np.ndarray  # int32 [N]
    masked_m: np.ndarray          # int32 [E]
    partition_counts: np.ndarray  # int32 [P]
    expected_m: int
    status: int

    @property
    def num_valid(self) -> int:
        return int(self.seg_indptr[-1])


def route_meta(topk_ids: np.ndarray, E: int, P: int = 1, M: int = 0) -> Meta:
    ids = np.ascontiguousarray(topk_ids, dtype=np.int32)
    T, K = ids.shape
    seg = np.zeros(E + 1, np.int64)
    s2d = np.empty(T * K, np.int32)
    reo = np.empty(max(T * K, 1), np.int32)
    mm = np.zeros(E, np.int32)
    pc = np.zeros(max(P, 1), np.int32)
    st = _load().oracle_route_meta(_ptr(ids), T, K, E, P, M, _ptr(seg), _ptr(s2d), _ptr(reo),
                                   _ptr(mm), _ptr(pc))
    n = int(seg[-1])
    return Meta(seg, s2d, reo[:n].copy(), mm, pc[:P], expected_m(T, K, E) if E else 0, int(st))


def quant_fp8_row(x_row: np.ndarray):
    x_row = np.ascontiguousarray(x_row, dtype=np.uint16)
    H = x_row.shape[0]
    q = np.empty(H, np.uint8)
    s = np.empty(H // 128, np.float32)
    _load().oracle_quant_fp8_g128_row(_ptr(x_row), H, _ptr(q), _ptr(s))
    return q, s


def quant_nvfp4_row(x_row: np.ndarray, g: float):
    x_row = np.ascontiguousarray(x_row, dtype=np.uint16)
    H = x_row.shape[0]
    q = np.empty(H // 2, np.uint8)
    sf = np.empty(H // 16, np.uint8)
    _load().oracle_quant_nvfp4_b16_row(_ptr(x_row), H, float(g), _ptr(q), _ptr(sf))
    return q, sf


def out_shapes(mode: str, quant: str, T: int, H: int, K: int, E: int, M: int, rows: Optional[int] = None):
    """(q shape, q dtype, scale shape, scale dtype) of the dispatch outputs."""
    lead = (rows if rows is not None else T * K,) if mode == "normal" else (E, M)
    if quant == "none":
        return lead + (H,), np.uint16, None, None
    if quant == "fp8_passthrough":
        return lead + (H,), np.uint8, None, None
    if quant == "fp8g128":
        return lead + (H,), np.uint8, lead + (H // 128,), np.float32
    return lead + (H // 2,), np.uint8, lead + (H // 16,), np.uint8


def _filled(shape, dtype, fill: int) -> np.ndarray:
    """Array of ``shape``/``dtype`` whose every byte is ``fill``."""
    n = int(np.prod(shape)) * np.dtype(dtype).itemsize
    return np.full(n, fill, np.uint8).view(dtype).reshape(shape)


def dispatch(mode: str, quant: str, x: np.ndarray, topk_ids: np.ndarray, meta: Meta, E: int,
             M: int = 0, global_scale: float = 0.0, rows: Optional[int] = None, fill: int = 0, out=None):
    """Returns (q, scales) in the layout of ``mode``; untouched bytes hold ``fill``.
    For quant "fp8_passthrough" x is [T, H] uint8 codes. ``out`` = (q, scales) reuses
    caller-owned arrays of the right shapes (their untouched bytes are left as they are)."""
    x = np.ascontiguousarray(x, dtype=np.uint8 if quant == "fp8_passthrough" else np.uint16)
    ids = np.ascontiguousarray(topk_ids, dtype=np.int32)
    T, H = x.shape
    K = ids.shape[1]
    qs, qd, ss, sd = out_shapes(mode, quant, T, H, K, E, M, rows)
    if out is not None:
        q, s = out
        assert q.shape == qs and q.dtype == qd and (ss is None or (s.shape == ss and s.dtype == sd))
    else:
        q = _filled(qs, qd, fill)
        s = _filled(ss, sd, fill) if ss is not None else None
    _load().oracle_dispatch(MODES[mode], QUANTS[quant], _ptr(x), T, H, _ptr(ids), K, E, M,
                            _ptr(meta.src2dst), _ptr(meta.seg_indptr), float(global_scale),
                            _ptr(q), _ptr(s))
    return q, s


def combine(mode: str, expert_out: np.ndarray, topk_ids: np.ndarray, topk_weights: np.ndarray,
            meta: Meta, E: int, M: int = 0) -> np.ndarray:
    """bf16 bits [T, H] of the weighted combine."""
    eo = np.ascontiguousarray(expert_out, dtype=np.uint16)
    ids = np.ascontiguousarray(topk_ids, dtype=np.int32)
    w = np.ascontiguousarray(topk_weights, dtype=np.float32)
    T, K = ids.shape
    H = eo.shape[-1]
    out = np.empty((T, H), np.uint16)
    _load().oracle_combine(MODES[mode], _ptr(eo), T, H, K, E, M, _ptr(ids), _ptr(meta.src2dst),
                           _ptr(meta.seg_indptr), _ptr(w), _ptr(out))
    return out


# ---------------------------------------------------------------------------
# per-partition layout (get_dispatch_layout) and the FlashInfer all-to-all layout
# ---------------------------------------------------------------------------

def dispatch_layout(topk_ids: np.ndarray, E: int, P: int):
    """(num_tokens_per_rank [P] int32, is_token_in_rank [T, P] bool, num_tokens_per_expert [E] int32)."""
    ids = np.ascontiguousarray(topk_ids, dtype=np.int32)
    T, K = ids.shape
    ntr = np.zeros(P, np.int32)
    itr = np.zeros((T, P), np.uint8)
    nte = np.zeros(E, np.int32)
    _load().oracle_dispatch_layout(_ptr(ids), T, K, E, P, _ptr(ntr), _ptr(itr), _ptr(nte))
    return ntr, itr.astype(bool), nte


def dispatch_partitioned(quant: str, x: np.ndarray, topk_ids: np.ndarray, topk_weights: np.ndarray, E: int,
                         P: int, invalid_id: int = -1, global_scale: float = 0.0, num_slots=None, fill: int = 0):
    """FlashInfer-style receive buffers of one source rank: (recv_x, recv_sf, recv_ids, recv_w)."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    ids = np.ascontiguousarray(topk_ids, dtype=np.int32)
    w = np.ascontiguousarray(topk_weights, dtype=np.float32)
    T, H = x.shape
    K = ids.shape[1]
    S = T if num_slots is None else num_slots
    if quant == "nvfp4b16":
        rx = _filled((P, S, H // 2), np.uint8, fill)
        rsf = _filled((P, S, H // 16), np.uint8, fill)
    else:
        rx = _filled((P, S, H), np.uint16, fill)
        rsf = None
    rids = _filled((P, S, K), np.int32, fill)
    rw = _filled((P, S, K), np.float32, fill)
    _load().oracle_dispatch_partitioned(QUANTS[quant], _ptr(x), T, S, H, _ptr(ids), _ptr(w), K, E, P,
                                        int(invalid_id), float(global_scale), _ptr(rx), _ptr(rsf), _ptr(rids),
                                        _ptr(rw))
    return rx, rsf, rids, rw


def combine_partitioned(partial: np.ndarray, topk_ids: np.ndarray, E: int, P: int) -> np.ndarray:
    """bf16 bits [T, H]: sum over the partitions each token was sent to of partial[p, t]."""
    pa = np.ascontiguousarray(partial, dtype=np.uint16)
    ids = np.ascontiguousarray(topk_ids, dtype=np.int32)
    T, K = ids.shape
    _, S, H = pa.shape
    out = np.empty((T, H), np.uint16)
    _load().oracle_combine_partitioned(_ptr(pa), T, S, H, _ptr(ids), K, E, P, _ptr(out))
    return out


# ---------------------------------------------------------------------------
# DeepGEMM consumer formats: expert alignment, UE8M0 scales
# ---------------------------------------------------------------------------

def route_meta_aligned(topk_ids: np.ndarray, E: int, A: int, P: int = 1, M: int = 0) -> Meta:
    """Metadata with every expert segment starting at a multiple of A; reorder_topk_ids holds
    seg_indptr[E] entries, -1 on padding rows."""
    ids = np.ascontiguousarray(topk_ids, dtype=np.int32)
    T, K = ids.shape
    seg = np.zeros(E + 1, np.int64)
    s2d = np.empty(T * K, np.int32)
    reo = np.empty(max(T * K + E * (A - 1), 1), np.int32)
    mm = np.zeros(E, np.int32)
    pc = np.zeros(max(P, 1), np.int32)
    st = _load().oracle_route_meta_aligned(_ptr(ids), T, K, E, P, M, A, _ptr(seg), _ptr(s2d), _ptr(reo),
                                           _ptr(mm), _ptr(pc))
    n = int(seg[-1])
    return Meta(seg, s2d, reo[:n].copy(), mm, pc[:P], expected_m(T, K, E) if E else 0, int(st))


def quant_fp8_ue8m0_row(x_row: np.ndarray):
    """(codes [H] uint8, UE8M0 scale bytes [H/128] uint8)."""
    x_row = np.ascontiguousarray(x_row, dtype=np.uint16)
    H = x_row.shape[0]
    q = np.empty(H, np.uint8)
    e = np.empty(H // 128, np.uint8)
    _load().oracle_quant_fp8_g128_ue8m0_row(_ptr(x_row), H, _ptr(q), _ptr(e))
    return q, e


# ---------------------------------------------------------------------------
# CUTLASS consumer format: interleaved NVFP4 block scales
# ---------------------------------------------------------------------------

def nvfp4_sf_interleave(sf: np.ndarray) -> np.ndarray:
    """nvfp4_block_scale_interleave of a [rows, cols] uint8 block-scale matrix: 1-D uint8 of
    round_up(rows, 128) * round_up(cols, 4) bytes in the 128 x 4 tile layout, zero padding."""
    sf = np.ascontiguousarray(sf, dtype=np.uint8)
    rows, cols = sf.shape
    n = (rows + 127) // 128 * 128 * ((cols + 3) // 4 * 4)
    out = np.empty(n, np.uint8)
    _load().oracle_nvfp4_sf_interleave(_ptr(sf), rows, cols, _ptr(out))
    return out
