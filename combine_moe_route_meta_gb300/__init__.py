"""GB300 (sm_103a) MoE token dispatch / combine.

Python binding of the C ABI in ``include/moe_dispatch.h``. The functions named like
the C entry points (``moe_route_meta``, ``moe_dispatch``, ``moe_combine``, ...) only
marshal arguments: every step of the path runs in the CUDA kernels of
``libmoe_dispatch.so``. PyTorch supplies device memory and streams.

The higher-level helpers (:func:`route_meta`, :func:`dispatch`, :func:`combine`,
:class:`MoEDispatcher`) allocate outputs with torch and return named tuples shaped
like the dispatcher pages' outputs (``DeepEPNormalDispatchOutput`` /
``DeepEPLLDispatchOutput`` on the "sglang token_dispatcher/deepep.py" page).

There is no CPU fallback: the first call raises when the library has not been built
(``python -m combine_moe_route_meta_gb300.build``), and every call requires CUDA tensors.
"""
from __future__ import annotations

import ctypes
import os
from typing import NamedTuple, Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_dispatch.so")

# ---------------------------------------------------------------------------
# C ABI constants (mirrors include/moe_dispatch.h)
# ---------------------------------------------------------------------------
MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_CAPACITY = 3
MOE_ERR_BAD_EXPERT_ID = 4
MOE_ERR_TIMEOUT = 5
MOE_ERR_CUDA = 6

MOE_MODE_NORMAL = 0
MOE_MODE_MASKED = 1
MODES = {"normal": MOE_MODE_NORMAL, "masked": MOE_MODE_MASKED}

MOE_QUANT_NONE = 0
MOE_QUANT_FP8_G128 = 1
MOE_QUANT_NVFP4_B16 = 2
MOE_QUANT_FP8_G128_UE8M0 = 3
QUANTS = {"none": MOE_QUANT_NONE, "fp8g128": MOE_QUANT_FP8_G128, "nvfp4b16": MOE_QUANT_NVFP4_B16,
          "fp8g128_ue8m0": MOE_QUANT_FP8_G128_UE8M0, "fp8_passthrough": 4}
MOE_QUANT_FP8_PASSTHROUGH = 4
MOE_SCALES_ROW_MAJOR = 0
MOE_SCALES_COL_MAJOR = 1
MOE_SCALES_SWIZZLED_128X4 = 2
SCALE_LAYOUTS = {"row": MOE_SCALES_ROW_MAJOR, "col": MOE_SCALES_COL_MAJOR, "swizzled": MOE_SCALES_SWIZZLED_128X4}

MOE_MAX_EXPERTS = 1024
MOE_MAX_TOPK = 16

_P = ctypes.c_void_p
_i32, _i64, _int, _f32, _sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_size_t

_SIGNATURES = {
    "moe_abi_version": (_int, []),
    "moe_status_string": (ctypes.c_char_p, [_int]),
    "moe_route_meta_workspace_size": (_sz, [_i64, _int, _int]),
    "moe_route_meta": (_int, [_P, _i64, _int, _int, _int, _int, _P, _P, _P, _P, _P, _P, _P, _sz, _P, _P]),
    "moe_dispatch": (_int, [_int, _int, _P, _i64, _int, _P, _int, _int, _int, _P, _P, _f32, _P, _P, _P, _P]),
    "moe_combine": (_int, [_int, _P, _i64, _int, _int, _int, _int, _P, _P, _P, _P, _P, _P, _P]),
    "moe_convert_probe": (_int, [_P, _i64, _P, _P, _P, _P]),
    "moe_fp8_division_check": (_int, [_P, _P]),
    "moe_wait_timeout_check": (_int, [_P, _i64, _int, _P]),
    "moe_route_meta_noalloc": (_int, [_P, _i64, _int, _int, _int, _int, _P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_route_dispatch": (_int, [_int, _int, _P, _i64, _int, _P, _int, _int, _int, _int, _f32, _P, _P, _P, _P,
                                  _P, _P, _P, _sz, _P, _P, _P, _P]),
    "moe_dispatch_layout": (_int, [_P, _i64, _int, _int, _int, _P, _P, _P, _P, _P]),
    "moe_route_meta_ex": (_int, [_P, _int, _i64, _int, _int, _int, _int, _int, _P, _P, _P, _P, _P, _P, _P, _P,
                                 _sz, _P, _P]),
    "moe_dispatch_ex": (_int, [_int, _int, _int, _P, _i64, _int, _P, _int, _int, _int, _i64, _P, _P, _f32, _P, _P,
                               _P, _P]),
    "moe_combine_ex": (_int, [_int, _P, _i64, _int, _int, _int, _int, _i64, _P, _P, _P, _P, _P, _P, _P]),
    "moe_dispatch_partitioned": (_int, [_int, _P, _i64, _i64, _int, _P, _P, _int, _int, _int, _i32, _f32, _P, _P,
                                        _P, _P, _P, _P]),
    "moe_combine_partitioned": (_int, [_P, _i64, _i64, _int, _P, _int, _int, _int, _P, _P, _P]),
    "moe_dispatch_partitioned_ex": (_int, [_int, _int, _P, _i64, _i64, _int, _P, _P, _int, _int, _int, _i32, _f32,
                                           _P, _P, _P, _P, _P, _P]),
}
_lib_handle = None


def load_library() -> ctypes.CDLL:
    """Load libmoe_dispatch.so (once). Raises when it has not been built: no CPU fallback."""
    global _lib_handle
    if _lib_handle is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build the CUDA library first "
                "(python -m combine_moe_route_meta_gb300.build); there is no CPU fallback")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib_handle = lib
    return _lib_handle


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = int(status)
        super().__init__(f"{where}: {moe_status_string(status)}" if where else moe_status_string(status))


def moe_status_string(status: int) -> str:
    return load_library().moe_status_string(int(status)).decode()


def moe_abi_version() -> int:
    return int(load_library().moe_abi_version())


def moe_route_meta_workspace_size(num_tokens: int, topk: int, num_experts: int) -> int:
    return int(load_library().moe_route_meta_workspace_size(int(num_tokens), int(topk), int(num_experts)))


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("device tensor expected (the library has no CPU path)")
    if not t.is_contiguous():
        raise ValueError("contiguous tensor expected")
    return ctypes.c_void_p(t.data_ptr())


def _nbytes(t: torch.Tensor) -> int:
    return t.numel() * t.dtype.itemsize


def _need(t: Optional[torch.Tensor], nbytes: int, name: str, dtype=None) -> None:
    """Reject, before any launch, a buffer the kernels would read or write past its end (the
    C ABI takes raw pointers and cannot see sizes) or of the wrong element type."""
    if t is None:
        return
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name}: {dtype} expected, got {t.dtype}")
    if _nbytes(t) < nbytes:
        raise ValueError(f"{name}: {nbytes} bytes needed, the tensor has {_nbytes(t)}")


def _shape_bytes(shape, dtype) -> int:
    n = 1
    for d in shape:
        n *= int(d)
    return n * dtype.itemsize


def _check_meta_buffers(T: int, K: int, E: int, P: int, seg_indptr, src2dst, reorder_topk_ids, masked_m,
                        partition_counts, dev_status) -> None:
    _need(seg_indptr, 8 * (E + 1), "seg_indptr", torch.int64)
    _need(src2dst, 4 * T * K, "src2dst", torch.int32)
    _need(reorder_topk_ids, 4 * T * K, "reorder_topk_ids", torch.int32)
    _need(masked_m, 4 * E, "masked_m", torch.int32)
    _need(partition_counts, 4 * P, "partition_counts", torch.int32)
    _need(dev_status, 4, "dev_status", torch.int32)


def _check_dispatch_buffers(mode: str, quant: str, T: int, H: int, K: int, E: int, M: int, out_q,
                            out_scales) -> None:
    """The masked layout fixes the output size ([E, M, .]); the contiguous layout needs
    N = seg_indptr[E] rows, known only on the device, so only the scale buffer's presence is
    checked there."""
    qs, qd, ss, sd = dispatch_out_shapes(mode, quant, T, H, K, E, M)
    if ss is not None and out_scales is None:
        raise ValueError(f"out_scales: a scale buffer is needed for quant {quant}")
    if mode == "masked":
        _need(out_q, _shape_bytes(qs, qd), "out_q")
        if ss is not None:
            _need(out_scales, _shape_bytes(ss, sd), "out_scales")


def _scale_bytes_ex(mode: str, quant: str, layout: str, rows: int, H: int, E: int, M: int) -> int:
    """Bytes of moe_dispatch_ex's scale buffer for `rows` destination rows (normal layout) or
    E x M slots (masked), in the given layout."""
    if quant in ("none", "fp8_passthrough"):
        return 0
    if layout == "swizzled":
        R = rows if mode == "normal" else E * M
        return (R + 127) // 128 * 128 * (H // 16)
    if quant == "nvfp4b16":
        return (rows if mode == "normal" else E * M) * (H // 16)
    G = H // 128
    elem = 4 if quant == "fp8g128" else 1
    if layout == "row":
        return (rows if mode == "normal" else E * M) * G * elem
    if quant == "fp8g128":                      # column-major fp32: [G, R4] (per expert in masked)
        R4 = ((rows if mode == "normal" else M) + 3) // 4 * 4
        return (1 if mode == "normal" else E) * G * R4 * 4
    R4 = ((rows if mode == "normal" else M) + 3) // 4 * 4      # column-major UE8M0 words
    return (1 if mode == "normal" else E) * ((G + 3) // 4) * R4 * 4


def _check_partitioned_buffers(quant: str, layout: str, T: int, H: int, K: int, S: int, P: int, topk_ids,
                               topk_weights, recv_x, recv_scales, recv_topk_ids, recv_topk_weights,
                               dev_status) -> None:
    _need(topk_ids, 4 * T * K, "topk_ids", torch.int32)
    _need(topk_weights, 4 * T * K, "topk_weights", torch.float32)
    _need(recv_x, P * S * (H // 2 if quant == "nvfp4b16" else 2 * H), "recv_x")
    if quant == "nvfp4b16":
        need = (P * S + 127) // 128 * 128 * (H // 16) if layout == "swizzled" else P * S * (H // 16)
        if recv_scales is None:
            raise ValueError("recv_scales: a scale buffer is needed for quant nvfp4b16")
        _need(recv_scales, need, "recv_scales")
    _need(recv_topk_ids, 4 * P * S * K, "recv_topk_ids", torch.int32)
    _need(recv_topk_weights, 4 * P * S * K, "recv_topk_weights", torch.float32)
    _need(dev_status, 4, "dev_status", torch.int32)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        # the raw handle of torch's current stream, without building a Stream object
        return ctypes.c_void_p(torch._C._cuda_getCurrentRawStream(torch.cuda.current_device()))
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(status: int, where: str):
    if status != MOE_OK:
        raise MoEError(status, where)


# ---------------------------------------------------------------------------
# thin wrappers with the C names
# ---------------------------------------------------------------------------

def moe_route_meta(topk_ids: torch.Tensor, num_experts: int, seg_indptr: torch.Tensor,
                   src2dst: torch.Tensor, reorder_topk_ids: torch.Tensor, masked_m: torch.Tensor,
                   dev_status: torch.Tensor, workspace: Optional[torch.Tensor] = None,
                   num_partitions: int = 1, max_tokens_per_expert: int = 0,
                   partition_counts: Optional[torch.Tensor] = None, stream=None) -> int:
    """Launch moe_route_meta; returns expected_m (computed on the host)."""
    T, K = topk_ids.shape
    _need(topk_ids, 4 * T * K, "topk_ids", torch.int32)
    _check_meta_buffers(T, K, num_experts, num_partitions, seg_indptr, src2dst, reorder_topk_ids, masked_m,
                        partition_counts, dev_status)
    em = ctypes.c_int32(0)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = load_library().moe_route_meta(_ptr(topk_ids), T, K, num_experts, num_partitions, max_tokens_per_expert,
                             _ptr(seg_indptr), _ptr(src2dst), _ptr(reorder_topk_ids), _ptr(masked_m),
                             _ptr(partition_counts), ctypes.byref(em), _ptr(workspace), ws_bytes,
                             _ptr(dev_status), _stream(stream))
    _check(st, "moe_route_meta")
    return int(em.value)


def moe_route_meta_noalloc(topk_ids: torch.Tensor, num_experts: int, seg_indptr: torch.Tensor,
                           src2dst: torch.Tensor, reorder_topk_ids: torch.Tensor, masked_m: torch.Tensor,
                           dev_status: torch.Tensor, num_partitions: int = 1, max_tokens_per_expert: int = 0,
                           partition_counts: Optional[torch.Tensor] = None, stream=None) -> int:
    """moe_route_meta for callers that cannot allocate device memory: no workspace argument.

    Scratch comes from a fixed 1 MiB array inside the library (held on every GPU that loads
    it); larger problems raise MoEError(MOE_ERR_UNSUPPORTED). The first call on a device
    looks up that array and should come before any stream capture. All calls share the
    array, so calls that could overlap on the GPU must not be issued. Returns expected_m.
    """
    T, K = topk_ids.shape
    _need(topk_ids, 4 * T * K, "topk_ids", torch.int32)
    _check_meta_buffers(T, K, num_experts, num_partitions, seg_indptr, src2dst, reorder_topk_ids, masked_m,
                        partition_counts, dev_status)
    em = ctypes.c_int32(0)
    st = load_library().moe_route_meta_noalloc(_ptr(topk_ids), T, K, num_experts, num_partitions,
                                               max_tokens_per_expert, _ptr(seg_indptr), _ptr(src2dst),
                                               _ptr(reorder_topk_ids), _ptr(masked_m), _ptr(partition_counts),
                                               ctypes.byref(em), _ptr(dev_status), _stream(stream))
    _check(st, "moe_route_meta_noalloc")
    return int(em.value)


def moe_dispatch(mode: str, quant: str, hidden_states: torch.Tensor, topk_ids: torch.Tensor,
                 num_experts: int, src2dst: torch.Tensor, seg_indptr: torch.Tensor,
                 out_q: torch.Tensor, out_scales: Optional[torch.Tensor], dev_status: torch.Tensor,
                 max_tokens_per_expert: int = 0, input_global_scale: float = 0.0, stream=None) -> None:
    T, H = hidden_states.shape
    K = topk_ids.shape[1]
    _need(topk_ids, 4 * T * K, "topk_ids", torch.int32)
    _need(src2dst, 4 * T * K, "src2dst", torch.int32)
    _need(seg_indptr, 8 * (num_experts + 1) if mode == "masked" else 0, "seg_indptr", torch.int64)
    _need(dev_status, 4, "dev_status", torch.int32)
    _check_dispatch_buffers(mode, quant, T, H, K, num_experts, max_tokens_per_expert, out_q, out_scales)
    st = load_library().moe_dispatch(MODES[mode], QUANTS[quant], _ptr(hidden_states), T, H, _ptr(topk_ids), K,
                           num_experts, max_tokens_per_expert, _ptr(src2dst), _ptr(seg_indptr),
                           float(input_global_scale), _ptr(out_q), _ptr(out_scales), _ptr(dev_status),
                           _stream(stream))
    _check(st, "moe_dispatch")


def moe_route_dispatch(mode: str, quant: str, hidden_states: torch.Tensor, topk_ids: torch.Tensor,
                       num_experts: int, seg_indptr: torch.Tensor, src2dst: torch.Tensor,
                       reorder_topk_ids: torch.Tensor, masked_m: torch.Tensor, out_q: torch.Tensor,
                       out_scales: Optional[torch.Tensor], dev_status: torch.Tensor,
                       workspace: Optional[torch.Tensor] = None, num_partitions: int = 1,
                       max_tokens_per_expert: int = 0, input_global_scale: float = 0.0,
                       partition_counts: Optional[torch.Tensor] = None, stream=None) -> int:
    """moe_route_meta + moe_dispatch in one call; returns expected_m."""
    T, H = hidden_states.shape
    K = topk_ids.shape[1]
    _need(topk_ids, 4 * T * K, "topk_ids", torch.int32)
    _check_meta_buffers(T, K, num_experts, num_partitions, seg_indptr, src2dst, reorder_topk_ids, masked_m,
                        partition_counts, dev_status)
    _check_dispatch_buffers(mode, quant, T, H, K, num_experts, max_tokens_per_expert, out_q, out_scales)
    em = ctypes.c_int32(0)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = load_library().moe_route_dispatch(
        MODES[mode], QUANTS[quant], _ptr(hidden_states), T, H, _ptr(topk_ids), K, num_experts, num_partitions,
        max_tokens_per_expert, float(input_global_scale), _ptr(seg_indptr), _ptr(src2dst), _ptr(reorder_topk_ids),
        _ptr(masked_m), _ptr(partition_counts), ctypes.byref(em), _ptr(workspace), ws_bytes, _ptr(out_q),
        _ptr(out_scales), _ptr(dev_status), _stream(stream))
    _check(st, "moe_route_dispatch")
    return int(em.value)


def moe_combine(mode: str, expert_out: torch.Tensor, topk_ids: torch.Tensor, topk_weights: torch.Tensor,
                num_experts: int, src2dst: torch.Tensor, seg_indptr: torch.Tensor, out: torch.Tensor,
                dev_status: torch.Tensor, max_tokens_per_expert: int = 0, stream=None) -> None:
    T, K = topk_ids.shape
    H = out.shape[1]
    # the contiguous layout reads N = seg_indptr[E] rows (known only on the device)
    rows = 0 if mode == "normal" else num_experts * max_tokens_per_expert
    _need(expert_out, 2 * rows * H, "expert_out", torch.bfloat16)
    _need(topk_ids, 4 * T * K, "topk_ids", torch.int32)
    _need(topk_weights, 4 * T * K, "topk_weights", torch.float32)
    _need(src2dst, 4 * T * K, "src2dst", torch.int32)
    _need(seg_indptr, 8 * (num_experts + 1) if mode == "masked" else 0, "seg_indptr", torch.int64)
    _need(out, 2 * T * H, "out", torch.bfloat16)
    _need(dev_status, 4, "dev_status", torch.int32)
    st = load_library().moe_combine(MODES[mode], _ptr(expert_out), T, H, K, num_experts, max_tokens_per_expert,
                          _ptr(topk_ids), _ptr(src2dst), _ptr(seg_indptr), _ptr(topk_weights), _ptr(out),
                          _ptr(dev_status), _stream(stream))
    _check(st, "moe_combine")


def moe_convert_probe(x: torch.Tensor, e4m3: Optional[torch.Tensor] = None, e2m1: Optional[torch.Tensor] = None,
                      e4m3_value: Optional[torch.Tensor] = None, stream=None) -> None:
    """Diagnostics: the quantisers' e4m3 / e2m1 conversions applied to fp32 values ``x``."""
    st = load_library().moe_convert_probe(_ptr(x), x.numel(), _ptr(e4m3), _ptr(e2m1), _ptr(e4m3_value), _stream(stream))
    _check(st, "moe_convert_probe")


def moe_fp8_division_check(result: torch.Tensor, stream=None) -> None:
    """Diagnostics: result ([4] int64) <- (pairs with different e4m3 codes, the first of them,
    quotient differences with |x/s| >= 2^-12, all quotient differences) of the FP8 quantiser's
    division against the IEEE division over its whole input domain."""
    st = load_library().moe_fp8_division_check(_ptr(result), _stream(stream))
    _check(st, "moe_fp8_division_check")


def moe_wait_timeout_check(dev_status: torch.Tensor, limit_ns: int, complete: bool, stream=None) -> None:
    """Diagnostics: the bulk dispatch kernels' bounded mbarrier wait on a barrier that is
    completed first (complete=True: dev_status stays MOE_OK) or never (complete=False: the
    wait gives up after limit_ns and dev_status becomes MOE_ERR_TIMEOUT)."""
    _need(dev_status, 4, "dev_status", torch.int32)
    st = load_library().moe_wait_timeout_check(_ptr(dev_status), int(limit_ns), 1 if complete else 0,
                                               _stream(stream))
    _check(st, "moe_wait_timeout_check")


def moe_route_meta_ex(topk_ids: torch.Tensor, num_experts: int, seg_indptr: torch.Tensor, src2dst: torch.Tensor,
                      reorder_topk_ids: torch.Tensor, masked_m: torch.Tensor, dev_status: torch.Tensor,
                      workspace: Optional[torch.Tensor] = None, num_partitions: int = 1,
                      max_tokens_per_expert: int = 0, expert_alignment: int = 1,
                      partition_counts: Optional[torch.Tensor] = None,
                      topk_ids_i32_out: Optional[torch.Tensor] = None, stream=None) -> int:
    """moe_route_meta with expert segments aligned to ``expert_alignment`` rows and int32 or int64
    ``topk_ids`` (optionally also written as int32 to ``topk_ids_i32_out``); returns expected_m."""
    T, K = topk_ids.shape
    E, A = num_experts, max(int(expert_alignment), 1)
    if topk_ids.dtype not in (torch.int32, torch.int64):
        raise ValueError(f"topk_ids: int32 or int64 expected, got {topk_ids.dtype}")
    _need(seg_indptr, 8 * (E + 1), "seg_indptr", torch.int64)
    _need(src2dst, 4 * T * K, "src2dst", torch.int32)
    _need(reorder_topk_ids, 4 * (T * K + E * (A - 1)), "reorder_topk_ids", torch.int32)
    _need(masked_m, 4 * E, "masked_m", torch.int32)
    _need(partition_counts, 4 * num_partitions, "partition_counts", torch.int32)
    _need(topk_ids_i32_out, 4 * T * K, "topk_ids_i32_out", torch.int32)
    _need(dev_status, 4, "dev_status", torch.int32)
    em = ctypes.c_int32(0)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = load_library().moe_route_meta_ex(_ptr(topk_ids), topk_ids.element_size(), T, K, num_experts,
                                          num_partitions, max_tokens_per_expert, expert_alignment, _ptr(seg_indptr),
                                          _ptr(src2dst), _ptr(reorder_topk_ids), _ptr(masked_m),
                                          _ptr(partition_counts), _ptr(topk_ids_i32_out), ctypes.byref(em),
                                          _ptr(workspace), ws_bytes, _ptr(dev_status), _stream(stream))
    _check(st, "moe_route_meta_ex")
    return int(em.value)


def moe_dispatch_ex(mode: str, quant: str, scale_layout: str, hidden_states: torch.Tensor, topk_ids: torch.Tensor,
                    num_experts: int, src2dst: torch.Tensor, seg_indptr: torch.Tensor, out_q: torch.Tensor,
                    out_scales: Optional[torch.Tensor], dev_status: torch.Tensor, max_tokens_per_expert: int = 0,
                    out_rows: int = 0, input_global_scale: float = 0.0, stream=None) -> None:
    T, H = hidden_states.shape
    K = topk_ids.shape[1]
    E, M = num_experts, max_tokens_per_expert
    rows = int(out_rows) if (mode == "normal" and out_rows) else T * K
    row_bytes = {"none": 2 * H, "nvfp4b16": H // 2}.get(quant, H)   # passthrough: H is already bytes
    # sizes are fixed by the masked layout, by a declared out_rows, or (swizzled scales) by
    # the row count the tile layout is built over; otherwise N rows, known only on the device
    declared = mode == "masked" or bool(out_rows)
    _need(out_q, (rows if mode == "normal" else E * M) * row_bytes if declared else 0, "out_q")
    need_s = _scale_bytes_ex(mode, quant, scale_layout, rows, H, E, M)
    if need_s and out_scales is None:
        raise ValueError(f"out_scales: a scale buffer is needed for quant {quant}")
    _need(out_scales, need_s if (declared or scale_layout == "swizzled") else 0, "out_scales")
    _need(topk_ids, 4 * T * K, "topk_ids", torch.int32)
    _need(src2dst, 4 * T * K, "src2dst", torch.int32)
    _need(seg_indptr, 8 * (E + 1) if mode == "masked" else 0, "seg_indptr", torch.int64)
    _need(dev_status, 4, "dev_status", torch.int32)
    st = load_library().moe_dispatch_ex(MODES[mode], QUANTS[quant], SCALE_LAYOUTS[scale_layout], _ptr(hidden_states),
                                        T, H, _ptr(topk_ids), K, num_experts, max_tokens_per_expert, int(out_rows),
                                        _ptr(src2dst), _ptr(seg_indptr), float(input_global_scale), _ptr(out_q),
                                        _ptr(out_scales), _ptr(dev_status), _stream(stream))
    _check(st, "moe_dispatch_ex")


def moe_combine_ex(mode: str, expert_out: torch.Tensor, topk_ids: torch.Tensor, topk_weights: torch.Tensor,
                   num_experts: int, src2dst: torch.Tensor, seg_indptr: torch.Tensor, out: torch.Tensor,
                   dev_status: torch.Tensor, max_tokens_per_expert: int = 0, expert_out_rows: int = 0,
                   stream=None) -> None:
    T, K = topk_ids.shape
    H = out.shape[1]
    if mode == "normal":
        rows = int(expert_out_rows)   # a declared capacity; 0: N rows, known only on the device
    else:
        rows = num_experts * max_tokens_per_expert
    _need(expert_out, 2 * rows * H, "expert_out", torch.bfloat16)
    _need(topk_ids, 4 * T * K, "topk_ids", torch.int32)
    _need(topk_weights, 4 * T * K, "topk_weights", torch.float32)
    _need(src2dst, 4 * T * K, "src2dst", torch.int32)
    _need(seg_indptr, 8 * (num_experts + 1) if mode == "masked" else 0, "seg_indptr", torch.int64)
    _need(out, 2 * T * H, "out", torch.bfloat16)
    _need(dev_status, 4, "dev_status", torch.int32)
    st = load_library().moe_combine_ex(MODES[mode], _ptr(expert_out), T, H, K, num_experts, max_tokens_per_expert,
                                       int(expert_out_rows), _ptr(topk_ids), _ptr(src2dst), _ptr(seg_indptr),
                                       _ptr(topk_weights), _ptr(out), _ptr(dev_status), _stream(stream))
    _check(st, "moe_combine_ex")


def moe_dispatch_layout(topk_ids: torch.Tensor, num_experts: int, num_partitions: int,
                        num_tokens_per_rank: torch.Tensor, is_token_in_rank: torch.Tensor, dev_status: torch.Tensor,
                        num_tokens_per_expert: Optional[torch.Tensor] = None, stream=None) -> None:
    T, K = topk_ids.shape
    _need(topk_ids, 4 * T * K, "topk_ids", torch.int32)
    _need(num_tokens_per_rank, 4 * num_partitions, "num_tokens_per_rank", torch.int32)
    _need(is_token_in_rank, T * num_partitions, "is_token_in_rank")
    _need(num_tokens_per_expert, 4 * num_experts, "num_tokens_per_expert", torch.int32)
    _need(dev_status, 4, "dev_status", torch.int32)
    st = load_library().moe_dispatch_layout(_ptr(topk_ids), T, K, num_experts, num_partitions,
                                            _ptr(num_tokens_per_rank), _ptr(is_token_in_rank),
                                            _ptr(num_tokens_per_expert), _ptr(dev_status), _stream(stream))
    _check(st, "moe_dispatch_layout")


def moe_dispatch_partitioned(quant: str, hidden_states: torch.Tensor, topk_ids: torch.Tensor,
                             topk_weights: torch.Tensor, num_experts: int, num_partitions: int,
                             recv_x: torch.Tensor, recv_scales: Optional[torch.Tensor], recv_topk_ids: torch.Tensor,
                             recv_topk_weights: torch.Tensor, dev_status: torch.Tensor, invalid_expert_id: int = -1,
                             input_global_scale: float = 0.0, stream=None) -> None:
    T, H = hidden_states.shape
    K = topk_ids.shape[1]
    S = recv_topk_ids.shape[1]
    _check_partitioned_buffers(quant, "row", T, H, K, S, num_partitions, topk_ids, topk_weights, recv_x,
                               recv_scales, recv_topk_ids, recv_topk_weights, dev_status)
    st = load_library().moe_dispatch_partitioned(
        QUANTS[quant], _ptr(hidden_states), T, S, H, _ptr(topk_ids), _ptr(topk_weights), K, num_experts,
        num_partitions, int(invalid_expert_id), float(input_global_scale), _ptr(recv_x), _ptr(recv_scales),
        _ptr(recv_topk_ids), _ptr(recv_topk_weights), _ptr(dev_status), _stream(stream))
    _check(st, "moe_dispatch_partitioned")


def moe_dispatch_partitioned_ex(quant: str, scale_layout: str, hidden_states: torch.Tensor, topk_ids: torch.Tensor,
                                topk_weights: torch.Tensor, num_experts: int, num_partitions: int,
                                recv_x: torch.Tensor, recv_scales: Optional[torch.Tensor], recv_topk_ids: torch.Tensor,
                                recv_topk_weights: torch.Tensor, dev_status: torch.Tensor, invalid_expert_id: int = -1,
                                input_global_scale: float = 0.0, stream=None) -> None:
    T, H = hidden_states.shape
    K = topk_ids.shape[1]
    S = recv_topk_ids.shape[1]
    _check_partitioned_buffers(quant, scale_layout, T, H, K, S, num_partitions, topk_ids, topk_weights, recv_x,
                               recv_scales, recv_topk_ids, recv_topk_weights, dev_status)
    st = load_library().moe_dispatch_partitioned_ex(
        QUANTS[quant], SCALE_LAYOUTS[scale_layout], _ptr(hidden_states), T, S, H, _ptr(topk_ids), _ptr(topk_weights),
        K, num_experts, num_partitions, int(invalid_expert_id), float(input_global_scale), _ptr(recv_x),
        _ptr(recv_scales), _ptr(recv_topk_ids), _ptr(recv_topk_weights), _ptr(dev_status), _stream(stream))
    _check(st, "moe_dispatch_partitioned_ex")


def swizzled_scale_bytes(rows: int, hidden: int) -> int:
    """Bytes of a MOE_SCALES_SWIZZLED_128X4 NVFP4 scale buffer for `rows` destination rows."""
    return (rows + 127) // 128 * 128 * (hidden // 16)


def moe_combine_partitioned(partial: torch.Tensor, topk_ids: torch.Tensor, num_experts: int, num_partitions: int,
                            out: torch.Tensor, dev_status: torch.Tensor, stream=None) -> None:
    T, K = topk_ids.shape
    _, S, H = partial.shape
    _need(partial, num_partitions * S * H * 2, "partial", torch.bfloat16)
    _need(topk_ids, 4 * T * K, "topk_ids", torch.int32)
    _need(out, 2 * T * H, "out", torch.bfloat16)
    _need(dev_status, 4, "dev_status", torch.int32)
    st = load_library().moe_combine_partitioned(_ptr(partial), T, S, H, _ptr(topk_ids), K, num_experts,
                                                num_partitions, _ptr(out), _ptr(dev_status), _stream(stream))
    _check(st, "moe_combine_partitioned")


# ---------------------------------------------------------------------------
# convenience layer: allocates outputs, returns the pages' tuple shapes
# ---------------------------------------------------------------------------

class RouteMeta(NamedTuple):
    seg_indptr: torch.Tensor        # int64 [E+1]
    src2dst: torch.Tensor           # int32 [T*K]
    reorder_topk_ids: torch.Tensor  # int32 [T*K]; first seg_indptr[E] entries valid
    masked_m: torch.Tensor          # int32 [E]
    partition_counts: torch.Tensor  # int32 [P]
    expected_m: int


class NormalDispatchOutput(NamedTuple):
    """Expert-contiguous dispatch (DeepEPNormalDispatchOutput with the permute metadata)."""
    hidden_states: torch.Tensor            # [T*K (capacity), H] bf16 / [.., H] uint8 / [.., H/2] uint8
    hidden_states_scale: Optional[torch.Tensor]
    topk_ids: torch.Tensor
    topk_weights: torch.Tensor
    seg_indptr: torch.Tensor
    reorder_topk_ids: torch.Tensor
    src2dst: torch.Tensor


class LLDispatchOutput(NamedTuple):
    """Masked-layout dispatch (DeepEPLLDispatchOutput)."""
    hidden_states: torch.Tensor            # [E, M, H] bf16 / [E, M, H] uint8 / [E, M, H/2] uint8
    hidden_states_scale: Optional[torch.Tensor]
    topk_ids: torch.Tensor
    topk_weights: torch.Tensor
    masked_m: torch.Tensor
    expected_m: int


def new_status(device=None) -> torch.Tensor:
    """A zeroed device status word."""
    return torch.zeros(1, dtype=torch.int32, device=device or "cuda")


def check_status(dev_status: torch.Tensor, where: str = "device") -> None:
    """Synchronise on the status word and raise MoEError if a kernel reported an error."""
    v = int(dev_status.item())
    if v != MOE_OK:
        raise MoEError(v, where)


def new_workspace(num_tokens: int, topk: int, num_experts: int, device=None) -> Optional[torch.Tensor]:
    n = moe_route_meta_workspace_size(num_tokens, topk, num_experts)
    if n == 0:
        return None
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def dispatch_out_shapes(mode: str, quant: str, T: int, H: int, K: int, E: int, M: int):
    lead = (T * K,) if mode == "normal" else (E, M)
    if quant == "none":
        return lead + (H,), torch.bfloat16, None, None
    if quant == "fp8g128":
        return lead + (H,), torch.uint8, lead + (H // 128,), torch.float32
    if quant == "fp8g128_ue8m0":
        return lead + (H,), torch.uint8, lead + (H // 128,), torch.uint8
    if quant == "fp8_passthrough":
        return lead + (H,), torch.uint8, None, None
    return lead + (H // 2,), torch.uint8, lead + (H // 16,), torch.uint8


def route_meta(topk_ids: torch.Tensor, num_experts: int, num_partitions: int = 1,
               max_tokens_per_expert: int = 0, workspace: Optional[torch.Tensor] = None,
               dev_status: Optional[torch.Tensor] = None, stream=None) -> RouteMeta:
    T, K = topk_ids.shape
    dev = topk_ids.device
    seg = torch.empty(num_experts + 1, dtype=torch.int64, device=dev)
    s2d = torch.empty(T * K, dtype=torch.int32, device=dev)
    reo = torch.empty(max(T * K, 1), dtype=torch.int32, device=dev)
    mm = torch.empty(num_experts, dtype=torch.int32, device=dev)
    pc = torch.empty(num_partitions, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = new_workspace(T, K, num_experts, dev)
    if dev_status is None:
        dev_status = new_status(dev)
    em = moe_route_meta(topk_ids, num_experts, seg, s2d, reo, mm, dev_status, workspace,
                        num_partitions, max_tokens_per_expert, pc, stream)
    return RouteMeta(seg, s2d, reo, mm, pc, em)


def dispatch(hidden_states: torch.Tensor, topk_ids: torch.Tensor, topk_weights: torch.Tensor,
             meta: RouteMeta, num_experts: int, mode: str = "normal", quant: str = "none",
             max_tokens_per_expert: int = 0, input_global_scale: float = 0.0,
             dev_status: Optional[torch.Tensor] = None, stream=None):
    T, H = hidden_states.shape
    K = topk_ids.shape[1]
    M = max_tokens_per_expert
    qs, qd, ss, sd = dispatch_out_shapes(mode, quant, T, H, K, num_experts, M)
    dev = hidden_states.device
    q = torch.empty(qs, dtype=qd, device=dev)
    s = torch.empty(ss, dtype=sd, device=dev) if ss is not None else None
    if dev_status is None:
        dev_status = new_status(dev)
    moe_dispatch(mode, quant, hidden_states, topk_ids, num_experts, meta.src2dst, meta.seg_indptr, q, s,
                 dev_status, M, input_global_scale, stream)
    if mode == "normal":
        return NormalDispatchOutput(q, s, topk_ids, topk_weights, meta.seg_indptr, meta.reorder_topk_ids,
                                    meta.src2dst)
    return LLDispatchOutput(q, s, topk_ids, topk_weights, meta.masked_m, meta.expected_m)


def combine(expert_out: torch.Tensor, topk_ids: torch.Tensor, topk_weights: torch.Tensor,
            meta: RouteMeta, num_experts: int, mode: str = "normal", max_tokens_per_expert: int = 0,
            out: Optional[torch.Tensor] = None, dev_status: Optional[torch.Tensor] = None,
            stream=None) -> torch.Tensor:
    T, K = topk_ids.shape
    H = expert_out.shape[-1]
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=expert_out.device)
    if dev_status is None:
        dev_status = new_status(expert_out.device)
    moe_combine(mode, expert_out, topk_ids, topk_weights, num_experts, meta.src2dst, meta.seg_indptr,
                out, dev_status, max_tokens_per_expert, stream)
    return out


class MoEDispatcher:
    """Pre-allocated buffers for repeated dispatch/combine of one shape (graph-capturable).

    Every launch goes to the current torch stream (or ``stream``); no call allocates
    after construction, so the three launches can be captured in a CUDA graph.
    """

    def __init__(self, num_tokens: int, hidden: int, topk: int, num_experts: int, *, mode: str = "normal",
                 quant: str = "none", num_partitions: int = 1, max_tokens_per_expert: int = 0,
                 device=None):
        self.T, self.H, self.K, self.E = num_tokens, hidden, topk, num_experts
        self.mode, self.quant, self.P, self.M = mode, quant, num_partitions, max_tokens_per_expert
        dev = torch.device(device or "cuda")
        T, K, E = num_tokens, topk, num_experts
        self.status = new_status(dev)
        self.workspace = new_workspace(T, K, E, dev)
        self.seg_indptr = torch.zeros(E + 1, dtype=torch.int64, device=dev)
        self.src2dst = torch.empty(max(T * K, 1), dtype=torch.int32, device=dev)
        self.reorder_topk_ids = torch.empty(max(T * K, 1), dtype=torch.int32, device=dev)
        self.masked_m = torch.zeros(E, dtype=torch.int32, device=dev)
        self.partition_counts = torch.zeros(num_partitions, dtype=torch.int32, device=dev)
        qs, qd, ss, sd = dispatch_out_shapes(mode, quant, T, hidden, K, E, max_tokens_per_expert)
        self.out_q = torch.empty(qs, dtype=qd, device=dev)
        self.out_scales = torch.empty(ss, dtype=sd, device=dev) if ss is not None else None
        self.out = torch.empty((T, hidden), dtype=torch.bfloat16, device=dev)
        self.expected_m = (T * K + E) // E

    def route(self, topk_ids: torch.Tensor, stream=None) -> int:
        self.expected_m = moe_route_meta(topk_ids, self.E, self.seg_indptr, self.src2dst, self.reorder_topk_ids,
                                         self.masked_m, self.status, self.workspace, self.P, self.M,
                                         self.partition_counts, stream)
        return self.expected_m

    def route_dispatch(self, hidden_states: torch.Tensor, topk_ids: torch.Tensor, input_global_scale: float = 0.0,
                       stream=None) -> int:
        """route() and dispatch() in one library call (one kernel for small batches)."""
        self.expected_m = moe_route_dispatch(self.mode, self.quant, hidden_states, topk_ids, self.E, self.seg_indptr,
                                             self.src2dst, self.reorder_topk_ids, self.masked_m, self.out_q,
                                             self.out_scales, self.status, self.workspace, self.P, self.M,
                                             input_global_scale, self.partition_counts, stream)
        return self.expected_m

    def dispatch(self, hidden_states: torch.Tensor, topk_ids: torch.Tensor, input_global_scale: float = 0.0,
                 stream=None) -> None:
        moe_dispatch(self.mode, self.quant, hidden_states, topk_ids, self.E, self.src2dst, self.seg_indptr,
                     self.out_q, self.out_scales, self.status, self.M, input_global_scale, stream)

    def combine(self, expert_out: torch.Tensor, topk_ids: torch.Tensor, topk_weights: torch.Tensor,
                stream=None) -> torch.Tensor:
        moe_combine(self.mode, expert_out, topk_ids, topk_weights, self.E, self.src2dst, self.seg_indptr,
                    self.out, self.status, self.M, stream)
        return self.out

    def check(self) -> None:
        check_status(self.status, "MoEDispatcher")
