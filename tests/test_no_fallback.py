"""The product path has no CPU fallback (CPU only, no compute call): the binding raises when
the CUDA library is missing, and rejects host tensors instead of computing on the CPU."""
import pytest
import torch

import combine_moe_route_meta_gb300 as moe


def test_missing_library_raises(monkeypatch, tmp_path):
    monkeypatch.setattr(moe, "LIB_PATH", str(tmp_path / "libmoe_dispatch.so"))
    monkeypatch.setattr(moe, "_lib_handle", None)
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        moe.load_library()
    ids = torch.zeros((4, 2), dtype=torch.int32)
    with pytest.raises(RuntimeError, match="missing"):
        moe.moe_route_meta(ids, 8, torch.zeros(9, dtype=torch.int64), torch.zeros(8, dtype=torch.int32),
                           torch.zeros(8, dtype=torch.int32), torch.zeros(8, dtype=torch.int32),
                           torch.zeros(1, dtype=torch.int32))


def test_host_tensors_are_rejected():
    T, K, E = 4, 2, 8
    ids = torch.zeros((T, K), dtype=torch.int32)
    with pytest.raises(ValueError, match="no CPU path"):
        moe.moe_route_meta(ids, E, torch.zeros(E + 1, dtype=torch.int64), torch.zeros(T * K, dtype=torch.int32),
                           torch.zeros(T * K, dtype=torch.int32), torch.zeros(E, dtype=torch.int32),
                           torch.zeros(1, dtype=torch.int32))
    x = torch.zeros((T, 128), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="no CPU path"):
        moe.moe_combine("normal", torch.zeros((T * K, 128), dtype=torch.bfloat16), ids,
                        torch.zeros((T, K), dtype=torch.float32), E, torch.zeros(T * K, dtype=torch.int32),
                        torch.zeros(E + 1, dtype=torch.int64), x, torch.zeros(1, dtype=torch.int32))
