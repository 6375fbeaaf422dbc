"""Host-side argument checks of the Python binding, with CPU tensors: the
shape, layout and dtype rules of the cache writes, and the refusal of
anything that is not a CUDA tensor (the binding has no CPU path)."""
import pytest
import torch

from paged_kv_cache_slot_gb300 import bkv


def _rows(n=5, h=8, d=128, dtype=torch.bfloat16):
    return torch.zeros(n, h, d, dtype=dtype)


def _cache(tb=3, bs=16, h=8, d=128, dtype=torch.bfloat16):
    return torch.zeros(tb, bs, h, d, dtype=dtype)


def test_check_kv_rows_accepts_and_returns_the_dtype_code():
    assert bkv._check_kv_rows(_rows(), _rows(), _cache(), _cache()) == bkv.BKV_BF16
    f32 = torch.float32
    assert bkv._check_kv_rows(_rows(dtype=f32), _rows(dtype=f32), _cache(dtype=f32), _cache(dtype=f32)) == bkv.BKV_F32
    u8 = torch.uint8
    assert bkv._check_kv_rows(_rows(dtype=f32), _rows(dtype=f32), _cache(dtype=u8), _cache(dtype=u8),
                              fp8=True) == bkv.BKV_F32
    # a row stride (rows sliced out of a fused buffer) is allowed
    fused = torch.zeros(5, 3, 8, 128, dtype=torch.bfloat16)
    assert bkv._check_kv_rows(fused[:, 1], fused[:, 2], _cache(), _cache()) == bkv.BKV_BF16


@pytest.mark.parametrize("case,exc", [
    ("cache_rank", ValueError), ("cache_shapes", ValueError), ("row_shape", ValueError), ("row_heads", ValueError),
    ("strided_inner", ValueError), ("mixed", TypeError), ("fp8_cache_dtype", TypeError), ("fp8_mixed", TypeError),
    ("int_rows", TypeError)])
def test_check_kv_rows_rejects(case, exc):
    k, v, kc, vc, fp8 = _rows(), _rows(), _cache(), _cache(), False
    if case == "cache_rank":
        kc = vc = torch.zeros(3, 16, 1024, dtype=torch.bfloat16)
    elif case == "cache_shapes":
        vc = _cache(tb=4)
    elif case == "row_shape":
        v = _rows(n=6)
    elif case == "row_heads":
        k = v = _rows(h=4)
    elif case == "strided_inner":
        k = v = torch.zeros(5, 8, 256, dtype=torch.bfloat16)[:, :, ::2]
    elif case == "mixed":
        v = _rows(dtype=torch.float32)
    elif case == "fp8_cache_dtype":
        fp8 = True
    elif case == "fp8_mixed":
        kc = vc = _cache(dtype=torch.uint8)
        v, fp8 = _rows(dtype=torch.float32), True
    elif case == "int_rows":
        k = v = _rows(dtype=torch.int16)
        kc = vc = _cache(dtype=torch.int16)
    with pytest.raises(exc):
        bkv._check_kv_rows(k, v, kc, vc, fp8=fp8)


def test_binding_refuses_host_tensors():
    """Every call marshals device pointers only; a CPU tensor is an error, never a CPU fallback."""
    table = torch.ones(2, 4, dtype=torch.int32)
    req = torch.zeros(3, dtype=torch.int32)
    pos = torch.zeros(3, dtype=torch.int64)
    slots = torch.zeros(3, dtype=torch.int64)
    with pytest.raises(TypeError, match="CUDA tensor"):
        bkv.bkv_compute_slot_mapping(table, req, pos, 16, slots)
    with pytest.raises(TypeError, match="CUDA tensor"):
        bkv.bkv_cache_write(_rows(3), _rows(3), slots, _cache(), _cache())
    with pytest.raises(TypeError, match="CUDA tensor"):
        bkv.bkv_slot_mapping_cache_write(table, req, pos, slots, _rows(3), _rows(3), _cache(), _cache())
