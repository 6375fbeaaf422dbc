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


class _FakeLib:
    """Records the arguments each entry point is called with."""

    def __init__(self):
        self.calls = {}

    def __getattr__(self, name):
        def f(*args):
            self.calls[name] = args
            return 0
        return f


@pytest.fixture
def fake(monkeypatch):
    lib = _FakeLib()
    monkeypatch.setattr(bkv, "load", lambda: lib)
    ptrs = {}
    monkeypatch.setattr(bkv, "_dev", lambda t, name, dtype=None, contiguous=True: ptrs.setdefault(name, len(ptrs) + 1))
    monkeypatch.setattr(bkv, "_stream", lambda s: 999)
    lib.ptrs = ptrs
    return lib


def test_cache_write_marshalling(fake):
    fused = torch.zeros(5, 3, 8, 128, dtype=torch.float32)
    k, v = fused[:, 1], fused[:, 2]                                   # row stride 3 * 8 * 128
    bkv.bkv_cache_write(k, v, torch.zeros(5, dtype=torch.int64), _cache(dtype=torch.float32),
                        _cache(dtype=torch.float32), num_tokens=4)
    p = fake.ptrs
    assert fake.calls["bkv_cache_write"] == (p["k_new"], p["v_new"], 4, 3 * 8 * 128, p["slot_mapping"], p["k_cache"],
                                             p["v_cache"], 3, 16, 8, 128, bkv.BKV_F32, None, 999)


def test_cache_write_fp8_marshalling(fake):
    u8 = torch.uint8
    bkv.bkv_cache_write_fp8(_rows(), _rows(), torch.zeros(5, dtype=torch.int64), _cache(dtype=u8), _cache(dtype=u8),
                            0.5, 0.25)
    p = fake.ptrs
    assert fake.calls["bkv_cache_write_fp8"] == (p["k_new"], p["v_new"], 5, 8 * 128, p["slot_mapping"],
                                                 p["k_cache"], p["v_cache"], 3, 16, 8, 128, bkv.BKV_BF16, 0.5, 0.25,
                                                 None, 999)


@pytest.mark.parametrize("fp8", [False, True])
def test_fused_write_marshalling(fake, fp8):
    wide = torch.ones(4, 10, dtype=torch.int32)
    table = wide[:, 2:8]                                              # row stride 10, 6 columns
    req = torch.zeros(7, dtype=torch.int32)
    pos = torch.zeros(7, dtype=torch.int64)
    slots = torch.zeros(9, dtype=torch.int64)
    cdt = torch.uint8 if fp8 else torch.bfloat16
    if fp8:
        bkv.bkv_slot_mapping_cache_write_fp8(table, req, pos, slots, _rows(7), _rows(7), _cache(dtype=cdt),
                                             _cache(dtype=cdt), 2.0, 3.0, num_tokens=6)
        name, tail = "bkv_slot_mapping_cache_write_fp8", (2.0, 3.0, None, 999)
    else:
        bkv.bkv_slot_mapping_cache_write(table, req, pos, slots, _rows(7), _rows(7), _cache(dtype=cdt),
                                         _cache(dtype=cdt), num_tokens=6)
        name, tail = "bkv_slot_mapping_cache_write", (None, 999)
    p = fake.ptrs
    assert fake.calls[name] == (p["block_table"], 4, 10, 6, p["req_indices"], p["positions"], 6, 9, p["slot_mapping"],
                                p["k_new"], p["v_new"], 8 * 128, p["k_cache"], p["v_cache"], 3, 16, 8, 128,
                                bkv.BKV_BF16) + tail
    with pytest.raises(ValueError):                                    # more tokens than rows
        bkv.bkv_slot_mapping_cache_write(table, req, pos, slots, _rows(3), _rows(3), _cache(), _cache())
