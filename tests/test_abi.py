"""CPU checks of the C ABI: libbkv.so builds, loads, exports every entry point
include/bkv.h declares, and rejects bad arguments on the host (before any
CUDA call) with the documented status codes."""
import os
import re

import pytest

from paged_kv_cache_slot_gb300 import bkv
from paged_kv_cache_slot_gb300 import build as bkv_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include")))
           if f.endswith(".h")]


@pytest.fixture(scope="module")
def lib():
    bkv_build.build()
    return bkv.load()


def _declared():
    names = set()
    for h in HEADERS:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b(bkv_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ("bkv_compute_slot_mapping", "bkv_map_to_kernel_blocks", "bkv_cache_write", "bkv_paged_decode",
              "bkv_paged_decode_workspace_size", "bkv_slot_mapping_cache_write", "bkv_slot_mapping_cache_write_fp8"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(lib):
    assert lib.bkv_status_string(0) == b"ok"
    assert b"invalid" in lib.bkv_status_string(1)
    assert lib.bkv_version().startswith(b"bkv ")


def test_package_version_is_the_library_version(lib):
    import paged_kv_cache_slot_gb300 as pkg
    assert lib.bkv_version().split()[1].decode() == pkg.__version__


NULL = None


def test_slot_mapping_rejects_bad_arguments(lib):
    f = lib.bkv_compute_slot_mapping
    # block_size <= 0
    assert f(NULL, 1, 4, 4, NULL, NULL, 1, 1, 0, NULL, NULL, NULL) == bkv.BKV_ERR_INVALID_ARG
    # max_num_tokens < num_tokens
    assert f(NULL, 1, 4, 4, NULL, NULL, 5, 4, 16, NULL, NULL, NULL) == bkv.BKV_ERR_INVALID_ARG
    # bt_stride < bt_cols
    assert f(NULL, 1, 2, 4, NULL, NULL, 1, 1, 16, NULL, NULL, NULL) == bkv.BKV_ERR_INVALID_ARG
    # null output / inputs
    assert f(NULL, 1, 4, 4, NULL, NULL, 1, 1, 16, NULL, NULL, NULL) == bkv.BKV_ERR_INVALID_ARG
    # nothing to do is fine and launches nothing
    assert f(NULL, 0, 0, 0, NULL, NULL, 0, 0, 16, NULL, NULL, NULL) == bkv.BKV_OK


def test_block_expansion_rejects_indivisible(lib):
    f = lib.bkv_map_to_kernel_blocks
    assert f(NULL, 2, 4, 4, 32, 12, NULL, 16, NULL) == bkv.BKV_ERR_INVALID_ARG
    assert f(NULL, 2, 4, 4, 32, 0, NULL, 16, NULL) == bkv.BKV_ERR_INVALID_ARG
    assert f(NULL, 2, 4, 4, 32, 16, NULL, 7, NULL) == bkv.BKV_ERR_INVALID_ARG   # kernel_stride < 4 * 2
    assert f(NULL, 0, 4, 4, 32, 16, NULL, 8, NULL) == bkv.BKV_OK                 # empty


def test_cache_write_rejects_bad_arguments(lib):
    f = lib.bkv_cache_write
    assert f(NULL, NULL, 1, 1024, NULL, NULL, NULL, 4, 16, 8, 128, 7, NULL, NULL) == bkv.BKV_ERR_UNSUPPORTED
    assert f(NULL, NULL, 1, 1023, NULL, NULL, NULL, 4, 16, 8, 128, 0, NULL, NULL) == bkv.BKV_ERR_INVALID_ARG
    assert f(NULL, NULL, 1, 1024, NULL, NULL, NULL, 4, 0, 8, 128, 0, NULL, NULL) == bkv.BKV_ERR_INVALID_ARG
    assert f(NULL, NULL, 1, 1024, NULL, NULL, NULL, 4, 16, 8, 128, 0, NULL, NULL) == bkv.BKV_ERR_INVALID_ARG
    assert f(NULL, NULL, 0, 1024, NULL, NULL, NULL, 4, 16, 8, 128, 0, NULL, NULL) == bkv.BKV_OK


def test_fused_slot_write_rejects_bad_arguments(lib):
    f = lib.bkv_slot_mapping_cache_write

    def call(**kw):
        a = dict(bt=NULL, nr=1, st=4, cols=4, req=NULL, pos=NULL, n=1, mx=1, slots=NULL, kn=NULL, vn=NULL, sst=1024,
                 kc=NULL, vc=NULL, tb=4, bs=16, h=8, d=128, dt=0)
        a.update(kw)
        return f(*a.values(), NULL, NULL)

    assert call(dt=7) == bkv.BKV_ERR_UNSUPPORTED
    assert call(bs=0) == bkv.BKV_ERR_INVALID_ARG
    assert call(n=5, mx=4) == bkv.BKV_ERR_INVALID_ARG          # max_num_tokens < num_tokens
    assert call(st=2) == bkv.BKV_ERR_INVALID_ARG               # bt_stride < bt_cols
    assert call(sst=1023) == bkv.BKV_ERR_INVALID_ARG           # source stride < H_kv * D
    assert call(h=0) == bkv.BKV_ERR_INVALID_ARG
    assert call() == bkv.BKV_ERR_INVALID_ARG                   # null pointers
    assert call(n=0, mx=0) == bkv.BKV_OK                       # nothing to do launches nothing


def test_fused_slot_write_fp8_rejects_bad_arguments(lib):
    f = lib.bkv_slot_mapping_cache_write_fp8

    def call(**kw):
        a = dict(bt=NULL, nr=1, st=4, cols=4, req=NULL, pos=NULL, n=1, mx=1, slots=NULL, kn=NULL, vn=NULL, sst=1024,
                 kc=NULL, vc=NULL, tb=4, bs=16, h=8, d=128, dt=0, ks=1.0, vs=1.0)
        a.update(kw)
        return f(*a.values(), NULL, NULL)

    assert call(dt=7) == bkv.BKV_ERR_UNSUPPORTED
    assert call(ks=0.0) == bkv.BKV_ERR_INVALID_ARG                  # scales must be positive and finite
    assert call(vs=float("inf")) == bkv.BKV_ERR_INVALID_ARG
    assert call(n=5, mx=4) == bkv.BKV_ERR_INVALID_ARG
    assert call(sst=1023) == bkv.BKV_ERR_INVALID_ARG
    assert call() == bkv.BKV_ERR_INVALID_ARG
    assert call(n=0, mx=0) == bkv.BKV_OK


@pytest.mark.parametrize("fn", ["bkv_paged_decode", "bkv_paged_decode_swa", "bkv_paged_decode_partition",
                                "bkv_paged_decode_merge"])
def test_paged_decode_rejects_bad_arguments(lib, fn):
    f = getattr(lib, fn)
    windowed = fn != "bkv_paged_decode"      # the survey's signature has no window argument
    base = dict(q=NULL, k=NULL, v=NULL, bt=NULL, bt_stride=4, bt_cols=4, ctx=NULL, max_ctx=16, num_reqs=2, q_len=1,
                hq=32, hkv=8, d=128, bs=16, tb=8, scale=0.0, mask=0, window=0, dtype=0, out=NULL, ws=NULL, wsb=0,
                err=NULL, stream=NULL)
    if not windowed:
        del base["window"]

    def call(**kw):
        a = dict(base, **kw)
        return f(*a.values())

    assert call(dtype=5) == bkv.BKV_ERR_UNSUPPORTED
    assert call(d=512) == bkv.BKV_ERR_UNSUPPORTED
    assert call(mask=2) == bkv.BKV_ERR_INVALID_ARG
    if windowed:
        assert call(window=-1) == bkv.BKV_ERR_INVALID_ARG
    assert call(bt_stride=2) == bkv.BKV_ERR_INVALID_ARG
    assert call(hq=30) == bkv.BKV_ERR_INVALID_ARG          # 30 % 8 != 0
    assert call(num_reqs=0) == bkv.BKV_ERR_INVALID_ARG
    assert call() == bkv.BKV_ERR_INVALID_ARG                # null pointers / no workspace


def test_paged_decode_has_the_survey_signature():
    """bkv_paged_decode is declared with exactly the argument list of the boundary's statement (no
    window: the sliding-window form is bkv_paged_decode_swa)."""
    text = re.sub(r"/\*.*?\*/", "", open(os.path.join(ROOT, "include", "bkv.h")).read(), flags=re.S)
    decl = re.search(r"int bkv_paged_decode\((.*?)\);", text, flags=re.S).group(1)
    names = [a.strip().split()[-1].lstrip("*") for a in decl.split(",")]
    assert names == ["q", "k_cache", "v_cache", "block_table", "bt_stride", "bt_cols", "context_lens",
                     "max_context_len", "num_reqs", "q_len", "num_q_heads", "num_kv_heads", "head_dim",
                     "block_size", "total_blocks", "softmax_scale", "mask_mode", "dtype", "out", "workspace",
                     "workspace_bytes", "err_count", "stream"]


def test_workspace_size_is_zero_for_invalid_sizes(lib):
    assert lib.bkv_paged_decode_workspace_size(2, 1, 30, 8, 128, 16, 100) == 0
    assert lib.bkv_paged_decode_workspace_size(0, 1, 32, 8, 128, 16, 100) == 0


def test_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    monkeypatch.setattr(bkv, "_lib", None)
    monkeypatch.setattr(bkv, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no fallback"):
        bkv.load()


def test_fp8_entry_points_reject_bad_arguments(lib):
    w = lib.bkv_cache_write_fp8
    # src_dtype, scale <= 0, scale inf / nan, stride too small, null pointers, empty
    assert w(NULL, NULL, 1, 1024, NULL, NULL, NULL, 4, 16, 8, 128, 7, 1.0, 1.0, NULL, NULL) == bkv.BKV_ERR_UNSUPPORTED
    assert w(NULL, NULL, 1, 1024, NULL, NULL, NULL, 4, 16, 8, 128, 0, 0.0, 1.0, NULL, NULL) == bkv.BKV_ERR_INVALID_ARG
    assert w(NULL, NULL, 1, 1024, NULL, NULL, NULL, 4, 16, 8, 128, 0, 1.0, float("inf"), NULL, NULL) == \
        bkv.BKV_ERR_INVALID_ARG
    assert w(NULL, NULL, 1, 1024, NULL, NULL, NULL, 4, 16, 8, 128, 0, float("nan"), 1.0, NULL, NULL) == \
        bkv.BKV_ERR_INVALID_ARG
    assert w(NULL, NULL, 1, 1023, NULL, NULL, NULL, 4, 16, 8, 128, 0, 1.0, 1.0, NULL, NULL) == bkv.BKV_ERR_INVALID_ARG
    assert w(NULL, NULL, 1, 1024, NULL, NULL, NULL, 4, 16, 8, 128, 0, 1.0, 1.0, NULL, NULL) == bkv.BKV_ERR_INVALID_ARG
    assert w(NULL, NULL, 0, 1024, NULL, NULL, NULL, 4, 16, 8, 128, 0, 1.0, 1.0, NULL, NULL) == bkv.BKV_OK
    base = dict(q=NULL, k=NULL, v=NULL, bt=NULL, bt_stride=4, bt_cols=4, ctx=NULL, max_ctx=16, num_reqs=2, q_len=1,
                hq=32, hkv=8, d=128, bs=16, tb=8, scale=0.0, ks=1.0, vs=1.0, mask=0, window=0, dtype=0, out=NULL,
                ws=NULL, wsb=0, err=NULL, stream=NULL)
    for fn in ("bkv_paged_decode_fp8", "bkv_paged_decode_fp8_partition", "bkv_paged_decode_fp8_merge"):
        f = getattr(lib, fn)

        def call(**kw):
            a = dict(base, **kw)
            return f(*a.values())

        assert call(dtype=5) == bkv.BKV_ERR_UNSUPPORTED
        assert call(d=512) == bkv.BKV_ERR_UNSUPPORTED
        assert call(ks=0.0) == bkv.BKV_ERR_INVALID_ARG
        assert call(vs=-1.0) == bkv.BKV_ERR_INVALID_ARG
        assert call(vs=float("inf")) == bkv.BKV_ERR_INVALID_ARG
        assert call(mask=2) == bkv.BKV_ERR_INVALID_ARG
        assert call(hq=30) == bkv.BKV_ERR_INVALID_ARG
        assert call() == bkv.BKV_ERR_INVALID_ARG            # null pointers / no workspace
