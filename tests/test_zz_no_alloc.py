"""GPU test of bkv_paged_decode_noalloc, the decode entry point that allocates
nothing: its split-KV scratch is a fixed device array inside libbkv.so, for
callers that cannot call cudaMalloc (code running under a stream capture that
forbids allocation, plugins whose host owns all device memory, plain C callers
with no allocator).  Called through the C ABI, it must match
bkv_paged_decode run with a caller-owned workspace, on two calls in a row.
The file is named so that pytest collects it last; it passes when run alone
in a fresh process as well as after the rest of the suite."""
import ctypes
import os
import re

import pytest
import torch

from paged_kv_cache_slot_gb300 import bkv
from paged_kv_cache_slot_gb300 import workloads as wl
from paged_kv_cache_slot_gb300.staging import DeviceWorkload

pytestmark = pytest.mark.gpu

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "bkv.h")
TOL = 1e-2   # the decode tests' bf16 tolerance


def _scratch_bytes():
    m = re.search(r"#define BKV_NOALLOC_SCRATCH_BYTES \(\(size_t\)(\d+) << (\d+)\)", open(HEADER).read())
    return int(m.group(1)) << int(m.group(2))


def _entry():
    f = bkv.load().bkv_paged_decode_noalloc
    i32, i64, vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
    f.restype = ctypes.c_int
    f.argtypes = [vp, vp, vp, vp, i64, i32, vp, i32, i32, i32, i32, i32, i32, i32, i64, ctypes.c_float,
                  ctypes.c_int, ctypes.c_int, vp, vp, vp]
    return f


def _call(f, dw, out):
    q, kc, t = dw.q, dw.k_cache, dw.kernel_table
    nr, ql, hq, d = q.shape
    tb, bs, hkv, _ = kc.shape
    return f(q.data_ptr(), kc.data_ptr(), dw.v_cache.data_ptr(), t.data_ptr(), t.stride(0), t.shape[1],
             dw.context_lens.data_ptr(), dw.max_context_len, nr, ql, hq, hkv, d, bs, tb, 0.0, bkv.BKV_MASK_CAUSAL,
             bkv.BKV_BF16, out.data_ptr(), dw.err_count.data_ptr(), torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("name", ["llama3_decode", "long_context"])
def test_noalloc_matches_workspace_entry_point(name):
    w = wl.make(name)
    dw = DeviceWorkload(w)
    dw.write_step()
    dw.workspace.fill_(0xFF)                     # NaN: no unwritten partial may be read
    ref = dw.decode().clone()                    # bkv_paged_decode with a caller workspace
    torch.cuda.synchronize()
    need = bkv.bkv_paged_decode_workspace_size(w.num_rows, w.q_len, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                               w.kernel_block_size, dw.max_context_len)
    assert 0 < need <= _scratch_bytes()
    f = _entry()
    dw.err_count.zero_()
    for _ in range(2):                           # the array keeps the previous call's contents
        out = torch.full_like(ref, float("nan"))
        assert _call(f, dw, out) == bkv.BKV_OK
        torch.cuda.synchronize()
        assert torch.isfinite(out.float()).all()
        diff = (out.float() - ref.float()).abs().max().item()
        assert diff <= TOL, f"{name}: max abs difference {diff}"
    assert int(dw.err_count.item()) == 0


def test_noalloc_rejects_sizes_beyond_its_scratch():
    # hybrid-shaped batch: 320 rows, 4 query tokens, kernel blocks of 16, contexts to 8196
    need = bkv.bkv_paged_decode_workspace_size(320, 4, 32, 8, 128, 16, 8196)
    assert need > _scratch_bytes()
    f = _entry()
    rc = f(None, None, None, None, 514, 514, None, 8196, 320, 4, 32, 8, 128, 16, 40000, 0.0, 0, bkv.BKV_BF16, None,
           None, None)
    assert rc == bkv.BKV_ERR_UNSUPPORTED
