"""GPU test of bkv_paged_decode_noalloc, the decode entry point that allocates
nothing: its split-KV scratch is a fixed device array inside libbkv.so, for
callers that cannot call cudaMalloc (code running under a stream capture that
forbids allocation, plugins whose host owns all device memory, plain C callers
with no allocator).

Called through the C ABI, it must give exactly the bits of bkv_paged_decode
run with a caller-owned workspace: the plan, the kernels and the partial-slot
layout depend only on the shape, not on where the scratch lives or how large
it is, and the stream-K merge is deterministic.  Each checked call follows a
call on a DIFFERENT workload, so the shared array holds unrelated partials
when it starts (a kernel reading a slot it did not write in this call would
show).  Covered: the tensor-core kernel (bf16, head_dim 128) on two
full-size workloads and the CUDA-core kernel (fp32, another layout of the
scratch).  The file is named so that pytest collects it last; it passes when
run alone in a fresh process as well as after the rest of the suite."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import oracle
from _parity import check_attention
from oracle.cases import fill_oracle_cache
from paged_kv_cache_slot_gb300 import bkv
from paged_kv_cache_slot_gb300 import workloads as wl
from paged_kv_cache_slot_gb300.staging import DeviceWorkload

pytestmark = pytest.mark.gpu

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "bkv.h")


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
    dt = bkv.BKV_BF16 if q.dtype == torch.bfloat16 else bkv.BKV_F32
    return f(q.data_ptr(), kc.data_ptr(), dw.v_cache.data_ptr(), t.data_ptr(), t.stride(0), t.shape[1],
             dw.context_lens.data_ptr(), dw.max_context_len, nr, ql, hq, hkv, d, bs, tb, 0.0, bkv.BKV_MASK_CAUSAL,
             dt, out.data_ptr(), dw.err_count.data_ptr(), torch.cuda.current_stream().cuda_stream)


def _fp32_small():
    """A CUDA-core (fp32, head_dim 32) batch: 3 requests, 2 query tokens, several partitions each."""
    prior = np.array([700, 3, 1500], np.int64)
    new = np.full(3, 2, np.int64)
    bs = 16
    need = -(-(prior + new) // bs)
    rng = np.random.default_rng(91)
    total = 1 + int(need.sum()) + 5
    ids = rng.permutation(np.arange(1, total))[: int(need.sum())]
    table = np.full((3, int(need.max()) + 1), -1, np.int32)
    k = 0
    for r, n in enumerate(need):
        table[r, :n] = ids[k:k + n]
        k += int(n)
    return wl.Workload("noalloc_f32", 91, "f32", 3, 3, 2, 8, 2, 32, bs, bs, prior, new, table, total,
                       max_num_tokens=8, qk_scale=1.0, v_scale=1.0)


def _staged(name):
    w = _fp32_small() if name == "fp32_small" else wl.make(name, loud=True)
    dw = DeviceWorkload(w)
    dw.write_step()
    torch.cuda.synchronize()
    return dw


# each checked workload, and the different one whose call leaves its partials in the array first
CASES = [("llama3_decode", "long_context"), ("long_context", "llama3_decode"), ("fp32_small", "llama3_decode")]


@pytest.mark.parametrize("name,other", CASES)
def test_noalloc_matches_workspace_entry_point_bitwise(name, other):
    dw = _staged(name)
    ow = _staged(other)
    w = dw.w
    dw.workspace.fill_(0xFF)                     # NaN: no unwritten partial may be read
    ref = dw.decode().clone()                    # bkv_paged_decode with a caller workspace
    torch.cuda.synchronize()
    need = bkv.bkv_paged_decode_workspace_size(w.num_rows, w.q_len, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                               w.kernel_block_size, dw.max_context_len)
    assert 0 < need <= _scratch_bytes()
    f = _entry()
    dw.err_count.zero_()
    for _ in range(2):                           # two calls in a row, each after an unrelated one
        junk = torch.empty_like(ow.out)
        assert _call(f, ow, junk) == bkv.BKV_OK
        out = torch.full_like(ref, float("nan"))
        assert _call(f, dw, out) == bkv.BKV_OK
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.uint8), ref.view(torch.uint8)), f"{name}: differs from bkv_paged_decode"
    assert int(dw.err_count.item()) == 0
    assert int(ow.err_count.item()) == 0


def test_noalloc_matches_the_oracle():
    dw = _staged("llama3_decode")
    w = dw.w
    out = torch.full_like(dw.out, float("nan"))
    assert _call(_entry(), dw, out) == bkv.BKV_OK
    torch.cuda.synchronize()
    kc, vc, table = fill_oracle_cache(w)
    want, err = oracle.paged_decode(w.q(), kc, vc, table, w.context_lens)
    assert err == 0
    check_attention(out.float().cpu().numpy(), want, "bf16", "noalloc llama3_decode", min_magnitude=0.1)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    # hybrid-shaped batch: 320 rows, 4 query tokens, kernel blocks of 16, contexts to 8196
    need = bkv.bkv_paged_decode_workspace_size(320, 4, 32, 8, 128, 16, 8196)
    assert need > _scratch_bytes()
    f = _entry()
    rc = f(None, None, None, None, 514, 514, None, 8196, 320, 4, 32, 8, 128, 16, 40000, 0.0, 0, bkv.BKV_BF16, None,
           None, None)
    assert rc == bkv.BKV_ERR_UNSUPPORTED
