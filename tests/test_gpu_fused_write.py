"""GPU parity of bkv_slot_mapping_cache_write (slot mapping and the cache
scatter in one kernel): the slot array, both caches and the error count are
bit-exact against the oracle's slot mapping followed by its cache write, and
equal to the library's own two-call sequence."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_slot_gb300 import bkv
from paged_kv_cache_slot_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _d(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    return (t.view(dtype) if dtype is not None else t).to(DEV)


def _bits(t):
    x = t.cpu()
    return x.view(torch.int16).numpy() if x.dtype == torch.bfloat16 else x.view(torch.int32).numpy()


def _oracle(table, req, pos, bs, n, mx, kn, vn, kc, vc):
    slots, serr = oracle.compute_slot_mapping(table, req, pos, bs, n, mx)
    kc_w, vc_w, werr = oracle.cache_write(kn, vn, slots, kc, vc, num_tokens=n)
    return slots, kc_w, vc_w, serr + werr


def _run_fused(table_t, req, pos, n, mx, kn_t, vn_t, kc_t, vc_t):
    slots = torch.full((mx,), 777, dtype=torch.int64, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    bkv.bkv_slot_mapping_cache_write(table_t, _d(req.astype(np.int32)), _d(pos.astype(np.int64)), slots, kn_t, vn_t,
                                     kc_t, vc_t, num_tokens=n, err_count=err)
    torch.cuda.synchronize()
    return slots.cpu().numpy(), int(err.item())


SMALL = ("tiny", "llama3_decode", "ragged_step")


@pytest.mark.parametrize("name", SMALL)
def test_fused_write_workloads_bit_exact(name):
    """Seeded workloads whose caches fit a whole-cache comparison: the step's tokens (padded tail
    included) against the oracle, every byte of both caches compared."""
    w = wl.make(name)
    req, pos = w.step_tokens()
    kn, vn = w.step_kv()
    shape = (w.total_blocks, w.block_size, w.num_kv_heads, w.head_dim)
    rng = np.random.default_rng(3)
    if w.dtype == "bf16":
        bg = rng.integers(0, 1 << 16, size=shape).astype(np.uint16)
        tdt = torch.bfloat16
    else:
        bg = rng.standard_normal(shape).astype(np.float32)
        tdt = None
    want_s, want_k, want_v, want_e = _oracle(w.block_table, req, pos, w.block_size, w.num_tokens, w.max_num_tokens,
                                             kn, vn, bg, bg[::-1].copy())
    kc, vc = _d(bg, tdt), _d(bg[::-1].copy(), tdt)
    got_s, got_e = _run_fused(_d(w.block_table), req, pos, w.num_tokens, w.max_num_tokens, _d(kn, tdt), _d(vn, tdt),
                              kc, vc)
    view = np.int16 if w.dtype == "bf16" else np.int32
    assert np.array_equal(got_s, want_s)
    assert got_e == want_e == 0
    assert np.array_equal(_bits(kc), want_k.view(view))
    assert np.array_equal(_bits(vc), want_v.view(view))


@pytest.mark.parametrize("name", [n for n in wl.WORKLOADS if n not in SMALL])
def test_fused_write_large_workloads(name):
    """The long-context and hybrid workloads (caches of GBs, the hybrid one in its manager view of
    32-token blocks): the slot array bit-exact against the oracle; the rows at the oracle's slots
    hold the new rows' bits and every other row still holds the NaN background."""
    w = wl.make(name)
    req, pos = w.step_tokens()
    kn, vn = w.step_kv()
    want_s, want_e = oracle.compute_slot_mapping(w.block_table, req, pos, w.block_size, w.num_tokens,
                                                 w.max_num_tokens)
    shape = (w.total_blocks, w.block_size, w.num_kv_heads, w.head_dim)
    kc = torch.full(shape, float("nan"), dtype=torch.bfloat16, device=DEV)
    vc = torch.full(shape, float("nan"), dtype=torch.bfloat16, device=DEV)
    got_s, got_e = _run_fused(_d(w.block_table), req, pos, w.num_tokens, w.max_num_tokens,
                              _d(kn, torch.bfloat16), _d(vn, torch.bfloat16), kc, vc)
    assert np.array_equal(got_s, want_s) and got_e == want_e == 0
    real = np.nonzero(want_s[: w.num_tokens] >= 0)[0]
    rows = torch.from_numpy(want_s[real]).to(DEV)
    for cache, new in ((kc, kn), (vc, vn)):
        flat = cache.view(-1, w.num_kv_heads * w.head_dim).view(torch.int16)
        assert torch.equal(flat[rows].cpu(), torch.from_numpy(new[real].reshape(len(real), -1).view(np.int16)))
        untouched = torch.ones(flat.shape[0], dtype=torch.bool, device=DEV)
        untouched[rows] = False
        assert torch.isnan(cache.view(-1, w.num_kv_heads * w.head_dim)[untouched]).all()


def _bad_case(seed, H, D, dtype, stride_extra):
    """A table of distinct ids (some null, some -1, some past the cache) and tokens with distinct
    (request, position) pairs plus bad request indices, negative positions and positions past the
    table width; valid slots are therefore distinct, as the cache write requires."""
    rng = np.random.default_rng(seed)
    nr, cols, bs, tb = 13, 6, 8, 60
    ids = rng.permutation(np.arange(1, tb + 25))[: nr * cols].astype(np.int32)   # some ids >= tb
    table = ids.reshape(nr, cols)
    table[rng.random(table.shape) < 0.1] = 0
    table[rng.random(table.shape) < 0.1] = -1
    pairs = rng.permutation(nr * cols * bs)[:300]
    req = (pairs // (cols * bs)).astype(np.int32)
    pos = (pairs % (cols * bs)).astype(np.int64)
    k = len(req)
    req[rng.random(k) < 0.05] = -1                                  # padded requests
    bad_r = rng.random(k) < 0.03
    req[bad_r] = nr + rng.integers(0, 3, size=int(bad_r.sum()))     # past the batch
    neg = rng.random(k) < 0.03
    pos[neg] = -1 - rng.integers(0, 5, size=int(neg.sum()))
    wide = rng.random(k) < 0.03
    pos[wide] = cols * bs + rng.integers(0, 40, size=int(wide.sum()))   # past the table width
    n, mx = 280, 320                                                # 20 token rows unused, 40 tail slots
    row = H * D
    npdt, tdt = (np.uint16, torch.bfloat16) if dtype == "bf16" else (np.float32, None)
    if dtype == "bf16":
        fused = rng.integers(0, 1 << 16, size=(k, 2 * (row + stride_extra))).astype(np.uint16)
        bg = rng.integers(0, 1 << 16, size=(tb, bs, H, D)).astype(np.uint16)
    else:
        fused = rng.standard_normal((k, 2 * (row + stride_extra))).astype(np.float32)
        bg = rng.standard_normal((tb, bs, H, D)).astype(np.float32)
    return table, req, pos, bs, n, mx, fused, bg, row, tdt


@pytest.mark.parametrize("dtype,H,D,stride_extra", [("bf16", 8, 128, 0), ("bf16", 8, 128, 1024), ("f32", 2, 64, 4),
                                                    ("bf16", 16, 256, 0), ("bf16", 1, 6, 0), ("bf16", 3, 10, 2),
                                                    ("f32", 1, 3, 1)])
def test_fused_write_bad_inputs_paths_and_strides(dtype, H, D, stride_extra):
    """The 16-byte path (rows of 2 KiB, 8 KiB, strided sources) and the element path, with every kind
    of padding and bad data: slots, caches and the error count equal the oracle's."""
    table, req, pos, bs, n, mx, fused, bg, row, tdt = _bad_case(H * 31 + D + stride_extra, H, D, dtype,
                                                                stride_extra)
    kn_h = np.ascontiguousarray(fused[:, :row]).reshape(-1, H, D)
    vn_h = np.ascontiguousarray(fused[:, row + stride_extra: 2 * row + stride_extra]).reshape(-1, H, D)
    want_s, want_k, want_v, want_e = _oracle(table, req, pos, bs, n, mx, kn_h, vn_h, bg, bg[::-1].copy())
    f = _d(fused, tdt)
    kn = f[:, :row].unflatten(1, (H, D))
    vn = f[:, row + stride_extra: 2 * row + stride_extra].unflatten(1, (H, D))
    kc, vc = _d(bg, tdt), _d(bg[::-1].copy(), tdt)
    got_s, got_e = _run_fused(_d(table), req, pos, n, mx, kn, vn, kc, vc)
    view = np.int16 if dtype == "bf16" else np.int32
    assert np.array_equal(got_s, want_s)
    assert got_e == want_e > 0
    assert np.array_equal(_bits(kc), want_k.view(view))
    assert np.array_equal(_bits(vc), want_v.view(view))


def test_fused_write_equals_the_two_calls():
    """Bitwise equal to bkv_compute_slot_mapping + bkv_cache_write on the same inputs, error count
    included, for a strided table view."""
    table, req, pos, bs, n, mx, fused, bg, row, tdt = _bad_case(11, 8, 128, "bf16", 0)
    wide = np.zeros((table.shape[0], table.shape[1] + 5), np.int32)
    wide[:, 2:2 + table.shape[1]] = table
    t = _d(wide)[:, 2:2 + table.shape[1]]
    f = _d(fused, tdt)
    kn, vn = f[:, :row].unflatten(1, (8, 128)), f[:, row:].unflatten(1, (8, 128))
    kc1, vc1 = _d(bg, tdt), _d(bg[::-1].copy(), tdt)
    kc2, vc2 = kc1.clone(), vc1.clone()
    s1, e1 = _run_fused(t, req, pos, n, mx, kn, vn, kc1, vc1)
    s2 = torch.full((mx,), 777, dtype=torch.int64, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    bkv.bkv_compute_slot_mapping(t, _d(req), _d(pos), bs, s2, num_tokens=n, err_count=err)
    bkv.bkv_cache_write(kn, vn, s2, kc2, vc2, num_tokens=n, err_count=err)
    torch.cuda.synchronize()
    assert np.array_equal(s1, s2.cpu().numpy()) and e1 == int(err.item()) > 0
    assert torch.equal(kc1.view(torch.int16), kc2.view(torch.int16))
    assert torch.equal(vc1.view(torch.int16), vc2.view(torch.int16))


def test_fused_write_no_tokens_fills_the_tail():
    """num_tokens = 0: the whole slot buffer becomes -1 and the caches are untouched."""
    bg = np.arange(4 * 8 * 2 * 16, dtype=np.float32).reshape(4, 8, 2, 16)
    kc, vc = _d(bg), _d(bg + 1)
    kn = torch.zeros((3, 2, 16), dtype=torch.float32, device=DEV)
    got_s, got_e = _run_fused(_d(np.ones((2, 4), np.int32)), np.zeros(3, np.int32), np.zeros(3, np.int64), 0, 50,
                              kn, kn.clone(), kc, vc)
    assert (got_s == -1).all() and got_e == 0
    assert np.array_equal(kc.cpu().numpy(), bg) and np.array_equal(vc.cpu().numpy(), bg + 1)
