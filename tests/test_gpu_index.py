"""GPU parity for the integer work: slot mapping, block expansion and the cache
scatter, all bit-exact against the oracle on the same seeded inputs."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from oracle.cases import BF16_NAN
from paged_kv_cache_slot_gb300 import bkv
from paged_kv_cache_slot_gb300 import workloads as wl
from paged_kv_cache_slot_gb300.staging import DeviceWorkload

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "slot_examples.json")
DEV = "cuda"


def _d(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    return (t.view(dtype) if dtype is not None else t).to(DEV)


def _gpu_slots(table, req, pos, bs, num_tokens, max_num_tokens):
    out = torch.full((max_num_tokens,), 777, dtype=torch.int64, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    bkv.bkv_compute_slot_mapping(_d(table.astype(np.int32)), _d(req.astype(np.int32)), _d(pos.astype(np.int64)), bs,
                                 out, num_tokens=num_tokens, err_count=err)
    torch.cuda.synchronize()
    return out.cpu().numpy(), int(err.item())


def test_slot_mapping_page_examples():
    from test_oracle_index import _expand
    for case in json.load(open(GOLDEN))["cases"]:
        n, mx = case["num_tokens"], case["max_num_tokens"]
        req = np.array(_expand(case["req_indices"], n) + [-1] * (mx - n), np.int32)
        pos = np.array(_expand(case["positions"], n) + [0] * (mx - n), np.int64)
        got, err = _gpu_slots(np.array(case["block_table"], np.int32), req, pos, case["block_size"], n, mx)
        assert got.tolist() == _expand(case["slots"], mx), case["id"]
        assert err == 0


@pytest.mark.parametrize("name", wl.WORKLOADS)
def test_slot_mapping_workloads_bit_exact(name):
    w = wl.make(name)
    req, pos = w.step_tokens()
    want, werr = oracle.compute_slot_mapping(w.block_table, req, pos, w.block_size, w.num_tokens, w.max_num_tokens)
    got, gerr = _gpu_slots(w.block_table, req, pos, w.block_size, w.num_tokens, w.max_num_tokens)
    assert np.array_equal(got, want) and gerr == werr == 0
    # prior tokens too (every position of every request), in one launch
    preq, ppos = w.prior_tokens()
    if len(ppos):
        want, _ = oracle.compute_slot_mapping(w.block_table, preq, ppos, w.block_size)
        got, _ = _gpu_slots(w.block_table, preq, ppos, w.block_size, len(ppos), len(ppos))
        assert np.array_equal(got, want)


def test_slot_mapping_bad_inputs_and_err_count():
    rng = np.random.default_rng(99)
    nr, cols, bs, n, mx = 37, 11, 16, 50_000, 65_536
    table = rng.integers(-1, 5000, size=(nr, cols)).astype(np.int32)
    table[rng.random(table.shape) < 0.1] = 0
    req = rng.integers(-3, nr + 3, size=mx).astype(np.int32)
    pos = rng.integers(-20, cols * bs + 40, size=mx).astype(np.int64)
    want, werr = oracle.compute_slot_mapping(table, req, pos, bs, n, mx)
    got, gerr = _gpu_slots(table, req, pos, bs, n, mx)
    assert np.array_equal(got, want)
    assert gerr == werr > 0


def test_slot_mapping_strided_table_and_empty():
    rng = np.random.default_rng(4)
    wide = rng.integers(1, 900, size=(9, 20)).astype(np.int32)
    t = _d(wide)[:, 3:15]                                    # row stride 20, 12 columns
    req = rng.integers(0, 9, size=300).astype(np.int32)
    pos = rng.integers(0, 12 * 8, size=300).astype(np.int64)
    out = torch.empty(300, dtype=torch.int64, device=DEV)
    bkv.bkv_compute_slot_mapping(t, _d(req), _d(pos), 8, out)
    want, _ = oracle.compute_slot_mapping(wide[:, 3:15], req, pos, 8)
    assert np.array_equal(out.cpu().numpy(), want)
    # zero tokens but a padded buffer: all -1
    out2 = torch.zeros(1000, dtype=torch.int64, device=DEV)
    bkv.bkv_compute_slot_mapping(t, _d(req), _d(pos), 8, out2, num_tokens=0)
    assert (out2.cpu().numpy() == -1).all()


@pytest.mark.parametrize("bs,kbs", [(32, 16), (64, 16), (16, 16), (128, 8), (48, 16), (16, 1)])
def test_block_expansion_bit_exact(bs, kbs):
    rng = np.random.default_rng(bs * 7 + kbs)
    rows, cols = 41, 33
    mgr = rng.integers(-1, 1 << 20, size=(rows, cols)).astype(np.int32)
    mgr[rng.random(mgr.shape) < 0.15] = 0
    want = oracle.map_to_kernel_blocks(mgr, bs, kbs)
    bpk = bs // kbs
    kt = torch.full((rows, cols * bpk + 5), 12345, dtype=torch.int32, device=DEV)   # 5 spare columns
    bkv.bkv_map_to_kernel_blocks(_d(mgr), bs, kbs, kt)
    got = kt.cpu().numpy()
    assert np.array_equal(got[:, : cols * bpk], want)
    assert (got[:, cols * bpk:] == 12345).all()


@pytest.mark.parametrize("bpk", [2, 3, 16])
def test_block_expansion_at_the_int32_edge_bit_exact(bpk):
    top = (2**31 - 1 - (bpk - 1)) // bpk
    mgr = np.array([[top, top + 1, 2**31 - 1, 7, -1, 0], [1, top - 1, top, top + 1, 2**31 - 2, 5]], np.int32)
    want = oracle.map_to_kernel_blocks(mgr, 16 * bpk, 16)
    kt = torch.full(want.shape, 12345, dtype=torch.int32, device=DEV)
    bkv.bkv_map_to_kernel_blocks(_d(mgr), 16 * bpk, 16, kt)
    assert np.array_equal(kt.cpu().numpy(), want)


def test_block_expansion_hybrid_workload_and_error():
    w = wl.make("hybrid_spec")
    want = oracle.map_to_kernel_blocks(w.block_table, w.block_size, w.kernel_block_size)
    kt = torch.empty(want.shape, dtype=torch.int32, device=DEV)
    bkv.bkv_map_to_kernel_blocks(_d(w.block_table), w.block_size, w.kernel_block_size, kt)
    assert np.array_equal(kt.cpu().numpy(), want)
    with pytest.raises(bkv.BkvError) as ei:
        bkv.bkv_map_to_kernel_blocks(_d(w.block_table), 32, 12, kt)
    assert ei.value.status == bkv.BKV_ERR_INVALID_ARG


def _host_bits(t):
    x = t.cpu()
    return x.view(torch.int16).numpy() if x.dtype == torch.bfloat16 else x.view(torch.int32).numpy()


@pytest.mark.parametrize("fused", [False, True])
def test_cache_write_ragged_step_bit_exact(fused):
    w = wl.make("ragged_step")
    dw = DeviceWorkload(w, fill_prior=False)
    dw.write_step(fused=fused)
    torch.cuda.synchronize()
    req, pos = w.step_tokens()
    slots, _ = oracle.compute_slot_mapping(w.block_table, req, pos, w.block_size, w.num_tokens, w.max_num_tokens)
    assert np.array_equal(dw.slot_mapping.cpu().numpy(), slots)
    kn, vn = w.step_kv()
    shape = (w.total_blocks, w.block_size, w.num_kv_heads, w.head_dim)
    kc, vc, err = oracle.cache_write(kn, vn, slots, np.full(shape, BF16_NAN, np.uint16),
                                     np.full(shape, BF16_NAN, np.uint16), num_tokens=w.num_tokens, inplace=True)
    assert err == 0 and int(dw.err_count.item()) == 0
    assert np.array_equal(_host_bits(dw.k_cache), kc.view(np.int16))
    assert np.array_equal(_host_bits(dw.v_cache), vc.view(np.int16))


def test_prior_fill_and_step_match_oracle_cache():
    from oracle.cases import fill_oracle_cache
    w = wl.make("llama3_decode")
    dw = DeviceWorkload(w)
    dw.write_step()
    torch.cuda.synchronize()
    kc, vc, _ = fill_oracle_cache(w)
    assert np.array_equal(_host_bits(dw.k_cache), kc.view(np.int16))
    assert np.array_equal(_host_bits(dw.v_cache), vc.view(np.int16))
    assert int(dw.err_count.item()) == 0


@pytest.mark.parametrize("dtype,H,D,stride_extra", [("bf16", 8, 128, 0), ("bf16", 8, 128, 1024), ("f32", 2, 64, 4),
                                                    ("bf16", 1, 6, 0), ("bf16", 3, 10, 2), ("f32", 1, 3, 1)])
def test_cache_write_paths_strides_and_out_of_range(dtype, H, D, stride_extra):
    rng = np.random.default_rng(H * 100 + D + stride_extra)
    tb, bs, n = 23, 8, 150
    row = H * D
    npdt, tdt = (np.uint16, torch.bfloat16) if dtype == "bf16" else (np.float32, torch.float32)
    bg = (rng.integers(0, 1 << 16, size=(tb, bs, H, D)).astype(np.uint16) if dtype == "bf16"
          else rng.standard_normal((tb, bs, H, D)).astype(np.float32))
    fused = (rng.integers(0, 1 << 16, size=(n, 2 * (row + stride_extra))).astype(np.uint16) if dtype == "bf16"
             else rng.standard_normal((n, 2 * (row + stride_extra))).astype(np.float32))
    slots = rng.permutation(tb * bs + 40)[:n].astype(np.int64) - 20     # some < 0, some past the cache
    slots[::7] = -1
    kn_h = np.ascontiguousarray(fused[:, :row]).reshape(n, H, D)
    vn_h = np.ascontiguousarray(fused[:, row + stride_extra: 2 * row + stride_extra]).reshape(n, H, D)
    kc_w, vc_w, werr = oracle.cache_write(kn_h, vn_h, np.where(slots < -1, -1, slots), bg, bg[::-1].copy())
    f = _d(fused, tdt if dtype == "bf16" else None)
    kn = f[:, :row].unflatten(1, (H, D))
    vn = f[:, row + stride_extra: 2 * row + stride_extra].unflatten(1, (H, D))
    kc = _d(bg, tdt if dtype == "bf16" else None)
    vc = _d(bg[::-1].copy(), tdt if dtype == "bf16" else None)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    bkv.bkv_cache_write(kn, vn, _d(slots), kc, vc, err_count=err)
    torch.cuda.synchronize()
    view = np.int16 if dtype == "bf16" else np.int32
    assert np.array_equal(_host_bits(kc), kc_w.view(view))
    assert np.array_equal(_host_bits(vc), vc_w.view(view))
    assert int(err.item()) == werr > 0
