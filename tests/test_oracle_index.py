"""Pins for the oracle's integer work: slot mapping, block expansion, cache write.

Each test ties the oracle to something other than itself: values printed on
the pages (tests/golden/slot_examples.json), a brute-force enumeration,
closed forms and invariants.
"""
import json
import os

import numpy as np
import pytest

import oracle
from paged_kv_cache_slot_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "slot_examples.json")


def _expand(spec, n):
    """Parse the fixture's shorthand: a list, 'v x n' or 'a..b' ranges joined by commas."""
    if isinstance(spec, list):
        return spec
    out = []
    for part in spec.replace("then", "").split(","):
        part = part.strip()
        if " x " in part:
            v, k = part.split(" x ")
            out += [int(v)] * int(k)
        elif ".." in part:
            a, b = part.split("..")
            out += list(range(int(a), int(b) + 1))
        else:
            out.append(int(part))
    return out


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


@pytest.mark.parametrize("case", _golden()["cases"], ids=lambda c: c["id"])
def test_slot_mapping_matches_page_examples(case):
    n, mx = case["num_tokens"], case["max_num_tokens"]
    req = _expand(case["req_indices"], n)
    pos = _expand(case["positions"], n)
    want = _expand(case["slots"], mx)
    req = np.array(req + [-1] * (mx - n), np.int32)
    pos = np.array(pos + [0] * (mx - n), np.int64)
    got, err = oracle.compute_slot_mapping(case["block_table"], req, pos, case["block_size"], n, mx)
    assert err == 0
    assert got.tolist() == want


def _brute_slots(table, bs, r):
    """All slots of row r in logical order, built by enumeration (no division)."""
    out = []
    for b in table[r]:
        for o in range(bs):
            out.append(int(b) * bs + o if b > 0 else -1)
    return out


def test_decode_batch_padding_page_example():
    g = _golden()["decode_batch_padding"]
    bs = 64
    table = np.array([[10, 15, -1], [8, 12, -1]] + [[-1, -1, -1]] * (g["bucket"] - 2), np.int32)
    pos = np.array([50, 75] + [g["pad_positions"]] * (g["bucket"] - g["active"]), np.int64)
    enum = [_brute_slots(table, bs, r) for r in range(2)]
    # padding marked by the token count (tail) ...
    req = np.array([0, 1] + [-1] * (g["bucket"] - 2), np.int32)
    got, err = oracle.compute_slot_mapping(table, req, pos, bs, num_tokens=g["active"], max_num_tokens=g["bucket"])
    assert got.tolist() == [enum[0][50], enum[1][75]] + [g["pad_slot"]] * 6 and err == 0
    # ... or by a negative request index, with all tokens counted
    got2, err2 = oracle.compute_slot_mapping(table, req, pos, bs, num_tokens=g["bucket"], max_num_tokens=g["bucket"])
    assert got2.tolist() == got.tolist() and err2 == 0
    # ... or a dummy pointing at a padded (all -1) table row
    req3 = np.array([0, 1] + list(range(2, g["bucket"])), np.int32)
    got3, _ = oracle.compute_slot_mapping(table, req3, pos, bs)
    assert got3.tolist() == got.tolist()


def test_dummy_on_valid_row_gets_a_real_slot_unless_marked():
    # The pages' dummies point at valid rows and only the later overwrite makes
    # their slot -1; the oracle gives such a token a real slot (reading R3).
    table = np.array([[10, 15]], np.int32)
    got, _ = oracle.compute_slot_mapping(table, np.array([0, 0], np.int32), np.array([5, 0], np.int64), 64)
    assert got.tolist() == [645, 640]


def test_null_block_and_sentinel_give_minus_one():
    table = np.array([[0, -1, 7]], np.int32)
    got, err = oracle.compute_slot_mapping(table, np.zeros(3, np.int32), np.array([1, 5, 9], np.int64), 4)
    assert got.tolist() == [-1, -1, 7 * 4 + 1] and err == 0


def test_out_of_range_inputs_are_minus_one_and_counted():
    table = np.array([[3, 4]], np.int32)
    req = np.array([0, 1, 0, 0], np.int32)
    pos = np.array([8, 0, -1, 7], np.int64)  # past width, bad request, negative position, ok
    got, err = oracle.compute_slot_mapping(table, req, pos, 4)
    assert got.tolist() == [-1, -1, -1, 4 * 4 + 3] and err == 3


@pytest.mark.parametrize("name", ["tiny", "llama3_decode", "ragged_step", "hybrid_spec"])
def test_slot_mapping_brute_force_and_invariants(name):
    w = wl.make(name)
    req, pos = w.step_tokens()
    got, err = oracle.compute_slot_mapping(w.block_table, req, pos, w.block_size, w.num_tokens, w.max_num_tokens)
    assert err == 0
    valid = req[: w.num_tokens] >= 0
    for i in np.nonzero(valid)[0][:400]:
        r, p = int(req[i]), int(pos[i])
        assert got[i] == _brute_slots(w.block_table, w.block_size, r)[p]
    s = got[: w.num_tokens][valid]
    p = pos[: w.num_tokens][valid]
    r = req[: w.num_tokens][valid]
    assert (s >= 0).all()
    assert (s % w.block_size == p % w.block_size).all()
    assert all(int(b) in set(w.block_table[rr].tolist()) for b, rr in zip(s // w.block_size, r))
    assert len(np.unique(s)) == len(s)  # distinct ids -> injective
    assert (got[w.num_tokens:] == -1).all()


@pytest.mark.parametrize("bs,kbs", [(32, 16), (64, 16), (16, 16), (64, 8), (48, 16)])
def test_kernel_block_expansion_preserves_slots(bs, kbs):
    rng = np.random.default_rng(5)
    rows, cols = 6, 5
    mgr = rng.permutation(np.arange(1, rows * cols + 1)).reshape(rows, cols).astype(np.int32)
    mgr[1, 3:] = -1
    mgr[2, 2] = 0
    kt = oracle.map_to_kernel_blocks(mgr, bs, kbs)
    assert kt.shape == (rows, cols * (bs // kbs))
    if bs == kbs:
        assert (kt == np.where(mgr > 0, mgr, -1)).all()
    req = np.repeat(np.arange(rows, dtype=np.int32), cols * bs)
    pos = np.tile(np.arange(cols * bs, dtype=np.int64), rows)
    s_mgr, e1 = oracle.compute_slot_mapping(mgr, req, pos, bs)
    s_ker, e2 = oracle.compute_slot_mapping(kt, req, pos, kbs)
    assert e1 == e2 == 0
    assert (s_mgr == s_ker).all()
    assert ((kt == -1) == np.repeat(mgr <= 0, bs // kbs, axis=1)).all()


@pytest.mark.parametrize("bpk", [2, 3, 16])
def test_kernel_block_expansion_at_the_int32_edge(bpk):
    """R17: the table holds int32 ids, so an expanded id above 2^31 - 1 names no block (-1); the largest
    manager id whose every kernel id fits expands normally (closed form m * bpk + t)."""
    top = (2**31 - 1 - (bpk - 1)) // bpk          # largest m with m * bpk + bpk - 1 <= INT32_MAX
    mgr = np.array([[top, top + 1, 2**31 - 1, 7]], np.int32)
    kt = oracle.map_to_kernel_blocks(mgr, 16 * bpk, 16)
    t = np.arange(bpk)
    assert kt[0, :bpk].tolist() == (top * bpk + t).tolist()
    assert max(kt[0, :bpk]) <= 2**31 - 1
    straddle = [(top + 1) * bpk + x for x in t]     # some (or all) of these exceed INT32_MAX
    assert kt[0, bpk:2 * bpk].tolist() == [v if v <= 2**31 - 1 else -1 for v in straddle]
    assert (kt[0, bpk:2 * bpk] == -1).any()
    assert (kt[0, 2 * bpk:3 * bpk] == -1).all()
    assert kt[0, 3 * bpk:].tolist() == (7 * bpk + t).tolist()


def test_kernel_block_expansion_rejects_indivisible():
    with pytest.raises(ValueError):
        oracle.map_to_kernel_blocks(np.ones((1, 2), np.int32), 32, 12)
    with pytest.raises(ValueError):
        oracle.map_to_kernel_blocks(np.ones((1, 2), np.int32), 32, 0)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_cache_write_invariants(dtype):
    rng = np.random.default_rng(11)
    tb, bs, h, d = 9, 4, 2, 8
    npdt = np.uint16 if dtype == "bf16" else np.float32
    kc = rng.integers(0, 2**16, size=(tb, bs, h, d)).astype(npdt) if dtype == "bf16" else \
        rng.standard_normal((tb, bs, h, d)).astype(np.float32)
    vc = kc[::-1].copy()
    n = 7
    kn = (rng.integers(0, 2**16, size=(n, h, d)).astype(npdt) if dtype == "bf16"
          else rng.standard_normal((n, h, d)).astype(np.float32))
    vn = kn[::-1].copy()
    slots = np.array([5, -1, 35, 0, 17, 36, -1], np.int64)  # 36 == tb*bs -> out of range
    k2, v2, err = oracle.cache_write(kn, vn, slots, kc, vc)
    assert err == 1
    flat_k, flat_v = k2.reshape(tb * bs, h, d), v2.reshape(tb * bs, h, d)
    written = [5, 35, 0, 17]
    src = [0, 2, 3, 4]
    for s, i in zip(written, src):
        assert flat_k[s].tobytes() == kn[i].tobytes()
        assert flat_v[s].tobytes() == vn[i].tobytes()
    untouched = np.setdiff1d(np.arange(tb * bs), written)
    assert flat_k[untouched].tobytes() == kc.reshape(tb * bs, h, d)[untouched].tobytes()
    assert flat_v[untouched].tobytes() == vc.reshape(tb * bs, h, d)[untouched].tobytes()


def test_cache_write_rejects_duplicate_slots():
    kc = np.zeros((2, 2, 1, 2), np.float32)
    kn = np.ones((2, 1, 2), np.float32)
    with pytest.raises(ValueError):
        oracle.cache_write(kn, kn, np.array([1, 1]), kc, kc)


def test_cache_write_all_padding_writes_nothing():
    kc = np.arange(16, dtype=np.float32).reshape(2, 2, 1, 4)
    kn = np.full((3, 1, 4), 99, np.float32)
    k2, v2, err = oracle.cache_write(kn, kn, np.full(3, -1, np.int64), kc, kc)
    assert err == 0 and (k2 == kc).all() and (v2 == kc).all()


def test_bucket_choice_matches_page_table():
    g = _golden()["bucket_selection_table"]
    for active, bucket in g["active_to_bucket"].items():
        # needed = max(num_computed) + 1 + spec: with num_computed = active - 1 this is `active`
        got = oracle.decode_bucket([int(active) - 1], 0, g["buckets"][:-1], g["buckets"][-1])
        assert got == bucket


def test_decode_bucket_needed_seq():
    # Decode Context-Length Bucketing, Examples: one 16384 bucket under max_model_len 131072.
    assert oracle.decode_bucket([100, 16382], 0, [16384], 131072) == 16384
    assert oracle.decode_bucket([100, 16383], 0, [16384], 131072) == 16384   # 16383 + 1 = 16384 still fits
    assert oracle.decode_bucket([16384], 0, [16384], 131072) == 131072      # 16385 falls back to max_model_len
    assert oracle.decode_bucket([16380], 3, [16384], 131072) == 16384       # 16380 + 1 + 3 = 16384
    assert oracle.decode_bucket([16381], 3, [16384], 131072) == 131072
    assert oracle.decode_bucket([131072], 0, [16384], 131072) == -1


def test_kv_cache_tensor_size_closed_form():
    g = _golden()["kv_cache_tensor_size"]
    k = np.empty((g["num_blocks"], g["block_size"], g["num_kv_heads"], g["head_size"]), np.uint16)
    assert 2 * k.nbytes == g["size"]
