"""Property-based pins of the oracle on random small inputs (hypothesis).

* The state merge is exact log-sum-exp algebra: merging parts in any grouping
  or order gives the same result (to fp64 rounding), and a part with lse -inf
  changes nothing.
* Slot mapping equals a brute-force enumeration of each row's slots in
  logical order, indexed by position, for random tables with null entries.
* Block expansion preserves every token's slot (the kernel view of the cache
  is the manager view's memory).
"""
import numpy as np
import pytest

hyp = pytest.importorskip("hypothesis")
st = pytest.importorskip("hypothesis.strategies")
from hypothesis import given, settings  # noqa: E402

import oracle  # noqa: E402


@settings(max_examples=60, deadline=None)
@given(seed=st.integers(0, 2**31 - 1), parts=st.integers(2, 6), rows=st.integers(1, 9), d=st.integers(1, 17))
def test_merge_is_associative_and_order_free(seed, parts, rows, d):
    rng = np.random.default_rng(seed)
    outs = rng.standard_normal((parts, rows, d))
    lses = rng.standard_normal((parts, rows)) * 4
    lses[rng.random((parts, rows)) < 0.2] = -np.inf
    whole, whole_lse = oracle.merge_attn_states(outs, lses)
    # (first k parts) merged, then merged with the rest
    k = int(rng.integers(1, parts))
    a, al = oracle.merge_attn_states(outs[:k], lses[:k])
    b, bl = oracle.merge_attn_states(outs[k:], lses[k:])
    two, two_lse = oracle.merge_attn_states(np.stack([a, b]), np.stack([al, bl]))
    np.testing.assert_allclose(two, whole, rtol=0, atol=1e-12)
    fin = np.isfinite(whole_lse)
    assert (np.isfinite(two_lse) == fin).all()
    np.testing.assert_allclose(two_lse[fin], whole_lse[fin], rtol=0, atol=1e-12)
    # any order
    perm = rng.permutation(parts)
    p, pl = oracle.merge_attn_states(outs[perm], lses[perm])
    np.testing.assert_allclose(p, whole, rtol=0, atol=1e-12)
    # an extra part that saw nothing changes nothing
    z, zl = oracle.merge_attn_states(np.concatenate([outs, rng.standard_normal((1, rows, d))]),
                                     np.concatenate([lses, np.full((1, rows), -np.inf)]))
    np.testing.assert_allclose(z, whole, rtol=0, atol=1e-12)


@settings(max_examples=60, deadline=None)
@given(seed=st.integers(0, 2**31 - 1), nr=st.integers(1, 6), cols=st.integers(1, 7),
       bs=st.sampled_from([1, 2, 4, 16, 64]))
def test_slot_mapping_equals_brute_force(seed, nr, cols, bs):
    rng = np.random.default_rng(seed)
    ids = rng.permutation(np.arange(1, nr * cols + 5))[: nr * cols].astype(np.int32).reshape(nr, cols)
    ids[rng.random(ids.shape) < 0.2] = 0
    ids[rng.random(ids.shape) < 0.1] = -1
    # every row's slots in logical order, by enumeration
    table_slots = {}
    for r in range(nr):
        for li in range(cols):
            for o in range(bs):
                b = int(ids[r, li])
                table_slots[(r, li * bs + o)] = b * bs + o if b > 0 else -1
    n = 40
    req = rng.integers(-1, nr, size=n).astype(np.int32)
    pos = rng.integers(0, cols * bs, size=n).astype(np.int64)
    got, err = oracle.compute_slot_mapping(ids, req, pos, bs, n, n + 3)
    want = [table_slots[(int(r), int(p))] if r >= 0 else -1 for r, p in zip(req, pos)] + [-1] * 3
    assert got.tolist() == want and err == 0


@settings(max_examples=40, deadline=None)
@given(seed=st.integers(0, 2**31 - 1), bpk=st.sampled_from([1, 2, 4, 8]), kbs=st.sampled_from([1, 4, 16]))
def test_expansion_preserves_slots(seed, bpk, kbs):
    rng = np.random.default_rng(seed)
    bs = bpk * kbs
    nr, cols = 4, 5
    mgr = rng.permutation(np.arange(1, nr * cols + 3))[: nr * cols].astype(np.int32).reshape(nr, cols)
    mgr[rng.random(mgr.shape) < 0.2] = -1
    kt = oracle.map_to_kernel_blocks(mgr, bs, kbs)
    req = np.repeat(np.arange(nr, dtype=np.int32), cols * bs)
    pos = np.tile(np.arange(cols * bs, dtype=np.int64), nr)
    a, _ = oracle.compute_slot_mapping(mgr, req, pos, bs)
    b, _ = oracle.compute_slot_mapping(kt, req, pos, kbs)
    assert np.array_equal(a, b)
