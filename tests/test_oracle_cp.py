"""Pins for the oracle's decode-context-parallel pieces (reading R14 of the
oracle source: position p belongs to rank (p / I) mod W and sits at local
position (p / (I W)) I + p mod I on it; a rank's decode reports its
normalised output and log-sum-exp; the merge weights ranks by exp(lse)).

* Worked example: slots written out by hand for W = 2, I = 1 and 2.
* Reductions: W = 1 is the plain slot mapping, bit for bit.
* Invariants: every token is real on exactly one rank, and a rank's tokens
  of a request fill local positions 0, 1, 2, ... in position order.
* Library routine: lse equals torch.logsumexp of the scaled scores (fp64).
* The split is exact: merging the ranks' (out, lse) of a cache sharded
  through the oracle's own CP slot mapping and cache write equals the
  unsplit attention to fp64 rounding, for several W, I, q_len and masks.
* Merge closed forms: equal lse gives the mean; -inf parts drop out; all
  -inf gives 0 and -inf.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle.cases import fill_oracle_cache, fill_oracle_cache_cp
from paged_kv_cache_slot_gb300 import workloads as wl


def test_cp_slot_mapping_worked_example():
    bs = 4
    t0 = np.array([[5, 7, -1]], np.int32)      # rank 0's table for request 0
    t1 = np.array([[3, 9, -1]], np.int32)      # rank 1's
    req = np.zeros(10, np.int32)
    pos = np.arange(10, dtype=np.int64)
    s0, e0 = oracle.compute_slot_mapping_cp(t0, req, pos, bs, 2, 0, 1)
    s1, e1 = oracle.compute_slot_mapping_cp(t1, req, pos, bs, 2, 1, 1)
    assert e0 == e1 == 0
    assert s0.tolist() == [20, -1, 21, -1, 22, -1, 23, -1, 28, -1]
    assert s1.tolist() == [-1, 12, -1, 13, -1, 14, -1, 15, -1, 36]
    s0, _ = oracle.compute_slot_mapping_cp(t0, req, pos, bs, 2, 0, 2)
    s1, _ = oracle.compute_slot_mapping_cp(t1, req, pos, bs, 2, 1, 2)
    assert s0.tolist() == [20, 21, -1, -1, 22, 23, -1, -1, 28, 29]
    assert s1.tolist() == [-1, -1, 12, 13, -1, -1, 14, 15, -1, -1]


def _random_tokens(rng, nr, width, bs, n):
    table = np.full((nr, width), -1, np.int32)
    ids = rng.permutation(np.arange(1, nr * width + 1))
    table[:, :] = ids.reshape(nr, width)
    req = rng.integers(-1, nr, n).astype(np.int32)
    pos = rng.integers(0, width * bs, n).astype(np.int64)
    return table, req, pos


def test_cp_world_one_is_the_plain_slot_mapping():
    rng = np.random.default_rng(1)
    table, req, pos = _random_tokens(rng, 5, 9, 8, 300)
    plain, e = oracle.compute_slot_mapping(table, req, pos, 8, num_tokens=250, max_num_tokens=300)
    for inter in (1, 3, 16):
        cp, e2 = oracle.compute_slot_mapping_cp(table, req, pos, 8, 1, 0, inter, num_tokens=250, max_num_tokens=300)
        assert e2 == e and cp.tobytes() == plain.tobytes()


@pytest.mark.parametrize("world,inter", [(2, 1), (3, 2), (4, 16), (8, 4)])
def test_cp_tokens_owned_once_and_local_positions_consecutive(world, inter):
    rng = np.random.default_rng(world * 100 + inter)
    bs, nr, width = 4, 3, 40
    L = 150
    req = np.repeat(np.arange(nr, dtype=np.int32), L)
    pos = np.tile(np.arange(L, dtype=np.int64), nr)
    owners = np.zeros(len(pos), np.int64)
    for k in range(world):
        table = rng.permutation(np.arange(1, nr * width + 1)).reshape(nr, width).astype(np.int32)
        slots, err = oracle.compute_slot_mapping_cp(table, req, pos, bs, world, k, inter)
        assert err == 0
        real = slots >= 0
        owners += real
        # invert slot -> local position through the table
        where = {int(b): (r, lb) for r in range(nr) for lb, b in enumerate(table[r])}
        for r in range(nr):
            sel = real & (req == r)
            locs = []
            for sl in slots[sel]:
                rr, lb = where[int(sl) // bs]
                assert rr == r
                locs.append(lb * bs + int(sl) % bs)
            assert locs == list(range(len(locs)))          # 0, 1, 2, ... in position order
    assert (owners == 1).all()


def _small(q_len=3, prior=(37, 0, 20, 61, 9)):
    prior = np.array(prior, np.int64)
    nr = len(prior)
    new = np.full(nr, q_len, np.int64)
    new[1] = 0
    bs = 4
    need = -(-(prior + new) // bs)
    width = int(need.max()) + 1
    rng = np.random.default_rng(9)
    total = 1 + int(need.sum()) + 3
    ids = rng.permutation(np.arange(1, total))[: int(need.sum())]
    table = np.full((nr, width), -1, np.int32)
    k = 0
    for r, n in enumerate(need):
        table[r, :n] = ids[k:k + n]
        k += int(n)
    return wl.Workload("cp", 515, "bf16", nr, nr - 1, q_len, 8, 2, 16, bs, bs, prior, new, table, total,
                       max_num_tokens=int(new.sum()), qk_scale=1.0, v_scale=0.7)


def test_lse_matches_torch_logsumexp():
    w = _small()
    kc, vc, table = fill_oracle_cache(w)
    out, lse, err = oracle.paged_decode_cp(w.q(), kc, vc, table, w.context_lens)
    assert err == 0
    q = wl.to_f32(w.q()).astype(np.float64)
    G = w.group_size
    for r in range(w.num_rows):
        L = int(w.context_lens[r])
        if L == 0:
            assert np.isneginf(lse[r]).all()
            continue
        k, _ = w.kv_rows(r, 0, L)
        k = torch.from_numpy(wl.to_f32(k).astype(np.float64))          # (L, H_kv, D)
        for t in range(w.q_len):
            vis = L - w.q_len + t + 1                                  # causal: keys 0..p_t
            for h in range(w.num_q_heads):
                s = k[:vis, h // G, :] @ torch.from_numpy(q[r, t, h]) / np.sqrt(w.head_dim)
                want = float(torch.logsumexp(s, dim=0)) if vis > 0 else -np.inf
                assert abs(lse[r, t, h] - want) <= 1e-12 * max(1.0, abs(want))


@pytest.mark.parametrize("world,inter,q_len,mask_mode", [(2, 1, 1, 0), (2, 4, 3, 0), (3, 2, 3, 1), (4, 1, 2, 0),
                                                          (4, 8, 3, 0), (5, 3, 1, 1)])
def test_merging_the_ranks_equals_the_unsplit_attention(world, inter, q_len, mask_mode):
    w = _small(q_len=q_len)
    kc, vc, table = fill_oracle_cache(w)
    want, want_lse, _ = oracle.paged_decode_cp(w.q(), kc, vc, table, w.context_lens, mask_mode=mask_mode)
    tables = wl.cp_block_tables(w, world)
    caches = fill_oracle_cache_cp(w, world, inter, tables)
    outs, lses = [], []
    for k, ((tab, _), (kk, vv)) in enumerate(zip(tables, caches)):
        o, l, err = oracle.paged_decode_cp(w.q(), kk, vv, tab, w.context_lens, world, k, inter, mask_mode=mask_mode)
        assert err == 0
        outs.append(o.reshape(-1, w.head_dim))
        lses.append(l.reshape(-1))
    got, got_lse = oracle.merge_attn_states(np.stack(outs), np.stack(lses))
    np.testing.assert_allclose(got, want.reshape(-1, w.head_dim), rtol=0, atol=1e-12)
    fin = np.isfinite(want_lse.reshape(-1))
    assert (np.isfinite(got_lse) == fin).all()
    np.testing.assert_allclose(got_lse[fin], want_lse.reshape(-1)[fin], rtol=0, atol=1e-12)


def test_merge_closed_forms():
    rng = np.random.default_rng(4)
    outs = rng.standard_normal((3, 5, 8))
    lses = np.full((3, 5), 0.7)
    out, lse = oracle.merge_attn_states(outs, lses)
    np.testing.assert_allclose(out, outs.mean(axis=0), rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse, 0.7 + np.log(3.0), rtol=0, atol=1e-15)
    lses2 = lses.copy()
    lses2[1] = -np.inf                                        # a rank that saw no key
    out, lse = oracle.merge_attn_states(outs, lses2)
    np.testing.assert_allclose(out, (outs[0] + outs[2]) / 2, rtol=0, atol=1e-15)
    out, lse = oracle.merge_attn_states(outs, np.full((3, 5), -np.inf))
    assert (out == 0).all() and np.isneginf(lse).all()
