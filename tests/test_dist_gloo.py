"""Multi-process paths on CPU with the gloo backend, world size 2.

* The decode-context-parallel exchange (``paged_kv_cache_slot_gb300.dcp``):
  each rank decodes its own share of every request's keys with the oracle,
  the ranks all-gather their (out, lse) states through ``gather_states``, and
  the merge of the gathered states (the oracle's, on the CPU) equals the
  unsplit attention.  On a GPU the same gather feeds the library's merge
  kernel (``merge_across_ranks``).
* The benchmark's replica aggregation: a step time is the maximum over ranks.
"""
import os

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from oracle.cases import fill_oracle_cache, fill_oracle_cache_cp
from paged_kv_cache_slot_gb300 import workloads as wl

WORLD = 2


def _workload(q_len=3):
    prior = np.array([37, 0, 20, 61, 9], np.int64)
    nr = len(prior)
    new = np.full(nr, q_len, np.int64)
    new[1] = 0                                  # a NULL row: nothing on any rank
    bs = 4
    need = -(-(prior + new) // bs)
    rng = np.random.default_rng(9)
    total = 1 + int(need.sum()) + 3
    ids = rng.permutation(np.arange(1, total))[: int(need.sum())]
    table = np.full((nr, int(need.max()) + 1), -1, np.int32)
    k = 0
    for r, n in enumerate(need):
        table[r, :n] = ids[k:k + n]
        k += int(n)
    return wl.Workload("dcp", 515, "bf16", nr, nr - 1, q_len, 8, 2, 16, bs, bs, prior, new, table, total,
                       max_num_tokens=int(new.sum()), qk_scale=1.0, v_scale=0.7)


def _init(rank, path):
    dist.init_process_group("gloo", init_method=f"file://{path}", rank=rank, world_size=WORLD)


def _dcp_rank(rank, path, inter, mask_mode, q):
    from paged_kv_cache_slot_gb300.dcp import gather_states
    _init(rank, path)
    try:
        w = _workload()
        tables = wl.cp_block_tables(w, WORLD)
        table, _ = tables[rank]
        kc, vc = fill_oracle_cache_cp(w, WORLD, inter, tables)[rank]   # this rank's share of the keys
        out, lse, err = oracle.paged_decode_cp(w.q(), kc, vc, table, w.context_lens, WORLD, rank, inter,
                                               mask_mode=mask_mode)
        assert err == 0
        outs, lses = gather_states(torch.from_numpy(out).float(), torch.from_numpy(lse).float())
        assert outs.shape == (WORLD,) + out.shape and lses.shape == (WORLD,) + lse.shape
        # index k holds rank k's state
        assert torch.equal(outs[rank], torch.from_numpy(out).float())
        assert torch.equal(lses[rank], torch.from_numpy(lse).float())
        merged, merged_lse = oracle.merge_attn_states(outs.double().reshape(WORLD, -1, w.head_dim).numpy(),
                                                      lses.double().reshape(WORLD, -1).numpy())
        q.put((rank, merged, merged_lse))
    finally:
        dist.destroy_process_group()


def _run(fn, *args):
    import tempfile
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    with tempfile.TemporaryDirectory() as d:
        path = os.path.join(d, "store")
        procs = [ctx.Process(target=fn, args=(r, path, *args, q)) for r in range(WORLD)]
        for p in procs:
            p.start()
        res = [q.get(timeout=300) for _ in range(WORLD)]
        for p in procs:
            p.join(timeout=60)
            assert p.exitcode == 0
    return sorted(res, key=lambda x: x[0])


@pytest.mark.parametrize("inter,mask_mode", [(1, 0), (4, 0), (2, 1)])
def test_dcp_exchange_merges_to_the_unsplit_attention(inter, mask_mode):
    oracle.build()                                  # once, before the ranks load it
    res = _run(_dcp_rank, inter, mask_mode)
    w = _workload()
    kc, vc, table = fill_oracle_cache(w)
    want, want_lse, _ = oracle.paged_decode_cp(w.q(), kc, vc, table, w.context_lens, mask_mode=mask_mode)
    want = want.reshape(-1, w.head_dim)
    want_lse = want_lse.reshape(-1)
    for rank, got, got_lse in res:
        # the gathered states went through fp32 (as the kernels keep them): fp32 rounding only
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-5)
        fin = np.isfinite(want_lse)
        assert (np.isfinite(got_lse) == fin).all()
        np.testing.assert_allclose(got_lse[fin], want_lse[fin], rtol=0, atol=1e-5)
    # both ranks hold the same merged result
    assert np.array_equal(res[0][1], res[1][1])


def _max_rank(rank, path, q):
    import bench
    _init(rank, path)
    try:
        mine = [1.0 + rank, 5.0 - rank, 3.0]
        q.put((rank, bench.max_over_ranks(mine, dist)))
    finally:
        dist.destroy_process_group()


def test_bench_step_time_is_the_max_over_ranks():
    res = _run(_max_rank)
    for _, got in res:
        assert got == [2.0, 5.0, 3.0]
    import bench
    assert bench.max_over_ranks([4.0, 2.0], None) == [4.0, 2.0]
