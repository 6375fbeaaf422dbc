"""GPU parity for decode context parallelism (ranks emulated on one GPU, no
collective): the CP slot filter is bit-exact with the oracle; each rank's
decode (out, lse) over caches written through the library's own CP slot
mapping and cache write matches the oracle's rank; and the ranks merged by
bkv_merge_attn_states match the UNSPLIT oracle attention.

Tolerances: out as the decode (tests/_parity.py: per output row, max abs
error <= 1e-2 of the row's largest oracle value for bf16, 1e-5 of it for
fp32; rows that see nothing exactly 0); lse (natural log) 4e-3 for bf16 (the kernel sums bf16-rounded weights, relative error up
to 2^-9 per weight) and 1e-5 for fp32.
"""
import numpy as np
import pytest
import torch

import oracle
from _parity import check_attention
from oracle.cases import fill_oracle_cache, fill_oracle_cache_cp
from paged_kv_cache_slot_gb300 import bkv
from paged_kv_cache_slot_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

LSE_TOL = {"bf16": 4e-3, "f32": 1e-5}


def _custom(q_len, H_q, H_kv, D, bs, prior, dtype, seed=606, null_rows=()):
    prior = np.array(prior, np.int64)
    nr = len(prior)
    new = np.full(nr, q_len, np.int64)
    for r in null_rows:
        prior[r] = 0
        new[r] = 0
    need = -(-(prior + new) // bs)
    width = int(need.max()) + 2
    rng = np.random.default_rng(seed)
    total = 1 + int(need.sum()) + 7
    ids = rng.permutation(np.arange(1, total))[: int(need.sum())]
    table = np.full((nr, width), -1, np.int32)
    k = 0
    for r, n in enumerate(need):
        table[r, :n] = ids[k:k + n]
        k += int(n)
    s = 1.0 / np.sqrt(D)
    return wl.Workload("cp_gpu", seed, dtype, nr, nr - len(null_rows), q_len, H_q, H_kv, D, bs, bs, prior, new,
                       table, total, max_num_tokens=int(new.sum()) + 3, qk_scale=1.0, v_scale=s)


def _tdtype(w):
    return torch.bfloat16 if w.dtype == "bf16" else torch.float32


def _dev(a, w=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if w is not None and w.dtype == "bf16":
        t = t.view(torch.bfloat16)
    return t.cuda()


def _rank_caches(w, world, inter, tables):
    """Every token of every request written into each rank's caches by the library's CP slot mapping."""
    rows = [r for r in range(w.num_rows) if int(w.context_lens[r]) > 0]
    k = np.concatenate([w.kv_rows(r, 0, int(w.context_lens[r]))[0] for r in rows])
    v = np.concatenate([w.kv_rows(r, 0, int(w.context_lens[r]))[1] for r in rows])
    req = np.concatenate([np.full(int(w.context_lens[r]), r, np.int32) for r in rows])
    pos = np.concatenate([np.arange(int(w.context_lens[r]), dtype=np.int64) for r in rows])
    kt, vt, rt, pt = _dev(k, w), _dev(v, w), _dev(req), _dev(pos)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = []
    for rank, (table, total) in enumerate(tables):
        shape = (total, w.kernel_block_size, w.num_kv_heads, w.head_dim)
        kc = torch.full(shape, float("nan"), dtype=_tdtype(w), device="cuda")
        vc = torch.full(shape, float("nan"), dtype=_tdtype(w), device="cuda")
        tab = _dev(table)
        slots = torch.empty(len(pos), dtype=torch.int64, device="cuda")
        bkv.bkv_compute_slot_mapping_cp(tab, rt, pt, w.kernel_block_size, slots, world, rank, inter, err_count=err)
        bkv.bkv_cache_write(kt, vt, slots, kc, vc, err_count=err)
        out.append((kc, vc, tab))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return out


@pytest.mark.parametrize("world,inter", [(1, 1), (2, 1), (2, 16), (4, 3), (8, 64)])
def test_cp_slot_mapping_bit_exact(world, inter):
    rng = np.random.default_rng(world * 31 + inter)
    nr, width, bs, n = 7, 30, 16, 5000
    table = rng.permutation(np.arange(1, nr * width + 1)).reshape(nr, width).astype(np.int32)
    table[2, 5:] = -1
    table[4, 3] = 0
    req = rng.integers(-1, nr + 1, n).astype(np.int32)       # includes padding and a bad request index
    pos = rng.integers(-2, width * bs * world + 40, n).astype(np.int64)
    num_tokens = n - 100
    for rank in range(world):
        want, want_err = oracle.compute_slot_mapping_cp(table, req, pos, bs, world, rank, inter,
                                                        num_tokens=num_tokens, max_num_tokens=n)
        got = torch.empty(n, dtype=torch.int64, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        bkv.bkv_compute_slot_mapping_cp(_dev(table), _dev(req), _dev(pos), bs, got, world, rank, inter,
                                        num_tokens=num_tokens, err_count=err)
        torch.cuda.synchronize()
        assert np.array_equal(got.cpu().numpy(), want)
        assert int(err.item()) == want_err


CASES = [
    # q_len, H_q, H_kv, D, bs, prior, dtype
    (1, 32, 8, 128, 64, (700, 1, 2300, 129, 64), "bf16"),      # tensor-core path
    (3, 16, 4, 128, 16, (90, 1500, 5, 400), "bf16"),          # tensor-core path, causal across 3 tokens
    (2, 8, 2, 32, 8, (50, 3, 260, 77), "f32"),                # generic path
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"q{c[0]}_h{c[1]}x{c[2]}_d{c[3]}_bs{c[4]}_{c[6]}")
@pytest.mark.parametrize("world,inter", [(2, 1), (2, 64), (4, 16), (3, 5)])
def test_cp_ranks_match_oracle_and_merge_to_unsplit(case, world, inter):
    q_len, H_q, H_kv, D, bs, prior, dtype = case
    w = _custom(q_len, H_q, H_kv, D, bs, list(prior) + [0], dtype, null_rows=(len(prior),))
    tables = wl.cp_block_tables(w, world)
    gpu = _rank_caches(w, world, inter, tables)
    host = fill_oracle_cache_cp(w, world, inter, tables)
    q = w.q()
    qt = _dev(q, w)
    ctx = _dev(w.context_lens)
    mx = int(w.context_lens.max())
    ws = bkv.alloc_workspace(w.num_rows, q_len, H_q, H_kv, D, bs, mx)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs, lses = [], []
    for rank in range(world):
        kc, vc, tab = gpu[rank]
        out = torch.empty_like(qt)
        lse = torch.empty((w.num_rows, q_len, H_q), dtype=torch.float32, device="cuda")
        ws.fill_(0xFF)
        bkv.bkv_paged_decode_cp(qt, kc, vc, tab, ctx, mx, out, lse, ws, world, rank, inter, err_count=err)
        torch.cuda.synchronize()
        want, want_lse, _ = oracle.paged_decode_cp(q, host[rank][0], host[rank][1], tables[rank][0], w.context_lens,
                                                   world, rank, inter)
        got = out.float().cpu().numpy().astype(np.float64)
        gl = lse.cpu().numpy().astype(np.float64)
        check_attention(got, want, dtype, f"rank {rank} of {world}")
        fin = np.isfinite(want_lse)
        assert (np.isfinite(gl) == fin).all()
        if fin.any():
            assert np.abs(gl[fin] - want_lse[fin]).max() <= LSE_TOL[dtype]
        outs.append(out)
        lses.append(lse)
    assert int(err.item()) == 0
    merged = torch.empty_like(qt)
    mlse = torch.empty((w.num_rows, q_len, H_q), dtype=torch.float32, device="cuda")
    bkv.bkv_merge_attn_states(torch.stack(outs), torch.stack(lses), merged, mlse)
    torch.cuda.synchronize()
    kc0, vc0, t0 = fill_oracle_cache(w)
    want, want_lse, _ = oracle.paged_decode_cp(q, kc0, vc0, t0, w.context_lens)
    got = merged.float().cpu().numpy().astype(np.float64)
    check_attention(got, want, dtype, f"merged {world} ranks")
    assert (got[w.num_rows - 1] == 0).all()                  # the NULL row
    fin = np.isfinite(want_lse)
    gl = mlse.cpu().numpy().astype(np.float64)
    assert np.abs(gl[fin] - want_lse[fin]).max() <= LSE_TOL[dtype]
    assert np.isneginf(gl[~fin]).all()


def test_cp_world_one_is_the_plain_decode_bitwise():
    w = _custom(2, 32, 8, 128, 64, (900, 40, 1700, 333), "bf16")
    tables = wl.cp_block_tables(w, 1)
    (kc, vc, tab), = _rank_caches(w, 1, 1, tables)
    qt, ctx = _dev(w.q(), w), _dev(w.context_lens)
    mx = int(w.context_lens.max())
    ws = bkv.alloc_workspace(w.num_rows, 2, 32, 8, 128, 64, mx)
    a = torch.empty_like(qt)
    b = torch.empty_like(qt)
    lse = torch.empty((w.num_rows, 2, 32), dtype=torch.float32, device="cuda")
    bkv.bkv_paged_decode(qt, kc, vc, tab, ctx, mx, a, ws)
    bkv.bkv_paged_decode_cp(qt, kc, vc, tab, ctx, mx, b, lse, ws, 1, 0, 1)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_merge_attn_states_matches_oracle(dtype):
    rng = np.random.default_rng(12)
    parts, rows, D = 5, 333, 96
    outs = rng.standard_normal((parts, rows, D)).astype(np.float32)
    lses = (rng.standard_normal((parts, rows)) * 3).astype(np.float32)
    lses[1, ::7] = -np.inf
    lses[:, 5] = -np.inf                                      # a row no part saw
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    o = torch.from_numpy(outs).to(tdt).cuda()
    ref_in = o.float().cpu().numpy().astype(np.float64)       # the values the kernel sees
    want, want_lse = oracle.merge_attn_states(ref_in, lses.astype(np.float64))
    out = torch.empty((rows, D), dtype=tdt, device="cuda")
    lse = torch.empty(rows, dtype=torch.float32, device="cuda")
    bkv.bkv_merge_attn_states(o, torch.from_numpy(lses).cuda(), out, lse)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().astype(np.float64)
    check_attention(got, want, dtype, "merge")               # outputs up to ~4: the bar scales with them
    fin = np.isfinite(want_lse)
    gl = lse.cpu().numpy().astype(np.float64)
    assert np.abs(gl[fin] - want_lse[fin]).max() <= 1e-5
    assert np.isneginf(gl[~fin]).all() and (got[5] == 0).all()


def test_dcp_merge_across_ranks_single_process_nccl(tmp_path):
    """The process-group exchange on the GPU (NCCL), in a one-rank group (two ranks need two GPUs, as
    their collectives wait on one another; the two-rank exchange runs on gloo in test_dist_gloo.py):
    gathering a rank's state and merging it equals the merge kernel on that state directly, bitwise."""
    import torch.distributed as dist
    from paged_kv_cache_slot_gb300.dcp import merge_across_ranks

    w = _custom(1, 32, 8, 128, 64, (700, 1, 2300, 129), "bf16")
    tables = wl.cp_block_tables(w, 2)
    kc, vc, tab = _rank_caches(w, 2, 16, tables)[0]
    qt, ctx = _dev(w.q(), w), _dev(w.context_lens)
    mx = int(w.context_lens.max())
    ws = bkv.alloc_workspace(w.num_rows, 1, 32, 8, 128, 64, mx)
    out = torch.empty_like(qt)
    lse = torch.empty((w.num_rows, 1, 32), dtype=torch.float32, device="cuda")
    bkv.bkv_paged_decode_cp(qt, kc, vc, tab, ctx, mx, out, lse, ws, 2, 0, 16)
    want = torch.empty_like(qt)
    want_lse = torch.empty_like(lse)
    bkv.bkv_merge_attn_states(out.unsqueeze(0), lse.unsqueeze(0), want, want_lse)
    dist.init_process_group("nccl", init_method=f"file://{tmp_path / 'store'}", rank=0, world_size=1)
    try:
        got = torch.empty_like(qt)
        got_lse = torch.empty_like(lse)
        merge_across_ranks(out, lse, got, got_lse)
        torch.cuda.synchronize()
    finally:
        dist.destroy_process_group()
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))
    assert torch.equal(got_lse, want_lse)
