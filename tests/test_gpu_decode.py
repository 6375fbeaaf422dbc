"""GPU parity for the paged decode (partition + merge kernels) against the fp64
oracle, plus bitwise invariants of the GPU path itself.

Error bars (tests/_parity.py): per output row (query token, query head)
max abs error <= 1e-2 of the row's largest oracle value (bf16 in/out, fp32
accumulation) or 1e-5 of it (fp32), which for outputs up to 1 is at least as
tight as the configuration's absolute 1e-2 / 1e-5; rows with nothing
visible must be exactly 0.  The "loud" variants (Q, K of variance 2, V
unscaled: outputs O(0.1 .. 1)) run the full-size workloads, where stream-K
splits streams over several CTAs and the merge combines several pieces, so
that a dropped or mis-weighted piece misses the bar by far.  Caches start as
NaN everywhere, so a read of any position that was never written (block 0,
slack blocks, the tail of a request's last block) poisons the output.
Error counts are compared with the oracle's exactly: every bad table entry
a request needs counts once per KV head.
"""

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


def _f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def _oracle_rows(w, rows, mask_mode=0, table=None, window=0):
    """Oracle outputs of ``rows`` and the bad-entry count over them."""
    kc, vc, ktable = fill_oracle_cache(w, rows=rows)
    table = ktable if table is None else table
    q = w.q()
    out, errs = {}, 0
    for r in rows:
        out[r], e = oracle.paged_decode_request(r, q, kc, vc, table, w.context_lens, mask_mode=mask_mode,
                                                sliding_window=window)
        errs += e
    return out, errs


def _check(dw, rows, mask_mode=0, label="", window=0, min_magnitude=None):
    w = dw.w
    dw.workspace.fill_(0xFF)   # NaN everywhere: reading a partial nobody wrote poisons the output
    got = _f64(dw.decode(mask_mode=mask_mode, sliding_window=window))
    torch.cuda.synchronize()
    want, _ = _oracle_rows(w, rows, mask_mode, window=window)
    rows = list(rows)
    worst = check_attention(np.stack([got[r] for r in rows]), np.stack([want[r] for r in rows]), w.dtype, label,
                            min_magnitude=min_magnitude)
    return got, worst


def _custom(q_len, H_q, H_kv, D, bs, prior, dtype="bf16", width=None, seed=4242, null_rows=(), sharp=False,
            holes=()):
    """A small seeded workload spanning several tiles and partitions, with ragged tails."""
    prior = np.array(prior, np.int64)
    nr = len(prior)
    new = np.full(nr, q_len, np.int64)
    for r in null_rows:
        prior[r] = 0
        new[r] = 0
    need = -(-(prior + new) // bs)
    width = int(need.max()) + 2 if width is None else width
    rng = np.random.default_rng(seed)
    total = 1 + int(need.sum()) + 7
    ids = rng.permutation(np.arange(1, total))[: int(need.sum())]
    table = np.full((nr, width), -1, np.int32)
    k = 0
    for r, n in enumerate(need):
        table[r, :n] = ids[k:k + n]
        k += int(n)
    for r, lb in holes:  # null entries inside a request's range: masked, never read
        table[r, lb] = 0
    s = 1.0 / np.sqrt(D)
    return wl.Workload("custom", seed, dtype, nr, nr - len(null_rows), q_len, H_q, H_kv, D, bs, bs, prior, new,
                       table, total, max_num_tokens=int(new.sum()) + 3, qk_scale=1.0 if sharp else s, v_scale=s)


@pytest.mark.parametrize("reading", ["record", "other"])
@pytest.mark.parametrize("mask_mode", [0, 1])
def test_tiny_fp32(reading, mask_mode):
    w = wl.make("tiny", tiny_reading=reading)
    dw = DeviceWorkload(w)
    dw.write_step()
    _check(dw, range(w.num_rows), mask_mode, f"tiny/{reading}/{mask_mode}")


SMALL = [
    # q_len, H_q, H_kv, D, bs, prior, dtype
    (1, 32, 8, 128, 64, (511, 1, 1300, 64, 2047, 129), "bf16"),
    (4, 32, 8, 128, 16, (0, 3, 700, 1025, 17, 250), "bf16"),
    (1, 64, 8, 128, 64, (3000, 70, 1), "bf16"),
    (2, 8, 8, 128, 32, (100, 600, 33), "bf16"),
    (3, 16, 2, 64, 16, (90, 1100, 5, 400), "bf16"),
    (1, 4, 1, 256, 8, (300, 17), "bf16"),
    (4, 8, 2, 32, 4, (50, 3, 260), "f32"),
    (1, 2, 1, 8, 4, (1, 2, 3, 9), "f32"),
    (5, 40, 8, 128, 64, (200, 1500), "bf16"),
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: f"q{c[0]}_h{c[1]}x{c[2]}_d{c[3]}_bs{c[4]}_{c[6]}")
@pytest.mark.parametrize("mask_mode", [0, 1])
def test_small_shapes(case, mask_mode):
    q_len, H_q, H_kv, D, bs, prior, dtype = case
    w = _custom(q_len, H_q, H_kv, D, bs, list(prior) + [0], dtype, null_rows=(len(prior),),
                holes=((0, 1),) if prior[0] >= 2 * bs else ())
    dw = DeviceWorkload(w)
    dw.write_step()
    got, _ = _check(dw, range(w.num_rows), mask_mode, f"{case}")
    assert (got[w.num_rows - 1] == 0).all()


# KV-head counts off the persistent grid: the tensor-core kernel runs P = floor(SMs / H_kv) groups of
# H_kv CTAs (152 SMs: 3 -> 150 CTAs, 7 -> 147), and one group of H_kv CTAs when H_kv exceeds the SM count
# (160: two waves); the merge recomputes each stream's slots from the same rule
OFF_GRID = [
    # q_len, H_q, H_kv, D, bs, prior
    (1, 6, 3, 128, 16, (900, 40, 2100, 5)),
    (2, 35, 7, 128, 32, (1500, 300, 4100)),
    (1, 160, 160, 128, 16, (200, 50, 700)),
]


@pytest.mark.parametrize("case", OFF_GRID, ids=lambda c: f"q{c[0]}_h{c[1]}x{c[2]}")
@pytest.mark.parametrize("mask_mode", [0, 1])
def test_kv_head_counts_off_the_sm_grid(case, mask_mode):
    q_len, H_q, H_kv, D, bs, prior = case
    w = _custom(q_len, H_q, H_kv, D, bs, list(prior) + [0], "bf16", null_rows=(len(prior),), seed=515)
    dw = DeviceWorkload(w)
    dw.write_step()
    got, _ = _check(dw, range(w.num_rows), mask_mode, f"off-grid {case}")   # (workspace NaN-filled first)
    assert (got[w.num_rows - 1] == 0).all()
    assert int(dw.err_count.item()) == 0


VARIANTS = {"literal": {}, "sharp": {"sharp": True}, "loud": {"loud": True}}


@pytest.mark.parametrize("variant", list(VARIANTS))
def test_llama3_decode_all_rows(variant):
    w = wl.make("llama3_decode", **VARIANTS[variant])
    dw = DeviceWorkload(w)
    dw.step()
    _check(dw, range(w.num_rows), 0, f"llama3/{variant}", min_magnitude=0.1 if variant == "loud" else None)
    assert int(dw.err_count.item()) == 0


@pytest.mark.parametrize("variant", ["sharp", "loud"])
def test_long_context_all_rows(variant):
    w = wl.make("long_context", **VARIANTS[variant])
    dw = DeviceWorkload(w)
    dw.step()
    _check(dw, range(w.num_rows), 0, f"long_context/{variant}", min_magnitude=0.1 if variant == "loud" else None)
    assert int(dw.err_count.item()) == 0


def test_hybrid_spec_sampled_rows_and_null_rows():
    w = wl.make("hybrid_spec", sharp=True)
    dw = DeviceWorkload(w)
    dw.step()
    lens = w.context_lens
    real = lens[: w.num_real]
    rows = sorted({int(np.argmax(real)), int(np.argmin(real)), 1, 17, 100, 255, 256, 319})
    got, _ = _check(dw, rows, 0, "hybrid")
    assert (got[w.num_real:] == 0).all()          # padded NULL rows
    assert int(dw.err_count.item()) == 0


def test_hybrid_spec_loud_longest_rows_and_null_rows():
    """The 20 longest requests of the hybrid batch (contexts near 8192, 4 query tokens, kernel blocks of
    16: the streams stream-K splits most) plus NULL rows, with loud values."""
    w = wl.make("hybrid_spec", loud=True)
    dw = DeviceWorkload(w)
    dw.step()
    real = w.context_lens[: w.num_real]
    rows = sorted({int(r) for r in np.argsort(real, kind="stable")[-20:]} | {256, 300, 319})
    got, _ = _check(dw, rows, 0, "hybrid/loud", min_magnitude=0.1)
    assert (got[w.num_real:] == 0).all()
    assert int(dw.err_count.item()) == 0


def _filled(w):
    dw = DeviceWorkload(w)
    dw.write_step()
    torch.cuda.synchronize()
    return dw


def test_block_permutation_invariance_bitwise():
    w = _custom(4, 32, 8, 128, 16, (900, 40, 1700, 333), "bf16", sharp=True)
    dw = _filled(w)
    base = dw.decode().clone()
    tb = dw.k_cache.shape[0]
    g = torch.Generator().manual_seed(8)
    perm = torch.cat([torch.zeros(1, dtype=torch.int64), torch.randperm(tb - 1, generator=g) + 1]).cuda()
    kc2, vc2 = torch.empty_like(dw.k_cache), torch.empty_like(dw.v_cache)
    kc2[perm] = dw.k_cache
    vc2[perm] = dw.v_cache
    t = dw.kernel_table.long()
    t2 = torch.where(t > 0, perm[t.clamp(min=0)], t).int()
    dw.k_cache, dw.v_cache = kc2, vc2
    moved = dw.decode(out=torch.empty_like(base), table=t2)
    torch.cuda.synchronize()
    assert torch.equal(moved.view(torch.int16), base.view(torch.int16))


def test_trim_and_garbage_past_range_and_zero_vs_minus_one_bitwise():
    w = _custom(1, 32, 8, 128, 64, (1000, 64, 3000, 5), "bf16", width=80, sharp=True, holes=((2, 3),))
    dw = _filled(w)
    base = dw.decode().clone()
    n_max = int(-(-w.context_lens.max() // w.kernel_block_size))
    trimmed = dw.kernel_table[:, :n_max].contiguous()
    a = dw.decode(out=torch.empty_like(base), table=trimmed)
    garbage = dw.kernel_table.clone()
    for r in range(w.num_rows):
        n = int(-(-int(w.context_lens[r]) // w.kernel_block_size))
        garbage[r, n:] = 10**7
    b = dw.decode(out=torch.empty_like(base), table=garbage)
    zero = dw.kernel_table.clone()
    zero[2, 3] = 0          # the hole as upstream 0 instead of -1
    c = dw.decode(out=torch.empty_like(base), table=zero)
    torch.cuda.synchronize()
    for x in (a, b, c):
        assert torch.equal(x.view(torch.int16), base.view(torch.int16))
    assert int(dw.err_count.item()) == 0


BAD_ENTRY_CASES = [
    # q_len, H_q, H_kv, D, bs, prior, dtype, bad (row, logical block) entries, window
    (1, 16, 4, 128, 16, (300, 90), "bf16", ((0, 2),), 0),                  # tensor-core kernel
    (3, 32, 8, 128, 64, (900, 1300, 40), "bf16", ((0, 1), (1, 5), (1, 19)), 0),
    (4, 32, 8, 128, 256, (1500, 700), "bf16", ((0, 2), (1, 1)), 0),        # blocks wider than a tile
    (4, 32, 8, 128, 256, (1500, 700), "bf16", ((0, 2), (0, 4), (1, 0)), 300),   # windowed: some not read
    (2, 8, 2, 32, 8, (50, 260, 3), "f32", ((1, 4), (1, 30)), 0),           # CUDA-core kernel
    (5, 40, 8, 128, 64, (200, 1500), "bf16", ((1, 3), (1, 20)), 0),        # 40 query rows: CUDA-core kernel
]


@pytest.mark.parametrize("case", BAD_ENTRY_CASES, ids=lambda c: f"q{c[0]}_h{c[1]}x{c[2]}_d{c[3]}_bs{c[4]}_W{c[8]}")
def test_bad_block_ids_are_masked_and_counted_exactly(case):
    """Ids past the cache inside the needed range: masked like null entries, each counted once per KV head
    (the oracle counts once per request; the counts must agree exactly)."""
    q_len, H_q, H_kv, D, bs, prior, dtype, bad_at, window = case
    w = _custom(q_len, H_q, H_kv, D, bs, prior, dtype, sharp=True)
    dw = _filled(w)
    bad = dw.kernel_table.clone()
    tab = w.block_table.copy()
    for r, lb in bad_at:
        bad[r, lb] = dw.k_cache.shape[0] + 5 + lb
        tab[r, lb] = dw.k_cache.shape[0] + 5 + lb
    dw.err_count.zero_()
    dw.workspace.fill_(0xFF)
    got = _f64(dw.decode(table=bad, sliding_window=window))
    torch.cuda.synchronize()
    rows = list(range(w.num_rows))
    want, errs = _oracle_rows(w, rows, table=tab, window=window)
    assert errs > 0 or window > 0
    assert int(dw.err_count.item()) == H_kv * errs
    check_attention(np.stack([got[r] for r in rows]), np.stack([want[r] for r in rows]), w.dtype, str(case))


def test_block_past_the_table_width_is_counted_exactly():
    """A request longer than its table row: the missing blocks are masked and counted once per KV head."""
    w = _custom(1, 32, 8, 128, 64, (1000, 64, 3000, 5), "bf16", sharp=True)
    dw = _filled(w)
    cols = 30                                   # request 2 needs 47 blocks
    narrow = dw.kernel_table[:, :cols].contiguous()
    dw.err_count.zero_()
    got = _f64(dw.decode(table=narrow))
    torch.cuda.synchronize()
    rows = list(range(w.num_rows))
    want, errs = _oracle_rows(w, rows, table=w.block_table[:, :cols].copy())
    assert errs == 47 - cols
    assert int(dw.err_count.item()) == w.num_kv_heads * errs
    check_attention(np.stack([got[r] for r in rows]), np.stack([want[r] for r in rows]), w.dtype, "narrow table")


@pytest.mark.parametrize("q_len,H_q,H_kv,dtype", [(1, 8, 8, "bf16"), (2, 8, 2, "f32")])
def test_context_len_above_host_bound_is_clamped_and_counted(q_len, H_q, H_kv, dtype):
    D = 128 if dtype == "bf16" else 32
    w = _custom(q_len, H_q, H_kv, D, 16, (100, 50, 300), dtype)
    dw = _filled(w)
    dw.err_count.zero_()
    dw.max_context_len = 80          # below requests 0 and 2
    dw.workspace = bkv.alloc_workspace(w.num_rows, q_len, H_q, H_kv, D, 16, 80)
    got = _f64(dw.decode())
    torch.cuda.synchronize()
    assert int(dw.err_count.item()) == 2        # once per clamped request
    assert np.isfinite(got).all()


def test_workspace_too_small_is_rejected():
    w = _custom(1, 8, 8, 128, 16, (100, 50), "bf16")
    dw = _filled(w)
    dw.workspace = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(bkv.BkvError) as ei:
        dw.decode()
    assert ei.value.status == bkv.BKV_ERR_INVALID_ARG


def test_repeated_steps_are_deterministic():
    w = wl.make("llama3_decode")
    dw = DeviceWorkload(w)
    dw.step()
    a = dw.out.clone()
    for _ in range(3):
        dw.step()
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), dw.out.view(torch.int16))


@pytest.mark.parametrize("name", ["llama3_decode", "hybrid_spec"])
def test_partition_then_merge_equals_one_call_bitwise(name):
    w = wl.make(name)
    dw = DeviceWorkload(w)
    dw.write_step()
    one = dw.decode(out=torch.empty_like(dw.out)).clone()
    two = torch.empty_like(dw.out)
    args = (dw.q, dw.k_cache, dw.v_cache, dw.kernel_table, dw.context_lens, dw.max_context_len, two, dw.workspace)
    bkv.bkv_paged_decode_partition(*args, err_count=dw.err_count)
    bkv.bkv_paged_decode_merge(*args, err_count=dw.err_count)
    torch.cuda.synchronize()
    assert torch.equal(one.view(torch.int16), two.view(torch.int16))
    assert int(dw.err_count.item()) == 0


# ---------------------------------------------------------------------------
# sliding window: key j visible for query t iff j >= L - q_len + t - W + 1
# ---------------------------------------------------------------------------
SWA_CASES = [(c, W, m) for c in range(len(SMALL)) for (W, m) in ((1, 0), (77, 0), (77, 1), (1000, 0))]


@pytest.mark.parametrize("ci,window,mask_mode", SWA_CASES,
                         ids=lambda v: str(v))
def test_sliding_window_small_shapes(ci, window, mask_mode):
    q_len, H_q, H_kv, D, bs, prior, dtype = SMALL[ci]
    w = _custom(q_len, H_q, H_kv, D, bs, list(prior) + [0], dtype, null_rows=(len(prior),))
    dw = DeviceWorkload(w)
    dw.write_step()
    got, _ = _check(dw, range(w.num_rows), mask_mode, f"{SMALL[ci]} W={window}", window=window)
    assert (got[w.num_rows - 1] == 0).all()


def test_sliding_window_long_context_all_rows():
    w = wl.make("long_context", loud=True)
    dw = DeviceWorkload(w)
    dw.step()
    _check(dw, range(w.num_rows), 0, "long_context W=4096", window=4096, min_magnitude=0.1)
    assert int(dw.err_count.item()) == 0


def test_sliding_window_hybrid_sampled_rows():
    w = wl.make("hybrid_spec", loud=True)
    dw = DeviceWorkload(w)
    dw.step()
    real = w.context_lens[: w.num_real]
    rows = sorted({int(r) for r in np.argsort(real, kind="stable")[-12:]} | {int(np.argmin(real)), 1, 17, 100, 255,
                                                                              256, 319})
    got, _ = _check(dw, rows, 0, "hybrid W=512", window=512, min_magnitude=0.1)
    assert (got[w.num_real:] == 0).all()
    assert int(dw.err_count.item()) == 0


def test_sliding_window_never_reads_blocks_before_it_bitwise():
    w = _custom(2, 32, 8, 128, 16, (900, 40, 1700, 333), "bf16", sharp=True)
    dw = _filled(w)
    window = 300
    base = dw.decode(sliding_window=window).clone()
    torch.cuda.synchronize()
    bs = w.kernel_block_size
    t_null, t_junk = dw.kernel_table.clone(), dw.kernel_table.clone()
    dropped = []
    for r in range(w.num_rows):
        L = int(w.context_lens[r])
        lo = max(0, L - w.q_len - window + 1)
        for lb in range(lo // bs):
            dropped.append(int(dw.kernel_table[r, lb]))
            t_null[r, lb] = -1
            t_junk[r, lb] = 10**7
    assert dropped
    dw.err_count.zero_()
    a = dw.decode(out=torch.empty_like(base), table=t_null, sliding_window=window)
    b = dw.decode(out=torch.empty_like(base), table=t_junk, sliding_window=window)
    ids = torch.tensor(dropped, device="cuda", dtype=torch.int64)
    dw.k_cache[ids] = float("nan")
    dw.v_cache[ids] = float("nan")
    c = dw.decode(out=torch.empty_like(base), sliding_window=window)
    torch.cuda.synchronize()
    for x in (a, b, c):
        assert torch.equal(x.view(torch.int16), base.view(torch.int16))
    assert int(dw.err_count.item()) == 0


def test_sliding_window_covering_every_key_is_bitwise_full_attention():
    w = _custom(3, 32, 8, 128, 64, (1000, 64, 3000, 5), "bf16", sharp=True)
    dw = _filled(w)
    base = dw.decode().clone()
    wide = dw.decode(out=torch.empty_like(base), sliding_window=int(w.context_lens.max()) + w.q_len)
    torch.cuda.synchronize()
    assert torch.equal(wide.view(torch.int16), base.view(torch.int16))
