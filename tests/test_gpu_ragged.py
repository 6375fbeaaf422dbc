"""GPU parity for the mixed-step (ragged) attention against the fp64 oracle:
packed query tokens of requests with different q_len (decode tokens,
drafts, prefill chunks), caches written through the library's slot
mapping and cache write, NaN everywhere else.  Error bars as the decode
(tests/_parity.py): per output row, max abs error <= 1e-2 of the row's
largest oracle value for bf16 (fp32 accumulation), 1e-5 of it for fp32.
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


def _ragged(new, prior, dtype="bf16", H_q=32, H_kv=8, D=128, bs=16, seed=777, holes=()):
    prior = np.array(prior, np.int64)
    new = np.array(new, np.int64)
    nr = len(prior)
    need = -(-(prior + new) // bs)
    width = int(need.max()) + 2
    rng = np.random.default_rng(seed)
    total = 1 + int(need.sum()) + 5
    ids = rng.permutation(np.arange(1, total))[: int(need.sum())]
    table = np.full((nr, width), -1, np.int32)
    k = 0
    for r, n in enumerate(need):
        table[r, :n] = ids[k:k + n]
        k += int(n)
    for r, lb in holes:
        table[r, lb] = -1
    return wl.Workload("ragged_gpu", seed, dtype, nr, nr, 0, H_q, H_kv, D, bs, bs, prior, new, table, total,
                       max_num_tokens=int(new.sum()) + 4, qk_scale=1.0, v_scale=1.0 / np.sqrt(D))


def _run(w, mask_mode=0, rows=None, max_query_len=None):
    dw = DeviceWorkload(w)
    dw.write_step()
    dt = dw.tdtype
    q = torch.from_numpy(w.q_tokens())
    q = (q.view(dt) if w.dtype == "bf16" else q).cuda()
    out = torch.full_like(q, float("nan"))
    qsl = torch.from_numpy(w.query_start_loc()).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    mq = int(w.new_tokens.max()) if max_query_len is None else max_query_len
    bkv.bkv_paged_attention_ragged(q, qsl, dw.k_cache, dw.v_cache, dw.kernel_table, dw.context_lens,
                                   dw.max_context_len, mq, out, mask_mode=mask_mode, err_count=err)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().astype(np.float64)
    kc, vc, table = fill_oracle_cache(w, rows=rows)
    want, _ = oracle.paged_attention_ragged(w.q_tokens(), w.query_start_loc(), kc, vc, table, w.context_lens,
                                            mask_mode=mask_mode)
    return got, want, int(err.item())


CASES = [
    # new tokens per request, prior lengths, dtype, H_q, H_kv, D, bs
    ((1, 5, 200, 0, 1, 77, 3), (300, 0, 1000, 40, 2047, 129, 7), "bf16", 32, 8, 128, 16),
    ((1, 1, 1, 1), (500, 64, 2, 1300), "bf16", 32, 8, 128, 64),
    ((129, 256, 1), (0, 128, 900), "bf16", 64, 8, 128, 32),
    ((40, 3, 1), (100, 9, 50), "bf16", 16, 2, 64, 16),
    ((17, 1, 33), (20, 70, 0), "f32", 8, 2, 32, 8),
    ((64, 1), (300, 12), "bf16", 8, 8, 128, 16),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"n{sum(c[0])}_h{c[3]}x{c[4]}_d{c[5]}_bs{c[6]}_{c[2]}")
@pytest.mark.parametrize("mask_mode", [0, 1])
def test_ragged_matches_oracle(case, mask_mode):
    new, prior, dtype, H_q, H_kv, D, bs = case
    w = _ragged(new, prior, dtype, H_q, H_kv, D, bs)
    got, want, err = _run(w, mask_mode)
    assert err == 0
    check_attention(got, want, dtype, f"{case}/{mask_mode}")


def test_ragged_null_entries_inside_the_range_are_masked():
    w = _ragged((50, 1), (300, 400), holes=((0, 3), (1, 10)))
    got, want, err = _run(w)
    assert err == 0
    check_attention(got, want, "bf16", "holes")


@pytest.mark.parametrize("loud", [False, True])
def test_ragged_step_workload_sampled_requests(loud):
    w = wl.make("ragged_step", loud=loud)
    multi = [int(r) for r in np.argsort(w.new_tokens)[-3:]]     # three prefill chunks
    single = [int(r) for r in np.nonzero(w.new_tokens == 1)[0][:3]]
    rows = sorted(multi + single)
    got, want, err = _run(w, rows=rows)
    assert err == 0
    qsl = w.query_start_loc()
    for r in rows:
        a, b = int(qsl[r]), int(qsl[r + 1])
        check_attention(got[a:b], want[a:b], "bf16", f"request {r}")


def test_ragged_request_above_query_bound_is_skipped_and_counted():
    w = _ragged((10, 3), (50, 20))
    got, want, err = _run(w, max_query_len=4)
    assert err == 1                                     # once per skipped request
    assert np.isnan(got[:10]).all()                     # request 0 (10 tokens > 4): rows untouched
    check_attention(got[10:13], want[10:13], "bf16", "request 1")
