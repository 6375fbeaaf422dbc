"""Pins for the oracle's attention over a mixed (ragged) step (reading R15:
request r's q_len_r packed query tokens sit at positions L_r - q_len_r + i).

* Library routine: torch SDPA in fp64 per request on its contiguous
  generator rows with the per-token causal mask.
* Reduction: with one q_len for every request it is the decode, bit for bit.
* Chunking: a request's tokens processed as one chunk or as two consecutive
  chunks (the first with the shorter cache) give the same bits.
* Closed form: a request's first token with nothing before it returns V[0].
"""
import numpy as np
import pytest
import torch

import oracle
from oracle.cases import fill_oracle_cache
from paged_kv_cache_slot_gb300 import workloads as wl


def _ragged(new=(1, 5, 37, 0, 1, 130), prior=(40, 0, 3, 9, 0, 70), dtype="bf16", H_q=8, H_kv=2, D=16, bs=4,
            seed=321):
    prior = np.array(prior, np.int64)
    new = np.array(new, np.int64)
    nr = len(prior)
    need = -(-(prior + new) // bs)
    width = int(need.max()) + 1
    rng = np.random.default_rng(seed)
    total = 1 + int(need.sum()) + 3
    ids = rng.permutation(np.arange(1, total))[: int(need.sum())]
    table = np.full((nr, width), -1, np.int32)
    k = 0
    for r, n in enumerate(need):
        table[r, :n] = ids[k:k + n]
        k += int(n)
    return wl.Workload("ragged_small", seed, dtype, nr, nr, 0, H_q, H_kv, D, bs, bs, prior, new, table, total,
                       max_num_tokens=int(new.sum()), qk_scale=1.0, v_scale=0.7)


def _sdpa(w, r, q, mask_mode):
    L = int(w.context_lens[r])
    qsl = w.query_start_loc()
    qr = wl.to_f32(q[qsl[r]:qsl[r + 1]]).astype(np.float64)         # (ql, H_q, D)
    ql = len(qr)
    if ql == 0 or L == 0:
        return np.zeros_like(qr)
    k, v = w.kv_rows(r, 0, L)
    k = torch.from_numpy(wl.to_f32(k).astype(np.float64)).permute(1, 0, 2).repeat_interleave(w.group_size, 0)
    v = torch.from_numpy(wl.to_f32(v).astype(np.float64)).permute(1, 0, 2).repeat_interleave(w.group_size, 0)
    qpos = L - ql + np.arange(ql)
    allowed = (np.arange(L)[None, :] <= qpos[:, None]) if mask_mode == 0 else np.ones((ql, L), bool)
    o = torch.nn.functional.scaled_dot_product_attention(torch.from_numpy(qr).permute(1, 0, 2), k, v,
                                                         attn_mask=torch.from_numpy(allowed)[None])
    return o.permute(1, 0, 2).numpy()


@pytest.mark.parametrize("mask_mode", [0, 1])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_ragged_matches_sdpa(mask_mode, dtype):
    w = _ragged(dtype=dtype)
    kc, vc, table = fill_oracle_cache(w)
    q = w.q_tokens()
    out, err = oracle.paged_attention_ragged(q, w.query_start_loc(), kc, vc, table, w.context_lens,
                                             mask_mode=mask_mode)
    assert err == 0 and np.isfinite(out).all()
    qsl = w.query_start_loc()
    for r in range(w.num_rows):
        np.testing.assert_allclose(out[qsl[r]:qsl[r + 1]], _sdpa(w, r, q, mask_mode), rtol=0, atol=1e-12)


def test_one_q_len_for_all_is_the_decode_bitwise():
    w = _ragged(new=(3, 3, 3, 3), prior=(40, 0, 9, 70))
    kc, vc, table = fill_oracle_cache(w)
    q = w.q_tokens()
    out, _ = oracle.paged_attention_ragged(q, w.query_start_loc(), kc, vc, table, w.context_lens)
    dec, _ = oracle.paged_decode(q.reshape(4, 3, w.num_q_heads, w.head_dim), kc, vc, table, w.context_lens)
    assert out.tobytes() == dec.reshape(out.shape).tobytes()


def test_chunked_prefill_equals_one_chunk_bitwise():
    w = _ragged(new=(1, 50, 1), prior=(20, 30, 7))
    kc, vc, table = fill_oracle_cache(w)
    q = w.q_tokens()
    qsl = w.query_start_loc()
    whole, _ = oracle.paged_attention_ragged(q, qsl, kc, vc, table, w.context_lens)
    # request 1's 50 tokens as 20 then 30: the first chunk sees a cache 30 tokens shorter
    r, a = 1, 20
    t0 = int(qsl[r])
    ctx1 = w.context_lens.copy()
    ctx1[r] -= 50 - a
    part1, _ = oracle.paged_attention_ragged(q[t0:t0 + a], np.array([0, 0, a, a], np.int32), kc, vc, table,
                                             np.array([0, ctx1[r], 0], np.int32))
    part2, _ = oracle.paged_attention_ragged(q[t0 + a:t0 + 50], np.array([0, 0, 50 - a, 50 - a], np.int32), kc, vc,
                                             table, np.array([0, w.context_lens[r], 0], np.int32))
    assert part1.tobytes() == whole[t0:t0 + a].tobytes()
    assert part2.tobytes() == whole[t0 + a:t0 + 50].tobytes()


def test_first_token_of_a_fresh_request_returns_its_value_row():
    w = _ragged(new=(6,), prior=(0,))
    kc, vc, table = fill_oracle_cache(w)
    out, _ = oracle.paged_attention_ragged(w.q_tokens(), w.query_start_loc(), kc, vc, table, w.context_lens)
    _, v = w.kv_rows(0, 0, 1)
    assert (out[0] == np.repeat(wl.to_f32(v[0]).astype(np.float64), w.group_size, axis=0)).all()
