"""Pins for the oracle's paged decode attention.

* Library special case: on small inputs the oracle equals torch's
  scaled_dot_product_attention in float64 on the CPU, run on each request's
  contiguous K/V rows taken from the generator (not from the paged cache),
  with KV heads repeated per GQA group and the mask built from the step's
  token positions.
* Closed forms: one visible key returns that V row; equal keys return the
  mean of V.
* Invariants: permuting physical block ids (moving the cache with them),
  poisoning unreferenced memory with NaN, trimming the table, and writing 0
  instead of -1 for unused entries leave every output bit unchanged;
  padded (NULL) rows give 0.
* Sliding window (reading R13): SDPA with the banded mask; a window that
  covers every key changes no bit; a window of one returns the query's own
  V row exactly; blocks wholly before the window may be null, garbage or
  NaN without changing a bit or counting an error.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_slot_gb300 import workloads as wl
from oracle.cases import BF16_NAN, fill_oracle_cache

F64 = torch.float64


def _sdpa_request(w, r, mask_mode, drop_logical_blocks=(), window=0):
    """torch SDPA (fp64, CPU) for request r on its contiguous generator rows."""
    L = int(w.context_lens[r])
    q = wl.to_f32(w.q()[r]).astype(np.float64)                # (q_len, H_q, D)
    if L == 0:
        return np.zeros_like(q)
    k, v = w.kv_rows(r, 0, L)
    k = wl.to_f32(k).astype(np.float64)
    v = wl.to_f32(v).astype(np.float64)
    req, pos = w.step_tokens()
    qpos = pos[req == r]                                       # this step's positions of request r
    assert len(qpos) == w.q_len
    keep = np.ones(L, bool)
    for lb in drop_logical_blocks:
        keep[lb * w.kernel_block_size:(lb + 1) * w.kernel_block_size] = False
    kpos = np.arange(L)[keep]
    k, v = k[keep], v[keep]
    if mask_mode == 0:
        allowed = kpos[None, :] <= qpos[:, None]
    else:
        allowed = np.ones((w.q_len, len(kpos)), bool)
    if window > 0:
        allowed &= kpos[None, :] > qpos[:, None] - window
    G = w.group_size
    qt = torch.from_numpy(q).permute(1, 0, 2)                  # (H_q, q_len, D)
    kt = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(G, dim=0)
    vt = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(G, dim=0)
    out = torch.nn.functional.scaled_dot_product_attention(
        qt, kt, vt, attn_mask=torch.from_numpy(allowed)[None], dropout_p=0.0)
    out = out.permute(1, 0, 2).numpy()
    rows_with_no_key = ~allowed.any(axis=1)
    out[rows_with_no_key] = 0.0
    return out


def _small(name="gqa", q_len=3, H_q=8, H_kv=2, D=16, bs=4, prior=(9, 0, 1, 22, 4), dtype="bf16", qk=1.0, v=0.7):
    prior = np.array(prior, np.int64)
    nr = len(prior)
    new = np.where(prior >= 0, q_len, 0).astype(np.int64)
    new[1] = 0                      # row 1 is a padded NULL row
    width = 9
    rng = np.random.default_rng(77)
    need = -(-(prior + new) // bs)
    total = 1 + int(need.sum()) + 3
    ids = rng.permutation(np.arange(1, total))[: int(need.sum())]
    table = np.full((nr, width), -1, np.int32)
    k = 0
    for r, n in enumerate(need):
        table[r, :n] = ids[k:k + n]
        k += int(n)
    return wl.Workload(name, 4242, dtype, nr, nr - 1, q_len, H_q, H_kv, D, bs, bs, prior, new, table, total,
                       max_num_tokens=int(new.sum()) + 2, qk_scale=qk, v_scale=v)


def _oracle_all(w, kc, vc, table, mask_mode=0, scale=None):
    out, err = oracle.paged_decode(w.q(), kc, vc, table, w.context_lens, scale=scale, mask_mode=mask_mode)
    return out, err


@pytest.mark.parametrize("reading", ["record", "other"])
@pytest.mark.parametrize("mask_mode", [0, 1])
def test_tiny_matches_sdpa(reading, mask_mode):
    w = wl.make("tiny", tiny_reading=reading)
    kc, vc, table = fill_oracle_cache(w)
    out, err = _oracle_all(w, kc, vc, table, mask_mode)
    assert err == 0
    for r in range(w.num_rows):
        np.testing.assert_allclose(out[r], _sdpa_request(w, r, mask_mode), rtol=0, atol=1e-12)


@pytest.mark.parametrize("mask_mode", [0, 1])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_gqa_multi_token_matches_sdpa(mask_mode, dtype):
    w = _small(dtype=dtype)
    kc, vc, table = fill_oracle_cache(w)
    out, err = _oracle_all(w, kc, vc, table, mask_mode)
    assert err == 0
    assert np.isfinite(out).all()
    for r in range(w.num_rows):
        np.testing.assert_allclose(out[r], _sdpa_request(w, r, mask_mode), rtol=0, atol=1e-12)
    assert (out[1] == 0).all()  # padded NULL row


@pytest.mark.parametrize("name", ["llama3_decode", "hybrid_spec"])
def test_full_shape_sampled_rows_match_sdpa(name):
    w = wl.make(name, sharp=True)
    lens = w.context_lens
    rows = [int(np.argmin(np.where(lens > 0, lens, 1 << 30))), int(np.argmax(lens)), 3]
    kc, vc, table = fill_oracle_cache(w, rows=rows)
    for r in rows:
        got, err = oracle.paged_decode_request(r, w.q(), kc, vc, table, lens)
        assert err == 0
        np.testing.assert_allclose(got, _sdpa_request(w, r, 0), rtol=0, atol=1e-11)


def test_null_entry_inside_range_is_masked_and_zero_equals_minus_one():
    w = _small(prior=(9, 0, 1, 22, 4))
    kc, vc, table = fill_oracle_cache(w)
    t_neg, t_zero = table.copy(), table.copy()
    t_neg[3, 2] = -1
    t_zero[3, 2] = 0
    a, ea = _oracle_all(w, kc, vc, t_neg)
    b, eb = _oracle_all(w, kc, vc, t_zero)
    assert ea == eb == 0
    assert a.tobytes() == b.tobytes()
    np.testing.assert_allclose(a[3], _sdpa_request(w, 3, 0, drop_logical_blocks=[2]), rtol=0, atol=1e-12)


def test_single_visible_key_returns_that_value_row():
    w = _small(prior=(0, 0, 0, 0, 0), q_len=1)
    kc, vc, table = fill_oracle_cache(w)
    out, _ = _oracle_all(w, kc, vc, table)
    for r in (0, 2, 3, 4):
        _, v = w.kv_rows(r, 0, 1)
        want = np.repeat(wl.to_f32(v[0]).astype(np.float64), w.group_size, axis=0)  # (H_q, D)
        assert (out[r, 0] == want).all()


def test_equal_keys_give_mean_of_values():
    w = _small(prior=(13, 0, 5, 2, 7), q_len=2)
    kc, vc, table = fill_oracle_cache(w)
    kc[...] = np.uint16(0x3F80) if w.dtype == "bf16" else np.float32(1.0)  # every key is 1.0
    out, _ = _oracle_all(w, kc, vc, table, mask_mode=1)
    for r in (0, 2, 3, 4):
        L = int(w.context_lens[r])
        _, v = w.kv_rows(r, 0, L)
        mean = wl.to_f32(v).astype(np.float64).mean(axis=0)           # (H_kv, D)
        want = np.repeat(mean, w.group_size, axis=0)
        for t in range(w.q_len):
            np.testing.assert_allclose(out[r, t], want, rtol=0, atol=1e-14)


def test_block_permutation_invariance_bitwise():
    w = _small(prior=(30, 0, 17, 22, 9))
    kc, vc, table = fill_oracle_cache(w)
    base, _ = _oracle_all(w, kc, vc, table)
    rng = np.random.default_rng(3)
    tb = kc.shape[0]
    perm = np.concatenate([[0], rng.permutation(np.arange(1, tb))])   # new id of old block b
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[perm], vc2[perm] = kc, vc
    t2 = np.where(table > 0, perm[np.maximum(table, 0)], table).astype(np.int32)
    moved, _ = _oracle_all(w, kc2, vc2, t2)
    assert moved.tobytes() == base.tobytes()


def test_poisoned_unreferenced_memory_and_trim_do_not_change_output():
    w = _small(prior=(30, 0, 17, 22, 9))
    kc, vc, table = fill_oracle_cache(w)
    base, _ = _oracle_all(w, kc, vc, table)
    assert np.isfinite(base).all()  # NaN background never leaks
    # garbage ids past each row's last needed block must not be read
    t2 = table.copy()
    for r in range(w.num_rows):
        n = -(-int(w.context_lens[r]) // w.kernel_block_size)
        t2[r, n:] = 10**6
    out2, err = _oracle_all(w, kc, vc, t2)
    assert err == 0 and out2.tobytes() == base.tobytes()
    # head trim to the smallest width that covers every row keeps absolute positions
    n_max = -(-int(w.context_lens.max()) // w.kernel_block_size)
    out3, _ = _oracle_all(w, kc, vc, np.ascontiguousarray(table[:, :n_max]))
    assert out3.tobytes() == base.tobytes()


def test_out_of_range_ids_are_counted():
    w = _small(prior=(30, 0, 17, 22, 9))
    kc, vc, table = fill_oracle_cache(w)
    t2 = table.copy()
    t2[0, 1] = kc.shape[0]        # id past the cache
    _, err = _oracle_all(w, kc, vc, t2)
    assert err >= 1


def test_query_rows_before_position_zero_are_zero():
    # cache length 2 with 4 query tokens: the first two queries sit at negative positions
    w = _small(prior=(0, 0, 0, 0, 0), q_len=4)
    w = dataclasses.replace(w, new_tokens=np.array([2, 0, 2, 2, 2], np.int64))
    kc, vc, table = fill_oracle_cache(w)
    out, _ = _oracle_all(w, kc, vc, table)
    assert (out[:, :2] == 0).all() and np.isfinite(out).all()
    assert (out[0, 2] != 0).any()


# ---------------------------------------------------------------------------
# sliding window (R13)
# ---------------------------------------------------------------------------
def _oracle_win(w, kc, vc, table, window, mask_mode=0):
    return oracle.paged_decode(w.q(), kc, vc, table, w.context_lens, mask_mode=mask_mode, sliding_window=window)


@pytest.mark.parametrize("mask_mode", [0, 1])
@pytest.mark.parametrize("window", [1, 2, 5, 9, 17])
def test_window_matches_sdpa_with_banded_mask(mask_mode, window):
    w = _small(prior=(30, 0, 17, 22, 9))
    kc, vc, table = fill_oracle_cache(w)
    out, err = _oracle_win(w, kc, vc, table, window, mask_mode)
    assert err == 0
    for r in range(w.num_rows):
        np.testing.assert_allclose(out[r], _sdpa_request(w, r, mask_mode, window=window), rtol=0, atol=1e-12)


def test_window_covering_every_key_changes_no_bit():
    w = _small(prior=(30, 0, 17, 22, 9))
    kc, vc, table = fill_oracle_cache(w)
    base, _ = _oracle_all(w, kc, vc, table)
    wide = int(w.context_lens.max()) + w.q_len
    out, _ = _oracle_win(w, kc, vc, table, wide)
    assert out.tobytes() == base.tobytes()
    out0, _ = _oracle_win(w, kc, vc, table, 0)
    assert out0.tobytes() == base.tobytes()


def test_window_of_one_returns_the_query_positions_value_row():
    w = _small(prior=(30, 0, 17, 22, 9), q_len=3)
    kc, vc, table = fill_oracle_cache(w)
    out, _ = _oracle_win(w, kc, vc, table, 1)
    for r in (0, 2, 3, 4):
        L = int(w.context_lens[r])
        _, v = w.kv_rows(r, 0, L)
        v = wl.to_f32(v).astype(np.float64)
        for t in range(w.q_len):
            p = L - w.q_len + t
            assert (out[r, t] == np.repeat(v[p], w.group_size, axis=0)).all()


def test_blocks_before_the_window_are_never_read():
    w = _small(prior=(30, 0, 17, 22, 9), q_len=2)
    kc, vc, table = fill_oracle_cache(w)
    window = 5
    base, err = _oracle_win(w, kc, vc, table, window)
    assert err == 0 and np.isfinite(base).all()
    bs = w.kernel_block_size
    t_null, t_junk = table.copy(), table.copy()
    kp, vp = kc.copy(), vc.copy()
    for r in range(w.num_rows):
        L = int(w.context_lens[r])
        lo = max(0, L - w.q_len - window + 1)          # first key any query of the row sees
        for lb in range(lo // bs):                     # logical blocks wholly before it
            b = int(table[r, lb])
            if b > 0:
                kp[b] = BF16_NAN if w.dtype == "bf16" else np.nan
                vp[b] = BF16_NAN if w.dtype == "bf16" else np.nan
            t_null[r, lb] = -1
            t_junk[r, lb] = 10**6
    for tab, k_, v_ in ((t_null, kc, vc), (t_junk, kc, vc), (table, kp, vp)):
        out, err = _oracle_win(w, k_, v_, tab, window)
        assert err == 0
        assert out.tobytes() == base.tobytes()
