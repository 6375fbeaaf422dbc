"""The seeded synthetic workloads against the configurations they stand for:
sizes, value ranges, block-table structure (distinct physical ids from the
pool, block 0 never handed out, -1 past a request's blocks, NULL rows empty)
and determinism.  No GPU."""
import numpy as np
import pytest

from paged_kv_cache_slot_gb300 import workloads as wl


def _table_ok(w: wl.Workload):
    t = w.block_table
    need = -(-(w.prior_lens + w.new_tokens) // w.block_size)
    used = []
    for r in range(w.num_rows):
        n = int(need[r])
        assert (t[r, :n] >= 1).all() and (t[r, :n] < w.total_blocks).all()
        assert (t[r, n:] == -1).all()
        used.extend(t[r, :n].tolist())
    assert len(used) == len(set(used)), "a physical block is handed out twice"
    # the pool holds the needed blocks, block 0 and about 25% slack
    assert w.total_blocks >= 1 + len(used)
    assert w.total_blocks <= 1 + len(used) + int(np.ceil(0.25 * len(used))) or w.name == "tiny"


@pytest.mark.parametrize("name", wl.WORKLOADS)
def test_workloads_are_deterministic_and_tables_valid(name):
    a, b = wl.make(name), wl.make(name)
    assert np.array_equal(a.block_table, b.block_table) and np.array_equal(a.prior_lens, b.prior_lens)
    _table_ok(a)
    req, pos = a.step_tokens()
    assert len(req) == a.max_num_tokens >= a.num_tokens
    assert (req[a.num_tokens:] == -1).all()
    # this step's tokens sit right after each request's prior tokens
    for r in range(a.num_rows):
        sel = req[: a.num_tokens] == r
        assert np.array_equal(pos[: a.num_tokens][sel], a.prior_lens[r] + np.arange(a.new_tokens[r]))


def test_tiny_configuration():
    w = wl.make("tiny")
    assert (w.num_rows, w.block_size, w.total_blocks, w.width) == (2, 4, 16, 4)
    assert (w.num_q_heads, w.num_kv_heads, w.head_dim, w.dtype) == (2, 1, 8, "f32")
    assert w.context_lens.tolist() == [4, 8]                           # {3, 7} + the decode token
    assert wl.make("tiny", tiny_reading="other").context_lens.tolist() == [3, 7]


def test_llama3_decode_configuration():
    w = wl.make("llama3_decode")
    assert (w.num_rows, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size, w.dtype) == (
        32, 32, 8, 128, 64, "bf16")
    assert (w.prior_lens >= 512).all() and (w.prior_lens <= 4096).all() and (w.new_tokens == 1).all()
    assert w.width == 65 and abs(w.qk_scale - 1 / np.sqrt(128)) < 1e-12


def test_ragged_step_configuration():
    w = wl.make("ragged_step")
    assert (w.num_rows, w.block_size, w.num_kv_heads, w.head_dim, w.width) == (64, 16, 8, 128, 192)
    ones = int((w.new_tokens == 1).sum())
    multi = w.new_tokens[w.new_tokens > 1]
    assert ones == 48 and len(multi) == 16 and (multi >= 64).all() and (multi <= 1024).all()
    assert (w.prior_lens >= 0).all() and (w.prior_lens <= 2048).all()
    assert w.num_tokens == 9691 and not w.has_decode


def test_long_context_configuration():
    w = wl.make("long_context")
    assert (w.num_rows, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size) == (8, 64, 8, 128, 64)
    assert w.width == 131072 // 64                                     # 2048-entry rows, unused = -1
    L = w.context_lens
    assert (L >= 257).all() and (L <= 131072).all()


def test_hybrid_spec_configuration():
    w = wl.make("hybrid_spec")
    assert (w.num_rows, w.num_real, w.q_len) == (320, 256, 4)
    assert (w.block_size, w.kernel_block_size, w.blocks_per_kv_block) == (32, 16, 2)
    assert (w.prior_lens[:256] >= 1).all() and (w.prior_lens[:256] <= 8192).all()
    assert (w.new_tokens[:256] == 4).all()
    # the 64 NULL padding rows: no tokens, no blocks, cache length 0
    assert (w.new_tokens[256:] == 0).all() and (w.block_table[256:] == -1).all() and (w.context_lens[256:] == 0).all()
    # Zipf(1.1): a large share at the clip and a small share of one-token contexts
    assert 0.2 < float((w.prior_lens[:256] == 8192).mean()) < 0.6
