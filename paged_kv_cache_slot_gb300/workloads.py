"""Seeded synthetic inputs for the paged KV cache hot path.

This module only draws inputs: block tables, request lengths, token lists and
K/V/Q values.  It holds none of the method's arithmetic (no slot formula, no
block expansion, no attention); the oracle and the CUDA library each compute
those on their own from what is drawn here.  Both sides import this module,
and nothing else is shared between them.

Five workloads follow the shapes, value distributions and length mixes the
pages and the benchmark configuration name (all synthetic; no dataset):

* ``tiny``          2 requests, block_size 4, 16 blocks (block 0 is the null
                    block), table width 4, H_q 2, H_kv 1, head_dim 8, fp32;
                    context lengths {3, 7} plus one decode token.
* ``llama3_decode`` Llama-3-8B-shaped decode layer: 32 requests, contexts
                    uniform in [512, 4096], 1 new token, H_q 32, H_kv 8,
                    head_dim 128, block_size 64, bf16.
* ``ragged_step``   64 requests (48 with 1 new token, 16 with 64..1024),
                    prior lengths uniform in [0, 2048], block_size 16, H_kv 8,
                    head_dim 128, bf16 (slot mapping + cache write only).
* ``long_context``  8 requests, contexts lognormal (median 4096, sigma 1.0)
                    clipped to [256, 131071], table width 2048 (131072 / 64),
                    H_q 64, H_kv 8, head_dim 128, block_size 64, bf16.
* ``hybrid_spec``   manager block_size 32 split into kernel blocks of 16,
                    256 real rows padded to 320 with NULL rows, contexts Zipf
                    (a = 1.1) clipped to [1, 8192], 4 query tokens per request
                    (1 + 3 speculative), H_q 32, H_kv 8, head_dim 128, bf16.

Physical block ids are a seeded permutation of 1..total_blocks-1 (block 0 is
never handed out, as the pages' block pool reserves it); the pool holds the
needed blocks plus 25% slack.  Unused table entries are -1.  K, V and Q are
N(0, 1) scaled by 1/sqrt(head_dim) for the bf16 workloads (unscaled for
``tiny``); ``sharp=True`` leaves Q and K unscaled so attention weights are far
from uniform; ``loud=True`` draws Q and K with variance 2 (scores of standard
deviation 2 at the 1/sqrt(head_dim) softmax scale, so a few dozen to a few
hundred keys, spread over the whole context, carry most of the weight) and V
unscaled, so that outputs are O(0.1 .. 1) and an absolute error bar of 1e-2
separates a right answer from a wrong one at every context length.  K/V rows
of request r are drawn in chunks of 1024 positions from
``default_rng([seed, 7, r, chunk])`` so that any position range can be
regenerated on its own.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

WORKLOADS = ("tiny", "llama3_decode", "ragged_step", "long_context", "hybrid_spec")
SEEDS = {name: 1001 + i for i, name in enumerate(WORKLOADS)}
KV_CHUNK = 1024


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); bit patterns as uint16."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float32."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def to_f32(a: np.ndarray) -> np.ndarray:
    return bf16_bits_to_f32(a) if a.dtype == np.uint16 else np.asarray(a, dtype=np.float32)


@dataclass
class Workload:
    """One seeded draw.  Arrays are numpy; the caller copies them where needed."""

    name: str
    seed: int
    dtype: str                       # "bf16" or "f32"
    num_rows: int                    # block-table rows (real + padded NULL rows)
    num_real: int
    q_len: int                       # query tokens per request this step
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int                  # manager block size (what the table's ids count in)
    kernel_block_size: int           # block size the attention reads with (== block_size unless hybrid)
    prior_lens: np.ndarray           # int64 (num_rows,) tokens already in the cache (num_computed_tokens)
    new_tokens: np.ndarray           # int64 (num_rows,) tokens written this step
    block_table: np.ndarray          # int32 (num_rows, width) manager ids, -1 unused
    total_blocks: int                # manager blocks in the pool, block 0 included
    max_num_tokens: int              # length of the slot buffer (>= sum(new_tokens))
    qk_scale: float                  # scale applied to drawn Q and K values
    v_scale: float
    has_decode: bool = True
    extra: dict = field(default_factory=dict)

    # ---- derived sizes (plain bookkeeping, no method arithmetic) ----
    @property
    def context_lens(self) -> np.ndarray:
        """Cache length per row after this step's tokens: prior + new (0 for NULL rows)."""
        return (self.prior_lens + self.new_tokens).astype(np.int32)

    @property
    def width(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def num_tokens(self) -> int:
        return int(self.new_tokens.sum())

    @property
    def group_size(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == "bf16" else 4

    @property
    def np_dtype(self):
        return np.uint16 if self.dtype == "bf16" else np.float32

    @property
    def blocks_per_kv_block(self) -> int:
        return self.block_size // self.kernel_block_size

    @property
    def total_kernel_blocks(self) -> int:
        return self.total_blocks * self.blocks_per_kv_block

    def cast(self, x: np.ndarray) -> np.ndarray:
        return f32_to_bf16_bits(x) if self.dtype == "bf16" else np.ascontiguousarray(x, dtype=np.float32)

    # ---- values ----
    def kv_rows(self, r: int, start: int = 0, stop: int | None = None):
        """K and V rows of request r at positions [start, stop): (n, H_kv, D) each."""
        L = int(self.prior_lens[r] + self.new_tokens[r])
        stop = L if stop is None else int(stop)
        if not (0 <= start <= stop <= L):
            raise ValueError(f"positions [{start},{stop}) outside request {r} of length {L}")
        shape = (self.num_kv_heads, self.head_dim)
        ks, vs = [], []
        for c in range(start // KV_CHUNK, (stop + KV_CHUNK - 1) // KV_CHUNK):
            rng = np.random.default_rng([self.seed, 7, int(r), c])
            k = rng.standard_normal((KV_CHUNK,) + shape, dtype=np.float32)
            v = rng.standard_normal((KV_CHUNK,) + shape, dtype=np.float32)
            lo, hi = max(start - c * KV_CHUNK, 0), min(stop - c * KV_CHUNK, KV_CHUNK)
            ks.append(k[lo:hi])
            vs.append(v[lo:hi])
        if not ks:
            z = np.zeros((0,) + shape, np.float32)
            return self.cast(z), self.cast(z)
        k = np.concatenate(ks) * np.float32(self.qk_scale)
        v = np.concatenate(vs) * np.float32(self.v_scale)
        return self.cast(k), self.cast(v)

    def q(self) -> np.ndarray:
        """Queries (num_rows, q_len, H_q, D); NULL rows get values too (they are ignored)."""
        rng = np.random.default_rng([self.seed, 3])
        x = rng.standard_normal((self.num_rows, self.q_len, self.num_q_heads, self.head_dim), dtype=np.float32)
        return self.cast(x * np.float32(self.qk_scale))

    def query_start_loc(self) -> np.ndarray:
        """int32 (num_rows + 1,): request r's query tokens are [qsl[r], qsl[r+1]) of the packed step."""
        return np.concatenate([[0], np.cumsum(self.new_tokens)]).astype(np.int32)

    def q_tokens(self) -> np.ndarray:
        """Packed queries of this step's tokens (num_tokens, H_q, D), one draw per token."""
        rng = np.random.default_rng([self.seed, 5])
        x = rng.standard_normal((self.num_tokens, self.num_q_heads, self.head_dim), dtype=np.float32)
        return self.cast(x * np.float32(self.qk_scale))

    # ---- token lists ----
    def step_tokens(self):
        """This step's tokens: req_indices (int32), positions (int64), both max_num_tokens long.

        Real tokens come first, request by request, at positions prior..prior+new-1.
        Entries past num_tokens are padding: request -1, position 0.
        """
        n, mx = self.num_tokens, self.max_num_tokens
        req = np.full(mx, -1, np.int32)
        pos = np.zeros(mx, np.int64)
        i = 0
        for r in range(self.num_rows):
            k = int(self.new_tokens[r])
            req[i:i + k] = r
            pos[i:i + k] = self.prior_lens[r] + np.arange(k)
            i += k
        assert i == n
        return req, pos

    def step_kv(self):
        """K/V rows of this step's tokens, (max_num_tokens, H_kv, D); padding rows are 0."""
        mx = self.max_num_tokens
        k = np.zeros((mx, self.num_kv_heads, self.head_dim), self.np_dtype)
        v = np.zeros_like(k)
        i = 0
        for r in range(self.num_rows):
            cnt = int(self.new_tokens[r])
            if cnt:
                p0 = int(self.prior_lens[r])
                k[i:i + cnt], v[i:i + cnt] = self.kv_rows(r, p0, p0 + cnt)
            i += cnt
        return k, v

    def prior_tokens(self, rows=None):
        """Tokens already in the cache before this step, for the given rows (default all)."""
        rows = range(self.num_rows) if rows is None else rows
        reqs, poss = [], []
        for r in rows:
            p = int(self.prior_lens[r])
            reqs.append(np.full(p, r, np.int32))
            poss.append(np.arange(p, dtype=np.int64))
        if not reqs:
            return np.zeros(0, np.int32), np.zeros(0, np.int64)
        return np.concatenate(reqs), np.concatenate(poss)


def cp_block_tables(w: Workload, world: int, slack: float = 0.25):
    """Per-rank kernel-block tables for splitting ``w``'s cache over ``world``
    context-parallel ranks: rank k draws its own seeded permutation of physical
    ids 1..total-1 and gives every request as many blocks as its unsplit row
    needs (more than any rank's share), so each rank's cache holds whichever
    positions the split gives it.  Returns [(table int32 (rows, width), total)]."""
    kbs = w.kernel_block_size
    needed = np.array([_ceil_div(int(n), kbs) for n in w.context_lens], np.int64)
    width = max(int(needed.max()) if len(needed) else 0, 1) + 1
    out = []
    for k in range(world):
        rng = np.random.default_rng([w.seed, 11, k])
        out.append(_assign_blocks(rng, needed, width, slack))
    return out


def _assign_blocks(rng, needed: np.ndarray, width: int, slack: float = 0.25):
    """Random distinct physical ids 1..total-1 for each row's needed blocks; -1 elsewhere."""
    total_needed = int(needed.sum())
    total_blocks = 1 + total_needed + int(math.ceil(slack * total_needed))
    ids = rng.permutation(np.arange(1, total_blocks, dtype=np.int64))[:total_needed]
    table = np.full((len(needed), width), -1, np.int32)
    k = 0
    for r, n in enumerate(needed):
        n = int(n)
        table[r, :n] = ids[k:k + n]
        k += n
    return table, total_blocks


def _ceil_div(a, b):
    return -(-np.asarray(a, dtype=np.int64) // b)


def _qk(s: float, sharp: bool, loud: bool) -> float:
    """Scale of the drawn Q and K values: s (the recipe), 1 (sharp) or sqrt(2) (loud)."""
    return math.sqrt(2.0) if loud else (1.0 if sharp else s)


def make(name: str, *, sharp: bool = False, loud: bool = False, tiny_reading: str = "record") -> Workload:
    """Draw workload ``name`` with its fixed seed (``sharp`` / ``loud``: the test variants above)."""
    if name not in WORKLOADS:
        raise KeyError(name)
    if sharp and loud:
        raise ValueError("sharp and loud are different variants")
    seed = SEEDS[name]
    rng = np.random.default_rng(seed)

    if name == "tiny":
        # context lengths {3, 7}; the record reading counts the decode token on top
        # (cache lengths 4 and 8); the other reading takes 3 and 7 as cache lengths.
        ctx = np.array([3, 7], np.int64)
        prior = ctx if tiny_reading == "record" else ctx - 1
        new = np.ones(2, np.int64)
        bs, width, total = 4, 4, 16
        needed = _ceil_div(prior + new, bs)
        ids = rng.permutation(np.arange(1, total, dtype=np.int64))[: int(needed.sum())]
        table = np.full((2, width), -1, np.int32)
        k = 0
        for r, n in enumerate(needed):
            table[r, :n] = ids[k:k + n]
            k += int(n)
        return Workload(name, seed, "f32", 2, 2, 1, 2, 1, 8, bs, bs, prior, new, table, total,
                        max_num_tokens=4, qk_scale=1.0, v_scale=1.0)

    if name == "llama3_decode":
        nr, bs, d = 32, 64, 128
        prior = rng.integers(512, 4096, size=nr, endpoint=True).astype(np.int64)
        new = np.ones(nr, np.int64)
        width = int(_ceil_div(4096 + 1, bs))
        table, total = _assign_blocks(rng, _ceil_div(prior + new, bs), width)
        s = 1.0 / math.sqrt(d)
        return Workload(name, seed, "bf16", nr, nr, 1, 32, 8, d, bs, bs, prior, new, table, total,
                        max_num_tokens=nr, qk_scale=_qk(s, sharp, loud), v_scale=1.0 if loud else s)

    if name == "ragged_step":
        nr, bs, d = 64, 16, 128
        prior = rng.integers(0, 2048, size=nr, endpoint=True).astype(np.int64)
        new = np.ones(nr, np.int64)
        multi = rng.choice(nr, size=16, replace=False)
        new[multi] = rng.integers(64, 1024, size=16, endpoint=True)
        width = 192
        table, total = _assign_blocks(rng, _ceil_div(prior + new, bs), width)
        n = int(new.sum())
        max_tokens = int(_ceil_div(n, 1024) * 1024)  # slot buffer sized for reuse, tail padded
        s = 1.0 / math.sqrt(d)
        return Workload(name, seed, "bf16", nr, nr, 0, 32, 8, d, bs, bs, prior, new, table, total,
                        max_num_tokens=max_tokens, qk_scale=_qk(s, sharp, loud), v_scale=1.0 if loud else s,
                        has_decode=False)

    if name == "long_context":
        nr, bs, d, max_model_len = 8, 64, 128, 131072
        prior = np.rint(rng.lognormal(mean=math.log(4096), sigma=1.0, size=nr)).astype(np.int64)
        prior = np.clip(prior, 256, max_model_len - 1)
        new = np.ones(nr, np.int64)
        width = max_model_len // bs
        table, total = _assign_blocks(rng, _ceil_div(prior + new, bs), width)
        s = 1.0 / math.sqrt(d)
        return Workload(name, seed, "bf16", nr, nr, 1, 64, 8, d, bs, bs, prior, new, table, total,
                        max_num_tokens=nr, qk_scale=_qk(s, sharp, loud), v_scale=1.0 if loud else s,
                        extra={"max_model_len": max_model_len, "buckets": [4096, 8192, 16384]})

    # hybrid_spec
    real, pad, mbs, kbs, d, q_len = 256, 64, 32, 16, 128, 4
    nr = real + pad
    prior = np.zeros(nr, np.int64)
    prior[:real] = np.clip(rng.zipf(1.1, size=real), 1, 8192)
    new = np.zeros(nr, np.int64)
    new[:real] = q_len
    width = int(_ceil_div(8192 + q_len, mbs))
    table, total = _assign_blocks(rng, _ceil_div(prior + new, mbs), width)
    s = 1.0 / math.sqrt(d)
    return Workload(name, seed, "bf16", nr, real, q_len, 32, 8, d, mbs, kbs, prior, new, table, total,
                    max_num_tokens=nr * q_len, qk_scale=_qk(s, sharp, loud), v_scale=1.0 if loud else s)
