"""The oracle's view of a seeded workload: host caches filled by the oracle's
own slot mapping and cache write.  TEST INFRASTRUCTURE, like the rest of
this package; it calls only the oracle and the seeded input generators."""
import numpy as np

from . import cache_write, cache_write_fp8, compute_slot_mapping, compute_slot_mapping_cp, map_to_kernel_blocks
from paged_kv_cache_slot_gb300 import workloads as wl

BF16_NAN = np.uint16(0x7FC0)
E4M3_NAN = np.uint8(0x7F)


def nan_cache(w: wl.Workload, total_blocks=None, block_size=None, sparse=False):
    """NaN-filled host caches; ``sparse`` leaves them uninitialised instead, so
    that the pages of a large cache are only committed where rows are written
    (the oracle never reads anything else)."""
    tb = w.total_kernel_blocks if total_blocks is None else total_blocks
    bs = w.kernel_block_size if block_size is None else block_size
    shape = (tb, bs, w.num_kv_heads, w.head_dim)
    if sparse:
        return np.empty(shape, w.np_dtype)
    if w.dtype == "bf16":
        return np.full(shape, BF16_NAN, np.uint16)
    return np.full(shape, np.nan, np.float32)


def kernel_table(w: wl.Workload):
    if w.kernel_block_size == w.block_size:
        return w.block_table.copy()
    return map_to_kernel_blocks(w.block_table, w.block_size, w.kernel_block_size)


def fill_oracle_cache(w: wl.Workload, rows=None, kcache=None, vcache=None, table=None):
    """Write every token (prior and this step's) of ``rows`` into NaN-poisoned
    caches through the oracle.  Returns (k_cache, v_cache, kernel_table)."""
    table = kernel_table(w) if table is None else table
    sparse = w.total_kernel_blocks * w.kernel_block_size * w.num_kv_heads * w.head_dim * w.elem_bytes > (256 << 20)
    kc = nan_cache(w, sparse=sparse) if kcache is None else kcache
    vc = nan_cache(w, sparse=sparse) if vcache is None else vcache
    rows = range(w.num_rows) if rows is None else rows
    for r in rows:
        L = int(w.context_lens[r])
        if L == 0:
            continue
        k, v = w.kv_rows(r, 0, L)
        req = np.full(L, r, np.int32)
        pos = np.arange(L, dtype=np.int64)
        slots, err = compute_slot_mapping(table, req, pos, w.kernel_block_size)
        assert err == 0
        kc, vc, err = cache_write(k, v, slots, kc, vc, inplace=True)
        assert err == 0
    return kc, vc, table


def fill_oracle_cache_cp(w: wl.Workload, world: int, interleave: int, tables, rows=None):
    """Each context-parallel rank's caches, written through the oracle's CP slot
    mapping (reading R14) and cache write from every token of ``rows``;
    ``tables`` are the ranks' (table, total_blocks) pairs.  Returns [(k, v)]."""
    rows = range(w.num_rows) if rows is None else rows
    out = []
    for k, (table, total) in enumerate(tables):
        kc = nan_cache(w, total_blocks=total)
        vc = nan_cache(w, total_blocks=total)
        for r in rows:
            L = int(w.context_lens[r])
            if L == 0:
                continue
            kr, vr = w.kv_rows(r, 0, L)
            req = np.full(L, r, np.int32)
            pos = np.arange(L, dtype=np.int64)
            slots, err = compute_slot_mapping_cp(table, req, pos, w.kernel_block_size, world, k, interleave)
            assert err == 0
            kc, vc, err = cache_write(kr, vr, slots, kc, vc, inplace=True)
            assert err == 0
        out.append((kc, vc))
    return out


def fill_oracle_cache_fp8(w: wl.Workload, k_scale: float, v_scale: float, rows=None, table=None):
    """E4M3 caches (uint8 codes, unwritten bytes the NaN code 0x7F) holding every
    token of ``rows``, written through the oracle's slot mapping and FP8 cache
    write (reading R16).  Returns (k_cache, v_cache, kernel_table)."""
    table = kernel_table(w) if table is None else table
    shape = (w.total_kernel_blocks, w.kernel_block_size, w.num_kv_heads, w.head_dim)
    kc = np.full(shape, E4M3_NAN, np.uint8)
    vc = np.full(shape, E4M3_NAN, np.uint8)
    rows = range(w.num_rows) if rows is None else rows
    for r in rows:
        L = int(w.context_lens[r])
        if L == 0:
            continue
        k, v = w.kv_rows(r, 0, L)
        req = np.full(L, r, np.int32)
        pos = np.arange(L, dtype=np.int64)
        slots, err = compute_slot_mapping(table, req, pos, w.kernel_block_size)
        assert err == 0
        kc, vc, err = cache_write_fp8(k, v, slots, kc, vc, k_scale, v_scale, inplace=True)
        assert err == 0
    return kc, vc, table
