"""Device staging of a seeded workload for the GPU tests and the benchmark.

Uploads a :class:`~paged_kv_cache_slot_gb300.workloads.Workload` and fills
the paged caches with every request's prior tokens THROUGH THE LIBRARY
(slot mapping + cache write kernels), exactly as a serving step would have
written them.  Caches start as NaN so that any read of a position that was
never written shows up in the output.

``DeviceWorkload.step()`` is one pass of the hot path over one batch:
block expansion (manager -> kernel ids), slot mapping of this step's tokens
and the K/V scatter (one fused kernel, or the two calls), and the paged
decode (partition + merge kernels).
"""
from __future__ import annotations

import numpy as np
import torch

from . import bkv
from .workloads import Workload
from .workloads import cp_block_tables as wl_cp_tables

PRIOR_FILL_TOKENS = 1 << 16  # tokens uploaded per prior-fill batch


def _t(a: np.ndarray, device, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.to(device)


class DeviceWorkload:
    def __init__(self, w: Workload, device="cuda", background: str = "nan", fill_prior: bool = True,
                 sliding_window: int = 0, cp_world: int = 1, cp_rank: int = 0, cp_interleave: int = 1,
                 kv_fp8=None, fused_write: bool = True, prior_values: str = "host"):
        self.w = w
        # values of the prior tokens: "host" draws the workload's own (what the oracle sees); "device"
        # draws N(0, 1) with the workload's scales on the GPU (seeded), for timing runs that compare
        # nothing with the oracle and would otherwise spend their time generating values on the host
        if prior_values not in ("host", "device"):
            raise ValueError("prior_values must be 'host' or 'device'")
        self.prior_values = prior_values
        # the step's slot mapping + cache write as one bkv_slot_mapping_cache_write(_fp8) call (without
        # context parallelism), else the two calls
        self.fused_write = bool(fused_write)
        self.window = int(sliding_window)   # decode's default sliding window (0: full attention)
        # FP8 (E4M3) caches: (k_scale, v_scale); new rows are quantised by the cache write
        self.fp8 = None if kv_fp8 is None else (float(kv_fp8[0]), float(kv_fp8[1]))
        if self.fp8 is not None and int(cp_world) > 1:
            raise ValueError("FP8 caches are not combined with context parallelism here")
        # decode context parallelism: this object is rank cp_rank of cp_world, holding only its
        # share of every request's tokens in a cache of its own (block_size == kernel block size)
        self.cp = (int(cp_world), int(cp_rank), int(cp_interleave))
        if self.cp[0] > 1 and w.block_size != w.kernel_block_size:
            raise ValueError("context-parallel staging needs block_size == kernel_block_size")
        self.device = torch.device(device)
        dev = self.device
        self.tdtype = torch.bfloat16 if w.dtype == "bf16" else torch.float32
        if self.cp[0] > 1:
            table, total = wl_cp_tables(w, self.cp[0])[self.cp[1]]
        else:
            table, total = w.block_table, w.total_kernel_blocks
        kshape = (total, w.kernel_block_size, w.num_kv_heads, w.head_dim)
        if self.fp8 is not None:
            code = 0x7F if background == "nan" else 0   # 0x7F: the E4M3 NaN code
            self.k_cache = torch.full(kshape, code, dtype=torch.uint8, device=dev)
            self.v_cache = torch.full(kshape, code, dtype=torch.uint8, device=dev)
        else:
            fill = float("nan") if background == "nan" else 0.0
            self.k_cache = torch.full(kshape, fill, dtype=self.tdtype, device=dev)
            self.v_cache = torch.full(kshape, fill, dtype=self.tdtype, device=dev)
        self.mgr_table = _t(table, dev)
        self.kernel_table = torch.empty((w.num_rows, table.shape[1] * w.blocks_per_kv_block), dtype=torch.int32,
                                        device=dev)
        bkv.bkv_map_to_kernel_blocks(self.mgr_table, w.block_size, w.kernel_block_size, self.kernel_table)
        self.context_lens = _t(w.context_lens, dev)
        self.max_context_len = int(w.context_lens.max()) if w.num_rows else 0
        req, pos = w.step_tokens()
        self.req_indices = _t(req, dev)
        self.positions = _t(pos, dev)
        self.slot_mapping = torch.empty(w.max_num_tokens, dtype=torch.int64, device=dev)
        kn, vn = w.step_kv()
        self.k_new = _t(kn, dev, self.tdtype if w.dtype == "bf16" else None)
        self.v_new = _t(vn, dev, self.tdtype if w.dtype == "bf16" else None)
        self.err_count = torch.zeros(1, dtype=torch.int32, device=dev)
        if w.has_decode:
            self.q = _t(w.q(), dev, self.tdtype if w.dtype == "bf16" else None)
            self.out = torch.empty_like(self.q)
            self.lse = torch.empty(self.q.shape[:3], dtype=torch.float32, device=dev)
            self.workspace = bkv.alloc_workspace(w.num_rows, w.q_len, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                                 w.kernel_block_size, self.max_context_len, device=dev)
        if fill_prior:
            self.fill_prior()

    # -- prior context ------------------------------------------------------
    def fill_prior(self, rows=None):
        """Write prior tokens of ``rows`` (default all) through slot mapping + cache write."""
        w, dev = self.w, self.device
        rows = list(range(w.num_rows)) if rows is None else list(rows)
        batch: list[int] = []
        ntok = 0
        for r in rows + [None]:
            if r is not None and int(w.prior_lens[r]) == 0:
                continue
            if r is None or (batch and ntok + int(w.prior_lens[r]) > PRIOR_FILL_TOKENS):
                if batch:
                    self._write_rows(batch)
                batch, ntok = [], 0
            if r is not None:
                batch.append(r)
                ntok += int(w.prior_lens[r])
        torch.cuda.synchronize(dev)

    def _write_rows(self, rows):
        w, dev = self.w, self.device
        req, pos = w.prior_tokens(rows)
        if self.prior_values == "device":
            g = torch.Generator(device=dev)
            g.manual_seed(int(w.seed) * 1000003 + int(rows[0]))
            shape = (len(pos), w.num_kv_heads, w.head_dim)
            kt = (torch.randn(shape, generator=g, device=dev) * w.qk_scale).to(self.tdtype)
            vt = (torch.randn(shape, generator=g, device=dev) * w.v_scale).to(self.tdtype)
        else:
            ks, vs = zip(*(w.kv_rows(r, 0, int(w.prior_lens[r])) for r in rows))
            k = np.concatenate(ks)
            v = np.concatenate(vs)
            cast = self.tdtype if w.dtype == "bf16" else None
            kt, vt = _t(k, dev, cast), _t(v, dev, cast)
        slots = torch.empty(len(pos), dtype=torch.int64, device=dev)
        self._slots(self.kernel_table, _t(req, dev), _t(pos, dev), slots)
        self._write(kt, vt, slots)

    def _write(self, k, v, slots, num_tokens=None, stream=None):
        if self.fp8 is not None:
            bkv.bkv_cache_write_fp8(k, v, slots, self.k_cache, self.v_cache, *self.fp8, num_tokens=num_tokens,
                                    err_count=self.err_count, stream=stream)
        else:
            bkv.bkv_cache_write(k, v, slots, self.k_cache, self.v_cache, num_tokens=num_tokens,
                                err_count=self.err_count, stream=stream)

    # -- the hot path ---------------------------------------------------------
    def expand_blocks(self, stream=None):
        w = self.w
        bkv.bkv_map_to_kernel_blocks(self.mgr_table, w.block_size, w.kernel_block_size, self.kernel_table,
                                     stream=stream)

    def _slots(self, table, req, pos, slots, num_tokens=None, stream=None):
        w = self.w
        if self.cp[0] > 1:
            bkv.bkv_compute_slot_mapping_cp(table, req, pos, w.kernel_block_size, slots, *self.cp,
                                            num_tokens=num_tokens, err_count=self.err_count, stream=stream)
        else:
            bkv.bkv_compute_slot_mapping(table, req, pos, w.kernel_block_size, slots, num_tokens=num_tokens,
                                         err_count=self.err_count, stream=stream)

    def write_step(self, stream=None, fused=None):
        """Slot mapping + cache write of this step's tokens: one fused call where it applies (``fused``
        None: the object's default), else the two calls."""
        w = self.w
        fused = self.fused_write if fused is None else fused
        if fused and self.cp[0] == 1:
            args = (self.kernel_table, self.req_indices, self.positions, self.slot_mapping, self.k_new, self.v_new,
                    self.k_cache, self.v_cache)
            if self.fp8 is not None:
                bkv.bkv_slot_mapping_cache_write_fp8(*args, *self.fp8, num_tokens=w.num_tokens,
                                                     err_count=self.err_count, stream=stream)
            else:
                bkv.bkv_slot_mapping_cache_write(*args, num_tokens=w.num_tokens, err_count=self.err_count,
                                                 stream=stream)
            return
        self._slots(self.kernel_table, self.req_indices, self.positions, self.slot_mapping, w.num_tokens, stream)
        self._write(self.k_new, self.v_new, self.slot_mapping, w.num_tokens, stream)

    def decode(self, stream=None, out=None, table=None, mask_mode=bkv.BKV_MASK_CAUSAL, sliding_window=None):
        out = self.out if out is None else out
        sliding_window = self.window if sliding_window is None else sliding_window
        table = self.kernel_table if table is None else table
        if self.cp[0] > 1:
            bkv.bkv_paged_decode_cp(self.q, self.k_cache, self.v_cache, table, self.context_lens,
                                    self.max_context_len, out, self.lse, self.workspace, *self.cp, mask_mode=mask_mode,
                                    err_count=self.err_count, stream=stream)
            return out
        if self.fp8 is not None:
            bkv.bkv_paged_decode_fp8(self.q, self.k_cache, self.v_cache, table, self.context_lens,
                                     self.max_context_len, out, self.workspace, *self.fp8, mask_mode=mask_mode,
                                     err_count=self.err_count, stream=stream, sliding_window=sliding_window)
            return out
        if sliding_window:
            bkv.bkv_paged_decode_swa(self.q, self.k_cache, self.v_cache, table, self.context_lens,
                                     self.max_context_len, out, self.workspace, sliding_window, mask_mode=mask_mode,
                                     err_count=self.err_count, stream=stream)
        else:
            bkv.bkv_paged_decode(self.q, self.k_cache, self.v_cache, table, self.context_lens, self.max_context_len,
                                 out, self.workspace, mask_mode=mask_mode, err_count=self.err_count, stream=stream)
        return out

    def decode_partition(self, stream=None):
        """Phase 1 of the decode alone (the partition kernel), for timing."""
        if self.fp8 is not None:
            bkv.bkv_paged_decode_fp8_partition(self.q, self.k_cache, self.v_cache, self.kernel_table,
                                               self.context_lens, self.max_context_len, self.out, self.workspace,
                                               *self.fp8, err_count=self.err_count, stream=stream,
                                               sliding_window=self.window)
            return
        bkv.bkv_paged_decode_partition(self.q, self.k_cache, self.v_cache, self.kernel_table, self.context_lens,
                                       self.max_context_len, self.out, self.workspace, err_count=self.err_count,
                                       stream=stream, sliding_window=self.window)

    def step(self, stream=None):
        """One pass of the whole path: a2 -> a1 -> a3 -> a4 + a5."""
        self.expand_blocks(stream)
        self.write_step(stream)
        if self.w.has_decode:
            self.decode(stream)

    # -- byte accounting (algorithmic, token granularity) ---------------------
    def decode_kv_bytes(self) -> int:
        """K and V bytes the decode must read: cache_len rows per request and KV head (with a
        sliding window W, only the rows from the first query's window start, L - q_len - W + 1; with
        context parallelism, only the rows this rank holds)."""
        w = self.w
        L = w.context_lens.astype(np.int64)
        if self.window > 0:
            L = L - np.maximum(0, L - w.q_len - self.window + 1)
        if self.cp[0] > 1:
            W, k, inter = self.cp
            cyc = inter * W
            L = (L // cyc) * inter + np.clip(L % cyc - k * inter, 0, inter)
        return int(L.sum()) * 2 * w.num_kv_heads * w.head_dim * self.cache_elem_bytes()

    def cache_elem_bytes(self) -> int:
        return 1 if self.fp8 is not None else self.w.elem_bytes

    def write_bytes(self) -> int:
        """Cache-write traffic: new K/V rows read + written, plus the slot ids."""
        w = self.w
        return w.num_tokens * (2 * w.num_kv_heads * w.head_dim * (w.elem_bytes + self.cache_elem_bytes()) + 8)
