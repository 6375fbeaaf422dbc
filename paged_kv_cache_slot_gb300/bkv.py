"""Thin Python binding of libbkv.so (ctypes).

Argument marshalling only: each function checks the tensors' device, dtype,
shape and contiguity, passes their device pointers and the current CUDA
stream to the C entry point of the same name, and raises :class:`BkvError`
on a non-zero status.  Every step of the path runs in the library's kernels;
there is no fallback of any kind.  If libbkv.so is missing or cannot be
loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

from . import build as _build

BKV_OK, BKV_ERR_INVALID_ARG, BKV_ERR_UNSUPPORTED, BKV_ERR_CUDA = 0, 1, 2, 3
BKV_BF16, BKV_F32 = 0, 1
BKV_MASK_CAUSAL, BKV_MASK_ALL = 0, 1

LIB_PATH = _build.LIB

_lib = None
_lock = threading.Lock()


class BkvError(RuntimeError):
    def __init__(self, fn: str, status: int):
        lib = load()
        msg = lib.bkv_status_string(status).decode()
        if status == BKV_ERR_CUDA:
            msg += ": " + lib.bkv_last_cuda_error().decode()
        super().__init__(f"{fn} -> status {status} ({msg})")
        self.status = status


def load() -> ctypes.CDLL:
    """Load libbkv.so (built in-tree by ``build()``); raise if it is absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libbkv.so not found at {LIB_PATH}: run paged_kv_cache_slot_gb300.build.build() "
                               "(there is no fallback path)")
        lib = ctypes.CDLL(LIB_PATH)
        i32, i64, vp, sz, f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_float
        cint = ctypes.c_int
        lib.bkv_status_string.restype = ctypes.c_char_p
        lib.bkv_status_string.argtypes = [cint]
        lib.bkv_last_cuda_error.restype = ctypes.c_char_p
        lib.bkv_last_cuda_error.argtypes = []
        lib.bkv_version.restype = ctypes.c_char_p
        lib.bkv_version.argtypes = []
        lib.bkv_compute_slot_mapping.restype = cint
        lib.bkv_compute_slot_mapping.argtypes = [vp, i32, i64, i32, vp, vp, i64, i64, i32, vp, vp, vp]
        lib.bkv_compute_slot_mapping_cp.restype = cint
        lib.bkv_compute_slot_mapping_cp.argtypes = [vp, i32, i64, i32, vp, vp, i64, i64, i32, i32, i32, i32, vp, vp,
                                                    vp]
        lib.bkv_paged_decode_cp.restype = cint
        lib.bkv_paged_decode_cp.argtypes = [vp, vp, vp, vp, i64, i32, vp, i32, i32, i32, i32, i32, i32, i32, i64, f32,
                                            cint, i32, i32, i32, cint, vp, vp, vp, sz, vp, vp]
        lib.bkv_paged_attention_ragged.restype = cint
        lib.bkv_paged_attention_ragged.argtypes = [vp, vp, vp, vp, vp, i64, i32, vp, i32, i32, i32, i64, i32, i32,
                                                   i32, i32, i64, f32, cint, cint, vp, vp, vp]
        lib.bkv_merge_attn_states.restype = cint
        lib.bkv_merge_attn_states.argtypes = [vp, vp, i32, i64, i32, cint, vp, vp, vp]
        lib.bkv_map_to_kernel_blocks.restype = cint
        lib.bkv_map_to_kernel_blocks.argtypes = [vp, i32, i64, i32, i32, i32, vp, i64, vp]
        lib.bkv_cache_write.restype = cint
        lib.bkv_cache_write.argtypes = [vp, vp, i64, i64, vp, vp, vp, i64, i32, i32, i32, cint, vp, vp]
        lib.bkv_slot_mapping_cache_write_fp8.restype = cint
        lib.bkv_slot_mapping_cache_write_fp8.argtypes = [vp, i32, i64, i32, vp, vp, i64, i64, vp, vp, vp, i64, vp,
                                                         vp, i64, i32, i32, i32, cint, f32, f32, vp, vp]
        lib.bkv_slot_mapping_cache_write.restype = cint
        lib.bkv_slot_mapping_cache_write.argtypes = [vp, i32, i64, i32, vp, vp, i64, i64, vp, vp, vp, i64, vp, vp,
                                                     i64, i32, i32, i32, cint, vp, vp]
        lib.bkv_paged_decode_workspace_size.restype = sz
        lib.bkv_paged_decode_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, i32]
        dec = [vp, vp, vp, vp, i64, i32, vp, i32, i32, i32, i32, i32, i32, i32, i64, f32, cint, i32, cint, vp, vp, sz,
               vp, vp]
        for fn in ("bkv_paged_decode_swa", "bkv_paged_decode_partition", "bkv_paged_decode_merge"):
            getattr(lib, fn).restype = cint
            getattr(lib, fn).argtypes = dec
        # the boundary's own form: no sliding_window argument
        lib.bkv_paged_decode.restype = cint
        lib.bkv_paged_decode.argtypes = dec[:17] + dec[18:]
        lib.bkv_paged_decode_noalloc.restype = cint
        lib.bkv_paged_decode_noalloc.argtypes = dec[:17] + [cint, vp, vp, vp]
        lib.bkv_cache_write_fp8.restype = cint
        lib.bkv_cache_write_fp8.argtypes = [vp, vp, i64, i64, vp, vp, vp, i64, i32, i32, i32, cint, f32, f32, vp, vp]
        dec8 = [vp, vp, vp, vp, i64, i32, vp, i32, i32, i32, i32, i32, i32, i32, i64, f32, f32, f32, cint, i32, cint,
                vp, vp, sz, vp, vp]
        for fn in ("bkv_paged_decode_fp8", "bkv_paged_decode_fp8_partition", "bkv_paged_decode_fp8_merge"):
            getattr(lib, fn).restype = cint
            getattr(lib, fn).argtypes = dec8
        _lib = lib
        return lib


def _check(fn: str, status: int):
    if status != BKV_OK:
        raise BkvError(fn, status)


def _stream(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _dev(t: torch.Tensor, name: str, dtype=None, contiguous=True):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _opt(t, name, dtype):
    return None if t is None else _dev(t, name, dtype)


def _kv_dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BKV_BF16
    if t.dtype == torch.float32:
        return BKV_F32
    raise TypeError(f"KV/Q tensors must be bfloat16 or float32, got {t.dtype}")


def bkv_compute_slot_mapping(block_table, req_indices, positions, block_size, slot_mapping, num_tokens=None,
                             err_count=None, stream=None):
    """slot_mapping[i] = block_table[req, pos // bs] * bs + pos % bs, -1 for padding (see include/bkv.h)."""
    return _slot_mapping("bkv_compute_slot_mapping", (), block_table, req_indices, positions, block_size,
                         slot_mapping, num_tokens, err_count, stream)


def bkv_compute_slot_mapping_cp(block_table, req_indices, positions, block_size, slot_mapping, cp_world, cp_rank,
                                cp_interleave=1, num_tokens=None, err_count=None, stream=None):
    """Rank ``cp_rank``'s slots under decode context parallelism, -1 for other ranks' tokens (see include/bkv.h)."""
    return _slot_mapping("bkv_compute_slot_mapping_cp", (int(cp_world), int(cp_rank), int(cp_interleave)),
                         block_table, req_indices, positions, block_size, slot_mapping, num_tokens, err_count, stream)


def _slot_mapping(fn, cp, block_table, req_indices, positions, block_size, slot_mapping, num_tokens, err_count,
                  stream):
    if block_table.dim() != 2 or block_table.stride(1) != 1:
        raise ValueError("block_table must be 2-D with unit column stride")
    n = positions.numel() if num_tokens is None else int(num_tokens)
    if n > positions.numel() or n > req_indices.numel() or n > slot_mapping.numel():
        raise ValueError("num_tokens exceeds positions / req_indices / slot_mapping")
    _check(fn, getattr(load(), fn)(
        _dev(block_table, "block_table", torch.int32, contiguous=False), block_table.shape[0],
        block_table.stride(0), block_table.shape[1], _dev(req_indices, "req_indices", torch.int32),
        _dev(positions, "positions", torch.int64), n, slot_mapping.numel(), int(block_size), *cp,
        _dev(slot_mapping, "slot_mapping", torch.int64), _opt(err_count, "err_count", torch.int32), _stream(stream)))
    return slot_mapping


def bkv_map_to_kernel_blocks(mgr_table, block_size, kernel_block_size, kernel_table, stream=None):
    """Expand manager block ids into kernel block ids m * bpk + t (see include/bkv.h)."""
    if mgr_table.dim() != 2 or kernel_table.dim() != 2 or mgr_table.stride(1) != 1 or kernel_table.stride(1) != 1:
        raise ValueError("tables must be 2-D with unit column stride")
    if kernel_table.shape[0] != mgr_table.shape[0]:
        raise ValueError("row count mismatch")
    _check("bkv_map_to_kernel_blocks", load().bkv_map_to_kernel_blocks(
        _dev(mgr_table, "mgr_table", torch.int32, contiguous=False), mgr_table.shape[0], mgr_table.stride(0),
        mgr_table.shape[1], int(block_size), int(kernel_block_size),
        _dev(kernel_table, "kernel_table", torch.int32, contiguous=False), kernel_table.stride(0), _stream(stream)))
    return kernel_table


def bkv_cache_write(k_new, v_new, slot_mapping, k_cache, v_cache, num_tokens=None, err_count=None, stream=None):
    """Scatter k_new/v_new rows (num_tokens, H_kv, D) into the caches at slot_mapping (see include/bkv.h)."""
    dt = _check_kv_rows(k_new, v_new, k_cache, v_cache)
    tb, bs, hkv, d = k_cache.shape
    n = k_new.shape[0] if num_tokens is None else int(num_tokens)
    if n > k_new.shape[0] or n > slot_mapping.numel():
        raise ValueError("num_tokens exceeds k_new / slot_mapping")
    _check("bkv_cache_write", load().bkv_cache_write(
        _dev(k_new, "k_new", contiguous=False), _dev(v_new, "v_new", contiguous=False), n, k_new.stride(0),
        _dev(slot_mapping, "slot_mapping", torch.int64), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"), tb, bs,
        hkv, d, dt, _opt(err_count, "err_count", torch.int32), _stream(stream)))


def bkv_slot_mapping_cache_write(block_table, req_indices, positions, slot_mapping, k_new, v_new, k_cache, v_cache,
                                 num_tokens=None, err_count=None, stream=None):
    """bkv_compute_slot_mapping then bkv_cache_write in one kernel, with the same results; the caches'
    block size is the table's (see include/bkv.h)."""
    if block_table.dim() != 2 or block_table.stride(1) != 1:
        raise ValueError("block_table must be 2-D with unit column stride")
    dt = _check_kv_rows(k_new, v_new, k_cache, v_cache)
    tb, bs, hkv, d = k_cache.shape
    n = positions.numel() if num_tokens is None else int(num_tokens)
    if n > positions.numel() or n > req_indices.numel() or n > slot_mapping.numel() or n > k_new.shape[0]:
        raise ValueError("num_tokens exceeds positions / req_indices / slot_mapping / k_new")
    _check("bkv_slot_mapping_cache_write", load().bkv_slot_mapping_cache_write(
        _dev(block_table, "block_table", torch.int32, contiguous=False), block_table.shape[0],
        block_table.stride(0), block_table.shape[1], _dev(req_indices, "req_indices", torch.int32),
        _dev(positions, "positions", torch.int64), n, slot_mapping.numel(),
        _dev(slot_mapping, "slot_mapping", torch.int64), _dev(k_new, "k_new", contiguous=False),
        _dev(v_new, "v_new", contiguous=False), k_new.stride(0), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
        tb, bs, hkv, d, dt, _opt(err_count, "err_count", torch.int32), _stream(stream)))
    return slot_mapping


def bkv_slot_mapping_cache_write_fp8(block_table, req_indices, positions, slot_mapping, k_new, v_new, k_cache,
                                     v_cache, k_scale, v_scale, num_tokens=None, err_count=None, stream=None):
    """bkv_compute_slot_mapping then bkv_cache_write_fp8 in one kernel, with the same results: k_new / v_new
    (num_tokens, H_kv, D) bf16 or fp32 quantised into uint8 E4M3 caches (see include/bkv.h)."""
    if block_table.dim() != 2 or block_table.stride(1) != 1:
        raise ValueError("block_table must be 2-D with unit column stride")
    dt = _check_kv_rows(k_new, v_new, k_cache, v_cache, fp8=True)
    tb, bs, hkv, d = k_cache.shape
    n = positions.numel() if num_tokens is None else int(num_tokens)
    if n > positions.numel() or n > req_indices.numel() or n > slot_mapping.numel() or n > k_new.shape[0]:
        raise ValueError("num_tokens exceeds positions / req_indices / slot_mapping / k_new")
    _check("bkv_slot_mapping_cache_write_fp8", load().bkv_slot_mapping_cache_write_fp8(
        _dev(block_table, "block_table", torch.int32, contiguous=False), block_table.shape[0],
        block_table.stride(0), block_table.shape[1], _dev(req_indices, "req_indices", torch.int32),
        _dev(positions, "positions", torch.int64), n, slot_mapping.numel(),
        _dev(slot_mapping, "slot_mapping", torch.int64), _dev(k_new, "k_new", contiguous=False),
        _dev(v_new, "v_new", contiguous=False), k_new.stride(0), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
        tb, bs, hkv, d, dt, float(k_scale), float(v_scale), _opt(err_count, "err_count", torch.int32),
        _stream(stream)))
    return slot_mapping


def _check_kv_rows(k_new, v_new, k_cache, v_cache, fp8=False):
    """Shape, layout and dtype checks shared by the cache writes; returns the dtype code of the rows.

    Caches (total_blocks, block_size, H_kv, D), equal in shape: bf16 / fp32 like the rows, or uint8 E4M3
    codes when ``fp8``.  Rows (num_tokens, H_kv, D), dense within a row (a row stride is allowed)."""
    if k_cache.dim() != 4 or k_cache.shape != v_cache.shape:
        raise ValueError("caches must be (total_blocks, block_size, H_kv, D) and equal in shape")
    _, _, hkv, d = k_cache.shape
    if k_new.dim() != 3 or tuple(k_new.shape[1:]) != (hkv, d) or k_new.shape != v_new.shape:
        raise ValueError("k_new/v_new must be (num_tokens, H_kv, D) matching the cache")
    if k_new.stride(2) != 1 or k_new.stride(1) != d or k_new.stride() != v_new.stride():
        raise ValueError("k_new/v_new rows must be dense (a row stride is allowed)")
    if fp8:
        if k_cache.dtype != torch.uint8 or v_cache.dtype != torch.uint8:
            raise TypeError("FP8 caches are uint8 tensors of E4M3 codes")
        if k_new.dtype != v_new.dtype:
            raise TypeError("mixed dtypes")
        return _kv_dtype(k_new)
    if k_new.dtype != k_cache.dtype or v_new.dtype != k_cache.dtype or v_cache.dtype != k_cache.dtype:
        raise TypeError("mixed dtypes")
    return _kv_dtype(k_cache)


def bkv_cache_write_fp8(k_new, v_new, slot_mapping, k_cache, v_cache, k_scale, v_scale, num_tokens=None,
                        err_count=None, stream=None):
    """Quantise k_new/v_new rows (num_tokens, H_kv, D; bf16 or fp32) into uint8 E4M3 caches at slot_mapping
    with per-tensor scales (see include/bkv.h)."""
    dt = _check_kv_rows(k_new, v_new, k_cache, v_cache, fp8=True)
    tb, bs, hkv, d = k_cache.shape
    n = k_new.shape[0] if num_tokens is None else int(num_tokens)
    if n > k_new.shape[0] or n > slot_mapping.numel():
        raise ValueError("num_tokens exceeds k_new / slot_mapping")
    _check("bkv_cache_write_fp8", load().bkv_cache_write_fp8(
        _dev(k_new, "k_new", contiguous=False), _dev(v_new, "v_new", contiguous=False), n, k_new.stride(0),
        _dev(slot_mapping, "slot_mapping", torch.int64), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"), tb, bs,
        hkv, d, dt, float(k_scale), float(v_scale), _opt(err_count, "err_count", torch.int32), _stream(stream)))


def bkv_paged_decode_workspace_size(num_reqs, q_len, num_q_heads, num_kv_heads, head_dim, block_size,
                                    max_context_len) -> int:
    return int(load().bkv_paged_decode_workspace_size(int(num_reqs), int(q_len), int(num_q_heads),
                                                      int(num_kv_heads), int(head_dim), int(block_size),
                                                      int(max_context_len)))


def bkv_paged_decode(q, k_cache, v_cache, block_table, context_lens, max_context_len, out, workspace,
                     softmax_scale=0.0, mask_mode=BKV_MASK_CAUSAL, err_count=None, stream=None):
    """GQA paged decode attention into ``out`` (num_reqs, q_len, H_q, D) (see include/bkv.h)."""
    return _decode("bkv_paged_decode", q, k_cache, v_cache, block_table, context_lens, max_context_len, out,
                   workspace, softmax_scale, mask_mode, None, err_count, stream)


def bkv_paged_decode_swa(q, k_cache, v_cache, block_table, context_lens, max_context_len, out, workspace,
                         sliding_window, softmax_scale=0.0, mask_mode=BKV_MASK_CAUSAL, err_count=None, stream=None):
    """bkv_paged_decode of a sliding-window layer: query t sees the last ``sliding_window`` positions up to its
    own (0: full attention) (see include/bkv.h)."""
    return _decode("bkv_paged_decode_swa", q, k_cache, v_cache, block_table, context_lens, max_context_len, out,
                   workspace, softmax_scale, mask_mode, sliding_window, err_count, stream)


def bkv_paged_decode_noalloc(q, k_cache, v_cache, block_table, context_lens, max_context_len, out,
                             softmax_scale=0.0, mask_mode=BKV_MASK_CAUSAL, err_count=None, stream=None):
    """bkv_paged_decode with its scratch in the library's fixed device array instead of a workspace (see
    include/bkv.h)."""
    return _decode("bkv_paged_decode_noalloc", q, k_cache, v_cache, block_table, context_lens, max_context_len, out,
                   False, softmax_scale, mask_mode, None, err_count, stream)


def bkv_paged_decode_partition(q, k_cache, v_cache, block_table, context_lens, max_context_len, out, workspace,
                               softmax_scale=0.0, mask_mode=BKV_MASK_CAUSAL, err_count=None, stream=None,
                               sliding_window=0):
    """Phase 1 of bkv_paged_decode: split-KV partials into ``workspace`` (see include/bkv.h)."""
    return _decode("bkv_paged_decode_partition", q, k_cache, v_cache, block_table, context_lens, max_context_len,
                   out, workspace, softmax_scale, mask_mode, sliding_window, err_count, stream)


def bkv_paged_decode_merge(q, k_cache, v_cache, block_table, context_lens, max_context_len, out, workspace,
                           softmax_scale=0.0, mask_mode=BKV_MASK_CAUSAL, err_count=None, stream=None,
                           sliding_window=0):
    """Phase 2 of bkv_paged_decode: merge the workspace partials into ``out`` (see include/bkv.h)."""
    return _decode("bkv_paged_decode_merge", q, k_cache, v_cache, block_table, context_lens, max_context_len, out,
                   workspace, softmax_scale, mask_mode, sliding_window, err_count, stream)


def _decode(fn, q, k_cache, v_cache, block_table, context_lens, max_context_len, out, workspace, softmax_scale,
            mask_mode, sliding_window, err_count, stream, scales=None):
    if q.dim() != 4 or out.shape != q.shape or k_cache.dim() != 4 or k_cache.shape != v_cache.shape:
        raise ValueError("q/out must be (num_reqs, q_len, H_q, D); caches (total_blocks, bs, H_kv, D)")
    nr, ql, hq, d = q.shape
    tb, bs, hkv, d2 = k_cache.shape
    if d2 != d:
        raise ValueError("head_dim mismatch")
    if block_table.dim() != 2 or block_table.shape[0] < nr or block_table.stride(1) != 1:
        raise ValueError("block_table must be (>= num_reqs, cols) with unit column stride")
    dt = _kv_dtype(q)
    cache_dtype = q.dtype if scales is None else torch.uint8
    for t, nm, want in ((k_cache, "k_cache", cache_dtype), (v_cache, "v_cache", cache_dtype), (out, "out", q.dtype)):
        if t.dtype != want:
            raise TypeError(f"{nm} must be {want}, got {t.dtype}")
    # workspace: a uint8 tensor, None (a null pointer), or False (the entry point takes none)
    if workspace is not None and workspace is not False and workspace.dtype != torch.uint8:
        raise TypeError("workspace must be a uint8 tensor")
    ws = ()
    if workspace is not False:
        ws = (None, 0) if workspace is None else (_dev(workspace, "workspace"), workspace.numel())
    window = () if sliding_window is None else (int(sliding_window),)
    _check(fn, getattr(load(), fn)(
        _dev(q, "q"), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
        _dev(block_table, "block_table", torch.int32, contiguous=False), block_table.stride(0),
        block_table.shape[1], _dev(context_lens, "context_lens", torch.int32), int(max_context_len), nr, ql, hq, hkv,
        d, bs, tb, float(softmax_scale), *(() if scales is None else (float(scales[0]), float(scales[1]))),
        int(mask_mode), *window, dt, _dev(out, "out"), *ws, _opt(err_count, "err_count", torch.int32),
        _stream(stream)))
    return out


def bkv_paged_decode_fp8(q, k_cache, v_cache, block_table, context_lens, max_context_len, out, workspace, k_scale,
                         v_scale, softmax_scale=0.0, mask_mode=BKV_MASK_CAUSAL, err_count=None, stream=None,
                         sliding_window=0):
    """bkv_paged_decode over uint8 E4M3 caches with per-tensor scales (see include/bkv.h)."""
    return _decode("bkv_paged_decode_fp8", q, k_cache, v_cache, block_table, context_lens, max_context_len, out,
                   workspace, softmax_scale, mask_mode, sliding_window, err_count, stream, scales=(k_scale, v_scale))


def bkv_paged_decode_fp8_partition(q, k_cache, v_cache, block_table, context_lens, max_context_len, out, workspace,
                                   k_scale, v_scale, softmax_scale=0.0, mask_mode=BKV_MASK_CAUSAL, err_count=None,
                                   stream=None, sliding_window=0):
    """Phase 1 of bkv_paged_decode_fp8 (see include/bkv.h)."""
    return _decode("bkv_paged_decode_fp8_partition", q, k_cache, v_cache, block_table, context_lens,
                   max_context_len, out, workspace, softmax_scale, mask_mode, sliding_window, err_count, stream,
                   scales=(k_scale, v_scale))


def bkv_paged_decode_fp8_merge(q, k_cache, v_cache, block_table, context_lens, max_context_len, out, workspace,
                               k_scale, v_scale, softmax_scale=0.0, mask_mode=BKV_MASK_CAUSAL, err_count=None,
                               stream=None, sliding_window=0):
    """Phase 2 of bkv_paged_decode_fp8 (see include/bkv.h)."""
    return _decode("bkv_paged_decode_fp8_merge", q, k_cache, v_cache, block_table, context_lens, max_context_len,
                   out, workspace, softmax_scale, mask_mode, sliding_window, err_count, stream,
                   scales=(k_scale, v_scale))


def bkv_paged_decode_cp(q, k_cache, v_cache, block_table, context_lens, max_context_len, out, lse, workspace,
                        cp_world, cp_rank, cp_interleave=1, softmax_scale=0.0, mask_mode=BKV_MASK_CAUSAL,
                        err_count=None, stream=None):
    """One rank's part of a context-parallel decode: its normalised ``out`` and fp32 ``lse`` (num_reqs, q_len,
    H_q) over the keys it holds; ``context_lens`` are global lengths (see include/bkv.h).  ``lse`` may be None."""
    if q.dim() != 4 or out.shape != q.shape or k_cache.dim() != 4 or k_cache.shape != v_cache.shape:
        raise ValueError("q/out must be (num_reqs, q_len, H_q, D); caches (total_blocks, bs, H_kv, D)")
    nr, ql, hq, d = q.shape
    tb, bs, hkv, d2 = k_cache.shape
    if d2 != d:
        raise ValueError("head_dim mismatch")
    if block_table.dim() != 2 or block_table.shape[0] < nr or block_table.stride(1) != 1:
        raise ValueError("block_table must be (>= num_reqs, cols) with unit column stride")
    if lse is not None and tuple(lse.shape) != (nr, ql, hq):
        raise ValueError("lse must be (num_reqs, q_len, H_q)")
    dt = _kv_dtype(q)
    for t, nm in ((k_cache, "k_cache"), (v_cache, "v_cache"), (out, "out")):
        if t.dtype != q.dtype:
            raise TypeError(f"{nm} dtype differs from q")
    ws_ptr = None if workspace is None else _dev(workspace, "workspace")
    ws_bytes = 0 if workspace is None else workspace.numel()
    _check("bkv_paged_decode_cp", load().bkv_paged_decode_cp(
        _dev(q, "q"), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
        _dev(block_table, "block_table", torch.int32, contiguous=False), block_table.stride(0),
        block_table.shape[1], _dev(context_lens, "context_lens", torch.int32), int(max_context_len), nr, ql, hq, hkv,
        d, bs, tb, float(softmax_scale), int(mask_mode), int(cp_world), int(cp_rank), int(cp_interleave), dt,
        _dev(out, "out"), _opt(lse, "lse", torch.float32), ws_ptr, ws_bytes, _opt(err_count, "err_count", torch.int32),
        _stream(stream)))
    return out, lse


def bkv_paged_attention_ragged(q, query_start_loc, k_cache, v_cache, block_table, context_lens, max_context_len,
                               max_query_len, out, softmax_scale=0.0, mask_mode=BKV_MASK_CAUSAL, err_count=None,
                               stream=None):
    """Attention over a mixed step: q / out packed (num_tokens, H_q, D), request r's tokens at
    [query_start_loc[r], query_start_loc[r+1]) (see include/bkv.h)."""
    if q.dim() != 3 or out.shape != q.shape or k_cache.dim() != 4 or k_cache.shape != v_cache.shape:
        raise ValueError("q/out must be (num_tokens, H_q, D); caches (total_blocks, bs, H_kv, D)")
    nt, hq, d = q.shape
    tb, bs, hkv, d2 = k_cache.shape
    nr = query_start_loc.numel() - 1
    if d2 != d or nr < 0 or context_lens.numel() < nr:
        raise ValueError("head_dim / query_start_loc / context_lens mismatch")
    if block_table.dim() != 2 or block_table.shape[0] < nr or block_table.stride(1) != 1:
        raise ValueError("block_table must be (>= num_reqs, cols) with unit column stride")
    dt = _kv_dtype(q)
    for t, nm in ((k_cache, "k_cache"), (v_cache, "v_cache"), (out, "out")):
        if t.dtype != q.dtype:
            raise TypeError(f"{nm} dtype differs from q")
    _check("bkv_paged_attention_ragged", load().bkv_paged_attention_ragged(
        _dev(q, "q"), _dev(query_start_loc, "query_start_loc", torch.int32), _dev(k_cache, "k_cache"),
        _dev(v_cache, "v_cache"), _dev(block_table, "block_table", torch.int32, contiguous=False),
        block_table.stride(0), block_table.shape[1], _dev(context_lens, "context_lens", torch.int32),
        int(max_context_len), int(max_query_len), nr, nt, hq, hkv, d, bs, tb, float(softmax_scale), int(mask_mode),
        dt, _dev(out, "out"), _opt(err_count, "err_count", torch.int32), _stream(stream)))
    return out


def bkv_merge_attn_states(outs, lses, out, lse_out=None, stream=None):
    """Merge ``parts`` partial results: outs (parts, rows, D), lses fp32 (parts, rows) -> out (rows, D) and
    optionally lse_out (rows) (see include/bkv.h).  Any leading shape with the same element count works."""
    parts = outs.shape[0]
    rows = lses[0].numel()
    d = outs.shape[-1]
    if outs.numel() != parts * rows * d or lses.numel() != parts * rows or out.numel() != rows * d:
        raise ValueError("outs (parts, rows, D), lses (parts, rows), out (rows, D) sizes disagree")
    if out.dtype != outs.dtype:
        raise TypeError("out dtype differs from outs")
    _check("bkv_merge_attn_states", load().bkv_merge_attn_states(
        _dev(outs, "outs"), _dev(lses, "lses", torch.float32), parts, rows, d, _kv_dtype(outs), _dev(out, "out"),
        _opt(lse_out, "lse_out", torch.float32), _stream(stream)))
    return out


def alloc_workspace(num_reqs, q_len, num_q_heads, num_kv_heads, head_dim, block_size, max_context_len, device=None):
    """Convenience: a uint8 device tensor of the size bkv_paged_decode needs."""
    n = bkv_paged_decode_workspace_size(num_reqs, q_len, num_q_heads, num_kv_heads, head_dim, block_size,
                                        max_context_len)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device or "cuda")


def default_scale(head_dim: int) -> float:
    return 1.0 / math.sqrt(head_dim)
