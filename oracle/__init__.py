"""CPU oracle for the paged (block) KV cache hot path -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline legs of
``bench.py`` may import this package.  The product library never loads it and
shares no code with it.  The arithmetic lives in ``bkv_oracle.c`` (plain C,
fp64); this module builds it with gcc and marshals numpy arrays through ctypes.

Functions and the passages they follow (page titles and sections):

* :func:`compute_slot_mapping` -- "Padding and Batching with Block KV",
  Slot Mapping / The Core Formula and Slot Mapping Computation; Special Block
  and Slot Values; "ブロック表" 設計動機 (the -1 tail).
* :func:`map_to_kernel_blocks` -- "ブロック表" 設計動機 and 境界と失敗.
* :func:`cache_write` -- "Padding and Batching with Block KV", Block
  Structure and Slot ID -1: Padding Tokens.
* :func:`paged_decode` / :func:`paged_decode_request` -- "Padding and
  Batching with Block KV", Cache Masking (mask_cache, mask_active).
* :func:`decode_bucket` -- "Decode Context-Length Bucketing", Design /
  Per-step bucket selection (used to report bytes only).
* :func:`paged_attention_ragged` -- the decode's attention over a mixed
  step with per-request query counts ("Padding and Batching with Block KV",
  Batching with Block KV; reading R15 of the C source).
* :func:`compute_slot_mapping_cp`, :func:`paged_decode_cp`,
  :func:`merge_attn_states` -- "ブロック表" 設計動機 (DCP / PCP interleave:
  a rank writes real slots only for the tokens it owns); the ownership,
  local-position and merge readings are R14 of the C source.
* :func:`e4m3_encode`, :func:`e4m3_decode`, :func:`cache_write_fp8`,
  :func:`paged_decode_fp8` -- the FP8 (E4M3) KV cache: "Padding and Batching
  with Block KV", Block ID 0 vs. Sentinel -1 names a non-FP8 pathway, nothing
  more; the format and per-tensor scale convention are reading R16 of the C
  source.

Every function is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_*.py`` against worked values printed on the pages, brute
force, closed forms and a library routine (torch SDPA in fp64).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bkv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

DT_BF16 = 0
DT_F32 = 1
DT_E4M3 = 2

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile ``bkv_oracle.c`` into ``liboracle.so`` (gcc, -O2, portable)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    # -ffp-contract=off: no fused multiply-adds, so every product and sum is
    # rounded to fp64 exactly as written.
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i32, i64, vp, dbl = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_double
            lib.orc_compute_slot_mapping.restype = i64
            lib.orc_compute_slot_mapping.argtypes = [vp, i32, i64, i32, vp, vp, i64, i64, i32, vp]
            lib.orc_map_to_kernel_blocks.restype = ctypes.c_int
            lib.orc_map_to_kernel_blocks.argtypes = [vp, i32, i64, i32, i32, i32, vp, i64]
            lib.orc_cache_write.restype = i64
            lib.orc_cache_write.argtypes = [vp, vp, i64, i64, vp, vp, vp, i64, i32, i32, i32, ctypes.c_int]
            dec = [vp, vp, vp, vp, i64, i32, vp, i32, i32, i32, i32, i32, i32, i64, dbl, ctypes.c_int, i32,
                   ctypes.c_int, vp]
            lib.orc_paged_decode.restype = i64
            lib.orc_paged_decode.argtypes = dec
            lib.orc_paged_decode_request.restype = i64
            lib.orc_paged_decode_request.argtypes = [i32] + dec
            lib.orc_compute_slot_mapping_cp.restype = i64
            lib.orc_compute_slot_mapping_cp.argtypes = [vp, i32, i64, i32, vp, vp, i64, i64, i32, i32, i32, i32, vp]
            lib.orc_paged_decode_cp_request.restype = i64
            lib.orc_paged_decode_cp_request.argtypes = [i32, vp, vp, vp, vp, i64, i32, vp, i32, i32, i32, i32, i32,
                                                        i32, i64, dbl, ctypes.c_int, i32, i32, i32, i32,
                                                        ctypes.c_int, vp, vp]
            lib.orc_paged_attention_ragged.restype = i64
            lib.orc_paged_attention_ragged.argtypes = [vp, vp, vp, vp, vp, i64, i32, vp, i32, i64, i32, i32, i32, i32,
                                                       i64, dbl, ctypes.c_int, ctypes.c_int, vp]
            lib.orc_merge_attn_states.restype = ctypes.c_int
            lib.orc_merge_attn_states.argtypes = [vp, vp, i32, i64, i32, vp, vp]
            lib.orc_e4m3_decode.restype = dbl
            lib.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.orc_e4m3_encode_array.restype = None
            lib.orc_e4m3_encode_array.argtypes = [vp, i64, vp]
            lib.orc_cache_write_fp8.restype = i64
            lib.orc_cache_write_fp8.argtypes = [vp, vp, i64, i64, vp, vp, vp, i64, i32, i32, i32, ctypes.c_int,
                                                ctypes.c_float, ctypes.c_float]
            lib.orc_paged_decode_fp8_request.restype = i64
            lib.orc_paged_decode_fp8_request.argtypes = [i32, vp, vp, vp, vp, i64, i32, vp, i32, i32, i32, i32, i32,
                                                         i32, i64, dbl, dbl, dbl, ctypes.c_int, i32, ctypes.c_int,
                                                         vp]
            lib.orc_decode_bucket.restype = i64
            lib.orc_decode_bucket.argtypes = [vp, i64, i64, vp, i64, i64]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=dtype))


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.uint16:
        return DT_BF16  # bf16 bit patterns
    if a.dtype == np.float32:
        return DT_F32
    raise TypeError(f"oracle takes bf16 bit patterns (uint16) or float32, got {a.dtype}")


def compute_slot_mapping(block_table, req_indices, positions, block_size, num_tokens=None, max_num_tokens=None):
    """Slot ids (int64, length ``max_num_tokens``) and the count of bad tokens."""
    bt = _c(block_table, np.int32)
    if bt.ndim != 2:
        raise ValueError("block_table must be 2-D")
    req = _c(req_indices, np.int32)
    pos = _c(positions, np.int64)
    n = len(pos) if num_tokens is None else int(num_tokens)
    mx = n if max_num_tokens is None else int(max_num_tokens)
    if len(req) < n or len(pos) < n:
        raise ValueError("req_indices/positions shorter than num_tokens")
    out = np.empty(max(mx, 1), np.int64)
    err = _load().orc_compute_slot_mapping(_ptr(bt), bt.shape[0], bt.shape[1], bt.shape[1], _ptr(req), _ptr(pos),
                                           n, mx, int(block_size), _ptr(out))
    if err < 0:
        raise ValueError("invalid slot-mapping arguments")
    return out[:mx], int(err)


def compute_slot_mapping_cp(block_table, req_indices, positions, block_size, cp_world, cp_rank, cp_interleave,
                            num_tokens=None, max_num_tokens=None):
    """Slot ids of rank ``cp_rank`` under decode context parallelism (reading R14) and the bad-token count."""
    bt = _c(block_table, np.int32)
    if bt.ndim != 2:
        raise ValueError("block_table must be 2-D")
    req = _c(req_indices, np.int32)
    pos = _c(positions, np.int64)
    n = len(pos) if num_tokens is None else int(num_tokens)
    mx = n if max_num_tokens is None else int(max_num_tokens)
    out = np.empty(max(mx, 1), np.int64)
    err = _load().orc_compute_slot_mapping_cp(_ptr(bt), bt.shape[0], bt.shape[1], bt.shape[1], _ptr(req),
                                              _ptr(pos), n, mx, int(block_size), int(cp_world), int(cp_rank),
                                              int(cp_interleave), _ptr(out))
    if err < 0:
        raise ValueError("invalid slot-mapping arguments")
    return out[:mx], int(err)


def map_to_kernel_blocks(mgr_table, block_size, kernel_block_size):
    """Kernel-block table (rows, mgr_cols * bs/kbs) int32; ValueError if bs % kbs."""
    m = _c(mgr_table, np.int32)
    if int(kernel_block_size) <= 0 or int(block_size) % int(kernel_block_size):
        raise ValueError("block_size must be a multiple of kernel_block_size")
    bpk = int(block_size) // int(kernel_block_size)
    out = np.zeros((m.shape[0], m.shape[1] * bpk), np.int32)
    rc = _load().orc_map_to_kernel_blocks(_ptr(m), m.shape[0], m.shape[1], m.shape[1], int(block_size),
                                          int(kernel_block_size), _ptr(out), out.shape[1])
    if rc != 0:
        raise ValueError("invalid map_to_kernel_blocks arguments")
    return out


def cache_write(k_new, v_new, slot_mapping, k_cache, v_cache, num_tokens=None, inplace=False):
    """Scatter rows into copies of the caches (or into the caches themselves when
    ``inplace``); returns (k_cache, v_cache, errors).

    ``k_new``/``v_new`` are (num_tokens, H_kv, D); caches are
    (total_blocks, block_size, H_kv, D), all bf16 bits (uint16) or float32.
    """
    if inplace:
        if not (k_cache.flags.c_contiguous and v_cache.flags.c_contiguous):
            raise ValueError("in-place cache_write needs C-contiguous caches")
        kc, vc = k_cache, v_cache
    else:
        kc = np.array(k_cache, copy=True, order="C")
        vc = np.array(v_cache, copy=True, order="C")
    kn = np.ascontiguousarray(k_new)
    vn = np.ascontiguousarray(v_new)
    dt = _dtype_code(kc)
    if not (kn.dtype == vn.dtype == kc.dtype == vc.dtype):
        raise TypeError("mixed dtypes")
    sl = _c(slot_mapping, np.int64)
    n = kn.shape[0] if num_tokens is None else int(num_tokens)
    tb, bs, hkv, d = kc.shape
    err = _load().orc_cache_write(_ptr(kn), _ptr(vn), n, hkv * d, _ptr(sl), _ptr(kc), _ptr(vc), tb, bs, hkv, d, dt)
    if err == -2:
        raise ValueError("duplicate non-negative slot ids")
    if err < 0:
        raise ValueError("invalid cache_write arguments")
    return kc, vc, int(err)


def _decode_args(q, k_cache, v_cache, block_table, context_lens, scale, mask_mode, sliding_window=0):
    qa = np.ascontiguousarray(q)
    kc = np.ascontiguousarray(k_cache)
    vc = np.ascontiguousarray(v_cache)
    dt = _dtype_code(kc)
    if not (qa.dtype == kc.dtype == vc.dtype):
        raise TypeError("mixed dtypes")
    bt = _c(block_table, np.int32)
    cl = _c(context_lens, np.int32)
    nr, ql, hq, d = qa.shape
    tb, bs, hkv, d2 = kc.shape
    if d2 != d:
        raise ValueError("head_dim mismatch")
    sc = (1.0 / np.sqrt(d)) if scale is None else float(scale)
    args = (_ptr(qa), _ptr(kc), _ptr(vc), _ptr(bt), bt.shape[1], bt.shape[1], _ptr(cl), nr, ql, hq, hkv, d, bs, tb,
            sc, int(mask_mode), int(sliding_window), dt)
    return args, (qa, kc, vc, bt, cl), (nr, ql, hq, d)


def paged_decode(q, k_cache, v_cache, block_table, context_lens, scale=None, mask_mode=0, sliding_window=0):
    """fp64 attention output (num_reqs, q_len, H_q, D) and the bad-entry count.

    ``sliding_window`` W > 0: query t of a request of length L sees only keys
    j >= L - q_len + t - W + 1 (reading R13 of the C source)."""
    args, keep, shape = _decode_args(q, k_cache, v_cache, block_table, context_lens, scale, mask_mode,
                                     sliding_window)
    out = np.zeros(shape, np.float64)
    err = _load().orc_paged_decode(*args, _ptr(out))
    if err < 0:
        raise ValueError("invalid paged_decode arguments")
    del keep
    return out, int(err)


def paged_decode_request(r, q, k_cache, v_cache, block_table, context_lens, scale=None, mask_mode=0,
                         sliding_window=0):
    """fp64 output of request ``r`` only, (q_len, H_q, D)."""
    args, keep, shape = _decode_args(q, k_cache, v_cache, block_table, context_lens, scale, mask_mode,
                                     sliding_window)
    out = np.zeros(shape, np.float64)
    err = _load().orc_paged_decode_request(int(r), *args, _ptr(out))
    if err < 0:
        raise ValueError("invalid paged_decode arguments")
    del keep
    return out[r], int(err)


def paged_decode_cp(q, k_cache, v_cache, block_table, context_lens, cp_world=1, cp_rank=0, cp_interleave=1,
                    scale=None, mask_mode=0, sliding_window=0, rows=None):
    """Rank ``cp_rank``'s decode over its own keys (reading R14; context_lens are global lengths).

    Returns fp64 out (num_reqs, q_len, H_q, D), lse (num_reqs, q_len, H_q) (natural log of the sum of
    exp of the scaled scores over the visible keys, -inf where none) and the bad-entry count; ``rows``
    limits the work to those requests (the others stay 0 / -inf)."""
    args, keep, shape = _decode_args(q, k_cache, v_cache, block_table, context_lens, scale, mask_mode,
                                     sliding_window)
    out = np.zeros(shape, np.float64)
    lse = np.full(shape[:3], -np.inf, np.float64)
    err = 0
    lib = _load()
    base, tail = args[:-2], args[-1]   # everything up to the mask / window, then dtype
    for r in (range(shape[0]) if rows is None else rows):
        e = lib.orc_paged_decode_cp_request(int(r), *base, int(sliding_window), int(cp_world), int(cp_rank),
                                            int(cp_interleave), tail, _ptr(out), _ptr(lse))
        if e < 0:
            raise ValueError("invalid paged_decode_cp arguments")
        err += e
    del keep
    return out, lse, int(err)


def paged_attention_ragged(q, query_start_loc, k_cache, v_cache, block_table, context_lens, scale=None,
                           mask_mode=0):
    """fp64 attention of a mixed step (reading R15): q packed (num_tokens, H_q, D), request r's tokens at
    [query_start_loc[r], query_start_loc[r+1]) ending at position context_lens[r] - 1.  Returns (out, errors)."""
    qa = np.ascontiguousarray(q)
    kc = np.ascontiguousarray(k_cache)
    vc = np.ascontiguousarray(v_cache)
    if not (qa.dtype == kc.dtype == vc.dtype):
        raise TypeError("mixed dtypes")
    dt = _dtype_code(kc)
    qsl = _c(query_start_loc, np.int32)
    bt = _c(block_table, np.int32)
    cl = _c(context_lens, np.int32)
    nt, hq, d = qa.shape
    tb, bs, hkv, d2 = kc.shape
    if d2 != d or len(qsl) != len(cl) + 1:
        raise ValueError("shape mismatch")
    sc = (1.0 / np.sqrt(d)) if scale is None else float(scale)
    out = np.zeros((nt, hq, d), np.float64)
    err = _load().orc_paged_attention_ragged(_ptr(qa), _ptr(qsl), _ptr(kc), _ptr(vc), _ptr(bt), bt.shape[1],
                                             bt.shape[1], _ptr(cl), len(cl), nt, hq, hkv, d, bs, tb, sc,
                                             int(mask_mode), dt, _ptr(out))
    if err < 0:
        raise ValueError("invalid paged_attention_ragged arguments")
    return out, int(err)


def merge_attn_states(outs, lses):
    """Merge of partial attention results (R14): outs (parts, rows, D), lses (parts, rows) -> (out, lse)."""
    o = np.ascontiguousarray(outs, np.float64)
    l = np.ascontiguousarray(lses, np.float64)
    parts, rows, d = o.shape
    if l.shape != (parts, rows):
        raise ValueError("lses must be (parts, rows)")
    out = np.zeros((rows, d), np.float64)
    lse = np.zeros(rows, np.float64)
    if _load().orc_merge_attn_states(_ptr(o), _ptr(l), parts, rows, d, _ptr(out), _ptr(lse)) != 0:
        raise ValueError("invalid merge arguments")
    return out, lse


def e4m3_decode(codes):
    """float64 values of E4M3 codes (uint8 array; NaN for 0x7F / 0xFF), reading R16."""
    c = np.asarray(codes, np.uint8)
    lib = _load()
    table = np.array([lib.orc_e4m3_decode(i) for i in range(256)], np.float64)
    return table[c]


def e4m3_encode(x):
    """E4M3 codes (uint8) of float32 values: nearest, ties to even, saturating at 448, NaN -> 0x7F (R16)."""
    xa = np.ascontiguousarray(np.asarray(x, np.float32))
    out = np.empty(xa.shape, np.uint8)
    _load().orc_e4m3_encode_array(_ptr(xa), xa.size, _ptr(out))
    return out


def cache_write_fp8(k_new, v_new, slot_mapping, k_cache, v_cache, k_scale, v_scale, num_tokens=None,
                    inplace=False):
    """Scatter bf16 (uint16 bits) / float32 rows into E4M3 caches (uint8, (total_blocks, bs, H_kv, D)), each
    element stored as the code of float32(x) / float32(scale) (reading R16).  Returns (k_cache, v_cache,
    errors)."""
    if inplace:
        if not (k_cache.flags.c_contiguous and v_cache.flags.c_contiguous):
            raise ValueError("in-place cache_write_fp8 needs C-contiguous caches")
        kc, vc = k_cache, v_cache
    else:
        kc = np.array(k_cache, copy=True, order="C")
        vc = np.array(v_cache, copy=True, order="C")
    if kc.dtype != np.uint8 or vc.dtype != np.uint8:
        raise TypeError("FP8 caches are uint8 codes")
    kn = np.ascontiguousarray(k_new)
    vn = np.ascontiguousarray(v_new)
    if kn.dtype != vn.dtype:
        raise TypeError("mixed dtypes")
    dt = _dtype_code(kn)
    sl = _c(slot_mapping, np.int64)
    n = kn.shape[0] if num_tokens is None else int(num_tokens)
    tb, bs, hkv, d = kc.shape
    err = _load().orc_cache_write_fp8(_ptr(kn), _ptr(vn), n, hkv * d, _ptr(sl), _ptr(kc), _ptr(vc), tb, bs, hkv,
                                      d, dt, float(k_scale), float(v_scale))
    if err == -2:
        raise ValueError("duplicate non-negative slot ids")
    if err < 0:
        raise ValueError("invalid cache_write_fp8 arguments")
    return kc, vc, int(err)


def paged_decode_fp8(q, k_cache, v_cache, block_table, context_lens, k_scale, v_scale, scale=None, mask_mode=0,
                     sliding_window=0, rows=None):
    """fp64 decode over E4M3 caches (uint8 codes; key value = code value * k_scale, value = * v_scale,
    reading R16); q is bf16 bits (uint16) or float32.  ``rows`` limits the work to those requests (the others
    stay 0).  Returns (out, errors)."""
    qa = np.ascontiguousarray(q)
    kc = np.ascontiguousarray(k_cache)
    vc = np.ascontiguousarray(v_cache)
    if kc.dtype != np.uint8 or vc.dtype != np.uint8:
        raise TypeError("FP8 caches are uint8 codes")
    dt = _dtype_code(qa)
    bt = _c(block_table, np.int32)
    cl = _c(context_lens, np.int32)
    nr, ql, hq, d = qa.shape
    tb, bs, hkv, d2 = kc.shape
    if d2 != d:
        raise ValueError("head_dim mismatch")
    sc = (1.0 / np.sqrt(d)) if scale is None else float(scale)
    out = np.zeros((nr, ql, hq, d), np.float64)
    err = 0
    lib = _load()
    for r in (range(nr) if rows is None else rows):
        e = lib.orc_paged_decode_fp8_request(int(r), _ptr(qa), _ptr(kc), _ptr(vc), _ptr(bt), bt.shape[1],
                                             bt.shape[1], _ptr(cl), nr, ql, hq, hkv, d, bs, tb, sc, float(k_scale),
                                             float(v_scale), int(mask_mode), int(sliding_window), dt, _ptr(out))
        if e < 0:
            raise ValueError("invalid paged_decode_fp8 arguments")
        err += e
    return out, int(err)


def decode_bucket(num_computed, num_speculative_tokens, buckets, max_model_len):
    """Smallest bucket >= max(num_computed) + 1 + spec, else max_model_len (or -1)."""
    nc = _c(num_computed, np.int64)
    bk = _c(buckets, np.int64)
    return int(_load().orc_decode_bucket(_ptr(nc), len(nc), int(num_speculative_tokens), _ptr(bk), len(bk),
                                         int(max_model_len)))
