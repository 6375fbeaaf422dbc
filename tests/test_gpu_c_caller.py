"""The hot path from a plain C program written against the boundary's own
argument lists (tests/c/sec8b_caller.c declares the five calls by hand, with
no bkv.h): block expansion, slot mapping, cache write, workspace sizing and
the decode, on a hybrid-block-size batch with multi-token queries and a NULL
row.  Its results must be the oracle's: the kernel table and the slots bit
for bit, the attention within the parity bars (tests/_parity.py).

The CPU test only compiles and links the program (nvcc cross-compiles
without a GPU); the GPU test runs it."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from _parity import check_attention
from oracle.cases import fill_oracle_cache
from paged_kv_cache_slot_gb300 import build as bkv_build
from paged_kv_cache_slot_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c", "sec8b_caller.c")


def _nvcc():
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    return None


def _compile(tmp_path):
    """gcc (plain C11), the CUDA runtime from the toolkit that builds the library, and libbkv.so."""
    lib = bkv_build.build()
    cuda = os.path.dirname(os.path.dirname(os.path.realpath(_nvcc())))
    exe = str(tmp_path / "sec8b_caller")
    libdir = os.path.dirname(lib)
    cudalib = os.path.join(cuda, "lib64")
    p = subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(cuda, "include"), SRC, "-o", exe,
                        "-L", libdir, "-lbkv", "-L", cudalib, "-lcudart", "-Wl,-rpath," + libdir,
                        "-Wl,-rpath," + cudalib], capture_output=True, text=True)
    assert p.returncode == 0, p.stderr
    return exe


@pytest.mark.skipif(_nvcc() is None or shutil.which("gcc") is None, reason="gcc and the CUDA toolkit are needed")
def test_sec8b_caller_compiles_and_links(tmp_path):
    assert os.path.exists(_compile(tmp_path))


def _workload():
    """Manager blocks of 32 split into kernel blocks of 16, 4 query tokens, a NULL row, loud values."""
    prior = np.array([700, 3, 1500, 0, 260], np.int64)
    new = np.array([4, 4, 4, 0, 4], np.int64)
    mbs, kbs = 32, 16
    need = -(-(prior + new) // mbs)
    rng = np.random.default_rng(2024)
    total = 1 + int(need.sum()) + 6
    ids = rng.permutation(np.arange(1, total))[: int(need.sum())]
    table = np.full((len(prior), int(need.max()) + 2), -1, np.int32)
    k = 0
    for r, n in enumerate(need):
        table[r, :n] = ids[k:k + n]
        k += int(n)
    return wl.Workload("c_caller", 2024, "bf16", 5, 4, 4, 32, 8, 128, mbs, kbs, prior, new, table, total,
                       max_num_tokens=int(new.sum()), qk_scale=np.sqrt(2.0), v_scale=1.0)


@pytest.mark.gpu
@pytest.mark.skipif(_nvcc() is None or shutil.which("gcc") is None, reason="gcc and the CUDA toolkit are needed")
def test_sec8b_caller_matches_the_oracle(tmp_path):
    exe = _compile(tmp_path)
    w = _workload()
    L = w.context_lens
    rows = [r for r in range(w.num_rows) if L[r] > 0]
    req = np.concatenate([np.full(int(L[r]), r, np.int32) for r in rows])
    pos = np.concatenate([np.arange(int(L[r]), dtype=np.int64) for r in rows])
    kv = [w.kv_rows(r, 0, int(L[r])) for r in rows]
    k_new = np.concatenate([a for a, _ in kv])
    v_new = np.concatenate([b for _, b in kv])
    T = len(pos)
    max_tokens = T + 5                                   # a padded tail, written as -1
    q = w.q()
    sizes = np.array([w.num_rows, w.width, w.block_size, w.kernel_block_size, T, max_tokens, w.num_q_heads,
                      w.num_kv_heads, w.head_dim, w.q_len, w.total_blocks, 0, int(L.max()), 0, 0, 0], np.int64)
    parts = [sizes, w.block_table, req, pos, k_new, v_new, q, L]
    with open(tmp_path / "in.bin", "wb") as f:
        for a in parts:
            b = np.ascontiguousarray(a).tobytes()
            f.write(b + b"\0" * (-len(b) % 8))
    p = subprocess.run([exe, str(tmp_path / "in.bin"), str(tmp_path / "out.bin")], capture_output=True, text=True,
                       timeout=120)
    assert p.returncode == 0, p.stdout + p.stderr
    raw = open(tmp_path / "out.bin", "rb").read()
    bpk = w.blocks_per_kv_block
    n_kt = w.num_rows * w.width * bpk
    kt = np.frombuffer(raw, np.int32, n_kt).reshape(w.num_rows, -1)
    slots = np.frombuffer(raw, np.int64, max_tokens, offset=4 * n_kt)
    out_off = 4 * n_kt + 8 * max_tokens
    out = np.frombuffer(raw, np.uint16, q.size, offset=out_off).reshape(q.shape)
    err = int(np.frombuffer(raw, np.int32, 1, offset=out_off + 2 * q.size)[0])

    want_kt = oracle.map_to_kernel_blocks(w.block_table, w.block_size, w.kernel_block_size)
    assert np.array_equal(kt, want_kt)
    want_slots, serr = oracle.compute_slot_mapping(want_kt, req, pos, w.kernel_block_size, T, max_tokens)
    assert np.array_equal(slots, want_slots) and serr == 0
    kc, vc, table = fill_oracle_cache(w)
    want, derr = oracle.paged_decode(q, kc, vc, table, L)
    assert err == 0 and derr == 0
    got = wl.bf16_bits_to_f32(out).astype(np.float64)
    check_attention(got, want, "bf16", "C caller", min_magnitude=0.1)
    assert (got[3] == 0).all()                           # the NULL row
