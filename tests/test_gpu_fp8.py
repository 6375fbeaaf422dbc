"""GPU parity for the FP8 (E4M3) KV cache against the fp64 oracle (reading
R16 of the oracle source: per-tensor scales, code = nearest to float32(x) /
scale with ties to even and saturation at 448, value = code value * scale).

* bkv_cache_write_fp8: every byte of both caches equals the oracle's, for
  bf16 and fp32 sources, 16-byte and element paths, a strided source,
  padding (-1) and out-of-range slots, NaN, saturating and subnormal inputs.
* bkv_paged_decode_fp8: per output row, max abs error <= 1e-2 (bf16 q / out)
  or 1e-5 (fp32) of the row's largest oracle value (tests/_parity.py; at
  least as tight as the absolute 1e-2 / 1e-5 for outputs up to 1), against
  the oracle on caches written by the library; unwritten cache bytes
  hold the NaN code 0x7F, so any read of them poisons the output; both mask
  modes, sliding windows, null entries inside a range, NULL rows; partition
  + merge equals the one call bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from _parity import check_attention
from oracle.cases import fill_oracle_cache_fp8
from paged_kv_cache_slot_gb300 import bkv
from paged_kv_cache_slot_gb300 import workloads as wl
from paged_kv_cache_slot_gb300.staging import DeviceWorkload

pytestmark = pytest.mark.gpu

K_SCALE = 2.0 ** -9
V_SCALE = 1e-3
NAN8 = 0x7F


def _f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def _custom(q_len, H_q, H_kv, D, bs, prior, dtype="bf16", seed=4242, null_rows=(), holes=(), qk=None, v=None):
    prior = np.array(prior, np.int64)
    nr = len(prior)
    new = np.full(nr, q_len, np.int64)
    for r in null_rows:
        prior[r] = 0
        new[r] = 0
    need = -(-(prior + new) // bs)
    width = int(need.max()) + 2
    rng = np.random.default_rng(seed)
    total = 1 + int(need.sum()) + 7
    ids = rng.permutation(np.arange(1, total))[: int(need.sum())]
    table = np.full((nr, width), -1, np.int32)
    k = 0
    for r, n in enumerate(need):
        table[r, :n] = ids[k:k + n]
        k += int(n)
    for r, lb in holes:
        table[r, lb] = 0
    s = 1.0 / np.sqrt(D)
    return wl.Workload("fp8", seed, dtype, nr, nr - len(null_rows), q_len, H_q, H_kv, D, bs, bs, prior, new, table,
                       total, max_num_tokens=int(new.sum()) + 3, qk_scale=s if qk is None else qk,
                       v_scale=s if v is None else v)


# ---------------------------------------------------------------------------
# cache write
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("shape", [(8, 128), (2, 12), (1, 8)])    # H_kv * D: 1024 (16-byte path), 24, 8
def test_cache_write_fp8_bytes_match_oracle(dtype, shape):
    hkv, d = shape
    rng = np.random.default_rng(11)
    n, tb, bs = 300, 40, 16
    cast = wl.f32_to_bf16_bits if dtype == "bf16" else (lambda x: x.astype(np.float32))
    # normal, saturating, subnormal and NaN inputs
    x = rng.standard_normal((2, n, hkv, d)).astype(np.float32) * np.float32(0.05)
    x[:, :20] *= np.float32(1e4)                                     # past 448 * scale: saturates
    x[:, 20:40] *= np.float32(1e-4)                                  # E4M3 subnormals and zeros
    x[0, 41, 0, 0] = np.nan
    x[1, 42, 0, d - 1] = -np.inf
    k, v = cast(x[0]), cast(x[1])
    slots = rng.permutation(tb * bs)[:n].astype(np.int64)
    slots[::7] = -1
    slots[5] = tb * bs + 3                                           # past the cache: skipped, counted
    kc0 = np.full((tb, bs, hkv, d), NAN8, np.uint8)
    want_k, want_v, want_err = oracle.cache_write_fp8(k, v, slots, kc0, kc0, K_SCALE, V_SCALE)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    kt = torch.from_numpy(k).view(tdt).cuda() if dtype == "bf16" else torch.from_numpy(k).cuda()
    vt = torch.from_numpy(v).view(tdt).cuda() if dtype == "bf16" else torch.from_numpy(v).cuda()
    kc = torch.full((tb, bs, hkv, d), NAN8, dtype=torch.uint8, device="cuda")
    vc = torch.full_like(kc, NAN8)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bkv.bkv_cache_write_fp8(kt, vt, torch.from_numpy(slots).cuda(), kc, vc, K_SCALE, V_SCALE, err_count=err)
    torch.cuda.synchronize()
    got_k, got_v = kc.cpu().numpy(), vc.cpu().numpy()
    assert int(err.item()) == want_err == 1
    for got, want in ((got_k, want_k), (got_v, want_v)):
        nan_g = (got & 0x7F) == 0x7F
        nan_w = (want & 0x7F) == 0x7F
        assert (nan_g == nan_w).all()
        assert (got[~nan_w] == want[~nan_w]).all()


def test_cache_write_fp8_strided_source_and_num_tokens():
    hkv, d, n = 8, 128, 64
    rng = np.random.default_rng(2)
    fused = torch.from_numpy(rng.standard_normal((n, 3, hkv, d)).astype(np.float32) * 0.05).cuda().to(torch.bfloat16)
    k, v = fused[:, 1], fused[:, 2]                                   # row stride 3 * hkv * d
    slots = torch.arange(n, dtype=torch.int64, device="cuda") * 2
    kc = torch.full((16, 16, hkv, d), NAN8, dtype=torch.uint8, device="cuda")
    vc = torch.full_like(kc, NAN8)
    bkv.bkv_cache_write_fp8(k, v, slots, kc, vc, K_SCALE, V_SCALE, num_tokens=40)
    torch.cuda.synchronize()
    kh = k.contiguous().view(torch.uint16).cpu().numpy()
    vh = v.contiguous().view(torch.uint16).cpu().numpy()
    want_k, want_v, _ = oracle.cache_write_fp8(kh, vh, slots.cpu().numpy(), np.full(kc.shape, NAN8, np.uint8),
                                               np.full(kc.shape, NAN8, np.uint8), K_SCALE, V_SCALE, num_tokens=40)
    assert (kc.cpu().numpy() == want_k).all()
    assert (vc.cpu().numpy() == want_v).all()


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("shape", [(8, 128), (2, 12)])            # 16-byte path, element path
def test_fused_slot_write_fp8_matches_oracle_and_two_calls(dtype, shape):
    """bkv_slot_mapping_cache_write_fp8: slots, E4M3 cache bytes and the error count equal the oracle's
    slot mapping followed by its quantising write, and the library's two calls, with padded requests, a
    padded tail, null entries, bad request indices and positions, a block id past the cache, and
    saturating, subnormal and NaN inputs."""
    hkv, d = shape
    rng = np.random.default_rng(23)
    nr, cols, bs, tb = 11, 6, 16, 70
    table = rng.permutation(np.arange(1, nr * cols + 10))[: nr * cols].astype(np.int32).reshape(nr, cols)
    table[rng.random(table.shape) < 0.1] = 0                      # null entries; some ids >= tb: counted
    pairs = rng.permutation(nr * cols * bs)[:250]
    req = (pairs // (cols * bs)).astype(np.int32)
    pos = (pairs % (cols * bs)).astype(np.int64)
    req[::13] = -1
    req[5] = nr + 2
    pos[7] = -3
    pos[9] = cols * bs + 5
    n, mx = 230, 260
    cast = wl.f32_to_bf16_bits if dtype == "bf16" else (lambda x: x.astype(np.float32))
    x = rng.standard_normal((2, len(req), hkv, d)).astype(np.float32) * np.float32(0.05)
    x[:, :15] *= np.float32(1e4)
    x[:, 15:30] *= np.float32(1e-4)
    x[0, 31, 0, 0] = np.nan
    k, v = cast(x[0]), cast(x[1])
    want_s, serr = oracle.compute_slot_mapping(table, req, pos, bs, n, mx)
    kc0 = np.full((tb, bs, hkv, d), NAN8, np.uint8)
    want_k, want_v, werr = oracle.cache_write_fp8(k, v, want_s, kc0, kc0, K_SCALE, V_SCALE, num_tokens=n)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    kt = torch.from_numpy(k).cuda().view(tdt) if dtype == "bf16" else torch.from_numpy(k).cuda()
    vt = torch.from_numpy(v).cuda().view(tdt) if dtype == "bf16" else torch.from_numpy(v).cuda()
    tab, rq, ps = torch.from_numpy(table).cuda(), torch.from_numpy(req).cuda(), torch.from_numpy(pos).cuda()
    results = []
    for fused in (True, False):
        kc = torch.full((tb, bs, hkv, d), NAN8, dtype=torch.uint8, device="cuda")
        vc = torch.full_like(kc, NAN8)
        slots = torch.full((mx,), 777, dtype=torch.int64, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        if fused:
            bkv.bkv_slot_mapping_cache_write_fp8(tab, rq, ps, slots, kt, vt, kc, vc, K_SCALE, V_SCALE, num_tokens=n,
                                                 err_count=err)
        else:
            bkv.bkv_compute_slot_mapping(tab, rq, ps, bs, slots, num_tokens=n, err_count=err)
            bkv.bkv_cache_write_fp8(kt, vt, slots, kc, vc, K_SCALE, V_SCALE, num_tokens=n, err_count=err)
        torch.cuda.synchronize()
        results.append((slots.cpu().numpy(), kc.cpu().numpy(), vc.cpu().numpy(), int(err.item())))
    (s1, k1, v1, e1), (s2, k2, v2, e2) = results
    assert np.array_equal(s1, want_s) and np.array_equal(s2, want_s)
    assert e1 == e2 == serr + werr > 0
    assert np.array_equal(k1, k2) and np.array_equal(v1, v2)
    for got, want in ((k1, want_k), (v1, want_v)):
        nan_w = (want & 0x7F) == 0x7F
        assert (((got & 0x7F) == 0x7F) == nan_w).all()
        assert (got[~nan_w] == want[~nan_w]).all()


# ---------------------------------------------------------------------------
# decode
# ---------------------------------------------------------------------------
def _decode_check(w, mask_mode=0, window=0, scales=(K_SCALE, V_SCALE), label=""):
    dw = DeviceWorkload(w, kv_fp8=scales)
    dw.write_step()
    dw.workspace.fill_(0xFF)
    got = _f64(dw.decode(mask_mode=mask_mode, sliding_window=window))
    torch.cuda.synchronize()
    assert int(dw.err_count.item()) == 0
    kc, vc, table = fill_oracle_cache_fp8(w, *scales)
    # the caches the library wrote are the oracle's, byte for byte
    assert (dw.k_cache.cpu().numpy() == kc).all() and (dw.v_cache.cpu().numpy() == vc).all()
    want, err = oracle.paged_decode_fp8(w.q(), kc, vc, table, w.context_lens, *scales, mask_mode=mask_mode,
                                        sliding_window=window)
    assert err == 0
    check_attention(got, want, w.dtype, label)
    return dw, got


SMALL = [
    # q_len, H_q, H_kv, D, bs, prior, dtype
    (1, 32, 8, 128, 64, (511, 1, 1300, 64, 2047, 129), "bf16"),
    (4, 32, 8, 128, 16, (0, 3, 700, 1025, 17, 250), "bf16"),
    (1, 64, 8, 128, 64, (3000, 70, 1), "bf16"),
    (2, 8, 8, 128, 32, (100, 600, 33), "bf16"),
    (3, 16, 2, 64, 16, (90, 1100, 5, 400), "bf16"),
    (4, 8, 2, 32, 4, (50, 3, 260), "f32"),
    (1, 32, 8, 128, 16, (900, 4), "f32"),
    (1, 15, 5, 128, 64, (1200, 77, 3000), "bf16"),      # 5 KV heads: a grid of 150 CTAs on 152 SMs
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: f"q{c[0]}_h{c[1]}x{c[2]}_d{c[3]}_bs{c[4]}_{c[6]}")
@pytest.mark.parametrize("mask_mode", [0, 1])
def test_decode_fp8_matches_oracle(case, mask_mode):
    q_len, H_q, H_kv, D, bs, prior, dtype = case
    w = _custom(q_len, H_q, H_kv, D, bs, list(prior) + [0], dtype, null_rows=(len(prior),),
                holes=((0, 1),) if prior[0] >= 2 * bs else ())
    _, got = _decode_check(w, mask_mode, label=f"{case}/{mask_mode}")
    assert (got[-1] == 0).all()                                       # NULL row


@pytest.mark.parametrize("window", [1, 77, 1000])
def test_decode_fp8_sliding_window(window):
    w = _custom(2, 32, 8, 128, 16, (1500, 40, 700, 3000))
    _decode_check(w, 0, window, label=f"W={window}")


def test_decode_fp8_saturating_scales():
    # scales so small that many codes saturate at 448: still the oracle's numbers
    w = _custom(1, 32, 8, 128, 64, (800, 2000, 31), qk=1.0, v=1.0)
    _decode_check(w, 0, scales=(2.0 ** -7, 1.0 / 300.0), label="saturating")


def test_decode_fp8_partition_then_merge_equals_one_call():
    w = _custom(1, 32, 8, 128, 64, (700, 1900, 65, 4000))
    dw, got = _decode_check(w)
    out2 = torch.empty_like(dw.out)
    args = (dw.q, dw.k_cache, dw.v_cache, dw.kernel_table, dw.context_lens, dw.max_context_len, out2, dw.workspace,
            K_SCALE, V_SCALE)
    bkv.bkv_paged_decode_fp8_partition(*args)
    bkv.bkv_paged_decode_fp8_merge(*args)
    torch.cuda.synchronize()
    assert torch.equal(out2.view(torch.uint16), dw.out.view(torch.uint16))


@pytest.mark.parametrize("variant", ["literal", "loud"])
def test_decode_fp8_llama_shape_all_rows(variant):
    """Every request of the Llama-shaped batch: the literal draw (scales as the benchmark's) and the loud one
    (K, V values up to ~7: scales 1/32, a few codes saturate), where outputs are O(0.1 .. 1)."""
    loud = variant == "loud"
    w = wl.make("llama3_decode", loud=loud)
    scales = (1.0 / 32, 1.0 / 32) if loud else (K_SCALE, V_SCALE)
    dw = DeviceWorkload(w, kv_fp8=scales)
    dw.write_step()
    dw.workspace.fill_(0xFF)
    got = _f64(dw.decode())
    torch.cuda.synchronize()
    assert int(dw.err_count.item()) == 0
    kc, vc, table = fill_oracle_cache_fp8(w, *scales)
    want, err = oracle.paged_decode_fp8(w.q(), kc, vc, table, w.context_lens, *scales)
    assert err == 0
    check_attention(got, want, "bf16", f"fp8 llama/{variant}", min_magnitude=0.1 if loud else None)
