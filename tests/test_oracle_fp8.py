"""Pins for the oracle's FP8 (E4M3) KV cache (reading R16 of the oracle source:
OCP E4M3 codes, one scale per tensor, code = nearest to float32(x) / scale,
ties to even, saturation at 448; value = code value * scale).

The pages name a non-FP8 pathway ("Padding and Batching with Block KV",
Block ID 0 vs. Sentinel -1) and print nothing about the format or the scale
convention, so these pins fix the oracle to that reading, not to the pages:

* Library special case: every code's value equals torch.float8_e4m3fn's,
  and the encoding of a sweep of binary32 values (every code value, every
  exact midpoint between neighbours, one ulp either side of it, a log-uniform
  random sample, zeros, infinities, NaN) equals torch's round-to-nearest-even
  conversion after clamping to +-448.
* Worked values from the format's definition: 448, 1, 2^-9, the ties at
  2^-10 and 3 * 2^-10, 1.0625 and 1.1875, -0, saturation.
* Cache write: the bytes of the named rows equal torch's conversion of the
  float32 quotient, nothing else changes, -1 writes nothing, duplicates are
  rejected.
* Decode: torch SDPA in float64 on keys and values dequantised by torch; a
  cache whose values are exactly representable with scale 1 gives the bf16
  cache's output bit for bit; NaN codes in unreferenced memory change nothing.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle.cases import E4M3_NAN, fill_oracle_cache, fill_oracle_cache_fp8
from paged_kv_cache_slot_gb300 import workloads as wl

K_SCALE = 2.0 ** -6
V_SCALE = 0.0123


def _torch_codes(x_f32):
    """torch's E4M3 codes of float32 values (saturated to +-448 first; NaN stays NaN)."""
    t = torch.from_numpy(np.ascontiguousarray(x_f32, np.float32))
    t = torch.where(torch.isnan(t), t, t.clamp(-448.0, 448.0))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _torch_values(codes):
    return torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_every_code_value_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.e4m3_decode(codes)
    want = _torch_values(codes)
    nan = np.isnan(want)
    assert (np.isnan(got) == nan).all()
    assert set(np.nonzero(nan)[0].tolist()) == {0x7F, 0xFF}
    assert (got[~nan] == want[~nan]).all()
    # sign symmetry and monotone magnitudes 0x00..0x7E
    assert (got[0x80:0xFF] == -got[0x00:0x7F]).all()
    assert (np.diff(got[0x00:0x7F]) > 0).all()


def _sweep():
    vals = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))      # 0 .. 448
    mids = (vals[:-1] + vals[1:]) / 2                                # exact ties
    x = [vals, mids, np.nextafter(mids.astype(np.float32), np.float32(np.inf)),
         np.nextafter(mids.astype(np.float32), np.float32(-np.inf)), np.array([460.0, 464.0, 465.0, 1e6, 3e38])]
    rng = np.random.default_rng(5)
    x.append(np.exp2(rng.uniform(-14, 10, 4000)))
    x.append(rng.uniform(0, 2 ** -9, 500))                           # below the smallest subnormal
    pos = np.concatenate([np.asarray(a, np.float64) for a in x]).astype(np.float32)
    return np.concatenate([pos, -pos, np.array([0.0, -0.0, np.inf, -np.inf], np.float32)])


def test_encode_matches_torch_round_to_nearest_even_with_saturation():
    x = _sweep()
    got = oracle.e4m3_encode(x)
    assert (got == _torch_codes(x)).all()
    nan = oracle.e4m3_encode(np.array([np.nan], np.float32))
    assert nan[0] & 0x7F == 0x7F


@pytest.mark.parametrize("x, code", [
    (448.0, 0x7E), (1.0, 0x38), (2.0 ** -9, 0x01), (2.0 ** -10, 0x00), (3 * 2.0 ** -10, 0x02),
    (1.0625, 0x38), (1.1875, 0x3A), (-0.0, 0x80), (-2.0 ** -11, 0x80), (1e6, 0x7E), (-1e6, 0xFE),
    (464.0, 0x7E), (np.inf, 0x7E), (-np.inf, 0xFE), (0.015625, 0x08), (-1.5, 0xBC),
])
def test_worked_values(x, code):
    assert int(oracle.e4m3_encode(np.array([x], np.float32))[0]) == code


def _small(dtype="bf16", q_len=2, prior=(9, 0, 30, 5), bs=4, H_q=8, H_kv=2, D=16, qk=1.0, v=0.7):
    prior = np.array(prior, np.int64)
    nr = len(prior)
    new = np.full(nr, q_len, np.int64)
    new[1] = 0                      # a padded NULL row
    rng = np.random.default_rng(31)
    need = -(-(prior + new) // bs)
    total = 1 + int(need.sum()) + 3
    ids = rng.permutation(np.arange(1, total))[: int(need.sum())]
    table = np.full((nr, int(need.max()) + 2), -1, np.int32)
    k = 0
    for r, n in enumerate(need):
        table[r, :n] = ids[k:k + n]
        k += int(n)
    return wl.Workload("fp8_small", 99, dtype, nr, nr - 1, q_len, H_q, H_kv, D, bs, bs, prior, new, table, total,
                       max_num_tokens=int(new.sum()) + 2, qk_scale=qk, v_scale=v)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_cache_write_bytes_match_torch_quotient(dtype):
    w = _small(dtype=dtype, qk=40.0, v=9.0)    # magnitudes that reach saturation
    kc, vc, table = fill_oracle_cache_fp8(w, K_SCALE, V_SCALE)
    for r in range(w.num_rows):
        L = int(w.context_lens[r])
        if L == 0:
            continue
        k, v = w.kv_rows(r, 0, L)
        slots, _ = oracle.compute_slot_mapping(table, np.full(L, r, np.int32), np.arange(L), w.kernel_block_size)
        kf = torch.from_numpy(wl.to_f32(k)) / torch.tensor(K_SCALE, dtype=torch.float32)
        vf = torch.from_numpy(wl.to_f32(v)) / torch.tensor(V_SCALE, dtype=torch.float32)
        ks = kc.reshape(-1, w.num_kv_heads, w.head_dim)[slots]
        vs = vc.reshape(-1, w.num_kv_heads, w.head_dim)[slots]
        assert (ks == _torch_codes(kf.numpy())).all()
        assert (vs == _torch_codes(vf.numpy())).all()
    assert ((kc == 0x7E) | (kc == 0xFE)).any()                      # saturation was exercised
    # every byte not named by a slot keeps its poison
    written = np.zeros(kc.shape[0] * kc.shape[1], bool)
    for r in range(w.num_rows):
        L = int(w.context_lens[r])
        s, _ = oracle.compute_slot_mapping(table, np.full(L, r, np.int32), np.arange(L), w.kernel_block_size)
        written[s[s >= 0]] = True
    flat = kc.reshape(-1, w.num_kv_heads * w.head_dim)
    assert (flat[~written] == E4M3_NAN).all()


def test_cache_write_padding_duplicates_and_nan():
    kc = np.full((3, 4, 1, 8), E4M3_NAN, np.uint8)
    vc = kc.copy()
    k = np.linspace(-1, 1, 3 * 8, dtype=np.float32).reshape(3, 1, 8)
    k[2, 0, 3] = np.nan
    kc2, vc2, err = oracle.cache_write_fp8(k, k, np.array([5, -1, 11]), kc, vc, 0.5, 0.25)
    assert err == 0
    assert (kc2.reshape(12, 8)[[0, 1, 2, 3, 4, 6, 7, 8, 9, 10]] == E4M3_NAN).all()   # -1 wrote nothing
    assert (kc2.reshape(12, 8)[5] == _torch_codes(k[0, 0] / np.float32(0.5))).all()
    assert kc2.reshape(12, 8)[11, 3] & 0x7F == 0x7F                                  # NaN stays NaN
    with pytest.raises(ValueError):
        oracle.cache_write_fp8(k, k, np.array([5, 5, 6]), kc, vc, 0.5, 0.25)
    _, _, err = oracle.cache_write_fp8(k, k, np.array([5, 12, 6]), kc, vc, 0.5, 0.25)   # 12 is past the cache
    assert err == 1


def _sdpa_fp8(w, r, mask_mode, window=0):
    """torch SDPA (fp64) for request r on keys / values quantised and dequantised by torch."""
    L = int(w.context_lens[r])
    q = wl.to_f32(w.q()[r]).astype(np.float64)
    if L == 0:
        return np.zeros_like(q)
    k, v = w.kv_rows(r, 0, L)
    kq = _torch_values(_torch_codes((torch.from_numpy(wl.to_f32(k)) / torch.tensor(K_SCALE)).numpy())) * K_SCALE
    vq = _torch_values(_torch_codes((torch.from_numpy(wl.to_f32(v)) / torch.tensor(np.float32(V_SCALE))).numpy()))
    vq = vq * np.float64(np.float32(V_SCALE))
    qpos = L - w.q_len + np.arange(w.q_len)
    kpos = np.arange(L)
    allowed = kpos[None, :] <= qpos[:, None] if mask_mode == 0 else np.ones((w.q_len, L), bool)
    if window > 0:
        allowed &= kpos[None, :] > qpos[:, None] - window
    G = w.group_size
    qt = torch.from_numpy(q).permute(1, 0, 2)
    kt = torch.from_numpy(kq).permute(1, 0, 2).repeat_interleave(G, dim=0)
    vt = torch.from_numpy(vq).permute(1, 0, 2).repeat_interleave(G, dim=0)
    out = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=torch.from_numpy(allowed)[None])
    out = out.permute(1, 0, 2).numpy()
    out[~allowed.any(axis=1)] = 0.0
    return out


@pytest.mark.parametrize("mask_mode", [0, 1])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("window", [0, 7])
def test_decode_matches_sdpa_on_dequantised_values(mask_mode, dtype, window):
    w = _small(dtype=dtype, qk=3.0, v=2.0)
    kc, vc, table = fill_oracle_cache_fp8(w, K_SCALE, np.float32(V_SCALE))
    out, err = oracle.paged_decode_fp8(w.q(), kc, vc, table, w.context_lens, K_SCALE, np.float32(V_SCALE),
                                       mask_mode=mask_mode, sliding_window=window)
    assert err == 0 and np.isfinite(out).all()
    for r in range(w.num_rows):
        np.testing.assert_allclose(out[r], _sdpa_fp8(w, r, mask_mode, window), rtol=0, atol=1e-12)
    assert (out[1] == 0).all()


def test_representable_values_with_unit_scale_equal_the_bf16_cache_bitwise():
    # K/V drawn from the E4M3 grid and stored exactly in bf16: the FP8 cache with
    # scale 1 holds the same numbers, so the decode is the same computation
    w = _small(dtype="bf16")
    rng = np.random.default_rng(3)
    grid = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))[16:100]   # 2^-5 .. ~24
    kb, vb, table = fill_oracle_cache(w)
    for c in (kb, vb):
        vals = rng.choice(np.concatenate([grid, -grid]), size=c.shape)
        c[...] = wl.f32_to_bf16_bits(vals.astype(np.float32))
    k8 = oracle.e4m3_encode(wl.bf16_bits_to_f32(kb))
    v8 = oracle.e4m3_encode(wl.bf16_bits_to_f32(vb))
    assert (oracle.e4m3_decode(k8) == wl.bf16_bits_to_f32(kb)).all()    # exactly representable
    a, ea = oracle.paged_decode(w.q(), kb, vb, table, w.context_lens)
    b, eb = oracle.paged_decode_fp8(w.q(), k8, v8, table, w.context_lens, 1.0, 1.0)
    assert ea == eb == 0
    assert a.tobytes() == b.tobytes()


def test_nan_codes_in_unreferenced_memory_change_nothing():
    w = _small()
    kc, vc, table = fill_oracle_cache_fp8(w, K_SCALE, V_SCALE)
    a, _ = oracle.paged_decode_fp8(w.q(), kc, vc, table, w.context_lens, K_SCALE, V_SCALE)
    used = np.zeros(kc.shape[0], bool)
    used[table[table > 0]] = True
    kz, vz = kc.copy(), vc.copy()
    kz[~used] = 0
    vz[~used] = 0
    b, _ = oracle.paged_decode_fp8(w.q(), kz, vz, table, w.context_lens, K_SCALE, V_SCALE)
    assert np.isfinite(a).all()
    assert a.tobytes() == b.tobytes()
