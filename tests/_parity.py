"""Error bars of the attention parity tests (GPU output against the fp64 oracle).

Every attention output row (one query token and query head: head_dim values)
is checked against a bar scaled to that row of the oracle's output:

    max_d |got - want|  <=  REL[dtype] * max_d |want| + FLOOR[dtype]

For outputs of magnitude at most 1 (every workload of the benchmark
configuration) this is at least as tight as the configuration's absolute bar
(1e-2 for bf16 in/out with fp32 accumulation, 1e-5 for fp32), and unlike
that bar it cannot be met by a wrong answer whose outputs are small: a row
whose attention dropped a partition or came out as zero misses it by far.
bf16 rounding of the output alone costs up to 2^-9 of the row's largest
element, the bf16 weights of the P.V product about as much again, so 1e-2
leaves a margin of about 2.5x.

Guards, so that no bar can silently stop biting:
* a row whose oracle output is exactly zero (nothing visible: a NULL row)
  must come out exactly zero;
* every other checked row must have a bar below a tenth of its magnitude
  (fails on rows the oracle puts near zero, where no bar can tell right from
  wrong);
* ``min_magnitude`` (the loud variants): the median row magnitude must reach
  it, so that the absolute bar bites as well.
"""
import os

import numpy as np

ABS = {"bf16": 1e-2, "f32": 1e-5}
REL = {"bf16": 1e-2, "f32": 1e-5}
FLOOR = {"bf16": 1e-6, "f32": 1e-9}

# worst errors seen per test (node id -> [dtype, rows checked, worst |got - want|, worst of that over the
# row's magnitude]); tests/conftest.py prints them at the end of the session
WORST = {}


def _record(dtype, rows, err_abs, err_rel):
    key = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    e = WORST.setdefault(key, [dtype, 0, 0.0, 0.0])
    e[1] += rows
    e[2] = max(e[2], err_abs)
    e[3] = max(e[3], err_rel)


def check_attention(got, want, dtype, label="", min_magnitude=None):
    """Checks ``got`` against ``want`` (same shape, last axis head_dim) row by
    row; returns (worst absolute error, worst error relative to its row's
    magnitude) over the non-zero rows."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, f"{label}: shape {got.shape} != {want.shape}"
    d = got.shape[-1]
    g = got.reshape(-1, d)
    w = want.reshape(-1, d)
    assert np.isfinite(g).all(), f"{label}: non-finite output"
    err = np.abs(g - w).max(axis=1)
    mag = np.abs(w).max(axis=1)
    zero = mag == 0.0
    if zero.any():
        bad = np.nonzero(zero & (np.abs(g).max(axis=1) != 0.0))[0]
        assert bad.size == 0, f"{label}: {bad.size} rows must be exactly 0 (nothing visible), e.g. row {bad[0]}"
    nz = ~zero
    if not nz.any():
        return 0.0, 0.0
    bar = REL[dtype] * mag[nz] + FLOOR[dtype]
    weak = np.nonzero(bar >= 0.1 * mag[nz])[0]
    assert weak.size == 0, (f"{label}: {weak.size} rows too close to zero for any bar to bite "
                            f"(magnitude {mag[nz][weak[0]]:.3e})")
    over = np.nonzero(err[nz] > bar)[0]
    if over.size:
        i = over[np.argmax(err[nz][over] / bar[over])]
        raise AssertionError(f"{label}: {over.size} rows over the bar; worst row {np.nonzero(nz)[0][i]}: "
                             f"err {err[nz][i]:.3e} > {bar[i]:.3e} (magnitude {mag[nz][i]:.3e})")
    small = mag[nz] <= 1.0
    if small.any():
        assert err[nz][small].max() <= ABS[dtype], f"{label}: absolute error above {ABS[dtype]}"
    if min_magnitude is not None:
        med = float(np.median(mag[nz]))
        assert med >= min_magnitude, f"{label}: median row magnitude {med:.3e} < {min_magnitude} (not loud)"
    worst = (float(err[nz].max()), float((err[nz] / mag[nz]).max()))
    _record(dtype, int(nz.sum()), *worst)
    return worst
