"""Host-side model of the tensor-core decode's head-grouped schedule, checked for the invariants the
partition kernel and the merge kernel rely on (no GPU needed).

The partition grid is P groups of H_kv CTAs (P = floor(SMs / H_kv), one group when H_kv exceeds the SM
count).  The requests' 128-position tiles are laid end to end (TP in all); group q takes tiles
[floor(q TP / peff), floor((q + 1) TP / peff)) with peff = min(P, TP), its CTA g for KV head g, and the
CTA computes floor(TP q / peff) as A q + floor(B q / peff) with TP = A peff + B.  The piece of request
r held by group q writes partial slots 2 (g (P + R) + q + r) + {0, 1}.  The merge recomputes, per
stream (r, g), the first and last group from the tiles before r: q0 = floor(((before + 1) peff - 1) /
TP), q1 = floor(((before + Ts) peff - 1) / TP), and reads slots 2 (g (P + R) + q0 + r) .. + 2 (q1 - q0
+ 1).  The workspace holds 2 (P H_kv + R H_kv) slots.

Checked on seeded random batches (tile counts 0..300, 1..600 requests) and on the edge shapes (fewer
tiles than groups, one tile, H_kv not dividing the SM count, H_kv above it): every tile of every
stream is covered exactly once; the kernel's 32-bit split equals the exact floor; slots are distinct
and inside the workspace; each stream's slots are exactly the merge's contiguous range.
"""
import numpy as np
import pytest

SMS = 152


def grid_of(h_kv, sms=SMS):
    return (sms // h_kv) * h_kv if h_kv <= sms else h_kv


def kernel_pieces(tiles, h_kv, sms=SMS):
    """(group q, head g, request r, first tile, end tile) of every unit, as the partition kernel walks them."""
    R = len(tiles)
    pre = np.concatenate([[0], np.cumsum(tiles)]).astype(np.int64)
    TP = int(pre[-1])
    grid = grid_of(h_kv, sms)
    P = grid // h_kv
    peff = min(TP, P)
    out = []
    for cta in range(grid):
        q, g = divmod(cta, h_kv)
        if q >= peff:
            continue
        A, B = divmod(TP, peff)
        t = A * q + (B * q) // peff
        t1 = A * (q + 1) + (B * (q + 1)) // peff
        assert t == (TP * q) // peff and t1 == (TP * (q + 1)) // peff   # the 32-bit split is exact
        assert t1 > t                                                   # every participating CTA has a tile
        r = int(np.searchsorted(pre[1:], t, side="right"))             # first request ending after t
        while t < t1:
            while r < R and pre[r + 1] <= t:
                r += 1
            S, Tr = int(pre[r]), int(pre[r + 1] - pre[r])
            lo, hi = t - S, min(t1 - S, Tr)
            out.append((q, g, r, lo, hi))
            t = S + hi
    return out, P, R


def merge_range(tiles, h_kv, r, g, P, sms=SMS):
    """The merge kernel's (first slot, slot count) of stream (r, g)."""
    TP = int(np.sum(tiles))
    before = int(np.sum(tiles[:r]))
    Ts = int(tiles[r])
    if Ts == 0:
        return None, 0
    peff = min(TP, P)
    q0 = ((before + 1) * peff - 1) // TP
    q1 = ((before + Ts) * peff - 1) // TP
    return 2 * (g * (P + len(tiles)) + q0 + r), 2 * (q1 - q0 + 1)


def check(tiles, h_kv, sms=SMS):
    tiles = np.asarray(tiles, np.int64)
    pieces, P, R = kernel_pieces(tiles, h_kv, sms)
    grid = grid_of(h_kv, sms)
    nslots = 2 * (grid + R * h_kv)
    # coverage: per stream, a difference array of the tile ranges its units hold
    diff = {}
    owner = np.full(nslots, -1, np.int64)              # slot -> stream r * H_kv + g
    for q, g, r, lo, hi in pieces:
        assert 0 <= lo < hi <= tiles[r]
        d = diff.setdefault((r, g), np.zeros(int(tiles[r]) + 1, np.int64))
        d[lo] += 1
        d[hi] -= 1
        base = 2 * (g * (P + R) + q + r)
        for slot in (base, base + 1):
            assert 0 <= slot < nslots, f"slot {slot} outside {nslots}"
            assert owner[slot] == -1, f"slot {slot} twice"
            owner[slot] = r * h_kv + g
    for r in range(R):
        for g in range(h_kv):
            if tiles[r] == 0:
                assert (r, g) not in diff
                continue
            cover = np.cumsum(diff[(r, g)])[:-1]
            assert (cover == 1).all(), f"stream {(r, g)}: tiles covered {set(cover.tolist())} times"
            first, n = merge_range(tiles, h_kv, r, g, P, sms)
            mine = np.nonzero(owner == r * h_kv + g)[0]
            assert mine.tolist() == list(range(first, first + n)), (r, g, mine, first, n)


@pytest.mark.parametrize("h_kv", [1, 2, 3, 5, 7, 8, 16, 40, 152, 160])
def test_schedule_random_batches(h_kv):
    rng = np.random.default_rng(100 + h_kv)
    for _ in range(12):
        R = int(rng.integers(1, 80))
        tiles = rng.integers(0, 300, R)
        tiles[rng.random(R) < 0.15] = 0            # empty (NULL) rows
        if tiles.sum() == 0:
            tiles[0] = 1
        check(tiles, h_kv)


@pytest.mark.parametrize("tiles,h_kv", [
    ([1], 8),                    # one tile: one group participates
    ([3, 0, 2], 8),              # fewer tiles than groups
    ([0, 0, 5], 3),              # leading empty rows
    ([7] * 600, 8),              # many requests, one group ends mid-request everywhere
    ([300, 1, 299, 2], 7),       # H_kv not dividing the SM count
    ([5, 9], 160),               # H_kv above the SM count: one group of 160 CTAs
    (list(range(1, 200)), 4),    # every tile count once
])
def test_schedule_edge_shapes(tiles, h_kv):
    check(tiles, h_kv)


def test_slot_bound_is_the_workspace_bound():
    # the largest slot index any unit can take is below 2 (P H_kv + R H_kv), the tensor-core part of
    # the workspace size
    for h_kv in (1, 3, 8, 160):
        grid = grid_of(h_kv)
        P = grid // h_kv
        R = 37
        top = 2 * ((h_kv - 1) * (P + R) + (P - 1) + (R - 1)) + 1
        assert top < 2 * (grid + R * h_kv)
