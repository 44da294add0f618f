"""The host-packed static schedule of dense masked prefill (attn_dense_schedule).

The schedule decides only which CTA runs which work item (a 256-row query
block of one (batch, head)), never how an item is computed; GPU tests check
that outputs do not depend on it.  Here, on the CPU, its host logic is
checked against what its contract states: every item exactly once, each
CTA's list lightest first, and a makespan within the list-scheduling bound
(mean load + the largest item) and no worse than the plain snake order.
Item costs are recomputed by brute force from the mask definition (a key
tile counts when some (row, key) pair of the block keeps it; Composable
Kernel mask from window_size_left / right, bottom-right aligned unless
top-left), independent of the library's own arithmetic."""
import numpy as np
import pytest

import attention_forward_13_gb300 as A

GRID = 152


def block_steps(Lq, Lk, mb, wl, wr, top_left, qpt=128):
    """K/V tiles (128 keys) from the first to the last one that some row of
    the block's two tiles keeps a key in; a tile covers qpt queries (128, or
    128 / g with g query heads packed per tile)."""
    diag = 0 if top_left else Lk - Lq
    lo, hi = None, None
    j = np.arange(Lk)
    for t in range(2):
        r0 = mb * 2 * qpt + t * qpt
        if r0 >= Lq:
            continue
        rows = np.arange(r0, min(r0 + qpt, Lq))[:, None] + diag
        keep = np.ones((rows.shape[0], Lk), dtype=bool)
        if wr >= 0:
            keep &= j[None, :] <= rows + wr
        if wl >= 0:
            keep &= j[None, :] >= rows - wl
        cols = np.nonzero(keep.any(axis=0))[0]
        if cols.size:
            b, e = cols[0] // 128, cols[-1] // 128 + 1
            lo = b if lo is None else min(lo, b)
            hi = e if hi is None else max(hi, e)
    return 0 if lo is None else hi - lo


def costs(B, H, Lq, Lk, wl, wr, top_left, Hkv=None):
    """Item costs in the documented item order: items are (query block, batch,
    head group), a group being the g = H / Hkv heads of a kv head when g is
    2, 4, 8 or 16 (PackGQA), else one head."""
    g = H // (Hkv or H)
    pack = g if g in (2, 4, 8, 16) else 1
    qpt = 128 // pack
    nbh, M = B * (H // pack), (Lq + 2 * qpt - 1) // (2 * qpt)
    per_block = [10 * block_steps(Lq, Lk, mb, wl, wr, top_left, qpt) + 40 for mb in range(M)]
    return [per_block[M - 1 - i // nbh] for i in range(M * nbh)]


def snake_loads(cost, grid):
    loads = [0] * grid
    n = len(cost)
    for r in range((n + grid - 1) // grid):
        for c in range(grid):
            i = r * grid + (grid - 1 - c if r & 1 else c)
            if i < n:
                loads[c] += cost[i]
    return loads


# B, H, Hkv, Lq, Lk, causal, window (left, right), top_left
SHAPES = [
    (4, 16, 16, 2048, 2048, True, None, False),
    (8, 16, 16, 1024, 1024, True, None, False),
    (2, 16, 16, 4096, 4096, True, None, False),
    (4, 16, 16, 2048, 2048, False, (512, 0), False),
    (4, 16, 16, 1000, 3000, True, None, False),
    (2, 8, 8, 3000, 1000, True, None, False),
    (1, 16, 16, 4096, 4096, False, (300, 200), True),
    (3, 7, 7, 2500, 2600, False, (-1, 64), False),
    (2, 32, 8, 2048, 2048, True, None, False),      # PackGQA g = 4: 32 queries per tile
    (4, 16, 2, 1500, 1700, True, (200, -1), False),  # g = 8 with a window
    (2, 12, 4, 2048, 2048, True, None, False),      # g = 3: not packed
]


def _wlr(causal, window):
    wl, wr = (-1, -1) if window is None else window
    if causal:
        wr = 0
    return wl, wr


@pytest.mark.parametrize("shape", SHAPES, ids=[str(i) for i in range(len(SHAPES))])
def test_schedule_contract(shape):
    B, H, Hkv, Lq, Lk, causal, window, tl = shape
    sched = A.attn_dense_schedule(B, H, Lq, Lk, GRID, causal=causal, window=window, top_left=tl,
                                  Hkv=Hkv)
    assert sched is not None and len(sched) == GRID
    cost = costs(B, H, Lq, Lk, *_wlr(causal, window), tl, Hkv=Hkv)
    n = len(cost)
    flat = [i for lst in sched for i in lst]
    assert sorted(flat) == list(range(n)), "every work item exactly once"
    for lst in sched:
        cl = [cost[i] for i in lst]
        assert cl == sorted(cl), "each CTA's list runs lightest first"
    loads = [sum(cost[i] for i in lst) for lst in sched]
    assert max(loads) <= sum(cost) / GRID + max(cost), "list-scheduling bound"
    assert max(loads) <= max(snake_loads(cost, GRID)), "no worse than the snake order"


def test_schedule_balances_the_headline_shape():
    """B4 H16 L2048 causal: the snake order's most loaded CTA carries 9.6 %
    more than the mean (costs in tenths of a K/V step); the schedule's is
    within 1 % of it."""
    cost = costs(4, 16, 2048, 2048, -1, 0, False)
    mean = sum(cost) / GRID
    assert max(snake_loads(cost, GRID)) / mean > 1.05
    sched = A.attn_dense_schedule(4, 16, 2048, 2048, GRID, causal=True)
    loads = [sum(cost[i] for i in lst) for lst in sched]
    assert max(loads) / mean < 1.01


@pytest.mark.parametrize("args,kw", [
    ((4, 16, 2048, 2048, GRID), {}),                                  # no mask: plain order
    ((4, 16, 2048, 2048, GRID), {"window": (-1, -1)}),                # a window that keeps all
    ((1, 2, 2048, 2048, GRID), {"causal": True}),                     # 16 items <= 152 CTAs
    ((16, 16, 2048, 2048, GRID), {"causal": True}),                   # 2048 items > 1408
    ((11, 16, 2176, 2176, GRID), {"causal": True}),                   # 1584 items > 1408
    ((4, 16, 2048, 2048, 200), {"causal": True}),                     # grid > 160
])
def test_schedule_not_used(args, kw):
    assert A.attn_dense_schedule(*args, **kw) is None


@pytest.mark.parametrize("args", [(0, 16, 2048, 2048, GRID), (4, 16, 0, 2048, GRID),
                                  (4, 16, 2048, -1, GRID), (4, 16, 2048, 2048, 0)])
def test_schedule_rejects_bad_sizes(args):
    with pytest.raises(A.AttnError):
        A.attn_dense_schedule(*args, causal=True)


def test_schedule_query_block_count_does_not_overflow():
    """Lq near 2^31: the block count is taken in 64 bits, so the problem is
    simply too large for the static schedule (no wrapped-around count)."""
    assert A.attn_dense_schedule(1, 1, 2 ** 31 - 10, 100, GRID, causal=True) is None


def test_schedule_item_bound_is_inclusive():
    """11 x 16 heads x 8 query blocks = 1408 items: the most the launch
    parameters carry, scheduled."""
    assert A.attn_dense_schedule(11, 16, 2048, 2048, GRID, causal=True) is not None

