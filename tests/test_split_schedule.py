"""The split-sequence schedule that the attention kernels derive on the device, restated in Python
and checked on random length mixes (CPU only).

The schedule: each (sequence bi, KV head j) "segment" has ceil(L_bi / T) tiles of T cache rows
(none if L_bi is out of range); segments are laid end to end in (bi, j) order; CTA c of P takes
tiles [c*W/P, (c+1)*W/P). A CTA writes the partial state of a segment it covers only in part
into slot c + (bi*g + j); the merge step finds the CTAs covering a segment with
cta_of(x) = ((x+1)*P - 1) // W, skipping CTAs whose range is empty. These checks show every
tile is processed once, slots never collide, the slot count P + b*g suffices, and cta_of agrees
with the CTA ranges.
"""
from __future__ import annotations

import random

import pytest

T = 64


def tiles_of(L: int, n_max: int) -> int:
    return (L + T - 1) // T if 1 <= L <= n_max else 0


def prefix(lens, n_max):
    pre = [0]
    for L in lens:
        pre.append(pre[-1] + tiles_of(L, n_max))
    return pre


def cursor_start(x, pre, g):
    B = len(pre) - 1
    lo, hi = 0, B - 1
    while lo < hi:
        mid = (lo + hi + 1) >> 1
        if g * pre[mid] <= x:
            lo = mid
        else:
            hi = mid - 1
    bi = lo
    nt = pre[bi + 1] - pre[bi]
    rem = x - g * pre[bi]
    return [bi, rem // nt, rem % nt, nt]


def cursor_advance(cur, pre, g):
    B = len(pre) - 1
    bi, j, tile, nt = cur
    tile += 1
    if tile < nt:
        return [bi, j, tile, nt]
    tile = 0
    j += 1
    if j < g:
        return [bi, j, tile, nt]
    j = 0
    bi += 1
    while bi < B and pre[bi + 1] == pre[bi]:
        bi += 1
    nt = pre[bi + 1] - pre[bi] if bi < B else 0
    return [bi, j, tile, nt]


def simulate(lens, g, n_max, P):
    pre = prefix(lens, n_max)
    W = g * pre[-1]
    seen = []
    slots = {}
    for c in range(P):
        x0, x1 = W * c // P, W * (c + 1) // P
        if x0 >= x1:
            continue
        cur = cursor_start(x0, pre, g)
        began_at_zero = None
        for k in range(x1 - x0):
            bi, j, tile, nt = cur
            assert 0 <= bi < len(lens) and 0 <= j < g and 0 <= tile < nt
            if k == 0 or tile == 0:
                began_at_zero = tile == 0
            seen.append((bi, j, tile))
            seg_end = tile == nt - 1
            if seg_end or k == x1 - x0 - 1:
                complete = began_at_zero and seg_end
                if not complete:
                    slot = c + bi * g + j
                    assert slot not in slots, "two partial states in one slot"
                    slots[slot] = (c, bi, j)
                    assert slot < P + len(lens) * g
            cur = cursor_advance(cur, pre, g)
    return pre, W, seen, slots


@pytest.mark.parametrize("seed", range(40))
def test_schedule_covers_every_tile_once_and_slots_are_unique(seed):
    rng = random.Random(seed)
    B = rng.choice([1, 2, 3, 8, 17, 64])
    g = rng.choice([1, 2, 8, 32])
    n_max = rng.choice([1, 63, 64, 65, 129, 4097])
    lens = [rng.choice([rng.randint(1, n_max), n_max, 1, 0, n_max + 1, -3]) for _ in range(B)]
    P = rng.choice([1, 2, 3, 7, 148, 1000])
    pre, W, seen, slots = simulate(lens, g, n_max, P)
    expect = [(bi, j, t) for bi, L in enumerate(lens) for j in range(g)
              for t in range(tiles_of(L, n_max))]
    assert sorted(seen) == sorted(expect)
    # the merge step's view: pieces of each segment and where they are
    for bi, L in enumerate(lens):
        nt = tiles_of(L, n_max)
        if nt == 0:
            continue
        for j in range(g):
            s0 = g * pre[bi] + j * nt
            s1 = s0 + nt - 1
            c_first = ((s0 + 1) * P - 1) // W
            c_last = ((s1 + 1) * P - 1) // W
            def owns_tiles(c):
                return W * c // P < W * (c + 1) // P
            owners = sorted({c for c in range(P) if owns_tiles(c)
                             and W * c // P <= s1 and W * (c + 1) // P > s0})
            # the merge walks c_first..c_last and skips CTAs whose range is empty
            assert owners == [c for c in range(c_first, c_last + 1) if owns_tiles(c)]
            assert owns_tiles(c_first) and owns_tiles(c_last)
            seg = bi * g + j
            if c_first == c_last:
                assert all(v[1:] != (bi, j) for v in slots.values())
            else:
                for c in owners:
                    assert slots[c + seg] == (c, bi, j)


def test_single_cta_finishes_every_segment_itself():
    _, _, _, slots = simulate([5, 700, 64, 65], g=4, n_max=1000, P=1)
    assert slots == {}
