"""The persistent prefill kernels' unit schedule, restated on the host.  Units are numbered
heaviest first; CTA c of G takes units c, 2G-1-c, 2G+c, 4G-1-c, ... (a zig-zag over the
sorted list), and the head_dim-256 kernel takes the same units in the reverse order, its
lightest round first.  Checks that both orders hand every unit to exactly one CTA, that a
CTA's reversed sequence is its zig-zag sequence backwards (so each CTA's work is the same
either way), and that the first units of the reversed order differ in length from CTA to CTA
on the head_dim-256 window workload (the reason for the reversal)."""
import random

import pytest


def zigzag_unit(cta, rnd, grid):
    return rnd * grid + (grid - 1 - cta) if rnd & 1 else rnd * grid + cta


def zigzag_unit_rev(cta, rnd, grid, nunits):
    rounds = nunits // grid
    if rounds * grid + ((grid - 1 - cta) if rounds & 1 else cta) < nunits:
        rounds += 1
    return zigzag_unit(cta, rounds - 1 - rnd, grid) if rnd < rounds else 1 << 31


def units_of(cta, grid, nunits, order):
    out, r = [], 0
    while True:
        w = order(cta, r, grid, nunits)
        if w >= nunits:
            return out
        out.append(w)
        r += 1


def forward(cta, rnd, grid, nunits):
    return zigzag_unit(cta, rnd, grid)


CASES = [(4096, 152), (256, 152), (152, 152), (153, 152), (303, 152), (1, 1), (7, 3)]
random.seed(0x5C4ED)
CASES += [(random.randint(1, 5000), random.randint(1, 200)) for _ in range(200)]


@pytest.mark.parametrize("nunits,grid", CASES)
def test_both_orders_cover_every_unit_once_with_the_same_units_per_cta(nunits, grid):
    grid = min(grid, nunits)  # the launch never has more CTAs than units
    fwd = [units_of(c, grid, nunits, forward) for c in range(grid)]
    rev = [units_of(c, grid, nunits, zigzag_unit_rev) for c in range(grid)]
    assert sorted(w for ws in fwd for w in ws) == list(range(nunits))
    assert sorted(w for ws in rev for w in ws) == list(range(nunits))
    for f, r in zip(fwd, rev):
        assert r == f[::-1]


def test_reversed_order_staggers_the_first_units_of_the_window_workload():
    """8K head_dim-256 causal window 1024, b = 2, 32 heads: 64-key tiles, 128-row units.
    A unit's KV-tile count is the reversed order's first-unit length on each CTA."""
    sq, window, bm, bn, nbh, grid = 8192, 1024, 128, 64, 64, 152
    nqt = sq // bm

    def ntiles(qt):
        q0, q1 = qt * bm, qt * bm + bm - 1
        return q1 // bn - max(0, q0 - window + 1) // bn + 1

    nunits = nqt * nbh
    qt_of = lambda w: nqt - 1 - w // nbh  # heaviest first
    firsts = {ntiles(qt_of(zigzag_unit_rev(c, 0, grid, nunits))) for c in range(grid)}
    firsts_fwd = {ntiles(qt_of(zigzag_unit(c, 0, grid))) for c in range(grid)}
    assert firsts_fwd == {18}  # every CTA starts on a full 18-tile unit in the forward order
    assert len(firsts) >= 3 and max(firsts) < 18
