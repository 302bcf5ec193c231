"""The packed two-tile prefill's Q ring, modelled on the host as a discrete-event simulation.

The K producer loads the Q tiles of each unit in order (tile A, then tile B) into a ring of
three shared-memory slots: load n goes to slot n mod 3 and is issued once load n - 3's tile
has had its last S product (the slot's release).  The issuer of a tile waits for its load on
the slot's full barrier by phase parity, (n div 3) mod 2.  A parity wait is sound only if the
slot's previous phase has completed when the wait starts: with the barrier two phases behind,
the parity already matches and the wait passes before the load has landed.  The two issuers
take turns (A, B, A, B, ...) through each unit that has KV tiles, two turns or more each.

The model checks that soundness condition at every wait, over random unit sequences (tile B
present or not, tiles with and without KV tiles) and random load, product and issue delays,
for the protocol the kernel uses: a Q load only for tiles that have KV tiles.  It also checks
that the model finds the race in the earlier protocol, which loaded Q for every tile, so that
a run of units without KV tiles took no turns to order one issuer's wait after the other's."""
import random

import pytest

from tests.event_sim import Sim

NQ = 3


def simulate(units, rng, load_all_tiles):
    """One schedule; returns the number of waits that started with their slot two phases
    behind.  units: (has_b, n_a, n_b) per unit, n_x = KV tiles of tile X (0: none); tile X
    issues its S products in the unit's first n_x turns."""
    loads = []  # (unit, tile) in load order
    for r, (has_b, na, nb) in enumerate(units):
        for x, n in ((0, na), (1, nb)):
            if (x == 0 or has_b) and (n > 0 or load_all_tiles):
                loads.append((r, x))
    index = {lx: n for n, lx in enumerate(loads)}
    sim = Sim(rng)
    landed, released = [0] * NQ, [0] * NQ  # completed phases of each slot's barriers
    turn = [0]                             # whose turn: 0 = tile A's issuer, 1 = B's
    unsound = [0]
    finished = [0, 0]

    def land(s):
        landed[s] += 1

    def release(s):
        released[s] += 1

    def producer():
        for n in range(len(loads)):
            s, u = n % NQ, n // NQ
            if n >= NQ:
                yield "until", lambda s=s, u=u: released[s] >= u
            sim.at(sim.now + rng.uniform(0.5, 3.0), lambda s=s: land(s))
            yield "sleep", rng.uniform(0.0, 0.2)

    def issuer(x):
        for r, (has_b, na, nb) in enumerate(units):
            mine = na if x == 0 else nb
            slot = None
            if (r, x) in index:
                n = index[(r, x)]
                s, u = n % NQ, n // NQ
                if landed[s] < u:
                    unsound[0] += 1
                yield "until", lambda s=s, u=u: landed[s] >= u + 1
                slot = s
                if mine == 0:  # no product reads it: released at once
                    release(s)
            if na > 0 or (has_b and nb > 0):  # the unit takes turns
                steps = max(na, nb if has_b else 0) + 1
                for step in range(steps):
                    yield "until", lambda: turn[0] == x
                    yield "sleep", rng.uniform(0.05, 1.0)  # this turn's products are issued
                    if slot is not None and step == mine - 1:  # tile X's last S product
                        sim.at(sim.now + rng.uniform(0.1, 0.8), lambda s=slot: release(s))
                    turn[0] = 1 - x
        finished[x] = 1

    sim.start(producer())
    sim.start(issuer(0))
    sim.start(issuer(1))
    sim.run()
    assert finished == [1, 1], "the model deadlocked"
    return unsound[0]


def random_units(rng, count, p_empty):
    out = []
    for _ in range(count):
        has_b = rng.random() < 0.8
        empty = rng.random() < p_empty
        na = 0 if empty or rng.random() < 0.1 else rng.randint(1, 4)
        nb = 0 if empty or rng.random() < 0.1 else rng.randint(1, 4)
        out.append((has_b, na, nb))
    return out


@pytest.mark.parametrize("seed", range(40))
def test_q_loads_only_for_tiles_with_kv_tiles_keep_every_wait_sound(seed):
    rng = random.Random(seed)
    for p_empty in (0.0, 0.3, 0.6):
        units = random_units(rng, 24, p_empty)
        assert simulate(units, rng, load_all_tiles=False) == 0


def test_the_model_finds_the_race_of_loading_every_tile():
    """With a Q load for every tile, runs of units without KV tiles take no turns, and some
    schedule lets a wait start with its slot two phases behind."""
    found = 0
    for seed in range(300):
        rng = random.Random(seed)
        units = random_units(rng, 24, 0.6)
        found += simulate(units, rng, load_all_tiles=True) > 0
    assert found > 0
