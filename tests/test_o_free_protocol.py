"""The two-tile prefill's hand-over of each tile's O accumulator in TMEM, modelled on the host
as a discrete-event simulation.  Per tile, the MMA issuer accumulates a unit's P.V products
into O and commits `o_done` after the last one; the tile's softmax warps, as its epilogue, wait
for `o_done`, read O out of TMEM and arrive on `o_free`; the issuer's first P.V of its next unit
with products waits on `o_free` by phase parity.  That wait is sound only if, when it starts,
the barrier has completed one phase fewer than the wait needs or exactly as many: one fewer
still and it passes at once (O overwritten before it is read); one more and it waits for a
phase nobody completes (a hang, which the bounded waits turn into a reported timeout).

Both sides count only units in which the tile has KV tiles.  The model checks the soundness
condition at every wait over random unit sequences (units where the tile has no KV tile, with
and without the other tile's turns) and random delays, and that it finds the hang of an
epilogue that arrived for every unit (the fault a multi-unit test once reported)."""
import random

import pytest

from tests.event_sim import Sim


def simulate(units, rng, arrive_every_unit):
    """units: (n, other) per unit: this tile's KV tiles and the other tile's.  A unit with
    any KV tile takes max(n, other) + 1 issue turns; this tile's P.V of its tile j - 1 is
    issued in turn j."""
    sim = Sim(rng)
    o_free = [0]     # completed phases
    o_done = [0]
    bad = [0]
    finished = [0, 0]

    def issuer():
        uo = 0  # units with products so far
        for n, other in units:
            steps = max(n, other) + 1 if (n > 0 or other > 0) else 0
            for step in range(steps):
                in_v = 1 <= step <= n
                if in_v and step == 1 and uo > 0:
                    need = uo  # the previous product unit's read-out: phase uo - 1 complete
                    if not (need - 1 <= o_free[0] <= need):
                        bad[0] += 1
                        if o_free[0] > need:
                            finished[0] = -1  # would wait for a phase nobody completes
                            return
                    yield "until", lambda need=need: o_free[0] >= need
                yield "sleep", rng.uniform(0.05, 1.0)
                if in_v and step == n:
                    def done():
                        o_done[0] += 1
                    sim.at(sim.now + rng.uniform(0.1, 0.8), done)
            if n > 0:
                uo += 1
        finished[0] = 1

    def epilogue():
        ocnt = 0
        for n, _ in units:
            if n > 0:
                # the softmax of this unit's tiles, then the read-out of O
                yield "until", lambda ocnt=ocnt: o_done[0] >= ocnt + 1
                ocnt += 1
                yield "sleep", rng.uniform(0.2, 1.5)
            if n > 0 or arrive_every_unit:
                o_free[0] += 1
        finished[1] = 1

    sim.start(issuer())
    sim.start(epilogue())
    try:
        sim.run()
    except AssertionError:
        pass  # a hung issuer leaves the queue to run dry
    return bad[0] + (finished[0] != 1)


def random_units(rng, count):
    out = []
    for _ in range(count):
        n = 0 if rng.random() < 0.35 else rng.randint(1, 4)
        other = 0 if rng.random() < 0.35 else rng.randint(1, 4)
        out.append((n, other))
    return out


@pytest.mark.parametrize("seed", range(40))
def test_counting_only_units_with_products_keeps_every_wait_sound(seed):
    rng = random.Random(seed)
    assert simulate(random_units(rng, 30), rng, arrive_every_unit=False) == 0


def test_the_model_finds_the_hang_of_arriving_for_every_unit():
    found = sum(simulate(random_units(random.Random(s), 30), random.Random(s), True) > 0
                for s in range(100))
    assert found > 0
