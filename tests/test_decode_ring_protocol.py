"""The decode split pass's KV ring, modelled on the host as a discrete-event simulation.  The
producer loads tile i into ring slot i mod S once tile i - S has been consumed, and consumer
warp w of W takes tiles w, w + W, w + 2W, ..., waiting for each on its slot's full barrier by
phase parity, (i div S) mod 2.  A parity wait is sound only if the slot's previous phase has
completed when it starts.  When S is a multiple of W a slot only ever holds one warp's tiles,
and that warp's own earlier wait orders it; otherwise a warp can reach a slot whose previous
tile, another warp's, has not landed yet.  (A timing variant with six slots and four consumer
warps once faulted on the GPU that way.)  The model checks the ring shapes the kernel uses and
that it finds the race in the six-slot shape."""
import random

import pytest

from tests.event_sim import Sim


def simulate(ntiles, stages, consumers, rng):
    sim = Sim(rng)
    landed, released = [0] * stages, [0] * stages
    unsound = [0]
    finished = [0] * consumers

    def land(s):
        landed[s] += 1

    def release(s):
        released[s] += 1

    def producer():
        for i in range(ntiles):
            s, u = i % stages, i // stages
            if i >= stages:
                yield "until", lambda s=s, u=u: released[s] >= u
            sim.at(sim.now + rng.uniform(0.5, 4.0), lambda s=s: land(s))
            yield "sleep", rng.uniform(0.0, 0.1)

    def consumer(w):
        for i in range(w, ntiles, consumers):
            s, u = i % stages, i // stages
            if landed[s] < u:  # two phases behind: the parity wait passes early
                unsound[0] += 1
            yield "until", lambda s=s, u=u: landed[s] >= u + 1
            yield "sleep", rng.uniform(0.2, 2.0)  # the tile's products
            release(s)
        finished[w] = 1

    sim.start(producer())
    for w in range(consumers):
        sim.start(consumer(w))
    sim.run()
    assert all(finished), "the model deadlocked"
    return unsound[0]


@pytest.mark.parametrize("stages", [4, 8])  # the bf16 and the e4m3 rings
@pytest.mark.parametrize("seed", range(20))
def test_slots_owned_by_one_warp_keep_every_wait_sound(stages, seed):
    assert simulate(80, stages, 4, random.Random(seed)) == 0


def test_the_model_finds_the_race_of_six_slots_for_four_warps():
    found = sum(simulate(80, 6, 4, random.Random(seed)) > 0 for seed in range(100))
    assert found > 0
