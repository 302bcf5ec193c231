"""The head_dim-256 prefill kernel's S issue, modelled on the host as a discrete-event
simulation.  Two S issuers take the even and the odd KV tiles.  K tile T lands in slot T mod 3
of a three-slot ring, loaded once S(T - 3) has finished with the slot, and S(T) waits for it on
the slot's full barrier by phase parity, (T div 3) mod 2.  S(T) also needs S buffer T mod 4,
free once P.V of tile T - 4 is done.  The softmax and the P.V issuer take the tiles in order.

A parity wait is sound only if the slot's previous phase has completed when the wait starts.
The slot's previous tile, T - 3, belongs to the other issuer, and with four S buffers the two
issuers can drift apart by more than that.  The kernel passes a turn token from tile T's
issuer to tile T+1's once T's waits are done, so every wait runs in tile order.  The model
checks the soundness condition at every wait with the token, and that it finds unsound waits
without it (the race that the kernel's bounded waits once reported on the GPU)."""
import random

import pytest

from tests.event_sim import Sim

NK, NS = 3, 4


def simulate(ntiles, rng, turn_token):
    sim = Sim(rng)
    landed, released = [0] * NK, [0] * NK  # completed phases of each K slot's barriers
    s_done = [False] * ntiles
    pv_done = [False] * ntiles
    turn = [0]  # the tile whose issuer may do its waits
    unsound = [0]
    finished = [0, 0, 0]

    def land(s):
        landed[s] += 1

    def release(s):
        released[s] += 1

    def s_complete(t):
        s_done[t] = True
        release(t % NK)

    def k_producer():
        for t in range(ntiles):
            s, u = t % NK, t // NK
            if t >= NK:
                yield "until", lambda s=s, u=u: released[s] >= u
            sim.at(sim.now + rng.uniform(0.3, 3.0), lambda s=s: land(s))
            yield "sleep", rng.uniform(0.0, 0.1)

    def s_issuer(par):
        for t in range(par, ntiles, 2):
            if turn_token:
                yield "until", lambda t=t: turn[0] == t
            if t >= NS:
                yield "until", lambda t=t: pv_done[t - NS]
            s, u = t % NK, t // NK
            if landed[s] < u:  # the slot is two phases behind: the parity wait passes early
                unsound[0] += 1
            yield "until", lambda s=s, u=u: landed[s] >= u + 1
            if turn_token:
                turn[0] = t + 1
            yield "sleep", rng.uniform(0.2, 1.0)  # the tile's products are issued
            sim.at(sim.now + rng.uniform(0.1, 0.8), lambda t=t: s_complete(t))
        finished[par] = 1

    def softmax_and_pv():
        for t in range(ntiles):
            yield "until", lambda t=t: s_done[t]
            yield "sleep", rng.uniform(0.2, 1.5)  # softmax, P written
            yield "sleep", rng.uniform(0.1, 0.6)  # P.V issued

            def done(t=t):
                pv_done[t] = True
            sim.at(sim.now + rng.uniform(0.1, 0.5), done)
        finished[2] = 1

    sim.start(k_producer())
    sim.start(s_issuer(0))
    sim.start(s_issuer(1))
    sim.start(softmax_and_pv())
    sim.run()
    assert finished == [1, 1, 1], "the model deadlocked"
    return unsound[0]


@pytest.mark.parametrize("seed", range(40))
def test_turn_token_keeps_every_k_slot_wait_sound(seed):
    rng = random.Random(seed)
    assert simulate(60, rng, turn_token=True) == 0


def test_the_model_finds_the_race_without_the_turn_token():
    found = sum(simulate(60, random.Random(seed), turn_token=False) > 0 for seed in range(200))
    assert found > 0
