"""The decode split pass's work partition, restated on the host: the KV tiles of all
(sequence, kv head) pairs form one stream, CTA c of G takes tiles [c tpc, (c+1) tpc) with
tpc = max(ceil(NT / G), kv_chunk / 32), and a CTA's run is cut into pieces at pair
boundaries.  Checks that every tile is read exactly once, that the piece index of every
piece stays below the partial slots the workspace holds per row
(ceil(max_cache_len / kv_chunk) + 1, fewer with a window), and that the pieces of a pair
are numbered 0 .. npieces - 1 as the merge reads them."""
import random

import pytest

TILE = 32


def pair_tiles(n, sa, window, circular, cap):
    if n < sa or (not circular and n > cap):
        return 0
    nslots = min(n, cap) if circular else n
    first = (max(0, n - sa - window + 1) & ~(TILE - 1)) if (window > 0 and not circular) else 0
    return (nslots - first + TILE - 1) // TILE


def slots_bound(cap, chunk, window, sa, circular):
    slots = -(-cap // chunk) + 1
    if window > 0 and not circular:
        span = min(cap, window + sa - 1 + TILE - 1)
        slots = min(slots, -(-span // chunk) + 1)
    return slots


def partition(lens, hkv, sa, window, circular, cap, chunk, grid):
    nt = [pair_tiles(n, sa, window, circular, cap) for n in lens]
    total = sum(nt) * hkv
    tpc = max(-(-total // grid), chunk // TILE)
    cover, npieces, ks = {}, {}, {}
    for c in range(grid):
        lo, hi = c * tpc, min(total, c * tpc + tpc)
        if lo >= hi:
            continue
        base, b = 0, None
        for bb, t in enumerate(nt):  # the sequence holding tile lo
            if t > 0 and base <= lo < base + t * hkv:
                b, bstart = bb, base
                break
            base += t * hkv
        g, t_off = divmod(lo - bstart, nt[b])
        pstart = bstart + g * nt[b]
        i = 0
        while i < hi - lo:
            npc = min(nt[b] - t_off, hi - lo - i)
            k = c - pstart // tpc
            for x in range(npc):
                key = (b, g, t_off + x)
                assert key not in cover, key
                cover[key] = k
            ks.setdefault((b, g), set()).add(k)
            if t_off + npc == nt[b]:
                npieces[(b, g)] = k + 1
            i += npc
            t_off, pstart, g = 0, pstart + nt[b], g + 1
            if g == hkv:
                g = 0
                b += 1
                while b < len(nt) and nt[b] == 0:
                    b += 1
    return nt, cover, npieces, ks


def check(lens, hkv, sa, window, circular, cap, chunk, grid):
    nt, cover, npieces, ks = partition(lens, hkv, sa, window, circular, cap, chunk, grid)
    bound = slots_bound(cap, chunk, window, sa, circular)
    assert len(cover) == sum(nt) * hkv
    for b, t in enumerate(nt):
        for g in range(hkv):
            if t == 0:
                assert (b, g) not in npieces
                continue
            assert all((b, g, x) in cover for x in range(t))
            assert ks[(b, g)] == set(range(npieces[(b, g)]))
            assert npieces[(b, g)] <= bound


def window_default_chunk(cap, chunk, window, sa):
    """The decode call's least CTA share for a window with kv_chunk = 0: the smallest
    multiple of 32 tokens for which the window's span still fits the scratch's slots."""
    slots = -(-cap // chunk) + 1
    span = min(cap, window + sa - 1 + TILE - 1)
    share = -(-span // (slots - 1))
    return max(TILE, -(-share // TILE) * TILE)


def test_benchmark_shapes():
    rnd = random.Random(7)
    lens = [rnd.randint(1024, 32768) for _ in range(64)]
    check(lens, 8, 4, 0, False, 32768, 4096, 456)        # 4 new tokens, 3 CTAs x 152 SMs
    check(lens, 8, 4, 4096, False, 32768, window_default_chunk(32768, 4096, 4096, 4), 456)
    check(lens[:16], 8, 4, 4096, False, 32768, window_default_chunk(32768, 4096, 4096, 4), 456)
    check(lens[:32], 8, 1, 0, False, 32768, 4096, 152)   # head_dim 256: one CTA per SM
    check((40, 3000, 300, 33, 1000, 64, 2999, 700), 8, 4, 0, False, 3000, 256, 456)


@pytest.mark.parametrize("seed", range(4))
def test_random_shapes(seed):
    rnd = random.Random(seed)
    for _ in range(300):
        b, hkv, sa = rnd.randint(1, 12), rnd.choice([1, 2, 4, 8]), rnd.randint(1, 4)
        cap = rnd.choice([32, 64, 100, 1000, 5000])
        circular = rnd.random() < 0.2
        window = rnd.choice([0, 0, 1, 40, 333, 1000])
        if circular:
            window = rnd.randint(1, cap - sa + 1) if cap - sa + 1 >= 1 else 0
            if window == 0:
                continue
            lens = [rnd.randint(sa, 3 * cap) for _ in range(b)]
        else:  # lengths in range, out of range (skipped) and at the edges
            lens = [rnd.choice([rnd.randint(0, cap), rnd.randint(sa, cap), cap, cap + 5])
                    for _ in range(b)]
        chunk = TILE * rnd.randint(1, 40)
        if window > 0 and not circular and rnd.random() < 0.5:
            chunk = window_default_chunk(cap, chunk, window, sa)
        check(lens, hkv, sa, window, circular, cap, chunk, rnd.choice([1, 3, 7, 456]))
