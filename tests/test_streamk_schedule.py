"""Invariants of the stream-K work split that the kernel relies on (host model, CPU).

The kernel's schedule: CTA (pair) c of G first runs whole tiles c, c+G, ... < dp_tiles,
then the contiguous unit range [c*U/G, (c+1)*U/G) of the U = (tiles - dp_tiles) * nsb
remaining (tile, stage-block) units, cut at tile boundaries.  dp_tiles = (tiles//G - 1)*G
when tiles >= 2G, else 0.  The owner of a split tile holds its first unit; the other
holders are found from the range bounds.  These checks mirror that arithmetic and verify:
every unit is covered once, the owner's contributor set is exactly the other holders,
a split tile is each contributor's first stream-K item (so partials are written
before any owner can wait for them), and a split tile is its owner's last item, at most one
per CTA (so the owner's stage ring is idle while it gathers the partials there).
"""
import random

import pytest


def schedule(c, G, tiles, nsb, dp):
    items = []
    t = c
    while t < dp:
        items.append((t, 0, nsb))
        t += G
    U = (tiles - dp) * nsb
    u, ue = U * c // G, U * (c + 1) // G
    while u < ue:
        gu = dp * nsb + u
        tt, s0 = divmod(gu, nsb)
        s1 = s0 + min(ue - u, nsb - s0)
        items.append((tt, s0, s1))
        u += s1 - s0
    return items


def owner_of(v, G, U, dp, nsb):
    return ((v - dp * nsb + 1) * G + U - 1) // U - 1


def has_units(c, G, U):
    return U * (c + 1) // G > U * c // G


@pytest.mark.parametrize("seed", range(4))
def test_stream_k_split_invariants(seed):
    rnd = random.Random(seed)
    for _ in range(800):
        G = rnd.randint(1, 160)
        nsb = rnd.randint(1, 70)
        tiles = rnd.randint(1, 300)
        full = tiles // G
        dp = (full - 1) * G if full >= 2 else 0
        U = (tiles - dp) * nsb
        cover = {}
        for c in range(G):
            for t, s0, s1 in schedule(c, G, tiles, nsb, dp):
                cover.setdefault(t, []).append((s0, s1, c))
        assert sorted(cover) == list(range(tiles))
        owned_split = {}
        for t, parts in cover.items():
            parts.sort()
            assert parts[0][0] == 0 and parts[-1][1] == nsb
            for a, b in zip(parts, parts[1:]):
                assert a[1] == b[0]
            if len(parts) == 1:
                continue
            owner = parts[0]
            assert schedule(owner[2], G, tiles, nsb, dp)[-1] == (t, owner[0], owner[1])
            owned_split[owner[2]] = owned_split.get(owner[2], 0) + 1
            lo = owner_of(t * nsb + owner[1], G, U, dp, nsb)
            hi = owner_of((t + 1) * nsb - 1, G, U, dp, nsb)
            got = [c for c in range(lo, hi + 1) if has_units(c, G, U)]
            assert got == sorted(c for _, _, c in parts[1:])
            for _, _, c in parts[1:]:
                sk_items = schedule(c, G, tiles, nsb, dp)[len(range(c, dp, G)):]
                assert sk_items[0][0] == t
        assert all(n == 1 for n in owned_split.values())


def test_balance():
    """No CTA gets more than one unit above the average of its stream-K share."""
    for G, tiles, nsb in [(76, 1024, 64), (76, 256, 32), (152, 240, 65), (76, 16, 64)]:
        full = tiles // G
        dp = (full - 1) * G if full >= 2 else 0
        work = [sum(s1 - s0 for _, s0, s1 in schedule(c, G, tiles, nsb, dp)) for c in range(G)]
        assert max(work) - min(work) <= 1
