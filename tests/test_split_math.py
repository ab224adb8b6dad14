"""Arithmetic of the decode split, checked exhaustively on small sizes.

The persistent decode kernel gives CTA c (of P = min(CTAs, T)) the tile share
[floor(c T / P), floor((c+1) T / P)) of the flattened (b, kv head, tile)
space and finds the owner of tile t as ceil((t+1) P / T) - 1.  A pair's
pieces are the non-empty intersections of its tile range with the shares;
the piece count the in-kernel merge waits for is owner(last) - owner(first) + 1.
These identities must hold for every T >= 1 and every P <= T: each tile has
exactly one owner, every share is non-empty, and the owners of a pair's
tiles form a contiguous run with one piece each.
"""
import itertools


def share(c, T, P):
    return (c * T) // P, ((c + 1) * T) // P


def owner(t, T, P):
    return -(-((t + 1) * P) // T) - 1


def test_owner_matches_shares():
    for T in range(1, 70):
        for P in range(1, T + 1):
            seen = []
            for c in range(P):
                s, e = share(c, T, P)
                assert e > s, (T, P, c)          # non-empty shares when P <= T
                for t in range(s, e):
                    assert owner(t, T, P) == c
                seen.extend(range(s, e))
            assert seen == list(range(T))


def test_piece_count_of_a_pair():
    for T in range(1, 40):
        for P in range(1, T + 1):
            for o, n in itertools.product(range(T), range(1, 9)):
                if o + n > T:
                    continue
                owners = {owner(t, T, P) for t in range(o, o + n)}
                lo, hi = owner(o, T, P), owner(o + n - 1, T, P)
                assert owners == set(range(lo, hi + 1))


def stage_of(i, NG, SG):
    """Stage of a CTA's i-th tile: tile group i % NG, private ring of SG stages."""
    return (i % NG) * SG + (i // NG) % SG


def parity_of(i, NG, SG):
    return ((i // NG) // SG) & 1


def test_tile_groups_never_share_a_stage():
    """With NG consumer groups on alternate tiles, every stage is used by one
    group only, its uses alternate in parity, and the producer's wait for a
    free stage names the parity of that stage's previous use -- the property
    that keeps a parity wait from being satisfied by an older phase."""
    for NG, stages in [(1, 2), (1, 5), (1, 8), (2, 4), (2, 6), (2, 8)]:
        SG = stages // NG
        last = {}
        for i in range(500):
            s = stage_of(i, NG, SG)
            assert 0 <= s < NG * SG
            if s in last:
                j = last[s]
                assert j % NG == i % NG
                assert (i // NG) - (j // NG) == SG        # the group's previous use
                assert parity_of(j, NG, SG) == parity_of(i, NG, SG) ^ 1
            else:
                assert i // NG < SG                        # first use needs no wait
            last[s] = i
        # the producer's drain: the last NG*SG tiles cover every stage once
        for issued in range(NG * SG, 60):
            assert sorted(stage_of(i, NG, SG) for i in range(issued - NG * SG, issued)) == list(range(NG * SG))


def test_incremental_counters_match_the_closed_form():
    """The decode kernel keeps the ring position incrementally instead of
    dividing per tile.  Producer: (ig, us, lap) advance once per tile; tile i
    goes to stage ig*SG + us and, once lap > 0, first waits for the stage's
    previous use with parity (lap - 1) & 1.  Consumers: each tile group walks
    only its own tiles, piece by piece (a piece: the share's tiles of one
    (b, kv head) pair), starting at offset (grp - i0) mod NG of a piece that
    begins at share index i0, and keeps (us, ph) per own tile.  Both must name
    the closed-form stage and parity of every tile, for any cut into pieces."""
    import random
    rng = random.Random(7)
    for NG, stages in [(1, 2), (1, 6), (2, 4), (2, 6), (2, 8), (3, 9), (3, 12)]:
        SG = stages // NG
        for trial in range(40):
            n = rng.randint(1, 120)
            # producer
            ig = us = lap = 0
            for i in range(n):
                s = ig * SG + us
                assert s == stage_of(i, NG, SG)
                if lap > 0:
                    assert (lap - 1) & 1 == parity_of(i - NG * SG, NG, SG)
                else:
                    assert i // NG < SG
                ig += 1
                if ig == NG:
                    ig = 0
                    us += 1
                    if us == SG:
                        us = 0
                        lap += 1
            # consumers, over a random cut of the share into pieces
            cuts = sorted(rng.sample(range(1, n), min(n - 1, rng.randint(0, 6)))) if n > 1 else []
            bounds = [0] + cuts + [n]
            for grp in range(NG):
                us = ph = 0
                seen = []
                for i0, i1 in zip(bounds, bounds[1:]):
                    first = ((grp - i0) % NG + NG) % NG
                    for k in range(first, i1 - i0, NG):
                        i = i0 + k
                        assert i % NG == grp
                        assert grp * SG + us == stage_of(i, NG, SG)
                        assert ph == parity_of(i, NG, SG)
                        seen.append(i)
                        us += 1
                        if us == SG:
                            us = 0
                            ph ^= 1
                assert seen == [i for i in range(n) if i % NG == grp]
