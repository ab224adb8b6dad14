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
