"""The stream-K work partition of the persistent kernel, checked on the CPU.

The kernel cuts the sequence of total = units * KB K-blocks into G contiguous
ranges [floor(total*c/G), floor(total*(c+1)/G)) and finds a block's CTA in
closed form (largest c with floor(total*c/G) <= g); a unit's parts are
numbered by CTA.  These are the same integer formulas the kernel and the host
use; here they are checked against a direct enumeration for many shapes, so
that every block is streamed by exactly one CTA and every part index, flag
index and partial slot stays inside its buffer.
"""
from __future__ import annotations

import itertools

import pytest


def cta_of_block(g, total, G):
    return ((g + 1) * G + total - 1) // total - 1


def begin(total, G, c):
    return total * c // G


SHAPES = list(itertools.product([1, 2, 3, 64, 129], [1, 2, 4, 8, 64], [1, 3, 56, 104], [1, 2, 5, 148, 152]))


@pytest.mark.parametrize("tiles,R,KB,G", SHAPES)
def test_partition_covers_every_block_once(tiles, R, KB, G):
    units = tiles * R
    total = units * KB
    G = min(G, total)
    owner = [None] * total
    for c in range(G):
        b, e = begin(total, G, c), begin(total, G, c + 1)
        assert e > b, "every CTA gets at least one block"
        for g in range(b, e):
            assert owner[g] is None
            owner[g] = c
    assert all(o is not None for o in owner)
    assert all(cta_of_block(g, total, G) == owner[g] for g in range(total))
    pmax = 0
    for u in range(units):
        first = cta_of_block(u * KB, total, G)
        last = cta_of_block((u + 1) * KB - 1, total, G)
        parts = last - first + 1
        pmax = max(pmax, parts)
        seen = sorted({owner[g] for g in range(u * KB, (u + 1) * KB)})
        assert seen == list(range(first, last + 1))
        for g in range(u * KB, (u + 1) * KB):
            p = owner[g] - first
            assert 0 <= p < parts
    for t in range(tiles):
        C = sum(cta_of_block((u + 1) * KB - 1, total, G) - cta_of_block(u * KB, total, G) + 1
                for u in range(t * R, (t + 1) * R))
        assert R <= C <= R * pmax
        # flags of tile t: t * pmax + p < tiles * pmax
        assert (t + 1) * pmax <= tiles * pmax
    # with at least one unit per CTA, each range is >= KB blocks long, so no
    # unit is split into more than two parts
    if G <= units:
        assert pmax <= 2
