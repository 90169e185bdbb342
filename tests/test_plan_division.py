"""The work planner divides token positions by a chunk size C = 16 c with a
precomputed multiplier (no division per dividend in the attention kernel's
prologue): with l = ceil(log2 c), k = 26 + l and m = ceil(2^k / c),
floor((x >> 4) m / 2^k) = floor(x / C) for 0 <= x < 2^30 and 4 <= c <= 2^26
(division by invariant integers, Granlund and Montgomery 1994).  The kernel's
integer steps are restated here in exact Python integers and checked against
floor division on edge cases and dense samples, including the extremes of
both ranges.
"""
import numpy as np


def chunk_div(C):
    c = C >> 4
    k = 26 + (c - 1).bit_length()          # 32 - clz(c - 1) for c >= 2
    m = ((1 << k) + c - 1) // c
    assert m < (1 << 32)                    # the multiplier fits the 32-bit register
    return m, k


def div_c(x, d):
    m, k = d
    return ((x >> 4) * m) >> k


def test_multiplier_division_is_exact():
    rng = np.random.default_rng(20260331)
    top = (1 << 30) - 1
    cs = sorted(set([4, 5, 6, 7, 8, 9, 15, 16, 17, 31, 32, 33, 1 << 20, (1 << 20) + 1, (1 << 25) + 3,
                     (1 << 26) - 1, 1 << 26] + rng.integers(4, 1 << 26, 3000).tolist() + list(range(4, 2048))))
    for c in cs:
        C = int(c) * 16
        d = chunk_div(C)
        xs = set(rng.integers(0, 1 << 30, 400).tolist())
        xs.update(range(0, 48))
        xs.update(range(top - 48, top + 1))
        for j in (1, 2, 3, 17, 1000):          # multiples of C and their neighbours
            for dx in (-1, 0, 1):
                v = j * C + dx
                if 0 <= v <= top:
                    xs.add(v)
        for x in xs:
            assert div_c(x, d) == x // C, (x, C)
