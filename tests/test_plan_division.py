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


def _chunk_div_device_steps(C, ulp_off):
    """The kernel's steps for m: a float quotient 2^k / c (perturbed by
    ulp_off units in the last place, the fast division's error bound is 2),
    then +1 / -1 steps to the smallest m with m c >= 2^k."""
    c = C >> 4
    k = 26 + (c - 1).bit_length()
    q = np.float32(np.float32(2.0 ** k) / np.float32(c))
    for _ in range(abs(ulp_off)):
        q = np.nextafter(q, np.float32(np.inf) if ulp_off > 0 else np.float32(0), dtype=np.float32)
    m = int(q)
    steps = 0
    while m * c < (1 << k):
        m += 1
        steps += 1
    while (m - 1) * c >= (1 << k):
        m -= 1
        steps += 1
    return m, k, steps


def test_device_multiplier_steps_reach_the_exact_multiplier():
    rng = np.random.default_rng(20261202)
    cs = sorted(set([4, 5, 7, 8, 9, 31, 32, 33, 1 << 20, (1 << 25) + 3, (1 << 26) - 1, 1 << 26]
                    + rng.integers(4, 1 << 26, 2000).tolist() + list(range(4, 600))))
    for c in cs:
        for off in (-2, 0, 2):
            m, k, steps = _chunk_div_device_steps(int(c) * 16, off)
            assert (m, k) == chunk_div(int(c) * 16), (c, off)
            assert steps <= 40, (c, off, steps)
