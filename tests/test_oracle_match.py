"""Pins of the oracle's Match stage against exact rational arithmetic (no GPU).

"MAC-Attention", Figure 2(a) and abstract: the pre-RoPE query is compared by
L2 distance with a small ring of recent pre-RoPE queries; the nearest entry p
is reused if it passes the threshold.  Readings: the threshold is relative to
the current query's norm and strict; ties go to the most recent entry.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from conftest import bf16_value, bits


def _exact(q_bits, ring_bits, pos, tau):
    q = [Fraction(float(x)) for x in bf16_value(q_bits)]
    qn2 = sum(x * x for x in q)
    best, bestD, bestPos = -1, None, None
    for e in range(ring_bits.shape[0]):
        if pos[e] <= 0:
            continue
        r = [Fraction(float(x)) for x in bf16_value(ring_bits[e])]
        D = sum((a - b) * (a - b) for a, b in zip(q, r))
        if best < 0 or D < bestD or (D == bestD and pos[e] > bestPos):
            best, bestD, bestPos = e, D, pos[e]
    hit = best >= 0 and bestD < Fraction(tau) * Fraction(tau) * qn2
    return best, bestD, qn2, hit


@pytest.mark.parametrize("trial", range(20))
def test_distances_argmin_and_threshold_are_exact(rng, trial):
    L, d = 8, 64
    q = bits(rng.standard_normal(d))
    noise = rng.uniform(0.05, 0.8, size=L)[:, None]
    ring = bits(bf16_value(q)[None, :] + noise * rng.standard_normal((L, d)))
    pos = rng.permutation(np.arange(100, 100 + L)).astype(np.int64)
    pos[rng.integers(0, L)] = 0            # one empty slot
    tau = float(rng.uniform(0.1, 0.6))
    got = oracle.match(q, ring, pos, tau)
    slot, D, qn2, hit = _exact(q, ring, pos, tau)
    assert got["slot"] == slot
    assert Fraction(got["D"]) == D          # the fp64 sum is exact for bf16 inputs of this size
    assert Fraction(got["qn2"]) == qn2
    assert got["hit"] == hit


def test_empty_ring_is_a_miss(rng):
    q = bits(rng.standard_normal(16))
    got = oracle.match(q, bits(np.zeros((4, 16))), np.zeros(4, np.int64), 0.5)
    assert got["slot"] == -1 and not got["hit"]


def test_tie_goes_to_most_recent_entry(rng):
    d = 16
    q = bits(rng.standard_normal(d))
    other = bits(rng.standard_normal(d))
    ring = np.stack([other, q, other, q])            # entries 1 and 3 identical to q
    pos = np.array([9, 5, 10, 7], np.int64)
    got = oracle.match(q, ring, pos, 0.3)
    assert got["slot"] == 3 and got["D"] == 0.0 and got["hit"]
    pos = np.array([9, 8, 10, 7], np.int64)
    assert oracle.match(q, ring, pos, 0.3)["slot"] == 1


def test_threshold_is_strict():
    d = 4
    q = bits([2.0, 0, 0, 0])
    at = bits([[3.0, 0, 0, 0]])                      # D = 1 = 0.5^2 * 4 exactly
    below = bits([[2.984375, 0, 0, 0]])               # D < 1 (a bf16 value)
    pos = np.array([1], np.int64)
    assert not oracle.match(q, at, pos, 0.5)["hit"]
    assert oracle.match(q, below, pos, 0.5)["hit"]


def test_zero_threshold_never_hits(rng):
    q = bits(rng.standard_normal(8))
    ring = np.stack([q, q])
    got = oracle.match(q, ring, np.array([3, 4], np.int64), 0.0)
    assert got["D"] == 0.0 and not got["hit"] and got["slot"] == 1


def test_distance_is_on_pre_rope_values_not_positions(rng):
    # the same query vector stored at a far older position still matches exactly
    q = bits(rng.standard_normal(32))
    ring = np.stack([bits(rng.standard_normal(32)), q])
    got = oracle.match(q, ring, np.array([1000, 1], np.int64), 0.1)
    assert got["slot"] == 1 and got["hit"]


def test_runner_up_distance_is_reported(rng):
    d = 8
    q = bits(np.zeros(d))
    ring = bits(np.array([[1.0] + [0] * 7, [2.0] + [0] * 7, [0.5] + [0] * 7]))
    got = oracle.match(q, ring, np.array([1, 2, 3], np.int64), 1.0)
    assert got["slot"] == 2 and got["D"] == 0.25 and got["D2"] == 1.0
