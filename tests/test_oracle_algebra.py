"""Pins of the oracle's log-domain merge and removal (no GPU).

"MAC-Attention", Figure 2 caption: (+) merges the attention summaries of two
disjoint KV segments, (-) removes one segment's summary from a merged one
("online subtraction").  Both are fixed by what they must equal: the summary
of the union, and of the difference, computed directly over the tokens.
"""
import math

import mpmath
import numpy as np
import pytest

import oracle
from conftest import bf16_value, bits


def _kvq(rng, n, d):
    K = bits(rng.standard_normal((n, d)))
    V = bits(rng.standard_normal((n, d)))
    q = bf16_value(bits(rng.standard_normal(d)))
    return K, V, q


@pytest.mark.parametrize("trial", range(5))
def test_merge_over_any_partition_equals_attention_over_union(rng, trial):
    n, d = 257, 32
    K, V, q = _kvq(rng, n, d)
    s = 1 / math.sqrt(d)
    cuts = np.sort(rng.choice(np.arange(1, n), size=rng.integers(1, 9), replace=False))
    bounds = [0, *cuts.tolist(), n]
    segs = [(bounds[i], bounds[i + 1]) for i in range(len(bounds) - 1)]
    rng.shuffle(segs)   # merge order must not matter
    o, l = np.zeros(d), -math.inf
    for lo, hi in segs:
        os_, ls = oracle.attention_summary(q, K, V, lo, hi, s)
        o, l = oracle.merge(o, l, os_, ls)
    o_ref, l_ref = oracle.attention_summary(q, K, V, 0, n, s)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    assert l == pytest.approx(l_ref, abs=1e-12)


def test_merge_identity_and_commutativity(rng):
    d = 8
    oa, ob = rng.standard_normal(d), rng.standard_normal(d)
    o, l = oracle.merge(oa, 1.5, np.zeros(d), -math.inf)
    np.testing.assert_array_equal(o, oa)
    assert l == 1.5
    o, l = oracle.merge(np.zeros(d), -math.inf, np.zeros(d), -math.inf)
    assert l == -math.inf and not o.any()
    o1, l1 = oracle.merge(oa, 0.3, ob, -2.0)
    o2, l2 = oracle.merge(ob, -2.0, oa, 0.3)
    np.testing.assert_allclose(o1, o2, atol=1e-15)
    assert l1 == pytest.approx(l2, abs=1e-15)
    # weights: e^{la}/(e^{la}+e^{lb})
    w = math.exp(0.3) / (math.exp(0.3) + math.exp(-2.0))
    np.testing.assert_allclose(o1, w * oa + (1 - w) * ob, atol=1e-15)
    assert l1 == pytest.approx(math.log(math.exp(0.3) + math.exp(-2.0)), abs=1e-15)


@pytest.mark.parametrize("split", [1, 40, 150, 255])
def test_removal_recovers_the_remaining_segment(rng, split):
    n, d = 256, 32
    K, V, q = _kvq(rng, n, d)
    s = 1 / math.sqrt(d)
    oa, la = oracle.attention_summary(q, K, V, 0, split, s)
    ob, lb = oracle.attention_summary(q, K, V, split, n, s)
    oab, lab = oracle.attention_summary(q, K, V, 0, n, s)
    o, l, cond = oracle.remove(oab, lab, ob, lb)
    assert 0 < cond < 1
    # error is amplified by 1/cond; stay well inside it
    tol = 1e-13 / cond
    np.testing.assert_allclose(o, oa, rtol=0, atol=tol)
    assert l == pytest.approx(la, abs=tol)


def test_removal_undoes_merge(rng):
    d = 16
    oa, ob = rng.standard_normal(d), rng.standard_normal(d)
    for la, lb in [(0.0, 0.0), (3.0, -1.0), (-4.0, 2.0), (10.0, 9.5)]:
        oab, lab = oracle.merge(oa, la, ob, lb)
        o, l, cond = oracle.remove(oab, lab, ob, lb)
        np.testing.assert_allclose(o, oa, atol=1e-12 / cond)
        assert l == pytest.approx(la, abs=1e-12 / cond)


def test_removing_the_empty_summary_is_a_no_op(rng):
    o_in = rng.standard_normal(4)
    o, l, cond = oracle.remove(o_in, 0.7, np.zeros(4), -math.inf)
    np.testing.assert_array_equal(o, o_in)
    assert l == 0.7 and cond == 1.0


def test_removal_sign_convention():
    # A u B with B twice as heavy as A: delta = log(2/3)
    oa, ob = np.array([1.0, 0.0]), np.array([0.0, 1.0])
    la, lb = math.log(1.0), math.log(2.0)
    oab, lab = oracle.merge(oa, la, ob, lb)
    np.testing.assert_allclose(oab, [1 / 3, 2 / 3], atol=1e-15)
    assert lab == pytest.approx(math.log(3.0), abs=1e-15)
    o, l, cond = oracle.remove(oab, lab, ob, lb)
    assert cond == pytest.approx(1 / 3, abs=1e-15)
    np.testing.assert_allclose(o, oa, atol=1e-15)
    assert l == pytest.approx(0.0, abs=1e-15)


@pytest.mark.parametrize("x", [-1e-300, -1e-12, -1e-5, -0.01, -0.5, -0.6931471805599, -0.6931471805600,
                               -0.7, -1.0, -5.0, -30.0, -700.0])
def test_log1mexp_against_high_precision(x):
    mpmath.mp.dps = 60
    ref = float(mpmath.log(-mpmath.expm1(mpmath.mpf(x))))
    assert oracle.log1mexp(x) == pytest.approx(ref, rel=2e-15, abs=1e-300)


def test_log1mexp_at_zero_is_minus_infinity():
    assert oracle.log1mexp(0.0) == -math.inf
