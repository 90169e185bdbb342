"""Pins of the oracle's attention summary against closed forms and library
routines (no GPU).

The attention summary AS of a token set is (normalised attention output,
log-sum-exp of the scaled scores); "MAC-Attention", Figure 2 caption.  Each
case below has a value fixed by the mathematics alone.
"""
import math

import numpy as np
import pytest
import scipy.special

import oracle
from conftest import bf16_value, bits


def _as(q, K, V, lo, hi, scale):
    return oracle.attention_summary(np.asarray(q, np.float64), K, V, lo, hi, scale)


def test_single_token_gives_its_value_and_score(rng):
    d = 16
    K = bits(rng.standard_normal((5, d)))
    V = bits(rng.standard_normal((5, d)))
    q = bf16_value(bits(rng.standard_normal(d)))
    s = 0.37
    o, lse = _as(q, K, V, 3, 4, s)
    np.testing.assert_array_equal(o, bf16_value(V[3]))
    assert lse == pytest.approx(s * float(q @ bf16_value(K[3])), abs=1e-14)


def test_equal_keys_give_mean_value_and_log_count(rng):
    d, n = 8, 37
    k = rng.standard_normal(d)
    K = np.repeat(bits(k)[None, :], n, axis=0)
    V = bits(rng.standard_normal((n, d)))
    q = bf16_value(bits(rng.standard_normal(d)))
    s = 1 / math.sqrt(d)
    o, lse = _as(q, K, V, 0, n, s)
    z = s * float(q @ bf16_value(K[0]))
    np.testing.assert_allclose(o, bf16_value(V).mean(axis=0), rtol=0, atol=1e-13)
    assert lse == pytest.approx(z + math.log(n), abs=1e-12)


def test_zero_query_gives_uniform_attention(rng):
    d, n = 8, 50
    K = bits(rng.standard_normal((n, d)))
    V = bits(rng.standard_normal((n, d)))
    o, lse = _as(np.zeros(d), K, V, 10, 40, 0.5)
    np.testing.assert_allclose(o, bf16_value(V[10:40]).mean(axis=0), rtol=0, atol=1e-13)
    assert lse == pytest.approx(math.log(30), abs=1e-13)


def test_dominant_key_selects_its_value(rng):
    d, n = 8, 20
    K = bits(rng.standard_normal((n, d)) * 0.01)
    K[7] = bits(np.full(d, 4.0))
    V = bits(rng.standard_normal((n, d)))
    q = np.full(d, 4.0)
    o, lse = _as(q, K, V, 0, n, 1.0)
    np.testing.assert_allclose(o, bf16_value(V[7]), atol=1e-40 + 1e-30)
    assert lse == pytest.approx(128.0, abs=1e-9)


def test_empty_set_is_the_identity_summary(rng):
    K = bits(rng.standard_normal((4, 8)))
    o, lse = _as(np.ones(8), K, K, 2, 2, 1.0)
    assert lse == -math.inf
    assert not o.any()


@pytest.mark.parametrize("n,d", [(1, 4), (7, 16), (300, 128)])
def test_matches_scipy_softmax_and_logsumexp(rng, n, d):
    K = bits(rng.standard_normal((n, d)))
    V = bits(rng.standard_normal((n, d)))
    q = bf16_value(bits(rng.standard_normal(d)))
    s = 1 / math.sqrt(d)
    o, lse = _as(q, K, V, 0, n, s)
    z = s * (bf16_value(K) @ q)
    p = scipy.special.softmax(z)
    np.testing.assert_allclose(o, p @ bf16_value(V), rtol=1e-12, atol=1e-14)
    assert lse == pytest.approx(float(scipy.special.logsumexp(z)), rel=1e-13, abs=1e-13)


def test_large_scores_do_not_overflow(rng):
    d, n = 8, 64
    K = bits(rng.standard_normal((n, d)) * 30)
    V = bits(rng.standard_normal((n, d)))
    q = bf16_value(bits(rng.standard_normal(d) * 30))
    o, lse = _as(q, K, V, 0, n, 1.0)
    z = bf16_value(K) @ q
    assert np.isfinite(o).all() and math.isfinite(lse)
    np.testing.assert_allclose(o, scipy.special.softmax(z) @ bf16_value(V), rtol=1e-10, atol=1e-12)
    assert lse == pytest.approx(float(scipy.special.logsumexp(z)), rel=1e-13)
