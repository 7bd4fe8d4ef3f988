"""Pins for the oracle's truncation (temperature, top-k, top-p, renormalisation)
and its inverse-CDF sampler: closed forms, library routines, brute force."""
import itertools
import math

import numpy as np
import pytest
from scipy.special import softmax

from oracle.sampler import descending_order, inverse_cdf, truncate


def _rows(rng, n, V, ties=False):
    for _ in range(n):
        if ties:
            yield rng.integers(-3, 3, size=V).astype(np.float64)
        else:
            yield rng.normal(0, 2, size=V)


def test_no_truncation_is_plain_softmax():
    rng = np.random.default_rng(0)
    for z in _rows(rng, 20, 50):
        for T in (0.3, 1.0, 1.7):
            p = truncate(z, T, 0, 1.0).probs
            np.testing.assert_allclose(p, softmax(z / T), rtol=1e-12, atol=1e-15)
            p2 = truncate(z, T, 50, 1.5).probs      # top_k >= V and top_p > 1 are "off"
            np.testing.assert_array_equal(p, p2)


def test_top1_is_argmax_lowest_id():
    rng = np.random.default_rng(1)
    for z in _rows(rng, 50, 9, ties=True):
        p = truncate(z, 0.8, 1, 0.9).probs
        one_hot = np.zeros(9)
        one_hot[np.argmax(z)] = 1.0
        np.testing.assert_array_equal(p, one_hot)


def test_order_is_logit_desc_then_id_asc():
    z = np.array([1.0, 3.0, 1.0, 3.0, -0.0, 0.0, 2.0])
    assert list(descending_order(z)) == [1, 3, 6, 0, 2, 4, 5]


def _brute_force_kept(z, T, k, P):
    """Smallest upward-closed set (w.r.t. logit desc, id asc) inside the top-k set whose
    renormalised mass reaches P; found by enumerating every subset."""
    V = len(z)

    def above(a, b):          # a ranks strictly before b
        return z[a] > z[b] or (z[a] == z[b] and a < b)

    kk = k if 0 < k < V else V
    subsets = [s for r in range(1, V + 1) for s in itertools.combinations(range(V), r)]
    closed = [set(s) for s in subsets
              if all(all(y in s for y in range(V) if above(y, x)) for x in s)]
    top = [s for s in closed if len(s) == kk][0]
    e = np.exp((z - z.max()) / T)
    mass_top = sum(e[x] for x in top)
    if P >= 1.0:
        return top
    cands = [s for s in closed if s <= top and sum(e[x] for x in s) / mass_top >= P]
    return min(cands, key=len)


@pytest.mark.parametrize("ties", [False, True])
def test_kept_set_matches_subset_enumeration(ties):
    rng = np.random.default_rng(2 + ties)
    for z in _rows(rng, 12, 6, ties=ties):
        for T, k, P in [(1.0, 0, 0.9), (0.5, 3, 1.0), (2.0, 4, 0.6), (1.0, 2, 0.99),
                        (0.7, 0, 0.3), (1.3, 5, 0.75)]:
            got = set(int(x) for x in truncate(z, T, k, P).kept)
            assert got == _brute_force_kept(z, T, k, P), (z, T, k, P)


def test_truncation_invariants_large_row():
    rng = np.random.default_rng(4)
    V = 5000
    for _ in range(10):
        z = -1.1 * np.log(rng.permutation(V) + 1.0) + rng.normal(0, 0.5, V)
        T = rng.uniform(0.3, 1.2)
        k = int(rng.choice([0, 20, 50]))
        P = float(rng.choice([0.8, 0.95, 1.0]))
        t = truncate(z, T, k, P)
        assert math.isclose(t.probs.sum(), 1.0, rel_tol=0, abs_tol=1e-12)
        assert len(t.kept) <= (k if k else V)
        assert np.all(t.probs[t.kept] > 0) and np.count_nonzero(t.probs) == len(t.kept)
        # renormalised on the kept set: ratios are exp((z_a - z_b)/T)
        a, b = t.kept[0], t.kept[-1]
        assert math.isclose(t.probs[a] / t.probs[b], math.exp((z[a] - z[b]) / T), rel_tol=1e-9)
        if P < 1.0:
            kk = k if k else V
            top = descending_order(z)[:kk]
            w = np.exp((z[top] - z.max()) / T)
            w /= w.sum()
            n = len(t.kept)
            assert w[:n - 1].sum() < P <= w[:n].sum() + 1e-15


def test_temperature_limits():
    z = np.array([2.0, 1.0, 0.5, -1.0])
    hot = truncate(z, 1e6, 0, 1.0).probs           # T -> inf: uniform
    np.testing.assert_allclose(hot, 0.25, atol=1e-6)
    cold = truncate(z, 1e-3, 0, 1.0).probs         # T -> 0+: one-hot at argmax
    np.testing.assert_allclose(cold, [1, 0, 0, 0], atol=1e-200)


def test_inverse_cdf_closed_forms():
    n = 7
    w = np.full(n, 1.0 / n)
    for k in range(0, 2**24, 2**24 // 97):
        v = k * 2.0**-24
        assert inverse_cdf(w, v)[0] == math.floor(v * n)
    one_hot = np.array([0, 0, 0.0, 5.0, 0])
    for v in (0.0, 0.5, 1 - 2**-24):
        j, margin = inverse_cdf(one_hot, v)
        assert j == 3 and margin == math.inf
    # zero-mass ids are never chosen, whatever v
    w = np.array([0.0, 0.2, 0.0, 0.0, 0.3, 0.0, 0.5, 0.0])
    for k in range(0, 2**24, 2**24 // 301):
        j = inverse_cdf(w, k * 2.0**-24)[0]
        assert w[j] > 0


def test_inverse_cdf_margin_is_distance_to_nearest_interior_boundary():
    w = np.array([0.25, 0.25, 0.5])
    j, m = inverse_cdf(w, 0.3)
    assert j == 1 and math.isclose(m, 0.05)
    j, m = inverse_cdf(w, 0.1)
    assert j == 0 and math.isclose(m, 0.15)
    j, m = inverse_cdf(w, 0.9)
    assert j == 2 and math.isclose(m, 0.4)
