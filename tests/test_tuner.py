"""Acceptance telemetry and depth tuning (host logic), pinned to the method.

The rates and expected-token formulas are checked against hand-made histograms
and their closed forms. They are also checked against the float64 oracle:
sequences whose K positions share one (p, q) pair have the per-position
acceptance probability sum_x min(p(x), q(x)) (the exactness argument of
rejection sampling), and the tuner must recover it from the histogram of the
oracle's accepted-prefix lengths."""
import math

import numpy as np
import pytest

from oracle import sampler
from speculative_decoding_verification_30_gb300 import tuner


def test_rates_from_a_hand_made_histogram():
    # 10 calls stopped at n=0, 5 at n=1, 5 at n=2 (all accepted, K=2), 3 errors
    h = [10, 5, 5, 3]
    a = tuner.acceptance_rates(h)
    assert a == [10 / 20, 5 / 10]
    assert tuner.acceptance_rates([0, 0, 0, 0])[0] != tuner.acceptance_rates([0, 0, 0, 0])[0]   # NaN


@pytest.mark.parametrize("a", [0.0, 0.3, 0.7, 0.95, 1.0])
@pytest.mark.parametrize("k", [0, 1, 4, 8])
def test_expected_tokens_matches_the_closed_form(a, k):
    assert tuner.expected_tokens([a] * max(k, 1), k) == pytest.approx(tuner.iid_expected_tokens(a, k))


def test_choose_depth_balances_tokens_against_draft_cost():
    alpha = [0.8] * 8
    best_free, _ = tuner.choose_depth(alpha, tuner.linear_cost(0.0))
    assert best_free == 8                                   # free drafts: draft deepest
    best, score = tuner.choose_depth(alpha, tuner.linear_cost(0.2))
    brute = max(range(1, 9), key=lambda k: (tuner.iid_expected_tokens(0.8, k) / (1 + 0.2 * k), -k))
    assert best == brute and 1 < best < 8
    # falling acceptance: deeper positions are rarely reached
    best2, _ = tuner.choose_depth([0.9, 0.5, 0.1, 0.05], tuner.linear_cost(0.1))
    assert best2 <= 2


def test_rates_recover_the_exact_acceptance_probability_of_the_oracle():
    V, K, T, topk, topp = 6, 3, 1.0, 0, 1.0
    zp = np.array([2.0, 1.0, 0.5, 0.0, -1.0, -3.0])
    zq = np.array([1.0, 1.5, 0.0, 0.5, -2.0, -1.0])
    p = sampler.truncated_probs(zp, T, topk, topp)
    q = sampler.truncated_probs(zq, T, topk, topp)
    alpha = float(np.minimum(p, q).sum())                   # exact per-position acceptance
    target = np.tile(zp, (K + 1, 1))
    draft = np.tile(zq, (K, 1))
    N = 3000
    counts = np.zeros(K + 2, dtype=np.int64)
    for b in range(N):
        d = [sampler.draft_sample(zq, T, topk, topp, 99, 0, b, i) for i in range(K)]
        r = sampler.verify_sequence(target, draft, d, T, topk, topp, 7, 0, b)
        counts[r.n_accepted if r.n_accepted >= 0 else K + 1] += 1
    rates = tuner.acceptance_rates(counts.tolist())
    reached = [counts[i:K + 1].sum() for i in range(K)]
    for i in range(K):
        sigma = math.sqrt(alpha * (1 - alpha) / reached[i])
        assert abs(rates[i] - alpha) < 4 * sigma, (i, rates[i], alpha)
    measured = float(sum((n + 1) * c for n, c in enumerate(counts[: K + 1])) / N)
    assert measured == pytest.approx(tuner.iid_expected_tokens(alpha, K), abs=0.1)


def test_unreached_positions_do_not_poison_the_expected_tokens():
    # every call stopped at n = 0: later rates are undefined, the expectation is 1 token
    h = [50, 0, 0, 0, 0, 0]
    a = tuner.acceptance_rates(h)
    assert a[0] == 0.0 and all(x != x for x in a[1:])
    assert tuner.expected_tokens(a, 4) == 1.0
