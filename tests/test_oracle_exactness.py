"""Pins for the oracle's acceptance / residual / bonus logic.

The pages state the method is exact: the emitted tokens are distributed as the
(truncated) target distribution ("MTPLX: native MTP speculative decoding on
Apple Silicon", section 3.3; "Speculative decoding: draft models, VRAM
economics, 3x", section "Core mechanism", corrected-sampling step). The tests
enumerate the oracle's output distribution exactly on tiny vocabularies and
compare it with the truncated target; planted mistakes must be caught.
"""
import math

import numpy as np
import pytest

from oracle import sampler
from oracle.philox import uniforms
from tests.oracle_enum import check_exactness, exact_distribution

CASES = [
    # (seed, K, V, T, top_k, top_p)
    (0, 1, 6, 1.0, 0, 1.0),
    (1, 2, 5, 0.8, 0, 1.0),
    (2, 2, 6, 1.0, 4, 0.9),
    (3, 1, 8, 0.6, 0, 0.85),
    (4, 2, 5, 1.2, 3, 1.0),
]


def _logits(seed, K, V, alpha=0.5):
    rng = np.random.default_rng(seed)
    tgt = rng.normal(0, 1.2, size=(K + 1, V))
    drf = alpha * tgt[:K] + (1 - alpha) * rng.normal(0, 1.2, size=(K, V))
    return tgt, drf


@pytest.mark.parametrize("case", CASES)
def test_output_distribution_equals_truncated_target(case):
    seed, K, V, T, k, P = case
    tgt, drf = _logits(seed, K, V)
    worst, _ = check_exactness(tgt, drf, T, k, P)
    assert worst < 1e-5, worst


def test_acceptance_probability_is_overlap_of_p_and_q():
    # P(d_0 accepted) = sum_x min(p(x), q(x)): follows from accepting with min(1, p/q)
    tgt, drf = _logits(7, 1, 6)
    dist = exact_distribution(tgt, drf, 1.0, 0, 0.9)
    p = sampler.truncate(tgt[0], 1.0, 0, 0.9).probs
    q = sampler.truncate(drf[0], 1.0, 0, 0.9).probs
    acc = sum(pr for (toks, n), pr in dist.items() if n >= 1)
    assert abs(acc - np.minimum(p, q).sum()) < 1e-5


def test_worked_example_by_hand():
    # p = (1/2, 1/4, 1/8, 1/8), q = (1/4, 1/2, 1/8, 1/8), d = 1: p/q = 1/2.
    tgt = np.log(np.array([[0.5, 0.25, 0.125, 0.125], [0.1, 0.2, 0.3, 0.4]]))
    drf = np.log(np.array([[0.25, 0.5, 0.125, 0.125]]))
    # u = 0.75 >= 1/2: reject; (p - q)+ = (1/4, 0, 0, 0) so the replacement is token 0
    r = sampler.verify_sequence(tgt, drf, [1], 1.0, 0, 1.0, 0, 0, 0,
                                uniform_fn=lambda b, i: (0.75, 0.9))
    assert list(r.tokens) == [0, -1] and r.n_accepted == 0
    # u = 0.25 < 1/2: accept; bonus from p_1 = (.1,.2,.3,.4) at v = 0.35 -> cumulative .1,.3,.6 -> token 2
    r = sampler.verify_sequence(tgt, drf, [1], 1.0, 0, 1.0, 0, 0, 0,
                                uniform_fn=lambda b, i: (0.25, 0.35))
    assert list(r.tokens) == [1, 2] and r.n_accepted == 1


def test_identical_draft_is_always_accepted():
    rng = np.random.default_rng(11)
    for trial in range(40):
        K, V = 3, 40
        tgt = rng.normal(0, 2, size=(K + 1, V))
        d = [int(rng.integers(V)) for _ in range(K)]
        r = sampler.verify_sequence(tgt, tgt[:K], d, 0.9, 5, 0.9, 123, trial, 0)
        # a draft token outside the kept set has p = q = 0: always rejected, else accepted
        kept = [set(sampler.truncate(tgt[i], 0.9, 5, 0.9).kept.tolist()) for i in range(K)]
        n_expect = next((i for i in range(K) if d[i] not in kept[i]), K)
        assert r.n_accepted == n_expect


def test_monte_carlo_acceptance_rate_with_philox():
    rng = np.random.default_rng(5)
    V = 64
    tgt = rng.normal(0, 2, size=(2, V))
    drf = 0.6 * tgt[:1] + 0.4 * rng.normal(0, 2, size=(1, V))
    T, k, P = 1.0, 20, 0.95
    p = sampler.truncate(tgt[0], T, k, P).probs
    q = sampler.truncate(drf[0], T, k, P).probs
    expect = np.minimum(p, q).sum()
    N = 3000
    acc = 0
    for step in range(N):
        d = sampler.draft_sample(drf[0], T, k, P, 999, step, 0, 0)
        r = sampler.verify_sequence(tgt, drf, [d], T, k, P, 42, step, 0)
        acc += r.n_accepted
    sigma = math.sqrt(expect * (1 - expect) / N)
    assert abs(acc / N - expect) < 3 * sigma


def test_sampling_path_tends_to_greedy_as_temperature_goes_to_zero():
    rng = np.random.default_rng(6)
    for trial in range(30):
        K, V = 3, 30
        tgt = np.round(rng.normal(0, 3, size=(K + 1, V)), 1)
        drf = np.round(rng.normal(0, 3, size=(K, V)), 1)
        d = [int(np.argmax(drf[i])) if rng.random() < 0.5 else int(np.argmax(tgt[i]))
             for i in range(K)]
        g = sampler.verify_sequence(tgt, drf, d, 0.0, 0, 1.0, 1, trial, 0)
        s = sampler.verify_sequence(tgt, drf, d, 1e-4, 0, 1.0, 1, trial, 0)
        assert list(g.tokens) == list(s.tokens) and g.n_accepted == s.n_accepted


def test_greedy_argmax_prefix_with_ties_picks_lowest_id():
    tgt = np.array([[1.0, 3.0, 3.0, 0.0], [2.0, 2.0, 1.0, 0.0], [0.0, 0.0, 0.0, 5.0]])
    r = sampler.verify_sequence(tgt, None, [1, 0], 0.0, 0, 1.0, 0, 0, 0)
    assert list(r.tokens) == [1, 0, 3] and r.n_accepted == 2
    r = sampler.verify_sequence(tgt, None, [2, 0], 0.0, 0, 1.0, 0, 0, 0)
    assert list(r.tokens) == [1, -1, -1] and r.n_accepted == 0


def test_data_errors():
    tgt = np.zeros((2, 4))
    drf = np.zeros((1, 4))
    bad = [
        dict(d=[4]), dict(d=[-1]), dict(T=-1.0), dict(T=float("nan")),
        dict(P=0.0), dict(k=-2),
    ]
    for kw in bad:
        r = sampler.verify_sequence(tgt, drf, kw.get("d", [0]), kw.get("T", 1.0),
                                    kw.get("k", 0), kw.get("P", 1.0), 0, 0, 0)
        assert r.n_accepted == -1 and list(r.tokens) == [-1, -1]
    for val in (float("nan"), float("inf")):
        t2 = tgt.copy()
        t2[1, 2] = val
        assert sampler.verify_sequence(t2, drf, [0], 1.0, 0, 1.0, 0, 0, 0).n_accepted == -1
    t3 = tgt.copy()
    t3[0, :] = -np.inf
    assert sampler.verify_sequence(t3, drf, [0], 0.0, 0, 1.0, 0, 0, 0).n_accepted == -1
    t4 = tgt.copy()
    t4[0, 1:] = -np.inf              # -inf is legal: probability zero
    r = sampler.verify_sequence(t4, drf, [2], 1.0, 0, 1.0, 0, 0, 0)
    assert r.n_accepted == 0 and r.tokens[0] == 0


# ---------------------------------------------------------------------------
# Negative controls: mistakes planted in the oracle must break exactness.
# ---------------------------------------------------------------------------
MUTANT_CASE = (2, 2, 6, 1.0, 4, 0.9)


def _mutant_worst(monkeypatch, **patches):
    seed, K, V, T, k, P = MUTANT_CASE
    tgt, drf = _logits(seed, K, V)
    for name, fn in patches.items():
        monkeypatch.setattr(sampler, name, fn)
    worst, _ = check_exactness(tgt, drf, T, k, P)
    return worst


def test_mutant_swapped_ratio_is_caught(monkeypatch):
    assert _mutant_worst(monkeypatch, accepts=lambda u, p, q: u * p < q) > 1e-3


def test_mutant_residual_sign_is_caught(monkeypatch):
    def bad(p, q):
        r = np.maximum(q - p, 0.0)
        return r if r.sum() > 0 else p
    assert _mutant_worst(monkeypatch, residual_weights=bad) > 1e-3


def test_mutant_residual_from_target_is_caught(monkeypatch):
    # resampling from p instead of (p - q)+ (a "dropped term")
    assert _mutant_worst(monkeypatch, residual_weights=lambda p, q: p) > 1e-3


def test_mutant_independent_sample_comparison_is_caught(monkeypatch):
    # The bug the deniz.in page describes: accept iff an independent target sample
    # equals the draft. Acceptance then depends on p only through a fresh draw.
    def accepts_if_target_sample_matches(u, p_d, q_d):
        return u < p_d          # P(target sample == d) = p(d), independent of q
    assert _mutant_worst(monkeypatch, accepts=accepts_if_target_sample_matches) > 1e-3


def test_mutant_unmatched_truncation_is_caught(monkeypatch):
    # Verifying against the untruncated target while the draft is truncated
    # (deniz.in, "Truncation must match on both sides").
    real = sampler.truncate
    calls = {"n": 0}

    def half_truncated(z, T, k, P):
        calls["n"] += 1
        return real(z, T, 0, 1.0) if calls["n"] % 2 == 1 else real(z, T, k, P)
    seed, K, V, T, k, P = MUTANT_CASE
    tgt, drf = _logits(seed, K, V)
    monkeypatch.setattr(sampler, "truncate", half_truncated)
    dist_bad = exact_distribution(tgt, drf, T, k, P)
    monkeypatch.setattr(sampler, "truncate", real)
    p0 = real(tgt[0], T, k, P).probs
    marg = np.zeros(V)
    for (toks, n), pr in dist_bad.items():
        marg[toks[0]] += pr
    assert np.max(np.abs(marg - p0)) > 1e-3
