"""Pins for the oracle's decision margins: the top-p cut margin of truncate() and
the acceptance margin of verify_sequence().

Parity forgives a token mismatch only where a draw lies within 1e-6 of its
decision boundary ("MTPLX: native MTP speculative decoding on Apple Silicon",
section 3.3: the verifier is exact, so any other difference is an error). The
margins therefore decide which mismatches are forgiven, and each is pinned here
to something other than its own formula:

* closed forms on hand-made rows whose cumulative masses are known exactly;
* brute force: the margin equals the distance from the parameter (top_p, or the
  uniform u) to the nearest value at which the oracle's own decision (the kept
  set, or accept / reject) actually changes, found by bisection on that decision;
* planted mistakes put into the oracle (inclusive instead of exclusive mass, the
  top-k mass left unrenormalised, |u - q/p| instead of |u - p/q|, the margin of a
  q = 0 draw) each fail at least one of the pins above.
"""
import math

import numpy as np
import pytest

from oracle import sampler

# Row with known renormalised masses 0.5, 0.3, 0.15, 0.05 (T = 1, ids in order).
W4 = np.array([0.5, 0.3, 0.15, 0.05])
Z4 = np.log(W4)


# ----------------------------------------------------------------- top-p margin
def _topp_closed_form_failures():
    """(case, got, want) for every closed-form case the oracle gets wrong."""
    cases = [
        # (top_k, top_p, kept ids, margin): exclusive masses 0, .5, .8, .95
        (0, 0.78, [0, 1], 0.02),        # kept while excl < P: 0, .5; next excl .8
        (0, 0.60, [0, 1], 0.10),        # min(.6 - .5, .8 - .6)
        (0, 0.85, [0, 1, 2], 0.05),     # min(.85 - .8, .95 - .85)
        (0, 0.97, [0, 1, 2, 3], 0.02),  # every token kept: only the lower side
        (0, 0.30, [0], 0.20),           # first token alone: .5 - .3 (kept for any P > 0)
        (0, 0.10, [0], 0.40),           # not .1: P cannot go below 0 to drop token 0
        # top-3 renormalises onto .5/.95, .3/.95, .15/.95: excl 0, .5263.., .8421..
        (3, 0.90, [0, 1, 2], 0.90 - 0.8 / 0.95),
        (3, 0.70, [0, 1], min(0.70 - 0.5 / 0.95, 0.8 / 0.95 - 0.70)),
    ]
    bad = []
    for k, P, kept, want in cases:
        t = sampler.truncate(Z4, 1.0, k, P)
        if list(t.kept) != kept or not math.isclose(t.topp_margin, want, abs_tol=1e-12):
            bad.append(((k, P), (list(t.kept), t.topp_margin), (kept, want)))
    # no top-p cut: infinite margin
    if sampler.truncate(Z4, 1.0, 2, 1.0).topp_margin != math.inf:
        bad.append(("no top-p", sampler.truncate(Z4, 1.0, 2, 1.0).topp_margin, math.inf))
    return bad


def _kept(z, T, k, P):
    return tuple(int(x) for x in sampler.truncate(z, T, k, P).kept)


def _flip_distance(z, T, k, P, direction, limit):
    """Smallest |P' - P| (to 1e-13) in the given direction at which the kept set
    differs from the one at P, or None if it does not change up to `limit`."""
    base = _kept(z, T, k, P)
    far = P + direction * limit
    if _kept(z, T, k, far) == base:
        return None
    lo, hi = 0.0, limit                   # kept(P + d*lo) == base, kept(P + d*hi) != base
    while hi - lo > 1e-13:
        mid = 0.5 * (lo + hi)
        if _kept(z, T, k, P + direction * mid) == base:
            lo = mid
        else:
            hi = mid
    return hi


def _topp_bruteforce_failures(n_rows=40):
    rng = np.random.default_rng(21)
    bad = []
    for r in range(n_rows):
        V = int(rng.integers(3, 12))
        z = rng.normal(0, 1.5, V) if r % 2 else rng.integers(-2, 3, V).astype(np.float64)
        T = float(rng.uniform(0.5, 1.5))
        k = int(rng.choice([0, 0, 2, 4, V + 3]))
        P = float(rng.uniform(0.05, 0.95))
        m = sampler.truncate(z, T, k, P).topp_margin
        # the kept set flips at the nearest exclusive mass on either side; P' stays in (0, 1)
        down = _flip_distance(z, T, k, P, -1, P - 1e-12)
        up = _flip_distance(z, T, k, P, +1, (1.0 - 1e-12) - P)
        dists = [d for d in (down, up) if d is not None]
        want = min(dists) if dists else math.inf
        if not (math.isclose(m, want, abs_tol=1e-11) or (m == want == math.inf)):
            bad.append((r, m, want))
    return bad


def test_topp_margin_closed_forms():
    assert _topp_closed_form_failures() == []


def test_topp_margin_is_distance_to_the_nearest_kept_set_change():
    assert _topp_bruteforce_failures() == []


def _inclusive_mass_margin(excl, n_keep, top_p):
    # planted mistake: the cumulative mass including the token instead of before it
    incl = np.append(excl[1:], 1.0)
    margin = abs(top_p - incl[n_keep - 1])
    if n_keep < len(excl):
        margin = min(margin, abs(incl[n_keep] - top_p))
    return float(margin)


def _unrenormalised_margin(excl, n_keep, top_p):
    # planted mistake: measured on the mass of the whole row, not of the top-k set L1
    # (the excl passed in is renormalised onto L1; undo that with the row W4's
    # known L1 mass when L1 is its first three tokens)
    scale = 0.95 if len(excl) == 3 else 1.0
    e = excl * scale
    margin = top_p - e[n_keep - 1]
    if n_keep < len(e):
        margin = min(margin, e[n_keep] - top_p)
    return float(margin)


def _one_sided_margin(excl, n_keep, top_p):
    # planted mistake: only the distance to the last kept token's exclusive mass
    return float(top_p - excl[n_keep - 1])


@pytest.mark.parametrize("mutant", [_inclusive_mass_margin, _unrenormalised_margin,
                                    _one_sided_margin])
def test_planted_topp_margin_mistakes_fail_a_pin(monkeypatch, mutant):
    monkeypatch.setattr(sampler, "topp_margin", mutant)
    assert _topp_closed_form_failures() or _topp_bruteforce_failures(), mutant.__name__


# ------------------------------------------------------------- acceptance margin
def _accept_closed_form_failures():
    """Worked example p = (1/2, 1/4, 1/8, 1/8), q = (1/4, 1/2, 1/8, 1/8), K = 1."""
    tgt = np.log(np.array([[0.5, 0.25, 0.125, 0.125], [0.1, 0.2, 0.3, 0.4]]))
    drf = np.log(np.array([[0.25, 0.5, 0.125, 0.125]]))
    cases = [
        # (draft token, u, margin): p/q is 1/2 at d = 1, 2 at d = 0, 1 at d = 2
        (1, 0.75, 0.25),
        (1, 0.40, 0.10),
        (0, 0.30, 1.70),
        (2, 0.90, 0.10),     # p = q: the ratio is 1, u is never above it
    ]
    bad = []
    for d, u, want in cases:
        r = sampler.verify_sequence(tgt, drf, [d], 1.0, 0, 1.0, 0, 0, 0,
                                    uniform_fn=lambda b, i, u=u: (u, 0.5))
        got = r.accept_margins
        if len(got) != 1 or not math.isclose(got[0], want, abs_tol=1e-12):
            bad.append((d, u, got, want))
    # q(d) = 0 < p(d): accepted whatever u is, no margin recorded
    tgt0 = np.log(np.array([[0.25, 0.25, 0.5], [1.0, 1.0, 1.0]]))
    drf0 = np.array([[0.0, 0.0, -np.inf]])
    r = sampler.verify_sequence(tgt0, drf0, [2], 1.0, 0, 1.0, 0, 0, 0,
                                uniform_fn=lambda b, i: (0.999, 0.5))
    if r.accept_margins != [] or r.n_accepted != 1:
        bad.append(("q=0", r.accept_margins, r.n_accepted))
    return bad


def _accept_bruteforce_failures(n=60):
    """The margin equals the distance from u to the nearest u' at which the oracle's
    own accept/reject outcome (n_accepted of a K = 1 call) changes."""
    rng = np.random.default_rng(33)
    bad = []
    for t in range(n):
        V = 6
        tgt = rng.normal(0, 1.2, (2, V))
        drf = 0.5 * tgt[:1] + 0.5 * rng.normal(0, 1.2, (1, V))
        T, k, P = 1.0, int(rng.choice([0, 4])), float(rng.choice([1.0, 0.9]))
        q = sampler.truncate(drf[0], T, k, P).probs
        d = int(rng.choice(np.nonzero(q)[0]))
        u = float(rng.uniform(0, 1))

        def n_acc(uu):
            return sampler.verify_sequence(tgt, drf, [d], T, k, P, 0, 0, 0,
                                           uniform_fn=lambda b, i: (uu, 0.5)).n_accepted

        r = sampler.verify_sequence(tgt, drf, [d], T, k, P, 0, 0, 0,
                                    uniform_fn=lambda b, i: (u, 0.5))
        base = n_acc(u)
        # nearest flip of the outcome over u' in [0, 1), by bisection on each side
        best = math.inf
        for direction, limit in ((-1, u), (+1, 1.0 - 1e-15 - u)):
            if limit <= 0 or n_acc(u + direction * limit) == base:
                continue
            lo, hi = 0.0, limit
            while hi - lo > 1e-13:
                mid = 0.5 * (lo + hi)
                if n_acc(u + direction * mid) == base:
                    lo = mid
                else:
                    hi = mid
            best = min(best, hi)
        got = r.accept_margins[0] if r.accept_margins else math.inf
        # a flip point outside [0, 1) is not reachable by u: the margin may exceed `best`
        # only in that case (then best is inf); otherwise they agree
        if best == math.inf:
            if got < min(u, 1.0 - u) - 1e-12:
                bad.append((t, got, best))
        elif not math.isclose(got, best, abs_tol=1e-11):
            bad.append((t, got, best))
    return bad


def test_accept_margin_closed_forms():
    assert _accept_closed_form_failures() == []


def test_accept_margin_is_distance_to_the_outcome_flip():
    assert _accept_bruteforce_failures() == []


@pytest.mark.parametrize("mutant", [
    lambda u, p, q: abs(u - q / p) if p > 0 else math.inf,     # inverted ratio
    lambda u, p, q: abs(u - p) if q > 0 else math.inf,          # ratio dropped
    lambda u, p, q: abs(u * q - p) if q > 0 else math.inf,      # unscaled difference
])
def test_planted_accept_margin_mistakes_fail_a_pin(monkeypatch, mutant):
    monkeypatch.setattr(sampler, "accept_margin", mutant)
    assert _accept_closed_form_failures() or _accept_bruteforce_failures()


def test_boundary_flag_uses_the_smallest_margin():
    # a sequence is a boundary sequence iff one of its draws is within 1e-6
    tgt = np.log(np.array([[0.5, 0.25, 0.125, 0.125], [0.1, 0.2, 0.3, 0.4]]))
    drf = np.log(np.array([[0.25, 0.5, 0.125, 0.125]]))
    near = sampler.verify_sequence(tgt, drf, [1], 1.0, 0, 1.0, 0, 0, 0,
                                   uniform_fn=lambda b, i: (0.5 + 5e-7, 0.9))
    far = sampler.verify_sequence(tgt, drf, [1], 1.0, 0, 1.0, 0, 0, 0,
                                  uniform_fn=lambda b, i: (0.5 + 5e-6, 0.9))
    assert near.boundary and not far.boundary
