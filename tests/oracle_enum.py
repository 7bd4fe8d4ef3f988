"""Exact output distribution of oracle.verify_sequence on tiny inputs.

Enumerates every draft tuple d ~ q (exact weights) and, for each position, the
cells of the uniform grid {k * 2**-24} on which the oracle's outcome is
constant: a coarse scan finds the cells, bisection finds each cell edge to the
exact grid index. The outcome is always computed by calling the oracle itself,
so a mistake planted anywhere in it changes the enumerated distribution.
"""
from __future__ import annotations

from collections import defaultdict
import itertools

import numpy as np

from oracle import sampler

GRID = 1 << 24


def _cells(f, coarse=192):
    """Partition [0, GRID) into maximal runs where f(k) is constant (assuming at most
    one switch between consecutive coarse points). Returns [(outcome, count, first)]."""
    pts = [int(round(i * (GRID - 1) / coarse)) for i in range(coarse + 1)]
    vals = [f(k) for k in pts]
    edges = []                          # first grid index of every new run
    for a, b, fa, fb in zip(pts, pts[1:], vals, vals[1:]):
        if fa == fb:
            continue
        lo, hi = a, b                   # f(lo) == fa, f(hi) != fa
        while hi - lo > 1:
            mid = (lo + hi) // 2
            if f(mid) == fa:
                lo = mid
            else:
                hi = mid
        edges.append(hi)
    bounds = [0] + edges + [GRID]
    return [(f(s), e - s, s) for s, e in zip(bounds, bounds[1:])]


def exact_distribution(target, draft, T, k, P):
    """{(tuple(tokens), n): probability} of verify_sequence over d ~ q and the uniforms."""
    K = len(draft)
    V = target.shape[1]
    qs = [sampler.truncate(draft[i], T, k, P).probs for i in range(K)]
    supports = [np.nonzero(q)[0] for q in qs]
    dist = defaultdict(float)

    for d in itertools.product(*supports):
        w_d = float(np.prod([qs[i][d[i]] for i in range(K)]))

        def run(us, vs):
            def ufn(b, i):
                return us.get(i, 0.0), vs.get(i, 0.0)
            r = sampler.verify_sequence(target, draft, d, T, k, P, 0, 0, 0, uniform_fn=ufn)
            return tuple(int(x) for x in r.tokens), r.n_accepted

        def walk(i, us, weight):
            if weight == 0.0:
                return
            if i == K:                                   # bonus: only v_K matters
                for out, cnt, _ in _cells(lambda kk: run(us, {K: kk / GRID})):
                    dist[out] += weight * cnt / GRID
                return
            # acceptance at position i is a function of u_i (earlier u's accept)
            for acc, cnt, first in _cells(lambda kk: run({**us, i: kk / GRID}, {})[1] > i):
                u_rep = first / GRID                     # any grid point of this cell
                if acc:
                    walk(i + 1, {**us, i: u_rep}, weight * cnt / GRID)
                else:
                    for out, c2, _ in _cells(lambda kk: run({**us, i: u_rep}, {i: kk / GRID})):
                        dist[out] += weight * (cnt / GRID) * (c2 / GRID)

        walk(0, {}, w_d)
    return dict(dist)


def check_exactness(target, draft, T, k, P, tol=1e-5):
    """Return the largest deviation of the enumerated output from the truncated target:
    P(out_0 = x) vs p_0(x), and P(out_j = y | n >= j) vs p_j(y)."""
    K = len(draft)
    dist = exact_distribution(target, draft, T, k, P)
    ps = [sampler.truncate(target[j], T, k, P).probs for j in range(K + 1)]
    total = sum(dist.values())
    worst = abs(total - 1.0)
    for j in range(K + 1):
        reach = sum(pr for (toks, n), pr in dist.items() if n >= j)
        if reach < 1e-9:
            continue
        marg = np.zeros(target.shape[1])
        for (toks, n), pr in dist.items():
            if n >= j:
                marg[toks[j]] += pr
        worst = max(worst, float(np.max(np.abs(marg / reach - ps[j]))))
    return worst, dist
