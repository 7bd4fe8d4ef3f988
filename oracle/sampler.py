"""Float64 CPU oracle of the speculative-decoding verify-and-sample step.

TEST INFRASTRUCTURE: only tests/, the smoke check and bench.py's CPU-baseline
leg may import or run this module. The library never calls it, and it shares
no code, header, table or constant with the CUDA path.

What it computes, and where the pages say so (page titles as cited):

* "after three fixes, Qwen3.5/3.6 MTP head reaches 1.4x on Apple Silicon"
  (deniz.in), section "Verification under sampling was wrong": a draft token
  d is accepted with probability min(1, p_main(d)/q_draft(d)); on rejection a
  replacement is drawn from the clipped and rescaled difference of the two
  distributions. Greedy verification compares the draft with the target
  argmax. Section "Truncation must match on both sides": both distributions
  are restricted to the same deck (best 20 tokens, best 0.95 of cumulative
  mass) before the ratio is taken.
* "MTPLX: native MTP speculative decoding on Apple Silicon", section 3.3
  (exact rejection sampling): accept with min(1, p/q); on rejection sample
  from (p - q)+; the output distribution equals plain decoding.
* "Speculative decoding: draft models, VRAM economics, 3x" (tinycto.tv),
  section "Core mechanism": the four steps (draft K, verify all positions in
  one pass, accept in order with min(1, p/q), on rejection sample from
  (p(x) - q(x))+ and drop the remaining drafts).

Readings where the pages are silent:
* truncation order: top-k first, renormalise, then top-p on that mass;
* nucleus = shortest prefix of (logit desc, id asc) whose mass reaches top_p,
  i.e. keep x iff the mass strictly before x is < top_p (at least one token);
* ties in logits break by lower token id; top_k <= 0 or >= V means off,
  top_p >= 1 means off; temperature == 0 exactly means greedy;
* acceptance test u*q(d) < p(d) with u in [0, 1) (so q == p always accepts,
  p(d) == 0 always rejects, q(d) == 0 < p(d) always accepts);
* inverse CDF in token-id order: smallest j with C_j > v*S, S = total mass;
  if the residual mass S is 0, sample from p instead;
* bonus token when all K drafts are accepted: sample from p_K with v_K.

Everything is float64; the loops are plain Python over positions.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

from .philox import uniforms

BOUNDARY = 1e-6  # draws closer than this to a decision boundary are "boundary draws"


# --------------------------------------------------------------------------
# Truncation: temperature, top-k, top-p, renormalisation (one logit row)
# --------------------------------------------------------------------------
@dataclass
class Truncated:
    probs: np.ndarray          # float64 [V], zero outside the kept set
    kept: np.ndarray           # token ids of the kept set, in (logit desc, id asc) order
    topp_margin: float         # distance of the nucleus cut from top_p (inf if no top-p cut)


def descending_order(z: np.ndarray) -> np.ndarray:
    """Token ids sorted by logit descending, ties by ascending id (a total order)."""
    ids = np.arange(z.shape[0])
    return np.lexsort((ids, -z))


def topp_margin(excl: np.ndarray, n_keep: int, top_p: float) -> float:
    """Distance of top_p from the nearest value at which the nucleus changes.

    excl[j] is the renormalised mass strictly before the j-th token of L1 (in
    (logit desc, id asc) order) and the first n_keep tokens are kept (those with
    excl < top_p). Lowering top_p to excl[n_keep-1] drops the last kept token;
    raising it above excl[n_keep] (the mass before the first dropped token) keeps
    one more. The margin is the smaller of the two distances (only the first when
    no token was dropped). The first token is kept for every top_p > 0 (its
    exclusive mass is 0), so with a single kept token only the upper side counts."""
    margin = top_p - excl[n_keep - 1] if n_keep > 1 else math.inf
    if n_keep < len(excl):
        margin = min(margin, excl[n_keep] - top_p)
    return float(margin)


def truncate(z, temperature: float, top_k: int, top_p: float) -> Truncated:
    """Temperature-scaled softmax restricted by top-k then top-p, renormalised.

    z: one row of raw logits (any float dtype; converted to float64 exactly).
    """
    z = np.asarray(z, dtype=np.float64)
    V = z.shape[0]
    order = descending_order(z)
    kk = top_k if 0 < top_k < V else V
    top = order[:kk]                              # L1: the k best tokens
    m = z[order[0]]
    e = np.exp((z - m) / temperature)             # unnormalised weights, max weight 1
    w = e[top] / np.sum(e[top])                   # renormalised onto L1
    margin = math.inf
    n_keep = kk
    if top_p < 1.0:
        excl = np.concatenate(([0.0], np.cumsum(w)[:-1]))   # mass strictly before each token
        n_keep = int(np.count_nonzero(excl < top_p))         # excl is increasing: a prefix
        n_keep = max(n_keep, 1)
        margin = topp_margin(excl, n_keep, top_p)
    kept = top[:n_keep]
    probs = np.zeros(V, dtype=np.float64)
    probs[kept] = e[kept] / np.sum(e[kept])
    return Truncated(probs=probs, kept=kept, topp_margin=float(margin))


def truncated_probs(z, temperature: float, top_k: int, top_p: float) -> np.ndarray:
    return truncate(z, temperature, top_k, top_p).probs


# --------------------------------------------------------------------------
# Inverse-CDF sampling in token-id order
# --------------------------------------------------------------------------
def inverse_cdf(weights: np.ndarray, v: float) -> tuple[int, float]:
    """Smallest id j with sum(weights[:j+1]) > v * sum(weights); returns (j, margin).

    margin is the distance of v from the nearest interior CDF boundary of the
    chosen interval, in units of the normalised CDF (inf when both sides of the
    chosen interval are the ends of the support).
    """
    c = np.cumsum(np.asarray(weights, dtype=np.float64))
    s = c[-1]
    t = v * s
    j = int(np.searchsorted(c, t, side="right"))
    j = min(j, len(c) - 1)
    lo = c[j - 1] if j > 0 else 0.0
    margin = math.inf
    if lo > 0.0:                       # a positive-mass token lies before j
        margin = min(margin, (t - lo) / s)
    if c[j] < s:                       # a positive-mass token lies after j
        margin = min(margin, (c[j] - t) / s)
    return j, margin


# --------------------------------------------------------------------------
# One sequence: greedy or rejection-sampling verification
# --------------------------------------------------------------------------
@dataclass
class SeqResult:
    tokens: np.ndarray                 # int64 [K+1], -1 beyond n
    n_accepted: int                    # -1 on a data error
    n_draws: int = 0                   # acceptance tests evaluated + 1 sample (0 for greedy)
    accept_margins: list = field(default_factory=list)
    sample_margin: float = math.inf
    topp_margin: float = math.inf      # min over the rows that decided the output
    error: bool = False

    @property
    def min_margin(self) -> float:
        return min([self.sample_margin, self.topp_margin, *self.accept_margins])

    @property
    def boundary(self) -> bool:
        return self.min_margin < BOUNDARY


def _row_ok(z: np.ndarray) -> bool:
    return not (np.isnan(z).any() or np.isposinf(z).any() or np.isneginf(z).all())


def _error(K: int) -> SeqResult:
    return SeqResult(tokens=np.full(K + 1, -1, dtype=np.int64), n_accepted=-1, error=True)


def accepts(u: float, p_d: float, q_d: float) -> bool:
    """Accept the draft with probability min(1, p/q): u*q < p for u uniform in [0, 1)."""
    return u * q_d < p_d


def accept_margin(u: float, p_d: float, q_d: float) -> float:
    """Distance of the acceptance uniform u from the value at which accepts() flips.

    For q > 0 the test u*q < p flips at u = p/q, so the margin is |u - p/q|; for
    q == 0 the outcome does not depend on u (accept iff p > 0) and the margin is
    infinite."""
    return abs(u - p_d / q_d) if q_d > 0.0 else math.inf


def residual_weights(p: np.ndarray, q: np.ndarray) -> np.ndarray:
    """(p - q)+, the distribution a rejected position is resampled from (unnormalised);
    falls back to p when its mass is zero."""
    r = np.maximum(p - q, 0.0)
    return r if r.sum() > 0.0 else p


def verify_sequence(target, draft, draft_tokens, temperature: float, top_k: int,
                    top_p: float, seed: int, offset: int, b: int,
                    uniform_fn=None) -> SeqResult:
    """Verify K drafted tokens of sequence b against K+1 target rows.

    target: [K+1, V] logits, draft: [K, V] logits (unused when temperature == 0),
    draft_tokens: [K] ids. Uniforms come from Philox (oracle.philox.uniforms);
    uniform_fn(b, i) -> (u, v) replaces them (used by the exact-enumeration tests).
    """
    if uniform_fn is None:
        def uniform_fn(bb, ii):
            return uniforms(seed, offset, bb, ii)
    target = np.asarray(target, dtype=np.float64)
    K1, V = target.shape
    K = K1 - 1
    d = [int(x) for x in draft_tokens]
    T = float(temperature)
    if (math.isnan(T) or T < 0.0 or math.isnan(top_p) or top_p <= 0.0 or top_k < 0
            or any(x < 0 or x >= V for x in d)):
        return _error(K)
    if not all(_row_ok(target[i]) for i in range(K + 1)):
        return _error(K)
    out = np.full(K + 1, -1, dtype=np.int64)

    if T == 0.0:                                   # greedy: argmax-prefix matching
        amax = [int(np.argmax(target[i])) for i in range(K + 1)]   # first max = lowest id
        n = 0
        while n < K and d[n] == amax[n]:
            n += 1
        out[:n] = d[:n]
        out[n] = amax[n]
        return SeqResult(tokens=out, n_accepted=n)

    draft = np.asarray(draft, dtype=np.float64)
    if not all(_row_ok(draft[i]) for i in range(K)):
        return _error(K)

    res = SeqResult(tokens=out, n_accepted=0)
    n = K
    for i in range(K):                              # accept in order, stop at first rejection
        p = truncate(target[i], T, top_k, top_p)
        q = truncate(draft[i], T, top_k, top_p)
        res.topp_margin = min(res.topp_margin, p.topp_margin, q.topp_margin)
        u, v = uniform_fn(b, i)
        pd, qd = p.probs[d[i]], q.probs[d[i]]
        res.n_draws += 1
        if qd > 0.0:
            res.accept_margins.append(accept_margin(u, pd, qd))
        if accepts(u, pd, qd):
            continue
        n = i
        tok, res.sample_margin = inverse_cdf(residual_weights(p.probs, q.probs), v)
        break
    if n == K:                                      # all accepted: bonus token from p_K
        p = truncate(target[K], T, top_k, top_p)
        res.topp_margin = min(res.topp_margin, p.topp_margin)
        _, v = uniform_fn(b, K)
        tok, res.sample_margin = inverse_cdf(p.probs, v)
    res.n_draws += 1
    out[:n] = d[:n]
    out[n] = tok
    res.n_accepted = n
    return res


def verify_batch(target, draft, draft_tokens, temperature, top_k, top_p,
                 seed: int, offset: int) -> list[SeqResult]:
    """target [B,K+1,V], draft [B,K,V] (or None when every temperature is 0),
    draft_tokens [B,K], per-sequence temperature/top_k/top_p arrays."""
    B = len(target)
    return [verify_sequence(target[b], None if draft is None else draft[b], draft_tokens[b],
                            float(temperature[b]), int(top_k[b]), float(top_p[b]),
                            seed, offset, b) for b in range(B)]


# --------------------------------------------------------------------------
# Draft-side sampler: d ~ q (the truncated draft distribution)
# --------------------------------------------------------------------------
def sample_row(z, temperature: float, top_k: int, top_p: float, v: float) -> tuple[int, float]:
    """Sample one token from the truncated distribution of row z at uniform v
    (argmax, lowest id, when temperature == 0). Returns (token, margin)."""
    if temperature == 0.0:
        return int(np.argmax(np.asarray(z, dtype=np.float64))), math.inf
    t = truncate(z, temperature, top_k, top_p)
    return inverse_cdf(t.probs, v)


def draft_sample(z, temperature: float, top_k: int, top_p: float, seed: int,
                 offset: int, b: int, i: int) -> int:
    """The drafter's own draw d_i ~ q_i, with the sampling word of Philox at (b, i)."""
    _, v = uniforms(seed, offset, b, i)
    return sample_row(z, temperature, top_k, top_p, v)[0]
