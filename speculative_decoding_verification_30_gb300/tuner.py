"""Acceptance telemetry and draft-depth tuning for the verify step.

The pages treat the draft acceptance rate as the main operating signal, and the
draft depth as something to choose from it on the machine at hand:
- "Speculative decoding: draft models, VRAM economics, 3x" (tinycto.tv), sections
  on monitoring and tuning: watch the acceptance-rate telemetry (a draft
  accepted less than about 40% of the time can make decoding slower), and set
  the speculation length between 3 and 6 according to the measured acceptance.
- "MTPLX" (text-matrix.pages.dev), the tune command: measure the acceptance at
  each depth on the user's own machine and keep only the depths that beat plain
  decoding.
- "after three fixes, Qwen3.5/3.6 MTP head reaches 1.4x on Apple Silicon"
  (deniz.in), section on draft depth: on Apple GPUs depth 1 was best, and a
  heuristic that raises the depth after fully accepted rounds lost 4-17% against
  it; on CUDA, verifying extra positions is nearly free. So the depth depends on
  the cost of a step, which the cost model below makes explicit.

This module turns an acceptance histogram (`spec_accept_histogram`: counts of
the accepted-prefix length n in 0..K over verify calls) into:
- per-position acceptance rates alpha_i = P(position i accepted | positions
  before it accepted),
- the expected tokens per step at any depth k <= K: one emitted token plus the
  expected accepted prefix, E_k = sum_{j=0..k} prod_{i<j} alpha_i,
- the depth that maximises tokens per unit of step cost under a cost model.

`sweep` measures all of this on the GPU: synthetic batches with a chosen
draft/target similarity, drafts drawn by the library's draft-side sampler,
verified by the library.

Usage: python -m speculative_decoding_verification_30_gb300.tuner --alpha 0.7 --depths 1 2 4 8
"""
from __future__ import annotations

import argparse
import json
from typing import Callable, Sequence


def acceptance_rates(hist: Sequence[int], K: int | None = None) -> list[float]:
    """Per-position conditional acceptance rates from a histogram of the
    accepted-prefix length n (hist[n] for n in 0..K; a trailing error bin, if
    present, is ignored). alpha_i = #{n > i} / #{n >= i}; NaN where no call
    reached position i."""
    h = [int(x) for x in hist]
    if K is None:
        K = len(h) - 2
    h = h[: K + 1]
    rates = []
    for i in range(K):
        reached = sum(h[i:])
        passed = sum(h[i + 1:])
        rates.append(passed / reached if reached else float("nan"))
    return rates


def expected_tokens(alpha: Sequence[float], k: int) -> float:
    """Expected tokens emitted per step when drafting k tokens: the accepted
    prefix plus the one replacement or bonus token, 1 + sum_{j=1..k} prod_{i<j} alpha_i."""
    if k < 0 or k > len(alpha):
        raise ValueError("k must lie in [0, len(alpha)]")
    total, run = 1.0, 1.0
    for i in range(k):
        if run == 0.0:
            break                       # no later position is reached (its rate may be NaN)
        run *= alpha[i]
        total += run
    return total


def iid_expected_tokens(a: float, k: int) -> float:
    """Closed form for a constant acceptance rate a: (1 - a^(k+1)) / (1 - a)."""
    if a == 1.0:
        return float(k + 1)
    return (1.0 - a ** (k + 1)) / (1.0 - a)


def linear_cost(draft_cost: float) -> Callable[[int], float]:
    """Step cost in target-forward units: one target pass plus k draft passes, each
    draft_cost of a target pass (the verify step itself reads B(2k+1) logit rows and
    is part of the target pass)."""
    return lambda k: 1.0 + draft_cost * k


def choose_depth(alpha: Sequence[float], cost: Callable[[int], float] | None = None,
                 depths: Sequence[int] | None = None) -> tuple[int, dict[int, float]]:
    """The depth k (>= 1) with the most expected tokens per unit of step cost.
    Returns (best k, {k: tokens per cost}); ties go to the smaller depth."""
    cost = cost or linear_cost(0.0)
    depths = list(depths or range(1, len(alpha) + 1))
    score = {k: expected_tokens(alpha, k) / cost(k) for k in depths}
    best = min(depths, key=lambda k: (-score[k], k))
    return best, score


def sweep(alpha: float, depths: Sequence[int], B: int = 64, V: int = 151_936, T: float = 0.6,
          top_p: float = 0.95, steps: int = 4, seed: int = 1, device: str = "cuda") -> dict:
    """Measured acceptance per depth: for each K, `steps` synthetic batches (Zipf-like
    target rows, draft rows alpha * target + (1 - alpha) * independent), drafts d ~ q
    from spec_sample, verified by spec_verify, lengths counted by
    spec_accept_histogram. Returns per-K histograms, rates, measured and predicted
    tokens per step (inputs: the same seeded recipe as the benchmark workloads)."""
    import torch

    import speculative_decoding_verification_30_gb300 as sv
    from speculative_decoding_verification_30_gb300.workloads import Workload, make_batch

    out = {}
    for K in depths:
        w = Workload("nucleus_batch", B, K, V, torch.bfloat16, steps, cid=3)
        hist = torch.zeros(K + 2, dtype=torch.int64, device=device)
        ws = sv.Workspace(B, K, device)
        for step in range(steps):
            b = make_batch(w, 7000 + 2 * step, device=device)
            other = make_batch(w, 7001 + 2 * step, device=device).target[:, :K]   # independent rows
            b.draft.copy_((alpha * b.target[:, :K].float() + (1 - alpha) * other.float())
                          .to(b.draft.dtype))
            Tt = torch.full((B,), T, device=device)
            kk = torch.zeros(B, dtype=torch.int32, device=device)
            P = torch.full((B,), top_p, device=device)
            d = sv.spec_sample(b.draft, Tt, kk, P, seed=seed + 17, offset=step)
            _, n = sv.spec_verify(b.target, b.draft, d, Tt, kk, P, seed=seed, offset=step,
                                  workspace=ws)
            sv.spec_accept_histogram(n, K, hist)
        h = hist.cpu().tolist()
        rates = acceptance_rates(h, K)
        valid = sum(h[: K + 1])
        measured = sum((n + 1) * c for n, c in enumerate(h[: K + 1])) / max(1, valid)
        out[K] = {"hist": h, "rates": rates, "tokens_per_step": measured,
                  "predicted": expected_tokens(rates, K) if valid else float("nan")}
    return out


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--alpha", type=float, default=0.7, help="draft/target similarity of the synthetic rows")
    ap.add_argument("--depths", type=int, nargs="+", default=[1, 2, 3, 4, 6, 8])
    ap.add_argument("--B", type=int, default=64)
    ap.add_argument("--steps", type=int, default=4)
    ap.add_argument("--draft-cost", type=float, default=0.1,
                    help="one draft forward as a fraction of a target forward")
    args = ap.parse_args()
    res = sweep(args.alpha, args.depths, B=args.B, steps=args.steps)
    deepest = max(args.depths)
    best, score = choose_depth(res[deepest]["rates"], linear_cost(args.draft_cost),
                               [k for k in args.depths if k <= deepest])
    print(json.dumps({"alpha": args.alpha, "per_depth": res, "tokens_per_cost": score,
                      "chosen_depth": best}, indent=1))


if __name__ == "__main__":
    main()
