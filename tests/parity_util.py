"""Helpers for GPU-vs-oracle parity tests: run the CPU oracle on the same
inputs (optionally in a spawn-started process pool) and classify differences."""
from __future__ import annotations

import multiprocessing as mp
import os
from dataclasses import dataclass, field

import numpy as np
import torch

from oracle import sampler


def f64(t: torch.Tensor) -> np.ndarray:
    """Exact float64 copy of a bf16/fp32 tensor (host)."""
    return t.detach().to("cpu").float().double().numpy()


def _one(args):
    tgt, drf, d, T, k, P, seed, off, b = args
    r = sampler.verify_sequence(tgt, drf, d, T, k, P, seed, off, b)
    draw_margin = min([r.sample_margin, *r.accept_margins])
    return (list(r.tokens), r.n_accepted, r.n_draws, draw_margin, r.topp_margin, r.error)


_POOL = None


def pool():
    global _POOL
    if _POOL is None:
        n = min(16, max(1, (os.cpu_count() or 2) - 1))
        _POOL = mp.get_context("spawn").Pool(n)
    return _POOL


def oracle_verify(target, draft, dtok, T, k, P, seed, offset, seqs=None, parallel=True):
    """Oracle results for the selected sequences (all by default)."""
    B = target.shape[0]
    seqs = range(B) if seqs is None else seqs
    tg = f64(target)
    dr = None if draft is None else f64(draft)
    dt = dtok.cpu().numpy()
    Tn, kn, Pn = T.cpu().numpy(), k.cpu().numpy(), P.cpu().numpy()
    jobs = [(tg[b], None if dr is None else dr[b], dt[b].tolist(), float(Tn[b]), int(kn[b]),
             float(Pn[b]), seed, offset, b) for b in seqs]
    if parallel and len(jobs) > 4:
        res = pool().map(_one, jobs, chunksize=max(1, len(jobs) // 64))
    else:
        res = [_one(j) for j in jobs]
    return dict(zip(seqs, res))


@dataclass
class ParityReport:
    sequences: int = 0
    draws: int = 0
    greedy: int = 0
    boundary: int = 0          # sequences with a draw within 1e-6 of its decision boundary
    cut_near: int = 0          # sequences whose nucleus cut lies within 1e-6 of top_p
    mismatches: int = 0
    excused: int = 0           # mismatches on boundary-draw sequences
    bad_mismatches: list = field(default_factory=list)

    def add(self, other: "ParityReport"):
        for f in ("sequences", "draws", "greedy", "boundary", "cut_near", "mismatches",
                  "excused"):
            setattr(self, f, getattr(self, f) + getattr(other, f))
        self.bad_mismatches += other.bad_mismatches

    def __str__(self):
        return (f"seqs={self.sequences} draws={self.draws} greedy={self.greedy} "
                f"boundary_draw_seqs={self.boundary} cut_near_top_p_seqs={self.cut_near} "
                f"mismatches={self.mismatches} excused={self.excused} "
                f"non_boundary_mismatches={len(self.bad_mismatches)}")


def compare(gpu_tokens, gpu_n, oracle_res, T) -> ParityReport:
    """Tokens and n must match exactly, except for sequences with a boundary draw:
    an acceptance uniform or a sampling uniform within 1e-6 of its decision
    boundary. A nucleus cut near top_p is counted but excuses nothing (it is not
    a draw). Greedy sequences must match exactly."""
    rep = ParityReport()
    gt = gpu_tokens.cpu().numpy()
    gn = gpu_n.cpu().numpy()
    Tn = T.cpu().numpy()
    for b, (toks, n, draws, draw_margin, topp_margin, err) in oracle_res.items():
        rep.sequences += 1
        rep.draws += draws
        greedy = Tn[b] == 0.0
        boundary = draw_margin < sampler.BOUNDARY
        rep.greedy += int(greedy)
        rep.boundary += int(boundary)
        rep.cut_near += int(topp_margin < sampler.BOUNDARY)
        same = list(gt[b]) == toks and int(gn[b]) == n
        if not same:
            rep.mismatches += 1
            if greedy or not boundary:
                rep.bad_mismatches.append((b, list(gt[b]), int(gn[b]), toks, n, draw_margin))
            else:
                rep.excused += 1
    return rep
