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
    return (list(r.tokens), r.n_accepted, r.n_draws, r.boundary, r.min_margin, r.error)


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
    boundary: int = 0
    mismatches: int = 0
    bad_mismatches: list = field(default_factory=list)

    def add(self, other: "ParityReport"):
        self.sequences += other.sequences
        self.draws += other.draws
        self.greedy += other.greedy
        self.boundary += other.boundary
        self.mismatches += other.mismatches
        self.bad_mismatches += other.bad_mismatches

    def __str__(self):
        return (f"seqs={self.sequences} draws={self.draws} greedy={self.greedy} "
                f"boundary_draw_seqs={self.boundary} mismatches={self.mismatches} "
                f"non_boundary_mismatches={len(self.bad_mismatches)}")


def compare(gpu_tokens, gpu_n, oracle_res, T) -> ParityReport:
    """Tokens and n must match exactly, except for sequences whose oracle draws
    include a boundary draw (margin < 1e-6); greedy sequences must match exactly."""
    rep = ParityReport()
    gt = gpu_tokens.cpu().numpy()
    gn = gpu_n.cpu().numpy()
    Tn = T.cpu().numpy()
    for b, (toks, n, draws, boundary, margin, err) in oracle_res.items():
        rep.sequences += 1
        rep.draws += draws
        greedy = Tn[b] == 0.0
        rep.greedy += int(greedy)
        rep.boundary += int(boundary)
        same = list(gt[b]) == toks and int(gn[b]) == n
        if not same:
            rep.mismatches += 1
            if greedy or not boundary:
                rep.bad_mismatches.append((b, list(gt[b]), int(gn[b]), toks, n, margin))
    return rep
