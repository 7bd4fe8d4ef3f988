"""GPU parity of the key-histogram path (bf16 rows, 16-byte aligned, at least 16
verify units per call) against the float64 oracle, over its edge cases.

Tokens and n_accepted must equal the oracle's except on sequences with a
boundary draw (an acceptance or sampling uniform within 1e-6 of its decision
boundary); data errors must be reported as n = -1 with all tokens -1.
"""
import numpy as np
import pytest
import torch

import speculative_decoding_verification_30_gb300 as sv
from tests.parity_util import ParityReport, compare, oracle_verify

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _check(tgt, drf, dtok, T, k, P, seed, offset, label):
    out, n = sv.spec_verify(tgt.to(DEV), drf.to(DEV), dtok.to(DEV), T.to(DEV), k.to(DEV),
                            P.to(DEV), seed=seed, offset=offset)
    torch.cuda.synchronize()
    res = oracle_verify(tgt, drf, dtok, T, k, P, seed, offset)
    rep = compare(out.cpu(), n.cpu(), res, T)
    print(label, rep)
    assert not rep.bad_mismatches, (label, rep.bad_mismatches[:3])
    return out.cpu(), n.cpu(), rep


def _zipf(B, R, V, s, g, noise=0.5):
    """Rows z = -s ln(rank) + noise (a random permutation gives the ranks)."""
    ranks = torch.argsort(torch.rand(B * R, V, generator=g), dim=1).float() + 1.0
    return (-s * torch.log(ranks) + noise * torch.randn(B * R, V, generator=g)).view(B, R, V)


def _batch(B, K, V, g, s=1.1, alpha=0.7, quant=None):
    tgt = _zipf(B, K + 1, V, s, g)
    drf = alpha * tgt[:, :K] + (1 - alpha) * _zipf(B, K, V, s, g)
    if quant is not None:                         # coarse logits: long runs of equal values
        tgt = torch.round(tgt / quant) * quant
        drf = torch.round(drf / quant) * quant
    return tgt.to(torch.bfloat16), drf.to(torch.bfloat16)


def _drafts(drf, g):
    """Drafted tokens: mostly a high-ranked draft token, sometimes a random one."""
    B, K, V = drf.shape
    top = torch.topk(drf.float(), 8, dim=-1).indices
    pick = top.gather(-1, torch.randint(0, 8, (B, K, 1), generator=g)).squeeze(-1)
    rnd = torch.randint(0, V, (B, K), generator=g)
    return torch.where(torch.rand(B, K, generator=g) < 0.8, pick, rnd).to(torch.int32)


@pytest.mark.parametrize("V", [4096, 151_936])
def test_truncation_settings(V):
    # top-k only, top-p only, both, neither; several temperatures
    g = torch.Generator().manual_seed(V)
    B, K = 16, 4
    tgt, drf = _batch(B, K, V, g)
    dtok = _drafts(drf, g)
    T = torch.tensor([0.6, 1.0, 0.3, 1.5] * 4)
    k = torch.tensor([0, 20, 50, 0] * 2 + [1, 0, V - 1, 7] * 2, dtype=torch.int32)
    P = torch.tensor([0.95, 1.0, 0.8, 1.0] * 2 + [1.0, 0.5, 0.99, 0.9] * 2)
    total = ParityReport()
    for step in range(3 if V > 10_000 else 12):
        total.add(_check(tgt, drf, dtok, T, k, P, 11 + step, step, f"V={V} step {step}")[2])
    assert total.sequences > 0


def test_quantized_logits_force_tie_splits():
    # runs of equal bf16 logits at the cuts: target ties split from the kept
    # list, draft ties deferred to the finalizer
    g = torch.Generator().manual_seed(7)
    B, K, V = 16, 4, 8192
    total = ParityReport()
    for q in (0.25, 0.5, 1.0):
        tgt, drf = _batch(B, K, V, g, quant=q)
        dtok = _drafts(drf, g)
        T = torch.full((B,), 1.0)
        k = torch.tensor([0, 20, 100, 0] * 4, dtype=torch.int32)
        P = torch.tensor([0.9, 1.0, 0.95, 0.7] * 4)
        for step in range(6):
            total.add(_check(tgt, drf, dtok, T, k, P, 3, step, f"quant {q} step {step}")[2])
    assert total.sequences == 3 * 6 * 16


def test_drafted_tokens_on_the_draft_cut_value():
    # every drafted token sits on its draft row's cut value, so each acceptance
    # test needs the deferred id split of a partial cut bin
    g = torch.Generator().manual_seed(21)
    B, K, V = 16, 4, 4096
    tgt, drf = _batch(B, K, V, g, quant=0.5)
    T = torch.full((B,), 1.0)
    k = torch.full((B,), 40, dtype=torch.int32)
    P = torch.ones(B)
    zs = drf.float()
    dtok = torch.empty(B, K, dtype=torch.int32)
    for b in range(B):
        for i in range(K):
            kth = torch.sort(zs[b, i], descending=True).values[39]
            on = torch.nonzero(zs[b, i] == kth).flatten()
            dtok[b, i] = int(on[int(torch.randint(0, len(on), (1,), generator=g))])
    for step in range(4):
        _check(tgt, drf, dtok, T, k, P, 5, step, f"drafts on the cut, step {step}")


def test_flat_targets_use_the_full_row_pass():
    # flat targets: the nucleus is far below 2^-12 of the maximum, so no kept list
    g = torch.Generator().manual_seed(3)
    B, K, V = 16, 4, 32_768
    tgt, drf = _batch(B, K, V, g, s=0.3)
    dtok = _drafts(drf, g)
    T = torch.full((B,), 1.2)
    k = torch.zeros(B, dtype=torch.int32)
    P = torch.full((B,), 0.9)
    for step in range(3):
        _check(tgt, drf, dtok, T, k, P, 8, step, f"flat step {step}")


def test_masked_rows_and_data_errors():
    g = torch.Generator().manual_seed(5)
    B, K, V = 16, 4, 4096
    tgt, drf = _batch(B, K, V, g)
    dtok = _drafts(drf, g)
    ninf = -float("inf")
    tgt[0, :, 100:] = ninf                       # a heavily masked target
    drf[1, :, ::2] = ninf                        # a half-masked draft
    tgt[2, 3, :] = ninf                          # a target row with no finite logit: error
    drf[3, 1, 17] = float("nan")                 # NaN in a draft row: error
    tgt[4, 4, 99] = float("inf")                 # +inf in the bonus row: error
    T = torch.full((B,), 0.8)
    k = torch.tensor([0, 5] * 8, dtype=torch.int32)
    P = torch.tensor([0.9, 1.0] * 8)
    out, n, _ = _check(tgt, drf, dtok, T, k, P, 2, 0, "masked / errors")
    for b in (2, 3, 4):
        assert int(n[b]) == -1 and (out[b] == -1).all()


def test_count_overflow_and_constant_rows():
    # more than 65535 equal logits in one row overflows a 16-bit bin count: the
    # sequence is handed to the cluster kernel and must still match the oracle
    g = torch.Generator().manual_seed(9)
    B, K, V = 4, 4, 151_936
    tgt, drf = _batch(B, K, V, g)
    tgt[0, 1, :100_000] = 0.0
    drf[1, 2, 1000:80_000] = -3.0
    tgt[2] = 1.0                                  # constant target rows
    drf[3] = -2.0                                 # constant draft rows
    dtok = _drafts(drf, g)
    T = torch.tensor([1.0, 0.7, 1.0, 0.9])
    k = torch.tensor([0, 10, 0, 3], dtype=torch.int32)
    P = torch.tensor([0.9, 1.0, 0.5, 0.95])
    for step in range(3):
        _check(tgt, drf, dtok, T, k, P, 4, step, f"overflow step {step}")


def test_tiny_logits_share_the_merged_bin():
    # logits below 2^-40 in magnitude share one bin; a cut inside it with a
    # partial quota is handed to the cluster kernel
    g = torch.Generator().manual_seed(13)
    B, K, V = 16, 4, 4096
    tgt, drf = _batch(B, K, V, g)
    tiny = (torch.rand(V, generator=g) - 0.5) * 2.0 ** -42
    for b in range(0, B, 2):
        tgt[b, :, :] = tiny.to(torch.bfloat16)
        tgt[b, :, :3] = 5.0
    dtok = _drafts(drf, g)
    T = torch.full((B,), 1.0)
    k = torch.tensor([10, 0, 2000, 0] * 4, dtype=torch.int32)
    P = torch.tensor([1.0, 0.9, 1.0, 1.0] * 4)
    for step in range(3):
        _check(tgt, drf, dtok, T, k, P, 6, step, f"tiny logits step {step}")


@pytest.mark.parametrize("T", [3e-5, 0.05, 8.0, 1000.0])
def test_extreme_temperatures(T):
    g = torch.Generator().manual_seed(int(T * 100) + 1)
    B, K, V = 16, 4, 4096
    tgt, drf = _batch(B, K, V, g)
    dtok = _drafts(drf, g)
    Tt = torch.full((B,), T)
    k = torch.tensor([0, 20] * 8, dtype=torch.int32)
    P = torch.tensor([0.9, 1.0, 0.5, 1.0] * 4)
    for step in range(3):
        _check(tgt, drf, dtok, Tt, k, P, 1, step, f"T={T} step {step}")


def test_keyhist_workspace_stays_zeroed_and_calls_repeat():
    g = torch.Generator().manual_seed(17)
    B, K, V = 16, 4, 151_936
    tgt, drf = _batch(B, K, V, g, quant=0.25)
    dtok = _drafts(drf, g).to(DEV)
    T = torch.full((B,), 0.6, device=DEV)
    k = torch.tensor([0, 20] * 8, dtype=torch.int32, device=DEV)
    P = torch.full((B,), 0.95, device=DEV)
    ws = sv.Workspace(B, K)
    t, d = tgt.to(DEV), drf.to(DEV)
    outs = [sv.spec_verify(t, d, dtok, T, k, P, seed=9, offset=4, workspace=ws) for _ in range(4)]
    torch.cuda.synchronize()
    for o, n in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(n, outs[0][1])
    assert int(ws.buf.count_nonzero()) == 0


def test_huge_logits():
    # magnitudes far outside real logits (|z| >= 2^24): point masses and zero
    # weights at the ends of the bin range; every sequence must match the oracle
    g = torch.Generator().manual_seed(23)
    B, K, V = 16, 4, 4096
    tgt, drf = _batch(B, K, V, g)
    tgt[0, 1, 7] = 3.0e7                     # one huge positive logit (a point mass)
    drf[1, 0, 9] = -5.0e7                    # one huge negative logit (weight 0)
    tgt[2, :, 100] = 2.0e9
    drf[2, :, 100] = 2.0e9
    dtok = _drafts(drf, g)
    dtok[2, :] = 100
    T = torch.full((B,), 1.0)
    k = torch.tensor([0, 20] * 8, dtype=torch.int32)
    P = torch.tensor([0.95, 1.0] * 8)
    for step in range(3):
        _check(tgt, drf, dtok, T, k, P, 12, step, f"huge logits step {step}")


def _sample_check(drf, T, k, P, seed, offset, label):
    """spec_sample against the oracle's sample_row at Philox (b, i). A mismatch is
    allowed only for a sampling uniform within 1e-6 of a CDF boundary, or, where the
    nucleus cut lies within 1e-6 of top_p, for the token on either side of the cut
    (the only token that a cut decided the other way adds or drops)."""
    from oracle import sampler
    from oracle.philox import uniforms
    got = sv.spec_sample(drf.to(DEV), T.to(DEV), k.to(DEV), P.to(DEV), seed=seed,
                         offset=offset).cpu().numpy()
    z = drf.float().double().numpy()
    B, K, V = drf.shape
    bad, near_draw, near_cut = [], 0, 0
    for b in range(B):
        Tb, kb, Pb = float(T[b]), int(k[b]), float(P[b])
        for i in range(K):
            row = z[b, i]
            if np.isnan(row).any() or np.isposinf(row).any() or np.isneginf(row).all() or Pb <= 0:
                if got[b, i] != -1:
                    bad.append((b, i, int(got[b, i]), "error expected"))
                continue
            _, v = uniforms(seed, offset, b, i)
            tok, margin = sampler.sample_row(row, Tb, kb, Pb, v)
            edge = set()
            if Tb > 0:
                t = sampler.truncate(row, Tb, kb, Pb)
                if t.topp_margin < 1e-6:
                    near_cut += 1
                    order = sampler.descending_order(row)
                    n = len(t.kept)
                    edge = {int(order[n - 1])} | ({int(order[n])} if n < V else set())
            near_draw += int(margin < 1e-6)
            if got[b, i] != tok and margin >= 1e-6 and int(got[b, i]) not in edge:
                bad.append((b, i, int(got[b, i]), tok))
    print(label, "rows", B * K, "draws near a CDF boundary", near_draw,
          "cuts near top_p", near_cut, "bad", len(bad))
    assert not bad, bad[:4]


def test_draft_sampler_full_size_and_edge_rows():
    from speculative_decoding_verification_30_gb300.workloads import WORKLOADS, make_batch
    w = WORKLOADS["nucleus_batch"]
    b = make_batch(w, 3)
    _sample_check(b.draft, b.temperature, b.top_k, b.top_p, 4242, 10, "nucleus drafts B=64")
    g = torch.Generator().manual_seed(31)
    B, K, V = 16, 4, 8192
    _, drf = _batch(B, K, V, g, quant=0.5)
    drf[3, 1, :] = -float("inf")
    drf[3, 1, 5] = 2.0                                  # a single finite token
    drf[5, 2, 9] = float("nan")                         # data error
    T = torch.tensor([1.0, 0.6, 0.0, 1.3] * 4)          # T = 0 rows go to the cluster kernel
    k = torch.tensor([0, 20, 0, 3] * 4, dtype=torch.int32)
    P = torch.tensor([0.9, 1.0, 1.0, 0.7] * 4)
    P[7] = 0.0                                          # parameter error (top_p <= 0)
    for step in range(3):
        _sample_check(drf, T, k, P, 9, step, f"edge drafts step {step}")


def test_draft_sampler_many_rows_per_cta():
    # 640 rows on at most 304 CTAs: each CTA samples two or three rows in turn, so
    # the histogram and the shared scratch must be left clean between rows
    g = torch.Generator().manual_seed(77)
    B, K, V = 160, 4, 8192
    _, drf = _batch(B, K, V, g, quant=None)
    drf[::7] = torch.round(drf[::7].float() / 0.25).to(torch.bfloat16) * 0.25   # tie-heavy rows
    T = torch.tensor([0.6, 1.0, 0.8, 1.5] * (B // 4))
    k = torch.tensor([0, 40, 0, 7] * (B // 4), dtype=torch.int32)
    P = torch.tensor([0.95, 1.0, 0.5, 0.9] * (B // 4))
    _sample_check(drf, T, k, P, 2024, 3, "many rows per CTA")
