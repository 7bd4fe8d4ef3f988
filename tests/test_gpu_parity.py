"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle.

Bar (from the method's statement of exactness): token ids and n_accepted are
bit-exact, except for sequences whose oracle draws include a boundary draw
(an acceptance or sampling uniform within 1e-6 of its decision boundary); those
are counted and reported. A nucleus cut within 1e-6 of top_p is counted but
excuses no token mismatch; for the truncated probabilities such rows are left
out of the 1e-5 comparison (one tail token may sit on either side of the cut).
Temperature-0 rows are bit-exact with no exception. Truncated probabilities
agree within 1e-5.
"""
import math

import numpy as np
import pytest
import torch

import speculative_decoding_verification_30_gb300 as sv
from speculative_decoding_verification_30_gb300.workloads import (WORKLOADS, draft_tokens_by_rank,
                                                                   make_batch)
from oracle import sampler
from oracle.philox import philox4x32_10
from tests.parity_util import ParityReport, compare, f64, oracle_verify

pytestmark = pytest.mark.gpu
DEV = "cuda"
PROB_TOL = 1e-5


def _to(batch, dev=DEV):
    return (batch.target.to(dev), batch.draft.to(dev), batch.temperature.to(dev),
            batch.top_k.to(dev), batch.top_p.to(dev))


def _run(batch, dtok, seed, offset):
    tgt, drf, T, k, P = _to(batch)
    out, n = sv.spec_verify(tgt, drf, dtok.to(DEV), T, k, P, seed=seed, offset=offset)
    torch.cuda.synchronize()
    return out.cpu(), n.cpu()


# ------------------------------------------------------------------ Philox
def test_philox_stream_is_bit_exact():
    for seed, off in [(0, 0), (2**40 + 5, 2**33 + 17), (12345, 999)]:
        got = sv.spec_philox_uniforms(seed, off, 7, 5).cpu().numpy()
        for b in range(7):
            for i in range(5):
                w = philox4x32_10((i, b, off & 0xFFFFFFFF, off >> 32),
                                  (seed & 0xFFFFFFFF, seed >> 32))
                assert got[b, i, 0] == w[0] >> 8 and got[b, i, 1] == w[1] >> 8


# ------------------------------------------------------- truncated probs
def _ambiguous(z, T, k, P):
    """Tokens that may sit on either side of the nucleus cut: those whose exclusive
    renormalised mass (oracle, float64) lies within 1e-6 of top_p. Elsewhere the
    kernel's kept set must equal the oracle's."""
    if P >= 1.0:
        return set()
    V = z.shape[0]
    order = sampler.descending_order(z)
    kk = k if 0 < k < V else V
    top = order[:kk]
    e = np.exp((z[top] - z[order[0]]) / T)
    w = e / e.sum()
    excl = np.concatenate(([0.0], np.cumsum(w)[:-1]))
    return set(int(top[j]) for j in np.nonzero(np.abs(excl - P) < 1e-6)[0])


def _probs_case(rows, T, k, P):
    """Worst |p_gpu - p_ref| over the rows and the number of cut-near rows.

    p_ref is the oracle's float64 distribution on the kernel's kept set. That set
    must equal the oracle's kept set except for tokens whose exclusive mass lies
    within 1e-6 of top_p (where float64 and the kernel's exact fixed-point sums may
    place the cut on either side of one token); every other token is compared."""
    R = rows.shape[0]
    Tt = torch.full((R,), T) if np.isscalar(T) else T
    kt = torch.full((R,), k, dtype=torch.int32) if np.isscalar(k) else k
    Pt = torch.full((R,), P) if np.isscalar(P) else P
    got = sv.spec_truncated_probs(rows.to(DEV).contiguous(), Tt.float().to(DEV),
                                  kt.to(DEV), Pt.float().to(DEV)).cpu().double().numpy()
    z = f64(rows)
    worst, cut_near = 0.0, 0
    for r in range(R):
        Tr, kr, Pr = float(Tt[r]), int(kt[r]), float(Pt[r])
        t = sampler.truncate(z[r], Tr, kr, Pr)
        amb = _ambiguous(z[r], Tr, kr, Pr) if Tr > 0 else set()
        cut_near += int(bool(amb))
        kept_o = set(t.kept.tolist())
        kept_g = set(np.nonzero(got[r])[0].tolist())
        # weights below 2^-44 of the maximum are zero in the kernel's fixed point
        sig_o = set(np.nonzero(t.probs > 1e-12)[0].tolist())
        assert kept_g <= kept_o | amb, (r, sorted(kept_g - kept_o)[:5])
        assert sig_o <= kept_g | amb, (r, sorted(sig_o - kept_g)[:5])
        if Tr > 0:
            ref_set = np.array(sorted(kept_g | (kept_o - amb)))
            e = np.exp((z[r][ref_set] - z[r].max()) / Tr)
            ref = np.zeros_like(got[r])
            ref[ref_set] = e / e.sum()
        else:
            ref = t.probs
        worst = max(worst, float(np.max(np.abs(got[r] - ref))))
    return worst, cut_near


@pytest.mark.parametrize("name,B", [("tiny", 16), ("mtp_decode", 16), ("nucleus_batch", 4),
                                    ("mixed", 4)])
@pytest.mark.parametrize("side", ["target", "draft"])
def test_truncated_probs_match_oracle(name, B, side):
    # bf16 batches of at least 16 rows run the per-row code of the sampled verify path
    # (the key-histogram kernel); fp32 and smaller batches the cluster kernel
    w = WORKLOADS[name]
    b = make_batch(w, 0, B=B)
    rows = (b.target if side == "target" else b.draft).reshape(-1, w.V)
    per = w.K + 1 if side == "target" else w.K
    T = b.temperature.repeat_interleave(per)
    k = b.top_k.repeat_interleave(per)
    P = b.top_p.repeat_interleave(per)
    worst, cut_near = _probs_case(rows, T, k, P)
    print(name, side, "rows", rows.shape[0], "worst", worst, "cut-near rows", cut_near)
    assert worst < PROB_TOL, worst


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("V", [2, 3, 7, 33, 1000, 1023, 4096])
def test_truncated_probs_edge_shapes(dtype, V):
    g = torch.Generator().manual_seed(V)
    rows = (torch.randn(12, V, generator=g) * 3).to(dtype)
    rows[3] = torch.round(rows[3].float()).to(dtype)               # many ties
    rows[4, : V // 2] = -float("inf")                               # -inf is legal
    params = [(1.0, 0, 1.0), (0.7, 5, 1.0), (1.3, 0, 0.8), (0.5, 3, 0.5), (2.0, V, 0.99),
              (1.0, 1, 1.0), (0.9, 0, 0.05), (1e-3, 0, 1.0), (50.0, 0, 0.9), (1.0, 2, 0.999),
              (0.8, V - 1, 1.0), (1.0, 0, 0.5)]
    T = torch.tensor([p[0] for p in params])
    k = torch.tensor([p[1] for p in params], dtype=torch.int32)
    P = torch.tensor([p[2] for p in params])
    worst, cut_b = _probs_case(rows, T, k, P)
    assert worst < PROB_TOL, worst


@pytest.mark.parametrize("V", [4, 1000, 4096, 151_936])
def test_truncated_probs_fp32_rows_edge_cases(V):
    # 24 fp32 rows: ties, -inf, a top-k cut inside a run of equal logits, a maximum
    # far above the first load wave, flat rows, tiny and large temperatures
    g = torch.Generator().manual_seed(V + 5)
    rows = torch.randn(24, V, generator=g) * 2
    rows[1] = torch.round(rows[1])                                   # many ties
    rows[2, : V // 2] = -float("inf")
    rows[3] = torch.randn(V, generator=g) * 0.05                     # flat
    if V > 8:
        rows[4, -3:] = 60.0                                          # far above the first wave
        rows[5, V // 3: V // 3 + V // 4] = 1.5                       # a long run of equal logits
    params = [(1.0, 0, 0.9), (0.7, 5, 1.0), (1.3, 0, 0.8), (0.5, 3, 0.5), (2.0, V, 0.99),
              (1.0, 1, 1.0), (0.9, 0, 0.05), (1e-3, 0, 1.0), (50.0, 0, 0.9), (1.0, 2, 0.999),
              (0.8, V - 1, 1.0), (1.0, 0, 0.5)] * 2
    T = torch.tensor([p[0] for p in params])
    k = torch.tensor([p[1] for p in params], dtype=torch.int32)   # k = V - 1 > 256: handed back
    P = torch.tensor([p[2] for p in params])
    worst, cut_b = _probs_case(rows, T, k, P)
    assert worst < PROB_TOL, worst


def test_truncated_probs_top_k_large_and_ties_at_cut():
    # bf16 ties straddling the top-k and top-p cuts must split by token id
    V = 5000
    base = torch.zeros(V)
    base[100:400] = 2.0          # 300-way tie at the top
    base[4000:4100] = 1.0
    rows = torch.stack([base, base, base, base]).to(torch.bfloat16)
    T = torch.tensor([1.0, 1.0, 0.5, 1.0])
    k = torch.tensor([20, 700, 0, 350], dtype=torch.int32)
    P = torch.tensor([1.0, 0.3, 0.5, 0.9])
    worst, cut_b = _probs_case(rows, T, k, P)
    assert worst < PROB_TOL


# --------------------------------------------------------------- greedy
@pytest.mark.parametrize("B", [8, 256])
def test_greedy_is_bit_exact(B):
    w = WORKLOADS["greedy"]
    b = make_batch(w, 0, B=B)
    # drafted tokens: argmax of the draft row (the greedy drafter)
    dtok = b.draft.float().argmax(-1).to(torch.int32)
    out, n = _run(b, dtok, 1, 2)
    res = oracle_verify(b.target, None, dtok, b.temperature, b.top_k, b.top_p, 1, 2)
    rep = compare(out, n, res, b.temperature)
    assert rep.mismatches == 0, rep.bad_mismatches[:3]
    # every 5th sequence has draft == target: all K drafts accepted
    assert all(int(n[s]) == w.K for s in range(0, B, 5))


def test_greedy_without_draft_logits():
    w = WORKLOADS["greedy"]
    b = make_batch(w, 1, B=6)
    dtok = b.draft.float().argmax(-1).to(torch.int32)
    tgt, _, T, k, P = _to(b)
    out, n = sv.spec_verify(tgt, None, dtok.to(DEV), T, k, P, seed=0, offset=0)
    res = oracle_verify(b.target, None, dtok, b.temperature, b.top_k, b.top_p, 0, 0)
    assert compare(out.cpu(), n.cpu(), res, b.temperature).mismatches == 0


# ------------------------------------------------------------- sampling
@pytest.mark.parametrize("name,B,steps", [("tiny", 1, 60), ("mtp_decode", 1, 12),
                                           ("nucleus_batch", 16, 1), ("mixed", 24, 1)])
def test_verify_matches_oracle(name, B, steps):
    w = WORKLOADS[name]
    total = ParityReport()
    for step in range(steps):
        b = make_batch(w, step, B=B)
        dtok = draft_tokens_by_rank(b.draft, step, w.cid)
        out, n = _run(b, dtok, 1000 + step, step)
        res = oracle_verify(b.target, b.draft, dtok, b.temperature, b.top_k, b.top_p,
                            1000 + step, step)
        total.add(compare(out, n, res, b.temperature))
    print(name, total)
    assert not total.bad_mismatches, total.bad_mismatches[:3]


def test_identical_draft_rows_are_always_accepted():
    w = WORKLOADS["mixed"]
    b = make_batch(w, 3, B=16)
    b.draft.copy_(b.target[:, : w.K])
    dtok = draft_tokens_by_rank(b.draft, 3, w.cid)
    out, n = _run(b, dtok, 5, 5)
    # a drafted token outside the kept set has p = q = 0 and is rejected: compare to the oracle
    res = oracle_verify(b.target, b.draft, dtok, b.temperature, b.top_k, b.top_p, 5, 5)
    rep = compare(out, n, res, b.temperature)
    assert rep.mismatches == 0, [(m[0], m[1], m[2], m[3], m[4]) for m in rep.bad_mismatches]
    kept_all = [all(res[s][0][i] == int(dtok[s, i]) for i in range(w.K)) for s in range(16)]
    assert sum(kept_all) >= 4
    for s in range(16):
        if kept_all[s]:
            assert int(n[s]) == w.K


def test_repeated_calls_are_deterministic_and_reuse_the_workspace():
    w = WORKLOADS["nucleus_batch"]
    b = make_batch(w, 2, B=8)
    dtok = draft_tokens_by_rank(b.draft, 2, w.cid).to(DEV)
    tgt, drf, T, k, P = _to(b)
    ws = sv.Workspace(8, w.K)
    outs = [sv.spec_verify(tgt, drf, dtok, T, k, P, seed=9, offset=4, workspace=ws)
            for _ in range(5)]
    torch.cuda.synchronize()
    for o, n in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(n, outs[0][1])
    assert int(ws.buf.count_nonzero()) == 0       # the call leaves the workspace zeroed


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("V,K", [(2, 1), (7, 3), (33, 2), (1023, 4), (4097, 16)])
def test_verify_edge_shapes(dtype, V, K):
    g = torch.Generator().manual_seed(V * 31 + K)
    B = 6
    tgt = (torch.randn(B, K + 1, V, generator=g) * 2).to(dtype)
    drf = (0.5 * tgt[:, :K].float() + torch.randn(B, K, V, generator=g)).to(dtype)
    tgt[1] = torch.round(tgt[1].float()).to(dtype)        # ties
    tgt[2, :, : V // 2] = -float("inf")
    dtok = torch.randint(0, V, (B, K), generator=g, dtype=torch.int32)
    T = torch.tensor([1.0, 0.8, 1.1, 0.0, 0.5, 2.0])
    k = torch.tensor([0, 3, 0, 0, 1, V], dtype=torch.int32)
    P = torch.tensor([1.0, 0.9, 0.7, 1.0, 1.0, 0.95])
    out, n = sv.spec_verify(tgt.to(DEV), drf.to(DEV), dtok.to(DEV), T.to(DEV), k.to(DEV),
                            P.to(DEV), seed=3, offset=V)
    res = oracle_verify(tgt, drf, dtok, T, k, P, 3, V, parallel=False)
    rep = compare(out.cpu(), n.cpu(), res, T)
    assert not rep.bad_mismatches, rep.bad_mismatches


def test_verify_top_k_with_many_ties_at_the_kth_logit():
    # fp32 rows whose k-th largest logit is shared by hundreds or thousands of
    # tokens: the kept set is split by token id (ties ranked by ascending id)
    V, K, B = 8192, 2, 8
    g = torch.Generator().manual_seed(77)
    tgt = torch.randn(B, K + 1, V, generator=g) - 6.0
    drf = torch.randn(B, K, V, generator=g) - 6.0
    for s in range(B):
        ties = [3000, 500, 3000, 40, 1500, 700, 3000, 4000][s]
        idx = torch.randperm(V, generator=g)
        tgt[s, :, idx[:50]] = 2.0 + torch.rand(K + 1, 50, generator=g)
        tgt[s, :, idx[50:50 + ties]] = 1.0
        drf[s, :, idx[:50 + ties]] = 1.5
    dtok = torch.randint(0, V, (B, K), generator=g, dtype=torch.int32)
    T = torch.tensor([1.0, 0.7, 1.0, 1.2, 0.9, 1.0, 2.0, 1.0])
    k = torch.tensor([60, 60, 45, 80, 200, 256, 120, 100], dtype=torch.int32)
    P = torch.tensor([1.0, 1.0, 1.0, 0.9, 0.6, 1.0, 0.95, 1.0])
    out, n = sv.spec_verify(tgt.to(DEV), drf.to(DEV), dtok.to(DEV), T.to(DEV), k.to(DEV),
                            P.to(DEV), seed=8, offset=3)
    res = oracle_verify(tgt, drf, dtok, T, k, P, 8, 3, parallel=False)
    rep = compare(out.cpu(), n.cpu(), res, T)
    assert not rep.bad_mismatches, rep.bad_mismatches


def test_verify_top_p_with_maximum_far_above_the_first_wave():
    # fp32 top-p rows whose first 8192 logits are far below the row maximum: logits
    # 2^24 or more times heavier than the first wave's maximum are handled apart
    # from the binned bulk; the cut lies among them (P small), below them (many
    # tokens between), or they are too many and the row is served another way
    V, K, B = 32768, 2, 8
    g = torch.Generator().manual_seed(91)
    tgt = torch.randn(B, K + 1, V, generator=g) * 0.3
    drf = torch.randn(B, K, V, generator=g) * 0.3
    ln2 = math.log(2.0)
    for s in range(B):
        idx = 8192 + torch.randperm(V - 8192, generator=g)
        mode = s % 4
        for x in (tgt[s], drf[s]):
            if mode == 0:        # three tokens 30-45 binades up: the cut among them
                x[:, idx[:3]] = torch.tensor([45.0, 40.0, 30.0]) * ln2
            elif mode == 1:      # one token 25 binades up, 10000 tokens 20 binades up
                x[:, idx[:1]] = 25.0 * ln2
                x[:, idx[1:10001]] = 20.0 * ln2 + 0.3 * torch.randn(x.shape[0], 10000, generator=g)
            elif mode == 2:      # 300 tokens 30 binades up (more than are listed)
                x[:, idx[:300]] = 30.0 * ln2 + 0.1 * torch.randn(x.shape[0], 300, generator=g)
            else:                # the bulk 10 binades up, a ramp of single tokens above
                x[:, idx[:2000]] = 10.0 * ln2 + torch.randn(x.shape[0], 2000, generator=g)
                x[:, idx[2000:2040]] = torch.arange(40, dtype=torch.float32) * 0.8 * ln2
    dtok = torch.randint(0, V, (B, K), generator=g, dtype=torch.int32)
    T = torch.ones(B)
    k = torch.zeros(B, dtype=torch.int32)
    P = torch.tensor([0.5, 0.9, 0.95, 0.8, 0.99, 0.7, 0.6, 0.95])
    out, n = sv.spec_verify(tgt.to(DEV), drf.to(DEV), dtok.to(DEV), T.to(DEV), k.to(DEV),
                            P.to(DEV), seed=4, offset=12)
    res = oracle_verify(tgt, drf, dtok, T, k, P, 4, 12, parallel=False)
    rep = compare(out.cpu(), n.cpu(), res, T)
    assert not rep.bad_mismatches, rep.bad_mismatches


def test_verify_fp32_large_logits_and_small_temperatures():
    # fp32 rows offset by hundreds and low temperatures: (z - m) c must not pick up
    # the rounding of z c and m c separately (|m c| reaches 1e5 here)
    V, K, B = 8192, 2, 8
    g = torch.Generator().manual_seed(123)
    tgt = torch.randn(B, K + 1, V, generator=g) * 3 + 400.0
    drf = 0.6 * tgt[:, :K] + 0.4 * (torch.randn(B, K, V, generator=g) * 3 + 400.0)
    T = torch.tensor([0.01, 0.003, 0.05, 0.2, 0.01, 1.0, 0.02, 0.004])
    # drafted tokens the draft could have produced: its top token at the lowest
    # temperatures (where every other weight is below fp32's range on both rows),
    # its second one elsewhere
    ranks = drf.argsort(dim=-1, descending=True)
    dtok = torch.where((T < 0.05)[:, None], ranks[..., 0], ranks[..., 1]).to(torch.int32)
    k = torch.tensor([0, 0, 20, 0, 50, 0, 0, 5], dtype=torch.int32)
    P = torch.tensor([0.9, 1.0, 0.95, 0.8, 1.0, 0.99, 0.5, 1.0])
    out, n = sv.spec_verify(tgt.to(DEV), drf.to(DEV), dtok.to(DEV), T.to(DEV), k.to(DEV),
                            P.to(DEV), seed=6, offset=2)
    res = oracle_verify(tgt, drf, dtok, T, k, P, 6, 2, parallel=False)
    rep = compare(out.cpu(), n.cpu(), res, T)
    assert not rep.bad_mismatches, rep.bad_mismatches
    # the same rows' truncated probabilities
    rows = tgt.reshape(-1, V)
    worst, _ = _probs_case(rows, T.repeat_interleave(K + 1), k.repeat_interleave(K + 1),
                           P.repeat_interleave(K + 1))
    assert worst < PROB_TOL, worst


def test_data_errors_are_reported_in_band():
    V, K, B = 64, 2, 9
    tgt = torch.randn(B, K + 1, V)
    drf = torch.randn(B, K, V)
    dtok = torch.randint(0, V, (B, K), dtype=torch.int32)
    T = torch.ones(B)
    k = torch.zeros(B, dtype=torch.int32)
    P = torch.ones(B)
    tgt[0, 1, 5] = float("nan")
    drf[1, 0, 7] = float("inf")
    tgt[2, 2, :] = -float("inf")
    dtok[3, 1] = V
    T[4] = -1.0
    P[5] = 0.0
    k[6] = -3
    T[7] = float("nan")
    tgt[8, 0, 3] = float("nan")
    T[8] = 0.0                                        # greedy rows check their target rows too
    out, n = sv.spec_verify(tgt.to(DEV), drf.to(DEV), dtok.to(DEV), T.to(DEV), k.to(DEV),
                            P.to(DEV), seed=1, offset=1)
    out, n = out.cpu(), n.cpu()
    for s in range(B):
        assert int(n[s]) == -1 and bool((out[s] == -1).all()), s
    res = oracle_verify(tgt, drf, dtok, T, k, P, 1, 1, parallel=False)
    assert all(r[1] == -1 for r in res.values())


def test_missing_draft_with_positive_temperature_is_a_data_error():
    V, K, B = 64, 2, 3
    tgt = torch.randn(B, K + 1, V).to(DEV)
    dtok = torch.zeros(B, K, dtype=torch.int32, device=DEV)
    T = torch.tensor([0.0, 1.0, 0.0], device=DEV)
    out, n = sv.spec_verify(tgt, None, dtok, T, torch.zeros(B, dtype=torch.int32, device=DEV),
                            torch.ones(B, device=DEV), seed=0, offset=0)
    assert n.tolist()[1] == -1 and n.tolist()[0] >= 0 and n.tolist()[2] >= 0


# ------------------------------------------------------- draft sampler
@pytest.mark.parametrize("name", ["tiny", "nucleus_batch", "mixed"])
def test_draft_sampler_matches_oracle(name):
    w = WORKLOADS[name]
    b = make_batch(w, 4, B=8)
    got = sv.spec_sample(b.draft.to(DEV), b.temperature.to(DEV), b.top_k.to(DEV),
                         b.top_p.to(DEV), seed=77, offset=8).cpu().numpy()
    z = f64(b.draft)
    bad = 0
    for s in range(8):
        for i in range(w.K):
            from oracle.philox import uniforms
            _, v = uniforms(77, 8, s, i)
            tok, margin = sampler.sample_row(z[s, i], float(b.temperature[s]), int(b.top_k[s]),
                                             float(b.top_p[s]), v)
            # only a sampling uniform within 1e-6 of a CDF boundary excuses a difference
            if got[s, i] != tok and margin >= 1e-6:
                bad += 1
    assert bad == 0


# --------------------------------------------------- distribution (GPU)
@pytest.mark.parametrize("dtype,V", [(torch.float32, 8), (torch.bfloat16, 64)])
def test_gpu_output_distribution_is_the_truncated_target(dtype, V):
    # Monte Carlo over the sequences of one call (each with its own Philox
    # counter): the first emitted token is distributed as p_0, the truncated target
    # ("MTPLX", section 3.3: the verifier is exact). fp32 rows run the cluster
    # kernel; bf16 rows of a batch this size run the key-histogram kernel.
    # Marginals within 3 sigma, read for many tokens at once: with ~30 kept tokens
    # one of them lies beyond 3 sigma by chance in ~8% of runs, so at most one may,
    # none beyond 4 sigma; and a chi-square test over all kept tokens.
    from scipy.stats import chi2
    K, N = 2, 20000
    g = torch.Generator().manual_seed(5 + V)
    tgt = (torch.randn(1, K + 1, V, generator=g) * 1.5).to(dtype)
    drf = (0.5 * tgt[:, :K].float() + torch.randn(1, K, V, generator=g)).to(dtype)
    T, k, P = 1.0, 0, 0.9
    q = [sampler.truncate(f64(drf[0, i]), T, k, P).probs for i in range(K)]
    p0 = sampler.truncate(f64(tgt[0, 0]), T, k, P).probs
    rng = np.random.default_rng(0)
    dt = torch.tensor(np.stack([rng.choice(V, size=N, p=q[i] / q[i].sum()) for i in range(K)], 1),
                      dtype=torch.int32)
    tg = tgt.expand(N, K + 1, V).contiguous()
    dr = drf.expand(N, K, V).contiguous()
    out, n = sv.spec_verify(tg.to(DEV), dr.to(DEV), dt.to(DEV), torch.full((N,), T, device=DEV),
                            torch.zeros(N, dtype=torch.int32, device=DEV),
                            torch.full((N,), P, device=DEV), seed=11, offset=0)
    first = out[:, 0].cpu().numpy()
    assert (first >= 0).all()
    cnt = np.bincount(first, minlength=V)
    assert cnt[p0 == 0].sum() == 0                     # never a token outside the nucleus
    freq = cnt / N
    sigma = np.sqrt(p0 * (1 - p0) / N)
    z = np.abs(freq - p0) / np.maximum(sigma, 1e-300)
    print(dtype, "kept tokens", int((p0 > 0).sum()), "beyond 3 sigma", int((z > 3).sum()),
          "max sigma", float(z[p0 > 0].max()))
    assert int((z > 3).sum()) <= 1 and np.all(z <= 4), (freq, p0)
    kept = p0 > 0
    stat = float(np.sum((cnt[kept] - N * p0[kept]) ** 2 / (N * p0[kept])))
    assert chi2.sf(stat, int(kept.sum()) - 1) > 1e-3, stat
    acc = (n.cpu().numpy() >= 1).mean()
    expect = np.minimum(p0, q[0]).sum()
    assert abs(acc - expect) < 3 * math.sqrt(expect * (1 - expect) / N)
